"""Pins for the oracle's per-token group quantisation (group 128).

Checked against properties the definition fixes, not against a retyped copy
of it: the element of largest magnitude in every group encodes to +-448, the
scale times 448 recovers amax to within one fp32 rounding, every element's
dequantised value is within half an e4m3 step of x, row- and column-major
scale layouts hold the same numbers, a bf16 input equals its exact fp32
widening, and ragged K only looks at the group's real elements.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_02_gb300 import workloads


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _groups(M, K):
    G = (K + 127) // 128
    return [(g * 128, min(K, g * 128 + 128)) for g in range(G)]


def _e4m3_ulp(y):
    """Spacing of e4m3 values around |y| (2^-9 in the subnormal range)."""
    y = np.abs(y)
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    return 2.0 ** (e - 3)


CASES = [
    ("normal", 7, 1024, False),
    ("student_t3", 5, 1000, False),      # ragged K: last group has 104 elements
    ("student_t3", 3, 300, False),
    ("uniform448", 4, 7168, True),       # the page's fp32 activations
]


def _make(kind, M, K, is_f32, seed=0):
    g = torch.Generator().manual_seed(seed)
    if kind == "uniform448":
        x = (torch.rand(M, K, generator=g) - 0.5) * 2 * 448
        return x.numpy().astype(np.float32), x.numpy().astype(np.float32)
    x = workloads.activations(M, K, seed, kind)
    bits = _bf16_bits(x)
    return bits, _widen(bits)


@pytest.mark.parametrize("kind,M,K,is_f32", CASES)
@pytest.mark.parametrize("col_major", [False, True])
def test_quant_invariants(oracle_mod, kind, M, K, is_f32, col_major):
    x_in, xf = _make(kind, M, K, is_f32)
    q, s = oracle_mod.group_quant(x_in, is_f32, col_major)
    tab = oracle_mod.e4m3_table()
    G = (K + 127) // 128
    scale = s[:G, :M].T if col_major else s[:, :G]          # [M, G]
    assert scale.shape == (M, G)
    for gi, (k0, k1) in enumerate(_groups(M, K)):
        blk = xf[:, k0:k1].astype(np.float64)
        amax = np.abs(blk).max(axis=1)
        sc = scale[:, gi].astype(np.float64)
        # scale * 448 recovers amax within one fp32 rounding of the division
        assert (np.abs(sc * 448.0 - amax) <= amax * 2.0 ** -23 + 1e-30).all()
        # the largest-magnitude element of the group encodes to +-448
        idx = np.abs(blk).argmax(axis=1)
        top = q[np.arange(M), k0 + idx]
        assert np.isin(top, [0x7E, 0xFE]).all()
        # dequantised values are within half an e4m3 step (plus the division's rounding)
        y = blk / sc[:, None]
        deq = tab[q[:, k0:k1]]
        err = np.abs(deq - y)
        assert (err <= 0.5 * _e4m3_ulp(y) + np.abs(y) * 2.0 ** -23).all()
        # sign is kept
        assert (np.signbit(deq) == np.signbit(blk)).all()


@pytest.mark.parametrize("kind,M,K,is_f32", CASES)
def test_layouts_hold_the_same_scales(oracle_mod, kind, M, K, is_f32):
    x_in, _ = _make(kind, M, K, is_f32)
    q_r, s_r = oracle_mod.group_quant(x_in, is_f32, False)
    q_c, s_c = oracle_mod.group_quant(x_in, is_f32, True)
    G = (K + 127) // 128
    assert (q_r == q_c).all()
    assert (s_c[:, :M].T == s_r[:, :G]).all()
    ld = s_c.shape[1]
    assert ld % 4 == 0 and ld >= M
    assert (s_c[:, M:] == 0).all()          # padding of the column-major layout


def test_bf16_input_equals_its_fp32_widening(oracle_mod):
    x_in, xf = _make("student_t3", 6, 640, False)
    q1, s1 = oracle_mod.group_quant(x_in, False, True)
    q2, s2 = oracle_mod.group_quant(xf, True, True)
    assert (q1 == q2).all() and (s1 == s2).all()


def test_zero_group_and_tiny_groups(oracle_mod):
    x = np.zeros((2, 256), dtype=np.float32)
    x[1, 128:] = -0.0
    x[1, 200] = 1e-12                       # amax below the 1e-10 floor
    q, s = oracle_mod.group_quant(x, True, False)
    assert (q[0] == 0).all()
    assert (s > 0).all()
    # floor: the scale is 1e-10/448 within an fp32 rounding when amax < 1e-10
    assert abs(float(s[0, 0]) * 448 - 1e-10) <= 1e-10 * 2.0 ** -22
    assert float(s[1, 1]) == float(s[0, 0])
    # 1e-12 / (1e-10/448) = 4.48 -> e4m3 4.5 (0x49)
    assert q[1, 200] == 0x49
    assert (q[1, 128:200] == 0x80).all()    # -0.0 keeps its sign


def test_ragged_k_uses_only_real_elements(oracle_mod):
    K = 1000                                # groups of 128 x 7 + 104
    x = np.ones((1, K), dtype=np.float32)
    x[0, 900] = 10.0                        # in the last (partial) group
    q, s = oracle_mod.group_quant(x, True, False)
    assert s.shape[1] == 8
    assert float(s[0, 7]) * 448 == pytest.approx(10.0, rel=2 ** -22)
    assert float(s[0, 0]) * 448 == pytest.approx(1.0, rel=2 ** -22)
    assert q[0, 900] == 0x7E


def test_agrees_with_an_independent_vectorised_restatement(oracle_mod):
    """Brute-force cross-check of indexing: numpy computes the groups' scales
    and quotients, torch's own float8_e4m3fn cast encodes them (all quotients
    are below 464 in magnitude, where torch's cast rounds the same way)."""
    x_in, xf = _make("normal", 9, 1000, False)
    q, s = oracle_mod.group_quant(x_in, False, False)
    for gi, (k0, k1) in enumerate(_groups(9, 1000)):
        blk = xf[:, k0:k1]
        amax = np.abs(blk).max(axis=1)
        sc = (np.maximum(amax, np.float32(1e-10)) / np.float32(448.0)).astype(np.float32)
        y = (blk / sc[:, None]).astype(np.float32)
        ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert (q[:, k0:k1] == ref).all()
        assert (s[:, gi] == sc).all()
