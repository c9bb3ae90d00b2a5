"""Pins for the oracle's UE8M0 scale variant.

The transformers DeepGEMM integration (`_ceil_to_ue8m0`, and
`_select_fp8_cast_kwargs` with use_ue8m0) rounds every fp32 scale up to the
nearest power of two -- the UE8M0 format keeps only the biased exponent -- and
quantises the activations with the rounded scale.  The oracle writes the
rounding from its definition (frexp); it is pinned here by hand-computed
values, by the page's own bit formulation of the same rounding (add 2^23 - 1
to the fp32 bit pattern, clear the 23 mantissa bits), by torch's float8 cast
of the exact quotients, and by the invariants the rounding implies."""
import numpy as np
import pytest
import torch


def _bits_round_up(s: np.ndarray) -> np.ndarray:
    """The page's formulation: (bits + 2^23 - 1) & ~(2^23 - 1) on the fp32 bits."""
    b = np.asarray(s, dtype=np.float32).view(np.int32).astype(np.int64)
    return ((b + (1 << 23) - 1) & ~((1 << 23) - 1)).astype(np.int32).view(np.float32)


def test_ceil_pow2_hand_values(oracle_mod):
    f32 = np.float32
    cases = {
        0.25: 0.25, 1.0: 1.0, 2.0 ** -42: 2.0 ** -42, 2.0 ** 20: 2.0 ** 20,   # already powers
        0.3: 0.5, 3.0: 4.0, 448.0: 512.0, 1.0 / 448.0: 2.0 ** -8,             # rounded up
        float(np.nextafter(f32(0.25), f32(1))): 0.5,                           # just above a power
        float(np.nextafter(f32(0.25), f32(0))): 0.25,                          # just below a power
        float(f32(1e-10) / f32(448.0)): 2.0 ** -42,                            # the amax floor's scale
        float(f32(5.0) / f32(448.0)): 2.0 ** -6,
    }
    got = oracle_mod.ceil_pow2(np.array(list(cases), dtype=np.float32))
    assert got.tolist() == [f32(v) for v in cases.values()]


def test_ceil_pow2_equals_the_pages_bit_formulation(oracle_mod):
    rng = np.random.default_rng(0)
    # random positive normal fp32 patterns, plus every power of two and its neighbours
    bits = rng.integers(0x00800000, 0x7F000000, size=20000, dtype=np.int64).astype(np.int32)
    pw = (np.arange(1, 254, dtype=np.int32) << 23)
    s = np.concatenate([bits.view(np.float32), pw.view(np.float32), (pw + 1).view(np.float32),
                        (pw - 1).view(np.float32)])
    s = s[np.isfinite(s) & (s > 0) & (s < 2.0 ** 127)]
    assert np.array_equal(oracle_mod.ceil_pow2(s), _bits_round_up(s))


@pytest.mark.parametrize("dist", ["normal", "student_t3"])
@pytest.mark.parametrize("M,K", [(7, 4096), (33, 1000), (2, 128)])
def test_ue8m0_group_quant_invariants(oracle_mod, dist, M, K):
    from block_scaled_fp8_02_gb300 import workloads as wl
    x = wl.activations(M, K, seed=M + K, dist=dist)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle_mod.group_quant(xb, False, False, ue8m0=True)
    q32, s32 = oracle_mod.group_quant(xb, False, False)
    xf = x.float().numpy()
    G = (K + 127) // 128
    for g in range(G):
        k0, k1 = 128 * g, min(128 * g + 128, K)
        amax = np.abs(xf[:, k0:k1]).max(axis=1)
        sc = s[:, g]
        # a power of two, the smallest one >= the fp32 scale amax / 448
        m, _ = np.frexp(sc.astype(np.float64))
        assert (m == 0.5).all()
        assert (sc >= s32[:, g]).all() and (sc / 2 < s32[:, g]).all()
        # the codes are torch's float8 cast of the exact quotients x / s
        want = torch.from_numpy(xf[:, k0:k1] / sc[:, None]).to(torch.float8_e4m3fn)
        assert np.array_equal(q[:, k0:k1], want.view(torch.uint8).numpy())
        # no saturation: |x / s| <= 448, and the group's largest element lands in (224, 448]
        top = np.abs(xf[:, k0:k1] / sc[:, None]).max(axis=1)
        assert ((top > 224) & (top <= 448)).all()
        # when amax / 448 is already a power of two the two variants coincide
        same = s32[:, g] == sc
        assert np.array_equal(q[same, k0:k1], q32[same, k0:k1])


def test_ue8m0_power_of_two_amax_matches_fp32_scales(oracle_mod):
    """amax = 448 * 2^-3: the fp32 scale is already 2^-3, so both variants give
    the same codes and scales; amax = 450 * 2^-3 rounds the scale up to 2^-2."""
    x = np.zeros((2, 128), dtype=np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 56.0, -7.0, 1.0           # 448 / 8 = 56
    x[1, 0], x[1, 1] = 56.25, 7.0                          # 450 / 8
    q, s = oracle_mod.group_quant(x, True, False, ue8m0=True)
    q32, s32 = oracle_mod.group_quant(x, True, False)
    assert s[0, 0] == 0.125 and s32[0, 0] == 0.125 and np.array_equal(q[0], q32[0])
    assert q[0, 0] == 0x7E and q[0, 1] == 0xE6 and q[0, 2] == 0x50   # 448, -56, 8
    assert s[1, 0] == 0.25
    # 56.25 / 0.25 = 225 -> 224 (0x76); 7 / 0.25 = 28 (0x5E)
    assert q[1, 0] == 0x76 and q[1, 1] == 0x5E


def test_ue8m0_all_zero_group(oracle_mod):
    q, s = oracle_mod.group_quant(np.zeros((1, 256), dtype=np.float32), True, True, ue8m0=True)
    assert (s[:, 0] == np.float32(2.0 ** -42)).all() and not q.any()
