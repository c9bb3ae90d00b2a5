"""Pins for the oracle's blocked GEMM.

out[m,n] = bf16( sum_kb (A[m,kb].B[n,kb]) As[m,kb] Bs[n/128,kb] )

Checked against: an exact integer matmul (numpy int64) when every scale is 1;
an exact power-of-two-scaled integer result that exposes any mistake in the
(m, kb) / (n/128, kb) scale indexing or a transposed operand; a brute-force
dequantise-then-fp64-matmul (numpy, with torch decoding the fp8 codes) on
small ragged shapes; layout, row-subset and thread-count invariance; and the
pages' own acceptance bar on the page's correctness inputs.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_02_gb300 import workloads
from block_scaled_fp8_02_gb300.metrics import cdiv


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _int_codes(rng, shape, tab):
    """e4m3 codes whose values are the integers -16..16 (all exactly representable)."""
    vals = {int(v): c for c, v in enumerate(tab) if np.isfinite(v) and v == int(v) and abs(v) <= 16}
    keys = np.array(sorted(vals))
    pick = rng.integers(0, keys.size, size=shape)
    lut = np.array([vals[k] for k in keys], dtype=np.uint8)
    return lut[pick], keys[pick].astype(np.int64)


def _expand_as(As, col_major, M, K):
    G = cdiv(K, 128)
    a = As[:G, :M].T if col_major else As[:M, :G]
    return np.repeat(a.astype(np.float64), 128, axis=1)[:, :K]


def _expand_bs(Bs, N, K):
    return np.repeat(np.repeat(Bs.astype(np.float64), 128, axis=0), 128, axis=1)[:N, :K]


@pytest.mark.parametrize("M,N,K", [(37, 300, 1000), (5, 128, 128), (130, 257, 384)])
def test_unit_scales_give_the_exact_integer_matmul(oracle_mod, M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    tab = oracle_mod.e4m3_table()
    A, Ai = _int_codes(rng, (M, K), tab)
    B, Bi = _int_codes(rng, (N, K), tab)
    G = cdiv(K, 128)
    As = np.ones((M, G), dtype=np.float32)
    Bs = np.ones((cdiv(N, 128), G), dtype=np.float32)
    got = oracle_mod.blocked_gemm(A, B, As, False, Bs, want_f64=True)
    exact = Ai @ Bi.T                                  # |values| < 2^24: exact in fp32
    assert (got["f64"] == exact).all()
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
    ref = ref.view(torch.int16).numpy().view(np.uint16)
    assert (got["bf16"] == ref).all()


@pytest.mark.parametrize("col_major", [False, True])
def test_power_of_two_scales_are_indexed_by_m_kb_and_nblock_kb(oracle_mod, col_major):
    """Distinct power-of-two scales per (m, kb) and per (n/128, kb): the result is
    exact in fp64, so a swapped index, a transposed Bs or a dropped scale shows."""
    M, N, K = 9, 300, 700
    G, NT = cdiv(K, 128), cdiv(N, 128)
    rng = np.random.default_rng(3)
    tab = oracle_mod.e4m3_table()
    A, Ai = _int_codes(rng, (M, K), tab)
    B, Bi = _int_codes(rng, (N, K), tab)
    ea = rng.integers(-6, 7, size=(M, G))
    eb = rng.integers(-6, 7, size=(NT, G))
    As_mg = np.ldexp(1.0, ea).astype(np.float32)
    Bs = np.ldexp(1.0, eb).astype(np.float32)
    if col_major:
        ld = (M + 3) // 4 * 4
        As = np.zeros((G, ld), dtype=np.float32)
        As[:, :M] = As_mg.T
    else:
        As = As_mg
    got = oracle_mod.blocked_gemm(A, B, As, col_major, Bs, want_f64=True)["f64"]
    want = np.zeros((M, N))
    for kb in range(G):
        k0, k1 = kb * 128, min(K, kb * 128 + 128)
        d = Ai[:, k0:k1] @ Bi[:, k0:k1].T                         # exact integers
        want += d * np.ldexp(1.0, ea[:, kb])[:, None] * np.ldexp(1.0, eb[np.arange(N) // 128, kb])[None, :]
    assert (got == want).all()


@pytest.mark.parametrize("M,N,K,col_major", [(3, 130, 260, True), (17, 256, 129, False),
                                             (1, 1, 1, False), (64, 200, 1000, True)])
def test_matches_dequantise_then_fp64_matmul(oracle_mod, M, N, K, col_major):
    case = workloads.ragged_case(M, N, K, seed=M + N + K)
    x = case["x"].view(torch.int16).numpy().view(np.uint16)
    A, As = oracle_mod.group_quant(x, False, col_major)
    B = case["B"].view(torch.uint8).numpy()
    Bs = case["Bs"].numpy()
    res = oracle_mod.blocked_gemm(A, B, As, col_major, Bs, want_f64=True, want_abs=True)
    a = _torch_decode(A) * _expand_as(As, col_major, M, K)
    b = _torch_decode(B) * _expand_bs(Bs, N, K)
    ref = a @ b.T
    tol = res["abs"] * 1e-13 + 1e-300
    assert (np.abs(res["f64"] - ref) <= tol).all()
    # bf16 results agree except where ref sits within the fp64 noise of a tie
    ref_bf16 = oracle_mod.bf16_from_f64(ref)
    diff = np.nonzero(ref_bf16 != res["bf16"])[0]
    assert diff.size <= max(1, ref.size // 10000)


def test_layouts_rows_and_threads_do_not_change_the_result(oracle_mod):
    M, N, K = 23, 384, 1000
    case = workloads.ragged_case(M, N, K, seed=11)
    x = case["x"].view(torch.int16).numpy().view(np.uint16)
    A, As_r = oracle_mod.group_quant(x, False, False)
    _, As_c = oracle_mod.group_quant(x, False, True)
    B = case["B"].view(torch.uint8).numpy()
    Bs = case["Bs"].numpy()
    full = oracle_mod.blocked_gemm(A, B, As_r, False, Bs, threads=1)["bf16"]
    full_c = oracle_mod.blocked_gemm(A, B, As_c, True, Bs, threads=5)["bf16"]
    assert (full == full_c).all()
    rows = [22, 0, 7, 7]
    sub = oracle_mod.blocked_gemm(A, B, As_c, True, Bs, rows=rows, threads=3)["bf16"]
    assert (sub == full[rows]).all()


def test_page_correctness_case_meets_the_pages_bar(oracle_mod):
    """The vLLM PR 49932 digest's test (M=83, N=576, K=7168, seed 0) accepts
    rel_diff = mean|out-ref| / mean|ref| < 1e-3.  The oracle against an
    independent dequantise-then-matmul reference must be far inside it."""
    c = workloads.correctness_case()
    x = c["x"].numpy()
    A, As = oracle_mod.group_quant(x, True, True)
    B = c["B"].view(torch.uint8).numpy()
    Bs = c["Bs"].numpy()
    assert As.shape == (56, 84) and Bs.shape == (5, 56)
    res = oracle_mod.blocked_gemm(A, B, As, True, Bs, want_f64=True)
    ref = (_torch_decode(A) * _expand_as(As, True, 83, 7168)) @ \
          (_torch_decode(B) * _expand_bs(Bs, 576, 7168)).T
    def as_f64(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    out = as_f64(res["bf16"])
    # the page compares two bf16 outputs (kernel vs reference, both out_dtype=bf16)
    ref_bf16 = as_f64(oracle_mod.bf16_from_f64(ref))
    rel = np.abs(out - ref_bf16).mean() / np.abs(ref_bf16).mean()
    assert rel < 1e-6
    # against the unrounded reference only the final bf16 rounding remains
    rel_f64 = np.abs(out - ref).mean() / np.abs(ref).mean()
    assert rel_f64 < 2.0 ** -8
