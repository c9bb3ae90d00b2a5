"""Pins for the oracle's M-grouped (mixture-of-experts) GEMM and fused linear.

The grouped GEMM of the transformers DeepGEMM integration (contiguous layout,
SM100 cumulative form) applies the plain blocked GEMM to each expert's block
of rows.  Pinned against: the row -> expert map written out by hand; brute
force (dequantise, fp64 matmul per expert) on tiny shapes; and the fact that a
row's result depends on its own expert's weights only."""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore")


def _case(oracle_mod, counts, N, K, seed):
    rng = np.random.default_rng(seed)
    E = len(counts)
    aligned = [((c + 127) // 128) * 128 for c in counts]
    psum = np.cumsum(aligned).astype(np.int32)
    M = int(psum[-1]) + 64                                       # rows past the last expert
    # integer-valued codes in [-16, 16] and power-of-two scales in [2^-2, 2^2]:
    # every product and every partial sum is exact in fp64, so any correct
    # evaluation order gives the same bf16
    tab = oracle_mod.e4m3_table()
    codes = np.array([c for c in range(256) if np.isfinite(tab[c]) and abs(tab[c]) <= 16
                      and tab[c] == np.round(tab[c])], dtype=np.uint8)
    A = rng.choice(codes, size=(M, K)).astype(np.uint8)
    B = rng.choice(codes, size=(E, N, K)).astype(np.uint8)
    G = (K + 127) // 128
    As = (2.0 ** rng.integers(-2, 3, size=(M, G))).astype(np.float32)
    Bs = (2.0 ** rng.integers(-2, 3, size=(E, (N + 127) // 128, G))).astype(np.float32)
    return A, B, As, Bs, psum


def test_rows_map_to_the_expert_whose_block_holds_them(oracle_mod):
    psum = np.array([128, 128, 384, 512], dtype=np.int32)         # expert 1 is empty
    rows = np.array([0, 127, 128, 383, 384, 511, 512, 900])
    assert oracle_mod.expert_of_rows(psum, rows).tolist() == [0, 0, 2, 2, 3, 3, -1, -1]


def test_grouped_equals_dequantised_fp64_matmul_per_expert(oracle_mod):
    A, B, As, Bs, psum = _case(oracle_mod, [100, 0, 130, 5], N=136, K=200, seed=3)
    res = oracle_mod.grouped_gemm(A, B, As, False, Bs, psum)
    tab = oracle_mod.e4m3_table()
    M = A.shape[0]
    E, N, K = B.shape
    G = (K + 127) // 128
    kb = np.arange(K) // 128
    ref_rows = 0
    for m in range(M):
        e = res["expert"][m]
        if e < 0:
            assert not res["bf16"][m].any()
            continue
        a = tab[A[m]] * As[m, kb].astype(np.float64)
        b = tab[B[e]] * Bs[e][np.arange(N)[:, None] // 128, kb[None, :]].astype(np.float64)
        want = oracle_mod.bf16_from_f64(b @ a)
        assert np.array_equal(res["bf16"][m], want)
        ref_rows += 1
    assert ref_rows == int(psum[-1])


def test_a_row_depends_on_its_own_experts_weights_only(oracle_mod):
    A, B, As, Bs, psum = _case(oracle_mod, [128, 256, 128], N=64, K=256, seed=5)
    base = oracle_mod.grouped_gemm(A, B, As, False, Bs, psum)["bf16"]
    B2 = B.copy()
    Bs2 = Bs.copy()
    B2[1] = np.flip(B2[1], axis=0)                              # change expert 1 only
    Bs2[1] *= 2.0
    got = oracle_mod.grouped_gemm(A, B2, As, False, Bs2, psum)["bf16"]
    rows_e1 = slice(int(psum[0]), int(psum[1]))
    others = np.ones(A.shape[0], dtype=bool)
    others[rows_e1] = False
    assert np.array_equal(got[others], base[others])
    assert not np.array_equal(got[rows_e1], base[rows_e1])


def test_one_expert_is_the_plain_blocked_gemm(oracle_mod):
    A, B, As, Bs, psum = _case(oracle_mod, [300], N=200, K=384, seed=7)
    got = oracle_mod.grouped_gemm(A, B, As, False, Bs, psum)
    plain = oracle_mod.blocked_gemm(A, B[0], As, False, Bs[0])["bf16"]
    n = int(psum[0])
    assert np.array_equal(got["bf16"][:n], plain[:n])


def test_bias_add_is_the_bf16_tensor_addition(oracle_mod):
    """The bias step is torch's bf16 + bf16 (computed in fp32, rounded once to
    bf16); compare with torch on CPU over random values and hand-made ties."""
    import torch
    rng = np.random.default_rng(11)
    y = rng.standard_normal((64, 300)).astype(np.float32) * np.float32(2.0) ** rng.integers(-20, 20, size=(64, 300))
    b = rng.standard_normal(300).astype(np.float32) * np.float32(2.0) ** rng.integers(-20, 20, size=300)
    yt = torch.from_numpy(y).to(torch.bfloat16)
    bt = torch.from_numpy(b).to(torch.bfloat16)
    want = (yt + bt).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.bias_add_bf16(yt.view(torch.int16).numpy().view(np.uint16),
                                   bt.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, want)
    # 1 + 2^-8 is a bf16 tie between 1 and 1 + 2^-7: to even (1.0)
    one = np.array([0x3F80], dtype=np.uint16)
    tiny = np.array([0x3B80], dtype=np.uint16)            # 2^-8
    assert oracle_mod.bias_add_bf16(one, tiny)[0] == 0x3F80


def test_fused_linear_is_gemm_then_bias_then_group_quant(oracle_mod):
    A, B, As, Bs, _ = _case(oracle_mod, [256], N=256, K=256, seed=13)
    B0, Bs0 = B[0], Bs[0]
    bias = np.random.default_rng(1).standard_normal(256).astype(np.float32)
    bias_bits = (bias.view(np.uint32) >> 16).astype(np.uint16)
    res = oracle_mod.fused_linear(A, B0, As, False, Bs0, bias_bits)
    y = oracle_mod.bias_add_bf16(oracle_mod.blocked_gemm(A, B0, As, False, Bs0)["bf16"], bias_bits)
    assert np.array_equal(res["bf16"], y)
    q, s = oracle_mod.group_quant(y, False, True)
    assert np.array_equal(res["q"], q) and np.array_equal(res["s"], s)


# Hand-made fused-linear cases.  Every GEMM value below is exact (one nonzero
# product per output, a power-of-two weight scale), so the expected bf16
# values, codes and scales follow from the definitions by hand:
#   e4m3 codes: 0x28 = 0.25, 0x38 = 1, 0x40 = 2, 0x48 = 4, 0x68 = 64, 0x70 = 128, 0x78 = 256,
#   0x71 = 144, 0x73 = 176, 0x76 = 224, 0x7E = 448 (bias 7, 3 mantissa bits).
_E4M3 = {1.0: 0x38, 2.0: 0x40, 4.0: 0x48, 64.0: 0x68, 128.0: 0x70, 256.0: 0x78, 0.25: 0x28}


def _bf16_bits(vals):
    return np.array([np.float32(v).view(np.uint32) >> 16 for v in vals], dtype=np.uint16)


def _one_group_case(b_rows, bs):
    """M=1, N=128, K=128; A[0] = (1, 1, 1, 0, ...); row n of B holds the codes
    b_rows[n] in its first columns; As = 1, Bs = bs."""
    A = np.zeros((1, 128), dtype=np.uint8)
    A[0, :3] = 0x38
    B = np.zeros((128, 128), dtype=np.uint8)
    for n, vals in b_rows.items():
        for k, v in enumerate(vals):
            B[n, k] = _E4M3[v]
    As = np.ones((1, 1), dtype=np.float32)
    Bs = np.full((1, 1), bs, dtype=np.float32)
    return A, B, As, Bs


def test_fused_linear_bias_moves_the_group_amax(oracle_mod):
    """GEMM row = (2, 1, 0, ...), bias = (0, 4, 0, ...): y = (2, 5, 0, ...).
    The amax is 5 at column 1 (it was 2 at column 0 before the bias), so
    scale = fl32(5 / 448), column 1 encodes to 448 (0x7E) and column 0 to
    e4m3(2 / scale) = e4m3(179.2...) = 176 (0x73); zeros stay 0x00."""
    A, B, As, Bs = _one_group_case({0: [128.0], 1: [64.0]}, 2.0 ** -6)
    bias = _bf16_bits([0.0, 4.0] + [0.0] * 126)
    res = oracle_mod.fused_linear(A, B, As, True, Bs, bias)
    assert res["bf16"][0, :2].tolist() == [0x4000, 0x40A0]          # 2.0, 5.0
    assert not res["bf16"][0, 2:].any()
    assert res["q"][0, 0] == 0x73 and res["q"][0, 1] == 0x7E
    assert not res["q"][0, 2:].any()
    assert res["s"][0, 0] == np.float32(5.0) / np.float32(448.0)


def test_fused_linear_rounds_the_gemm_to_bf16_before_the_bias(oracle_mod):
    """Column 0: the GEMM value is (256 + 1 + 0.25) * 2^-8 = 1 + 2^-8 + 2^-10,
    which rounds to bf16 1 + 2^-7; with bias -1 the layer output is
    bf16(2^-7) = 2^-7.  (Adding the bias before rounding would give
    2^-8 + 2^-10 = 1.25 * 2^-8 instead.)  Column 1: 4 * 2^-8 = 2^-6, no bias,
    the group's amax.  So scale = fl32(2^-6 / 448), column 1 encodes to 448
    (0x7E) and column 0 to e4m3(224) (0x76); the single-rounding value would
    have encoded to e4m3(140) = 144 (0x71)."""
    A, B, As, Bs = _one_group_case({0: [256.0, 1.0, 0.25], 1: [4.0]}, 2.0 ** -8)
    bias = _bf16_bits([-1.0] + [0.0] * 127)
    res = oracle_mod.fused_linear(A, B, As, True, Bs, bias)
    gemm = oracle_mod.blocked_gemm(A, B, As, True, Bs)["bf16"]
    assert gemm[0, 0] == 0x3F81                                      # 1 + 2^-7
    assert res["bf16"][0, 0] == 0x3C00                               # 2^-7
    assert res["bf16"][0, 1] == 0x3C80                               # 2^-6
    assert res["q"][0, 0] == 0x76 and res["q"][0, 1] == 0x7E
    assert res["s"][0, 0] == np.float32(2.0 ** -6) / np.float32(448.0)
