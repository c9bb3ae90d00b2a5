"""GPU parity of the UE8M0 scale variant (transformers DeepGEMM integration,
`_ceil_to_ue8m0` and `_select_fp8_cast_kwargs` with use_ue8m0): activation
scales rounded up to powers of two -- codes and scales bit for bit against the
oracle's UE8M0 quantisation -- weight scales rounded the same way, and the
blocked GEMM on those scales against the oracle GEMM (every element)."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild
from block_scaled_fp8_02_gb300 import workloads as wl

from parity import check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    bfbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _oracle_quant(oracle_mod, x: torch.Tensor, col_major: bool):
    if x.dtype == torch.float32:
        return oracle_mod.group_quant(x.numpy(), True, col_major, ue8m0=True)
    return oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, col_major,
                                  ue8m0=True)


def _check_quant(oracle_mod, dev, x: torch.Tensor, col_major: bool):
    M, K = x.shape
    G = (K + 127) // 128
    q_ref, s_ref = _oracle_quant(oracle_mod, x, col_major)
    q, s = bf.bfp8_group_quant(x.to(dev), col_major=col_major, ue8m0=True)
    torch.cuda.synchronize()
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_ref)
    s_want = s_ref[:, :M].T if col_major else s_ref[:, :G]
    assert np.array_equal(s.cpu().numpy().view(np.uint32), np.ascontiguousarray(s_want).view(np.uint32))


@pytest.mark.parametrize("M,K,dist", [(1, 4096, "normal"), (64, 4096, "normal"), (2048, 4096, "normal"),
                                      (83, 7168, "student_t3"), (1000, 1000, "student_t3"),
                                      (3, 200, "student_t3"), (1, 1, "normal")])
@pytest.mark.parametrize("col_major", [True, False])
def test_ue8m0_quant_bitwise_vs_oracle(oracle_mod, dev, M, K, dist, col_major):
    _check_quant(oracle_mod, dev, wl.activations(M, K, seed=3 * M + K, dist=dist), col_major)


def test_ue8m0_quant_fp32_page_inputs_and_special_groups(oracle_mod, dev):
    _check_quant(oracle_mod, dev, wl.correctness_case()["x"], True)
    x = torch.zeros(3, 384, dtype=torch.float32)
    x[1, 200] = 1e-12                            # below the 1e-10 floor
    x[2, :] = torch.linspace(-1000, 1000, 384)
    x[2, 5] = 56.0 * 8                           # amax / 448 a power of two
    _check_quant(oracle_mod, dev, x, True)
    _check_quant(oracle_mod, dev, x.to(torch.bfloat16), False)


def test_scale_ceil_matches_the_oracle(oracle_mod, dev):
    rng = np.random.default_rng(3)
    s = np.concatenate([np.exp(rng.uniform(np.log(1e-12), np.log(1e6), 5000)),
                        2.0 ** np.arange(-40, 40), [1.0 / 448.0, 1e-10 / 448.0]]).astype(np.float32)
    s = np.concatenate([s, np.nextafter(s, np.float32(np.inf)), np.nextafter(s, np.float32(0))])
    got = bf.bfp8_scale_ceil_ue8m0(torch.from_numpy(s).to(dev)).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), oracle_mod.ceil_pow2(s).view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (64, 4096, 4096),
                                   (256, 4096, 4096), (2048, 4096, 4096), (83, 576, 7168),
                                   (1000, 1000, 1000)])
def test_ue8m0_linear_against_the_oracle(oracle_mod, dev, M, N, K):
    """The whole UE8M0 layer: activations quantised with power-of-two scales,
    weight scales rounded up by the library, then the blocked GEMM."""
    case = wl.linear_case(M, N, K, seed=M + 5) if K == 4096 else wl.ragged_case(M, N, K, seed=M)
    x = case["x"]
    Bs_pow2 = bf.bfp8_scale_ceil_ue8m0(case["Bs"].to(dev))
    out = bf.linear(x.to(dev), case["B"].to(dev), Bs_pow2, ue8m0=True)
    torch.cuda.synchronize()
    A, As = oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, True, ue8m0=True)
    Bs_ref = oracle_mod.ceil_pow2(case["Bs"].numpy())
    assert np.array_equal(Bs_pow2.cpu().numpy(), Bs_ref)
    ref = oracle_mod.blocked_gemm(A, case["B"].view(torch.uint8).numpy(), As, True, Bs_ref, want_abs=True)
    check_gemm(out, ref, (K + 127) // 128, label=f"ue8m0 linear {M}x{N}x{K}")
