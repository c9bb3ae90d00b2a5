"""bfp8_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Such callers (code inside a CUDA-graph capture that forbids cudaMalloc, plug-ins
whose host framework owns every device allocation, latency-critical loops that
must not allocate) cannot hand libbfp8 a workspace; this entry point uses the
scratch array built into the library instead.  Its results must match the
regular entry point's, within the same acceptance the other GEMM tests use,
on two calls in a row (the second call finds the first call's leftovers in the
shared scratch).  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild
from block_scaled_fp8_02_gb300 import workloads as wl

from parity import bf16_bits, bits_to_f64, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    bfbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _call_noalloc(A, B, As, Bs, out):
    M, K = A.shape
    N = B.shape[0]
    col = 1 if As.stride(0) == 1 else 0
    ld = As.stride(1) if col else As.stride(0)
    return bf.lib().bfp8_gemm_noalloc(
        A.data_ptr(), B.data_ptr(), As.data_ptr(), col, ld, Bs.data_ptr(), out.data_ptr(),
        M, N, K, torch.cuda.current_stream().cuda_stream)


def _same_within_tolerance(got: torch.Tensor, want: torch.Tensor):
    g = bits_to_f64(bf16_bits(got))
    w = bits_to_f64(bf16_bits(want))
    err = abs(g - w)
    assert (err <= 2 * ulp_bf16(w)).all()
    assert err.mean() / max(abs(w).mean(), 1e-30) < 1e-3


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (64, 4096, 4096), (32, 576, 7168),
                                   (3, 1000, 1000)])
def test_noalloc_matches_the_regular_entry_point_twice_in_a_row(dev, M, N, K):
    case = wl.ragged_case(M, N, K, seed=11 * M + N)
    q, s = bf.bfp8_group_quant(case["x"].to(dev))
    B = case["B"].to(dev)
    Bs = case["Bs"].to(dev)
    want = bf.bfp8_gemm(q, B, s, Bs)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        st = _call_noalloc(q, B, s, Bs, out)
        assert st == 0, bf.bfp8_last_error()
        torch.cuda.synchronize()
        _same_within_tolerance(out, want)


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    M, N, K = 2048, 5120, 8192            # 320 tiles: stream-K needs ~40 MB of partial sums
    need = bf.bfp8_gemm_workspace_size(M, N, K)
    assert need > ctypes.c_size_t(16 << 20).value
    G, NT = K // 128, N // 128
    A = torch.zeros((M, K), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    B = torch.zeros((N, K), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    As = torch.ones((G, M), device=dev).t()
    Bs = torch.ones((NT, G), device=dev)
    out = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    assert _call_noalloc(A, B, As, Bs, out) == 5            # BFP8_ERR_WORKSPACE
    assert "scratch" in bf.bfp8_last_error()
    torch.cuda.synchronize()
    assert float(out.float().abs().sum()) == 0.0            # nothing was launched
