"""bfp8_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Such callers (code inside a CUDA-graph capture that forbids cudaMalloc, plug-ins
whose host framework owns every device allocation, latency-critical loops that
must not allocate) cannot hand libbfp8 a workspace; this entry point uses the
scratch array built into the library instead.  Its results must equal the
regular entry point's bit for bit on two calls in a row (the second call finds
the first call's leftovers in the shared scratch) on every kernel family a
decode-sized call can take -- the warp-MMA decode kernel, 128- and 256-wide
tiles in clusters, swap-AB tiles, re-laid-out operands and scales in the
scratch -- and must meet the GEMM acceptance against the oracle.  (The
default plans split no decode-sized problem stream-K within the scratch: a
wide tile's fp32 partials need ~38 MB on a full grid; such problems are
rejected.)  This file is collected last on purpose.
"""
import ctypes

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


def _call_noalloc(A, B, As, Bs, out):
    M, K = A.shape
    N = B.shape[0]
    col = 1 if As.stride(0) == 1 else 0
    ld = As.stride(1) if col else As.stride(0)
    return bf.lib().bfp8_gemm_noalloc(
        A.data_ptr(), B.data_ptr(), As.data_ptr(), col, ld, Bs.data_ptr(), out.data_ptr(),
        M, N, K, torch.cuda.current_stream().cuda_stream)


def _shapes():
    # M = 1, 16: warp-MMA decode kernel; 64: 128-wide tiles, clusters of 4;
    # 200 x 2048: 256-wide tiles; 32 x 576: 128-wide, clusters of 8;
    # 3 x 1000 x 1000: re-laid-out operands and scales in the scratch
    return [(1, 4096, 4096), (16, 4096, 4096), (64, 4096, 4096), (200, 2048, 4096),
            (32, 576, 7168), (3, 1000, 1000)]


@pytest.mark.parametrize("shape", _shapes())
def test_noalloc_matches_the_regular_entry_point_twice_in_a_row(oracle_mod, dev, shape):
    """Bit for bit equal to bfp8_gemm (same plan, same kernels) on two calls in
    a row -- the second call finds the first call's leftovers in the shared
    scratch -- and, once, within the GEMM acceptance of the oracle."""
    M, N, K = shape
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
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    G = (K + 127) // 128
    s_st = torch.zeros((G, bf.bfp8_scale_ld(M)), dtype=torch.float32, device=dev)
    s_st[:, :M] = s.t()
    ref = oracle_mod.blocked_gemm(q.view(torch.uint8).cpu().numpy(), case["B"].view(torch.uint8).numpy(),
                                  s_st.cpu().numpy(), True, case["Bs"].numpy(), want_abs=True)
    check_gemm(out, ref, G, label=f"noalloc {M}x{N}x{K}")


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
