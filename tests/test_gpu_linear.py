"""End to end on the GPU: the whole layer (quantise, then GEMM) against the
oracle's quantise-then-GEMM; the bounded-wait failure path; and a clean
device failure word after all the work above."""
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


@pytest.mark.parametrize("M,N,K", [(83, 576, 7168), (1, 4096, 4096), (200, 1000, 1000),
                                   (1024, 4096, 4096)])
def test_linear_end_to_end(oracle_mod, dev, M, N, K):
    case = wl.correctness_case() if (M, N, K) == (83, 576, 7168) else wl.ragged_case(M, N, K, seed=M)
    x = case["x"]
    out = bf.linear(x.to(dev), case["B"].to(dev), case["Bs"].to(dev))
    torch.cuda.synchronize()
    if x.dtype == torch.float32:
        A, As = oracle_mod.group_quant(x.numpy(), True, True)
    else:
        A, As = oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, True)
    ref = oracle_mod.blocked_gemm(A, case["B"].view(torch.uint8).numpy(), As, True,
                                  case["Bs"].numpy(), want_abs=True)
    check_gemm(out, ref, (K + 127) // 128, label=f"linear {M}x{N}x{K}")


def _quant_then_gemm(x, B, Bs, options):
    q, s = bf.bfp8_group_quant(x, col_major=True)
    return bf.bfp8_gemm(q, B, s, Bs, options=options)


@pytest.mark.parametrize("M,N,K,ld_pad,options", [
    (1, 4096, 4096, 0, None), (16, 4096, 4096, 64, None), (3, 576, 7168, 0, {"k_split": 2}),
    (3, 1000, 1040, 0, None),          # K % 128 != 0
    (4, 4096, 4096, 3, None),          # rows of x not 16-byte aligned
    (100, 1000, 1024, 0, {"k_split": 1}),
    (1, 5120, 25600, 0, None),
    (8, 1000, 128, 0, None), (5, 4100, 384, 8, None), (13, 2000, 1152, 0, None),
    (7, 16, 4096, 0, {"max_ctas": 3}), (2, 51200, 5120, 0, None),
    (2048, 4096, 4096, 0, None)])
def test_bfp8_linear(oracle_mod, dev, M, N, K, ld_pad, options):
    """bfp8_linear (one library call: quantisation into the workspace, then
    the GEMM) is bitwise the two-call result and matches the oracle; x may
    have a row stride other than K."""
    case = wl.ragged_case(M, N, K, seed=5 * M + K)
    xs = torch.zeros((M, K + ld_pad), dtype=torch.bfloat16)
    xs[:, :K] = case["x"]
    x = xs.to(dev)[:, :K]
    B, Bs = case["B"].to(dev), case["Bs"].to(dev)
    out = bf.bfp8_linear(x, B, Bs, options=options)
    two = _quant_then_gemm(x, B, Bs, dict(options or {}, prefetch_weights=1))
    torch.cuda.synchronize()
    assert bf.bfp8_device_status() == 0
    assert torch.equal(out.view(torch.int16), two.view(torch.int16))
    rows = None if M * N * K <= 2e9 else np.arange(0, M, 97)
    A, As = oracle_mod.group_quant(case["x"].view(torch.int16).numpy().view(np.uint16), False, True)
    ref = oracle_mod.blocked_gemm(A, case["B"].view(torch.uint8).numpy(), As, True,
                                  case["Bs"].numpy(), rows=rows, want_abs=True)
    check_gemm(out, ref, (K + 127) // 128, rows=rows, label=f"bfp8_linear {M}x{N}x{K}")


def test_bounded_wait_gives_up_and_reports(dev):
    """A wait on a barrier nothing arrives on returns an error status after its
    cycle budget instead of hanging the GPU; the context stays usable."""
    st, elapsed = bf.bfp8_selftest_bounded_wait(2_000_000)      # ~1 ms
    assert st == 6, bf.bfp8_last_error()
    assert elapsed >= 2_000_000
    x = torch.ones(4, 4, device=dev)
    assert float((x * 2).sum()) == 32.0


def test_device_failure_word_is_clean(dev):
    case = wl.linear_case(16, 512, 512, seed=1)
    bf.linear(case["x"].to(dev), case["B"].to(dev), case["Bs"].to(dev))
    assert bf.bfp8_device_status(clear=True) == 0
