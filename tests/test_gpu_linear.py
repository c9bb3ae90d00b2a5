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
