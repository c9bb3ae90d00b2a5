"""GPU parity of the paired wide tiles (BFP8_PAIRS_ALWAYS): 256 x 256 output
tiles computed by CTA pairs with 2-SM MMAs.  Every row (or, at the largest
sizes, sampled rows) against the oracle: the prefill sweep, Qwen3-32B shapes,
ragged M, N and K (a tile's second half wholly past M; re-laid-out operands),
both scale layouts, weight prefetch, and bitwise determinism."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild
from block_scaled_fp8_02_gb300 import workloads as wl

from parity import check_gemm

pytestmark = pytest.mark.gpu

PAIRS = {"pairs": bf.PAIRS_ALWAYS}


@pytest.fixture(scope="module")
def dev():
    bfbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _run(oracle_mod, dev, case, col_major=True, options=PAIRS, rows=None, label=""):
    x = case["x"]
    M, N, K = case["M"], case["N"], case["K"]
    if x.dtype == torch.float32:
        A, As = oracle_mod.group_quant(x.numpy(), True, col_major)
    else:
        A, As = oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, col_major)
    B = case["B"].view(torch.uint8).numpy()
    Bs = case["Bs"].numpy()
    A_d = torch.from_numpy(A).to(dev).view(torch.float8_e4m3fn)
    B_d = torch.from_numpy(B).to(dev).view(torch.float8_e4m3fn)
    As_st = torch.from_numpy(As).to(dev)
    As_d = As_st[:, :M].t() if col_major else As_st
    Bs_d = torch.from_numpy(Bs).to(dev)
    plan = bf.bfp8_gemm_plan(M, N, K, 0, options)
    assert plan["pair"] == 1 and plan["grid"] % 2 == 0
    out = bf.bfp8_gemm(A_d, B_d, As_d, Bs_d, options=options)
    torch.cuda.synchronize()
    assert bf.bfp8_device_status() == 0
    ref = oracle_mod.blocked_gemm(A, B, As, col_major, Bs, rows=rows, want_abs=True)
    return check_gemm(out, ref, (K + 127) // 128, rows=rows, label=label), out


@pytest.mark.parametrize("M", [256, 512, 1024, 2048])
def test_prefill_sweep(oracle_mod, dev, M):
    _run(oracle_mod, dev, wl.linear_case(M, 4096, 4096, seed=100 + M), label=f"pairs M={M}")


def test_prefill_8192_sampled_rows(oracle_mod, dev):
    rows = np.concatenate([np.arange(0, 8192, 61), np.arange(8192 - 130, 8192)])
    _run(oracle_mod, dev, wl.linear_case(8192, 4096, 4096, seed=108), rows=rows, label="pairs M=8192")


@pytest.mark.parametrize("layer", list(wl.QWEN3_32B_LAYERS))
def test_qwen3_32b_layers_m2048(oracle_mod, dev, layer):
    N, K = wl.QWEN3_32B_LAYERS[layer]
    rows = np.arange(0, 2048, 29)
    _run(oracle_mod, dev, wl.linear_case(2048, N, K, seed=N + K), rows=rows, label=f"pairs {layer}")


@pytest.mark.parametrize("M,N,K", [(65, 256, 128), (300, 1000, 1000), (257, 384, 256),
                                   (1000, 576, 7168), (383, 4096, 2048), (129, 130, 4112)])
@pytest.mark.parametrize("col_major", [True, False])
def test_ragged(oracle_mod, dev, M, N, K, col_major):
    _run(oracle_mod, dev, wl.ragged_case(M, N, K, seed=M + N + K), col_major,
         label=f"pairs ragged {M}x{N}x{K}")


def test_prefetch_and_cta_cap(oracle_mod, dev):
    case = wl.linear_case(1024, 4096, 4096, seed=7)
    _run(oracle_mod, dev, case, options=dict(PAIRS, prefetch_weights=1), label="pairs prefetch")
    _run(oracle_mod, dev, case, options=dict(PAIRS, max_ctas=10), label="pairs 5 pairs")


def test_deterministic(dev):
    case = wl.linear_case(768, 2048, 4096, seed=3)
    q, s = bf.bfp8_group_quant(case["x"].to(dev))
    B, Bs = case["B"].to(dev), case["Bs"].to(dev)
    outs = [bf.bfp8_gemm(q, B, s, Bs, options=PAIRS).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
