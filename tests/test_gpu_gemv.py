"""GPU parity of the warp-MMA kernel for a few activation rows (M <= 32,
BFP8_SCHEDULE_GEMV, TMA-fed mma.sync): every output element against the
oracle, on the decode sweep shapes, the Qwen3-32B layer shapes, ragged M and
N (a partial last weight tile, partial column groups, fewer k-blocks than a
stage or a box holds), both scale layouts and weight prefetch."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild
from block_scaled_fp8_02_gb300 import workloads as wl

from parity import check_gemm

pytestmark = pytest.mark.gpu

GEMV = {"schedule": bf.SCHEDULE_GEMV}


@pytest.fixture(scope="module")
def dev():
    bfbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _run(oracle_mod, dev, case, col_major=True, options=GEMV, label=""):
    x = case["x"]
    M, N, K = case["M"], case["N"], case["K"]
    A, As = oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, col_major)
    B = case["B"].view(torch.uint8).numpy()
    Bs = case["Bs"].numpy()
    A_d = torch.from_numpy(A).to(dev).view(torch.float8_e4m3fn)
    B_d = torch.from_numpy(B).to(dev).view(torch.float8_e4m3fn)
    As_st = torch.from_numpy(As).to(dev)
    As_d = As_st[:, :M].t() if col_major else As_st
    Bs_d = torch.from_numpy(Bs).to(dev)
    plan = bf.bfp8_gemm_plan(M, N, K, 0, options)
    assert plan["gemv"] == 1
    out = bf.bfp8_gemm(A_d, B_d, As_d, Bs_d, options=options)
    torch.cuda.synchronize()
    assert bf.bfp8_device_status() == 0
    ref = oracle_mod.blocked_gemm(A, B, As, col_major, Bs, want_abs=True)
    return check_gemm(out, ref, (K + 127) // 128, label=label)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 17, 24, 25, 31, 32])
def test_decode_sweep_shape(oracle_mod, dev, M):
    _run(oracle_mod, dev, wl.linear_case(M, 4096, 4096, seed=100 + M), label=f"gemv decode M={M}")


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("layer", list(wl.QWEN3_32B_LAYERS))
def test_qwen3_32b_layers(oracle_mod, dev, layer, M):
    N, K = wl.QWEN3_32B_LAYERS[layer]
    _run(oracle_mod, dev, wl.linear_case(M, N, K, seed=N + K + M), label=f"gemv {layer} M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (2, 130, 256), (3, 1000, 1024), (4, 576, 7168),
                                   (1, 300, 640), (8, 129, 4224), (6, 8, 2048 + 128),
                                   (8, 4100, 1024), (13, 1000, 7168), (32, 200, 384),
                                   (20, 4100, 1152), (27, 16, 512 + 128 * 3), (7, 5000, 1152),
                                   (3, 6000, 128 * 3)])
@pytest.mark.parametrize("col_major", [True, False])
def test_ragged(oracle_mod, dev, M, N, K, col_major):
    _run(oracle_mod, dev, wl.ragged_case(M, N, K, seed=M + N + K), col_major,
         label=f"gemv ragged {M}x{N}x{K}")


@pytest.mark.parametrize("M,ld", [(3, 16), (5, 5), (8, 12), (13, 36)])
def test_column_major_scale_strides(oracle_mod, dev, M, ld):
    """Column-major As whose stride rules out copying each stage's slice whole
    (ld_as above 8 x the column groups, or not a multiple of 4): the scale
    warp reads the scales instead."""
    case = wl.linear_case(M, 1000, 2048 + 128, seed=M + ld)
    x = case["x"]
    N, K = case["N"], case["K"]
    A, As = oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, True)
    G = (K + 127) // 128
    wide = np.zeros((G, ld), dtype=np.float32)
    wide[:, :M] = As[:, :M]
    A_d = torch.from_numpy(A).to(dev).view(torch.float8_e4m3fn)
    B_d = case["B"].to(dev)
    As_d = torch.from_numpy(wide).to(dev)[:, :M].t()
    out = bf.bfp8_gemm(A_d, B_d, As_d, case["Bs"].to(dev), options=GEMV)
    torch.cuda.synchronize()
    assert bf.bfp8_device_status() == 0
    ref = oracle_mod.blocked_gemm(A, case["B"].view(torch.uint8).numpy(), As, True, case["Bs"].numpy(),
                                  want_abs=True)
    check_gemm(out, ref, G, label=f"gemv As ld={ld} M={M}")


@pytest.mark.parametrize("M", [2, 24])
def test_prefetch_weights(oracle_mod, dev, M):
    _run(oracle_mod, dev, wl.linear_case(M, 4096, 4096, seed=5 + M),
         options=dict(GEMV, prefetch_weights=1), label=f"gemv prefetch M={M}")


@pytest.mark.parametrize("M,N,K,max_ctas", [(2, 5000, 2048, 7), (8, 6000, 1024, 0), (20, 3000, 1152, 0),
                                             (13, 5200, 640, 11), (1, 4880, 384, 0)])
def test_multi_wave(oracle_mod, dev, M, N, K, max_ctas):
    """More 16-row tiles than a wave of CTAs: persistent CTAs take tiles
    round-robin (three per SM up to 8 rows; few CTAs when capped; three
    activation column groups)."""
    options = dict(GEMV, max_ctas=max_ctas) if max_ctas else GEMV
    _run(oracle_mod, dev, wl.ragged_case(M, N, K, seed=M + N + K + max_ctas), True,
         options=options, label=f"gemv multi-wave {M}x{N}x{K} cap {max_ctas}")


def test_multi_wave_deterministic(dev):
    case = wl.linear_case(3, 5120, 25600, seed=11)
    q, s = bf.bfp8_group_quant(case["x"].to(dev))
    B, Bs = case["B"].to(dev), case["Bs"].to(dev)
    outs = [bf.bfp8_gemm(q, B, s, Bs, options=GEMV).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert bf.bfp8_device_status() == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("M,max_ctas", [(5, 1), (5, 3), (1, 7), (13, 5), (30, 2)])
def test_max_ctas(oracle_mod, dev, M, max_ctas):
    """Few persistent CTAs: many tiles per CTA, the stage ring wraps many times."""
    _run(oracle_mod, dev, wl.linear_case(M, 1000, 2048 + 384, seed=M + max_ctas),
         options=dict(GEMV, max_ctas=max_ctas), label=f"gemv M={M} max_ctas={max_ctas}")


def test_deterministic(dev):
    case = wl.linear_case(20, 2048, 4096, seed=9)
    q, s = bf.bfp8_group_quant(case["x"].to(dev))
    B, Bs = case["B"].to(dev), case["Bs"].to(dev)
    outs = [bf.bfp8_gemm(q, B, s, Bs, options=GEMV).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
