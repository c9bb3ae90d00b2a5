"""GPU parity of the fused linear epilogue (bias add and the next layer's
1x128 group quantisation inside the GEMM).

The fused result must equal, bit for bit, the unfused composition on the GPU
(the GEMM on the same schedule, torch's bf16 bias addition, bfp8_group_quant),
and its codes and scales must equal the oracle's quantisation of the bf16
values the GEMM produced; the bf16 values themselves are checked against the
oracle GEMM with the usual GEMM acceptance."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild
from block_scaled_fp8_02_gb300 import workloads as wl

from parity import bf16_bits, check_gemm

pytestmark = pytest.mark.gpu

SCHED = {"schedule": 2, "k_split": 1}          # the schedule the fused epilogue runs


@pytest.fixture(scope="module")
def dev():
    bfbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _inputs(dev, M, N, K, seed):
    case = wl.ragged_case(M, N, K, seed=seed)
    x = case["x"].to(dev)
    q, s = bf.bfp8_group_quant(x)
    g = torch.Generator().manual_seed(seed)
    bias = (torch.randn(N, generator=g) * 0.5).to(torch.bfloat16).to(dev)
    return q, s, case["B"].to(dev), case["Bs"].to(dev), bias


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (300, 1000, 1000), (1000, 576, 7168),
                                   (2048, 4096, 4096), (129, 200, 384)])
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("col_major", [True, False])
def test_fused_equals_the_unfused_composition(dev, M, N, K, with_bias, col_major):
    A, As, B, Bs, bias = _inputs(dev, M, N, K, seed=M + N + K)
    b = bias if with_bias else None
    out, q, s = bf.bfp8_gemm_fused(A, B, As, Bs, bias=b, s_col_major=col_major)
    ref = bf.bfp8_gemm(A, B, As, Bs, options=SCHED)
    if with_bias:
        ref = ref + bias                       # torch: fp32 addition, rounded to bf16
    rq, rs = bf.bfp8_group_quant(ref, col_major=col_major)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(q.view(torch.uint8), rq.view(torch.uint8))
    assert torch.equal(s, rs)


def test_fused_quantisation_without_the_bf16_output(dev):
    A, As, B, Bs, bias = _inputs(dev, 512, 1024, 2048, seed=3)
    out, q, s = bf.bfp8_gemm_fused(A, B, As, Bs, bias=bias, want_out=False)
    assert out is None
    y = bf.bfp8_gemm(A, B, As, Bs, options=SCHED) + bias
    rq, rs = bf.bfp8_group_quant(y)
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.uint8), rq.view(torch.uint8)) and torch.equal(s, rs)


@pytest.mark.parametrize("M,N,K", [(300, 1000, 1000), (1000, 576, 7168)])
def test_fused_against_the_oracle(oracle_mod, dev, M, N, K):
    case = wl.ragged_case(M, N, K, seed=5 * M + K)
    A, As = oracle_mod.group_quant(case["x"].view(torch.int16).numpy().view(np.uint16), False, True)
    Bn = case["B"].view(torch.uint8).numpy()
    Bsn = case["Bs"].numpy()
    bias = (torch.randn(N, generator=torch.Generator().manual_seed(M)) * 0.25).to(torch.bfloat16)
    A_d = torch.from_numpy(A).to(dev).view(torch.float8_e4m3fn)
    As_d = torch.from_numpy(As).to(dev)[:, :M].t()
    out, q, s = bf.bfp8_gemm_fused(A_d, torch.from_numpy(Bn).to(dev).view(torch.float8_e4m3fn),
                                   As_d, torch.from_numpy(Bsn).to(dev), bias=bias.to(dev))
    torch.cuda.synchronize()
    bias_bits = bias.view(torch.int16).numpy().view(np.uint16)
    ref = oracle_mod.fused_linear(A, Bn, As, True, Bsn, bias_bits)
    check_gemm(out, ref, (K + 127) // 128, label=f"fused {M}x{N}x{K}")
    # codes and scales: the oracle's quantisation of the bf16 values the GPU produced
    y_gpu = bf16_bits(out)
    oq, osc = oracle_mod.group_quant(y_gpu, False, True)
    assert np.array_equal(q.cpu().view(torch.uint8).numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), osc[:, :M].T)
