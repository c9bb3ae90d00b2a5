"""Seeded synthetic inputs for the blocked W8A8 FP8 linear layer.

This module only draws random numbers (torch's CPU generator, so the same
seed gives the same bytes on every machine) and holds none of the method's
arithmetic: activation quantisation and the GEMM are done by the library or
by the test oracle, never here.  Weights are produced the way the pages
produce them -- uniform values in [-448, 448], clamped and cast to
float8_e4m3fn by torch -- because a linear layer receives its weights already
in e4m3.

Workloads (shapes and distributions follow the pages):
  correctness  M=83, N=576, K=7168, seed 0, the exact draw order of
               test_w8a8_block_fp8_torch_scaled_mm_matmul (vLLM PR 49932
               digest, section "key source snippet").
  sweep        N=K=4096 and the M values of the H200 latency table
               (lmdeploy PR 4830, section "Performance"); activations bf16
               N(0,1), weight scales U[1e-4, 1e-2).
  qwen3_32b    the four linear shapes of a Qwen3-32B-sized decoder layer (the
               model the vLLM PR 19085 page serves); weights are synthetic.
  ragged       M in {3,83,127,1000}, N in {576,1000}, K in {7168,1000};
               heavy-tailed bf16 activations (Student-t, df=3), log-uniform
               weight scales in [1e-5, 1e-1].
"""
from __future__ import annotations

import math

import torch

FP8_MAX = 448.0
DECODE_MS = (1, 8, 9, 16, 24, 32, 64, 128, 160, 192, 224, 256)
PREFILL_MS = (512, 1024, 2048, 4096, 8192)
SWEEP_NK = 4096
QWEN3_32B_LAYERS = {          # name: (N, K)
    "qkv_proj": (10240, 5120),
    "o_proj": (5120, 8192),
    "gate_up_proj": (51200, 5120),
    "down_proj": (5120, 25600),
}
QWEN3_32B_MS = (1, 16, 64, 256, 2048)
RAGGED_MS = (3, 83, 127, 1000)
RAGGED_NS = (576, 1000)
RAGGED_KS = (7168, 1000)


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _weights_e4m3(N: int, K: int, g: torch.Generator) -> torch.Tensor:
    w = (torch.rand(N, K, generator=g, dtype=torch.float32) - 0.5) * 2 * FP8_MAX
    return w.clamp(min=-FP8_MAX, max=FP8_MAX).to(torch.float8_e4m3fn)


def correctness_case():
    """The page-2 correctness test's inputs, drawn in its order with seed 0.

    Returns dict(M, N, K, x_f32 [M,K] float32, B [N,K] e4m3, Bs [5,56] float32).
    x_f32 is the activation that the test quantises per token group.
    """
    M, N, K = 83, 576, 7168
    torch.manual_seed(0)
    a = (torch.rand(M, K, dtype=torch.float32) - 0.5) * 2 * FP8_MAX
    b = (torch.rand(N, K, dtype=torch.float32) - 0.5) * 2 * FP8_MAX
    B = b.clamp(min=-FP8_MAX, max=FP8_MAX).to(torch.float8_e4m3fn)
    Bs = torch.rand(cdiv(N, 128), cdiv(K, 128), dtype=torch.float32) * 1e-2
    return dict(M=M, N=N, K=K, x=a, x_is_f32=True, B=B, Bs=Bs)


def linear_case(M: int, N: int, K: int, seed: int):
    """Decode/prefill-style inputs: bf16 N(0,1) activations, e4m3 weights from
    U[-448, 448], weight scales U[1e-4, 1e-2)."""
    g = _gen(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    B = _weights_e4m3(N, K, g)
    Bs = 1e-4 + torch.rand(cdiv(N, 128), cdiv(K, 128), generator=g) * (1e-2 - 1e-4)
    return dict(M=M, N=N, K=K, x=x, x_is_f32=False, B=B, Bs=Bs.float())


def ragged_case(M: int, N: int, K: int, seed: int):
    """Tail-stress inputs: bf16 Student-t (df=3) activations, e4m3 weights from
    U[-448, 448], weight scales log-uniform in [1e-5, 1e-1]."""
    g = _gen(seed)
    # Student-t(3) = Z / sqrt(chi2_3 / 3), with chi2_3 the sum of 3 squared normals
    z = torch.randn(M, K, generator=g, dtype=torch.float64)
    chi2 = (torch.randn(3, M, K, generator=g, dtype=torch.float64) ** 2).sum(0)
    t = z / torch.sqrt(chi2 / 3.0)
    x = t.to(torch.float32).to(torch.bfloat16)
    B = _weights_e4m3(N, K, g)
    u = torch.rand(cdiv(N, 128), cdiv(K, 128), generator=g, dtype=torch.float64)
    Bs = torch.exp(math.log(1e-5) + u * (math.log(1e-1) - math.log(1e-5))).float()
    return dict(M=M, N=N, K=K, x=x, x_is_f32=False, B=B, Bs=Bs)


def activations(M: int, K: int, seed: int, dist: str = "normal") -> torch.Tensor:
    """bf16 activations only (quantisation-kernel workloads)."""
    g = _gen(seed)
    if dist == "normal":
        return torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if dist == "student_t3":
        z = torch.randn(M, K, generator=g, dtype=torch.float64)
        chi2 = (torch.randn(3, M, K, generator=g, dtype=torch.float64) ** 2).sum(0)
        return (z / torch.sqrt(chi2 / 3.0)).to(torch.float32).to(torch.bfloat16)
    raise ValueError(dist)


def e4m3_codes(N: int, K: int, seed: int) -> torch.Tensor:
    """Weights only, as e4m3 codes viewed as uint8."""
    return _weights_e4m3(N, K, _gen(seed)).view(torch.uint8)


def grouped_case(counts, N: int, K: int, seed: int, extra_rows: int = 0):
    """Mixture-of-experts inputs in the M-grouped contiguous layout: expert e
    owns counts[e] token rows, padded to a multiple of 128 (padding rows are
    zero activations); `extra_rows` rows past the last expert stand for the
    caller's upper bound on the row count.  bf16 N(0,1) activations, e4m3
    weights from U[-448, 448] per expert, weight scales U[1e-4, 1e-2).

    Returns dict(M, N, K, E, x [M,K] bf16, B [E,N,K] e4m3, Bs [E,NT,G] f32,
    psum [E] int32, valid [M] bool (rows that hold a token))."""
    g = _gen(seed)
    E = len(counts)
    aligned = [cdiv(c, 128) * 128 for c in counts]
    psum = torch.tensor(aligned, dtype=torch.int64).cumsum(0).to(torch.int32)
    M = int(psum[-1]) + extra_rows
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    valid = torch.zeros(M, dtype=torch.bool)
    start = 0
    for c, a in zip(counts, aligned):
        if c:
            x[start:start + c] = torch.randn(c, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
            valid[start:start + c] = True
        start += a
    B = torch.stack([_weights_e4m3(N, K, g) for _ in range(E)])
    Bs = 1e-4 + torch.rand(E, cdiv(N, 128), cdiv(K, 128), generator=g) * (1e-2 - 1e-4)
    return dict(M=M, N=N, K=K, E=E, x=x, B=B, Bs=Bs.float(), psum=psum, valid=valid)
