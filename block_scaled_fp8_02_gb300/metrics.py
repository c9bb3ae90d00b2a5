"""Work and traffic accounting for the blocked W8A8 FP8 linear layer.

Throughput is 2*M*N*K / t, the convention of the H200 latency table in
lmdeploy PR 4830 ("Performance" section), whose TFLOP/s column it reproduces.
Algorithmic bytes are what the method has to move at least once: the fp8
operands, their fp32 scales and the bf16 output (split-K scratch excluded).
"""
from __future__ import annotations


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def gemm_bytes(M: int, N: int, K: int) -> int:
    G = cdiv(K, 128)
    return M * K + 4 * M * G + N * K + 4 * cdiv(N, 128) * G + 2 * M * N


def quant_bytes(M: int, K: int, in_bytes: int = 2) -> int:
    """Activation read (bf16 or fp32), e4m3 write, fp32 scale write."""
    return in_bytes * M * K + M * K + 4 * M * cdiv(K, 128)


def tflops(M: int, N: int, K: int, us: float) -> float:
    return gemm_flops(M, N, K) / (us * 1e-6) / 1e12


def roofline_us(M: int, N: int, K: int, fp8_tflops: float, hbm_gbs: float) -> float:
    """max(compute time at the fp8 dense peak, algorithmic bytes at HBM bandwidth)."""
    t_c = gemm_flops(M, N, K) / (fp8_tflops * 1e12)
    t_m = gemm_bytes(M, N, K) / (hbm_gbs * 1e9)
    return max(t_c, t_m) * 1e6


def gemm_bound(M: int, N: int, K: int, fp8_tflops: float, hbm_gbs: float) -> str:
    t_c = gemm_flops(M, N, K) / (fp8_tflops * 1e12)
    t_m = gemm_bytes(M, N, K) / (hbm_gbs * 1e9)
    return "tensor" if t_c >= t_m else "hbm"
