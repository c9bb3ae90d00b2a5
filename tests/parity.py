"""Helpers shared by the GPU parity tests: moving seeded inputs between the
oracle (numpy, CPU) and libbfp8 (torch, CUDA), and the acceptance checks.

Acceptance for the GEMM (bf16 outputs):
  - rel_diff = mean|out - ref| / mean|ref| < 1e-3, the bar of the vLLM PR
    49932 digest's test (section "key source snippet"), on bf16 vs bf16;
  - every element within 2 bf16 ulps of the oracle, except where the
    accumulation cancels: there |out - ref| may reach
    2 ulp(ref) + (G + 8) * 2^-24 * sum_kb |D_kb As Bs| -- the worst-case fp32
    accumulation error of G scaled block sums plus the tensor core's fp32
    block sums (the oracle reports that sum of magnitudes).
Elements beyond 2 ulps are counted; their share of a case's elements must
stay at or below OVER_2ULP_CEILING.  Every check records its statistics in
STATS, which the test session prints at the end (tests/conftest.py).
Quantisation is compared bit for bit (codes and fp32 scales).
"""
from __future__ import annotations

import numpy as np
import torch

# Largest share of a case's elements allowed beyond 2 bf16 ulps of the oracle
# (each of them must still satisfy the cancellation bound); a case of fewer
# than 1 / OVER_2ULP_CEILING elements may have one.
OVER_2ULP_CEILING = 1e-4

STATS: list[dict] = []


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(r: np.ndarray) -> np.ndarray:
    a = np.abs(r)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.maximum(2.0 ** (e - 7), 2.0 ** -133)


def check_gemm(out: torch.Tensor, ref: dict, G: int, rows=None, label: str = "") -> dict:
    """Compare a GPU bf16 output with the oracle's result (dict with 'bf16' bits
    and 'abs'); rows selects the output rows the oracle computed."""
    got_bits = bf16_bits(out if rows is None else out[torch.as_tensor(rows, device=out.device)])
    got = bits_to_f64(got_bits)
    want = bits_to_f64(ref["bf16"])
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = np.abs(got - want)
    denom = np.abs(want).mean()
    rel = float(err.mean() / denom) if denom > 0 else float(err.mean())
    two_ulp = 2 * ulp_bf16(want)
    over = err > two_ulp
    n_over = int(over.sum())
    if n_over:
        allowed = two_ulp + (G + 8) * 2.0 ** -24 * ref["abs"]
        bad = np.nonzero(err > allowed)
        assert bad[0].size == 0, (
            f"{label}: {bad[0].size} elements beyond the cancellation bound, e.g. "
            f"{[(int(i), int(j), got[i, j], want[i, j]) for i, j in zip(*bad)][:4]}")
    assert rel < 1e-3, f"{label}: rel_diff {rel}"
    exact = float((got_bits == ref["bf16"]).mean())
    frac = n_over / max(got.size, 1)
    # how much of the cancellation allowance the worst element used, in units
    # of 2^-24 * sum|terms|
    excess = 0.0
    if n_over:
        excess = float(((err - two_ulp)[over] / (2.0 ** -24 * np.maximum(ref["abs"][over], 1e-300))).max())
    stats = {"label": label, "elements": int(got.size), "rel_diff": rel, "over_2ulp": n_over,
             "over_2ulp_frac": frac, "max_excess_units": excess, "bitwise_equal_frac": exact}
    STATS.append(stats)
    assert n_over <= max(1, int(OVER_2ULP_CEILING * got.size)), (
        f"{label}: {n_over} of {got.size} elements beyond 2 ulp ({frac:.2e} > {OVER_2ULP_CEILING})")
    return stats
