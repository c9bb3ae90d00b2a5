"""The throughput formula bench.py reports, pinned to the pages' own table.

lmdeploy PR 4830 ("Performance" section) prints, for N=K=4096, each M's Gluon
latency and its TFLOP/s; 2*M*N*K / t must reproduce that column.
"""
import os

import pytest

from block_scaled_fp8_02_gb300 import metrics

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "h200_n4096_k4096.txt")


def _rows():
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                M, tri, glu, dg, tf = line.split()
                yield int(M), float(glu), float(tf)


@pytest.mark.parametrize("M,us,tf", list(_rows()))
def test_tflops_formula_reproduces_the_page_table(M, us, tf):
    assert metrics.tflops(M, 4096, 4096, us) == pytest.approx(tf, rel=5e-3, abs=0.01)


def test_algorithmic_bytes_and_bound():
    # M=1: one fp8 activation row, its 32 scales, the whole 16.8 MB weight, 32x32 scales, out
    assert metrics.gemm_bytes(1, 4096, 4096) == 4096 + 4 * 32 + 4096 * 4096 + 4 * 32 * 32 + 2 * 4096
    assert metrics.gemm_bound(1, 4096, 4096, 3948.0, 6684.0) == "hbm"
    assert metrics.gemm_bound(8192, 4096, 4096, 3948.0, 6684.0) == "tensor"
    assert metrics.quant_bytes(2, 256) == 2 * 512 + 512 + 4 * 2 * 2
