"""Shared pytest configuration.

Markers:
  gpu   -- needs a CUDA device (a GB300, sm_103a); run with ``-m gpu``.
Everything unmarked runs on a CPU-only machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: test needs a CUDA GB300 device (sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Per-case GEMM parity statistics of the GPU tests (elements beyond 2 bf16
    ulps of the oracle, bitwise-equal share, rel_diff)."""
    try:
        from parity import OVER_2ULP_CEILING, STATS
    except ImportError:
        return
    if not STATS:
        return
    tr = terminalreporter
    tr.section("GEMM parity against the oracle")
    n_el = sum(s["elements"] for s in STATS)
    n_over = sum(s["over_2ulp"] for s in STATS)
    worst = max(STATS, key=lambda s: s["over_2ulp_frac"])
    tr.write_line(f"{len(STATS)} checks, {n_el} elements compared; {n_over} beyond 2 ulp "
                  f"({n_over / max(n_el, 1):.2e}); ceiling per case {OVER_2ULP_CEILING:.0e}; "
                  f"worst case {worst['label']!r} {worst['over_2ulp_frac']:.2e}; max rel_diff "
                  f"{max(s['rel_diff'] for s in STATS):.2e}; largest cancellation excess "
                  f"{max(s['max_excess_units'] for s in STATS):.2f} x 2^-24 sum|terms|")
    for s in sorted(STATS, key=lambda s: -s["over_2ulp_frac"])[:25]:
        tr.write_line(f"  {s['label'][:60]:60s} n={s['elements']:>10d} over2ulp={s['over_2ulp']:>6d} "
                      f"({s['over_2ulp_frac']:.1e}) bitwise={s['bitwise_equal_frac']:.5f} "
                      f"rel={s['rel_diff']:.2e} excess={s['max_excess_units']:.2f}")
