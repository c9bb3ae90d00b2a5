"""GPU parity of the per-token group quantisation kernel: codes and fp32 scales
must equal the oracle's bit for bit, for both scale layouts, on the pages'
workloads (fp32 page inputs, bf16 N(0,1) activations at the sweep and
Qwen3-32B shapes, heavy-tailed ragged inputs) and on edge shapes."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild
from block_scaled_fp8_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    bfbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _oracle_quant(oracle_mod, x: torch.Tensor, col_major: bool):
    if x.dtype == torch.float32:
        return oracle_mod.group_quant(x.numpy(), True, col_major)
    return oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, col_major)


def _check(oracle_mod, dev, x_cpu: torch.Tensor, col_major: bool, x_dev=None):
    M, K = x_cpu.shape
    q_ref, s_ref = _oracle_quant(oracle_mod, x_cpu, col_major)
    x_dev = x_cpu.to(dev) if x_dev is None else x_dev
    q, s = bf.bfp8_group_quant(x_dev, col_major=col_major)
    torch.cuda.synchronize()
    q_np = q.view(torch.uint8).cpu().numpy()
    G = (K + 127) // 128
    s_np = s.cpu().numpy()                       # [M, G] view in either layout
    s_want = s_ref[:, :M].T if col_major else s_ref[:, :G]
    bad = np.nonzero(q_np != q_ref)
    assert bad[0].size == 0, f"{bad[0].size} codes differ, first at {bad[0][0], bad[1][0]}"
    assert (s_np.view(np.uint32) == np.ascontiguousarray(s_want).view(np.uint32)).all()


CASES = [(m, 4096, "normal") for m in (1, 9, 64, 256, 2048)] + \
        [(64, k, "normal") for k in (5120, 8192, 25600)] + \
        [(m, k, "student_t3") for m in (3, 83, 127, 1000) for k in (7168, 1000)] + \
        [(1, 1, "normal"), (5, 127, "student_t3"), (2, 129, "normal"), (7, 16, "normal"),
         (3, 200, "student_t3")]


@pytest.mark.parametrize("M,K,dist", CASES)
@pytest.mark.parametrize("col_major", [True, False])
def test_quant_bitwise_vs_oracle(oracle_mod, dev, M, K, dist, col_major):
    x = wl.activations(M, K, seed=M * 31 + K, dist=dist)
    _check(oracle_mod, dev, x, col_major)


@pytest.mark.parametrize("M,K,dist", [(1001, 4608, "normal"), (1024, 7168, "student_t3"),
                                      (4097, 1024, "normal")])
@pytest.mark.parametrize("col_major", [True, False])
def test_quant_large_dense_inputs(oracle_mod, dev, M, K, dist, col_major):
    """Large dense bf16 inputs: a step count that is not a multiple of the
    warps' walk, heavy tails, rows of two 512-element steps."""
    x = wl.activations(M, K, seed=M + 7 * K, dist=dist)
    _check(oracle_mod, dev, x, col_major)


@pytest.mark.parametrize("col_major", [True, False])
def test_quant_page_fp32_inputs(oracle_mod, dev, col_major):
    c = wl.correctness_case()
    _check(oracle_mod, dev, c["x"], col_major)


def test_quant_full_size_prefill(oracle_mod, dev):
    x = wl.activations(8192, 4096, seed=5)
    _check(oracle_mod, dev, x, True)


def test_quant_unaligned_rows_take_the_scalar_path(oracle_mod, dev):
    M, K = 9, 1000
    x = wl.activations(M, K + 1, seed=9, dist="student_t3")
    x_dev = x.to(dev)[:, 1:]                     # row stride K+1 elements: not 16-byte aligned
    _check(oracle_mod, dev, x[:, 1:].contiguous(), True, x_dev=x_dev)


def test_quant_special_groups(oracle_mod, dev):
    x = torch.zeros(3, 384, dtype=torch.float32)
    x[1, 128:256] = -0.0
    x[1, 200] = 1e-12                            # below the 1e-10 floor
    x[2, :] = torch.linspace(-1000, 1000, 384)   # max element encodes to +-448
    x[2, 300] = 3.0e-8
    _check(oracle_mod, dev, x, True)
    _check(oracle_mod, dev, x.to(torch.bfloat16), False)


def test_quotients_next_to_e4m3_rounding_boundaries(oracle_mod, dev):
    """Elements placed so that x / scale falls within a few fp32 ulps of the
    midpoints between e4m3 values (and in the e4m3 subnormal range), where a
    quotient that is not correctly rounded would change the code."""
    rng = np.random.default_rng(7)
    tab = oracle_mod.e4m3_table()
    mags = np.sort(np.unique(np.abs(tab[np.isfinite(tab)])))
    mids = (mags[:-1] + mags[1:]) / 2                       # every rounding boundary
    rows = []
    for amax in rng.uniform(0.5, 50.0, size=24).astype(np.float32):
        scale = np.float32(amax) / np.float32(448.0)          # the group's scale
        vals = []
        for mid in mids:
            base = np.float32(mid * np.float64(scale))
            for k in (-3, -2, -1, 0, 1, 2, 3):
                v = base
                step = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
                for _ in range(abs(k)):
                    v = np.nextafter(v, step)
                vals.append(v if rng.random() < 0.5 else -v)
        vals = np.array(vals, dtype=np.float32)
        vals = vals[np.abs(vals) < amax]
        for i in range(0, vals.size, 127):
            row = np.zeros(128, dtype=np.float32)
            chunk = vals[i:i + 127]
            row[:chunk.size] = chunk
            row[127] = amax                                   # fixes the group's scale
            rows.append(row)
    x = torch.from_numpy(np.stack(rows))
    _check(oracle_mod, dev, x, True)
    _check(oracle_mod, dev, x, False)


def test_exact_ties_from_bf16_inputs(oracle_mod, dev):
    """Groups whose amax is 448 have scale exactly 1, so x / scale = x: every
    bf16 value that is a midpoint between e4m3 values is an exact tie (to the
    even code).  bf16 activations meet such exact ties often."""
    rng = np.random.default_rng(17)
    tab = oracle_mod.e4m3_table()
    mags = np.sort(np.unique(np.abs(tab[np.isfinite(tab)])))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    rows = []
    for r in range(64):
        vals = rng.choice(mids, size=127) * rng.choice([-1.0, 1.0], size=127)
        vals = np.concatenate([vals.astype(np.float32), [np.float32(448.0)]])
        rng.shuffle(vals)
        rows.append(vals)
    x32 = torch.from_numpy(np.stack(rows).astype(np.float32))
    xb = x32.to(torch.bfloat16)
    assert torch.equal(xb.float(), x32)            # every midpoint is a bf16 value
    _check(oracle_mod, dev, xb, True)
    _check(oracle_mod, dev, xb, False)


@pytest.mark.parametrize("M,K,frac", [(300, 4096, 1.0), (97, 768, 1.0), (512, 4096, 0.02),
                                      (64, 25600, 0.3), (1024, 4096, 1.0), (1100, 4096, 0.3)])
def test_exact_ties_on_the_bf16_fast_path(oracle_mod, dev, M, K, frac):
    """Exact ties on the bf16 fast path (K a multiple of 256): a fraction
    `frac` of the elements are e4m3 midpoints in groups whose amax is 448
    (scale 1), up to every element of every warp step, so that the
    bracketing products disagree everywhere and the IEEE divisions decide."""
    rng = np.random.default_rng(M + K)
    tab = oracle_mod.e4m3_table()
    mags = np.sort(np.unique(np.abs(tab[np.isfinite(tab)])))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32) * 40.0
    tie = rng.random((M, K)) < frac
    x[tie] = rng.choice(mids, size=int(tie.sum())) * rng.choice([-1.0, 1.0], size=int(tie.sum()))
    x = np.clip(x, -447.0, 447.0)
    x[:, ::128] = 448.0                                  # every group's amax: scale 1
    xb = torch.from_numpy(x).to(torch.bfloat16)
    _check(oracle_mod, dev, xb, True)
    _check(oracle_mod, dev, xb, False)
