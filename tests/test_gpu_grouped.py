"""GPU parity of the M-grouped (mixture-of-experts) blocked FP8 GEMM against
the oracle: the contiguous layout with 128-aligned expert blocks and the
cumulative row-count form of the transformers DeepGEMM integration."""
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


def _run(oracle_mod, dev, case, options=None, rows=None, label=""):
    M, N, K, E = case["M"], case["N"], case["K"], case["E"]
    A, As = oracle_mod.group_quant(case["x"].view(torch.int16).numpy().view(np.uint16), False, True)
    B = case["B"].view(torch.uint8).numpy()
    Bs = case["Bs"].numpy()
    psum = case["psum"].numpy()
    A_d = torch.from_numpy(A).to(dev).view(torch.float8_e4m3fn)
    As_d = torch.from_numpy(As).to(dev)[:, :M].t()
    B_d = torch.from_numpy(B).to(dev).view(torch.float8_e4m3fn)
    Bs_d = torch.from_numpy(Bs).to(dev)
    ps_d = torch.from_numpy(psum).to(dev)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    bf.bfp8_gemm_grouped(A_d, B_d, As_d, Bs_d, ps_d, out=out, options=options)
    torch.cuda.synchronize()
    last = int(psum[-1])
    # rows past the last expert are not written
    assert torch.isnan(out[last:].float()).all(), f"{label}: rows past the last expert written"
    if rows is None:
        rows = list(range(last))
    rows = [r for r in rows if r < last]
    ref = oracle_mod.grouped_gemm(A, B, As, True, Bs, psum, rows=rows, want_abs=True)
    return check_gemm(out, ref, (K + 127) // 128, rows=rows, label=label)


@pytest.mark.parametrize("counts,N,K", [
    ([300], 512, 1024),                       # one expert
    ([100, 0, 300, 37], 576, 2048),           # an empty expert, ragged blocks
    ([256] * 8, 1024, 1024),                  # DeepSeek-like: many experts, equal loads
    ([5, 130, 1, 260], 200, 1000),            # ragged N, K % 16 != 0 (re-laid operands)
])
@pytest.mark.parametrize("options", [None, {"k_split": 1}, {"tile_n": 128}])
def test_grouped_matches_oracle(oracle_mod, dev, counts, N, K, options):
    case = wl.grouped_case(counts, N, K, seed=sum(counts) + N + K, extra_rows=96)
    _run(oracle_mod, dev, case, options, label=f"grouped {counts} N={N} K={K} {options}")


def test_grouped_with_one_expert_equals_the_plain_gemm(dev):
    case = wl.grouped_case([384], 512, 768, seed=9)
    x = case["x"].to(dev)
    q, s = bf.bfp8_group_quant(x)
    B = case["B"].to(dev)
    Bs = case["Bs"].to(dev)
    ps = case["psum"].to(dev)
    plain = bf.bfp8_gemm(q, B[0].contiguous(), s, Bs[0].contiguous(), options={"schedule": 2})
    grouped = bf.bfp8_gemm_grouped(q, B, s, Bs, ps)
    torch.cuda.synchronize()
    assert torch.equal(plain.view(torch.int16), grouped.view(torch.int16))


def test_grouped_is_deterministic(dev):
    case = wl.grouped_case([200, 70, 0, 500], 1024, 2048, seed=4)
    x = case["x"].to(dev)
    q, s = bf.bfp8_group_quant(x)
    args = (q, case["B"].to(dev), s, case["Bs"].to(dev), case["psum"].to(dev))
    outs = [bf.bfp8_gemm_grouped(*args).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("layout", [[100, 256], [256, 128], [128, 130]])
def test_invalid_grouped_layout_is_reported_not_computed(dev, layout):
    """grouped_layout lives on the device, so the kernel checks it: entries
    that are not non-decreasing multiples of 128 make every CTA return before
    any copy, store or TMEM allocation and set the failure word; the output is
    left untouched and the context stays usable."""
    case = wl.grouped_case([128, 128], 256, 512, seed=2)
    x = case["x"].to(dev)
    q, s = bf.bfp8_group_quant(x)
    bad = torch.tensor(layout, dtype=torch.int32, device=dev)
    out = torch.zeros((case["M"], 256), dtype=torch.bfloat16, device=dev)
    assert bf.bfp8_device_status(clear=True) == 0
    bf.bfp8_gemm_grouped(q, case["B"].to(dev), s, case["Bs"].to(dev), bad, out=out)
    assert bf.bfp8_device_status(clear=True) == 5          # BFP8_DEV_BAD_GROUPED_LAYOUT
    assert not out.view(torch.int16).any()
    good = bf.bfp8_gemm_grouped(q, case["B"].to(dev), s, case["Bs"].to(dev), case["psum"].to(dev))
    torch.cuda.synchronize()
    assert good.view(torch.int16).any() and bf.bfp8_device_status(clear=True) == 0
