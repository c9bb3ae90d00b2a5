"""GPU parity of the blocked FP8 GEMM against the oracle.

Every schedule computes the same function, so the page's correctness case is
run through each of them, through forced stream-K splits and through cluster
split-K at several cluster sizes.  Every output element is compared with the
oracle: the whole sweep at N=K=4096 (decode and prefill sizes, in the launch
configuration the bench times), the Qwen3-32B layer shapes and the
ragged/tail shapes (heavy-tailed activations, log-uniform weight scales,
K = 1000 with 1000-byte rows)."""
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


_cache = {}


def _prepare(oracle_mod, case, col_major=True):
    """Quantise the case's activations with the oracle and hand the same codes
    and scales to both sides."""
    key = (case["M"], case["N"], case["K"], id(case), col_major)
    if key in _cache:
        return _cache[key]
    x = case["x"]
    if x.dtype == torch.float32:
        A, As = oracle_mod.group_quant(x.numpy(), True, col_major)
    else:
        A, As = oracle_mod.group_quant(x.view(torch.int16).numpy().view(np.uint16), False, col_major)
    B = case["B"].view(torch.uint8).numpy()
    Bs = case["Bs"].numpy()
    _cache[key] = (A, As, B, Bs)
    return A, As, B, Bs


def _to_dev(dev, A, As, B, Bs, col_major, M):
    A_d = torch.from_numpy(A).to(dev).view(torch.float8_e4m3fn)
    B_d = torch.from_numpy(B).to(dev).view(torch.float8_e4m3fn)
    As_st = torch.from_numpy(As).to(dev)
    As_d = As_st[:, :M].t() if col_major else As_st
    Bs_d = torch.from_numpy(Bs).to(dev)
    return A_d, As_d, B_d, Bs_d


def _run(oracle_mod, dev, case, col_major=True, options=None, rows=None, label=""):
    M, N, K = case["M"], case["N"], case["K"]
    A, As, B, Bs = _prepare(oracle_mod, case, col_major)
    A_d, As_d, B_d, Bs_d = _to_dev(dev, A, As, B, Bs, col_major, M)
    out = bf.bfp8_gemm(A_d, B_d, As_d, Bs_d, options=options)
    torch.cuda.synchronize()
    ref = oracle_mod.blocked_gemm(A, B, As, col_major, Bs, rows=rows, want_abs=True)
    return check_gemm(out, ref, (K + 127) // 128, rows=rows, label=label), out


PAGE = wl.correctness_case()


@pytest.mark.parametrize("col_major", [True, False])
@pytest.mark.parametrize("options", [None, {"schedule": 1}, {"schedule": 2},
                                     {"schedule": 2, "tile_n": 128}, {"max_ctas": 7},
                                     {"schedule": 2, "max_ctas": 3}, {"schedule": 1, "max_ctas": 150},
                                     {"k_split": 1}, {"k_split": 2}, {"k_split": 2, "cluster_size": 3},
                                     {"schedule": 2, "k_split": 2}, {"k_split": 3},
                                     {"schedule": 2, "k_split": 3, "max_ctas": 3}])
def test_page_correctness_case_every_schedule(oracle_mod, dev, col_major, options):
    stats, _ = _run(oracle_mod, dev, PAGE, col_major, options, label=f"page {options}")
    assert stats["rel_diff"] < 1e-3


@pytest.mark.parametrize("M", wl.DECODE_MS)
@pytest.mark.parametrize("options", [None, {"schedule": 1}, {"schedule": 2, "tile_n": 256}])
def test_decode_sweep_full(oracle_mod, dev, M, options):
    """AUTO (warp-MMA decode kernel or wide tiles) and, explicitly, swap-AB and
    256-wide tiles with partial activation rows."""
    case = wl.linear_case(M, 4096, 4096, seed=100 + M)
    _run(oracle_mod, dev, case, options=options, label=f"decode M={M} {options}")


@pytest.mark.parametrize("M", wl.PREFILL_MS)
def test_prefill_sweep_full(oracle_mod, dev, M):
    case = wl.linear_case(M, 4096, 4096, seed=100 + M)
    _run(oracle_mod, dev, case, label=f"prefill M={M}")


@pytest.mark.parametrize("layer", list(wl.QWEN3_32B_LAYERS))
@pytest.mark.parametrize("M", wl.QWEN3_32B_MS)
def test_qwen3_32b_layers(oracle_mod, dev, layer, M):
    N, K = wl.QWEN3_32B_LAYERS[layer]
    case = wl.linear_case(M, N, K, seed=M + N + K)
    _run(oracle_mod, dev, case, label=f"{layer} M={M}")


@pytest.mark.parametrize("M", wl.RAGGED_MS)
@pytest.mark.parametrize("N", wl.RAGGED_NS)
@pytest.mark.parametrize("K", wl.RAGGED_KS)
@pytest.mark.parametrize("col_major", [True, False])
def test_ragged_tails(oracle_mod, dev, M, N, K, col_major):
    case = wl.ragged_case(M, N, K, seed=M * 7 + N + K)
    _run(oracle_mod, dev, case, col_major, label=f"ragged {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 8, 16), (2, 130, 129), (17, 256, 128),
                                   (129, 16, 300), (257, 384, 256), (300, 136, 4096)])
@pytest.mark.parametrize("options", [None, {"schedule": 1}, {"schedule": 2}])
def test_edge_shapes(oracle_mod, dev, M, N, K, options):
    case = wl.ragged_case(M, N, K, seed=M + 3 * N + 5 * K)
    _run(oracle_mod, dev, case, options=options, label=f"edge {M}x{N}x{K} {options}")


@pytest.mark.parametrize("options", [{"schedule": 2, "k_split": 1, "max_ctas": 7},
                                     {"schedule": 2, "k_split": 1, "max_ctas": 45},
                                     {"schedule": 2, "k_split": 3, "max_ctas": 5},
                                     {"schedule": 2, "tile_n": 128, "k_split": 1, "max_ctas": 11}])
def test_wide_weight_scale_windows(oracle_mod, dev, options):
    """Wide tiles read each column block's weight scales 32 k-blocks at a
    time, reloading at every segment start and every 32 units: stream-K runs
    over odd CTA counts start segments at k-blocks that are not multiples of
    32, and 56 k-blocks per tile cross a window boundary inside a segment."""
    case = wl.ragged_case(1000, 1000, 7168, seed=41)
    _run(oracle_mod, dev, case, label=f"windows {options}")


def test_unaligned_operands_and_output(oracle_mod, dev):
    """A and B starting 1 byte past a 16-byte boundary take the re-layout path;
    an output whose rows are not 16-byte aligned takes the element stores."""
    M, N, K = 37, 260, 512
    case = wl.ragged_case(M, N, K, seed=77)
    A, As, B, Bs = _prepare(oracle_mod, case, True)
    A_big = torch.zeros(M * K + 1, dtype=torch.uint8, device=dev)
    A_big[1:] = torch.from_numpy(A).reshape(-1).to(dev)
    B_big = torch.zeros(N * K + 1, dtype=torch.uint8, device=dev)
    B_big[1:] = torch.from_numpy(B).reshape(-1).to(dev)
    A_d = A_big[1:].view(M, K).view(torch.float8_e4m3fn)
    B_d = B_big[1:].view(N, K).view(torch.float8_e4m3fn)
    _, As_d, _, Bs_d = _to_dev(dev, A, As, B, Bs, True, M)
    out_big = torch.zeros(M * N + 1, dtype=torch.bfloat16, device=dev)
    out = out_big[1:].view(M, N)
    bf.bfp8_gemm(A_d, B_d, As_d, Bs_d, out=out)
    torch.cuda.synchronize()
    ref = oracle_mod.blocked_gemm(A, B, As, True, Bs, want_abs=True)
    check_gemm(out, ref, (K + 127) // 128, label="unaligned")
    assert float(out_big[0]) == 0.0


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (83, 576, 7168),
                                   (100, 1000, 1000), (129, 16, 300), (256, 4096, 1024),
                                   (600, 512, 4096), (257, 384, 256), (2, 130, 129)])
@pytest.mark.parametrize("cs", [0, 2, 3, 5, 8])
@pytest.mark.parametrize("schedule", [0, 1])
def test_cluster_split_k(oracle_mod, dev, M, N, K, cs, schedule):
    """Cluster split-K at every cluster size the planner may pick (0 = its
    own choice; explicit sizes are clamped to the tile's k-blocks): swap and
    wide tiles, ragged M, N and K, re-laid-out operands."""
    opts = {"k_split": 2, "cluster_size": cs, "schedule": schedule}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = bf.bfp8_gemm_plan(M, N, K, 0, opts)          # this device's plan
    G = plan["k_blocks"]
    if cs:
        assert plan["cluster"] == (min(cs, G) if G >= 2 else 1)
    elif G >= 2 and 2 * plan["tiles"] <= sms:
        assert 2 <= plan["cluster"] <= min(8, G) and plan["grid"] <= sms
    case = wl.ragged_case(M, N, K, seed=5 * M + N + K + cs)
    _run(oracle_mod, dev, case, options=opts, label=f"cluster {cs} s{schedule} {M}x{N}x{K}")


@pytest.mark.parametrize("options", [None, {"max_ctas": 5}, {"schedule": 2}, {"k_split": 2},
                                     {"k_split": 2, "cluster_size": 8}, {"k_split": 1},
                                     {"k_split": 3}])
def test_deterministic_across_calls(dev, options):
    case = wl.linear_case(96, 1024, 2048, seed=3)
    x = case["x"].to(dev)
    q, s = bf.bfp8_group_quant(x)
    B = case["B"].to(dev)
    Bs = case["Bs"].to(dev)
    outs = [bf.bfp8_gemm(q, B, s, Bs, options=options).clone() for _ in range(5)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_one_workspace_serves_problems_of_every_layout(oracle_mod, dev):
    """Calls with different workspace layouts (whole tiles only, stream-K,
    re-laid-out operands) share one workspace in turn; every result must stay
    correct, i.e. no call may leave non-zero counters for the next."""
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=dev)
    shapes = [(1, 8, 1), (2, 130, 129), (83, 576, 7168), (1, 8, 1), (300, 1000, 1000),
              (16, 4096, 512), (2, 130, 129), (1000, 576, 7168)]
    for M, N, K in shapes:
        case = wl.ragged_case(M, N, K, seed=M + N + K)
        A, As, B, Bs = _prepare(oracle_mod, case, True)
        A_d, As_d, B_d, Bs_d = _to_dev(dev, A, As, B, Bs, True, M)
        out = bf.bfp8_gemm(A_d, B_d, As_d, Bs_d, workspace=ws)
        torch.cuda.synchronize()
        ref = oracle_mod.blocked_gemm(A, B, As, True, Bs, want_abs=True)
        check_gemm(out, ref, (K + 127) // 128, label=f"shared ws {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (64, 4096, 4096), (300, 1024, 2048),
                                   (2048, 4096, 4096), (83, 576, 7168)])
def test_weight_prefetch_right_after_quantisation(oracle_mod, dev, M, N, K):
    """prefetch_weights=1: the GEMM requests weight tiles before the
    quantisation kernel launched just before it has finished (programmatic
    dependent launch), then waits for it before reading the activations."""
    case = wl.linear_case(M, N, K, seed=M + 17)
    x = case["x"].to(dev)
    B = case["B"].to(dev)
    Bs = case["Bs"].to(dev)
    for _ in range(3):
        q, s = bf.bfp8_group_quant(x)
        out = bf.bfp8_gemm(q, B, s, Bs, options={"prefetch_weights": 1})
    torch.cuda.synchronize()
    A, As = oracle_mod.group_quant(case["x"].view(torch.int16).numpy().view(np.uint16), False, True)
    ref = oracle_mod.blocked_gemm(A, case["B"].view(torch.uint8).numpy(), As, True,
                                  case["Bs"].numpy(), want_abs=True)
    check_gemm(out, ref, (K + 127) // 128, label=f"prefetch {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 16, 32, 33, 64])
@pytest.mark.parametrize("k_split", [0, 1, 2, 3])
def test_wide_tiles_with_partial_activation_rows(oracle_mod, dev, M, k_split):
    """Decode-sized M on 256-wide tiles loads only 32 or 64 activation rows per
    stage; the MMA still spans 128 rows and the promotion warps of the unused
    lane quadrants stay idle.  Every schedule, full comparison."""
    case = wl.linear_case(M, 4096, 4096, seed=900 + M)
    _run(oracle_mod, dev, case, options={"schedule": 2, "k_split": k_split},
         label=f"wide-rows M={M} k_split={k_split}")


@pytest.mark.parametrize("M,N,K", [(5, 1000, 1000), (40, 576, 7168), (64, 300, 129)])
def test_wide_partial_rows_ragged(oracle_mod, dev, M, N, K):
    case = wl.ragged_case(M, N, K, seed=M + N + K)
    for col_major in (True, False):
        _run(oracle_mod, dev, case, col_major, options={"schedule": 2},
             label=f"wide-rows ragged {M}x{N}x{K}")
