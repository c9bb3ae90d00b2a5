"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, rejects bad arguments on the host before touching a device, and
plans schedules whose work split covers every (tile, k-block) unit once."""
import ctypes
import os
import re

import numpy as np
import pytest

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import build as bfbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bfp8.h")


@pytest.fixture(scope="module")
def L():
    bfbuild.build()
    return bf.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bfp8_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_what_the_binding_expects():
    assert _declared() == sorted(bf.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings_and_helpers(L):
    assert bf.bfp8_version() == 1
    assert L.bfp8_status_string(0) == b"BFP8_OK"
    assert L.bfp8_status_string(6) == b"BFP8_ERR_DEVICE_TIMEOUT"
    assert [bf.bfp8_scale_ld(m) for m in (0, 1, 4, 5, 83, 84)] == [0, 4, 4, 8, 84, 84]


def _quant(L, **kw):
    a = dict(x=16, in_dtype=0, M=4, K=256, ld_x=256, group=128, col_major=1, q=16, ld_q=256,
             s=16, ld_s=4, stream=None)
    a.update(kw)
    return L.bfp8_group_quant(a["x"], a["in_dtype"], a["M"], a["K"], a["ld_x"], a["group"],
                              a["col_major"], a["q"], a["ld_q"], a["s"], a["ld_s"], a["stream"])


def test_group_quant_rejects_bad_arguments_on_the_host(L):
    assert _quant(L, group=64) == 1
    assert _quant(L, in_dtype=7) == 1
    assert _quant(L, col_major=2) == 1
    assert _quant(L, M=-1) == 1
    assert _quant(L, x=None) == 1
    assert _quant(L, ld_x=100) == 1
    assert _quant(L, ld_q=10) == 1
    assert _quant(L, ld_s=3) == 1                     # column-major needs ld_s >= M
    assert _quant(L, col_major=0, ld_s=1) == 1        # row-major needs ld_s >= G = 2
    assert _quant(L, x=17) == 2                       # bf16 input must be 2-byte aligned
    assert _quant(L, s=18) == 2
    assert "ld_s" in bf.bfp8_last_error() or "aligned" in bf.bfp8_last_error()
    assert _quant(L, M=0) == 0 and _quant(L, K=0, x=None) == 0   # empty: nothing to do


def test_ue8m0_entry_points_reject_bad_arguments_on_the_host(L):
    def q(fmt, **kw):
        a = dict(x=256, in_dtype=0, M=4, K=200, ld_x=200, group=128, col=1, q=256, ld_q=200, s=256,
                 ld_s=4)
        a.update(kw)
        return L.bfp8_group_quant_ex(a["x"], a["in_dtype"], a["M"], a["K"], a["ld_x"], a["group"],
                                     a["col"], fmt, a["q"], a["ld_q"], a["s"], a["ld_s"], None)
    assert q(2) == 1 and "scale_fmt" in bf.bfp8_last_error()
    assert q(-1) == 1
    assert q(1, group=64) == 1
    assert q(1, M=0) == 0 and q(0, M=0) == 0
    assert L.bfp8_scale_ceil_ue8m0(256, 256, -1, None) == 1
    assert L.bfp8_scale_ceil_ue8m0(None, 256, 4, None) == 1
    assert L.bfp8_scale_ceil_ue8m0(258, 256, 4, None) == 2
    assert L.bfp8_scale_ceil_ue8m0(None, None, 0, None) == 0      # empty: nothing to do


def _gemm(L, **kw):
    a = dict(A=256, B=256, As=256, col=1, ld_as=4, Bs=256, out=256, M=4, N=128, K=256, ws=256,
             wsb=1 << 30, opt=None, stream=None)
    a.update(kw)
    return L.bfp8_gemm_ex(a["A"], a["B"], a["As"], a["col"], a["ld_as"], a["Bs"], a["out"], a["M"],
                          a["N"], a["K"], a["ws"], a["wsb"], a["opt"], a["stream"])


def test_gemm_rejects_bad_arguments_on_the_host(L):
    assert _gemm(L, M=0) == 1
    assert _gemm(L, K=-5) == 1
    assert _gemm(L, N=1 << 31) == 1
    assert _gemm(L, A=None) == 1
    assert _gemm(L, out=None) == 1
    assert _gemm(L, col=3) == 1
    assert _gemm(L, ld_as=3) == 1                     # column-major ld_as >= M
    assert _gemm(L, col=0, ld_as=1) == 1              # row-major ld_as >= G = 2
    assert _gemm(L, As=258) == 2
    assert _gemm(L, out=257) == 2
    bad = bf.GemmOptions()
    bad.schedule = 9
    assert _gemm(L, opt=ctypes.pointer(bad)) == 1
    bad.schedule = 4
    assert _gemm(L, opt=ctypes.pointer(bad)) == 1
    bad.schedule, bad.tile_n = 0, 48
    assert _gemm(L, opt=ctypes.pointer(bad)) == 1
    bad.schedule, bad.tile_n = 2, 64                # wide tiles are 128 or 256 wide
    assert _gemm(L, opt=ctypes.pointer(bad)) == 1
    bad.schedule = 0
    bad.tile_n, bad.k_split = 0, 4
    assert _gemm(L, opt=ctypes.pointer(bad)) == 1
    for cs in (1, 9, -2):
        bad.k_split, bad.cluster_size = 2, cs
        assert _gemm(L, opt=ctypes.pointer(bad)) == 1
    bad.cluster_size = 0
    # a valid call reaches the device check, which fails cleanly without a GPU
    import torch
    if not torch.cuda.is_available():
        assert _gemm(L) == 3
        assert "device" in bf.bfp8_last_error().lower() or "driver" in bf.bfp8_last_error().lower()


def test_grouped_gemm_rejects_bad_arguments_on_the_host(L):
    def call(E=4, layout=512, M=256, N=128, K=256):
        return L.bfp8_gemm_grouped(256, 256, 256, 1, 256, 256, layout, E, 256, M, N, K, 256,
                                   1 << 30, None, None)
    assert call(E=0) == 1
    assert call(E=1025) == 1
    assert call(layout=0) == 1                    # null grouped_layout
    assert call(layout=514) == 2                  # not 4-byte aligned
    assert call(M=0) == 1
    import torch
    if not torch.cuda.is_available():
        assert call() == 3                        # valid: fails at the device check


def _cover(M, N, K, sms, options=None):
    plan = bf.bfp8_gemm_plan(M, N, K, sms, options)
    seen = {}
    for cta in range(plan["grid"]):
        n, _, _ = bf.bfp8_plan_unit(M, N, K, sms, cta, -1, options)
        prev = None
        for j in range(n):
            _, t, kb = bf.bfp8_plan_unit(M, N, K, sms, cta, j, options)
            assert 0 <= t < plan["tiles"] and 0 <= kb < plan["k_blocks"]
            assert (t, kb) not in seen, (t, kb, cta, seen.get((t, kb)))
            seen[(t, kb)] = cta
            if prev is not None and prev[0] == t:
                assert kb == prev[1] + 1          # a CTA's units within a tile are contiguous
            prev = (t, kb)
    assert len(seen) == plan["tiles"] * plan["k_blocks"]
    return plan


@pytest.mark.parametrize("M,N,K,sms,opts", [
    (1, 4096, 4096, 152, None), (83, 576, 7168, 152, None), (83, 576, 7168, 7, None),
    (2048, 4096, 4096, 152, None), (1000, 1000, 1000, 152, None), (3, 576, 1000, 152, None),
    (300, 1000, 7168, 152, {"schedule": 1}), (16, 512, 256, 152, {"schedule": 2}),
    (1, 1, 1, 152, None), (4096, 4096, 512, 19, {"tile_n": 128}),
    (1, 4096, 4096, 152, {"k_split": 1}), (3, 576, 7168, 152, {"k_split": 2}),
    (1, 4096, 300, 152, {"k_split": 2}), (5, 256, 1024, 152, {"k_split": 2, "cluster_size": 5}),
    (600, 512, 4096, 152, {"schedule": 2}), (7, 1000, 1000, 152, {"k_split": 2, "cluster_size": 7}),
    (8192, 4096, 4096, 152, None), (1000, 1000, 1000, 152, {"k_split": 3}),
    (3000, 4096, 512, 152, {"k_split": 3}), (1, 4096, 4096, 152, {"k_split": 3}),
])
def test_work_split_covers_every_unit_once(L, M, N, K, sms, opts):
    _cover(M, N, K, sms, opts)


def test_auto_plans_cover_every_unit_on_random_shapes(L):
    """The planner's automatic choice (stream-K, whole tiles or clusters,
    swap-AB or wide tiles) hands every (tile, k-block) unit to exactly one
    CTA, in contiguous runs, on seeded random shapes and SM counts."""
    rng = np.random.default_rng(2024)
    done = 0
    while done < 40:
        M = int(rng.integers(1, 6000))
        N = int(rng.integers(1, 9000))
        K = int(rng.integers(1, 9000))
        sms = int(rng.choice([152, 148, 132, 19, 7]))
        plan = bf.bfp8_gemm_plan(M, N, K, sms)
        if plan["tiles"] * plan["k_blocks"] > 20000:
            continue
        assert 1 <= plan["grid"] <= max(sms, plan["tiles"] * max(plan["cluster"], 1))
        _cover(M, N, K, sms, None)
        done += 1


def _cluster_units(M, N, K, sms, options):
    """Per tile, the k-blocks each cluster rank takes, from the plan's walk."""
    plan = bf.bfp8_gemm_plan(M, N, K, sms, options)
    cs = plan["cluster"]
    per_tile = {}
    for cta in range(plan["grid"]):
        n, _, _ = bf.bfp8_plan_unit(M, N, K, sms, cta, -1, options)
        kbs = []
        for j in range(n):
            _, t, kb = bf.bfp8_plan_unit(M, N, K, sms, cta, j, options)
            assert t == cta // cs                    # a cluster's CTAs share one tile
            kbs.append(kb)
        per_tile.setdefault(cta // cs, []).append(kbs)
    return plan, per_tile


@pytest.mark.parametrize("M,N,K,opts,cs", [
    (1, 4096, 4096, None, 4), (200, 4096, 4096, None, 4), (3, 576, 7168, {"k_split": 2}, 8),
    (1, 4096, 300, {"k_split": 2}, 3), (600, 512, 4096, {"schedule": 2}, 8),
    (5, 256, 1024, {"k_split": 2, "cluster_size": 5}, 5),
])
def test_cluster_split_gives_each_rank_one_nonempty_contiguous_slice(L, M, N, K, opts, cs):
    plan, per_tile = _cluster_units(M, N, K, 152, opts)
    assert plan["cluster"] == cs and plan["grid"] == plan["tiles"] * cs
    assert plan["dp_tiles"] == 0 and plan["sk_units"] == 0
    G = plan["k_blocks"]
    for t, slices in per_tile.items():
        assert len(slices) == cs
        assert [kb for sl in slices for kb in sl] == list(range(G))     # rank order = K order
        sizes = [len(sl) for sl in slices]
        assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def test_plans_choose_the_documented_schedules(L):
    SW = {"schedule": bf.SCHEDULE_SWAP_AB}
    p = bf.bfp8_gemm_plan(1, 4096, 4096, 152, SW)
    assert p["swap_ab"] == 1 and p["tile_n"] == 16 and p["cluster"] == 4 and p["grid"] == 128
    p = bf.bfp8_gemm_plan(1, 4096, 4096, 152, dict(SW, k_split=1))
    assert p["cluster"] == 1 and p["grid"] == 152 and p["dp_tiles"] == 0
    # AUTO, M <= 256: 256- or 128-wide tiles by the split model (a 128-wide
    # step weighs 0.7 of a 256-wide one).  N = K = 4096: 128-wide tiles in
    # clusters of 4 up to M = 128 (measured 8.96 against 10.13 us at M = 32,
    # 10.61 against 14.33 at M = 128), 256-wide from M = 160 (13.58 against 14.09)
    for M in (9, 32, 128):
        p = bf.bfp8_gemm_plan(M, 4096, 4096, 152)
        assert (p["swap_ab"], p["tile_n"], p["cluster"]) == (0, 128, 4)
    for M in (160, 256):
        p = bf.bfp8_gemm_plan(M, 4096, 4096, 152)
        assert (p["swap_ab"], p["tile_n"], p["cluster"]) == (0, 256, 4)
    # Qwen3-32B shapes: 256-wide (qkv at M = 256: 23.6 us against 36.3 with
    # swap-AB tiles; down at M = 64: 30.0 against 41.5)
    assert bf.bfp8_gemm_plan(256, 10240, 5120, 152)["tile_n"] == 256
    p = bf.bfp8_gemm_plan(64, 5120, 25600, 152)
    assert p["swap_ab"] == 0 and p["tile_n"] == 256 and p["cluster"] == 6
    # five narrow tiles (N = 576): 128-wide in clusters of 8 (7.99 us at M =
    # 83, against 9.50 swap-AB and 11.72 256-wide)
    p = bf.bfp8_gemm_plan(83, 576, 7168, 152)
    assert (p["swap_ab"], p["tile_n"], p["cluster"]) == (0, 128, 8)
    # swap-AB tiles, explicitly: five tiles of 56 k-blocks would be spread over
    # ~30 CTAs each by stream-K (a long fixup chain); clusters of 8 win
    assert bf.bfp8_gemm_plan(83, 576, 7168, 152, SW)["cluster"] == 8
    # 40 tiles of 200 k-blocks: stream-K's 53 steps per CTA beat 67 in clusters of 3
    assert bf.bfp8_gemm_plan(1, 5120, 25600, 152, SW)["cluster"] == 1
    # ... but not with 256-wide swap tiles, whose 128 KB partials are costly
    # to write and read (measured: clusters of 3 60.9 us, stream-K 65.8 us)
    assert bf.bfp8_gemm_plan(256, 5120, 25600, 152, SW)["cluster"] == 3
    # 80 tiles of 40 k-blocks: stream-K over 152 CTAs beats one wave of 80
    # whole tiles (measured 37.4 against 39.3 us)
    p = bf.bfp8_gemm_plan(256, 10240, 5120, 152, SW)
    assert p["cluster"] == 1 and p["sk_units"] > 0
    # wide tiles: 64 of them at M = 512, clusters of 2
    p = bf.bfp8_gemm_plan(512, 4096, 4096, 152)
    assert p["swap_ab"] == 0 and p["cluster"] == 2 and p["grid"] == 128
    # 80 tiles: not even clusters of 2 fit in one wave
    assert bf.bfp8_gemm_plan(1, 10240, 5120, 152, SW)["cluster"] == 1
    # cluster schedules need no stream-K partials in the workspace
    assert (bf.bfp8_gemm_plan(1, 4096, 4096, 152, SW)["workspace_bytes"]
            < bf.bfp8_gemm_plan(1, 4096, 4096, 152, dict(SW, k_split=1))["workspace_bytes"])
    p = bf.bfp8_gemm_plan(64, 4096, 4096, 152, SW)
    assert p["swap_ab"] == 1 and p["tile_n"] == 64
    # an explicit narrow tile width exists only as a swap-AB tile
    assert bf.bfp8_gemm_plan(64, 4096, 4096, 152, {"tile_n": 32})["swap_ab"] == 1
    p = bf.bfp8_gemm_plan(8192, 4096, 4096, 152)
    assert p["swap_ab"] == 0 and p["tile_n"] == 256 and p["tiles"] == 64 * 16
    # 1024 tiles = 6.7 waves: seven balanced waves of whole tiles on 147 CTAs
    # beat splitting the last 112 tiles' 256-wide partials stream-K
    assert p["dp_tiles"] == 1024 and p["sk_units"] == 0 and p["grid"] == 147
    p = bf.bfp8_gemm_plan(1024, 4096, 4096, 152)         # 128 tiles: one wave, 24 SMs idle
    assert p["grid"] == 128 and p["dp_tiles"] == 128 and p["sk_units"] == 0
    # 192 tiles: two balanced waves of whole tiles beat splitting 40 tiles'
    # 256-wide partials over 152 CTAs
    p = bf.bfp8_gemm_plan(1536, 4096, 4096, 152)
    assert p["grid"] == 96 and p["dp_tiles"] == 192 and p["sk_units"] == 0
    p = bf.bfp8_gemm_plan(1536, 4096, 4096, 152, {"k_split": 1})
    assert p["dp_tiles"] == 152 and p["sk_units"] == 40 * 32
    p = bf.bfp8_gemm_plan(4096, 4096, 4096, 152)         # 512 tiles: four waves of 128
    assert p["grid"] == 128 and p["sk_units"] == 0
    # 320 tiles of 64 k-blocks: a third wave of 16 tiles costs more than
    # sharing their k-blocks stream-K
    p = bf.bfp8_gemm_plan(2048, 5120, 8192, 152)
    assert p["dp_tiles"] == 304 and p["sk_units"] == 16 * 64
    p = bf.bfp8_gemm_plan(3, 1000, 1000, 152)
    assert p["relayout"] == 1                       # 1000-byte rows break the TMA stride rule
    assert bf.bfp8_gemm_plan(3, 1000, 1024, 152)["relayout"] == 0
    assert bf.bfp8_gemm_plan(3, 1000, 1024, 152, operands_unaligned=True)["relayout"] == 1


def test_linear_rejects_bad_arguments_on_the_host(L):
    P = 256  # any 256-aligned fake device address: nothing is dereferenced on the host
    def lin(x=P, ld_x=256, B=P, Bs=P, out=P, M=4, N=8, K=256, ws=P, wsb=1 << 20, opt=None):
        return L.bfp8_linear(x, ld_x, B, Bs, out, M, N, K, ws, wsb, opt, None)
    assert lin(M=0) == 1
    assert lin(K=-1) == 1
    assert lin(x=None) == 1
    assert lin(out=None) == 1
    assert lin(ld_x=255) == 1                       # ld_x >= K
    assert lin(x=P + 1) == 2                        # bf16 rows: 2-byte aligned
    assert lin(Bs=P + 2) == 2
    bad = bf.GemmOptions()
    bad.k_split = 7
    assert lin(opt=ctypes.pointer(bad)) == 1
    n = ctypes.c_size_t(0)
    assert L.bfp8_linear_workspace_size(4, 8, 0, None, 0, ctypes.byref(n)) == 1
    assert L.bfp8_linear_workspace_size(4, 8, 256, None, 0, None) == 1


def test_gemv_plans(L):
    """BFP8_SCHEDULE_GEMV: M <= 32, K % 128 == 0, aligned operands; else refused."""
    G = {"schedule": bf.SCHEDULE_GEMV}
    for M in (1, 2, 3, 4, 8, 9, 16, 24, 32):
        assert bf.bfp8_gemm_plan(M, 4096, 4096, 152, G)["gemv"] == 1
    for M, N, K, kw in ((33, 4096, 4096, {}), (1, 4096, 1000, {}), (1, 4096, 4112, {}),
                        (2, 64, 4096, {"operands_unaligned": True})):
        with pytest.raises(bf.BFP8Error):
            bf.bfp8_gemm_plan(M, N, K, 152, G, **kw)
    assert bf.bfp8_gemm_plan(64, 4096, 4096, 152)["gemv"] == 0
    # AUTO, M <= 16: one wave of 2 x SMs, or past it SMs balanced to 3/4 or
    # weight streams up to 64 MB
    for M, N, K in ((1, 4096, 4096), (8, 10240, 5120), (1, 5120, 8192), (1, 51200, 5120),
                    (1, 576, 7168), (9, 4096, 4096), (16, 4864, 4096), (16, 10240, 5120),
                    (16, 51200, 5120), (12, 6144, 4096), (16, 5120, 8192), (16, 4880, 4096)):
        assert bf.bfp8_gemm_plan(M, N, K, 152)["gemv"] == 1, (M, N, K)
    for M, N, K in ((17, 4096, 4096), (24, 4864, 4096)):          # M 17..24: one wave only
        assert bf.bfp8_gemm_plan(M, N, K, 152)["gemv"] == 1, (M, N, K)
    for M, N, K in ((1, 5120, 25600), (16, 5120, 25600), (17, 4880, 4096), (24, 10240, 5120),
                    (25, 4096, 4096), (1, 4096, 4112)):
        assert bf.bfp8_gemm_plan(M, N, K, 152)["gemv"] == 0, (M, N, K)
    assert bf.bfp8_gemm_plan(1, 4096, 4096, 152, {"schedule": bf.SCHEDULE_SWAP_AB})["gemv"] == 0


def test_pair_plans(L):
    """Paired 256 x 256 tiles: plain calls on 256-wide tiles with more than 64
    rows, whole tiles over the pairs; refused otherwise when forced."""
    P = {"pairs": bf.PAIRS_ALWAYS}
    p = bf.bfp8_gemm_plan(2048, 4096, 4096, 152, P)
    assert p["pair"] == 1 and p["tiles"] == 8 * 16 and p["grid"] % 2 == 0 and p["sk_units"] == 0
    p = bf.bfp8_gemm_plan(8192, 4096, 4096, 152, P)
    assert p["pair"] == 1 and p["tiles"] == 32 * 16 and p["dp_tiles"] == p["tiles"]
    assert bf.bfp8_gemm_plan(2048, 4096, 4096, 152, {"pairs": bf.PAIRS_NEVER})["pair"] == 0
    assert bf.bfp8_gemm_plan(2048, 4096, 4096, 152, dict(P, max_ctas=10))["grid"] == 10
    for M, o in ((64, {}), (2048, {"k_split": 1}), (2048, {"tile_n": 128}), (2048, {"schedule": 1})):
        with pytest.raises(bf.BFP8Error):
            bf.bfp8_gemm_plan(M, 4096, 4096, 152, dict(P, **o))
    bad = bf.GemmOptions()
    bad.pairs = 3
    assert _gemm(L, opt=ctypes.pointer(bad)) == 1

