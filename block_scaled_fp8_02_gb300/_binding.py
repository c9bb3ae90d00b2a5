"""ctypes binding to libbfp8 (include/bfp8.h).

Argument marshalling only: every step of the computation runs in libbfp8's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There
is no fallback: if the library is missing or the device is not an sm_103
part, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libbfp8.so")

BFP8_OK = 0
BFP8_IN_BF16 = 0
BFP8_IN_F32 = 1
SCALE_FP32, SCALE_UE8M0 = 0, 1
SCHEDULE_AUTO, SCHEDULE_SWAP_AB, SCHEDULE_WIDE, SCHEDULE_GEMV = 0, 1, 2, 3
KSPLIT_AUTO, KSPLIT_STREAM_K, KSPLIT_CLUSTER, KSPLIT_NONE = 0, 1, 2, 3
PAIRS_AUTO, PAIRS_NEVER, PAIRS_ALWAYS = 0, 1, 2
STATUS_NAMES = {0: "BFP8_OK", 1: "BFP8_ERR_INVALID_ARG", 2: "BFP8_ERR_ALIGNMENT",
                3: "BFP8_ERR_UNSUPPORTED", 4: "BFP8_ERR_CUDA", 5: "BFP8_ERR_WORKSPACE",
                6: "BFP8_ERR_DEVICE_TIMEOUT"}

# Every symbol include/bfp8.h declares.
EXPORTS = ("bfp8_group_quant", "bfp8_group_quant_ex", "bfp8_scale_ceil_ue8m0", "bfp8_scale_ld", "bfp8_gemm", "bfp8_gemm_ex",
           "bfp8_gemm_workspace_size", "bfp8_gemm_plan", "bfp8_plan_unit", "bfp8_last_error",
           "bfp8_status_string", "bfp8_device_status", "bfp8_selftest_bounded_wait",
           "bfp8_version", "bfp8_gemm_noalloc", "bfp8_gemm_grouped",
           "bfp8_gemm_grouped_workspace_size", "bfp8_gemm_fused", "bfp8_gemm_fused_workspace_size",
           "bfp8_linear", "bfp8_linear_workspace_size")


class BFP8Error(RuntimeError):
    def __init__(self, status: int, where: str, reason: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {reason}")
        self.status = status


class GemmOptions(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int), ("max_ctas", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("prefetch_weights", ctypes.c_int), ("k_split", ctypes.c_int),
                ("cluster_size", ctypes.c_int), ("pairs", ctypes.c_int),
                ("reserved", ctypes.c_int * 1)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("swap_ab", ctypes.c_int), ("tile_n", ctypes.c_int), ("stages", ctypes.c_int),
                ("grid", ctypes.c_int), ("tiles", ctypes.c_int64), ("k_blocks", ctypes.c_int64),
                ("dp_tiles", ctypes.c_int64), ("sk_units", ctypes.c_int64),
                ("relayout", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("cluster", ctypes.c_int), ("gemv", ctypes.c_int), ("pair", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libbfp8 (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libbfp8 is not built ({LIB_PATH} missing): run "
                    "`python -m block_scaled_fp8_02_gb300.build` or __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.bfp8_group_quant.restype = i32
            L.bfp8_group_quant.argtypes = [P, i32, i64, i64, i64, i32, i32, P, i64, P, i64, P]
            L.bfp8_group_quant_ex.restype = i32
            L.bfp8_group_quant_ex.argtypes = [P, i32, i64, i64, i64, i32, i32, i32, P, i64, P, i64, P]
            L.bfp8_scale_ceil_ue8m0.restype = i32
            L.bfp8_scale_ceil_ue8m0.argtypes = [P, P, i64, P]
            L.bfp8_scale_ld.restype = i64
            L.bfp8_scale_ld.argtypes = [i64]
            L.bfp8_gemm.restype = i32
            L.bfp8_gemm.argtypes = [P, P, P, i32, i64, P, P, i64, i64, i64, P, sz, P]
            L.bfp8_gemm_ex.restype = i32
            L.bfp8_gemm_ex.argtypes = [P, P, P, i32, i64, P, P, i64, i64, i64, P, sz,
                                       ctypes.POINTER(GemmOptions), P]
            L.bfp8_gemm_workspace_size.restype = i32
            L.bfp8_gemm_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(GemmOptions), i32,
                                                   ctypes.POINTER(sz)]
            L.bfp8_gemm_plan.restype = i32
            L.bfp8_gemm_plan.argtypes = [i64, i64, i64, i32, ctypes.POINTER(GemmOptions), i32,
                                         ctypes.POINTER(PlanInfo)]
            L.bfp8_plan_unit.restype = i32
            L.bfp8_plan_unit.argtypes = [i64, i64, i64, i32, ctypes.POINTER(GemmOptions), i32, i64,
                                         ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]
            L.bfp8_last_error.restype = ctypes.c_char_p
            L.bfp8_last_error.argtypes = []
            L.bfp8_status_string.restype = ctypes.c_char_p
            L.bfp8_status_string.argtypes = [i32]
            L.bfp8_device_status.restype = i32
            L.bfp8_device_status.argtypes = [ctypes.POINTER(i32), i32]
            L.bfp8_selftest_bounded_wait.restype = i32
            L.bfp8_selftest_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64), P]
            L.bfp8_version.restype = i32
            L.bfp8_version.argtypes = []
            L.bfp8_gemm_noalloc.restype = i32
            L.bfp8_gemm_noalloc.argtypes = [P, P, P, i32, i64, P, P, i64, i64, i64, P]
            L.bfp8_gemm_grouped.restype = i32
            L.bfp8_gemm_grouped.argtypes = [P, P, P, i32, i64, P, P, i32, P, i64, i64, i64, P, sz,
                                            ctypes.POINTER(GemmOptions), P]
            L.bfp8_gemm_fused.restype = i32
            L.bfp8_gemm_fused.argtypes = [P, P, P, i32, i64, P, P, P, P, P, i32, i64, i64, i64, i64,
                                          P, sz, ctypes.POINTER(GemmOptions), P]
            L.bfp8_gemm_fused_workspace_size.restype = i32
            L.bfp8_gemm_fused_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(GemmOptions),
                                                         i32, ctypes.POINTER(sz)]
            L.bfp8_linear.restype = i32
            L.bfp8_linear.argtypes = [P, i64, P, P, P, i64, i64, i64, P, sz,
                                      ctypes.POINTER(GemmOptions), P]
            L.bfp8_linear_workspace_size.restype = i32
            L.bfp8_linear_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(GemmOptions), i32,
                                                     ctypes.POINTER(sz)]
            L.bfp8_gemm_grouped_workspace_size.restype = i32
            L.bfp8_gemm_grouped_workspace_size.argtypes = [i64, i64, i64, i32,
                                                           ctypes.POINTER(GemmOptions), i32,
                                                           ctypes.POINTER(sz)]
            _lib = L
    return _lib


def bfp8_last_error() -> str:
    return lib().bfp8_last_error().decode()


def _check(status: int, where: str):
    if status != BFP8_OK:
        raise BFP8Error(status, where, bfp8_last_error())


def _stream_ptr(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _opts(options) -> ctypes.POINTER(GemmOptions) | None:
    if options is None:
        return None
    if isinstance(options, GemmOptions):
        return ctypes.pointer(options)
    o = GemmOptions()
    o.schedule = int(options.get("schedule", 0))
    o.max_ctas = int(options.get("max_ctas", 0))
    o.tile_n = int(options.get("tile_n", 0))
    o.prefetch_weights = int(options.get("prefetch_weights", 0))
    o.k_split = int(options.get("k_split", 0))
    o.cluster_size = int(options.get("cluster_size", 0))
    o.pairs = int(options.get("pairs", 0))
    unknown = set(options) - {"schedule", "max_ctas", "tile_n", "prefetch_weights", "k_split",
                              "cluster_size", "pairs"}
    if unknown:
        raise ValueError(f"unknown GEMM options {sorted(unknown)}")
    return ctypes.pointer(o)


def bfp8_version() -> int:
    return int(lib().bfp8_version())


def bfp8_scale_ld(M: int) -> int:
    return int(lib().bfp8_scale_ld(M))


def bfp8_group_quant(x: torch.Tensor, col_major: bool = True, group: int = 128,
                     q: torch.Tensor | None = None, s_storage: torch.Tensor | None = None,
                     stream=None, ue8m0: bool = False):
    """Quantise x [M, K] (bf16 or fp32, CUDA, unit inner stride) per 128-group.

    Returns (q, s): q [M, K] float8_e4m3fn and s [M, G] fp32; for col_major the
    scales live in a [G, bfp8_scale_ld(M)] buffer and s is its transposed view
    (stride (1, ld)), the layout the pages hand to the GEMM.  ue8m0: every
    scale rounded up to a power of two (the UE8M0 variant).
    """
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit inner stride")
    if x.dtype == torch.bfloat16:
        in_dtype = BFP8_IN_BF16
    elif x.dtype == torch.float32:
        in_dtype = BFP8_IN_F32
    else:
        raise ValueError(f"x dtype {x.dtype}: expected bfloat16 or float32")
    M, K = x.shape
    G = (K + 127) // 128
    if q is None:
        q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=x.device)
    if col_major:
        ld_s = bfp8_scale_ld(M) if s_storage is None else s_storage.shape[1]
        if s_storage is None:
            s_storage = torch.empty((G, max(ld_s, 1)), dtype=torch.float32, device=x.device)
        s_view = s_storage[:, :M].t()
    else:
        ld_s = G if s_storage is None else s_storage.shape[1]
        if s_storage is None:
            s_storage = torch.empty((M, max(ld_s, 1)), dtype=torch.float32, device=x.device)
        s_view = s_storage[:, :G]
    st = lib().bfp8_group_quant_ex(x.data_ptr(), in_dtype, M, K, x.stride(0), group, int(col_major),
                                   SCALE_UE8M0 if ue8m0 else SCALE_FP32, q.data_ptr(),
                                   q.stride(0) if M > 0 else K, s_storage.data_ptr(), ld_s,
                                   _stream_ptr(stream))
    _check(st, "bfp8_group_quant")
    return q, s_view


def bfp8_scale_ceil_ue8m0(s: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Every element of the fp32 scale tensor s rounded up to a power of two
    (contiguous tensors; out may be s itself)."""
    if s.dtype != torch.float32 or not s.is_contiguous():
        raise ValueError("s must be a contiguous float32 tensor")
    if out is None:
        out = torch.empty_like(s)
    if out.shape != s.shape or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor shaped like s")
    _check(lib().bfp8_scale_ceil_ue8m0(s.data_ptr(), out.data_ptr(), s.numel(), _stream_ptr(stream)),
           "bfp8_scale_ceil_ue8m0")
    return out


def _as_layout(As: torch.Tensor, M: int, G: int):
    """(col_major, ld) of an As tensor of shape [M, G]."""
    if As.shape != (M, G):
        raise ValueError(f"As has shape {tuple(As.shape)}, expected ({M}, {G})")
    s0, s1 = As.stride()
    if s0 == 1 and (G == 1 or s1 >= M):
        return 1, (s1 if G > 1 else max(M, 1))
    if s1 == 1 and (M == 1 or s0 >= G):
        return 0, (s0 if M > 1 else G)
    raise ValueError(f"As strides {As.stride()} are neither row- nor column-major")


_ws_cache: dict[tuple[int, int], torch.Tensor] = {}


def workspace_for(nbytes: int, device: torch.device, stream=None) -> torch.Tensor:
    """A zero-initialised workspace of at least nbytes on `device` for calls
    on `stream` (None: the current stream), cached per (device, stream).

    libbfp8 leaves the workspace zeroed after every completed call, so one
    buffer serves every call issued in order on one stream; calls on streams
    without ordering between them get separate buffers.  A new buffer is
    allocated and zeroed on that stream, so its zeroing is ordered before the
    calls that use it, and a replaced buffer is only ever reused by later work
    on the same stream (the caching allocator's stream-ordered reuse)."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    sp = _stream_ptr(stream)
    ws = _ws_cache.get((idx, sp))
    if ws is None or ws.numel() < nbytes:
        s = stream if isinstance(stream, torch.cuda.Stream) else (
            torch.cuda.current_stream(device) if stream is None else
            torch.cuda.ExternalStream(sp, device=device))
        with torch.cuda.stream(s):
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[(idx, sp)] = ws
    return ws


def drop_workspaces() -> None:
    """Forget every cached workspace (after a kernel gave up on a wait, one may
    hold non-zero stream-K counters)."""
    _ws_cache.clear()


def bfp8_gemm_workspace_size(M: int, N: int, K: int, options=None,
                             operands_unaligned: bool = False) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().bfp8_gemm_workspace_size(M, N, K, _opts(options), int(operands_unaligned),
                                          ctypes.byref(n)), "bfp8_gemm_workspace_size")
    return int(n.value)


def bfp8_gemm_plan(M: int, N: int, K: int, num_sms: int, options=None,
                   operands_unaligned: bool = False) -> dict:
    info = PlanInfo()
    _check(lib().bfp8_gemm_plan(M, N, K, num_sms, _opts(options), int(operands_unaligned),
                                ctypes.byref(info)), "bfp8_gemm_plan")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


def bfp8_plan_unit(M: int, N: int, K: int, num_sms: int, cta: int, j: int = -1, options=None):
    n, t, kb = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().bfp8_plan_unit(M, N, K, num_sms, _opts(options), cta, j, ctypes.byref(n),
                                ctypes.byref(t), ctypes.byref(kb)), "bfp8_plan_unit")
    return int(n.value), int(t.value), int(kb.value)


def bfp8_gemm(A: torch.Tensor, B: torch.Tensor, As: torch.Tensor, Bs: torch.Tensor,
              out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              options=None, stream=None) -> torch.Tensor:
    """out [M, N] bf16 = blocked-FP8 GEMM of A [M, K], B [N, K] (float8_e4m3fn),
    As [M, G] (row- or column-major strides) and Bs [ceil(N/128), G]."""
    if A.dtype != torch.float8_e4m3fn or B.dtype != torch.float8_e4m3fn:
        raise ValueError("A and B must be float8_e4m3fn")
    if not (A.is_contiguous() and B.is_contiguous() and Bs.is_contiguous()):
        raise ValueError("A, B and Bs must be contiguous")
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("A and B disagree on K")
    G = (K + 127) // 128
    if Bs.shape != ((N + 127) // 128, G) or Bs.dtype != torch.float32:
        raise ValueError(f"Bs must be float32 of shape {((N + 127) // 128, G)}")
    col, ld = _as_layout(As, M, G)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    unaligned = (A.data_ptr() % 16 != 0) or (B.data_ptr() % 16 != 0)
    if workspace is None:
        need = bfp8_gemm_workspace_size(M, N, K, options, unaligned)
        workspace = workspace_for(need, A.device, stream)
    st = lib().bfp8_gemm_ex(A.data_ptr(), B.data_ptr(), As.data_ptr(), col, ld, Bs.data_ptr(),
                            out.data_ptr(), M, N, K, workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _opts(options),
                            _stream_ptr(stream))
    _check(st, "bfp8_gemm")
    return out


def bfp8_gemm_grouped_workspace_size(M: int, N: int, K: int, num_experts: int, options=None,
                                     operands_unaligned: bool = False) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().bfp8_gemm_grouped_workspace_size(M, N, K, num_experts, _opts(options),
                                                  int(operands_unaligned), ctypes.byref(n)),
           "bfp8_gemm_grouped_workspace_size")
    return int(n.value)


def bfp8_gemm_grouped(A: torch.Tensor, B: torch.Tensor, As: torch.Tensor, Bs: torch.Tensor,
                      grouped_layout: torch.Tensor, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, options=None,
                      stream=None) -> torch.Tensor:
    """M-grouped (mixture-of-experts) blocked-FP8 GEMM: A [M, K] rows grouped by
    expert in 128-aligned blocks, B [E, N, K], Bs [E, ceil(N/128), G],
    grouped_layout int32 [E] = cumulative aligned row counts (device).  Rows
    past the last expert's block are left untouched in `out`."""
    if A.dtype != torch.float8_e4m3fn or B.dtype != torch.float8_e4m3fn:
        raise ValueError("A and B must be float8_e4m3fn")
    if B.dim() != 3:
        raise ValueError("B must be [experts, N, K]")
    if not (A.is_contiguous() and B.is_contiguous() and Bs.is_contiguous()
            and grouped_layout.is_contiguous()):
        raise ValueError("A, B, Bs and grouped_layout must be contiguous")
    M, K = A.shape
    E, N, K2 = B.shape
    if K2 != K:
        raise ValueError("A and B disagree on K")
    G = (K + 127) // 128
    if Bs.shape != (E, (N + 127) // 128, G) or Bs.dtype != torch.float32:
        raise ValueError(f"Bs must be float32 of shape {(E, (N + 127) // 128, G)}")
    if grouped_layout.dtype != torch.int32 or grouped_layout.shape != (E,):
        raise ValueError(f"grouped_layout must be int32 of shape ({E},)")
    col, ld = _as_layout(As, M, G)
    if out is None:
        out = torch.zeros((M, N), dtype=torch.bfloat16, device=A.device)
    unaligned = (A.data_ptr() % 16 != 0) or (B.data_ptr() % 16 != 0)
    if workspace is None:
        need = bfp8_gemm_grouped_workspace_size(M, N, K, E, options, unaligned)
        workspace = workspace_for(need, A.device, stream)
    st = lib().bfp8_gemm_grouped(A.data_ptr(), B.data_ptr(), As.data_ptr(), col, ld,
                                 Bs.data_ptr(), grouped_layout.data_ptr(), E, out.data_ptr(),
                                 M, N, K, workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _opts(options),
                                 _stream_ptr(stream))
    _check(st, "bfp8_gemm_grouped")
    return out


def bfp8_gemm_fused(A: torch.Tensor, B: torch.Tensor, As: torch.Tensor, Bs: torch.Tensor,
                    bias: torch.Tensor | None = None, want_out: bool = True,
                    quantise: bool = True, s_col_major: bool = True,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    options=None, stream=None):
    """Blocked-FP8 GEMM with the fused epilogue: y = bf16(bf16(A B^T scaled) +
    bias), returned as (out or None, q or None, s or None); q, s = the 1x128
    group quantisation of y (s a [M, G] view, column-major storage by default)."""
    if A.dtype != torch.float8_e4m3fn or B.dtype != torch.float8_e4m3fn:
        raise ValueError("A and B must be float8_e4m3fn")
    if not (A.is_contiguous() and B.is_contiguous() and Bs.is_contiguous()):
        raise ValueError("A, B and Bs must be contiguous")
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("A and B disagree on K")
    G = (K + 127) // 128
    if Bs.shape != ((N + 127) // 128, G) or Bs.dtype != torch.float32:
        raise ValueError(f"Bs must be float32 of shape {((N + 127) // 128, G)}")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.shape != (N,)
                             or not bias.is_contiguous()):
        raise ValueError(f"bias must be a contiguous bfloat16 tensor of shape ({N},)")
    col, ld = _as_layout(As, M, G)
    if want_out and out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if not want_out:
        out = None
    q = s_view = s_st = None
    Gn = (N + 127) // 128
    ld_s = 0
    if quantise:
        q = torch.empty((M, N), dtype=torch.float8_e4m3fn, device=A.device)
        if s_col_major:
            ld_s = bfp8_scale_ld(M)
            s_st = torch.zeros((Gn, ld_s), dtype=torch.float32, device=A.device)
            s_view = s_st[:, :M].t()
        else:
            ld_s = Gn
            s_st = torch.zeros((M, Gn), dtype=torch.float32, device=A.device)
            s_view = s_st
    unaligned = (A.data_ptr() % 16 != 0) or (B.data_ptr() % 16 != 0)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check(lib().bfp8_gemm_fused_workspace_size(M, N, K, _opts(options), int(unaligned),
                                                    ctypes.byref(n)),
               "bfp8_gemm_fused_workspace_size")
        workspace = workspace_for(int(n.value), A.device, stream)
    st = lib().bfp8_gemm_fused(
        A.data_ptr(), B.data_ptr(), As.data_ptr(), col, ld, Bs.data_ptr(),
        bias.data_ptr() if bias is not None else None, out.data_ptr() if out is not None else None,
        q.data_ptr() if q is not None else None, s_st.data_ptr() if s_st is not None else None,
        int(s_col_major), ld_s, M, N, K, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _opts(options), _stream_ptr(stream))
    _check(st, "bfp8_gemm_fused")
    return out, q, s_view


def bfp8_device_status(clear: bool = True) -> int:
    """The device failure word (0: no kernel gave up on a wait).  A nonzero
    word also drops the cached workspaces, which may hold stale counters."""
    code = ctypes.c_int(0)
    _check(lib().bfp8_device_status(ctypes.byref(code), int(clear)), "bfp8_device_status")
    if code.value != 0:
        drop_workspaces()
    return int(code.value)


def bfp8_selftest_bounded_wait(limit_cycles: int, stream=None):
    """Returns (status, elapsed_cycles); status BFP8_ERR_DEVICE_TIMEOUT (6) is
    the expected outcome: the wait gave up instead of hanging."""
    el = ctypes.c_uint64(0)
    st = lib().bfp8_selftest_bounded_wait(limit_cycles, ctypes.byref(el), _stream_ptr(stream))
    return int(st), int(el.value)


def bfp8_linear_workspace_size(M: int, N: int, K: int, options=None,
                               weights_unaligned: bool = False) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().bfp8_linear_workspace_size(M, N, K, _opts(options), int(weights_unaligned),
                                            ctypes.byref(n)), "bfp8_linear_workspace_size")
    return int(n.value)


def bfp8_linear(x: torch.Tensor, B: torch.Tensor, Bs: torch.Tensor, out: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, options=None, stream=None) -> torch.Tensor:
    """out [M, N] bf16 = the blocked linear layer of bf16 x [M, K] (rows may be
    strided) against e4m3 weights B [N, K] with scales Bs: the 1 x 128 group
    quantisation into the workspace, then the GEMM, in one library call."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 tensor with unit column stride")
    if B.dtype != torch.float8_e4m3fn or not B.is_contiguous() or not Bs.is_contiguous():
        raise ValueError("B must be contiguous float8_e4m3fn and Bs contiguous")
    M, K = x.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("x and B disagree on K")
    G = (K + 127) // 128
    if Bs.shape != ((N + 127) // 128, G) or Bs.dtype != torch.float32:
        raise ValueError(f"Bs must be float32 of shape {((N + 127) // 128, G)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        need = bfp8_linear_workspace_size(M, N, K, options, B.data_ptr() % 16 != 0)
        workspace = workspace_for(need, x.device, stream)
    st = lib().bfp8_linear(x.data_ptr(), x.stride(0), B.data_ptr(), Bs.data_ptr(), out.data_ptr(),
                           M, N, K, workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), _opts(options),
                           _stream_ptr(stream))
    _check(st, "bfp8_linear")
    return out


def linear(x: torch.Tensor, B: torch.Tensor, Bs: torch.Tensor, out: torch.Tensor | None = None,
           stream=None, ue8m0: bool = False) -> torch.Tensor:
    """The whole W8A8 blocked linear layer: quantise x per 128-group (column-major
    scales) and run the blocked GEMM against e4m3 weights B with scales Bs
    (bfp8_linear).  ue8m0: the UE8M0 variant (activation scales rounded up to
    powers of two; pass weight scales rounded the same way, e.g. by
    bfp8_scale_ceil_ue8m0) and fp32 activations run as two calls."""
    if not ue8m0 and x.dtype == torch.bfloat16:
        return bfp8_linear(x, B, Bs, out=out, stream=stream)
    q, s = bfp8_group_quant(x, col_major=True, stream=stream, ue8m0=ue8m0)
    # the quantisation kernel writes neither B nor Bs: the GEMM may start
    # streaming the weights while it runs
    return bfp8_gemm(q, B, s, Bs, out=out, options={"prefetch_weights": 1}, stream=stream)
