"""CPU oracle for the blocked W8A8 FP8 linear layer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library (``libbfp8``) and
its Python binding never touch it, and it shares no code with them: the C
source next to this file (oracle.c) restates every definition from the pages
on DeepSeek-style blocked FP8 linear layers and from the OCP E4M3 format.

Functions and the passages they follow:
  e4m3_table / e4m3_encode   OCP E4M3 "fn" format; fp8 limits +-448 from
                             torch.finfo(float8_e4m3fn) in the vLLM PR 49932
                             digest, section "key source snippet".
  group_quant                per_token_group_quant_fp8 (group 128, row- or
                             column-major scales), same snippet.
  blocked_gemm               native_w8a8_block_matmul with block_size [128, 128],
                             bf16 output, same snippet.
  bf16_from_f64              round-to-nearest-even to bfloat16 (the snippet's
                             out_dtype = torch.bfloat16).
  ceil_pow2 / group_quant(ue8m0=True)
                             the UE8M0 scale variant of the transformers DeepGEMM
                             integration (`_ceil_to_ue8m0`; `_select_fp8_cast_kwargs`
                             with use_ue8m0): each scale amax/448 rounded up to a
                             power of two before the codes are computed; weight
                             scales rounded the same way.
  bias_add_bf16              the bias addition of the transformers DeepGEMM
                             integration's `deepgemm_fp8_fp4_linear`
                             (`output.add_(bias)` on bf16 tensors): one IEEE fp32
                             addition, rounded to bf16.
  fused_linear               blocked_gemm, bias_add_bf16, then group_quant of the
                             bf16 result (the next layer's activations).
  grouped_gemm               the M-grouped contiguous layout of the transformers
                             DeepGEMM integration (`_build_deepgemm_contiguous_
                             layout`, SM100 "psum" form): blocked_gemm applied to
                             each expert's block of rows with that expert's
                             weights and weight scales.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# The same command __graft_entry__.build() runs; no fast-math and no FMA
# contraction, so every operation is one IEEE operation on x86-64 and aarch64.
GCC_CMD = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-o", _LIB, _SRC, "-lpthread", "-lm"]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so if missing or stale."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h")))
    if force or stale:
        subprocess.run(GCC_CMD, check=True)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_table.argtypes = [P]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode_array.argtypes = [P, P, i64]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_double_array.argtypes = [P, P, i64]
            lib.oracle_group_quant.restype = ctypes.c_int
            lib.oracle_group_quant.argtypes = [P, ctypes.c_int, i64, i64, i64, ctypes.c_int, i64,
                                               P, i64, P]
            lib.oracle_group_quant_ue8m0.restype = ctypes.c_int
            lib.oracle_group_quant_ue8m0.argtypes = lib.oracle_group_quant.argtypes
            lib.oracle_ceil_pow2.restype = ctypes.c_float
            lib.oracle_ceil_pow2.argtypes = [ctypes.c_float]
            lib.oracle_blocked_gemm.restype = ctypes.c_int
            lib.oracle_blocked_gemm.argtypes = [P, P, P, ctypes.c_int, i64, P, i64, i64, i64,
                                                P, i64, P, P, P, ctypes.c_int]
            lib.oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def e4m3_table() -> np.ndarray:
    """float64[256]: the value of every float8_e4m3fn code (NaN at 0x7F, 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even, saturating fp32 -> e4m3fn codes (uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_from_f64(v) -> np.ndarray:
    """Round float64 values to bfloat16 (ties to even); returns uint16 bits."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_from_double_array(_ptr(v), _ptr(out), v.size)
    return out


def scale_ld(M: int) -> int:
    """Leading dimension of a column-major scale array: M rounded up to 4."""
    return (M + 3) // 4 * 4


def ceil_pow2(s) -> np.ndarray:
    """Each positive finite fp32 scale rounded up to the nearest power of two."""
    s = np.asarray(s, dtype=np.float32)
    f = _load().oracle_ceil_pow2
    return np.array([f(float(v)) for v in s.reshape(-1)], dtype=np.float32).reshape(s.shape)


def group_quant(x: np.ndarray, is_f32: bool, col_major: bool, ld_s: int | None = None,
                ue8m0: bool = False):
    """Quantise x [M, K] (float32 values, or bfloat16 bits as uint16).

    Returns (q uint8 [M, K], s float32) where s is [G, ld_s] for column-major
    scales and [M, ld_s] for row-major ones (G = ceil(K/128)).  ue8m0: every
    scale rounded up to a power of two before the codes are computed.
    """
    x = np.ascontiguousarray(x, dtype=np.float32 if is_f32 else np.uint16)
    M, K = x.shape
    G = (K + 127) // 128
    if ld_s is None:
        ld_s = scale_ld(M) if col_major else G
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((G, ld_s) if col_major else (M, ld_s), dtype=np.float32)
    fn = _load().oracle_group_quant_ue8m0 if ue8m0 else _load().oracle_group_quant
    rc = fn(_ptr(x), int(is_f32), M, K, K, int(col_major), ld_s, _ptr(q), K, _ptr(s))
    if rc != 0:
        raise ValueError(f"oracle_group_quant rejected its arguments ({rc})")
    return q, s


def blocked_gemm(A: np.ndarray, B: np.ndarray, As: np.ndarray, as_col_major: bool,
                 Bs: np.ndarray, rows=None, want_f64: bool = False, want_abs: bool = False,
                 threads: int = 0):
    """out[r, n] = bf16( sum_kb (A[m,kb].B[n,kb]) As[m,kb] Bs[n/128,kb] ), m = rows[r].

    A uint8 [M, K], B uint8 [N, K] (e4m3 codes); As as returned by group_quant
    (layout given by as_col_major, leading dimension = As.shape[1]); Bs float32
    [ceil(N/128), ceil(K/128)].  Returns a dict with 'bf16' (uint16 bits) and,
    on request, 'f64' (sum before rounding) and 'abs' (sum of |terms|).
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    As = np.ascontiguousarray(As, dtype=np.float32)
    Bs = np.ascontiguousarray(Bs, dtype=np.float32)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    G = (K + 127) // 128
    assert Bs.shape == ((N + 127) // 128, G), Bs.shape
    ld_as = As.shape[1]
    if rows is None:
        rows_arr = None
        n_rows = M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
    out = np.empty((n_rows, N), dtype=np.uint16)
    f64 = np.empty((n_rows, N), dtype=np.float64) if want_f64 else None
    ab = np.empty((n_rows, N), dtype=np.float64) if want_abs else None
    rc = _load().oracle_blocked_gemm(
        _ptr(A), _ptr(B), _ptr(As), int(as_col_major), ld_as, _ptr(Bs), M, N, K,
        _ptr(rows_arr) if rows_arr is not None else None, n_rows, _ptr(out),
        _ptr(f64) if f64 is not None else None, _ptr(ab) if ab is not None else None,
        int(threads))
    if rc != 0:
        raise ValueError(f"oracle_blocked_gemm failed ({rc})")
    res = {"bf16": out}
    if f64 is not None:
        res["f64"] = f64
    if ab is not None:
        res["abs"] = ab
    return res


def expert_of_rows(psum: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Expert of each row under the cumulative layout psum [E] (rows
    [psum[e-1], psum[e]) belong to expert e); -1 for rows past psum[E-1]."""
    psum = np.asarray(psum, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    e = np.searchsorted(psum, rows, side="right")
    return np.where(e < psum.size, e, -1)


def grouped_gemm(A: np.ndarray, B: np.ndarray, As: np.ndarray, as_col_major: bool,
                 Bs: np.ndarray, psum: np.ndarray, rows=None, want_abs: bool = False,
                 threads: int = 0):
    """M-grouped blocked GEMM: row m of expert e = blocked_gemm with B[e], Bs[e].

    A uint8 [M, K]; B uint8 [E, N, K]; Bs float32 [E, ceil(N/128), G]; psum
    int [E] cumulative row counts.  Returns a dict with 'bf16' [n_rows, N]
    (rows past the last expert hold 0), 'expert' [n_rows] (-1 for those rows)
    and, on request, 'abs'.
    """
    M = A.shape[0]
    E, N, _ = B.shape
    rows_arr = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    experts = expert_of_rows(psum, rows_arr)
    out = np.zeros((rows_arr.size, N), dtype=np.uint16)
    ab = np.zeros((rows_arr.size, N), dtype=np.float64) if want_abs else None
    for e in range(E):
        sel = np.nonzero(experts == e)[0]
        if sel.size == 0:
            continue
        r = blocked_gemm(A, B[e], As, as_col_major, Bs[e], rows=rows_arr[sel],
                         want_abs=want_abs, threads=threads)
        out[sel] = r["bf16"]
        if ab is not None:
            ab[sel] = r["abs"]
    res = {"bf16": out, "expert": experts}
    if ab is not None:
        res["abs"] = ab
    return res


def bias_add_bf16(y_bits: np.ndarray, bias_bits: np.ndarray) -> np.ndarray:
    """bf16 [.., N] + bf16 [N]: each sum is one IEEE fp32 addition of the two
    values, rounded to nearest-even bf16 (bits in, bits out)."""
    y = (np.asarray(y_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    b = (np.asarray(bias_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    s32 = (y + b).astype(np.float32)          # numpy adds float32 in float32 (IEEE)
    return bf16_from_f64(s32.astype(np.float64))


def fused_linear(A: np.ndarray, B: np.ndarray, As: np.ndarray, as_col_major: bool,
                 Bs: np.ndarray, bias_bits=None, col_major_out: bool = True, rows=None,
                 threads: int = 0):
    """y = bf16 GEMM (+ bias as a bf16 addition), then y's 1x128 group
    quantisation.  Returns dict(y bf16 bits [n_rows, N], q [n_rows, N] codes,
    s scales in the requested layout, abs)."""
    r = blocked_gemm(A, B, As, as_col_major, Bs, rows=rows, want_abs=True, threads=threads)
    y = r["bf16"]
    if bias_bits is not None:
        y = bias_add_bf16(y, bias_bits)
    q, sc = group_quant(np.ascontiguousarray(y), False, col_major_out)
    return {"bf16": y, "q": q, "s": sc, "abs": r["abs"]}
