"""Oracle for the dense FP16 GEMM hot path: plain, slow, obviously correct.

TEST INFRASTRUCTURE ONLY. Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``dense_gemm_gb300``) never imports it, and this
package imports nothing from the product.

Contents
--------
``gemm`` / ``gemm_rows``
    C[i, j] = sum_k A[i, k] * B[k, j] with every fp16 input widened exactly to
    double and the sum taken in double, k ascending (C code in
    ``oracle_gemm.c``). Source of the semantics: "(1/n) Triton matmul 커널 탐험
    - persistent kernel은 그 자체로 빠르지 않다", section "naive tiled matmul"
    (masked loads with zero fill, FP32 accumulator from zero, C overwritten).
``tile_coord`` / ``schedule``
    Row-major and grouped ("CTA swizzle") tile maps, "(2/n) Triton matmul 커널
    탐험 - grouped ordering(CTA swizzle)...", section "구현"; persistent
    visiting order from "(1/n) ...", section "naive persistent matmul".
``fp16_to_f64`` / ``bf16_to_f64`` / ``f64_to_f16_bits`` / ``f64_to_bf16_bits``
    decoding and round-to-nearest-even encoding of binary16 and bfloat16 from
    the formats' definitions (for the 16-bit C outputs).
``counts``
    FLOP / HBM-byte / panel-size formulas of "4주차 정리: Roofline과 Tiling"
    (sections 1, 2 and 5) and of the "(2/n)" page's section "재사용 거리와 캐시
    용량".

Every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle.py`` and ``tests/test_oracle_counts.py``. No function is
"parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import counts  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    from .build import build
    path = build()
    lib = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_f64.restype = ctypes.c_double
    lib.oracle_gemm_block.argtypes = [p, p, i64, i64, i64, i64, i64, i64, i64,
                                      p, i64, i64, i64, p, ctypes.c_int]
    lib.oracle_gemm_block.restype = ctypes.c_int
    lib.oracle_tile_coord.argtypes = [i64, i64, i64, i64, ctypes.c_int,
                                      ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.oracle_tile_coord.restype = ctypes.c_int
    lib.oracle_schedule.argtypes = [i64, i64, i64, ctypes.c_int, i64, p]
    lib.oracle_schedule.restype = ctypes.c_int
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_init()
    _lib = lib
    return lib


def max_threads() -> int:
    """Threads the OpenMP runtime would use by default."""
    return int(_load().oracle_max_threads())


def fp16_to_f64(bits: int) -> float:
    return float(_load().oracle_fp16_to_f64(int(bits) & 0xFFFF))


def f64_to_f16_bits(x: float) -> int:
    """Nearest binary16 (ties to even) as a bit pattern."""
    return int(_load().oracle_f64_to_f16(float(x)))


def f64_to_bf16_bits(x: float) -> int:
    """Nearest bfloat16 (ties to even) as a bit pattern."""
    return int(_load().oracle_f64_to_bf16(float(x)))


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def round_output(C64: np.ndarray, dtype: str, alpha: float = 1.0) -> np.ndarray:
    """round_dtype(alpha * C) elementwise, returned as float64 values.

    dtype: "f32" (IEEE binary32 via numpy's float32 cast, nearest-even),
    "f16" or "bf16" (this module's rounding)."""
    x = np.asarray(C64, dtype=np.float64) * alpha
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    lib = _load()
    enc = lib.oracle_f64_to_f16 if dtype == "f16" else lib.oracle_f64_to_bf16
    dec = lib.oracle_fp16_to_f64 if dtype == "f16" else lib.oracle_bf16_to_f64
    flat = x.ravel()
    out = np.fromiter((dec(enc(float(v))) for v in flat), dtype=np.float64, count=flat.size)
    return out.reshape(x.shape)


def _as_f16(x):
    """Accept a numpy float16/uint16 array or a CPU torch fp16 tensor (any strides)."""
    if hasattr(x, "numpy") and hasattr(x, "dtype") and str(x.dtype) == "torch.float16":
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must live on the host")
        x = x.numpy()  # shares storage and strides
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise ValueError("expected a 2-D float16 (or uint16 bit-pattern) array")
    return x


def _elem_strides(x):
    return tuple(s // x.itemsize for s in x.strides)


def gemm_rows(A, B, rows=None, col0: int = 0, ncols=None, threads: int = 0) -> np.ndarray:
    """Rows ``rows`` and columns ``[col0, col0+ncols)`` of A @ B, in float64.

    A: [M, K], B: [K, N], fp16, any (non-negative) strides. Returns a dense
    float64 array [len(rows), ncols].
    """
    A = _as_f16(A)
    B = _as_f16(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    sam, sak = _elem_strides(A)
    sbk, sbn = _elem_strides(B)
    if min(sam, sak, sbk, sbn) < 0:
        raise ValueError("negative strides are not supported")
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if ncols is None:
        ncols = N - col0
    out = np.empty((rows.size, ncols), dtype=np.float64)
    lib = _load()
    rc = lib.oracle_gemm_block(
        A.ctypes.data, B.ctypes.data, M, N, K, sam, sak, sbk, sbn,
        rows.ctypes.data, rows.size, col0, ncols, out.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle_gemm_block rejected its arguments")
    return out


def gemm(A, B, threads: int = 0) -> np.ndarray:
    """Full A @ B in float64 (dense [M, N])."""
    return gemm_rows(A, B, threads=threads)


def tile_coord(tile_id: int, nm: int, nn: int, G: int, grouped: bool):
    lib = _load()
    tm, tn = ctypes.c_int64(), ctypes.c_int64()
    rc = lib.oracle_tile_coord(tile_id, nm, nn, G, 1 if grouped else 0,
                               ctypes.byref(tm), ctypes.byref(tn))
    if rc != 0:
        raise ValueError("oracle_tile_coord rejected its arguments")
    return tm.value, tn.value


def schedule(nm: int, nn: int, G: int, grouped: bool, grid: int) -> np.ndarray:
    """[T, 3] int32 array: row tile_id = (program id, tile_m, tile_n)."""
    out = np.empty((nm * nn, 3), dtype=np.int32)
    rc = _load().oracle_schedule(nm, nn, G, 1 if grouped else 0, grid, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_schedule rejected its arguments")
    return out
