"""CPU oracle for the int8 paged-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path (the C-ABI library and its Python
binding) never loads it; the two share no code.

The arithmetic lives in ``pa_q8_oracle.c`` (plain C, fp64, OpenMP over
independent rows); this module compiles it with gcc on first use and wraps
it with ctypes.  Every function takes and returns numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_q8_oracle.c")
_LIB = os.path.join(_HERE, "libpa_q8_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/libpa_q8_oracle.so (gcc, -O2, no FMA
    contraction, no fast-math; OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, _SRC, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_quantize_vector.argtypes = [P, i32, P]
        lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32]
        lib.oracle_decode_partial.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f64,
                                              i32, i32, i64, i64, P, P, P]
        lib.oracle_combine.argtypes = [P, P, P, i32, i32, P]
        lib.oracle_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P, i64]
        lib.oracle_decode_rows.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, f64]
        lib.oracle_cq_append.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i64]
        lib.oracle_cq_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, f64, P, i64]
        lib.oracle_reshape_and_cache_f32.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32]
        lib.oracle_decode_f32.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P, i64]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _need(a, dtype, name):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous numpy {np.dtype(dtype).name} array")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the parallel loops from now on (results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def quantize_vector(x: np.ndarray) -> np.ndarray:
    """Codes + scale word of one f32 vector: u32 [len(x)/4 + 1]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 1 or x.size % 4:
        raise ValueError("x must be 1-D with a length that is a multiple of 4")
    out = np.empty(x.size // 4 + 1, dtype=np.uint32)
    _load().oracle_quantize_vector(_ptr(x), x.size, _ptr(out))
    return out


def reshape_and_cache(key: np.ndarray, value: np.ndarray, key_cache: np.ndarray,
                      value_cache: np.ndarray, slot_mapping: np.ndarray, *,
                      num_kv_heads: int, head_size: int, block_size: int,
                      key_stride: int | None = None, value_stride: int | None = None) -> None:
    """Quantise and scatter rows into the caches in place.

    key/value: f32 arrays whose rows start ``key_stride`` / ``value_stride``
    elements apart (default: num_kv_heads * head_size, i.e. [T, Hk, D]).
    A strided 2-D view (rows of a wider fused buffer) is accepted.
    """
    T = int(slot_mapping.shape[0])
    _need(slot_mapping, np.uint32, "slot_mapping")
    _need(key_cache, np.uint32, "key_cache")
    _need(value_cache, np.uint32, "value_cache")

    def base_and_stride(a, stride):
        if a.dtype != np.float32:
            raise TypeError("key/value must be float32")
        if a.flags.c_contiguous:
            return a, (stride if stride is not None else num_kv_heads * head_size)
        # a 2-D row view into a larger buffer: rows stride apart, each row contiguous
        if a.ndim != 2 or a.strides[1] != 4:
            raise ValueError("strided key/value must be 2-D views with contiguous rows")
        return a, a.strides[0] // 4

    k, ks = base_and_stride(key, key_stride)
    v, vs = base_and_stride(value, value_stride)
    _load().oracle_reshape_and_cache(
        ctypes.c_void_p(k.ctypes.data), ctypes.c_void_p(v.ctypes.data),
        _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping), T, ks, vs,
        num_kv_heads, head_size, block_size)


def decode(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
           block_tables: np.ndarray, context_lens: np.ndarray, *, num_kv_heads: int,
           block_size: int, scale: float, rows: np.ndarray | None = None) -> np.ndarray:
    """fp64 decode.  Returns [S, H, D] (rows=None) or [n_rows, D] for the
    given int32 (s, h) pairs."""
    _need(q, np.float32, "q")
    for a, n in ((key_cache, "key_cache"), (value_cache, "value_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens")):
        _need(a, np.uint32, n)
    S, H, D = q.shape
    Nb = block_tables.shape[1]
    if rows is None:
        out = np.empty((S, H, D), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.empty((rows.shape[0], D), dtype=np.float64)
        rp, nr = _ptr(rows), rows.shape[0]
    _load().oracle_decode(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache),
                          _ptr(block_tables), _ptr(context_lens), S, H, num_kv_heads, D,
                          block_size, Nb, float(scale), rp, nr)
    return out


def decode_rows(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                block_tables: np.ndarray, context_lens: np.ndarray, *, num_kv_heads: int,
                block_size: int, scale: float) -> np.ndarray:
    """fp64 multi-row causal decode: q [S, R, H, D]; row b of sequence s
    attends to the first min(context_len, cap) - (R - 1 - b) tokens.
    Returns [S, R, H, D]."""
    _need(q, np.float32, "q")
    for a, n in ((key_cache, "key_cache"), (value_cache, "value_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens")):
        _need(a, np.uint32, n)
    S, R, H, D = q.shape
    out = np.empty((S, R, H, D), dtype=np.float64)
    _load().oracle_decode_rows(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache),
                               _ptr(block_tables), _ptr(context_lens), S, R, H, num_kv_heads, D,
                               block_size, block_tables.shape[1], float(scale))
    return out


def decode_partial(q, key_cache, value_cache, block_tables, *, num_kv_heads: int,
                   block_size: int, scale: float, s: int, h: int, t0: int, t1: int):
    """(m, l, acc[D]) of row (s, h) over logical tokens [t0, t1)."""
    S, H, D = q.shape
    acc = np.empty(D, dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    _load().oracle_decode_partial(_ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
                                  H, num_kv_heads, D, block_size, block_tables.shape[1],
                                  float(scale), s, h, t0, t1, ctypes.byref(m), ctypes.byref(l),
                                  _ptr(acc))
    return m.value, l.value, acc


def combine(m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
    """Log-sum-exp merge of n partials: m, l [n] f64, acc [n, D] f64."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    n, D = acc.shape
    out = np.empty(D, dtype=np.float64)
    _load().oracle_combine(_ptr(m), _ptr(l), _ptr(acc), n, D, _ptr(out))
    return out


# ----------------------------------------------------------------- f32 cache
# The f32 variant of the cache: [num_blocks, num_kv_heads, block_size,
# head_size] f32 (the q8 layout with f32 elements and no scale word).


def reshape_and_cache_f32(key: np.ndarray, value: np.ndarray, key_cache: np.ndarray,
                          value_cache: np.ndarray, slot_mapping: np.ndarray, *,
                          num_kv_heads: int, head_size: int, block_size: int) -> None:
    """Copy rows into the f32 caches in place (PAD slots skipped).  key/value:
    f32 [T, Hk, D] or a 2-D view of rows with contiguous elements."""
    T = int(slot_mapping.shape[0])
    _need(slot_mapping, np.uint32, "slot_mapping")
    _need(key_cache, np.float32, "key_cache")
    _need(value_cache, np.float32, "value_cache")

    def base_and_stride(a):
        if a.dtype != np.float32:
            raise TypeError("key/value must be float32")
        if a.flags.c_contiguous:
            return a, num_kv_heads * head_size
        if a.ndim != 2 or a.strides[1] != 4:
            raise ValueError("strided key/value must be 2-D views with contiguous rows")
        return a, a.strides[0] // 4

    k, ks = base_and_stride(key)
    v, vs = base_and_stride(value)
    _load().oracle_reshape_and_cache_f32(
        ctypes.c_void_p(k.ctypes.data), ctypes.c_void_p(v.ctypes.data),
        _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping), T, ks, vs,
        num_kv_heads, head_size, block_size)


def decode_f32(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
               block_tables: np.ndarray, context_lens: np.ndarray, *, num_kv_heads: int,
               block_size: int, scale: float, rows: np.ndarray | None = None) -> np.ndarray:
    """fp64 decode over the f32 caches.  Returns [S, H, D] (rows=None) or
    [n_rows, D] for the given int32 (s, h) pairs."""
    _need(q, np.float32, "q")
    _need(key_cache, np.float32, "key_cache")
    _need(value_cache, np.float32, "value_cache")
    _need(block_tables, np.uint32, "block_tables")
    _need(context_lens, np.uint32, "context_lens")
    S, H, D = q.shape
    Nb = block_tables.shape[1]
    if rows is None:
        out = np.empty((S, H, D), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.empty((rows.shape[0], D), dtype=np.float64)
        rp, nr = _ptr(rows), rows.shape[0]
    _load().oracle_decode_f32(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache),
                              _ptr(block_tables), _ptr(context_lens), S, H, num_kv_heads, D,
                              block_size, Nb, float(scale), rp, nr)
    return out


# -------------------------------------------------------- contiguous q8 cache
# Per sequence: [max_t][kv_row] int8 codes (u32 words), then [max_t][kv_row/32]
# f32 group scales; sequences back to back (see pa_q8_oracle.c).


def cq_seq_words(max_t: int, num_kv_heads: int, head_size: int) -> int:
    kv_row = num_kv_heads * head_size
    return max_t * kv_row // 4 + max_t * kv_row // 32


def cq_append(key: np.ndarray, value: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
              slot_mapping: np.ndarray, *, num_kv_heads: int, head_size: int, max_t: int) -> None:
    """Quantise rows (slot = sequence * max_t + position) into the contiguous
    caches in place, one scale per 32-element group."""
    T = int(slot_mapping.shape[0])
    _need(slot_mapping, np.uint32, "slot_mapping")
    _need(key_cache, np.uint32, "key_cache")
    _need(value_cache, np.uint32, "value_cache")

    def base_and_stride(a):
        if a.dtype != np.float32:
            raise TypeError("key/value must be float32")
        if a.flags.c_contiguous:
            return a, num_kv_heads * head_size
        if a.ndim != 2 or a.strides[1] != 4:
            raise ValueError("strided key/value must be 2-D views with contiguous rows")
        return a, a.strides[0] // 4

    k, ks = base_and_stride(key)
    v, vs = base_and_stride(value)
    _load().oracle_cq_append(ctypes.c_void_p(k.ctypes.data), ctypes.c_void_p(v.ctypes.data),
                             _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping), T, ks, vs,
                             num_kv_heads, head_size, int(max_t))


def cq_decode(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray, context_lens: np.ndarray, *,
              num_kv_heads: int, max_t: int, scale: float, rows: np.ndarray | None = None) -> np.ndarray:
    """fp64 decode over the contiguous caches: [S, H, D] or [n_rows, D]."""
    _need(q, np.float32, "q")
    for a, n in ((key_cache, "key_cache"), (value_cache, "value_cache"), (context_lens, "context_lens")):
        _need(a, np.uint32, n)
    S, H, D = q.shape
    if rows is None:
        out = np.empty((S, H, D), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.empty((rows.shape[0], D), dtype=np.float64)
        rp, nr = _ptr(rows), rows.shape[0]
    _load().oracle_cq_decode(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(context_lens),
                             S, H, num_kv_heads, D, int(max_t), float(scale), rp, nr)
    return out
