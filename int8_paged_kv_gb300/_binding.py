"""ctypes binding of libpa_q8.so -- argument marshalling only.

Every function here checks dtypes / devices / shapes of torch tensors,
passes their ``data_ptr()`` and the current CUDA stream to the C entry
point of the same name, and turns a negative status into an exception.
All arithmetic happens in the library's CUDA kernels; there is no fallback:
without the compiled library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_q8.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pa_q8.h")

PA_Q8_KERNEL_AUTO = 0
PA_Q8_KERNEL_CUDA_CORE = 1
PA_Q8_KERNEL_TENSOR_CORE = 2
PA_Q8_KERNEL_TCGEN05 = 3
PA_Q8_DEV_BAD_BLOCK = 0x1
PA_Q8_DEV_BAD_SLOT = 0x2
PA_Q8_DEV_WAIT_TIMEOUT = 0x4

_lock = threading.Lock()
_lib = None


class PaQ8Error(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


class DecodeOptions(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("partition_tokens", ctypes.c_int)]


def lib() -> ctypes.CDLL:
    """Load libpa_q8.so (built by int8_paged_kv_gb300.build); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m int8_paged_kv_gb300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                                     ctypes.c_float, ctypes.c_size_t)
        L.pa_q8_version.restype = i32
        L.pa_q8_version.argtypes = []
        L.pa_q8_status_string.restype = ctypes.c_char_p
        L.pa_q8_status_string.argtypes = [i32]
        L.pa_q8_reshape_and_cache.restype = i32
        L.pa_q8_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32, i64, P]
        dec = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, P, sz, P]
        L.pa_q8_decode.restype = i32
        L.pa_q8_decode.argtypes = dec
        L.pa_q8_decode_ex.restype = i32
        L.pa_q8_decode_ex.argtypes = dec + [ctypes.POINTER(DecodeOptions)]
        L.pa_q8_decode_rows.restype = i32
        L.pa_q8_decode_rows.argtypes = ([P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, f32,
                                         P, sz, P, ctypes.POINTER(DecodeOptions)])
        L.pa_q8_decode_append.restype = i32
        L.pa_q8_decode_append.argtypes = ([P, P, P, P, i64, i64, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                           i32, i64, f32, P, sz, P, ctypes.POINTER(DecodeOptions)])
        L.pa_q8c_cache_words.restype = sz
        L.pa_q8c_cache_words.argtypes = [i64, i32, i32]
        L.pa_q8c_append.restype = i32
        L.pa_q8c_append.argtypes = [P, P, i64, i64, P, P, P, i64, i32, i32, i64, i32, P]
        L.pa_q8c_decode.restype = i32
        L.pa_q8c_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, f32, P, sz, P,
                                    ctypes.POINTER(DecodeOptions)]
        L.pa_q8c_decode_workspace_size.restype = sz
        L.pa_q8c_decode_workspace_size.argtypes = [i32, i32, i32, i32, i64, ctypes.POINTER(DecodeOptions)]
        L.pa_f32_reshape_and_cache.restype = i32
        L.pa_f32_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32, i64, P]
        L.pa_f32_decode.restype = i32
        L.pa_f32_decode.argtypes = dec + [ctypes.POINTER(DecodeOptions)]
        L.pa_f32_decode_workspace_size.restype = sz
        L.pa_f32_decode_workspace_size.argtypes = [i32] * 6 + [ctypes.POINTER(DecodeOptions)]
        L.pa_q8_decode_rows_workspace_size.restype = sz
        L.pa_q8_decode_rows_workspace_size.argtypes = [i32] * 7 + [ctypes.POINTER(DecodeOptions)]
        L.pa_q8_decode_workspace_size.restype = sz
        L.pa_q8_decode_workspace_size.argtypes = [i32] * 6
        L.pa_q8_decode_workspace_size_ex.restype = sz
        L.pa_q8_decode_workspace_size_ex.argtypes = [i32] * 6 + [ctypes.POINTER(DecodeOptions)]
        L.pa_q8_decode_plan.restype = i32
        L.pa_q8_decode_plan.argtypes = [i32] * 6 + [ctypes.POINTER(DecodeOptions),
                                                    ctypes.POINTER(i32), ctypes.POINTER(i32),
                                                    ctypes.POINTER(i32), ctypes.POINTER(i64)]
        L.pa_q8_device_status.restype = i32
        L.pa_q8_device_status.argtypes = [ctypes.POINTER(u32), i32, P]
        L.pa_q8_selftest_wait_timeout.restype = i32
        L.pa_q8_selftest_wait_timeout.argtypes = [u32, P]
        _lib = L
        return L


def pa_q8_status_string(status: int) -> str:
    return lib().pa_q8_status_string(int(status)).decode()


def pa_q8_version() -> int:
    return int(lib().pa_q8_version())


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise PaQ8Error(fn, rc, pa_q8_status_string(rc))


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t, dtype, name):
    """Device pointer of a CUDA tensor; u32 buffers may also be int32 (same bits)."""
    import torch
    ok = (torch.uint32, torch.int32) if dtype is torch.uint32 else (dtype,)
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in ok:
        raise TypeError(f"{name} must be a CUDA tensor of dtype {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _opts(kernel: int, partition_tokens: int):
    return ctypes.byref(DecodeOptions(int(kernel), int(partition_tokens)))


def pa_q8_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, *, num_kv_heads: int,
                            head_size: int, block_size: int, num_blocks: int | None = None,
                            stream=None) -> None:
    """Quantise rows of `key`/`value` into the caches.

    key/value: float32 CUDA tensors whose first dimension is the token and
    whose rows hold num_kv_heads * head_size contiguous floats; rows may be
    further apart (e.g. K/V column slices of fused QKV rows): the row stride
    is taken from the tensor.  Caches: uint32 [num_blocks, Hk, B, D/4 + 1].
    """
    import torch
    for t, n in ((key, "key"), (value, "value")):
        if t.dim() < 2 or t.stride(-1) != 1:
            raise ValueError(f"{n} rows must be contiguous in their last dimension")
        inner = t[0] if t.dim() > 2 else None
        if inner is not None and not inner.is_contiguous():
            raise ValueError(f"{n} must be [T, Hk, D] with contiguous rows")
    T = int(slot_mapping.numel())
    if key.shape[0] != T or value.shape[0] != T:
        raise ValueError("key/value rows must match slot_mapping")
    nb = int(key_cache.shape[0]) if num_blocks is None else int(num_blocks)
    rc = lib().pa_q8_reshape_and_cache(
        _cuda(key, torch.float32, "key"), _cuda(value, torch.float32, "value"),
        _cuda(key_cache, torch.uint32, "key_cache"), _cuda(value_cache, torch.uint32, "value_cache"),
        _cuda(slot_mapping, torch.uint32, "slot_mapping"), T, int(key.stride(0)),
        int(value.stride(0)), int(num_kv_heads), int(head_size), int(block_size), nb, _stream(stream))
    _check("pa_q8_reshape_and_cache", rc)


def pa_q8_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                max_blocks_per_seq, *, kernel: int = 0,
                                partition_tokens: int = 0) -> int:
    return int(lib().pa_q8_decode_workspace_size_ex(int(num_seqs), int(num_heads), int(num_kv_heads),
                                                    int(head_size), int(block_size),
                                                    int(max_blocks_per_seq),
                                                    _opts(kernel, partition_tokens)))


def pa_q8_decode_plan(num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq,
                      *, kernel: int = 0, partition_tokens: int = 0) -> dict:
    k, pt, np_ = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    nc = ctypes.c_int64()
    rc = lib().pa_q8_decode_plan(int(num_seqs), int(num_heads), int(num_kv_heads), int(head_size),
                                 int(block_size), int(max_blocks_per_seq),
                                 _opts(kernel, partition_tokens), ctypes.byref(k),
                                 ctypes.byref(pt), ctypes.byref(np_), ctypes.byref(nc))
    _check("pa_q8_decode_plan", rc)
    return {"kernel": k.value, "partition_tokens": pt.value, "num_partitions": np_.value,
            "num_ctas": nc.value}


def pa_q8_decode(out, q, key_cache, value_cache, block_tables, context_lens, *, num_kv_heads: int,
                 block_size: int, scale: float, num_blocks: int | None = None, workspace=None,
                 kernel: int = 0, partition_tokens: int = 0, stream=None):
    """out[S, H, D] = paged int8 attention decode (see include/pa_q8.h).

    workspace: a uint8 CUDA tensor of >= pa_q8_decode_workspace_size bytes;
    allocated here (torch) when None.  Returns `out`.
    """
    import torch
    S, H, D = q.shape
    if out.shape != q.shape or not out.is_contiguous() or not q.is_contiguous():
        raise ValueError("q and out must be contiguous [num_seqs, num_heads, head_size]")
    Nb = int(block_tables.shape[1])
    if block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables / context_lens do not match num_seqs")
    nb = int(key_cache.shape[0]) if num_blocks is None else int(num_blocks)
    need = pa_q8_decode_workspace_size(S, H, num_kv_heads, D, block_size, Nb, kernel=kernel,
                                       partition_tokens=partition_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_q8_decode_ex(
        _cuda(out, torch.float32, "out"), _cuda(q, torch.float32, "q"),
        _cuda(key_cache, torch.uint32, "key_cache"), _cuda(value_cache, torch.uint32, "value_cache"),
        _cuda(block_tables, torch.uint32, "block_tables"),
        _cuda(context_lens, torch.uint32, "context_lens"), S, H, int(num_kv_heads), D,
        int(block_size), Nb, nb, float(scale), ws_ptr, ws_bytes, _stream(stream),
        _opts(kernel, partition_tokens))
    _check("pa_q8_decode", rc)
    return out


def pa_q8_decode_rows_workspace_size(num_seqs, num_rows, num_heads, num_kv_heads, head_size,
                                     block_size, max_blocks_per_seq, *, kernel: int = 0,
                                     partition_tokens: int = 0) -> int:
    return int(lib().pa_q8_decode_rows_workspace_size(
        int(num_seqs), int(num_rows), int(num_heads), int(num_kv_heads), int(head_size),
        int(block_size), int(max_blocks_per_seq), _opts(kernel, partition_tokens)))


def pa_q8_decode_rows(out, q, key_cache, value_cache, block_tables, context_lens, *,
                      num_kv_heads: int, block_size: int, scale: float,
                      num_blocks: int | None = None, workspace=None, kernel: int = 0,
                      partition_tokens: int = 0, stream=None):
    """out[S, R, H, D] = causal multi-row decode: row b of sequence s attends
    to the first c - (R - 1 - b) cached tokens (see include/pa_q8.h).
    Returns `out`."""
    import torch
    S, R, H, D = q.shape
    if out.shape != q.shape or not out.is_contiguous() or not q.is_contiguous():
        raise ValueError("q and out must be contiguous [num_seqs, num_rows, num_heads, head_size]")
    Nb = int(block_tables.shape[1])
    if block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables / context_lens do not match num_seqs")
    nb = int(key_cache.shape[0]) if num_blocks is None else int(num_blocks)
    need = pa_q8_decode_rows_workspace_size(S, R, H, num_kv_heads, D, block_size, Nb, kernel=kernel,
                                            partition_tokens=partition_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_q8_decode_rows(
        _cuda(out, torch.float32, "out"), _cuda(q, torch.float32, "q"),
        _cuda(key_cache, torch.uint32, "key_cache"), _cuda(value_cache, torch.uint32, "value_cache"),
        _cuda(block_tables, torch.uint32, "block_tables"),
        _cuda(context_lens, torch.uint32, "context_lens"), S, R, H, int(num_kv_heads), D,
        int(block_size), Nb, nb, float(scale), ws_ptr, ws_bytes, _stream(stream),
        _opts(kernel, partition_tokens))
    _check("pa_q8_decode_rows", rc)
    return out


def _rows2d(t, n_rows, name):
    """(tensor, row stride in floats) of new K/V rows given as [S, R, Hk, D]
    / [S, R, Hk * D] (contiguous) or [S * R, Hk * D] (rows may be strided)."""
    if t.dim() == 2:
        if t.shape[0] != n_rows or t.stride(1) != 1:
            raise ValueError(f"{name}: expected [num_seqs * num_rows, num_kv_heads * head_size] rows")
        return t, int(t.stride(0))
    if not t.is_contiguous() or t.shape[0] * t.shape[1] != n_rows:
        raise ValueError(f"{name}: expected contiguous [num_seqs, num_rows, ...] rows")
    return t, int(t[0].numel() // t.shape[1])


def pa_q8_decode_append(out, q, key, value, key_cache, value_cache, block_tables, context_lens, *,
                        num_kv_heads: int, block_size: int, scale: float,
                        num_blocks: int | None = None, workspace=None, kernel: int = 0,
                        partition_tokens: int = 0, stream=None):
    """Append the newest num_rows tokens' K/V (rows of key / value) to the
    caches and decode q [S, R, H, D] over them, in one attention launch (see
    include/pa_q8.h).  Returns `out`."""
    import torch
    S, R, H, D = q.shape
    if out.shape != q.shape or not out.is_contiguous() or not q.is_contiguous():
        raise ValueError("q and out must be contiguous [num_seqs, num_rows, num_heads, head_size]")
    Nb = int(block_tables.shape[1])
    if block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables / context_lens do not match num_seqs")
    k2, ks = _rows2d(key, S * R, "key")
    v2, vs = _rows2d(value, S * R, "value")
    nb = int(key_cache.shape[0]) if num_blocks is None else int(num_blocks)
    need = pa_q8_decode_rows_workspace_size(S, R, H, num_kv_heads, D, block_size, Nb, kernel=kernel,
                                            partition_tokens=partition_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_q8_decode_append(
        _cuda(out, torch.float32, "out"), _cuda(q, torch.float32, "q"),
        _cuda(k2, torch.float32, "key"), _cuda(v2, torch.float32, "value"), ks, vs,
        _cuda(key_cache, torch.uint32, "key_cache"), _cuda(value_cache, torch.uint32, "value_cache"),
        _cuda(block_tables, torch.uint32, "block_tables"),
        _cuda(context_lens, torch.uint32, "context_lens"), S, R, H, int(num_kv_heads), D,
        int(block_size), Nb, nb, float(scale), ws_ptr, ws_bytes, _stream(stream),
        _opts(kernel, partition_tokens))
    _check("pa_q8_decode_append", rc)
    return out


def pa_f32_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, *, num_kv_heads: int,
                             head_size: int, block_size: int, num_blocks: int | None = None,
                             stream=None) -> None:
    """Copy rows into the f32 caches [num_blocks, Hk, B, D] (see include/pa_q8.h)."""
    import torch
    T = int(slot_mapping.numel())
    if key.dim() != 2 or value.dim() != 2 or key.stride(1) != 1 or value.stride(1) != 1:
        raise ValueError("key/value must be 2-D [num_tokens, >= num_kv_heads * head_size] with unit column stride")
    nb = int(key_cache.shape[0]) if num_blocks is None else int(num_blocks)
    rc = lib().pa_f32_reshape_and_cache(
        _cuda(key, torch.float32, "key"), _cuda(value, torch.float32, "value"),
        _cuda(key_cache, torch.float32, "key_cache"), _cuda(value_cache, torch.float32, "value_cache"),
        _cuda(slot_mapping, torch.uint32, "slot_mapping"), T, int(key.stride(0)), int(value.stride(0)),
        int(num_kv_heads), int(head_size), int(block_size), nb, _stream(stream))
    _check("pa_f32_reshape_and_cache", rc)


def pa_f32_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                 max_blocks_per_seq, *, partition_tokens: int = 0) -> int:
    return int(lib().pa_f32_decode_workspace_size(int(num_seqs), int(num_heads), int(num_kv_heads),
                                                  int(head_size), int(block_size), int(max_blocks_per_seq),
                                                  _opts(0, partition_tokens)))


def pa_f32_decode(out, q, key_cache, value_cache, block_tables, context_lens, *, num_kv_heads: int,
                  block_size: int, scale: float, num_blocks: int | None = None, workspace=None,
                  partition_tokens: int = 0, stream=None):
    """out[S, H, D] = paged attention decode over the f32 caches.  Returns `out`."""
    import torch
    S, H, D = q.shape
    if out.shape != q.shape or not out.is_contiguous() or not q.is_contiguous():
        raise ValueError("q and out must be contiguous [num_seqs, num_heads, head_size]")
    Nb = int(block_tables.shape[1])
    if block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables / context_lens do not match num_seqs")
    nb = int(key_cache.shape[0]) if num_blocks is None else int(num_blocks)
    need = pa_f32_decode_workspace_size(S, H, num_kv_heads, D, block_size, Nb,
                                        partition_tokens=partition_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_f32_decode(
        _cuda(out, torch.float32, "out"), _cuda(q, torch.float32, "q"),
        _cuda(key_cache, torch.float32, "key_cache"), _cuda(value_cache, torch.float32, "value_cache"),
        _cuda(block_tables, torch.uint32, "block_tables"),
        _cuda(context_lens, torch.uint32, "context_lens"), S, H, int(num_kv_heads), D,
        int(block_size), Nb, nb, float(scale), ws_ptr, ws_bytes, _stream(stream), _opts(0, partition_tokens))
    _check("pa_f32_decode", rc)
    return out


def pa_q8c_cache_words(max_t: int, num_kv_heads: int, head_size: int) -> int:
    return int(lib().pa_q8c_cache_words(int(max_t), int(num_kv_heads), int(head_size)))


def pa_q8c_append(key, value, key_cache, value_cache, slot_mapping, *, num_kv_heads: int, head_size: int,
                  max_t: int, num_seqs: int | None = None, stream=None) -> None:
    """Quantise rows into the contiguous caches (u32 [num_seqs, cache_words]);
    slot = sequence * max_t + position (see include/pa_q8.h)."""
    import torch
    T = int(slot_mapping.numel())
    if key.dim() != 2 or value.dim() != 2 or key.stride(1) != 1 or value.stride(1) != 1:
        raise ValueError("key/value must be 2-D [num_tokens, >= num_kv_heads * head_size] with unit column stride")
    ns = int(key_cache.shape[0]) if num_seqs is None else int(num_seqs)
    rc = lib().pa_q8c_append(
        _cuda(key, torch.float32, "key"), _cuda(value, torch.float32, "value"), int(key.stride(0)),
        int(value.stride(0)), _cuda(key_cache, torch.uint32, "key_cache"),
        _cuda(value_cache, torch.uint32, "value_cache"), _cuda(slot_mapping, torch.uint32, "slot_mapping"), T,
        int(num_kv_heads), int(head_size), int(max_t), ns, _stream(stream))
    _check("pa_q8c_append", rc)


def pa_q8c_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_t, *,
                                 partition_tokens: int = 0) -> int:
    return int(lib().pa_q8c_decode_workspace_size(int(num_seqs), int(num_heads), int(num_kv_heads),
                                                  int(head_size), int(max_t), _opts(0, partition_tokens)))


def pa_q8c_decode(out, q, key_cache, value_cache, context_lens, *, num_kv_heads: int, max_t: int,
                  scale: float, workspace=None, partition_tokens: int = 0, stream=None):
    """out[S, H, D] = decode over the contiguous caches.  Returns `out`."""
    import torch
    S, H, D = q.shape
    if out.shape != q.shape or not out.is_contiguous() or not q.is_contiguous():
        raise ValueError("q and out must be contiguous [num_seqs, num_heads, head_size]")
    if context_lens.numel() != S:
        raise ValueError("context_lens does not match num_seqs")
    need = pa_q8c_decode_workspace_size(S, H, num_kv_heads, D, max_t, partition_tokens=partition_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_q8c_decode(
        _cuda(out, torch.float32, "out"), _cuda(q, torch.float32, "q"),
        _cuda(key_cache, torch.uint32, "key_cache"), _cuda(value_cache, torch.uint32, "value_cache"),
        _cuda(context_lens, torch.uint32, "context_lens"), S, H, int(num_kv_heads), D, int(max_t), float(scale),
        ws_ptr, ws_bytes, _stream(stream), _opts(0, partition_tokens))
    _check("pa_q8c_decode", rc)
    return out


def pa_q8_device_status(clear: bool = True, stream=None) -> int:
    bits = ctypes.c_uint32()
    _check("pa_q8_device_status", lib().pa_q8_device_status(ctypes.byref(bits), int(bool(clear)),
                                                              _stream(stream)))
    return int(bits.value)


def pa_q8_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    _check("pa_q8_selftest_wait_timeout",
           lib().pa_q8_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def header_functions() -> list[str]:
    """Names of the functions include/pa_q8.h declares."""
    import re
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_(?:q8c?|f32)_[a-z0-9_]+)\s*\(", text)))
