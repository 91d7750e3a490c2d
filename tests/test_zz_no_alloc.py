"""pa_q8_decode_noalloc, called through the C ABI, against pa_q8_decode.

Some callers cannot give the library device memory for scratch -- a plugin
inside another runtime that owns every device allocation, or a serving loop
that may not call an allocator -- so pa_q8_decode_noalloc keeps the
split-context partials in a fixed buffer compiled into the library.  This
test checks, on two calls in a row with different inputs, that its output
matches the workspace-taking entry point within the decode tolerance
(|a - b| <= 1e-5 + 1e-4 |b|), that a shape whose partials would not fit the
buffer is refused, and that nothing was flagged on the device.  The file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from int8_paged_kv_gb300 import build, _binding
    build.build()
    L = _binding.lib()
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.pa_q8_decode_noalloc.restype = i32
    L.pa_q8_decode_noalloc.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, P]
    return L


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, out, q, kc, vc, bt, cl, w, stream):
    cfg = w.cfg
    return L.pa_q8_decode_noalloc(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                                  cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size,
                                  cfg.block_size, cfg.max_blocks_per_seq, w.num_blocks,
                                  ctypes.c_float(w.scale), ctypes.c_void_p(stream))


def test_noalloc_matches_decode_on_two_calls(lib):
    import torch
    import int8_paged_kv_gb300 as pk
    from int8_paged_kv_gb300 import workloads as wl

    w = wl.build("llama8b")
    cfg = w.cfg
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    dev = torch.device("cuda")

    def u32(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)

    W = D // 4 + 1
    kc = torch.full((w.num_blocks, Hk, B, W), -1, dtype=torch.int32, device=dev)
    vc = torch.full_like(kc, -1)
    T = w.key.shape[0]
    pk.pa_q8_reshape_and_cache(torch.from_numpy(w.key.reshape(T, -1)).to(dev),
                               torch.from_numpy(w.value.reshape(T, -1)).to(dev), kc, vc,
                               u32(w.slot_mapping), num_kv_heads=Hk, head_size=D, block_size=B)
    need = pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq)
    assert 0 < need <= 64 << 20            # this shape uses the split-context partials
    stream = torch.cuda.current_stream().cuda_stream
    bt = u32(w.block_tables)
    rng = np.random.default_rng(99)

    for call in range(2):
        # second call: other queries and shorter contexts, so stale partials
        # left in the shared buffer by the first call would show
        qn = w.q if call == 0 else rng.standard_normal(w.q.shape).astype(np.float32)
        cln = w.context_lens if call == 0 else (w.context_lens // 3 + 1).astype(np.uint32)
        q = torch.from_numpy(qn).to(dev)
        cl = u32(cln)
        ref = torch.full_like(q, float("nan"))
        pk.pa_q8_decode(ref, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale)
        got = torch.full_like(q, float("nan"))
        rc = _noalloc(lib, got, q, kc, vc, bt, cl, w, stream)
        assert rc == 0, pk.pa_q8_status_string(rc)
        torch.cuda.synchronize()
        a = got.cpu().numpy().astype(np.float64)
        b = ref.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert np.all(np.abs(a - b) <= 1e-5 + 1e-4 * np.abs(b)), f"call {call}"
    assert pk.pa_q8_device_status(clear=True) == 0


def test_noalloc_refuses_shapes_beyond_its_buffer(lib):
    import torch
    import int8_paged_kv_gb300 as pk
    # 4096 sequences x 64 heads with contexts up to 8192 tokens need more than
    # the fixed buffer for their partials: refused on the host, nothing launched
    S, H, Hk, D, B, Nb = 4096, 64, 8, 128, 16, 512
    assert pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, Nb) > 64 << 20
    dummy = torch.empty(64, dtype=torch.float32, device="cuda")
    p = _ptr(dummy)
    rc = lib.pa_q8_decode_noalloc(p, p, p, p, p, p, S, H, Hk, D, B, Nb, 1 << 20, ctypes.c_float(0.1),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -5, pk.pa_q8_status_string(rc)
