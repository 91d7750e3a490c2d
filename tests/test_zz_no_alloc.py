"""pa_q8_decode_noalloc, called through the C ABI, against the fp64 oracle
and against pa_q8_decode.

Some callers cannot give the library device memory for scratch -- a plugin
inside another runtime that owns every device allocation, or a serving loop
that may not call an allocator -- so pa_q8_decode_noalloc keeps the
split-context partials in a fixed buffer compiled into the library.  This
test checks, on two calls in a row with different inputs (the second one
split into partitions), that its output is within the decode tolerance
(|gpu - oracle| <= 1e-5 + 1e-4 |oracle|) of the oracle's and of the
workspace-taking entry point's, that a shape whose scratch would not fit the
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


def _cache_from_rows(pk, key, value, slots, nblocks, Hk, D, B, dev):
    import torch
    W = D // 4 + 1
    kc = torch.full((nblocks, Hk, B, W), -1, dtype=torch.int32, device=dev)
    vc = torch.full_like(kc, -1)
    T = key.shape[0]
    pk.pa_q8_reshape_and_cache(key.reshape(T, -1), value.reshape(T, -1), kc, vc, slots,
                               num_kv_heads=Hk, head_size=D, block_size=B)
    return kc, vc


def test_noalloc_matches_oracle_and_decode_on_two_calls(lib):
    """Call 1: the 64-sequence workload (the buffer holds the sequence order
    and the CTA map, and the partials of any context the plan splits).  Call
    2: three ~20k-token contexts (split into partitions: the buffer holds
    their partials, over whatever call 1 left there).  Each output matches
    the oracle's (on caches the oracle writer built from the same rows) and
    pa_q8_decode's."""
    import torch
    import int8_paged_kv_gb300 as pk
    import oracle
    from int8_paged_kv_gb300 import workloads as wl
    from tests.gpu_helpers import assert_close, host_u32

    oracle.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def u32(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)

    def caches(w, key, value):
        """Device caches from the GPU writer and host caches from the oracle
        writer, from the same f32 rows (checked equal word for word)."""
        cfg = w.cfg
        Hk, D, B = cfg.num_kv_heads, cfg.head_size, cfg.block_size
        kc, vc = _cache_from_rows(pk, torch.from_numpy(key).to(dev), torch.from_numpy(value).to(dev),
                                  u32(w.slot_mapping), w.num_blocks, Hk, D, B, dev)
        W = D // 4 + 1
        ok_ = np.full((w.num_blocks, Hk, B, W), 0xFFFFFFFF, dtype=np.uint32)
        ov_ = ok_.copy()
        oracle.reshape_and_cache(key, value, ok_, ov_, w.slot_mapping, num_kv_heads=Hk, head_size=D,
                                 block_size=B)
        assert np.array_equal(host_u32(kc), ok_) and np.array_equal(host_u32(vc), ov_)
        return kc, vc, ok_, ov_

    cases = []
    w = wl.build("llama8b")
    cases.append((w, *caches(w, w.key, w.value)))
    w.key = w.value = None

    rng = np.random.default_rng(7)
    S, H, Hk, D, B = 3, 8, 2, 128, 16
    lens = np.array([20000, 17333, 19001], dtype=np.uint32)
    Nb = -(-int(lens.max()) // B)
    nblk = [-(-int(c) // B) for c in lens]
    perm = rng.permutation(sum(nblk)).astype(np.uint32)
    bt = np.full((S, Nb), 0xFFFFFFFF, dtype=np.uint32)
    pos, slots = 0, []
    for s_, c in enumerate(lens):
        bt[s_, :nblk[s_]] = perm[pos:pos + nblk[s_]]
        pos += nblk[s_]
        t = np.arange(int(c))
        slots.append(bt[s_, t // B].astype(np.int64) * B + t % B)
    slots = np.concatenate(slots).astype(np.uint32)
    T = slots.size
    key = rng.standard_normal((T, Hk, D)).astype(np.float32)
    value = rng.standard_normal((T, Hk, D)).astype(np.float32)
    cfg2 = wl.Config("three-long", 98, S, H, Hk, D, B, Nb * B)
    w2 = wl.Workload(cfg=cfg2, context_lens=lens, block_tables=bt, num_blocks=sum(nblk),
                     q=rng.standard_normal((S, H, D)).astype(np.float32),
                     scale=float(np.float32(D ** -0.5)), key=None, value=None, slot_mapping=slots,
                     row_seq=None)
    cases.append((w2, *caches(w2, key, value)))

    needs = [pk.pa_q8_decode_workspace_size(c.cfg.num_seqs, c.cfg.num_heads, c.cfg.num_kv_heads,
                                            c.cfg.head_size, c.cfg.block_size, c.cfg.max_blocks_per_seq)
             for c, *_ in cases]
    assert all(0 < n <= 64 << 20 for n in needs)    # both fit the fixed buffer

    for call, (wk, kck, vck, ok_, ov_) in enumerate(cases):
        c = wk.cfg
        want = oracle.decode(wk.q, ok_, ov_, wk.block_tables, wk.context_lens, num_kv_heads=c.num_kv_heads,
                             block_size=c.block_size, scale=wk.scale)
        q = torch.from_numpy(wk.q).to(dev)
        bt_d, cl_d = u32(wk.block_tables), u32(wk.context_lens)
        ref = torch.full_like(q, float("nan"))
        pk.pa_q8_decode(ref, q, kck, vck, bt_d, cl_d, num_kv_heads=c.num_kv_heads,
                        block_size=c.block_size, scale=wk.scale)
        got = torch.full_like(q, float("nan"))
        rc = _noalloc(lib, got, q, kck, vck, bt_d, cl_d, wk, stream)
        assert rc == 0, pk.pa_q8_status_string(rc)
        torch.cuda.synchronize()
        a = got.cpu().numpy().astype(np.float64)
        b = ref.cpu().numpy().astype(np.float64)
        assert_close(a, want, f"call {call}: noalloc against the oracle")
        assert_close(b, want, f"call {call}: pa_q8_decode against the oracle")
        assert np.all(np.abs(a - b) <= 1e-5 + 1e-4 * np.abs(b)), f"call {call}: noalloc against pa_q8_decode"
    assert pk.pa_q8_device_status(clear=True) == 0


def test_noalloc_refuses_shapes_beyond_its_buffer(lib):
    import torch
    import int8_paged_kv_gb300 as pk
    # 64 sequences x 64 heads (one kv head) with contexts up to 2^20 tokens
    # are split into many partitions whose partials need more than the fixed
    # buffer: refused on the host, nothing launched
    S, H, Hk, D, B, Nb = 64, 64, 1, 128, 16, 65536
    assert pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, Nb) > 64 << 20
    dummy = torch.empty(64, dtype=torch.float32, device="cuda")
    p = _ptr(dummy)
    rc = lib.pa_q8_decode_noalloc(p, p, p, p, p, p, S, H, Hk, D, B, Nb, 1 << 20, ctypes.c_float(0.1),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -5, pk.pa_q8_status_string(rc)
