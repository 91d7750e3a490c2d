"""The contiguous q8 cache (per-sequence code rows + side scale region,
32-element groups) on the GPU against its oracle: the append bit for bit
(oracle.cq_append), the decode within |gpu - oracle| <= 1e-5 + 1e-4 |oracle|
(oracle.cq_decode) on GQA ratios, head sizes, partition sizes, ragged, empty
and clamped contexts, and the 64-sequence workload's contexts."""
import numpy as np
import pytest

from int8_paged_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

PAD = 0xFFFFFFFF


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def _host(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("Hk,D", [(2, 64), (3, 128), (1, 256)])
def test_append_bit_exact_strided_pad_and_bad_slot(Hk, D):
    import torch
    import int8_paged_kv_gb300 as pk
    import oracle
    from tests.gpu_helpers import device_status
    rng = np.random.default_rng(D + Hk)
    S, max_t, T = 3, 40, 60
    kv_row = Hk * D
    slots = rng.choice(S * max_t, size=T, replace=False).astype(np.uint32)
    slots[[5, 17]] = PAD
    words = oracle.cq_seq_words(max_t, Hk, D)
    assert pk.pa_q8c_cache_words(max_t, Hk, D) == words
    for offset in (0, 1):                               # rows on and off 16-byte alignment
        buf = rng.standard_normal((T, 2 * kv_row + 5)).astype(np.float32)
        buf[3, offset:offset + 32] = 0.0                # an all-zero group
        buf[4, offset + 7] *= 30.0
        key = buf[:, offset:offset + kv_row]
        val = buf[:, offset + kv_row:offset + 2 * kv_row]
        ok_ = np.full((S, words), 0x33333333, dtype=np.uint32)
        ov_ = ok_.copy()
        oracle.cq_append(key, val, ok_, ov_, slots, num_kv_heads=Hk, head_size=D, max_t=max_t)
        dbuf = torch.from_numpy(buf).cuda()
        kc, vc = _dev(np.full_like(ok_, 0x33333333)), _dev(np.full_like(ok_, 0x33333333))
        pk.pa_q8c_append(dbuf[:, offset:offset + kv_row], dbuf[:, offset + kv_row:offset + 2 * kv_row], kc, vc,
                         _dev(slots), num_kv_heads=Hk, head_size=D, max_t=max_t)
        assert np.array_equal(_host(kc), ok_), f"offset {offset}"
        assert np.array_equal(_host(vc), ov_), f"offset {offset}"
    bad = slots.copy()
    bad[0] = S * max_t + 2
    device_status(clear=True)
    kc = _dev(np.zeros((S, words), dtype=np.uint32))
    pk.pa_q8c_append(torch.from_numpy(np.ascontiguousarray(key)).cuda(),
                     torch.from_numpy(np.ascontiguousarray(val)).cuda(), kc, _dev(np.zeros((S, words), np.uint32)),
                     _dev(bad), num_kv_heads=Hk, head_size=D, max_t=max_t)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_SLOT


def _case(S, H, Hk, D, max_t, lens, seed):
    """Caches written by the oracle (poison elsewhere) and the same words on the device."""
    import oracle
    rng = np.random.default_rng(seed)
    slots = np.array([s * max_t + t for s, c in enumerate(lens) for t in range(c)], dtype=np.uint32)
    T = slots.size
    key = rng.standard_normal((T, Hk * D)).astype(np.float32)
    val = rng.standard_normal((T, Hk * D)).astype(np.float32)
    words = oracle.cq_seq_words(max_t, Hk, D)
    kc = np.full((S, words), 0xFFFFFFFF, dtype=np.uint32)
    vc = kc.copy()
    if T:
        oracle.cq_append(key, val, kc, vc, slots, num_kv_heads=Hk, head_size=D, max_t=max_t)
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    return kc, vc, q, key, val, slots


def _gpu(kc, vc, q, cl, Hk, max_t, scale, pt=0):
    import torch
    import int8_paged_kv_gb300 as pk
    qd = torch.from_numpy(q).cuda()
    out = torch.full_like(qd, float("nan"))
    pk.pa_q8c_decode(out, qd, _dev(kc), _dev(vc), _dev(cl), num_kv_heads=Hk, max_t=max_t, scale=scale,
                     partition_tokens=pt)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("H,Hk,D", [(8, 2, 128), (32, 8, 128), (16, 1, 256), (4, 4, 256), (12, 3, 128)])
def test_decode_shapes_and_partitions(H, Hk, D):
    import oracle
    from tests.gpu_helpers import assert_close, device_status
    lens = [1, 31, 33, 700, 0, 129, 1000, 64]
    max_t = 1024
    kc, vc, q, *_ = _case(len(lens), H, Hk, D, max_t, lens, seed=H + D)
    cl = np.array(lens, dtype=np.uint32)
    scale = float(np.float32(D ** -0.5))
    want = oracle.cq_decode(q, kc, vc, cl, num_kv_heads=Hk, max_t=max_t, scale=scale)
    for pt in (0, 128, 256):
        got = _gpu(kc, vc, q, cl, Hk, max_t, scale, pt)
        assert_close(got, want, f"H {H} Hk {Hk} D {D} pt {pt}")
        assert np.all(got[4] == 0.0)
    assert device_status() == 0


def test_clamp_and_gpu_append_then_decode():
    """Contexts beyond max_t are clamped; the library's own append writes the
    oracle's words (same fill elsewhere), so the decode sees the same cache."""
    import torch
    import oracle
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import assert_close
    S, H, Hk, D, max_t = 3, 8, 2, 128, 300
    lens = [300, 5, 177]
    kc, vc, q, key, val, slots = _case(S, H, Hk, D, max_t, lens, seed=3)
    gk, gv = _dev(np.full_like(kc, 0xFFFFFFFF)), _dev(np.full_like(vc, 0xFFFFFFFF))
    pk.pa_q8c_append(torch.from_numpy(key).cuda(), torch.from_numpy(val).cuda(), gk, gv, _dev(slots),
                     num_kv_heads=Hk, head_size=D, max_t=max_t)
    assert np.array_equal(_host(gk), kc) and np.array_equal(_host(gv), vc)
    cl = np.array([10_000, 5, 177], dtype=np.uint32)
    want = oracle.cq_decode(q, kc, vc, cl, num_kv_heads=Hk, max_t=max_t, scale=0.09)
    assert_close(_gpu(kc, vc, q, cl, Hk, max_t, 0.09), want, "clamped")


def test_llama8b_contexts_all_rows():
    """The 64-sequence workload's contexts and queries in a contiguous cache
    (max_t = 4096); every row against the oracle."""
    import oracle
    from tests.gpu_helpers import assert_close, device_status
    w = wl.build("llama8b", with_append=False)
    cfg = w.cfg
    S, H, Hk, D, max_t = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.max_context
    slots = np.concatenate([s * max_t + np.arange(int(c)) for s, c in enumerate(w.context_lens)]).astype(np.uint32)
    rows_k = w.key.reshape(w.key.shape[0], -1)
    rows_v = w.value.reshape(w.value.shape[0], -1)
    words = oracle.cq_seq_words(max_t, Hk, D)
    kc = np.full((S, words), 0xFFFFFFFF, dtype=np.uint32)
    vc = kc.copy()
    oracle.cq_append(rows_k, rows_v, kc, vc, slots, num_kv_heads=Hk, head_size=D, max_t=max_t)
    w.key = w.value = None
    want = oracle.cq_decode(w.q, kc, vc, w.context_lens, num_kv_heads=Hk, max_t=max_t, scale=w.scale)
    got = _gpu(kc, vc, w.q, w.context_lens, Hk, max_t, w.scale)
    assert_close(got, want, "llama8b contiguous")
    assert device_status() == 0


def test_many_sequences_three_per_sm_build():
    """Enough (sequence, kv head) work for four or more waves of three CTAs
    per SM: the plan takes the head-size-128 kernel's three-per-SM build
    (the cases above, with few sequences, take the two-per-SM one)."""
    import torch
    import oracle
    from tests.gpu_helpers import assert_close, device_status
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hk, H, D, max_t = 8, 16, 128, 128
    S = (4 * 3 * sms + Hk - 1) // Hk + 16               # one partition each (max_t <= 8192)
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(0, max_t + 1, size=S)]
    lens[:4] = [0, 1, max_t, 33]
    kc, vc, q, *_ = _case(S, H, Hk, D, max_t, lens, seed=12)
    cl = np.array(lens, dtype=np.uint32)
    scale = float(np.float32(D ** -0.5))
    want = oracle.cq_decode(q, kc, vc, cl, num_kv_heads=Hk, max_t=max_t, scale=scale)
    got = _gpu(kc, vc, q, cl, Hk, max_t, scale)
    assert_close(got, want, f"S {S}")
    assert np.all(got[0] == 0.0)
    assert device_status() == 0
