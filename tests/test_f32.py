"""The f32-cache variant on the GPU against its oracle: the writer bit for
bit (oracle.reshape_and_cache_f32), the decode within
|gpu - oracle| <= 1e-5 + 1e-4 |oracle| (oracle.decode_f32), on GQA ratios,
head sizes, block sizes, partition sizes, ragged and empty contexts, a bad
block id, and the 64- and 256-sequence workloads."""
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


def _case(S, H, Hk, D, B, lens, seed):
    """f32 caches written by the oracle (NaN elsewhere) and by the GPU writer
    (checked equal), block tables over a shuffled pool, seeded q."""
    import torch
    import int8_paged_kv_gb300 as pk
    import oracle
    from tests.gpu_helpers import dev_u32
    rng = np.random.default_rng(seed)
    nblk = [-(-int(c) // B) for c in lens]
    Nb = max(1, max(nblk))
    pool = sum(nblk) + 3
    perm = rng.permutation(pool).astype(np.uint32)
    bt = np.full((S, Nb), PAD, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += nblk[s]
    T = int(sum(lens))
    key = rng.standard_normal((T, Hk, D)).astype(np.float32)
    val = rng.standard_normal((T, Hk, D)).astype(np.float32)
    slots = np.concatenate([bt[s, np.arange(c) // B].astype(np.int64) * B + np.arange(c) % B
                            for s, c in enumerate(lens) if c > 0] or [np.zeros(0, np.int64)]).astype(np.uint32)
    ok_ = np.full((pool, Hk, B, D), np.nan, dtype=np.float32)
    ov_ = ok_.copy()
    oracle.reshape_and_cache_f32(key, val, ok_, ov_, slots, num_kv_heads=Hk, head_size=D, block_size=B)
    kc = torch.full(ok_.shape, float("nan"), device="cuda")
    vc = torch.full(ok_.shape, float("nan"), device="cuda")
    if T:
        pk.pa_f32_reshape_and_cache(torch.from_numpy(key.reshape(T, -1)).cuda(),
                                    torch.from_numpy(val.reshape(T, -1)).cuda(), kc, vc, dev_u32(slots),
                                    num_kv_heads=Hk, head_size=D, block_size=B)
    assert np.array_equal(kc.cpu().numpy().view(np.uint32), ok_.view(np.uint32))
    assert np.array_equal(vc.cpu().numpy().view(np.uint32), ov_.view(np.uint32))
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    return dict(bt=bt, cl=np.asarray(lens, np.uint32), ok=ok_, ov=ov_, kc=kc, vc=vc, q=q, Hk=Hk, B=B,
                scale=float(np.float32(D ** -0.5)), pool=pool)


def _gpu(c, *, pt=0, cl=None, bt=None):
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32
    q = torch.from_numpy(c["q"]).cuda()
    out = torch.full_like(q, float("nan"))
    pk.pa_f32_decode(out, q, c["kc"], c["vc"], dev_u32(c["bt"] if bt is None else bt),
                     dev_u32(c["cl"] if cl is None else cl), num_kv_heads=c["Hk"], block_size=c["B"],
                     scale=c["scale"], num_blocks=c["pool"], partition_tokens=pt)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def _oracle(c, rows=None, cl=None):
    import oracle
    return oracle.decode_f32(c["q"], c["ok"], c["ov"], c["bt"], c["cl"] if cl is None else cl,
                             num_kv_heads=c["Hk"], block_size=c["B"], scale=c["scale"], rows=rows)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_writer_strided_unaligned_and_pad(D):
    """Rows that are column slices of fused rows, on and off 16-byte
    alignment, PAD slots and a slot out of range (skipped, flagged)."""
    import torch
    import int8_paged_kv_gb300 as pk
    import oracle
    from tests.gpu_helpers import dev_u32, device_status
    rng = np.random.default_rng(D)
    T, Hk, B, nb = 50, 3, 16, 10
    slots = rng.choice(nb * B, size=T, replace=False).astype(np.uint32)
    slots[[4, 20]] = PAD
    for offset in (0, 1):
        buf = rng.standard_normal((T, 2 * Hk * D + 5)).astype(np.float32)
        key = buf[:, offset:offset + Hk * D]
        val = buf[:, offset + Hk * D:offset + 2 * Hk * D]
        ok_ = np.full((nb, Hk, B, D), -3.0, dtype=np.float32)
        ov_ = ok_.copy()
        oracle.reshape_and_cache_f32(key, val, ok_, ov_, slots, num_kv_heads=Hk, head_size=D, block_size=B)
        dbuf = torch.from_numpy(buf).cuda()
        kc = torch.full(ok_.shape, -3.0, device="cuda")
        vc = torch.full(ok_.shape, -3.0, device="cuda")
        bad = slots.copy()
        bad[7] = nb * B + 3                                  # out of range: skipped, flagged
        want_k, want_v = ok_.copy(), ov_.copy()
        s7 = int(slots[7])
        want_k[s7 // B, :, s7 % B] = -3.0
        want_v[s7 // B, :, s7 % B] = -3.0
        device_status(clear=True)
        pk.pa_f32_reshape_and_cache(dbuf[:, offset:offset + Hk * D], dbuf[:, offset + Hk * D:offset + 2 * Hk * D],
                                    kc, vc, dev_u32(bad), num_kv_heads=Hk, head_size=D, block_size=B)
        assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_SLOT
        assert np.array_equal(kc.cpu().numpy().view(np.uint32), want_k.view(np.uint32)), f"offset {offset}"
        assert np.array_equal(vc.cpu().numpy().view(np.uint32), want_v.view(np.uint32)), f"offset {offset}"


@pytest.mark.parametrize("H,Hk,D,B", [(8, 2, 64, 16), (32, 8, 128, 16), (16, 1, 256, 32), (4, 4, 128, 8),
                                      (64, 8, 128, 64), (12, 3, 128, 128), (24, 2, 64, 256)])
def test_decode_shapes_and_partitions(H, Hk, D, B):
    from tests.gpu_helpers import assert_close, device_status
    lens = [1, 31, 33, 700, 0, 129, 2 * B, 1000]
    c = _case(len(lens), H, Hk, D, B, lens, seed=H + Hk + D + B)
    want = _oracle(c)
    for pt in (0, 128, 256):
        got = _gpu(c, pt=pt)
        assert_close(got, want, f"H {H} Hk {Hk} D {D} B {B} pt {pt}")
        assert np.all(got[4] == 0.0)
    assert device_status() == 0


def test_clamped_context_and_bad_block():
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import assert_close, device_status
    lens = [64, 208, 50]
    c = _case(3, 8, 2, 128, 16, lens, seed=5)
    cl = np.array([64, 10_000, 50], dtype=np.uint32)        # sequence 1 clamps to 208
    assert_close(_gpu(c, cl=cl), _oracle(c, cl=cl), "clamp")
    bt = c["bt"].copy()
    bt[1, 2] = 1 << 30                                      # inside the context, out of the pool
    device_status(clear=True)
    got = _gpu(c, bt=bt)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_BLOCK
    want = _oracle(c)
    assert_close(got[[0, 2]], want[[0, 2]], "untouched sequences")


def _workload_case(name):
    """A workload's context rows in f32 caches (GPU writer; oracle writer for
    the oracle's copy, checked equal)."""
    import torch
    import int8_paged_kv_gb300 as pk
    import oracle
    from tests.gpu_helpers import dev_u32
    w = wl.build(name, with_append=False)
    cfg = w.cfg
    Hk, D, B = cfg.num_kv_heads, cfg.head_size, cfg.block_size
    shape = (w.num_blocks, Hk, B, D)
    ok_ = np.full(shape, np.nan, dtype=np.float32)
    ov_ = ok_.copy()
    oracle.reshape_and_cache_f32(w.key, w.value, ok_, ov_, w.slot_mapping, num_kv_heads=Hk, head_size=D,
                                 block_size=B)
    kc = torch.full(shape, float("nan"), device="cuda")
    vc = torch.full(shape, float("nan"), device="cuda")
    T = w.key.shape[0]
    for i in range(0, T, 1 << 18):
        pk.pa_f32_reshape_and_cache(torch.from_numpy(w.key[i:i + (1 << 18)].reshape(-1, Hk * D)).cuda(),
                                    torch.from_numpy(w.value[i:i + (1 << 18)].reshape(-1, Hk * D)).cuda(),
                                    kc, vc, dev_u32(w.slot_mapping[i:i + (1 << 18)]), num_kv_heads=Hk,
                                    head_size=D, block_size=B)
    w.key = w.value = None
    assert np.array_equal(kc.cpu().numpy().view(np.uint32), ok_.view(np.uint32))
    assert np.array_equal(vc.cpu().numpy().view(np.uint32), ov_.view(np.uint32))
    return dict(bt=w.block_tables, cl=w.context_lens, ok=ok_, ov=ov_, kc=kc, vc=vc, q=w.q, Hk=Hk, B=B,
                scale=w.scale, pool=w.num_blocks)


def test_llama8b_all_rows():
    from tests.gpu_helpers import assert_close, device_status
    c = _workload_case("llama8b")
    assert_close(_gpu(c), _oracle(c), "llama8b f32")
    assert device_status() == 0


def test_large_batch_sampled_rows():
    from tests.gpu_helpers import assert_close, device_status
    c = _workload_case("large")
    got = _gpu(c)
    rng = np.random.default_rng(3)
    S, H = c["q"].shape[:2]
    picks = sorted({(int(rng.integers(S)), int(rng.integers(H))) for _ in range(120)} |
                   {(int(np.argmax(c["cl"])), 0), (int(np.argmin(c["cl"])), H - 1)})
    rows = np.array(picks, dtype=np.int32)
    assert_close(got[rows[:, 0], rows[:, 1]], _oracle(c, rows=rows), "large f32")
    assert np.all(np.isfinite(got))
    assert device_status() == 0
