"""Pins of the f32-cache oracle (oracle.reshape_and_cache_f32 /
oracle.decode_f32) against things other than itself: numpy indexing for the
layout, a dense numpy attention, closed forms, the q8 oracle on a cache
holding the same (dequantised) values, and metamorphic invariances."""
import numpy as np
import pytest

import oracle

PAD = 0xFFFFFFFF


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _paged(S, Hk, D, B, lens, seed, Nb=None, dist=1.0):
    """An f32 paged cache (poisoned with NaN) holding seeded rows of each
    sequence's context, written by the oracle's f32 writer."""
    rng = np.random.default_rng(seed)
    nblk = [-(-int(c) // B) for c in lens]
    Nb = Nb or max(1, max(nblk))
    pool = sum(nblk) + 2
    perm = rng.permutation(pool).astype(np.uint32)
    bt = np.full((S, Nb), PAD, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += nblk[s]
    T = int(sum(lens))
    key = (rng.standard_normal((T, Hk, D)) * dist).astype(np.float32)
    val = (rng.standard_normal((T, Hk, D)) * dist).astype(np.float32)
    slots = np.concatenate([bt[s, np.arange(c) // B].astype(np.int64) * B + np.arange(c) % B
                            for s, c in enumerate(lens) if c > 0] or [np.zeros(0, np.int64)]).astype(np.uint32)
    kc = np.full((pool, Hk, B, D), np.nan, dtype=np.float32)
    vc = kc.copy()
    oracle.reshape_and_cache_f32(key, val, kc, vc, slots, num_kv_heads=Hk, head_size=D, block_size=B)
    return bt, kc, vc, key, val, slots


def _dense(q, kc, vc, bt, lens, Hk, B, scale, cap=None):
    """numpy: gather each sequence's K/V by its block table, softmax in fp64."""
    S, H, D = q.shape
    r = H // Hk
    out = np.zeros((S, H, D))
    for s in range(S):
        c = int(lens[s]) if cap is None else min(int(lens[s]), cap)
        if c == 0:
            continue
        t = np.arange(c)
        blocks = bt[s, t // B].astype(np.int64)
        for h in range(H):
            K = kc[blocks, h // r, t % B].astype(np.float64)
            V = vc[blocks, h // r, t % B].astype(np.float64)
            z = scale * (K @ q[s, h].astype(np.float64))
            p = np.exp(z - z.max())
            out[s, h] = (p / p.sum()) @ V
    return out


def test_writer_layout_pad_and_strides():
    rng = np.random.default_rng(1)
    T, Hk, D, B, nb = 40, 3, 64, 8, 12
    fused = rng.standard_normal((T, 2 * Hk * D + 4)).astype(np.float32)
    key, val = fused[:, :Hk * D], fused[:, Hk * D:2 * Hk * D]        # strided 2-D row views
    slots = rng.choice(nb * B, size=T, replace=False).astype(np.uint32)
    slots[[3, 17]] = PAD
    kc = np.full((nb, Hk, B, D), -7.0, dtype=np.float32)
    vc = kc.copy()
    oracle.reshape_and_cache_f32(key, val, kc, vc, slots, num_kv_heads=Hk, head_size=D, block_size=B)
    want_k = np.full_like(kc, -7.0)
    want_v = want_k.copy()
    live = slots != PAD
    sl = slots[live].astype(np.int64)
    want_k.reshape(nb, Hk, B, D)[sl // B, :, sl % B] = key[live].reshape(-1, Hk, D)
    want_v.reshape(nb, Hk, B, D)[sl // B, :, sl % B] = val[live].reshape(-1, Hk, D)
    assert np.array_equal(kc.view(np.uint32), want_k.view(np.uint32))
    assert np.array_equal(vc.view(np.uint32), want_v.view(np.uint32))


@pytest.mark.parametrize("H,Hk,D,B", [(8, 2, 64, 16), (4, 4, 128, 8), (16, 1, 256, 32)])
def test_decode_vs_dense_numpy(H, Hk, D, B):
    lens = [1, 37, 100, 0, 2 * B]
    bt, kc, vc, *_ = _paged(len(lens), Hk, D, B, lens, seed=H + D)
    q = np.random.default_rng(D).standard_normal((len(lens), H, D)).astype(np.float32)
    scale = float(np.float32(D ** -0.5))
    got = oracle.decode_f32(q, kc, vc, bt, np.array(lens, np.uint32), num_kv_heads=Hk, block_size=B,
                            scale=scale)
    want = _dense(q, kc, vc, bt, lens, Hk, B, scale)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.all(got[3] == 0.0)                         # empty context


def test_single_token_is_its_value_row():
    bt, kc, vc, key, val, _ = _paged(2, 2, 64, 16, [1, 1], seed=3)
    q = np.random.default_rng(3).standard_normal((2, 4, 64)).astype(np.float32)
    got = oracle.decode_f32(q, kc, vc, bt, np.array([1, 1], np.uint32), num_kv_heads=2, block_size=16,
                            scale=0.125)
    for s in range(2):
        for h in range(4):
            assert np.array_equal(got[s, h], val[s, h // 2].astype(np.float64))


def test_equal_keys_give_the_mean_of_values():
    B, D, c = 16, 64, 50
    bt, kc, vc, *_ = _paged(1, 1, D, B, [c], seed=4)
    kc[...] = kc[int(bt[0, 0]), 0, 0]                    # every token the same key
    q = np.random.default_rng(4).standard_normal((1, 2, D)).astype(np.float32)
    got = oracle.decode_f32(q, kc, vc, bt, np.array([c], np.uint32), num_kv_heads=1, block_size=B,
                            scale=0.3)
    t = np.arange(c)
    mean = vc[bt[0, t // B].astype(np.int64), 0, t % B].astype(np.float64).mean(axis=0)
    assert np.allclose(got[0, 0], mean, rtol=1e-13, atol=1e-13)
    assert np.allclose(got[0, 1], mean, rtol=1e-13, atol=1e-13)


def test_matches_the_q8_oracle_on_a_dequantised_cache():
    """The q8 oracle decodes code * scale exactly; an f32 cache holding
    fl32(code * scale) gives the same outputs up to that one rounding."""
    S, H, Hk, D, B = 3, 8, 2, 128, 16
    lens = [5, 64, 133]
    rng = np.random.default_rng(5)
    nblk = [-(-c // B) for c in lens]
    pool = sum(nblk)
    perm = rng.permutation(pool).astype(np.uint32)
    bt = np.full((S, max(nblk)), PAD, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += nblk[s]
    T = sum(lens)
    key = rng.standard_normal((T, Hk, D)).astype(np.float32)
    val = rng.standard_normal((T, Hk, D)).astype(np.float32)
    slots = np.concatenate([bt[s, np.arange(c) // B].astype(np.int64) * B + np.arange(c) % B
                            for s, c in enumerate(lens)]).astype(np.uint32)
    W = D // 4 + 1
    qk = np.zeros((pool, Hk, B, W), dtype=np.uint32)
    qv = qk.copy()
    oracle.reshape_and_cache(key, val, qk, qv, slots, num_kv_heads=Hk, head_size=D, block_size=B)

    def dequant(cache):
        codes = cache[..., :D // 4].copy().view(np.int8).reshape(pool, Hk, B, D).astype(np.float64)
        scale = cache[..., D // 4].copy().view(np.float32).astype(np.float64)
        return (codes * scale[..., None]).astype(np.float32)
    fk, fv = dequant(qk), dequant(qv)
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    cl = np.array(lens, np.uint32)
    a = oracle.decode_f32(q, fk, fv, bt, cl, num_kv_heads=Hk, block_size=B, scale=0.0883883)
    b = oracle.decode(q, qk, qv, bt, cl, num_kv_heads=Hk, block_size=B, scale=0.0883883)
    assert np.allclose(a, b, rtol=1e-6, atol=1e-7)


def test_gqa_is_mha_over_repeated_kv_heads_and_block_order_is_irrelevant():
    S, H, Hk, D, B = 2, 8, 2, 64, 8
    lens = [30, 17]
    bt, kc, vc, *_ = _paged(S, Hk, D, B, lens, seed=6)
    q = np.random.default_rng(6).standard_normal((S, H, D)).astype(np.float32)
    cl = np.array(lens, np.uint32)
    base = oracle.decode_f32(q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=0.2)
    rep_k = np.ascontiguousarray(np.repeat(kc, H // Hk, axis=1))
    rep_v = np.ascontiguousarray(np.repeat(vc, H // Hk, axis=1))
    mha = oracle.decode_f32(q, rep_k, rep_v, bt, cl, num_kv_heads=H, block_size=B, scale=0.2)
    assert np.array_equal(base, mha)
    # move every block to a new physical id: same bits out
    perm = np.random.default_rng(7).permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(bt == PAD, bt, perm[np.minimum(bt, kc.shape[0] - 1)]).astype(np.uint32)
    assert np.array_equal(oracle.decode_f32(q, kc2, vc2, bt2, cl, num_kv_heads=Hk, block_size=B,
                                            scale=0.2), base)


def test_context_clamp():
    S, Hk, D, B = 1, 1, 64, 16
    bt, kc, vc, *_ = _paged(S, Hk, D, B, [48], seed=8)
    q = np.random.default_rng(8).standard_normal((1, 2, D)).astype(np.float32)
    a = oracle.decode_f32(q, kc, vc, bt, np.array([10_000], np.uint32), num_kv_heads=1, block_size=B,
                          scale=0.1)
    b = oracle.decode_f32(q, kc, vc, bt, np.array([48], np.uint32), num_kv_heads=1, block_size=B,
                          scale=0.1)
    assert np.array_equal(a, b)
