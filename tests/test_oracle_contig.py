"""Pins of the contiguous-cache oracle (oracle.cq_append / oracle.cq_decode)
against things other than itself: a numpy float32 group quantiser and numpy
indexing for the layout, a dense numpy attention over a numpy dequantisation,
a one-token closed form, and metamorphic invariances (repeated kv heads,
context clamp)."""
import numpy as np
import pytest

import oracle

PAD = 0xFFFFFFFF


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _np_group_quant(x):
    """numpy float32 steps for one 32-value group: (8 code words, scale word)."""
    x = x.astype(np.float32)
    amax = np.float32(np.max(np.abs(x)))
    inv = np.float32(127) / amax if amax > 0 else np.float32(0)
    t = (x * inv).astype(np.float32).astype(np.float64)
    codes = np.clip(np.sign(t) * np.floor(np.abs(t) + 0.5), -127, 127).astype(np.int8)
    scale = (amax / np.float32(127)) if amax > 0 else np.float32(1.0)
    return codes.view(np.uint32), np.float32(scale).view(np.uint32)


def _np_cache(rows, slots, S, Hk, D, max_t, fill=0x5A5A5A5A):
    """Expected cache words from numpy: per sequence [max_t][kv_row/4] code
    words then [max_t][kv_row/32] scales."""
    kv_row = Hk * D
    cw, sw = max_t * kv_row // 4, max_t * kv_row // 32
    cache = np.full((S, cw + sw), fill, dtype=np.uint32)
    for i, slot in enumerate(slots):
        if slot == PAD:
            continue
        s, t = divmod(int(slot), max_t)
        for j in range(kv_row // 32):
            words, scale = _np_group_quant(rows[i, 32 * j:32 * j + 32])
            cache[s, t * kv_row // 4 + 8 * j: t * kv_row // 4 + 8 * j + 8] = words
            cache[s, cw + t * kv_row // 32 + j] = scale
    return cache


def _rows(rng, T, kv_row):
    x = rng.standard_normal((T, kv_row)).astype(np.float32)
    x[1] *= np.float32(50.0)                       # a wide row
    x[2, :32] = 0.0                                # an all-zero group: scale word 1.0
    x[3, 5] *= np.float32(40.0)                    # an outlier in one group
    x[4] = (rng.integers(-254, 255, kv_row) / 128.0).astype(np.float32)   # half-way products
    return x


@pytest.mark.parametrize("Hk,D", [(2, 128), (1, 256), (4, 64)])
def test_append_matches_numpy_groups_and_layout(Hk, D):
    rng = np.random.default_rng(D + Hk)
    S, max_t, T = 3, 20, 24
    kv_row = Hk * D
    fused = rng.standard_normal((T, 2 * kv_row + 8)).astype(np.float32)
    fused[:, :kv_row] = _rows(rng, T, kv_row)
    key, value = fused[:, :kv_row], fused[:, kv_row:2 * kv_row]          # strided row views
    slots = rng.choice(S * max_t, size=T, replace=False).astype(np.uint32)
    slots[[6, 11]] = PAD
    sw = oracle.cq_seq_words(max_t, Hk, D)
    kc = np.full((S, sw), 0x5A5A5A5A, dtype=np.uint32)
    vc = kc.copy()
    oracle.cq_append(key, value, kc, vc, slots, num_kv_heads=Hk, head_size=D, max_t=max_t)
    assert np.array_equal(kc, _np_cache(np.ascontiguousarray(key), slots, S, Hk, D, max_t))
    assert np.array_equal(vc, _np_cache(np.ascontiguousarray(value), slots, S, Hk, D, max_t))


def _case(S, H, Hk, D, max_t, lens, seed):
    rng = np.random.default_rng(seed)
    kv_row = Hk * D
    slots, rows = [], []
    for s, c in enumerate(lens):
        for t in range(c):
            slots.append(s * max_t + t)
    T = len(slots)
    key = rng.standard_normal((T, kv_row)).astype(np.float32)
    val = rng.standard_normal((T, kv_row)).astype(np.float32)
    sw = oracle.cq_seq_words(max_t, Hk, D)
    kc = np.zeros((S, sw), dtype=np.uint32)
    vc = kc.copy()
    oracle.cq_append(key, val, kc, vc, np.array(slots, dtype=np.uint32), num_kv_heads=Hk, head_size=D,
                     max_t=max_t)
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    return kc, vc, q, key, val


def _np_dequant(cache, S, Hk, D, max_t):
    """numpy: [S][max_t][kv_row] float64 values = code * group scale."""
    kv_row = Hk * D
    cw = max_t * kv_row // 4
    codes = cache[:, :cw].copy().view(np.int8).reshape(S, max_t, kv_row).astype(np.float64)
    scales = cache[:, cw:].copy().view(np.float32).reshape(S, max_t, kv_row // 32).astype(np.float64)
    return codes * np.repeat(scales, 32, axis=2)


@pytest.mark.parametrize("H,Hk,D", [(8, 2, 128), (4, 1, 256), (8, 8, 64)])
def test_decode_vs_dense_numpy(H, Hk, D):
    S, max_t = 4, 70
    lens = [1, 33, 70, 0]
    kc, vc, q, *_ = _case(S, H, Hk, D, max_t, lens, seed=H * D)
    scale = float(np.float32(D ** -0.5))
    got = oracle.cq_decode(q, kc, vc, np.array(lens, np.uint32), num_kv_heads=Hk, max_t=max_t, scale=scale)
    K, V = _np_dequant(kc, S, Hk, D, max_t), _np_dequant(vc, S, Hk, D, max_t)
    r = H // Hk
    for s, c in enumerate(lens):
        for h in range(H):
            g = h // r
            if c == 0:
                assert np.all(got[s, h] == 0.0)
                continue
            Ks, Vs = K[s, :c, g * D:(g + 1) * D], V[s, :c, g * D:(g + 1) * D]
            z = scale * (Ks @ q[s, h].astype(np.float64))
            p = np.exp(z - z.max())
            assert np.allclose(got[s, h], (p / p.sum()) @ Vs, rtol=1e-12, atol=1e-12)


def test_single_position_is_its_value_row():
    S, H, Hk, D, max_t = 2, 4, 2, 128, 8
    kc, vc, q, *_ = _case(S, H, Hk, D, max_t, [1, 1], seed=3)
    got = oracle.cq_decode(q, kc, vc, np.array([1, 1], np.uint32), num_kv_heads=Hk, max_t=max_t, scale=0.1)
    V = _np_dequant(vc, S, Hk, D, max_t)
    for s in range(S):
        for h in range(H):
            g = h // 2
            assert np.array_equal(got[s, h], V[s, 0, g * D:(g + 1) * D])


def test_repeated_kv_heads_and_clamp():
    """A cache whose kv heads are repeated r times (numpy) decoded as MHA gives
    the same bits as the GQA decode; a context beyond max_t is clamped."""
    S, H, Hk, D, max_t = 2, 8, 2, 64, 40
    lens = [40, 17]
    kc, vc, q, *_ = _case(S, H, Hk, D, max_t, lens, seed=5)
    cl = np.array(lens, np.uint32)
    base = oracle.cq_decode(q, kc, vc, cl, num_kv_heads=Hk, max_t=max_t, scale=0.2)

    def repeat(cache):
        kv_row = Hk * D
        cw = max_t * kv_row // 4
        codes = cache[:, :cw].reshape(S, max_t, Hk, D // 4)
        scales = cache[:, cw:].reshape(S, max_t, Hk, D // 32)
        r = H // Hk
        c2 = np.repeat(codes, r, axis=2).reshape(S, -1)
        s2 = np.repeat(scales, r, axis=2).reshape(S, -1)
        return np.ascontiguousarray(np.concatenate([c2, s2], axis=1))
    mha = oracle.cq_decode(q, repeat(kc), repeat(vc), cl, num_kv_heads=H, max_t=max_t, scale=0.2)
    assert np.array_equal(base, mha)
    far = oracle.cq_decode(q, kc, vc, np.array([10_000, 17], np.uint32), num_kv_heads=Hk, max_t=max_t,
                           scale=0.2)
    assert np.array_equal(far, base)
