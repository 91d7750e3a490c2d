"""Test-side readers of the packed cache, written from the layout alone.

The cache layout is the one in the header comments of
"paged_attn_q8.comp" / "reshape_and_cache_q8.comp": u32 words
[num_blocks, num_kv_heads, block_size, head_size/4 + 1]; the first
head_size/4 words of a token vector hold the int8 codes (4 per word, code
l in byte l, little endian), the last word the f32 scale bits.  These
helpers use numpy views only, so they check the oracle (and the kernels)
through a route that shares nothing with either.
"""
import numpy as np

PAD = 0xFFFFFFFF


def split_cache(cache: np.ndarray, head_size: int):
    """(codes int8 [..., head_size], scales f32 [...]) of a u32 cache
    whose last axis is head_size/4 + 1 words."""
    W = head_size // 4 + 1
    assert cache.shape[-1] == W
    words = np.ascontiguousarray(cache)
    code_words = np.ascontiguousarray(words[..., : head_size // 4])
    codes = code_words.view("<i1").reshape(*words.shape[:-1], head_size)
    scales = np.ascontiguousarray(words[..., head_size // 4]).view("<f4")
    return codes, scales


def dequant_cache(cache: np.ndarray, head_size: int) -> np.ndarray:
    codes, scales = split_cache(cache, head_size)
    return codes.astype(np.float64) * scales.astype(np.float64)[..., None]


def dense_context(cache4: np.ndarray, block_tables: np.ndarray, s: int, c: int,
                  head_size: int) -> np.ndarray:
    """Dequantised [c, Hk, D] K or V of sequence s, gathered through its block table."""
    B = cache4.shape[2]
    deq = dequant_cache(cache4, head_size)                 # [nb, Hk, B, D]
    t = np.arange(c)
    blocks = block_tables[s, t // B].astype(np.int64)
    return deq[blocks, :, t % B, :]                         # [c, Hk, D]


def tolerance_ok(got, want, atol=1e-5, rtol=1e-4):
    """Elementwise |got - want| <= atol + rtol * |want| (want from the oracle)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = ~(err <= bound)
    return (not bad.any()), float(np.max(err / bound)) if err.size else 0.0, int(bad.sum())


def random_paged_case(rng, *, S, H, Hk, D, B, lens, pool_extra=3, dist="normal"):
    """A small random paged setup built by the oracle writer: returns dict."""
    import oracle
    Nb = max(1, max(-(-int(c) // B) for c in lens))
    nblk = [-(-int(c) // B) for c in lens]
    pool = sum(nblk) + pool_extra
    perm = rng.permutation(pool).astype(np.uint32)
    bt = np.full((S, Nb), PAD, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt[s, : nblk[s]] = perm[pos: pos + nblk[s]]
        pos += nblk[s]
    W = D // 4 + 1
    kc = np.full((pool, Hk, B, W), 0xA5A5A5A5, dtype=np.uint32)
    vc = np.full((pool, Hk, B, W), 0xA5A5A5A5, dtype=np.uint32)
    rows_k, rows_v, slots = [], [], []
    for s in range(S):
        c = int(lens[s])
        if dist == "normal":
            k = rng.standard_normal((c, Hk, D)).astype(np.float32)
            v = rng.standard_normal((c, Hk, D)).astype(np.float32)
        else:
            k = rng.uniform(-3, 3, (c, Hk, D)).astype(np.float32)
            v = rng.uniform(-3, 3, (c, Hk, D)).astype(np.float32)
        t = np.arange(c)
        rows_k.append(k)
        rows_v.append(v)
        slots.append((bt[s, t // B].astype(np.int64) * B + t % B).astype(np.uint32))
    key = np.concatenate(rows_k) if rows_k else np.zeros((0, Hk, D), np.float32)
    val = np.concatenate(rows_v) if rows_v else np.zeros((0, Hk, D), np.float32)
    sm = np.concatenate(slots) if slots else np.zeros(0, np.uint32)
    oracle.reshape_and_cache(np.ascontiguousarray(key), np.ascontiguousarray(val), kc, vc, sm,
                             num_kv_heads=Hk, head_size=D, block_size=B)
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    cl = np.asarray(lens, dtype=np.uint32)
    return dict(q=q, kc=kc, vc=vc, bt=bt, cl=cl, key=key, value=val, slots=sm,
                S=S, H=H, Hk=Hk, D=D, B=B, Nb=Nb, pool=pool)
