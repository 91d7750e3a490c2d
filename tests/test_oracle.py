"""Pins for the CPU oracle, checked against facts fixed outside the oracle.

Nothing here retypes the oracle's formulas.  The writer is pinned by
hand-derived golden words, by numpy's IEEE f32 arithmetic (a library route to
the same f32 operations), by exact rational arithmetic (fractions), and by
invariants the writer page states.  The decode is pinned by closed forms,
by a dense numpy / scipy brute force built from numpy views of the cache,
by metamorphic relations and by the log-sum-exp merge of partials.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from tests.helpers import PAD, dense_context, dequant_cache, random_paged_case, split_cache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "writer_vectors.txt")


def _golden_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key == "x":
                cur["x"] = np.array([float(v) for v in vals], dtype=np.float32)
            elif key == "words":
                cur["words"] = np.array([int(v, 16) for v in vals], dtype=np.uint32)
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_writer_golden_words(oracle_lib, case):
    got = oracle.quantize_vector(case["x"])
    assert [hex(w) for w in got] == [hex(w) for w in case["words"]]


def _round_half_away(t: np.ndarray) -> np.ndarray:
    t = t.astype(np.float64)
    return np.sign(t) * np.floor(np.abs(t) + 0.5)


def _vectors(rng, n, D):
    """Assorted vectors: normal, heavy tails, outlier channels, tiny and huge
    magnitudes, exact multiples of a power of two (many half-way products),
    and all-zero vectors."""
    out = []
    for i in range(n):
        kind = i % 7
        if kind == 0:
            x = rng.standard_normal(D)
        elif kind == 1:
            x = rng.standard_t(2, D)
        elif kind == 2:
            x = rng.standard_normal(D)
            x[rng.integers(D)] *= 20
        elif kind == 3:
            x = rng.standard_normal(D) * 1e-20
        elif kind == 4:
            x = rng.standard_normal(D) * 1e20
        elif kind == 5:
            x = rng.integers(-254, 255, D) / 128.0       # amax often 2^k: x*inv hits .5 exactly
            x[0] = 254 / 128.0
        else:
            x = np.zeros(D)
        out.append(x.astype(np.float32))
    return out


def test_writer_matches_numpy_f32_arithmetic(oracle_lib):
    """The page's steps done with numpy float32 operations (IEEE, correctly
    rounded) give the same words as the oracle's double-then-round route."""
    rng = np.random.default_rng(11)
    for x in _vectors(rng, 700, 128):
        words = oracle.quantize_vector(x)
        codes = words[:32].copy().view("<i1").astype(np.int64)
        amax = np.max(np.abs(x)) if x.size else np.float32(0)
        amax = np.float32(amax)
        inv = np.float32(127) / amax if amax > 0 else np.float32(0)
        t = (x * inv).astype(np.float32)                  # f32 product
        want = np.clip(_round_half_away(t), -127, 127).astype(np.int64)
        assert np.array_equal(codes, want)
        scale = (amax / np.float32(127)) if amax > 0 else np.float32(1.0)
        assert words[32] == np.float32(scale).view(np.uint32)


def test_writer_vs_exact_rational(oracle_lib):
    """Against round(x * 127 / amax) in exact rational arithmetic: the
    page's two-step f32 recipe (inv = 127/amax, then x * inv) may move a
    code by one only when the exact value sits within f32 rounding of a
    half-way point; everywhere else the codes are equal."""
    rng = np.random.default_rng(12)
    n_diff = n_tot = 0
    for x in _vectors(rng, 140, 64):
        words = oracle.quantize_vector(x)
        codes = words[:16].copy().view("<i1").astype(np.int64)
        amax = Fraction(float(np.max(np.abs(x))))
        for d in range(x.size):
            if amax == 0:
                exact = 0
                u = Fraction(0)
            else:
                u = Fraction(float(x[d])) * 127 / amax
                exact = int(np.sign(float(u))) * int((abs(u) + Fraction(1, 2)).__floor__())
            n_tot += 1
            if codes[d] != exact:
                n_diff += 1
                assert abs(int(codes[d]) - exact) == 1
                frac = abs(u) - int(abs(u))
                assert abs(frac - Fraction(1, 2)) < Fraction(1, 2**15)
    assert n_diff <= max(3, n_tot // 1000)


def test_writer_invariants(oracle_lib):
    """Page-stated invariants: |code| <= 127; the element attaining amax
    gets +-127; codes keep the sign of x (or are 0); codes are monotone in
    x; the scale word is amax/127 to within rounding (1.0 for amax = 0);
    round trip |x - code * scale| <= amax/254 (plus a few f32 ulps)."""
    rng = np.random.default_rng(13)
    for x in _vectors(rng, 700, 128):
        words = oracle.quantize_vector(x)
        codes = words[:32].copy().view("<i1").astype(np.int64)
        scale = np.float64(words[32:].view("<f4")[0])
        amax = float(np.max(np.abs(x)))
        assert np.all(np.abs(codes) <= 127)
        if amax == 0:
            assert np.all(codes == 0) and scale == 1.0
            continue
        i = int(np.argmax(np.abs(x)))
        assert codes[i] == (127 if x[i] > 0 else -127)
        assert np.all((codes == 0) | (np.sign(codes) == np.sign(x)))
        order = np.argsort(x, kind="stable")
        assert np.all(np.diff(codes[order]) >= 0)
        assert abs(scale * 127 - amax) <= amax * 2.0**-23
        err = np.abs(x.astype(np.float64) - codes * scale)
        assert np.all(err <= amax / 254 * (1 + 2.0**-14))


def test_writer_layout_pad_and_strides(oracle_lib):
    """Token vectors land at [slot // B, kv_head, slot % B, :]; PAD rows and
    every unmapped slot keep their previous words; a strided row view
    (rows of a wider fused buffer) writes the same words as contiguous rows."""
    rng = np.random.default_rng(14)
    Hk, D, B, nb = 3, 64, 8, 5
    W = D // 4 + 1
    T = 20
    fused = rng.standard_normal((T, 7 * Hk * D)).astype(np.float32)
    k_off, v_off = 2 * Hk * D, 5 * Hk * D
    key_view = fused[:, k_off:k_off + Hk * D]
    val_view = fused[:, v_off:v_off + Hk * D]
    slots = rng.choice(nb * B, size=T, replace=False).astype(np.uint32)
    slots[[3, 11, 17]] = PAD
    kc = np.full((nb, Hk, B, W), 0xA5A5A5A5, dtype=np.uint32)
    vc = kc.copy()
    oracle.reshape_and_cache(key_view, val_view, kc, vc, slots, num_kv_heads=Hk, head_size=D,
                             block_size=B)
    kc2 = np.full_like(kc, 0xA5A5A5A5)
    vc2 = kc2.copy()
    oracle.reshape_and_cache(np.ascontiguousarray(key_view).reshape(T, Hk, D),
                             np.ascontiguousarray(val_view).reshape(T, Hk, D), kc2, vc2, slots,
                             num_kv_heads=Hk, head_size=D, block_size=B)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)

    touched = np.zeros((nb, Hk, B), dtype=bool)
    for i in range(T):
        if slots[i] == PAD:
            continue
        b, o = divmod(int(slots[i]), B)
        for h in range(Hk):
            xk = key_view[i, h * D:(h + 1) * D]
            xv = val_view[i, h * D:(h + 1) * D]
            assert np.array_equal(kc[b, h, o], oracle.quantize_vector(xk))
            assert np.array_equal(vc[b, h, o], oracle.quantize_vector(xv))
            touched[b, h, o] = True
    assert np.all(kc[~touched] == 0xA5A5A5A5) and np.all(vc[~touched] == 0xA5A5A5A5)


# ----------------------------------------------------------------- decode


def _dec(case, **kw):
    return oracle.decode(case["q"], case["kc"], case["vc"], case["bt"], case["cl"],
                         num_kv_heads=case["Hk"], block_size=case["B"],
                         scale=kw.get("scale", 1.0 / np.sqrt(case["D"])))


def _brute(case, scale):
    """Dense attention from numpy views of the cache: gather each sequence's
    blocks, repeat kv heads over their query group, scipy softmax."""
    S, H, Hk, D = case["S"], case["H"], case["Hk"], case["D"]
    r = H // Hk
    cap = case["Nb"] * case["B"]
    out = np.zeros((S, H, D))
    for s in range(S):
        c = min(int(case["cl"][s]), cap)
        if c == 0:
            continue
        K = np.repeat(dense_context(case["kc"], case["bt"], s, c, D), r, axis=1)   # [c, H, D]
        V = np.repeat(dense_context(case["vc"], case["bt"], s, c, D), r, axis=1)
        z = scale * np.einsum("hd,chd->hc", case["q"][s].astype(np.float64), K)
        p = softmax(z, axis=1)
        out[s] = np.einsum("hc,chd->hd", p, V)
    return out


SHAPES = [
    dict(S=3, H=4, Hk=2, D=64, B=16, lens=[37, 100, 1]),
    dict(S=2, H=8, Hk=1, D=128, B=8, lens=[5, 70]),
    dict(S=2, H=6, Hk=6, D=32, B=4, lens=[9, 13]),
    dict(S=2, H=16, Hk=2, D=256, B=32, lens=[33, 64]),
    dict(S=3, H=4, Hk=1, D=16, B=16, lens=[0, 16, 17]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"H{s['H']}Hk{s['Hk']}D{s['D']}B{s['B']}")
def test_decode_vs_dense_brute_force(oracle_lib, shape):
    rng = np.random.default_rng(21)
    case = random_paged_case(rng, **shape)
    scale = float(np.float32(1.0 / np.sqrt(case["D"])))
    got = _dec(case, scale=scale)
    want = _brute(case, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_decode_single_token_is_its_value_row(oracle_lib):
    """context_len = 1 returns that token's dequantised V exactly (this also
    pins the no-epsilon reading of the softmax denominator)."""
    rng = np.random.default_rng(22)
    case = random_paged_case(rng, S=3, H=8, Hk=2, D=64, B=16, lens=[1, 1, 1], pool_extra=9)
    got = _dec(case)
    for s in range(3):
        V = dense_context(case["vc"], case["bt"], s, 1, 64)[0]       # [Hk, D]
        for h in range(8):
            assert np.array_equal(got[s, h], V[h // 4])


def test_decode_equal_logits_give_mean_value(oracle_lib):
    """Identical keys, q = 0 or scale = 0 make all logits equal: the output
    is the plain mean of the dequantised V rows."""
    rng = np.random.default_rng(23)
    case = random_paged_case(rng, S=2, H=4, Hk=2, D=64, B=16, lens=[37, 100])
    means = [dense_context(case["vc"], case["bt"], s, int(case["cl"][s]), 64).mean(axis=0)
             for s in range(2)]
    zero = _dec(case, scale=0.0)
    case_q0 = dict(case, q=np.zeros_like(case["q"]))
    q0 = _dec(case_q0)
    # identical keys: copy token 0's K vector into every slot of the sequence
    kc = case["kc"].copy()
    for s in range(2):
        c = int(case["cl"][s])
        t = np.arange(c)
        b, o = case["bt"][s, t // 16], t % 16
        kc[b, :, o] = kc[case["bt"][s, 0], :, 0]
    same = _dec(dict(case, kc=kc))
    for s in range(2):
        for h in range(4):
            for got in (zero, q0, same):
                np.testing.assert_allclose(got[s, h], means[s][h // 2], rtol=1e-13, atol=1e-15)


def test_decode_two_tokens_closed_form(oracle_lib):
    """Two tokens: out = v0 + sigmoid(z1 - z0) (v1 - v0)."""
    rng = np.random.default_rng(24)
    case = random_paged_case(rng, S=1, H=2, Hk=1, D=64, B=16, lens=[2])
    scale = 0.125
    got = _dec(case, scale=scale)
    K = dense_context(case["kc"], case["bt"], 0, 2, 64)[:, 0]
    V = dense_context(case["vc"], case["bt"], 0, 2, 64)[:, 0]
    for h in range(2):
        qh = case["q"][0, h].astype(np.float64)
        dz = scale * (qh @ K[1] - qh @ K[0])
        want = V[0] + (V[1] - V[0]) / (1.0 + np.exp(-dz))
        np.testing.assert_allclose(got[0, h], want, rtol=1e-12, atol=1e-14)


def test_decode_dominant_key(oracle_lib):
    """One key with a logit gap above 100 takes all the weight."""
    rng = np.random.default_rng(25)
    case = random_paged_case(rng, S=1, H=1, Hk=1, D=64, B=16, lens=[40])
    q = np.zeros_like(case["q"])
    q[0, 0, 0] = 1.0
    kc = case["kc"].copy()
    bt = case["bt"]
    for t in range(40):                       # every key: code 0 in dim 0 except token 29
        b, o = bt[0, t // 16], t % 16
        kc[b, 0, o, 0] &= np.uint32(0xFFFFFF00)
    b29, o29 = bt[0, 29 // 16], 29 % 16
    kc[b29, 0, o29, 0] = (kc[b29, 0, o29, 0] & np.uint32(0xFFFFFF00)) | np.uint32(127)
    kc[b29, 0, o29, 16] = np.float32(2.0).view(np.uint32)            # k[0] = 254
    got = oracle.decode(q, kc, case["vc"], bt, case["cl"], num_kv_heads=1, block_size=16,
                        scale=1.0)
    V = dense_context(case["vc"], bt, 0, 40, 64)[29, 0]
    # the other 39 tokens carry weight e^-254 each: far below double rounding
    np.testing.assert_allclose(got[0, 0], V, rtol=1e-15, atol=1e-100)


def test_decode_metamorphic(oracle_lib):
    """Moving blocks to other physical ids (table updated) changes nothing
    bit for bit; permuting the tokens of a context changes nothing beyond
    rounding; heads of one group given the same q agree exactly."""
    rng = np.random.default_rng(26)
    case = random_paged_case(rng, S=2, H=8, Hk=2, D=64, B=8, lens=[29, 50], pool_extra=5)
    base = _dec(case)

    perm = rng.permutation(case["pool"])
    kc = np.empty_like(case["kc"]); vc = np.empty_like(case["vc"])
    kc[perm] = case["kc"]; vc[perm] = case["vc"]
    bt = case["bt"].copy()
    used = bt != PAD
    bt[used] = perm[bt[used]].astype(np.uint32)
    moved = _dec(dict(case, kc=kc, vc=vc, bt=bt))
    assert np.array_equal(moved, base)

    kc = case["kc"].copy(); vc = case["vc"].copy()
    for s in range(2):
        c = int(case["cl"][s])
        t = np.arange(c)
        b, o = case["bt"][s, t // 8], t % 8
        p = rng.permutation(c)
        kc[b, :, o] = case["kc"][b[p], :, o[p]]
        vc[b, :, o] = case["vc"][b[p], :, o[p]]
    shuffled = _dec(dict(case, kc=kc, vc=vc))
    np.testing.assert_allclose(shuffled, base, rtol=1e-12, atol=1e-14)

    q = case["q"].copy()
    q[:, 1:4] = q[:, 0:1]
    same = _dec(dict(case, q=q))
    for h in range(1, 4):
        assert np.array_equal(same[:, h], same[:, 0])


def test_decode_gqa_is_contiguous_groups(oracle_lib):
    """GQA decode equals an MHA decode over a cache whose kv heads are each
    repeated over their group (head h reads kv head h // (H / Hk))."""
    rng = np.random.default_rng(27)
    case = random_paged_case(rng, S=2, H=8, Hk=2, D=64, B=16, lens=[45, 21])
    got = _dec(case)
    mha = dict(case, kc=np.ascontiguousarray(np.repeat(case["kc"], 4, axis=1)),
               vc=np.ascontiguousarray(np.repeat(case["vc"], 4, axis=1)), Hk=8)
    np.testing.assert_array_equal(_dec(mha), got)


def test_decode_context_clamp_and_empty(oracle_lib):
    """context_len beyond max_blocks_per_seq * block_size is clamped to it;
    context_len = 0 gives a zero row."""
    rng = np.random.default_rng(28)
    case = random_paged_case(rng, S=2, H=2, Hk=1, D=64, B=16, lens=[32, 5])
    base = _dec(case)
    big = dict(case, cl=np.array([10_000, 5], dtype=np.uint32))
    np.testing.assert_array_equal(_dec(big), base)
    empty = dict(case, cl=np.array([0, 5], dtype=np.uint32))
    e = _dec(empty)
    assert np.all(e[0] == 0) and np.array_equal(e[1], base[1])


@pytest.mark.parametrize("splits", [[20], [0, 20], [1, 2, 50, 99], [99], [33, 33, 66]])
def test_partials_merge_to_the_whole(oracle_lib, splits):
    """Split-context partials merged by log-sum-exp equal the whole row."""
    rng = np.random.default_rng(29)
    case = random_paged_case(rng, S=1, H=2, Hk=1, D=64, B=16, lens=[100])
    whole = _dec(case)
    for h in range(2):
        edges = [0] + sorted(splits) + [100]
        parts = [oracle.decode_partial(case["q"], case["kc"], case["vc"], case["bt"],
                                       num_kv_heads=1, block_size=16, scale=1 / 8.0, s=0, h=h,
                                       t0=a, t1=b) for a, b in zip(edges[:-1], edges[1:])]
        m = np.array([p[0] for p in parts]); l = np.array([p[1] for p in parts])
        acc = np.stack([p[2] for p in parts])
        np.testing.assert_allclose(oracle.combine(m, l, acc), whole[0, h], rtol=1e-12, atol=1e-15)
        # partial of the whole range, normalised, is the row itself
        m1, l1, a1 = oracle.decode_partial(case["q"], case["kc"], case["vc"], case["bt"],
                                           num_kv_heads=1, block_size=16, scale=1 / 8.0, s=0,
                                           h=h, t0=0, t1=100)
        np.testing.assert_allclose(a1 / l1, whole[0, h], rtol=1e-13, atol=1e-15)


def test_dequant_view_roundtrip(oracle_lib):
    """Dequantised rows from numpy views stay within amax/254 of the f32 input."""
    rng = np.random.default_rng(30)
    case = random_paged_case(rng, S=2, H=2, Hk=2, D=128, B=16, lens=[17, 40])
    K = np.concatenate([dense_context(case["kc"], case["bt"], s, int(case["cl"][s]), 128)
                        for s in range(2)])
    x = case["key"].astype(np.float64)
    amax = np.abs(x).max(axis=-1, keepdims=True)
    assert np.all(np.abs(K - x) <= amax / 254 * (1 + 2.0**-14))


# ---------------------------------------------------- multi-row causal decode


def _rows_case(rng, S, R, H, Hk, D, B, lens):
    case = random_paged_case(rng, S=S, H=H, Hk=Hk, D=D, B=B, lens=lens)
    case["qr"] = rng.standard_normal((S, R, H, D)).astype(np.float32)
    case["R"] = R
    return case


def _rows(case, cl=None, scale=0.125):
    return oracle.decode_rows(case["qr"], case["kc"], case["vc"], case["bt"],
                              case["cl"] if cl is None else cl, num_kv_heads=case["Hk"],
                              block_size=case["B"], scale=scale)


@pytest.mark.parametrize("R", [1, 2, 5])
def test_rows_vs_causal_brute_force(oracle_lib, R):
    """Row b of sequence s attends to its first c_s - (R - 1 - b) tokens
    ("attention.rs", attention_b: t_len = base_pos + b + 1): a dense
    numpy/scipy softmax over that prefix, kv heads repeated over their group."""
    rng = np.random.default_rng(40 + R)
    S, H, Hk, D, B = 3, 8, 2, 64, 16
    lens = [37, 3, 100]
    case = _rows_case(rng, S, R, H, Hk, D, B, lens)
    got = _rows(case, scale=0.125)
    r = H // Hk
    for s in range(S):
        c = lens[s]
        K = np.repeat(dense_context(case["kc"], case["bt"], s, c, D), r, axis=1)
        V = np.repeat(dense_context(case["vc"], case["bt"], s, c, D), r, axis=1)
        for b in range(R):
            n = c - (R - 1 - b)
            if n <= 0:
                assert np.all(got[s, b] == 0.0)
                continue
            z = 0.125 * np.einsum("hd,chd->hc", case["qr"][s, b].astype(np.float64), K[:n])
            want = np.einsum("hc,chd->hd", softmax(z, axis=1), V[:n])
            np.testing.assert_allclose(got[s, b], want, rtol=1e-12, atol=1e-13)


def test_rows_reduce_to_single_query_decode(oracle_lib):
    """R = 1 is the single-query decode; row b equals the single-query decode
    of the context cut to c - (R - 1 - b) tokens (clamp first, then cut)."""
    rng = np.random.default_rng(44)
    S, R, H, Hk, D, B = 2, 4, 4, 2, 64, 16
    case = _rows_case(rng, S, R, H, Hk, D, B, [50, 20])
    cap = case["Nb"] * B
    cl = np.array([10_000, 20], dtype=np.uint32)           # sequence 0 clamps to cap first
    got = _rows(case, cl=cl)
    for b in range(R):
        cut = np.array([min(int(c), cap) - (R - 1 - b) for c in cl], dtype=np.uint32)
        want = oracle.decode(np.ascontiguousarray(case["qr"][:, b]), case["kc"], case["vc"], case["bt"],
                             cut, num_kv_heads=Hk, block_size=B, scale=0.125)
        np.testing.assert_array_equal(got[:, b], want)
    one = dict(case, qr=np.ascontiguousarray(case["qr"][:, :1]))
    np.testing.assert_array_equal(
        _rows(one, cl=cl)[:, 0],
        oracle.decode(np.ascontiguousarray(case["qr"][:, 0]), case["kc"], case["vc"], case["bt"], cl,
                      num_kv_heads=Hk, block_size=B, scale=0.125))
