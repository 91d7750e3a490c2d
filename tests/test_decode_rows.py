"""GPU multi-row causal decode (pa_q8_decode_rows) against the fp64 oracle
(oracle.decode_rows: row b of R attends to the first c - (R-1-b) tokens,
"attention.rs", attention_b), |gpu - oracle| <= 1e-5 + 1e-4 |oracle|
elementwise, for both kernel families: row counts 1..16 (several head groups
per kv head), GQA ratios and head sizes, forced partitions whose last one
some rows see none of, contexts shorter than R (zero rows), clamped
contexts, and the full-size large-batch workload on sampled rows.  R = 1 is
pa_q8_decode bit for bit."""
import numpy as np
import pytest

from int8_paged_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TC, CC, T5 = 2, 1, 3          # T5: tcgen05 (5th-generation tensor cores, TMEM accumulators)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


_CACHE = {}


def _setup(name):
    if name in _CACHE:
        return _CACHE[name]
    from tests.gpu_helpers import dev_u32, oracle_write, poisoned_cache
    w = wl.build(name, with_append=False)
    ok_, ov_ = poisoned_cache(w), poisoned_cache(w)
    oracle_write(w.key, w.value, w.slot_mapping, ok_, ov_, w.cfg)
    w.key = w.value = None
    _CACHE.clear()
    _CACHE[name] = (w, ok_, ov_, dev_u32(ok_), dev_u32(ov_))
    return _CACHE[name]


@pytest.mark.parametrize("kernel", [TC, CC])
def test_one_row_is_single_query_decode_bitwise(kernel):
    """R = 1 runs the single-query launch: identical bits."""
    from tests.gpu_helpers import gpu_decode, gpu_decode_rows
    w, ok_, ov_, kc, vc = _setup("llama8b")
    for pt in (0, 512):
        a = gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt)
        b = gpu_decode_rows(w, kc, vc, w.q[:, None].copy(), kernel=kernel, partition_tokens=pt)
        assert np.array_equal(a, b[:, 0]), f"pt {pt}"


@pytest.mark.parametrize("kernel", [TC, CC, T5])
@pytest.mark.parametrize("name,R", [("tiny", 1), ("tiny", 3), ("tiny", 8), ("llama8b", 2),
                                    ("llama8b", 5), ("edge", 3)])
def test_workloads_all_rows(name, R, kernel):
    from tests.gpu_helpers import assert_close, device_status, gpu_decode_rows, oracle_decode_rows
    w, ok_, ov_, kc, vc = _setup(name)
    q = wl.query_rows(w, R)
    want = oracle_decode_rows(w, ok_, ov_, q)
    got = gpu_decode_rows(w, kc, vc, q, kernel=kernel)
    assert_close(got, want, f"{name} R {R} kernel {kernel}")
    assert device_status() == 0


@pytest.mark.parametrize("kernel", [TC, CC, T5])
def test_forced_partitions_with_rows_that_see_none_of_the_last(kernel):
    """Contexts 1 .. 3 tokens past a partition boundary: the lower rows see
    nothing of the last partition, the combine must give those partials no
    weight; contexts shorter than R give zero rows."""
    from tests.gpu_helpers import assert_close, gpu_decode_rows, oracle_decode_rows
    R, pt = 4, 256
    lens = [257, 258, 259, 513, 512, 1, 2, 3, 4, 0, 1000, 777]
    w, ok_, ov_, kc, vc = _random_case(len(lens), 8, 2, 128, 16, lens, seed=41)
    q = np.random.default_rng(41).standard_normal((len(lens), R, 8, 128)).astype(np.float32)
    want = oracle_decode_rows(w, ok_, ov_, q)
    for p in (0, pt, 128):
        got = gpu_decode_rows(w, kc, vc, q, kernel=kernel, partition_tokens=p)
        assert_close(got, want, f"pt {p}")
        # row b of a context c sees c - (3 - b) tokens: none -> exact zeros
        for s, c in enumerate(lens):
            for b in range(R):
                if c - (R - 1 - b) <= 0:
                    assert np.all(got[s, b] == 0.0), (s, b)


def _random_case(*args, **kw):
    from tests.gpu_helpers import random_case
    return random_case(*args, **kw)


@pytest.mark.parametrize("kernel", [TC, CC, T5])
@pytest.mark.parametrize("H,Hk,D,R", [(4, 4, 64, 16), (8, 4, 64, 7), (32, 1, 128, 2), (16, 2, 128, 4),
                                      (16, 1, 256, 3), (8, 8, 256, 2), (24, 2, 64, 5)])
def test_gqa_ratios_head_sizes_and_row_counts(kernel, H, Hk, D, R):
    from tests.gpu_helpers import assert_close, gpu_decode_rows, oracle_decode_rows
    lens = [1, 17, 300, 1000]
    w, ok_, ov_, kc, vc = _random_case(4, H, Hk, D, 16, lens, seed=H * 7 + Hk + D + R)
    q = np.random.default_rng(R).standard_normal((4, R, H, D)).astype(np.float32)
    want = oracle_decode_rows(w, ok_, ov_, q)
    for pt in (0, 256):
        assert_close(gpu_decode_rows(w, kc, vc, q, kernel=kernel, partition_tokens=pt), want,
                     f"H {H} Hk {Hk} D {D} R {R} pt {pt}")


@pytest.mark.parametrize("kernel", [TC, CC, T5])
def test_clamped_context(kernel):
    from tests.gpu_helpers import assert_close, gpu_decode_rows, oracle_decode_rows
    lens = [64, 208, 50]                                   # 208 = max_blocks_per_seq * 16
    w, ok_, ov_, kc, vc = _random_case(3, 8, 2, 128, 16, lens, seed=6)
    cl = np.array([64, 10_000, 50], dtype=np.uint32)       # seq 1 clamps to 208
    q = np.random.default_rng(6).standard_normal((3, 6, 8, 128)).astype(np.float32)
    want = oracle_decode_rows(w, ok_, ov_, q, cl=cl)
    assert_close(gpu_decode_rows(w, kc, vc, q, kernel=kernel, cl=cl), want, "clamped")


def _sampled_rows_oracle(w, ok_, ov_, q, picks):
    """fp64 rows (s, b, h) one by one: the oracle's partial over the first
    c - (R-1-b) tokens, normalised."""
    import oracle
    R = q.shape[1]
    cap = w.cfg.max_blocks_per_seq * w.cfg.block_size
    out = []
    for s, b, h in picks:
        t1 = max(0, min(int(w.context_lens[s]), cap) - (R - 1 - b))
        if t1 == 0:
            out.append(np.zeros(w.cfg.head_size))
            continue
        _, l, acc = oracle.decode_partial(np.ascontiguousarray(q[:, b]), ok_, ov_, w.block_tables,
                                          num_kv_heads=w.cfg.num_kv_heads,
                                          block_size=w.cfg.block_size, scale=w.scale, s=int(s),
                                          h=int(h), t0=0, t1=t1)
        out.append(acc / l)
    return np.array(out)


@pytest.mark.parametrize("kernel,R", [(0, 4), (TC, 4), (CC, 4), (T5, 4), (0, 5), (0, 8)])
def test_large_batch_many_rows_sampled(kernel, R):
    """The large-batch workload with 4, 5 or 8 query rows per sequence (the
    automatic plan takes tcgen05 from 24 pairs on: 32 and 40 pairs in partly
    filled CTAs, 64 in a full one), sampled (s, b, h) rows against the
    oracle."""
    from tests.gpu_helpers import assert_close, device_status, gpu_decode_rows
    w, ok_, ov_, kc, vc = _setup("large")
    q = wl.query_rows(w, R)
    got = gpu_decode_rows(w, kc, vc, q, kernel=kernel)
    rng = np.random.default_rng(kernel)
    S, H = w.cfg.num_seqs, w.cfg.num_heads
    picks = {(int(np.argmax(w.context_lens)), R - 1, 0), (int(np.argmin(w.context_lens)), 0, H - 1)}
    while len(picks) < 96:
        picks.add((int(rng.integers(S)), int(rng.integers(R)), int(rng.integers(H))))
    picks = sorted(picks)
    want = _sampled_rows_oracle(w, ok_, ov_, q, picks)
    sel = np.array([got[s, b, h] for s, b, h in picks])
    assert_close(sel, want, f"large R {R} kernel {kernel}")
    assert np.all(np.isfinite(got))
    assert device_status() == 0


@pytest.mark.parametrize("H,Hk,D", [(8, 2, 64), (32, 8, 128), (16, 1, 256), (64, 1, 128)])
def test_tcgen05_single_row_and_wide_groups(H, Hk, D):
    """The tcgen05 family asked for explicitly at R = 1, and a 64-head group
    (one full CTA of virtual heads), against the oracle."""
    from tests.gpu_helpers import assert_close, gpu_decode_rows, oracle_decode_rows
    lens = [1, 40, 333, 1500]
    w, ok_, ov_, kc, vc = _random_case(4, H, Hk, D, 16, lens, seed=H + D)
    for R in (1, 2):
        q = np.random.default_rng(R + H).standard_normal((4, R, H, D)).astype(np.float32)
        want = oracle_decode_rows(w, ok_, ov_, q)
        for pt in (0, 256):
            assert_close(gpu_decode_rows(w, kc, vc, q, kernel=T5, partition_tokens=pt), want,
                         f"H {H} Hk {Hk} D {D} R {R} pt {pt}")


@pytest.mark.parametrize("kernel", [TC, CC, T5])
def test_scale_sign_extreme_q_rows_and_growing_v(kernel):
    """Every family (tcgen05 at 32 pairs per kv head) against the oracle on:
    a negative, a zero and a large softmax scale; q rows of very different
    magnitudes in one kv group (1e-40 (subnormal) .. 1e-30, an all-zero row,
    and up to 8x), each row scaled by its own largest exponent; and V
    vectors whose magnitude grows 3 decades along each context, so the
    weight scale's exponent rises chunk by chunk (lazy rescales of O).
    The case stays well conditioned for f32 arithmetic: logits within a few
    hundred (beyond that the weights depend on logit differences below
    f32's resolution of the logits: a q row scaled by 1e15 failed on every
    family, the CUDA-core f32 one included), and V growth small enough that
    the weighted sum does not cancel (12 decades of growth, where large
    terms cancel to small outputs, failed on every family too)."""
    import dataclasses
    from tests.gpu_helpers import assert_close, device_status, gpu_decode_rows, oracle_decode_rows, random_case
    lens = [1, 33, 700, 2049]
    grow = lambda pos, ctx: 10.0 ** (-2.0 + 3.0 * pos / np.maximum(ctx - 1, 1))
    w, ok_, ov_, kc, vc = random_case(4, 16, 2, 128, 16, lens, seed=71, v_token_mult=grow)
    R = 4
    q = np.random.default_rng(72).standard_normal((4, R, 16, 128))
    q[:, :, 0] *= 1e-30
    q[:, :, 1] = 0.0
    q[:, :, 2] *= 8.0
    q[:, :, 3] *= 1e-40                      # subnormal in f32
    q[:, 1, 5] *= 1e-8
    q = q.astype(np.float32)
    for mult in (-1.0, 0.0, 3.0):
        ws = dataclasses.replace(w, scale=float(np.float32(mult / np.sqrt(128))))
        want = oracle_decode_rows(ws, ok_, ov_, q)
        for pt in (0, 256):
            got = gpu_decode_rows(ws, kc, vc, q, kernel=kernel, partition_tokens=pt)
            assert_close(got, want, f"kernel {kernel} scale x {mult} pt {pt}")
    assert device_status() == 0


@pytest.mark.parametrize("D,R,H", [(64, 8, 8), (128, 4, 8), (256, 2, 16)])
def test_tcgen05_many_waves_with_empty_contexts(D, R, H):
    """More (sequence, kv head) CTAs than fit at once, one partition each (the
    longest-first order across waves), with every 37th context empty (its
    rows must be zeros) and one of a single token; every row against the
    oracle."""
    from tests.gpu_helpers import (assert_close, device_status, gpu_decode_rows, oracle_decode_rows,
                                   random_case)
    S, Hk, B = 320, 1, 16
    rng = np.random.default_rng(D + R)
    lens = [int(x) for x in rng.integers(2, 300, S)]
    for s in range(0, S, 37):
        lens[s] = 0
    lens[5] = 1
    w, ok_, ov_, kc, vc = random_case(S, H, Hk, D, B, lens, seed=60 + D)
    q = rng.standard_normal((S, R, H, D)).astype(np.float32)
    got = gpu_decode_rows(w, kc, vc, q, kernel=T5, partition_tokens=384)
    want = oracle_decode_rows(w, ok_, ov_, q)
    assert_close(got, want, f"persistent D {D} R {R}")
    assert np.all(got[[s for s in range(S) if lens[s] == 0]] == 0.0)
    assert device_status() == 0
