"""The seeded synthetic inputs match their stated recipes (CPU only).

Every benchmark line and every parity case draws its inputs from
int8_paged_kv_gb300.workloads, so the recipe is pinned here: shapes, context
length distributions, the shuffled block pool and block tables, the slot
mapping the writer rows follow, the PAD rows, the large batch's strided
append, the MQA workload's value spread and zero vectors, the long-context
outlier channels, determinism, and the algorithmic byte counts the roofline
divides by (every token's K and V vector once, q and out, the block-table
entries walked, the context lengths)."""
import math

import numpy as np
import pytest

from int8_paged_kv_gb300 import workloads as wl

PAD = wl.PAD_SLOT
UNUSED = wl.UNUSED_BLOCK

SHAPES = {  # name: (S, H, Hk, D, B, max context)
    "tiny": (2, 4, 2, 64, 16, 112),
    "llama8b": (64, 32, 8, 128, 16, 4096),
    "long": (8, 32, 8, 128, 32, 131072),
    "large": (256, 64, 8, 128, 16, 8192),
    "edge": (32, 16, 1, 256, 32, 4096),
}


@pytest.fixture(scope="module")
def structure():
    return {name: wl.build(name, with_kv=False, with_append=False) for name in SHAPES}


@pytest.mark.parametrize("name", list(SHAPES))
def test_shapes_and_block_tables(structure, name):
    w = structure[name]
    S, H, Hk, D, B, max_ctx = SHAPES[name]
    cfg = w.cfg
    assert (cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size) == (S, H, Hk, D, B)
    assert cfg.max_blocks_per_seq * B >= max_ctx
    assert w.q.shape == (S, H, D) and w.q.dtype == np.float32
    assert w.context_lens.dtype == np.uint32 and w.context_lens.shape == (S,)
    assert w.block_tables.shape == (S, cfg.max_blocks_per_seq)
    assert math.isclose(w.scale, 1.0 / math.sqrt(D), rel_tol=1e-6)
    used = []
    for s in range(S):
        n = -(-int(w.context_lens[s]) // B)
        row = w.block_tables[s]
        assert np.all(row[:n] != UNUSED) and np.all(row[n:] == UNUSED), s
        used.extend(int(b) for b in row[:n])
    # every physical block belongs to at most one sequence, and all lie in the pool
    assert len(used) == len(set(used))
    assert max(used) < w.num_blocks


@pytest.mark.parametrize("name", list(SHAPES))
def test_writer_rows_follow_the_block_tables(structure, name):
    """Row i of the cache-building writer call is token t of sequence s, stored
    at slot block_tables[s][t / B] * B + t % B; only the tiny workload has PAD
    rows, and they belong to no sequence."""
    w = structure[name]
    B = w.cfg.block_size
    rows = np.flatnonzero(w.row_seq >= 0)
    assert np.all(w.slot_mapping[w.row_seq < 0] == PAD)
    t_of_row = np.zeros(w.row_seq.size, dtype=np.int64)
    for s in range(w.cfg.num_seqs):
        idx = np.flatnonzero(w.row_seq == s)
        assert idx.size == int(w.context_lens[s])
        t_of_row[idx] = np.arange(idx.size)
    s = w.row_seq[rows].astype(np.int64)
    t = t_of_row[rows]
    want = w.block_tables[s, t // B].astype(np.int64) * B + t % B
    assert np.array_equal(w.slot_mapping[rows].astype(np.int64), want)
    assert np.unique(want).size == want.size


def test_context_length_recipes(structure):
    tiny = structure["tiny"]
    assert list(tiny.context_lens) == [37, 100] and tiny.num_blocks == 16
    assert tiny.slot_mapping.size == 140 and int((tiny.slot_mapping == PAD).sum()) == 3
    c = structure["llama8b"].context_lens
    assert c.min() >= 512 and c.max() <= 4096
    c = structure["long"].context_lens
    assert c.min() >= 32768 and c.max() <= 131072
    c = structure["large"].context_lens.astype(np.float64)
    assert c.min() >= 16 and c.max() <= 8192
    # lognormal with median 2048 and sigma 1 (natural log): the sample median of
    # 256 draws lies within ~4 standard errors (0.078 in log space) of ln 2048
    assert abs(math.log(np.median(c)) - math.log(2048.0)) < 0.35
    assert (c == 8192).sum() >= 1                     # the clip at 8192 is reached
    e = structure["edge"].context_lens
    assert {1, 31, 33, 4095} <= set(int(x) for x in e)
    assert e.min() >= 1 and e.max() <= 4096
    assert int((e % 32 != 0).sum()) >= (32 - 4) // 2


def test_generation_is_deterministic(structure):
    again = wl.build("llama8b", with_kv=False, with_append=False)
    first = structure["llama8b"]
    assert np.array_equal(again.context_lens, first.context_lens)
    assert np.array_equal(again.block_tables, first.block_tables)
    assert np.array_equal(again.q, first.q)
    assert np.array_equal(again.slot_mapping, first.slot_mapping)


def test_large_batch_append_rows():
    """The large batch's writer workload: 16384 rows, 819 of them PAD (5%), the
    rest written to distinct slots of blocks no sequence owns, K and V taken as
    column slices of fused rows of (H + 2 Hk) * D = 10240 floats."""
    w = wl.build("large", with_kv=False, with_append=True)
    a = w.append
    H, Hk, D, B = w.cfg.num_heads, w.cfg.num_kv_heads, w.cfg.head_size, w.cfg.block_size
    assert a.num_tokens == 16384 and a.row_stride == 10240 == (H + 2 * Hk) * D
    assert (a.key_offset, a.value_offset) == (H * D, (H + Hk) * D)
    assert a.key_view().shape == (16384, Hk * D) and a.value_view().shape == (16384, Hk * D)
    sm = a.slot_mapping
    assert int((sm == PAD).sum()) == 819
    live = sm[sm != PAD].astype(np.int64)
    assert np.unique(live).size == live.size
    owned = set(int(b) for b in w.block_tables[w.block_tables != UNUSED])
    assert not (set((live // B).tolist()) & owned)
    assert live.max() < w.num_blocks * B
    assert abs(float(a.fused.std()) - 1.0) < 0.01


def test_edge_values_spread_and_zero_vectors():
    """MQA workload: K/V values ~N(0, variance 4) with about 2% of the token
    vectors all zero."""
    w = wl.build("edge", with_kv=True, with_append=False)
    for x in (w.key, w.value):
        zero = np.all(x == 0.0, axis=-1)
        frac = float(zero.mean())
        assert 0.015 < frac < 0.025, frac
        assert abs(float(x[~zero].std()) - 2.0) < 0.02


def test_long_context_outlier_channels(structure):
    """Long context: 1% of the kv_row channels (10 of 8 x 128) carry values x20."""
    ch = structure["long"].notes["outlier_channels"]
    assert ch.shape == (10, 2)
    assert len({(int(h), int(d)) for h, d in ch}) == 10
    assert np.all(ch[:, 0] < 8) and np.all(ch[:, 1] < 128)


def test_algorithmic_bytes_by_hand():
    """Tiny: contexts 37 and 100, Hk 2, D 64, B 16, S 2, H 4."""
    cfg = wl.CONFIGS["tiny"]
    c = np.array([37, 100], dtype=np.uint32)
    kv = (37 + 100) * 2 * 2 * (64 + 4)              # K and V vector of every token, code bytes + scale word
    qo = 2 * 2 * 4 * 64 * 4                           # q in and out back, f32
    bt = (3 + 7) * 4                                  # block-table entries walked
    assert wl.algorithmic_decode_bytes(cfg, c) == kv + qo + bt + 2 * 4
    assert wl.algorithmic_decode_bytes(cfg, c, num_rows=3) == kv + 3 * qo + bt + 2 * 4
    assert wl.algorithmic_decode_bytes(cfg, c, cache="f32") == (37 + 100) * 2 * 2 * 256 + qo + bt + 8
    slots = np.array([5, PAD, 7], dtype=np.uint32)
    assert wl.algorithmic_writer_bytes(2, 64, slots) == 2 * (2 * 64 * 4 * 2 + 2 * 68 * 2) + 3 * 4


def test_subset_keeps_the_first_sequences_with_a_compact_pool(structure):
    """subset(w, n): the first n sequences' contexts and queries, their blocks
    renumbered 0 .. pool-1 in pool order, and every writer row still landing at
    the same (sequence, position)."""
    w = structure["llama8b"]
    B = w.cfg.block_size
    n = 5
    sub = wl.subset(w, n)
    assert sub.cfg.num_seqs == n
    assert np.array_equal(sub.context_lens, w.context_lens[:n])
    assert np.array_equal(sub.q, w.q[:n])
    used_old = w.block_tables[:n][w.block_tables[:n] != UNUSED]
    used_new = sub.block_tables[sub.block_tables != UNUSED]
    assert sub.num_blocks == used_old.size == used_new.size
    assert sorted(used_new.tolist()) == list(range(sub.num_blocks))
    # the renumbering keeps the pool order of the blocks
    order_old = np.argsort(used_old, kind="stable")
    assert np.all(np.diff(used_new[order_old].astype(np.int64)) > 0)
    for s in range(n):
        idx = np.flatnonzero(sub.row_seq == s)
        t = np.arange(idx.size)
        want = sub.block_tables[s, t // B].astype(np.int64) * B + t % B
        assert np.array_equal(sub.slot_mapping[idx].astype(np.int64), want), s
