"""Seeded synthetic workloads for the int8 paged-KV decode path.

This module only *builds inputs*: random query / key / value values, context
lengths, a shuffled physical block pool, block tables and slot mappings.  It
holds none of the quantisation or attention arithmetic, so the CUDA path, the
CPU oracle, the tests and the benchmark can all draw the same inputs from it
without sharing any of the method.

The five workloads follow the shapes of the decode kernel and the writer on
the "paged_attn_q8.comp" and "reshape_and_cache_q8.comp" pages (push-constant
blocks and buffer bindings): q is f32 [num_seqs, num_heads, head_size];
block_tables is u32 [num_seqs, max_num_blocks_per_seq]; context_lens is u32
[num_seqs]; writer rows are f32 [num_tokens, num_kv_heads, head_size] with a
row stride; slot_mapping is u32 [num_tokens] with 0xFFFFFFFF meaning "skip".

Every random draw is seeded.  Bulk per-sequence tensors use a child generator
keyed by (seed, stream, sequence) so that any subset of sequences can be
regenerated on its own, and generation can run on several threads while
staying bit-identical to a single-threaded run.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

PAD_SLOT = 0xFFFFFFFF       # slot_mapping entry meaning "do not write this row"
UNUSED_BLOCK = 0xFFFFFFFF   # block_tables entry past the end of a sequence
BASE_SEED = 20261202

# generator streams (second element of the child seed)
_S_Q, _S_K, _S_V, _S_APPEND, _S_KZERO, _S_VZERO, _S_QROWS, _S_NEWKV = 1, 2, 3, 4, 5, 6, 7, 8


@dataclass(frozen=True)
class Config:
    name: str
    index: int
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    max_context: int          # largest context the distribution can produce
    description: str = ""

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_context // self.block_size)

    @property
    def n_rep(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        # softmax scale 1/sqrt(head_size), rounded once to f32 (the kernels' type)
        return float(np.float32(1.0 / math.sqrt(self.head_size)))


CONFIGS: dict[str, Config] = {c.name: c for c in [
    Config("tiny", 0, 2, 4, 2, 64, 16, 100,
           "S=2 H=4 Hk=2 D=64 B=16, context_lens {37,100}, 16-block shuffled pool, "
           "140 writer rows incl. 3 PAD"),
    Config("llama8b", 1, 64, 32, 8, 128, 16, 4096,
           "S=64 H=32 Hk=8 D=128 B=16, context_lens ~ U[512,4096]"),
    Config("long", 2, 8, 32, 8, 128, 32, 131072,
           "S=8 H=32 Hk=8 D=128 B=32, context_lens ~ U[32768,131072], "
           "10 of 1024 (kv_head, dim) channels x20"),
    Config("large", 3, 256, 64, 8, 128, 16, 8192,
           "S=256 H=64 Hk=8 D=128 B=16, context_lens = clip(LogNormal(ln 2048, 1), 16, 8192); "
           "append of 16384 rows with 5% PAD from fused rows of stride 10240"),
    Config("edge", 4, 32, 16, 1, 256, 32, 4096,
           "MQA S=32 H=16 Hk=1 D=256 B=32, context_lens incl. 1,31,33,4095, "
           "2% all-zero K/V vectors, rest ~N(0, var 4)"),
]}


@dataclass
class Append:
    """A writer call whose rows are slices of fused [T, (H + 2 Hk) * D] rows."""
    fused: np.ndarray          # f32 [T, row_floats]
    key_offset: int            # column of K within a fused row
    value_offset: int          # column of V within a fused row
    row_stride: int            # f32 elements between consecutive rows
    slot_mapping: np.ndarray   # u32 [T], PAD_SLOT = skip

    @property
    def num_tokens(self) -> int:
        return int(self.fused.shape[0])

    def key_view(self) -> np.ndarray:
        return self.fused[:, self.key_offset:self.value_offset]

    def value_view(self) -> np.ndarray:
        return self.fused[:, self.value_offset:self.value_offset + (self.value_offset - self.key_offset)]


@dataclass
class Workload:
    cfg: Config
    context_lens: np.ndarray       # u32 [S]
    block_tables: np.ndarray       # u32 [S, max_blocks_per_seq]
    num_blocks: int                # size of the physical pool
    q: np.ndarray                  # f32 [S, H, D]
    scale: float
    # rows that build the cache (one writer call): f32 [T, Hk, D] each
    key: np.ndarray | None
    value: np.ndarray | None
    slot_mapping: np.ndarray       # u32 [T] for key/value rows above
    row_seq: np.ndarray            # int32 [T]: sequence a row belongs to (-1 for PAD rows)
    append: Append | None = None   # extra writer workload (large batch only)
    notes: dict = field(default_factory=dict)

    @property
    def sum_context(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def _context_lens(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    S = cfg.num_seqs
    if cfg.name == "tiny":
        c = np.array([37, 100], dtype=np.int64)
    elif cfg.name == "llama8b":
        c = rng.integers(512, 4096, size=S, endpoint=True)
    elif cfg.name == "long":
        c = rng.integers(32768, 131072, size=S, endpoint=True)
    elif cfg.name == "large":
        # median 2048 = exp(mu); sigma = 1.0 in natural-log space; clipped to [16, 8192]
        c = np.clip(np.rint(rng.lognormal(math.log(2048.0), 1.0, size=S)), 16, 8192).astype(np.int64)
    elif cfg.name == "edge":
        fixed = np.array([1, 31, 33, 4095], dtype=np.int64)
        other = rng.integers(1, 4096, size=S - 4, endpoint=True)
        half = (S - 4 + 1) // 2
        for i in range(half):                      # at least half forced off multiples of 32
            if other[i] % cfg.block_size == 0:
                other[i] -= 1 if other[i] > 1 else -1
        c = np.concatenate([fixed, other])
        c = c[rng.permutation(S)]
    else:  # pragma: no cover
        raise KeyError(cfg.name)
    assert c.max() <= cfg.max_context and c.min() >= 1
    return c.astype(np.uint32)


def _fill_normal(out: np.ndarray, key: tuple[int, ...], sigma: float) -> None:
    _rng(*key).standard_normal(out.shape, dtype=np.float32, out=out)
    if sigma != 1.0:
        out *= np.float32(sigma)


def build(name: str, *, with_kv: bool = True, with_append: bool = True,
          threads: int | None = None) -> Workload:
    """Build the named workload.

    with_kv=False skips the bulk key/value rows (context-length / block-table
    structure and q only).  The rows of sequence s always come from the child
    generators (seed, 2, s) and (seed, 3, s), so `sequence_rows` can rebuild
    any subset later.
    """
    cfg = CONFIGS[name]
    rng = _rng(cfg.seed)
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    Nb = cfg.max_blocks_per_seq

    c = _context_lens(cfg, rng)
    nblk = -(-c.astype(np.int64) // B)
    n_ctx_blocks = int(nblk.sum())
    # the block pool (and so every block table) does not depend on with_append
    T_planned = 16384 if cfg.name == "large" else 0
    T_append = T_planned if with_append else 0
    n_extra = -(-(T_planned * 5 // 4) // B) if T_planned else 0
    if cfg.name == "tiny":
        pool = 16
    else:
        pool = n_ctx_blocks + n_extra
    assert pool >= n_ctx_blocks + n_extra
    perm = rng.permutation(pool).astype(np.uint32)
    bt = np.full((S, Nb), UNUSED_BLOCK, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += int(nblk[s])
    free_blocks = perm[pos:]

    outliers = None
    if cfg.name == "long":
        n_out = int(round(0.01 * Hk * D))
        ch = rng.choice(Hk * D, size=n_out, replace=False)
        outliers = np.stack([ch // D, ch % D], axis=1).astype(np.int64)

    q = np.empty((S, H, D), dtype=np.float32)
    _fill_normal(q, (cfg.seed, _S_Q), 1.0)

    # context rows, sequence-major; slot of token t of seq s = block_tables[s, t//B]*B + t%B
    offs = np.concatenate([[0], np.cumsum(c.astype(np.int64))])
    T = int(offs[-1])
    slots = np.empty(T, dtype=np.uint32)
    row_seq = np.empty(T, dtype=np.int32)
    for s in range(S):
        t = np.arange(int(c[s]), dtype=np.int64)
        slots[offs[s]:offs[s + 1]] = (bt[s, t // B].astype(np.int64) * B + t % B).astype(np.uint32)
        row_seq[offs[s]:offs[s + 1]] = s

    key = value = None
    if with_kv:
        key = np.empty((T, Hk, D), dtype=np.float32)
        value = np.empty((T, Hk, D), dtype=np.float32)
        jobs = []
        for s in range(S):
            jobs.append((key[offs[s]:offs[s + 1]], s, True))
            jobs.append((value[offs[s]:offs[s + 1]], s, False))
        with ThreadPoolExecutor(threads or _threads()) as ex:
            list(ex.map(lambda j: _seq_values(cfg, j[0], j[1], j[2], outliers), jobs))

    notes = {}
    if outliers is not None:
        notes["outlier_channels"] = outliers
    if cfg.name == "tiny":
        # 3 PAD rows at seeded positions among 140 writer rows
        n_pad = 3
        pad_pos = np.sort(rng.choice(T + n_pad, size=n_pad, replace=False))
        keep = np.ones(T + n_pad, dtype=bool)
        keep[pad_pos] = False
        slots2 = np.full(T + n_pad, PAD_SLOT, dtype=np.uint32)
        slots2[keep] = slots
        rs2 = np.full(T + n_pad, -1, dtype=np.int32)
        rs2[keep] = row_seq
        if with_kv:
            k2 = np.empty((T + n_pad, Hk, D), dtype=np.float32)
            v2 = np.empty((T + n_pad, Hk, D), dtype=np.float32)
            k2[keep], v2[keep] = key, value
            pad_rng = _rng(cfg.seed, _S_APPEND)
            k2[~keep] = pad_rng.standard_normal((n_pad, Hk, D), dtype=np.float32)
            v2[~keep] = pad_rng.standard_normal((n_pad, Hk, D), dtype=np.float32)
            key, value = k2, v2
        slots, row_seq = slots2, rs2
        notes["pad_rows"] = pad_pos

    append = None
    if T_append:
        row_floats = (H + 2 * Hk) * D
        fused = np.empty((T_append, row_floats), dtype=np.float32)
        chunk = 1024
        def fill(i):
            _fill_normal(fused[i:i + chunk], (cfg.seed, _S_APPEND, i // chunk), 1.0)
        with ThreadPoolExecutor(threads or _threads()) as ex:
            list(ex.map(fill, range(0, T_append, chunk)))
        n_pad = int(round(0.05 * T_append))          # 819
        arng = _rng(cfg.seed, _S_APPEND, 1 << 20)
        pad_pos = arng.choice(T_append, size=n_pad, replace=False)
        free_slots = (free_blocks.astype(np.int64)[:, None] * B + np.arange(B)[None, :]).reshape(-1)
        chosen = arng.choice(free_slots, size=T_append - n_pad, replace=False)
        sm = np.full(T_append, PAD_SLOT, dtype=np.uint32)
        mask = np.ones(T_append, dtype=bool)
        mask[pad_pos] = False
        sm[mask] = chosen.astype(np.uint32)
        append = Append(fused=fused, key_offset=H * D, value_offset=(H + Hk) * D,
                        row_stride=row_floats, slot_mapping=sm)

    return Workload(cfg=cfg, context_lens=c, block_tables=bt, num_blocks=pool, q=q,
                    scale=cfg.scale, key=key, value=value, slot_mapping=slots,
                    row_seq=row_seq, append=append, notes=notes)


def _seq_values(cfg: Config, out: np.ndarray, s: int, is_key: bool, outliers) -> None:
    stream = _S_K if is_key else _S_V
    sigma = 2.0 if cfg.name == "edge" else 1.0
    _fill_normal(out, (cfg.seed, stream, s), sigma)
    if cfg.name == "edge":
        zstream = _S_KZERO if is_key else _S_VZERO
        zero = _rng(cfg.seed, zstream, s).random(out.shape[:2]) < 0.02
        out[zero] = 0.0
    if outliers is not None:
        for h, d in outliers:
            out[:, h, d] *= np.float32(20.0)


def sequence_rows(w: Workload, seqs) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Context rows of the given sequences only: (key, value, slot_mapping).

    Regenerated from the per-sequence generators, so it does not need the
    bulk arrays of `build(..., with_kv=False)`.
    """
    cfg = w.cfg
    B = cfg.block_size
    keys, vals, slots = [], [], []
    outliers = w.notes.get("outlier_channels")
    for s in seqs:
        cs = int(w.context_lens[s])
        k = np.empty((cs, cfg.num_kv_heads, cfg.head_size), dtype=np.float32)
        v = np.empty_like(k)
        _seq_values(cfg, k, int(s), True, outliers)
        _seq_values(cfg, v, int(s), False, outliers)
        t = np.arange(cs, dtype=np.int64)
        keys.append(k)
        vals.append(v)
        slots.append((w.block_tables[s, t // B].astype(np.int64) * B + t % B).astype(np.uint32))
    return np.concatenate(keys), np.concatenate(vals), np.concatenate(slots)


def empty_cache(w: Workload, fill: int = 0) -> np.ndarray:
    """A u32 cache [num_blocks, Hk, B, head_size/4 + 1] filled with `fill`."""
    cfg = w.cfg
    W = cfg.head_size // 4 + 1
    return np.full((w.num_blocks, cfg.num_kv_heads, cfg.block_size, W), fill, dtype=np.uint32)


def query_rows(w: Workload, num_rows: int) -> np.ndarray:
    """Seeded queries for a multi-row causal decode: f32 [S, num_rows, H, D]
    ~ N(0, 1), the rows of the last num_rows positions of each sequence (as
    when a batch of draft tokens is verified in one pass)."""
    cfg = w.cfg
    q = np.empty((cfg.num_seqs, int(num_rows), cfg.num_heads, cfg.head_size), dtype=np.float32)
    _fill_normal(q, (cfg.seed, _S_QROWS, int(num_rows)), 1.0)
    return q


def new_token_rows(w: Workload, num_rows: int) -> tuple[np.ndarray, np.ndarray]:
    """Seeded K and V rows of the newest num_rows tokens of each sequence, as
    a decode step appends them: f32 [S, num_rows, Hk, D] each, ~N(0, 1)."""
    cfg = w.cfg
    shape = (cfg.num_seqs, int(num_rows), cfg.num_kv_heads, cfg.head_size)
    key = np.empty(shape, dtype=np.float32)
    value = np.empty(shape, dtype=np.float32)
    _fill_normal(key, (cfg.seed, _S_NEWKV, int(num_rows), 0), 1.0)
    _fill_normal(value, (cfg.seed, _S_NEWKV, int(num_rows), 1), 1.0)
    return key, value


def algorithmic_decode_bytes(cfg: Config, context_lens: np.ndarray, num_rows: int = 1,
                             cache: str = "q8") -> int:
    """Bytes a decode must move: every context token's K and V vector once
    (q8: head_size code bytes + a 4-byte scale word each; f32: 4 * head_size
    bytes; q8c, the contiguous cache: head_size code bytes + one 4-byte scale
    per 32 codes), q in, out back (one vector per query row and head), the
    block-table entries walked and the context lengths."""
    c = np.minimum(context_lens.astype(np.int64), cfg.max_blocks_per_seq * cfg.block_size)
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    vec = {"q8": D + 4, "f32": 4 * D, "q8c": D + D // 8}[cache]
    kv = int(c.sum()) * Hk * 2 * vec
    qo = 2 * S * int(num_rows) * H * D * 4
    bt = int((-(-c // B)).sum()) * 4
    return kv + qo + bt + S * 4


def algorithmic_writer_bytes(num_kv_heads: int, head_size: int, slot_mapping: np.ndarray) -> int:
    """Bytes a writer call must move: read K and V rows of every non-PAD
    token, write its K and V token vectors, read the slot mapping."""
    n = int((slot_mapping != PAD_SLOT).sum())
    rd = n * num_kv_heads * head_size * 4 * 2
    wr = n * num_kv_heads * (head_size + 4) * 2
    return rd + wr + slot_mapping.size * 4


def subset(w: Workload, n_seqs: int) -> Workload:
    """The first n_seqs sequences of a workload with a compact block pool
    (their blocks renumbered in pool order) and, if present, the matching
    share of the append rows redirected into fresh free blocks.  Used for
    small profiling captures of the same kernels."""
    cfg = w.cfg
    B = cfg.block_size
    n = int(n_seqs)
    c = w.context_lens[:n].copy()
    bt_old = w.block_tables[:n]
    used = bt_old[bt_old != UNUSED_BLOCK]
    remap = {int(b): i for i, b in enumerate(np.sort(used))}
    bt = np.full_like(bt_old, UNUSED_BLOCK)
    for s in range(n):
        k = -(-int(c[s]) // B)
        bt[s, :k] = [remap[int(b)] for b in bt_old[s, :k]]
    rows = w.row_seq < n
    rows &= w.row_seq >= 0
    slots = w.slot_mapping[rows].copy()
    slots = np.array([remap[int(sl) // B] * B + int(sl) % B for sl in slots], dtype=np.uint32) \
        if slots.size else slots
    pool = len(remap)
    append = None
    if w.append is not None:
        a = w.append
        T = max(1, a.num_tokens * n // cfg.num_seqs)
        sm = a.slot_mapping[:T].copy()
        live = sm != PAD_SLOT
        extra = -(-int(live.sum()) // B)
        sm[live] = (pool * B + np.random.default_rng([cfg.seed, 7]).permutation(extra * B)[:int(live.sum())]
                    ).astype(np.uint32)
        append = Append(fused=a.fused[:T], key_offset=a.key_offset, value_offset=a.value_offset,
                        row_stride=a.row_stride, slot_mapping=sm)
        pool += extra
    sub_cfg = Config(cfg.name, cfg.index, n, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, B,
                     cfg.max_context, cfg.description + f" (first {n} sequences)")
    return Workload(cfg=sub_cfg, context_lens=c, block_tables=bt, num_blocks=pool, q=w.q[:n].copy(),
                    scale=w.scale, key=None if w.key is None else w.key[rows],
                    value=None if w.value is None else w.value[rows], slot_mapping=slots,
                    row_seq=w.row_seq[rows].copy(), append=append, notes=dict(w.notes))
