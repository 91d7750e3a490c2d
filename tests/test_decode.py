"""GPU decode (pa_q8_decode) against the fp64 oracle:
|gpu - oracle| <= 1e-5 + 1e-4 |oracle| elementwise, for both kernel
families, on all five workloads (full-size ones on sampled rows, in the
launch configuration the benchmark times), and on edge cases: empty and
one-token contexts, ragged tails next to poisoned (NaN) cache words,
clamped contexts, every supported block size, GQA ratios 1..32, partition
sizes, a block id out of range, and the bounded-wait path."""
import numpy as np
import pytest

from int8_paged_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TC, CC = 2, 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


_CACHE = {}


def _setup(name):
    """Workload, oracle-written caches (numpy) and GPU-written caches (device)."""
    if name in _CACHE:
        return _CACHE[name]
    from tests.gpu_helpers import gpu_write, host_u32, oracle_write, poisoned_cache
    w = wl.build(name, with_append=False)
    cfg = w.cfg
    ok_, ov_ = poisoned_cache(w), poisoned_cache(w)
    oracle_write(w.key, w.value, w.slot_mapping, ok_, ov_, cfg)
    kc, vc = gpu_write(w.key, w.value, w.slot_mapping, poisoned_cache(w), poisoned_cache(w), cfg)
    assert np.array_equal(host_u32(kc), ok_) and np.array_equal(host_u32(vc), ov_)
    w.key = w.value = None                      # free host memory
    _CACHE.clear()
    _CACHE[name] = (w, ok_, ov_, kc, vc)
    return _CACHE[name]


def _rows(w, n, seed=0):
    """n sampled (s, h) rows, always including the longest and shortest contexts."""
    rng = np.random.default_rng(seed)
    S, H = w.cfg.num_seqs, w.cfg.num_heads
    pick = {(int(np.argmax(w.context_lens)), 0), (int(np.argmin(w.context_lens)), H - 1)}
    while len(pick) < min(n, S * H):
        pick.add((int(rng.integers(S)), int(rng.integers(H))))
    return np.array(sorted(pick), dtype=np.int32)


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("name", ["tiny", "llama8b", "edge"])
def test_small_configs_all_rows(name, kernel):
    from tests.gpu_helpers import assert_close, device_status, gpu_decode, oracle_decode
    w, ok_, ov_, kc, vc = _setup(name)
    want = oracle_decode(w, ok_, ov_)
    got = gpu_decode(w, kc, vc, kernel=kernel)
    assert_close(got, want, f"{name} kernel {kernel}")
    assert device_status() == 0


@pytest.mark.parametrize("kernel", [0, TC, CC])
@pytest.mark.parametrize("name", ["long", "large"])
def test_full_size_sampled_rows(name, kernel):
    """Full-size workloads in the benchmark's launch configuration (kernel 0 =
    the automatic plan); the oracle checks sampled rows."""
    from tests.gpu_helpers import assert_close, device_status, gpu_decode, oracle_decode
    w, ok_, ov_, kc, vc = _setup(name)
    rows = _rows(w, 48 if name == "long" else 160, seed=kernel)
    want = oracle_decode(w, ok_, ov_, rows=rows)
    got = gpu_decode(w, kc, vc, kernel=kernel)
    assert_close(got[rows[:, 0], rows[:, 1]], want, f"{name} kernel {kernel}")
    assert device_status() == 0


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("pt", [128, 256, 1024, 4096])
def test_partition_invariance(kernel, pt):
    """The split-context partition size changes nothing beyond tolerance."""
    from tests.gpu_helpers import assert_close, gpu_decode, oracle_decode
    w, ok_, ov_, kc, vc = _setup("llama8b")
    want = oracle_decode(w, ok_, ov_)
    got = gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt)
    assert_close(got, want, f"pt {pt}")


def _random_case(*args, **kw):
    from tests.gpu_helpers import random_case
    return random_case(*args, **kw)


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("B", [4, 8, 16, 32, 64, 128, 256])
def test_block_sizes_and_ragged_tails(kernel, B):
    from tests.gpu_helpers import assert_close, gpu_decode, oracle_decode
    lens = [1, B - 1, B + 1, 3 * B + 7, 700, 129, 0, 2 * B]
    w, ok_, ov_, kc, vc = _random_case(len(lens), 8, 2, 128, B, lens, seed=B)
    want = oracle_decode(w, ok_, ov_)
    for pt in (0, 128, 384):
        got = gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt)
        assert_close(got, want, f"B {B} pt {pt}")
        assert np.all(got[6] == 0.0)              # empty context -> zero rows


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("H,Hk,D", [(4, 4, 64), (8, 4, 64), (12, 1, 128), (16, 2, 128),
                                    (32, 1, 128), (16, 1, 256), (8, 8, 256), (24, 2, 64)])
def test_gqa_ratios_and_head_sizes(kernel, H, Hk, D):
    from tests.gpu_helpers import assert_close, gpu_decode, oracle_decode
    lens = [1, 17, 300, 1000]
    w, ok_, ov_, kc, vc = _random_case(4, H, Hk, D, 16, lens, seed=H * 7 + Hk + D)
    want = oracle_decode(w, ok_, ov_)
    for pt in (0, 256):
        assert_close(gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt), want,
                     f"H {H} Hk {Hk} D {D} pt {pt}")


@pytest.mark.parametrize("kernel", [TC, CC])
def test_clamped_context_and_value_ranges(kernel):
    """context_len beyond max_blocks*B is clamped; large and tiny value
    magnitudes and sharp softmax (scale x 30) stay within tolerance."""
    from tests.gpu_helpers import assert_close_scaled, f32_units, gpu_decode, oracle_decode
    lens = [64, 208, 50]                                   # 208 = max_blocks_per_seq * 16
    for dist, sm in ((1.0, 1.0), (1e3, 1e-3), (1e-3, 1e3), (1.0, 30.0)):
        w, ok_, ov_, kc, vc = _random_case(3, 8, 2, 128, 16, lens, seed=5, scale_mult=sm, dist=dist)
        cl = np.array([64, 10_000, 50], dtype=np.uint32)   # seq 1 clamps to 208
        want = oracle_decode(w, ok_, ov_, cl=cl)
        got = gpu_decode(w, kc, vc, kernel=kernel, cl=cl)
        # values N(0, dist^2), logits sigma dist * sm: beyond the workloads'
        # ranges the absolute part of the bound grows with sigma_v * sigma_z
        assert_close_scaled(got, want, f32_units(dist, dist * sm), f"dist {dist} scale x{sm}")


@pytest.mark.parametrize("kernel", [TC, CC])
def test_bad_block_id_is_skipped_and_flagged(kernel):
    from tests.gpu_helpers import device_status, gpu_decode
    import int8_paged_kv_gb300 as pk
    w, ok_, ov_, kc, vc = _random_case(2, 8, 2, 128, 16, [40, 40], seed=9)
    bt = w.block_tables.copy()
    bt[1, 1] = 1 << 30                         # inside the context, out of the pool
    device_status(clear=True)
    out = gpu_decode(w, kc, vc, kernel=kernel, bt=bt)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_BLOCK
    # sequence 0 is unaffected
    from tests.gpu_helpers import assert_close, oracle_decode
    want = oracle_decode(w, ok_, ov_)
    assert_close(out[0], want[0], "untouched sequence")


def test_bounded_wait_gives_up_and_context_survives():
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import device_status
    device_status(clear=True)
    pk.pa_q8_selftest_wait_timeout(2000)       # 2 ms on a barrier nothing releases
    torch.cuda.synchronize()
    assert device_status(clear=True) & pk.PA_Q8_DEV_WAIT_TIMEOUT
    x = torch.ones(1024, device="cuda")
    assert float((x * 2).sum()) == 2048.0      # the context still works
    assert device_status() == 0


def test_plan_is_what_the_benchmark_times():
    import int8_paged_kv_gb300 as pk
    cfg = wl.CONFIGS["large"]
    plan = pk.pa_q8_decode_plan(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size,
                                cfg.block_size, cfg.max_blocks_per_seq)
    assert plan["kernel"] in (TC, CC) and plan["partition_tokens"] % 128 == 0
    assert plan["num_partitions"] * plan["partition_tokens"] >= cfg.max_context


@pytest.mark.parametrize("S", [300, 1500, 9000])
def test_prep_orders_sequences_longest_first(S):
    """The order the prep kernel leaves at the start of the workspace (one
    u64 per sequence: clamped length << 32 | sequence) is longest first, ties
    by sequence index, for batches it ranks (<= 1024) and sorts (<= 8192),
    and the identity beyond; the grid runs sequences in that order."""
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, device_status
    rng = np.random.default_rng(S + 1)
    lens = rng.integers(0, 41, size=S)
    lens[:5] = [40, 40, 0, 40, 33]
    w, ok_, ov_, kc, vc = _random_case(S, 4, 2, 64, 16, lens.tolist(), seed=S)
    cap = w.block_tables.shape[1] * 16                # 48: sequence 3's three blocks are all in the table
    cl = lens.astype(np.uint32)
    cl[3] = 10_000                                   # clamped to the table's capacity
    plan = pk.pa_q8_decode_plan(S, 4, 2, 64, 16, w.block_tables.shape[1], kernel=TC)
    assert plan["num_ctas"] > 3 * torch.cuda.get_device_properties(0).multi_processor_count   # prep runs
    ws = torch.zeros(pk.pa_q8_decode_workspace_size(S, 4, 2, 64, 16, w.block_tables.shape[1], kernel=TC),
                     dtype=torch.uint8, device="cuda")
    q = torch.from_numpy(w.q).cuda()
    pk.pa_q8_decode(torch.empty_like(q), q, kc, vc, dev_u32(w.block_tables), dev_u32(cl),
                    num_kv_heads=2, block_size=16, scale=w.scale, workspace=ws, kernel=TC)
    assert device_status(clear=True) == 0
    keys = ws[:8 * S].cpu().numpy().view(np.uint64)
    seq = (keys & np.uint64(0xFFFFFFFF)).astype(np.int64)
    length = (keys >> np.uint64(32)).astype(np.int64)
    clamped = np.minimum(cl.astype(np.int64), cap)
    assert np.array_equal(np.sort(seq), np.arange(S))
    assert np.array_equal(length, clamped[seq])
    if S <= 8192:
        assert np.array_equal(seq, np.lexsort((np.arange(S), -clamped)))
    else:
        assert np.array_equal(seq, np.arange(S))


@pytest.mark.parametrize("S", [1500, 9000])
def test_many_sequences_take_every_ordering_path(S):
    """More sequences than one prep CTA ranks (sorting network) and more than
    it sorts (identity order): every row still matches the oracle."""
    from tests.gpu_helpers import assert_close, gpu_decode, oracle_decode
    rng = np.random.default_rng(S)
    lens = rng.integers(0, 41, size=S).tolist()
    w, ok_, ov_, kc, vc = _random_case(S, 4, 2, 64, 16, lens, seed=S)
    want = oracle_decode(w, ok_, ov_)
    for kernel in (TC, CC):
        for pt in (0, 128):
            assert_close(gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt), want,
                         f"S {S} kernel {kernel} pt {pt}")


MIXED_LENS = [0, 1, 31, 33, 5000, 20000, 700, 4096, 4097, 12345, 129, 64, 9000, 2, 16384, 333]


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("pt", [0, 256, 1024, 4096])
def test_mixed_per_sequence_splits_against_oracle(kernel, pt):
    """Contexts from empty to 20000 tokens in one batch, so some sequences are
    split into many equal partitions (the 20000-token one into 79 at 256,
    more than the 32 the combine keeps in shared memory), some into two and
    most not at all."""
    from tests.gpu_helpers import assert_close, device_status, gpu_decode, oracle_decode
    lens = MIXED_LENS
    w, ok_, ov_, kc, vc = _random_case(len(lens), 8, 2, 128, 16, lens, seed=32)
    want = oracle_decode(w, ok_, ov_)
    got = gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt)
    assert_close(got, want, f"kernel {kernel} pt {pt}")
    assert np.all(got[0] == 0.0)
    assert device_status() == 0


@pytest.mark.parametrize("R", [2, 5])
def test_mixed_per_sequence_splits_multi_row(R):
    """The same batch with R causal query rows per sequence on every family
    (the automatic plan takes tcgen05 from R * r = 24 pairs on)."""
    from tests.gpu_helpers import (assert_close, device_status, gpu_decode_rows, oracle_decode_rows,
                                   random_case)
    lens = MIXED_LENS
    w, ok_, ov_, kc, vc = random_case(len(lens), 16, 2, 128, 16, lens, seed=33)
    q = np.random.default_rng(R).standard_normal((len(lens), R, 16, 128)).astype(np.float32)
    want = oracle_decode_rows(w, ok_, ov_, q)
    for kernel in (0, CC, TC, 3):
        for pt in (0, 512):
            got = gpu_decode_rows(w, kc, vc, q, kernel=kernel, partition_tokens=pt)
            assert_close(got, want, f"R {R} kernel {kernel} pt {pt}")
    assert device_status() == 0


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("D", [128, 256])
def test_combine_of_many_partitions(kernel, D):
    """A 40000-token context split at 1024 tokens (40 partial records per
    head: the combine fetches a few heads' records per batch into shared
    memory) and at 128 tokens (313 records per head: more than shared memory
    holds, so the combine reads them with vector loads)."""
    from tests.gpu_helpers import assert_close, device_status, gpu_decode, oracle_decode
    lens = [40000, 3000, 0, 1]
    w, ok_, ov_, kc, vc = _random_case(len(lens), 8, 2, D, 32, lens, seed=41 + D)
    want = oracle_decode(w, ok_, ov_)
    for pt in (1024, 128):
        got = gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt)
        assert_close(got, want, f"D {D} kernel {kernel} pt {pt}")
        assert np.all(got[2] == 0.0)
    assert device_status() == 0


# (S, H, Hk, D, B, lens, pt, R): split contexts merged by each route.  The
# plan takes the separate combine grid when the split grid's expected CTAs
# (contexts at half the table's capacity) fit in one wave, else the merge by
# the last CTA of each group (arrival counters, prep kernel).
COMBINE_CASES = {
    # one wave, head size 256, 16-head CTAs (two head tiles): one record per
    # token-slot warp and head tile, every row (split or not) merged by the
    # combine grid, 16 records per row
    "grid_slot_records_256": (6, 16, 1, 256, 32, [0, 1, 33, 700, 3000, 4095], 1024, 1),
    # one wave, two causal rows per sequence (8 pairs per kv head)
    "grid_slot_records_rows": (5, 8, 2, 128, 16, [2, 40, 300, 1500, 2600], 256, 2),
    # one wave, more than 32 records per row (the (m, l) loop past one warp)
    "grid_many_records": (3, 8, 2, 128, 16, [9000, 1, 4000], 512, 1),
    # many waves: the last CTA of each group merges
    "last_cta_merge": (4, 32, 8, 128, 16, [8000, 100, 5000, 0], 128, 1),
}


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("case", sorted(COMBINE_CASES))
def test_split_context_merge_routes(case, kernel):
    """Both merge routes of split contexts against the oracle, on both
    kernel families (the CUDA-core family keeps one record per partition)."""
    from tests.gpu_helpers import (assert_close, device_status, gpu_decode, gpu_decode_rows, oracle_decode,
                                   oracle_decode_rows)
    S, H, Hk, D, B, lens, pt, R = COMBINE_CASES[case]
    w, ok_, ov_, kc, vc = _random_case(S, H, Hk, D, B, lens, seed=70 + len(case))
    if R == 1:
        got = gpu_decode(w, kc, vc, kernel=kernel, partition_tokens=pt)
        want = oracle_decode(w, ok_, ov_)
    else:
        q = np.random.default_rng(71).standard_normal((S, R, H, D)).astype(np.float32)
        got = gpu_decode_rows(w, kc, vc, q, kernel=kernel, partition_tokens=pt)
        want = oracle_decode_rows(w, ok_, ov_, q)
    assert_close(got, want, f"{case} kernel {kernel}")
    for s, c in enumerate(lens):
        if c == 0:
            assert np.all(got[s] == 0.0)
    assert device_status() == 0


@pytest.mark.parametrize("pt,lens", [(256, [1000, 2000, 37]),
                                     (128, [9000, 8800, 8000, 7000, 6600, 6000, 5000, 4400, 4000, 3000, 200, 20])])
def test_split_context_merge_routes_tcgen05(pt, lens):
    """The tcgen05 family (8 causal rows x 8 heads per kv head) on both merge
    routes: three sequences split at 256 tokens fit one wave (combine grid,
    one record per partition); twelve sequences at 128 tokens do not (the
    last CTA of each group merges)."""
    from tests.gpu_helpers import assert_close, device_status, gpu_decode_rows, oracle_decode_rows
    S, H, Hk, D, B, R = len(lens), 8, 1, 128, 16, 8
    w, ok_, ov_, kc, vc = _random_case(S, H, Hk, D, B, lens, seed=90 + pt)
    q = np.random.default_rng(91).standard_normal((S, R, H, D)).astype(np.float32)
    got = gpu_decode_rows(w, kc, vc, q, kernel=3, partition_tokens=pt)
    want = oracle_decode_rows(w, ok_, ov_, q)
    assert_close(got, want, f"tcgen05 pt {pt}")
    assert device_status() == 0
