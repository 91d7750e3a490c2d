"""Fused append + decode (pa_q8_decode_append) against the oracle applied in
the order the pages give (append, then attend): oracle.reshape_and_cache of
the new rows into the newest positions, then oracle.decode_rows.  The whole
cache must match bit for bit after the call and every output within
|gpu - oracle| <= 1e-5 + 1e-4 |oracle|; the fused step must also equal the
library's own writer-then-decode sequence bit for bit."""
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


def _new_slots(w, R):
    """Slot of new row (s, b): position min(c, cap) - R + b; PAD when that is
    negative or its block id is out of the pool."""
    B = w.cfg.block_size
    cap = w.cfg.max_blocks_per_seq * B
    S = w.context_lens.size
    slots = np.full((S, R), wl.PAD_SLOT, dtype=np.uint32)
    for s in range(S):
        c = min(int(w.context_lens[s]), cap)
        for b in range(R):
            p = c - R + b
            blk = int(w.block_tables[s, p // B]) if p >= 0 else -1
            if 0 <= blk < w.num_blocks:           # a bad block id: not written
                slots[s, b] = blk * B + p % B
    return slots.reshape(-1)


def _oracle_step(w, ok_, ov_, q, key, value, cl=None):
    import oracle
    S, R = q.shape[:2]
    k2, v2 = ok_.copy(), ov_.copy()
    oracle.reshape_and_cache(key.reshape(S * R, -1), value.reshape(S * R, -1), k2, v2, _new_slots(w, R),
                             num_kv_heads=w.cfg.num_kv_heads, head_size=w.cfg.head_size,
                             block_size=w.cfg.block_size)
    out = oracle.decode_rows(q, k2, v2, w.block_tables, w.context_lens if cl is None else cl,
                             num_kv_heads=w.cfg.num_kv_heads, block_size=w.cfg.block_size, scale=w.scale)
    return out, k2, v2


def _gpu_step(w, kc, vc, q, key, value, *, kernel=0, partition_tokens=0):
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32
    qd = torch.from_numpy(q).cuda()
    out = torch.full_like(qd, float("nan"))
    kd = torch.from_numpy(key).cuda() if isinstance(key, np.ndarray) else key
    vd = torch.from_numpy(value).cuda() if isinstance(value, np.ndarray) else value
    pk.pa_q8_decode_append(out, qd, kd, vd, kc, vc, dev_u32(w.block_tables), dev_u32(w.context_lens),
                           num_kv_heads=w.cfg.num_kv_heads, block_size=w.cfg.block_size, scale=w.scale,
                           num_blocks=w.num_blocks, kernel=kernel, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def _case(lens, H=8, Hk=2, D=128, B=16, seed=3):
    from tests.gpu_helpers import random_case
    return random_case(len(lens), H, Hk, D, B, lens, seed=seed)


def _rows(S, R, Hk, D, seed):
    rng = np.random.default_rng(seed)
    key = rng.standard_normal((S, R, Hk, D)).astype(np.float32)
    value = rng.standard_normal((S, R, Hk, D)).astype(np.float32)
    key[0, 0, 0] = 0.0                           # an all-zero vector: scale word 1.0
    return key, value


@pytest.mark.parametrize("kernel", [TC, CC])
@pytest.mark.parametrize("R", [1, 3])
@pytest.mark.parametrize("pt", [0, 128])
def test_fused_step_matches_oracle(kernel, R, pt):
    """Ragged contexts incl. 0, 1, 2 (some new rows have no position), new
    tokens straddling a 128-token partition boundary (c = 129, 130)."""
    from tests.gpu_helpers import assert_close, dev_u32, device_status, host_u32
    lens = [129, 130, 1, 2, 0, 700, 16, 33, 1000, 257]
    w, ok_, ov_, _, _ = _case(lens, seed=R + 10 * kernel)
    S, H, Hk, D = len(lens), 8, 2, 128
    q = np.random.default_rng(R).standard_normal((S, R, H, D)).astype(np.float32)
    key, value = _rows(S, R, Hk, D, seed=R + 1)
    want, wk, wv = _oracle_step(w, ok_, ov_, q, key, value)
    kc, vc = dev_u32(ok_), dev_u32(ov_)
    got = _gpu_step(w, kc, vc, q, key, value, kernel=kernel, partition_tokens=pt)
    assert np.array_equal(host_u32(kc), wk), "K cache words"
    assert np.array_equal(host_u32(vc), wv), "V cache words"
    assert_close(got, want, f"kernel {kernel} R {R} pt {pt}")
    assert device_status() == 0


@pytest.mark.parametrize("kernel", [TC, CC])
def test_fused_step_equals_writer_then_decode(kernel):
    """Same words and the same output bits as pa_q8_reshape_and_cache followed
    by pa_q8_decode_rows; strided new rows (column slices of fused rows)."""
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, gpu_decode_rows, host_u32
    lens = [300, 17, 4095, 64, 1]
    H, Hk, D, R = 16, 4, 64, 2
    w, ok_, ov_, _, _ = _case(lens, H=H, Hk=Hk, D=D, B=32, seed=7)
    S = len(lens)
    rng = np.random.default_rng(8)
    fused = torch.from_numpy(rng.standard_normal((S * R, (H + 2 * Hk) * D + 12)).astype(np.float32)).cuda()
    key = fused[:, H * D:(H + Hk) * D]
    value = fused[:, (H + Hk) * D:(H + 2 * Hk) * D]
    q = rng.standard_normal((S, R, H, D)).astype(np.float32)
    kc1, vc1 = dev_u32(ok_), dev_u32(ov_)
    got = _gpu_step(w, kc1, vc1, q, key, value, kernel=kernel)
    kc2, vc2 = dev_u32(ok_), dev_u32(ov_)
    pk.pa_q8_reshape_and_cache(key, value, kc2, vc2, dev_u32(_new_slots(w, R)), num_kv_heads=Hk,
                               head_size=D, block_size=32)
    ref = gpu_decode_rows(w, kc2, vc2, q, kernel=kernel)
    assert np.array_equal(host_u32(kc1), host_u32(kc2)) and np.array_equal(host_u32(vc1), host_u32(vc2))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("D", [64, 256])
def test_head_sizes(D):
    from tests.gpu_helpers import assert_close, dev_u32, host_u32
    lens = [31, 33, 1, 90]
    H, Hk, R = 16, 1, 2
    w, ok_, ov_, _, _ = _case(lens, H=H, Hk=Hk, D=D, B=32, seed=D)
    q = np.random.default_rng(D).standard_normal((len(lens), R, H, D)).astype(np.float32)
    key, value = _rows(len(lens), R, Hk, D, seed=D)
    want, wk, wv = _oracle_step(w, ok_, ov_, q, key, value)
    kc, vc = dev_u32(ok_), dev_u32(ov_)
    got = _gpu_step(w, kc, vc, q, key, value)
    assert np.array_equal(host_u32(kc), wk) and np.array_equal(host_u32(vc), wv)
    assert_close(got, want, f"D {D}")


def test_bad_block_of_a_new_token_is_flagged_and_not_written():
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, device_status, host_u32
    lens = [40, 40]
    w, ok_, ov_, _, _ = _case(lens, seed=9)
    w.block_tables = w.block_tables.copy()
    w.block_tables[1, 2] = 1 << 30               # the block of sequence 1's newest token
    q = np.random.default_rng(9).standard_normal((2, 1, 8, 128)).astype(np.float32)
    key, value = _rows(2, 1, 2, 128, seed=9)
    kc, vc = dev_u32(ok_), dev_u32(ov_)
    device_status(clear=True)
    _gpu_step(w, kc, vc, q, key, value)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_BLOCK
    # sequence 0's new token written, nothing else changed
    slot0 = int(_new_slots(w, 1)[0])
    gk = host_u32(kc)
    changed = np.argwhere(np.any(gk != ok_, axis=-1))
    assert all(int(b) * 16 + int(t) == slot0 for b, _, t in changed) and len(changed) >= 1


def test_large_batch_sampled():
    """The large-batch workload: one new token per sequence, automatic plan,
    new tokens' words bit for bit, sampled outputs against the oracle."""
    import oracle
    from tests.gpu_helpers import assert_close, dev_u32, device_status, host_u32, oracle_write, poisoned_cache
    w = wl.build("large", with_append=False)
    ok_, ov_ = poisoned_cache(w), poisoned_cache(w)
    oracle_write(w.key, w.value, w.slot_mapping, ok_, ov_, w.cfg)
    w.key = w.value = None
    cfg = w.cfg
    S, H, Hk, D = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size
    q = wl.query_rows(w, 1)
    key, value = _rows(S, 1, Hk, D, seed=11)
    slots = _new_slots(w, 1)
    wk, wv = ok_.copy(), ov_.copy()
    oracle.reshape_and_cache(key.reshape(S, -1), value.reshape(S, -1), wk, wv, slots,
                             num_kv_heads=Hk, head_size=D, block_size=cfg.block_size)
    kc, vc = dev_u32(ok_), dev_u32(ov_)
    got = _gpu_step(w, kc, vc, q, key, value)
    assert np.array_equal(host_u32(kc), wk) and np.array_equal(host_u32(vc), wv)
    rng = np.random.default_rng(12)
    picks = sorted({(int(rng.integers(S)), int(rng.integers(H))) for _ in range(80)} |
                   {(int(np.argmax(w.context_lens)), 0)})
    rows = np.array(picks, dtype=np.int32)
    want = oracle.decode(np.ascontiguousarray(q[:, 0]), wk, wv, w.block_tables, w.context_lens,
                         num_kv_heads=Hk, block_size=cfg.block_size, scale=w.scale, rows=rows)
    assert_close(got[rows[:, 0], 0, rows[:, 1]], want, "large fused step")
    assert device_status() == 0


@pytest.mark.parametrize("kernel", [3, 0])
def test_fused_step_on_tcgen05(kernel):
    """The tcgen05 family (asked for, and chosen automatically from 24 (row,
    head) pairs per kv head on: R = 8 rows x 8 heads) stores the new tokens too."""
    from tests.gpu_helpers import assert_close, dev_u32, device_status, host_u32
    import int8_paged_kv_gb300 as pk
    lens = [129, 1, 0, 700, 64, 2000]
    S, H, Hk, D, R = len(lens), 16, 2, 128, 8
    w, ok_, ov_, _, _ = _case(lens, H=H, Hk=Hk, D=D, seed=31)
    q = np.random.default_rng(31).standard_normal((S, R, H, D)).astype(np.float32)
    key, value = _rows(S, R, Hk, D, seed=32)
    want, wk, wv = _oracle_step(w, ok_, ov_, q, key, value)
    kc, vc = dev_u32(ok_), dev_u32(ov_)
    got = _gpu_step(w, kc, vc, q, key, value, kernel=kernel)
    assert np.array_equal(host_u32(kc), wk), "K cache words"
    assert np.array_equal(host_u32(vc), wv), "V cache words"
    assert_close(got, want, f"kernel {kernel}")
    assert device_status() == 0
