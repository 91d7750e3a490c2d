"""A block pool larger than 2^32 cache words: 1.1 M blocks x 8 kv heads x 16
tokens x 33 words is 4.6e9 words (18.6 GB) per cache, so the blocks at the
top of the pool sit past every 32-bit word offset.  The writer and the decode
on those blocks must give the same words and the same output bits as the
same tokens in a compact pool, and the output must match the oracle
(|gpu - oracle| <= 1e-5 + 1e-4 |oracle|).  A slot and a block id one past the
pool's end are flagged and skipped."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

PAD = 0xFFFFFFFF


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


def test_blocks_past_32bit_word_offsets():
    import torch
    import int8_paged_kv_gb300 as pk
    import oracle
    from tests.gpu_helpers import assert_close, device_status
    H, Hk, D, B = 32, 8, 128, 16
    W = D // 4 + 1
    NB = 1_100_000
    assert NB * Hk * B * W > 2 ** 32
    lens = [100, 1000, 333, 4096]
    S = len(lens)
    rng = np.random.default_rng(32)
    nblk = [-(-c // B) for c in lens]
    total = sum(nblk)
    Nb = max(nblk)
    big_ids = (NB - 1 - rng.permutation(total)).astype(np.int64)     # the top of the pool, shuffled
    big_ids[:3] = [0, 7, 123_456]                                      # and a few low ones
    bt_big = np.full((S, Nb), PAD, dtype=np.uint32)
    bt_small = np.full((S, Nb), PAD, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt_big[s, :nblk[s]] = big_ids[pos:pos + nblk[s]]
        bt_small[s, :nblk[s]] = np.arange(pos, pos + nblk[s])
        pos += nblk[s]
    tok = [(s, t) for s in range(S) for t in range(lens[s])]
    slots_big = np.array([int(bt_big[s, t // B]) * B + t % B for s, t in tok], dtype=np.uint32)
    slots_small = np.array([int(bt_small[s, t // B]) * B + t % B for s, t in tok], dtype=np.uint32)
    T = len(tok)
    key = rng.standard_normal((T, Hk * D)).astype(np.float32)
    val = rng.standard_normal((T, Hk * D)).astype(np.float32)
    q = rng.standard_normal((S, H, D)).astype(np.float32)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()

    dk, dv, dq = torch.from_numpy(key).cuda(), torch.from_numpy(val).cuda(), torch.from_numpy(q).cuda()
    device_status(clear=True)
    small_k = torch.zeros((total, Hk, B, W), dtype=torch.int32, device="cuda")
    small_v = torch.zeros_like(small_k)
    pk.pa_q8_reshape_and_cache(dk, dv, small_k, small_v, dev(slots_small), num_kv_heads=Hk, head_size=D,
                               block_size=B)
    big_k = torch.zeros((NB, Hk, B, W), dtype=torch.int32, device="cuda")
    big_v = torch.zeros_like(big_k)
    pk.pa_q8_reshape_and_cache(dk, dv, big_k, big_v, dev(slots_big), num_kv_heads=Hk, head_size=D, block_size=B)
    ids = torch.from_numpy(big_ids).cuda()
    assert torch.equal(big_k.index_select(0, ids), small_k)
    assert torch.equal(big_v.index_select(0, ids), small_v)
    assert device_status(clear=True) == 0

    cl = dev(np.array(lens, dtype=np.uint32))
    out_small = torch.full_like(dq, float("nan"))
    out_big = torch.full_like(dq, float("nan"))
    scale = float(np.float32(D ** -0.5))
    for kernel in (2, 1):
        pk.pa_q8_decode(out_small, dq, small_k, small_v, dev(bt_small), cl, num_kv_heads=Hk, block_size=B,
                        scale=scale, kernel=kernel)
        pk.pa_q8_decode(out_big, dq, big_k, big_v, dev(bt_big), cl, num_kv_heads=Hk, block_size=B,
                        scale=scale, kernel=kernel)
        torch.cuda.synchronize()
        assert torch.equal(out_big, out_small), f"kernel {kernel}"
    assert device_status(clear=True) == 0
    want = oracle.decode(q, small_k.cpu().numpy().view(np.uint32), small_v.cpu().numpy().view(np.uint32),
                         bt_small, np.array(lens, dtype=np.uint32), num_kv_heads=Hk, block_size=B, scale=scale)
    assert_close(out_big.cpu().numpy().astype(np.float64), want, "blocks past 2^32 words")

    # one past the end: a slot (writer) and a block id (decode) are flagged and skipped
    before = big_k[NB - 1].clone()
    bad_slots = slots_big[:2].copy()
    bad_slots[1] = NB * B
    pk.pa_q8_reshape_and_cache(dk[:2], dv[:2], big_k, big_v, dev(bad_slots), num_kv_heads=Hk, head_size=D,
                               block_size=B)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_SLOT
    assert torch.equal(big_k[NB - 1], before)
    bt_bad = bt_big.copy()
    bt_bad[0, 0] = NB
    pk.pa_q8_decode(out_big, dq, big_k, big_v, dev(bt_bad), cl, num_kv_heads=Hk, block_size=B, scale=scale)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_BLOCK
    del big_k, big_v
    torch.cuda.empty_cache()
