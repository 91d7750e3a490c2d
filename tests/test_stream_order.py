"""The writer and the decode back to back on one stream, no host sync between:
the writer overwrites every sequence's newest tokens and the decode's prep
and attention kernels (programmatic dependents, started while the writer's
last wave runs) must read the new words.  Outputs against the oracle over the
caches with the new rows; a decode that ran ahead of the writer would see the
old rows and miss the bound by far."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


@pytest.mark.parametrize("R", [1, 3])
def test_writer_then_decode_without_sync(R):
    import torch
    import oracle
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import (assert_close, dev_u32, device_status, oracle_decode_rows,
                                   random_case)
    S, H, Hk, D, B, NEW = 512, 16, 2, 128, 16, 16       # 1024 (sequence, kv head) units: ordered
    rng = np.random.default_rng(40 + R)
    lens = [int(x) for x in rng.integers(NEW + 1, 97, size=S)]
    w, ok_, ov_, kc, vc = random_case(S, H, Hk, D, B, lens, seed=41 + R)
    bt = w.block_tables
    new_slots = np.array([int(bt[s, t // B]) * B + t % B for s, c in enumerate(lens) for t in range(c - NEW, c)],
                         dtype=np.uint32)
    q = rng.standard_normal((S, R, H, D)).astype(np.float32)
    qd, btd, cld = torch.from_numpy(q).cuda(), dev_u32(bt), dev_u32(w.context_lens)
    out = torch.full_like(qd, float("nan"))
    ws = torch.empty(max(16, pk.pa_q8_decode_rows_workspace_size(S, R, H, Hk, D, B, bt.shape[1])),
                     dtype=torch.uint8, device="cuda")
    sd = dev_u32(new_slots)
    for rep in range(3):
        nk = (rng.standard_normal((S * NEW, Hk * D)) * (2.0 + rep)).astype(np.float32)
        nv = (rng.standard_normal((S * NEW, Hk * D)) * (2.0 + rep)).astype(np.float32)
        oracle.reshape_and_cache(nk, nv, ok_, ov_, new_slots, num_kv_heads=Hk, head_size=D, block_size=B)
        want = oracle_decode_rows(w, ok_, ov_, q)
        kd, vd = torch.from_numpy(nk).cuda(), torch.from_numpy(nv).cuda()
        torch.cuda.synchronize()
        pk.pa_q8_reshape_and_cache(kd, vd, kc, vc, sd, num_kv_heads=Hk, head_size=D, block_size=B)
        pk.pa_q8_decode_rows(out, qd, kc, vc, btd, cld, num_kv_heads=Hk, block_size=B, scale=w.scale,
                             num_blocks=w.num_blocks, workspace=ws)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy().astype(np.float64), want, f"rep {rep}")
    assert device_status() == 0
