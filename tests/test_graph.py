"""The library's calls inside a CUDA graph: a serving step (writer, then the
decode with its prep kernel and programmatic-dependent attention launch;
the multi-row and fused-append calls) is captured once on a side stream and
replayed.  Every replay must give the same cache words and the same output
bits as the same calls run eagerly, with new inputs copied into the captured
buffers between replays."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


def _inputs(seed, T, Hk, D):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, Hk * D)).astype(np.float32),
            rng.standard_normal((T, Hk * D)).astype(np.float32))


@pytest.mark.parametrize("kernel,R", [(0, 1), (2, 3), (1, 2), (3, 8)])
def test_step_captured_and_replayed(kernel, R):
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, device_status, random_case
    lens = [700, 1, 33, 2000, 129, 0, 64, 513]
    S, H, Hk, D, B = len(lens), 16, 2, 128, 16
    w, ok_, ov_, kc0, vc0 = random_case(S, H, Hk, D, B, lens, seed=50 + R)
    T = 24
    # the new rows overwrite positions 1600 .. 1623 of sequence 3 (2000 tokens)
    slots = np.array([int(w.block_tables[3, 100 + i // B]) * B + i % B for i in range(T)], dtype=np.uint32)
    bt, cl = dev_u32(w.block_tables), dev_u32(w.context_lens)
    q = torch.from_numpy(np.random.default_rng(R).standard_normal((S, R, H, D)).astype(np.float32)).cuda()
    key = torch.empty((T, Hk * D), device="cuda")
    val = torch.empty_like(key)
    out = torch.empty_like(q)
    ws = torch.empty(pk.pa_q8_decode_rows_workspace_size(S, R, H, Hk, D, B, w.block_tables.shape[1],
                                                         kernel=kernel), dtype=torch.uint8, device="cuda")
    slot_d = dev_u32(slots)

    def step(kc, vc):
        pk.pa_q8_reshape_and_cache(key, val, kc, vc, slot_d, num_kv_heads=Hk, head_size=D, block_size=B)
        pk.pa_q8_decode_rows(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale,
                             num_blocks=w.num_blocks, workspace=ws, kernel=kernel)

    kc, vc = kc0.clone(), vc0.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                     # warm up outside the capture
        k1, v1 = _inputs(1, T, Hk, D)
        key.copy_(torch.from_numpy(k1)); val.copy_(torch.from_numpy(v1))
        step(kc, vc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(kc, vc)
    for rep in range(3):
        kn, vn = _inputs(100 + rep, T, Hk, D)
        key.copy_(torch.from_numpy(kn)); val.copy_(torch.from_numpy(vn))
        kc.copy_(kc0); vc.copy_(vc0)
        g.replay()
        torch.cuda.synchronize()
        got_out, got_k, got_v = out.clone(), kc.clone(), vc.clone()
        # the same step, eagerly
        kc.copy_(kc0); vc.copy_(vc0)
        step(kc, vc)
        torch.cuda.synchronize()
        assert torch.equal(got_k, kc) and torch.equal(got_v, vc), f"rep {rep}: cache words"
        assert torch.equal(got_out, out), f"rep {rep}: output bits"
        assert torch.isfinite(out).all()
    assert device_status() == 0


def test_fused_append_captured_and_replayed():
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, device_status, random_case
    lens = [129, 1, 0, 700, 2000]
    S, H, Hk, D, B, R = len(lens), 8, 2, 128, 16, 2
    w, ok_, ov_, kc0, vc0 = random_case(S, H, Hk, D, B, lens, seed=77)
    bt, cl = dev_u32(w.block_tables), dev_u32(w.context_lens)
    q = torch.from_numpy(np.random.default_rng(3).standard_normal((S, R, H, D)).astype(np.float32)).cuda()
    key = torch.empty((S * R, Hk * D), device="cuda")
    val = torch.empty_like(key)
    out = torch.empty_like(q)
    ws = torch.empty(pk.pa_q8_decode_rows_workspace_size(S, R, H, Hk, D, B, w.block_tables.shape[1]),
                     dtype=torch.uint8, device="cuda")

    def step(kc, vc):
        pk.pa_q8_decode_append(out, q, key, val, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale,
                               num_blocks=w.num_blocks, workspace=ws)

    kc, vc = kc0.clone(), vc0.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        k1, v1 = _inputs(2, S * R, Hk, D)
        key.copy_(torch.from_numpy(k1)); val.copy_(torch.from_numpy(v1))
        step(kc, vc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(kc, vc)
    for rep in range(2):
        kn, vn = _inputs(200 + rep, S * R, Hk, D)
        key.copy_(torch.from_numpy(kn)); val.copy_(torch.from_numpy(vn))
        kc.copy_(kc0); vc.copy_(vc0)
        g.replay()
        torch.cuda.synchronize()
        got_out, got_k = out.clone(), kc.clone()
        kc.copy_(kc0); vc.copy_(vc0)
        step(kc, vc)
        torch.cuda.synchronize()
        assert torch.equal(got_k, kc) and torch.equal(got_out, out), f"rep {rep}"
    assert device_status() == 0
