"""GPU writer (pa_q8_reshape_and_cache) against the oracle: every cache word
bit for bit, on all five workloads and on edge inputs."""
import numpy as np
import pytest

from int8_paged_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CONFIGS = list(wl.CONFIGS)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_paged_kv_gb300 import build
    build.build()
    import oracle
    oracle.build()


@pytest.mark.parametrize("name", CONFIGS)
def test_context_build_bit_exact(name):
    from tests.gpu_helpers import device_status, gpu_write, host_u32, oracle_write, poisoned_cache
    w = wl.build(name, with_append=False)
    cfg = w.cfg
    ok_, ov_ = poisoned_cache(w), poisoned_cache(w)
    oracle_write(w.key, w.value, w.slot_mapping, ok_, ov_, cfg)
    kc, vc = gpu_write(w.key, w.value, w.slot_mapping, poisoned_cache(w), poisoned_cache(w), cfg)
    gk, gv = host_u32(kc), host_u32(vc)
    assert np.array_equal(gk, ok_), f"{name}: {int((gk != ok_).sum())} K words differ"
    assert np.array_equal(gv, ov_), f"{name}: {int((gv != ov_).sum())} V words differ"
    assert device_status() == 0


def test_large_append_strided_with_pad():
    """16384 rows whose K/V are column slices of fused rows (stride 10240),
    5% PAD, scattered into free slots of a populated cache."""
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, device_status, host_u32, poisoned_cache
    import oracle
    w = wl.build("large", with_kv=False)
    a, cfg = w.append, w.cfg
    base_k = poisoned_cache(w, 0x5A5A5A5A)
    base_v = poisoned_cache(w, 0x5A5A5A5A)
    ok_, ov_ = base_k.copy(), base_v.copy()
    oracle.reshape_and_cache(a.key_view(), a.value_view(), ok_, ov_, a.slot_mapping,
                             num_kv_heads=cfg.num_kv_heads, head_size=cfg.head_size,
                             block_size=cfg.block_size)
    fused = torch.from_numpy(a.fused).cuda()
    kc, vc = dev_u32(base_k), dev_u32(base_v)
    pk.pa_q8_reshape_and_cache(fused[:, a.key_offset:a.value_offset],
                               fused[:, a.value_offset:a.value_offset + (a.value_offset - a.key_offset)],
                               kc, vc, dev_u32(a.slot_mapping), num_kv_heads=cfg.num_kv_heads,
                               head_size=cfg.head_size, block_size=cfg.block_size)
    assert np.array_equal(host_u32(kc), ok_)
    assert np.array_equal(host_u32(vc), ov_)
    # PAD rows and unmapped slots untouched
    assert (a.slot_mapping == wl.PAD_SLOT).sum() == 819
    assert device_status() == 0


@pytest.mark.parametrize("D", [64, 128, 256])
def test_edge_values_and_unaligned_rows(D):
    """Zero vectors (scale word 1.0), half-way products, huge and tiny
    magnitudes, a subnormal amax (127/amax overflows), rows that start off a
    16-byte boundary (scalar-load kernel)."""
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, host_u32
    import oracle
    rng = np.random.default_rng(D)
    Hk, B, nb, T = 3, 8, 12, 64
    rows = rng.standard_normal((T, Hk, D)).astype(np.float32)
    rows[0] = 0.0
    rows[1] = (rng.integers(-254, 255, (Hk, D)) / 128.0).astype(np.float32)
    rows[1, :, 0] = 254 / 128.0
    rows[2] *= np.float32(1e30)
    rows[3] *= np.float32(1e-30)
    rows[4] = 0.0
    rows[4, :, 5] = np.float32(1e-40)           # subnormal amax
    rows[4, :, 6] = np.float32(-5e-41)
    rows[5, :, :] = rng.standard_normal((Hk, D)).astype(np.float32)
    rows[5, :, 7] *= 20
    slots = rng.choice(nb * B, size=T, replace=False).astype(np.uint32)
    slots[[9, 33]] = wl.PAD_SLOT
    W = D // 4 + 1
    for offset in (0, 1):                       # 1 float = 4 bytes off alignment
        buf = np.zeros((T, Hk * D + 3), dtype=np.float32)
        buf[:, offset:offset + Hk * D] = rows.reshape(T, -1)
        view = buf[:, offset:offset + Hk * D]
        ok_ = np.full((nb, Hk, B, W), 0xA5A5A5A5, dtype=np.uint32)
        ov_ = ok_.copy()
        oracle.reshape_and_cache(view, view, ok_, ov_, slots, num_kv_heads=Hk, head_size=D,
                                 block_size=B)
        dbuf = torch.from_numpy(buf).cuda()
        dview = dbuf[:, offset:offset + Hk * D]
        kc = dev_u32(np.full_like(ok_, 0xA5A5A5A5))
        vc = dev_u32(np.full_like(ok_, 0xA5A5A5A5))
        pk.pa_q8_reshape_and_cache(dview, dview, kc, vc, dev_u32(slots), num_kv_heads=Hk,
                                   head_size=D, block_size=B)
        assert np.array_equal(host_u32(kc), ok_), f"offset {offset}"
        assert np.array_equal(host_u32(vc), ov_), f"offset {offset}"
    zero = ok_[slots[0] // B, :, slots[0] % B]
    assert np.all(zero[:, :-1] == 0) and np.all(zero[:, -1] == 0x3F800000)


def test_bad_slot_is_skipped_and_flagged():
    import torch
    import int8_paged_kv_gb300 as pk
    from tests.gpu_helpers import dev_u32, device_status, host_u32
    Hk, D, B, nb, T = 2, 64, 16, 4, 8
    rows = torch.randn(T, Hk * D, device="cuda")
    slots = np.arange(T, dtype=np.uint32)
    slots[3] = nb * B + 5                        # out of range: must be skipped, never written
    W = D // 4 + 1
    init = np.full((nb, Hk, B, W), 0x11111111, dtype=np.uint32)
    kc, vc = dev_u32(init), dev_u32(init)
    device_status(clear=True)
    pk.pa_q8_reshape_and_cache(rows, rows, kc, vc, dev_u32(slots), num_kv_heads=Hk, head_size=D,
                               block_size=B)
    assert device_status(clear=True) & pk.PA_Q8_DEV_BAD_SLOT
    got = host_u32(kc)
    written = np.zeros((nb, Hk, B), dtype=bool)
    for i, s in enumerate(slots):
        if i != 3:
            written[s // B, :, s % B] = True
    assert np.all(got[~written] == 0x11111111)
    assert device_status() == 0
