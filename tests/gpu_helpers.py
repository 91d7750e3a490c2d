"""Shared pieces of the GPU parity tests: moving workloads to the device,
running the library through its binding, and running the oracle on the
same inputs.  u32 buffers travel as int32 tensors (same bits)."""
import numpy as np
import torch

import int8_paged_kv_gb300 as pk
import oracle
from int8_paged_kv_gb300 import workloads as wl

POISON = 0xFFFFFFFF      # a NaN bit pattern: unused cache words must never be read


def dev_u32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def host_u32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def poisoned_cache(w, fill=POISON):
    return wl.empty_cache(w, fill)


def gpu_write(key, value, slots, cache_k, cache_v, cfg, num_blocks=None):
    """Run the writer on device copies; key/value: numpy f32 (2-D row views allowed)."""
    kd = torch.from_numpy(np.ascontiguousarray(key)).cuda() if key.flags.c_contiguous else None
    if kd is None:
        raise ValueError("use gpu_write_rows for strided rows")
    vd = torch.from_numpy(np.ascontiguousarray(value)).cuda()
    kc, vc = dev_u32(cache_k), dev_u32(cache_v)
    pk.pa_q8_reshape_and_cache(kd.reshape(kd.shape[0], -1), vd.reshape(vd.shape[0], -1), kc, vc,
                               dev_u32(slots), num_kv_heads=cfg.num_kv_heads,
                               head_size=cfg.head_size, block_size=cfg.block_size,
                               num_blocks=num_blocks)
    return kc, vc


def oracle_write(key, value, slots, cache_k, cache_v, cfg):
    oracle.reshape_and_cache(key, value, cache_k, cache_v, slots, num_kv_heads=cfg.num_kv_heads,
                             head_size=cfg.head_size, block_size=cfg.block_size)


def gpu_decode(w, kc, vc, *, kernel=0, partition_tokens=0, q=None, bt=None, cl=None, out=None):
    q = torch.from_numpy(w.q if q is None else q).cuda()
    bt = dev_u32(w.block_tables if bt is None else bt)
    cl = dev_u32(w.context_lens if cl is None else cl)
    out = torch.full_like(q, float("nan")) if out is None else out
    pk.pa_q8_decode(out, q, kc, vc, bt, cl, num_kv_heads=w.cfg.num_kv_heads,
                    block_size=w.cfg.block_size, scale=w.scale, kernel=kernel,
                    partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def oracle_decode(w, kc, vc, rows=None, q=None, bt=None, cl=None):
    return oracle.decode(w.q if q is None else q, kc, vc,
                         w.block_tables if bt is None else bt,
                         w.context_lens if cl is None else cl,
                         num_kv_heads=w.cfg.num_kv_heads, block_size=w.cfg.block_size,
                         scale=w.scale, rows=rows)


def random_case(S, H, Hk, D, B, lens, seed, Nb=None, scale_mult=1.0, dist=1.0, v_token_mult=None):
    """A poisoned paged cache written by both writers (checked equal).
    v_token_mult(position, context) -> factor scales each token's V vectors
    (magnitudes that change along a context)."""
    rng = np.random.default_rng(seed)
    nblk = [-(-int(c) // B) for c in lens]
    Nb = Nb or max(1, max(nblk))
    pool = sum(nblk) + 3
    perm = rng.permutation(pool).astype(np.uint32)
    bt = np.full((S, Nb), 0xFFFFFFFF, dtype=np.uint32)
    pos = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += nblk[s]
    T = int(sum(lens))
    key = (rng.standard_normal((T, Hk, D)) * dist).astype(np.float32)
    val = (rng.standard_normal((T, Hk, D)) * dist).astype(np.float32)
    if v_token_mult is not None and T:
        pos = np.concatenate([np.arange(c) for c in lens if c > 0])
        ctx = np.concatenate([np.full(c, c) for c in lens if c > 0])
        val = (val * np.asarray(v_token_mult(pos, ctx), dtype=np.float64)[:, None, None]).astype(np.float32)
    slots = np.concatenate([(bt[s, np.arange(c) // B].astype(np.int64) * B + np.arange(c) % B)
                            for s, c in enumerate(lens) if c > 0] or [np.zeros(0, np.int64)]).astype(np.uint32)
    W = D // 4 + 1
    ok_ = np.full((pool, Hk, B, W), 0xFFFFFFFF, dtype=np.uint32)
    ov_ = ok_.copy()
    oracle.reshape_and_cache(key, val, ok_, ov_, slots, num_kv_heads=Hk, head_size=D, block_size=B)
    kc, vc = dev_u32(ok_.copy()), dev_u32(ov_.copy())
    kc.fill_(-1)
    vc.fill_(-1)
    if T:
        pk.pa_q8_reshape_and_cache(torch.from_numpy(key.reshape(T, -1)).cuda(),
                                   torch.from_numpy(val.reshape(T, -1)).cuda(), kc, vc,
                                   dev_u32(slots), num_kv_heads=Hk, head_size=D, block_size=B)
    assert np.array_equal(host_u32(kc), ok_) and np.array_equal(host_u32(vc), ov_)
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    cfg = wl.Config("case", 99, S, H, Hk, D, B, Nb * B)
    w = wl.Workload(cfg=cfg, context_lens=np.asarray(lens, dtype=np.uint32), block_tables=bt,
                    num_blocks=pool, q=q, scale=float(np.float32(scale_mult / np.sqrt(D))),
                    key=None, value=None, slot_mapping=slots, row_seq=None)
    return w, ok_, ov_, kc, vc


def gpu_decode_rows(w, kc, vc, q, *, kernel=0, partition_tokens=0, cl=None):
    """pa_q8_decode_rows on device copies; q: f32 [S, R, H, D] numpy."""
    qd = torch.from_numpy(q).cuda()
    out = torch.full_like(qd, float("nan"))
    pk.pa_q8_decode_rows(out, qd, kc, vc, dev_u32(w.block_tables),
                         dev_u32(w.context_lens if cl is None else cl),
                         num_kv_heads=w.cfg.num_kv_heads, block_size=w.cfg.block_size,
                         scale=w.scale, num_blocks=w.num_blocks, kernel=kernel,
                         partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def oracle_decode_rows(w, kc, vc, q, cl=None):
    return oracle.decode_rows(q, kc, vc, w.block_tables, w.context_lens if cl is None else cl,
                              num_kv_heads=w.cfg.num_kv_heads, block_size=w.cfg.block_size,
                              scale=w.scale)


def assert_close(got, want, what=""):
    """|got - want| <= 1e-5 + 1e-4 |want| elementwise (want from the oracle)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = 1e-5 + 1e-4 * np.abs(want)
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert np.all(err <= bound), (f"{what}: {int((err > bound).sum())} of {err.size} outside "
                                  f"tolerance; worst at {worst}: got {got[worst]}, want {want[worst]}")
    return float(ratio.max())


def f32_units(value_sigma, logit_sigma):
    """Factor on the 1e-5 absolute part of the bound for inputs beyond the
    workloads' ranges.

    An f32 evaluation of out = sum_t p_t v_t carries two rounding errors that
    matter: the logits' (a D-term dot product, wrong by a few units of f32
    rounding of the logit's size, sigma_z) and the weighted sum's (relative to
    the values' size, sigma_v).  To first order a logit error dz_t moves the
    output by sum_t p_t dz_t (v_t - out), so the absolute error grows as
    sigma_z * sigma_v.  The five workloads reach sigma_v = 2 and sigma_z = 2
    (the edge workload: values N(0, 4), q N(0, 1), scale 1/sqrt(256)), and the
    stated bound holds there as it stands.  Inputs with sigma_v * sigma_z
    above that product take the absolute part in proportion; inputs inside it
    get the bound unscaled (factor 1)."""
    return max(1.0, float(value_sigma) * float(logit_sigma) / 4.0)


def assert_close_scaled(got, want, units, what=""):
    """|got - want| <= 1e-5 * units + 1e-4 |want| elementwise (units >= 1
    from f32_units; units == 1 is assert_close)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert units >= 1.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = 1e-5 * units + 1e-4 * np.abs(want)
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert np.all(err <= bound), (f"{what}: {int((err > bound).sum())} of {err.size} outside "
                                  f"tolerance (x{units:g} absolute); worst at {worst}: got {got[worst]}, "
                                  f"want {want[worst]}")
    return float(ratio.max())


def device_status(clear=True):
    return pk.pa_q8_device_status(clear=clear)
