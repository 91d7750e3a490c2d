"""Benchmark of the int8 paged-KV hot path on one GB300 (or N replicas).

One step = one large-batch serving step, every row of the path once:
  1. pa_q8_reshape_and_cache: quantise and scatter 16384 new K/V rows
     (5% PAD, K/V column slices of fused rows of stride 10240) into the
     int8 paged caches;
  2. pa_q8_decode: single-query paged attention for 256 sequences x 64
     heads (8 kv heads, GQA 8), context lengths clip(LogNormal(ln 2048, 1),
     16, 8192), over the caches -- the attention kernel plus the
     log-sum-exp combine of split-context partials.
Metric: effective HBM GB/s = algorithmic bytes of the step / step time
(decode: every context token's K and V vector once + q + out + block-table
entries + context lengths; writer: K/V rows read + token vectors written +
slot mapping), also as % of the measured HBM copy peak, and seqs/s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 (launched by torch.distributed.run) every rank runs the same
workload on its own GPU (independent replicas, weak scaling; the path has
no exchange step).  --impl reference times the CPU oracle on bounded
samples of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from int8_paged_kv_gb300 import workloads as wl  # noqa: E402

WORKLOAD = "large"
METRIC = "q8 paged decode: effective KV HBM GB/s (% of GB300 peak) and seqs/s"
UNIT = "GB/s"
L2_FLUSH_MIN_BYTES = 256 << 20      # read (not written) between steps: evicts L2 with clean lines
def l2_flush_bytes(dev) -> int:
    """Twice the device's L2 (as the driver reports it), at least 256 MiB."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 0)
    return max(L2_FLUSH_MIN_BYTES, 2 * l2) // 4 * 4


NOMINAL_HBM_GBS = 8000.0            # GB300 HBM3e, nominal ~8 TB/s (reported beside the measured copy peak)
NVML_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                0x100: "display_clock_setting"}


def workload_description(cfg) -> str:
    return ("large batch serving step: num_seqs=256 num_heads=64 num_kv_heads=8 head_size=128 "
            "block_size=16, context_lens clip(LogNormal(ln 2048, 1), 16, 8192); append of 16384 "
            "rows, 5% PAD, K/V slices of fused rows of stride 10240")


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def recorded_traffic() -> dict | None:
    """DRAM bytes per decode launch from the committed ncu summary, if the
    kernel sources still match the ones profiled."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if not os.path.exists(p):
        return None
    rec = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("sources_sha256") != kernel_sources_sha():
        return None
    try:
        return {"bytes_per_launch": float(rec["dram_bytes_per_launch_scaled"]),
                "note": rec.get("note", "")}
    except (KeyError, ValueError):
        return None


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int8_paged_kv_gb300", "csrc")
    for name in ("decode.cu", "decode_common.cuh", "device_util.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Polls SM clock, power and clock-event reasons through NVML (ctypes)
    while running; falls back to nvidia-smi -lms if NVML is unavailable."""

    def __init__(self, index: int, period_s: float = 0.01):
        self.index, self.period = index, period_s
        self.samples: list[tuple[float, int, int]] = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        self._smi_path = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                raise OSError("no handle")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self._reasons = fn or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            self.nvml = None

    def _poll(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            ok = self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0
            ok = ok and self._reasons(self.h, ctypes.byref(rs)) == 0
            if ok:
                self.samples.append((time.time(), int(clk.value), int(rs.value)))
            time.sleep(self.period)

    def start(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        else:
            fd, self._smi_path = tempfile.mkstemp(prefix="pa_q8_clocks_", suffix=".csv")
            os.close(fd)
            self._smi = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=timestamp,clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self._smi_path, "w"), stderr=subprocess.DEVNULL)

    def stop(self) -> dict:
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            src = "nvml"
        elif self._smi is not None:
            self._smi.terminate()
            self._smi.wait()
            src = "nvidia-smi"
            with open(self._smi_path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    try:
                        self.samples.append((0.0, int(float(parts[1])), int(parts[3], 16)))
                        self.max_mhz = int(float(parts[2]))
                    except (ValueError, IndexError):
                        pass
            os.unlink(self._smi_path)
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s in self.samples if not (s[2] & 0x1)] or self.samples
        reasons = set()
        for _, _, r in busy:
            for bit, name in NVML_REASONS.items():
                if r & bit and bit != 0x1:
                    reasons.add(name)
        return {"sm_mhz": statistics.median([s[1] for s in busy]) if busy else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons), "samples": len(busy),
                "source": src}


# --------------------------------------------------------------- oracle legs

class OracleBench:
    """The CPU oracle on bounded samples of the workload.  Setup (untimed)
    writes every sequence's context into oracle-owned caches with the oracle
    writer; sample() then times the oracle writer on append rows and the
    oracle decode on whole sequences (all heads), resuming where the last
    sample stopped."""

    def __init__(self, w, key=None, value=None):
        import oracle
        self.oracle, self.w, cfg = oracle, w, w.cfg
        self.kc, self.vc = wl.empty_cache(w), wl.empty_cache(w)
        if key is None:
            for s in range(cfg.num_seqs):
                k, v, sm = wl.sequence_rows(w, [s])
                self._write(k, v, sm)
        else:
            self._write(key, value, w.slot_mapping)
        self.next_row, self.next_seq = 0, 0

    def _write(self, k, v, sm):
        cfg = self.w.cfg
        self.oracle.reshape_and_cache(k, v, self.kc, self.vc, sm, num_kv_heads=cfg.num_kv_heads,
                                      head_size=cfg.head_size, block_size=cfg.block_size)

    def sample(self, seconds: float, rows_per_chunk: int = 1024) -> dict:
        w, cfg, a = self.w, self.w.cfg, self.w.append
        t0 = time.perf_counter()
        rows, wbytes = 0, 0
        while rows == 0 or time.perf_counter() - t0 < seconds / 2:
            i = self.next_row
            sl = slice(i, min(i + rows_per_chunk, a.num_tokens))
            self._write(a.key_view()[sl], a.value_view()[sl], a.slot_mapping[sl])
            wbytes += wl.algorithmic_writer_bytes(cfg.num_kv_heads, cfg.head_size, a.slot_mapping[sl])
            rows += sl.stop - sl.start
            self.next_row = sl.stop % a.num_tokens
        tw = time.perf_counter() - t0
        t1 = time.perf_counter()
        nseq, dbytes = 0, 0
        while nseq == 0 or time.perf_counter() - t1 < seconds / 2:
            s = self.next_seq
            rws = np.array([[s, h] for h in range(cfg.num_heads)], dtype=np.int32)
            self.oracle.decode(w.q, self.kc, self.vc, w.block_tables, w.context_lens,
                               num_kv_heads=cfg.num_kv_heads, block_size=cfg.block_size,
                               scale=w.scale, rows=rws)
            c = int(w.context_lens[s])
            dbytes += (c * cfg.num_kv_heads * 2 * (cfg.head_size + 4) + 2 * cfg.num_heads * cfg.head_size * 4
                       + (-(-c // cfg.block_size)) * 4 + 4)
            nseq += 1
            self.next_seq = (s + 1) % cfg.num_seqs
        td = time.perf_counter() - t1
        return {"writer_s_per_byte": tw / wbytes, "decode_s_per_byte": td / dbytes,
                "writer_rows": rows, "decode_seqs": nseq, "seconds": tw + td,
                "sample_bytes": wbytes + dbytes, "cores": self.oracle.num_threads()}


def check_parity(ob, w, out, kc, vc) -> dict:
    """Sampled parity of the timed step's results against the oracle, once,
    before the timed loop: decode rows (all heads of the longest, the
    shortest and two seeded sequences) within 1e-5 + 1e-4 |oracle|, and the
    first 128 stored appended rows' cache words bit for bit (they go to free
    slots, which no sequence reads)."""
    import torch
    cfg, a = w.cfg, w.append
    H, Hk, B = cfg.num_heads, cfg.num_kv_heads, cfg.block_size
    lens = w.context_lens
    seqs = {int(np.argmax(lens)), int(np.argmin(lens))}
    seqs |= {int(x) for x in np.random.default_rng(7).choice(cfg.num_seqs, 2, replace=False)}
    seqs = sorted(seqs)
    rows = np.array([[s, h] for s in seqs for h in range(H)], dtype=np.int32)
    want = ob.oracle.decode(w.q, ob.kc, ob.vc, w.block_tables, w.context_lens, num_kv_heads=Hk,
                            block_size=B, scale=w.scale, rows=rows)
    got = out.cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    ratio = float(np.max(np.abs(got - want) / (1e-5 + 1e-4 * np.abs(want))))
    idx = np.nonzero(a.slot_mapping != wl.PAD_SLOT)[0][:128]
    sm = a.slot_mapping[idx]
    ob.oracle.reshape_and_cache(np.ascontiguousarray(a.key_view()[idx]), np.ascontiguousarray(a.value_view()[idx]),
                                ob.kc, ob.vc, sm, num_kv_heads=Hk, head_size=cfg.head_size, block_size=B)
    blk, off = (sm // B).astype(np.int64), (sm % B).astype(np.int64)
    tb, to = torch.from_numpy(blk).to(kc.device), torch.from_numpy(off).to(kc.device)
    same = (np.array_equal(kc[tb, :, to, :].cpu().numpy().view(np.uint32), ob.kc[blk, :, off, :]) and
            np.array_equal(vc[tb, :, to, :].cpu().numpy().view(np.uint32), ob.vc[blk, :, off, :]))
    return {"decode_rows": int(len(rows)), "sequences": seqs, "max_err_over_bound": round(ratio, 4),
            "writer_vectors": int(len(idx)) * Hk * 2, "writer_bit_exact": bool(same),
            "ok": bool(ratio <= 1.0 and same)}


def cpu_line_fields(samp: dict, step_bytes_w: int, step_bytes_d: int) -> dict:
    t_step = samp["writer_s_per_byte"] * step_bytes_w + samp["decode_s_per_byte"] * step_bytes_d
    return {"value": round((step_bytes_w + step_bytes_d) / t_step / 1e9, 4), "unit": UNIT,
            "cores": samp["cores"], "kind": "oracle",
            "sample": (f"fp64 C oracle (OpenMP) on {samp['writer_rows']} append rows (of 16384 per step, "
                       f"cycling) and {samp['decode_seqs']} sequence decodes (all 64 heads; 256 per "
                       f"step, cycling), {samp['seconds']:.1f} s; step time extrapolated by "
                       f"algorithmic bytes")}


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = wl.build(WORKLOAD, with_kv=False)
    cfg = w.cfg
    bw = wl.algorithmic_writer_bytes(cfg.num_kv_heads, cfg.head_size, w.append.slot_mapping)
    bd = wl.algorithmic_decode_bytes(cfg, w.context_lens)
    ob = OracleBench(w)
    for _ in range(args.warmup):
        ob.sample(seconds=0.05)
    vals, secs, last = [], 0.0, None
    for _ in range(args.steps):
        last = ob.sample(seconds=args.ref_step_seconds)
        vals.append(cpu_line_fields(last, bw, bd)["value"])
        secs += last["seconds"]
    value = float(statistics.median(vals))
    cpu = cpu_line_fields(last, bw, bd)
    cpu["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round((bw + bd) / (value * 1e9) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_description(cfg), "impl": "CPU oracle (fp64 C, OpenMP)"},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------- multi-rank glue

def dist_max(x: float, device=None) -> float:
    """Max of a per-rank float over all ranks (the bench's timing rule)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_step per step, the job
    takes the slowest rank's time."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------- the other four workloads

# sequences the oracle checks per workload (the first n): every sequence of
# tiny, a share of the others (long: one 32K-131K context of 32 heads)
PARITY_SEQS = {"tiny": 2, "llama8b": 4, "long": 1, "large": 8, "edge": 8}


def oracle_rows(w, n: int) -> np.ndarray:
    """The fp64 oracle's outputs for the first n sequences of a workload: their
    rows written into oracle-owned caches by the oracle writer, then decoded."""
    import oracle
    cfg = w.cfg
    sub = wl.subset(w, n)
    n = int(sub.context_lens.size)
    k, v, sm = wl.sequence_rows(sub, range(n))
    kc, vc = wl.empty_cache(sub), wl.empty_cache(sub)
    oracle.reshape_and_cache(k, v, kc, vc, sm, num_kv_heads=cfg.num_kv_heads, head_size=cfg.head_size,
                             block_size=cfg.block_size)
    return oracle.decode(np.ascontiguousarray(sub.q[:n]), kc, vc, sub.block_tables, sub.context_lens,
                         num_kv_heads=cfg.num_kv_heads, block_size=cfg.block_size, scale=sub.scale)


def time_workload_decodes(args, dev, peaks, flush_l2, names, with_parity: bool) -> dict:
    """pa_q8_decode on each named workload (automatic plan), timed like the
    bench step: L2 flushed between calls outside the events, CUDA events on the
    launching stream, median of args.steps calls after max(3, warmup) untimed
    ones.  With the oracle leg on, the first PARITY_SEQS[name] sequences'
    output rows are checked against the oracle (|gpu - oracle| <= 1e-5 +
    1e-4 |oracle|)."""
    import torch

    import int8_paged_kv_gb300 as pk
    res = {}
    stream = torch.cuda.current_stream()
    for name in names:
        w = wl.build(name, with_append=False)
        cfg = w.cfg
        S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size

        def u32(x):
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to(dev)

        kc = torch.empty((w.num_blocks, Hk, B, D // 4 + 1), dtype=torch.int32, device=dev)
        vc = torch.empty_like(kc)
        step = 1 << 18
        for i in range(0, w.key.shape[0], step):
            pk.pa_q8_reshape_and_cache(torch.from_numpy(w.key[i:i + step].reshape(-1, Hk * D)).to(dev),
                                       torch.from_numpy(w.value[i:i + step].reshape(-1, Hk * D)).to(dev),
                                       kc, vc, u32(w.slot_mapping[i:i + step]), num_kv_heads=Hk, head_size=D,
                                       block_size=B)
        w.key = w.value = None
        q = torch.from_numpy(w.q).to(dev)
        bt, cl = u32(w.block_tables), u32(w.context_lens)
        out = torch.empty_like(q)
        plan = pk.pa_q8_decode_plan(S, H, Hk, D, B, cfg.max_blocks_per_seq)
        ws = torch.empty(max(16, pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq)),
                         dtype=torch.uint8, device=dev)

        def run():
            pk.pa_q8_decode(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale, workspace=ws)
        for _ in range(max(3, args.warmup)):
            flush_l2()
            run()
        a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2()
            a[i].record(stream)
            run()
            b[i].record(stream)
        torch.cuda.synchronize()
        ms = float(statistics.median(x.elapsed_time(y) for x, y in zip(a, b)))
        nbytes = wl.algorithmic_decode_bytes(cfg, w.context_lens)
        gbps = nbytes / ms / 1e6
        entry = {"ms": round(ms, 4), "gbps": round(gbps, 1),
                 "pct_of_hbm_peak": round(100 * gbps / peaks["hbm_gbs"], 2),
                 "pct_of_nominal_hbm": round(100 * gbps / NOMINAL_HBM_GBS, 2),
                 "seqs_per_s": round(S / (ms * 1e-3), 1), "algorithmic_bytes": int(nbytes),
                 "partition_tokens": plan["partition_tokens"], "attention_ctas": plan["num_ctas"],
                 "device_status": pk.pa_q8_device_status(clear=True)}
        if with_parity:
            want = oracle_rows(w, PARITY_SEQS[name])
            got = out[:want.shape[0]].cpu().numpy().astype(np.float64)
            ratio = float(np.max(np.abs(got - want) / (1e-5 + 1e-4 * np.abs(want))))
            entry["parity"] = {"sequences": int(want.shape[0]), "rows": int(want.shape[0] * H),
                               "max_err_over_bound": round(ratio, 4),
                               "ok": bool(ratio <= 1.0 and entry["device_status"] == 0)}
        res[name] = entry
        del kc, vc, q, out, ws
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- our arm

def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import int8_paged_kv_gb300 as pk
    from int8_paged_kv_gb300 import build as pkbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        pkbuild.build()
    if world > 1:
        dist.barrier()
    pk.lib()

    w = wl.build(WORKLOAD)
    if args.seqs:
        w = wl.subset(w, args.seqs)                     # small case for profiler captures
    cfg, a = w.cfg, w.append
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    W = D // 4 + 1

    if args.seqs:
        args.no_cpu_baseline = True

    def u32(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to(dev)

    # resident state: the caches holding every sequence's context, built by the writer
    kc = torch.empty((w.num_blocks, Hk, B, W), dtype=torch.int32, device=dev)
    vc = torch.empty_like(kc)
    T = w.key.shape[0]
    chunk = 1 << 18
    for i in range(0, T, chunk):
        kk = torch.from_numpy(w.key[i:i + chunk].reshape(-1, Hk * D)).to(dev)
        vv = torch.from_numpy(w.value[i:i + chunk].reshape(-1, Hk * D)).to(dev)
        pk.pa_q8_reshape_and_cache(kk, vv, kc, vc, u32(w.slot_mapping[i:i + chunk]), num_kv_heads=Hk,
                                   head_size=D, block_size=B)
    del kk, vv
    ob = None
    if not args.no_cpu_baseline and world == 1 and rank == 0:
        ob = OracleBench(w, w.key, w.value)             # untimed setup of the CPU-baseline leg
    w.key = w.value = None
    q = torch.from_numpy(w.q).to(dev)
    bt, cl = u32(w.block_tables), u32(w.context_lens)
    out = torch.empty_like(q)
    fused = torch.from_numpy(a.fused).to(dev)
    k_new = fused[:, a.key_offset:a.value_offset]
    v_new = fused[:, a.value_offset:a.value_offset + Hk * D]
    slots = u32(a.slot_mapping)
    plan = pk.pa_q8_decode_plan(S, H, Hk, D, B, cfg.max_blocks_per_seq, kernel=args.kernel,
                                partition_tokens=args.partition_tokens)
    ws_bytes = pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq, kernel=args.kernel,
                                              partition_tokens=args.partition_tokens)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.ones(l2_flush_bytes(dev) // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int32, device=dev)

    def flush_l2():
        torch.sum(flush, dim=0, out=flush_sink)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    assert pk.pa_q8_device_status(clear=True) == 0

    def step():
        ev_w0.record(stream)
        pk.pa_q8_reshape_and_cache(k_new, v_new, kc, vc, slots, num_kv_heads=Hk, head_size=D,
                                   block_size=B)
        ev_d0.record(stream)
        pk.pa_q8_decode(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale,
                        workspace=ws, kernel=args.kernel, partition_tokens=args.partition_tokens)
        ev_d1.record(stream)

    bytes_w = wl.algorithmic_writer_bytes(Hk, D, a.slot_mapping)
    rows_w = int(np.count_nonzero(a.slot_mapping != wl.PAD_SLOT))    # token rows the writer stores
    bytes_d = wl.algorithmic_decode_bytes(cfg, w.context_lens)
    # writer, prep (sequence order; skipped when every CTA of a one-partition
    # plan is resident at once), attention.  A split plan that fits one wave
    # has no prep but a combine grid after the attention, so it also counts 3.
    per_sm = 3 if plan["kernel"] == 2 else 2
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    one_wave = plan["num_partitions"] == 1 and plan["num_ctas"] <= per_sm * sms
    launches_per_step = 2 if one_wave else 3

    ev_d0, ev_d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_w0 = torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    # the warm-up steps' results against the oracle, before anything is timed
    parity = check_parity(ob, w, out, kc, vc) if ob is not None else None
    if parity is not None and not parity["ok"]:
        print(json.dumps({"parity": parity}), flush=True)
        raise SystemExit("bench: the step's results do not match the oracle")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    wstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    # sustained, untimed load (back-to-back steps with the L2 flush) so clocks
    # and power settle, and a clock sampler sees the GPU busy, before timing
    sustained_steps, t_sus = 0, time.perf_counter()
    while time.perf_counter() - t_sus < args.sustain_seconds:
        for _ in range(64):
            flush_l2()
            step()
        torch.cuda.synchronize()
        sustained_steps += 64
    t_sus = time.perf_counter() - t_sus
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2()                                      # outside the timed events
        starts[i].record(stream)
        ev_d0, ev_d1, ev_w0 = dstarts[i], dends[i], wstarts[i]
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    clocks["window"] = "the sustained warm-up and the timed steps"
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dec_ms = [s.elapsed_time(e) for s, e in zip(dstarts, dends)]
    wr_ms = [s.elapsed_time(e) for s, e in zip(wstarts, dstarts)]
    total_ms = dist_max(sum(step_ms), dev)
    status = pk.pa_q8_device_status(clear=True)
    ms_per_step = total_ms / args.steps
    value = job_gbps(world, bytes_w + bytes_d, ms_per_step)
    # per-kernel figures: medians over the timed steps
    dec_med_ms = float(statistics.median(dec_ms))
    dec_gbs = bytes_d / (dec_med_ms * 1e-3) / 1e9
    wr_med_ms = float(statistics.median(wr_ms))

    # ---- end to end: host (pinned) inputs copied in, output copied back, every step
    e2e = None
    if not args.no_e2e:
        h_q = torch.from_numpy(w.q).pin_memory()
        h_k = torch.from_numpy(np.ascontiguousarray(a.key_view())).pin_memory()
        h_v = torch.from_numpy(np.ascontiguousarray(a.value_view())).pin_memory()
        h_slots = torch.from_numpy(a.slot_mapping.view(np.int32)).pin_memory()
        h_bt = torch.from_numpy(w.block_tables.view(np.int32)).pin_memory()
        h_cl = torch.from_numpy(w.context_lens.view(np.int32)).pin_memory()
        h_out = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        d_q, d_k, d_v = torch.empty_like(q), torch.empty(h_k.shape, device=dev), torch.empty(h_v.shape, device=dev)
        d_slots, d_bt, d_cl = torch.empty_like(slots), torch.empty_like(bt), torch.empty_like(cl)
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_slots, h_bt, h_cl))
        d2h = h_out.numel() * 4

        # Copies run on their own streams (waiting for the step's start event,
        # so none begins before the timed region): the small inputs first,
        # then the new K/V rows in chunks spread over the copy streams; the
        # compute stream appends each chunk as it lands, then decodes and
        # copies the output back.
        copy_streams = [torch.cuda.Stream(device=dev) for _ in range(max(1, args.e2e_streams))]
        n_chunks = max(1, args.e2e_chunks)
        rows = h_k.shape[0]
        cuts = [rows * j // n_chunks for j in range(n_chunks + 1)]

        def e2e_step(start):
            for cs in copy_streams:
                cs.wait_event(start)
            with torch.cuda.stream(copy_streams[0]):
                for src, dst in ((h_q, d_q), (h_slots, d_slots), (h_bt, d_bt), (h_cl, d_cl)):
                    dst.copy_(src, non_blocking=True)
                small = torch.cuda.Event()
                small.record(copy_streams[0])
            landed = []
            for j in range(n_chunks):
                cs = copy_streams[j % len(copy_streams)]
                lo, hi = cuts[j], cuts[j + 1]
                with torch.cuda.stream(cs):
                    d_k[lo:hi].copy_(h_k[lo:hi], non_blocking=True)
                    d_v[lo:hi].copy_(h_v[lo:hi], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                landed.append(ev)
            stream.wait_event(small)
            for j in range(n_chunks):
                lo, hi = cuts[j], cuts[j + 1]
                stream.wait_event(landed[j])
                pk.pa_q8_reshape_and_cache(d_k[lo:hi], d_v[lo:hi], kc, vc, d_slots[lo:hi], num_kv_heads=Hk,
                                           head_size=D, block_size=B)
            pk.pa_q8_decode(out, d_q, kc, vc, d_bt, d_cl, num_kv_heads=Hk, block_size=B, scale=w.scale,
                            workspace=ws, kernel=args.kernel, partition_tokens=args.partition_tokens)
            h_out.copy_(out, non_blocking=True)

        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for _ in range(args.warmup):
            flush_l2()
            es[0].record(stream)
            e2e_step(es[0])
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2()
            es[i].record(stream)
            e2e_step(es[i])
            ee[i].record(stream)
        torch.cuda.synchronize()
        e_total = dist_max(sum(s.elapsed_time(e) for s, e in zip(es, ee)), dev)
        e_ms = e_total / args.steps
        e2e = {"value": round(job_gbps(world, bytes_w + bytes_d, e_ms), 2), "unit": UNIT,
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "overlap": f"{len(copy_streams)} copy streams, append in {n_chunks} chunks as they land"}

    peaks = measured_peaks()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None
    if ob is not None:
        samp = ob.sample(seconds=args.cpu_seconds)
        cpu = cpu_line_fields(samp, bytes_w, bytes_d)

    # the other four workloads' decodes, each timed on its own (rank 0 only)
    configs = {}
    if not args.seqs and not args.no_configs:
        configs = time_workload_decodes(args, dev, peaks, flush_l2, ["tiny", "llama8b", "long", "edge"],
                                        with_parity=ob is not None)
    large_entry = {"ms": round(dec_med_ms, 4), "gbps": round(dec_gbs, 1),
                   "pct_of_hbm_peak": round(100 * dec_gbs / peaks["hbm_gbs"], 2),
                   "pct_of_nominal_hbm": round(100 * dec_gbs / NOMINAL_HBM_GBS, 2),
                   "seqs_per_s": round(S / (dec_med_ms * 1e-3), 1), "algorithmic_bytes": int(bytes_d),
                   "partition_tokens": plan["partition_tokens"], "attention_ctas": plan["num_ctas"],
                   "device_status": status}
    if parity is not None:
        large_entry["parity"] = {"sequences": len(parity["sequences"]), "rows": parity["decode_rows"],
                                 "max_err_over_bound": parity["max_err_over_bound"], "ok": parity["ok"]}
    if configs:
        configs = {"tiny": configs["tiny"], "llama8b": configs["llama8b"], "long": configs["long"],
                   "large": large_entry, "edge": configs["edge"]}

    traffic = recorded_traffic()
    kernel_name = {1: "CUDA-core (f32 FMA)", 2: "tensor-core (mma.sync f16 hi/lo)"}[plan["kernel"]]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_description(cfg), "kv_cache": "int8 codes + f32 scale per token",
                   "decode_kernel": kernel_name, "partition_tokens": plan["partition_tokens"],
                   "num_partitions": plan["num_partitions"], "attention_ctas": plan["num_ctas"],
                   "parallelism": f"{world} independent replica(s)" if world > 1 else "1 GPU",
                   "l2": f"{flush.numel() * 4 >> 20} MiB buffer read between steps (outside the timed events), so every "
                         "step starts with an L2 of clean foreign lines; the decode reads 1.6 GB of KV "
                         "per step"},
        "ms_per_step_median": round(float(statistics.median(step_ms)), 4),
        "pct_of_hbm_peak": round(100 * value / world / peaks["hbm_gbs"], 2),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "seqs_per_s": round(world * S / (ms_per_step * 1e-3), 1),
        "timing": ("value and ms_per_step: the K timed steps' total (max over ranks) / K; decode, writer, "
                   "roofline and configs: medians of per-call CUDA events"),
        "decode": {"ms": round(dec_med_ms, 4), "gbps": round(dec_gbs, 1),
                   "pct_of_hbm_peak": round(100 * dec_gbs / peaks["hbm_gbs"], 2),
                   "pct_of_nominal_hbm": round(100 * dec_gbs / NOMINAL_HBM_GBS, 2),
                   "seqs_per_s": round(S / (dec_med_ms * 1e-3), 1),
                   "algorithmic_bytes": int(bytes_d)},
        "writer": {"ms": round(wr_med_ms, 4),
                   "gbps": round(bytes_w / (wr_med_ms * 1e-3) / 1e9, 1),
                   "tokens_per_s": round(rows_w / (wr_med_ms * 1e-3), 1),
                   "algorithmic_bytes": int(bytes_w)},
        "configs": configs or None,
        "sustained_warmup": {"seconds": round(t_sus, 2), "steps": sustained_steps},
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(dec_gbs / peaks["hbm_gbs"], 4),
                     "traffic": (round(traffic["bytes_per_launch"]) if traffic else None),
                     "kernel": "pa_q8_decode call (prep kernel + attention kernel; one partition per "
                               "context, so no merge runs), CUDA events on the launching stream",
                     "peak_source": f"{peaks['source']} HBM copy peak (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cpu,
        "parity": parity,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------- per-workload table

def run_append_lines(args, name, w, kc, vc, bt, cl, q, flush, sink, peaks) -> None:
    """One decode step with one new token per sequence: the fused
    pa_q8_decode_append against pa_q8_reshape_and_cache followed by
    pa_q8_decode (same new tokens, same positions)."""
    import torch

    import int8_paged_kv_gb300 as pk
    cfg = w.cfg
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    dev = q.device
    key, value = wl.new_token_rows(w, 1)
    kd = torch.from_numpy(key.reshape(S, Hk * D)).to(dev)
    vd = torch.from_numpy(value.reshape(S, Hk * D)).to(dev)
    pos = np.minimum(w.context_lens.astype(np.int64), cfg.max_blocks_per_seq * B) - 1
    slots = (w.block_tables[np.arange(S), pos // B].astype(np.int64) * B + pos % B).astype(np.uint32)
    sm = torch.from_numpy(slots.view(np.int32)).to(dev)
    q4 = q.reshape(S, 1, H, D)
    out4 = torch.empty_like(q4)
    ws = torch.empty(pk.pa_q8_decode_rows_workspace_size(S, 1, H, Hk, D, B, cfg.max_blocks_per_seq),
                     dtype=torch.uint8, device=dev)
    nbytes = wl.algorithmic_decode_bytes(cfg, w.context_lens) + wl.algorithmic_writer_bytes(Hk, D, slots)

    def fused():
        pk.pa_q8_decode_append(out4, q4, kd, vd, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B,
                               scale=w.scale, workspace=ws)

    def unfused():
        pk.pa_q8_reshape_and_cache(kd, vd, kc, vc, sm, num_kv_heads=Hk, head_size=D, block_size=B)
        pk.pa_q8_decode(out4.view(S, H, D), q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B,
                        scale=w.scale, workspace=ws)
    for label, run in (("fused append+decode", fused), ("writer then decode", unfused)):
        for _ in range(max(3, args.warmup)):
            torch.sum(flush, dim=0, out=sink)
            run()
        ts = []
        for _ in range(args.steps):
            torch.sum(flush, dim=0, out=sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = float(np.median(ts))
        par = parity_fields(args, "append", out4.view(S, H, D))
        print(json.dumps({"kind": "decode step with append", "workload": name, "step": label,
                          "cpu_oracle_gbps": args.oracle_rates["append"], **par,
                          "new_tokens": S, "ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                          "gbps": round(nbytes / ms / 1e6, 1),
                          "pct_of_hbm_peak": round(100 * nbytes / ms / 1e6 / peaks["hbm_gbs"], 1),
                          "pct_of_nominal_hbm": round(100 * nbytes / ms / 1e6 / NOMINAL_HBM_GBS, 1)}),
              flush=True)


def run_f32_line(args, name, w, bt, cl, q, flush, sink, peaks) -> None:
    """The same decode over an f32 cache (pa_f32_decode): 4 * head_size bytes
    per token vector instead of head_size + 4."""
    import torch

    import int8_paged_kv_gb300 as pk
    cfg = w.cfg
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    dev = q.device
    kc = torch.empty((w.num_blocks, Hk, B, D), dtype=torch.float32, device=dev)
    vc = torch.empty_like(kc)
    T = w.key.shape[0]
    for i in range(0, T, 1 << 18):
        sm = torch.from_numpy(np.ascontiguousarray(w.slot_mapping[i:i + (1 << 18)]).view(np.int32)).to(dev)
        pk.pa_f32_reshape_and_cache(torch.from_numpy(w.key[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                    torch.from_numpy(w.value[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                    kc, vc, sm, num_kv_heads=Hk, head_size=D, block_size=B)
    out = torch.empty_like(q)
    ws = torch.empty(max(1, pk.pa_f32_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq)),
                     dtype=torch.uint8, device=dev)

    def run():
        pk.pa_f32_decode(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale, workspace=ws)
    for _ in range(max(3, args.warmup)):
        torch.sum(flush, dim=0, out=sink)
        run()
    ts = []
    for _ in range(args.steps):
        torch.sum(flush, dim=0, out=sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = float(np.median(ts))
    nbytes = wl.algorithmic_decode_bytes(cfg, w.context_lens, cache="f32")
    par = parity_fields(args, "f32", out)
    print(json.dumps({"kind": "decode per workload, f32 cache", "workload": name, "kernel": "f32 cuda-core",
                      "cpu_oracle_gbps": args.oracle_rates["f32"], **par,
                      "ms": round(ms, 4), "algorithmic_bytes": int(nbytes), "gbps": round(nbytes / ms / 1e6, 1),
                      "pct_of_hbm_peak": round(100 * nbytes / ms / 1e6 / peaks["hbm_gbs"], 1),
                      "pct_of_nominal_hbm": round(100 * nbytes / ms / 1e6 / NOMINAL_HBM_GBS, 1),
                      "seqs_per_s": round(S / (ms * 1e-3), 1)}), flush=True)
    del kc, vc
    torch.cuda.empty_cache()


def run_profile_rows(args) -> None:
    """A profiler case, not a bench line: pa_q8_decode_rows with
    --profile-rows R query rows per sequence over the large batch (its first
    --seqs sequences when given), kernel family --kernel; prints the median
    event time of --steps calls after --warmup."""
    import torch

    import int8_paged_kv_gb300 as pk
    from int8_paged_kv_gb300 import build as pkbuild

    pkbuild.build()
    dev = torch.device("cuda", 0)
    w = wl.build(WORKLOAD, with_append=False, with_kv=not args.seqs)
    if args.seqs:
        w = wl.subset(w, args.seqs)
        key, value, slots = wl.sequence_rows(w, range(w.context_lens.size))
    else:
        key, value, slots = w.key, w.value, w.slot_mapping
    cfg = w.cfg
    S = int(w.context_lens.size)
    H, Hk, D, B = cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    R = int(args.profile_rows)

    def u32(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to(dev)

    kc = torch.empty((w.num_blocks, Hk, B, D // 4 + 1), dtype=torch.int32, device=dev)
    vc = torch.empty_like(kc)
    for i in range(0, key.shape[0], 1 << 18):
        pk.pa_q8_reshape_and_cache(torch.from_numpy(key[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                   torch.from_numpy(value[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                   kc, vc, u32(slots[i:i + (1 << 18)]), num_kv_heads=Hk, head_size=D,
                                   block_size=B)
    key = value = w.key = w.value = None
    q = torch.from_numpy(np.ascontiguousarray(wl.query_rows(w, R)[:S])).to(dev)
    out = torch.empty_like(q)
    bt, cl = u32(w.block_tables), u32(w.context_lens)
    ws = torch.empty(max(16, pk.pa_q8_decode_rows_workspace_size(S, R, H, Hk, D, B, cfg.max_blocks_per_seq,
                                                                 kernel=args.kernel,
                                                                 partition_tokens=args.partition_tokens)),
                     dtype=torch.uint8, device=dev)

    def run():
        pk.pa_q8_decode_rows(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale,
                             workspace=ws, kernel=args.kernel, partition_tokens=args.partition_tokens)
    for _ in range(max(3, args.warmup)):
        run()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    sub = wl.Config(cfg.name, cfg.index, S, H, Hk, D, B, cfg.max_context)
    nbytes = wl.algorithmic_decode_bytes(sub, w.context_lens, R)
    ms = float(np.median(ts))
    print(json.dumps({"kind": "profile case: multi-row decode", "seqs": S, "query_rows": R,
                      "kernel": args.kernel, "ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                      "gbps": round(nbytes / ms / 1e6, 1), "device_status": pk.pa_q8_device_status()}))


def run_profile_workload(args) -> None:
    """A profiler case, not a bench line: pa_q8_decode on one named workload
    (--profile-workload), automatic plan unless --kernel / --partition-tokens,
    L2 flushed before every call; prints the median event time of --steps
    calls after --warmup."""
    import torch

    import int8_paged_kv_gb300 as pk
    from int8_paged_kv_gb300 import build as pkbuild

    pkbuild.build()
    dev = torch.device("cuda", 0)
    w = wl.build(args.profile_workload, with_append=False)
    cfg = w.cfg
    S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size

    def u32(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to(dev)

    kc = torch.empty((w.num_blocks, Hk, B, D // 4 + 1), dtype=torch.int32, device=dev)
    vc = torch.empty_like(kc)
    for i in range(0, w.key.shape[0], 1 << 18):
        pk.pa_q8_reshape_and_cache(torch.from_numpy(w.key[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                   torch.from_numpy(w.value[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                   kc, vc, u32(w.slot_mapping[i:i + (1 << 18)]), num_kv_heads=Hk, head_size=D,
                                   block_size=B)
    w.key = w.value = None
    q = torch.from_numpy(w.q).to(dev)
    out = torch.empty_like(q)
    bt, cl = u32(w.block_tables), u32(w.context_lens)
    opts = dict(kernel=args.kernel, partition_tokens=args.partition_tokens)
    ws = torch.empty(max(16, pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq, **opts)),
                     dtype=torch.uint8, device=dev)
    flush = torch.ones(l2_flush_bytes(dev) // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)

    def run():
        pk.pa_q8_decode(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale, workspace=ws,
                        **opts)
    for _ in range(max(3, args.warmup)):
        torch.sum(flush, dim=0, out=sink)
        run()
    ts = []
    for _ in range(args.steps):
        torch.sum(flush, dim=0, out=sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    nbytes = wl.algorithmic_decode_bytes(cfg, w.context_lens)
    ms = float(np.median(ts))
    print(json.dumps({"kind": "profile case: decode of one workload", "workload": args.profile_workload,
                      "plan": pk.pa_q8_decode_plan(S, H, Hk, D, B, cfg.max_blocks_per_seq, **opts),
                      "ms": round(ms, 4), "algorithmic_bytes": int(nbytes), "gbps": round(nbytes / ms / 1e6, 1),
                      "device_status": pk.pa_q8_device_status()}))


def run_contig_line(args, name, w, cl, q, flush, sink, peaks) -> None:
    """The same contexts in the contiguous q8 cache (per-sequence code rows +
    side scale region, max_t = the workload's largest context), appended by
    pa_q8c_append and decoded by pa_q8c_decode."""
    import torch

    import int8_paged_kv_gb300 as pk
    cfg = w.cfg
    S, H, Hk, D = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size
    max_t = cfg.max_context
    dev = q.device
    words = pk.pa_q8c_cache_words(max_t, Hk, D)
    kc = torch.empty((S, words), dtype=torch.int32, device=dev)
    vc = torch.empty_like(kc)
    seq = np.repeat(np.arange(S, dtype=np.int64), w.context_lens.astype(np.int64))
    pos = np.concatenate([np.arange(int(c), dtype=np.int64) for c in w.context_lens])
    slots = (seq * max_t + pos).astype(np.uint32)
    T = w.key.shape[0]
    for i in range(0, T, 1 << 18):
        sm = torch.from_numpy(np.ascontiguousarray(slots[i:i + (1 << 18)]).view(np.int32)).to(dev)
        pk.pa_q8c_append(torch.from_numpy(w.key[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                         torch.from_numpy(w.value[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                         kc, vc, sm, num_kv_heads=Hk, head_size=D, max_t=max_t)
    out = torch.empty_like(q)
    ws = torch.empty(max(16, pk.pa_q8c_decode_workspace_size(S, H, Hk, D, max_t)), dtype=torch.uint8, device=dev)

    def run():
        pk.pa_q8c_decode(out, q, kc, vc, cl, num_kv_heads=Hk, max_t=max_t, scale=w.scale, workspace=ws)
    for _ in range(max(3, args.warmup)):
        torch.sum(flush, dim=0, out=sink)
        run()
    ts = []
    for _ in range(args.steps):
        torch.sum(flush, dim=0, out=sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = float(np.median(ts))
    nbytes = wl.algorithmic_decode_bytes(cfg, w.context_lens, cache="q8c")
    par = parity_fields(args, "contig", out)
    print(json.dumps({"kind": "decode per workload, contiguous q8 cache", "workload": name,
                      "cpu_oracle_gbps": args.oracle_rates["contig"], **par,
                      "kernel": "tensor-core (32-element group scales)", "ms": round(ms, 4),
                      "algorithmic_bytes": int(nbytes), "gbps": round(nbytes / ms / 1e6, 1),
                      "pct_of_hbm_peak": round(100 * nbytes / ms / 1e6 / peaks["hbm_gbs"], 1),
                      "pct_of_nominal_hbm": round(100 * nbytes / ms / 1e6 / NOMINAL_HBM_GBS, 1),
                      "seqs_per_s": round(S / (ms * 1e-3), 1)}), flush=True)
    del kc, vc
    torch.cuda.empty_cache()


def run_profile_variant(args) -> None:
    """A profiler case, not a bench line: the f32-cache decode (--profile-f32)
    or the contiguous-cache decode (--profile-contig) over the large batch's
    contexts (its first --seqs sequences when given); prints the median event
    time of --steps calls after --warmup."""
    import torch

    import int8_paged_kv_gb300 as pk
    from int8_paged_kv_gb300 import build as pkbuild

    pkbuild.build()
    dev = torch.device("cuda", 0)
    w = wl.build(WORKLOAD, with_append=False, with_kv=not args.seqs)
    if args.seqs:
        w = wl.subset(w, args.seqs)
        key, value, slots = wl.sequence_rows(w, range(w.context_lens.size))
    else:
        key, value, slots = w.key, w.value, w.slot_mapping
    cfg = w.cfg
    S = int(w.context_lens.size)
    H, Hk, D, B = cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    scfg = wl.Config(cfg.name, cfg.index, S, H, Hk, D, B, cfg.max_context)

    def u32(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to(dev)

    q = torch.from_numpy(np.ascontiguousarray(w.q[:S])).to(dev)
    out = torch.empty_like(q)
    cl = u32(w.context_lens)
    step = 1 << 18
    if args.profile_f32:
        kc = torch.empty((w.num_blocks, Hk, B, D), dtype=torch.float32, device=dev)
        vc = torch.empty_like(kc)
        for i in range(0, key.shape[0], step):
            pk.pa_f32_reshape_and_cache(torch.from_numpy(key[i:i + step].reshape(-1, Hk * D)).to(dev),
                                        torch.from_numpy(value[i:i + step].reshape(-1, Hk * D)).to(dev),
                                        kc, vc, u32(slots[i:i + step]), num_kv_heads=Hk, head_size=D, block_size=B)
        bt = u32(w.block_tables)
        ws = torch.empty(max(16, pk.pa_f32_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq)),
                         dtype=torch.uint8, device=dev)

        def run():
            pk.pa_f32_decode(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale, workspace=ws)
        kind, nbytes = "f32 cache", wl.algorithmic_decode_bytes(scfg, w.context_lens, cache="f32")
    else:
        max_t = cfg.max_context
        words = pk.pa_q8c_cache_words(max_t, Hk, D)
        kc = torch.empty((S, words), dtype=torch.int32, device=dev)
        vc = torch.empty_like(kc)
        seq = np.repeat(np.arange(S, dtype=np.int64), w.context_lens.astype(np.int64))
        pos = np.concatenate([np.arange(int(c), dtype=np.int64) for c in w.context_lens])
        cs = (seq * max_t + pos).astype(np.uint32)
        for i in range(0, key.shape[0], step):
            pk.pa_q8c_append(torch.from_numpy(key[i:i + step].reshape(-1, Hk * D)).to(dev),
                             torch.from_numpy(value[i:i + step].reshape(-1, Hk * D)).to(dev),
                             kc, vc, u32(cs[i:i + step]), num_kv_heads=Hk, head_size=D, max_t=max_t)
        ws = torch.empty(max(16, pk.pa_q8c_decode_workspace_size(S, H, Hk, D, max_t)), dtype=torch.uint8,
                         device=dev)

        def run():
            pk.pa_q8c_decode(out, q, kc, vc, cl, num_kv_heads=Hk, max_t=max_t, scale=w.scale, workspace=ws)
        kind, nbytes = "contiguous q8 cache", wl.algorithmic_decode_bytes(scfg, w.context_lens, cache="q8c")
    for _ in range(max(3, args.warmup)):
        run()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = float(np.median(ts))
    print(json.dumps({"kind": f"profile case: {kind} decode", "seqs": S, "ms": round(ms, 4),
                      "algorithmic_bytes": int(nbytes), "gbps": round(nbytes / ms / 1e6, 1),
                      "device_status": pk.pa_q8_device_status()}))


def oracle_rates(w, n: int) -> dict:
    """GB/s of the CPU oracle on the first n sequences of a workload, for the
    report's variants (single query, 4 and 8 query rows, f32 cache,
    contiguous cache, append + decode); caches are written untimed, the
    timed call is the oracle's function for the variant."""
    import oracle
    cfg = w.cfg
    sub = wl.subset(w, n)
    n = int(sub.context_lens.size)
    Hk, D, B = cfg.num_kv_heads, cfg.head_size, cfg.block_size
    scfg = wl.Config(cfg.name, cfg.index, n, cfg.num_heads, Hk, D, B, cfg.max_context)
    k, v, sm = wl.sequence_rows(sub, range(n))
    kc, vc = wl.empty_cache(sub), wl.empty_cache(sub)
    oracle.reshape_and_cache(k, v, kc, vc, sm, num_kv_heads=Hk, head_size=D, block_size=B)
    q = np.ascontiguousarray(sub.q[:n])
    args = dict(num_kv_heads=Hk, block_size=B, scale=sub.scale)
    out, refs = {}, {}

    def rate(name, fn, nbytes):
        t0 = time.perf_counter()
        res = fn()
        out[name] = round(nbytes / (time.perf_counter() - t0) / 1e9, 4)
        if res is not None and name not in refs:
            refs[name] = res
    rate("q8", lambda: oracle.decode(q, kc, vc, sub.block_tables, sub.context_lens, **args),
         wl.algorithmic_decode_bytes(scfg, sub.context_lens))
    if cfg.name in ("tiny", "llama8b", "edge"):          # also on one host core
        cores = oracle.num_threads()
        oracle.set_num_threads(1)
        try:
            rate("q8_one_core", lambda: oracle.decode(q, kc, vc, sub.block_tables, sub.context_lens, **args),
                 wl.algorithmic_decode_bytes(scfg, sub.context_lens))
        finally:
            oracle.set_num_threads(cores)
    for R in (4, 8):
        qr = np.ascontiguousarray(wl.query_rows(w, R)[:n])
        rate(f"rows{R}", lambda: oracle.decode_rows(qr, kc, vc, sub.block_tables, sub.context_lens, **args),
             wl.algorithmic_decode_bytes(scfg, sub.context_lens, R))
    fk = np.zeros((sub.num_blocks, Hk, B, D), dtype=np.float32)
    fv = np.zeros_like(fk)
    oracle.reshape_and_cache_f32(k, v, fk, fv, sm, num_kv_heads=Hk, head_size=D, block_size=B)
    rate("f32", lambda: oracle.decode_f32(q, fk, fv, sub.block_tables, sub.context_lens, **args),
         wl.algorithmic_decode_bytes(scfg, sub.context_lens, cache="f32"))
    max_t = cfg.max_context
    words = oracle.cq_seq_words(max_t, Hk, D)
    ck = np.zeros((n, words), dtype=np.uint32)
    cv = np.zeros_like(ck)
    cslots = np.concatenate([s * max_t + np.arange(int(c)) for s, c in enumerate(sub.context_lens)]).astype(np.uint32)
    oracle.cq_append(k, v, ck, cv, cslots, num_kv_heads=Hk, head_size=D, max_t=max_t)
    rate("contig", lambda: oracle.cq_decode(q, ck, cv, sub.context_lens, num_kv_heads=Hk, max_t=max_t,
                                            scale=sub.scale),
         wl.algorithmic_decode_bytes(scfg, sub.context_lens, cache="q8c"))
    nk, nv = wl.new_token_rows(w, 1)
    nk, nv = np.ascontiguousarray(nk[:n].reshape(n, -1)), np.ascontiguousarray(nv[:n].reshape(n, -1))
    pos = np.minimum(sub.context_lens.astype(np.int64), cfg.max_blocks_per_seq * B) - 1
    nslots = (sub.block_tables[np.arange(n), pos // B].astype(np.int64) * B + pos % B).astype(np.uint32)

    def append_decode():
        oracle.reshape_and_cache(nk, nv, kc, vc, nslots, num_kv_heads=Hk, head_size=D, block_size=B)
        return oracle.decode(q, kc, vc, sub.block_tables, sub.context_lens, **args)
    rate("append", append_decode, wl.algorithmic_decode_bytes(scfg, sub.context_lens) +
         wl.algorithmic_writer_bytes(Hk, D, nslots))
    out["sample"] = f"first {n} sequences ({int(sub.context_lens.sum())} context tokens), fp64 C oracle"
    out["cores"] = oracle.num_threads()
    out["_refs"] = refs              # the oracle's outputs for these sequences (parity of the GPU lines)
    return out


def parity_fields(args, variant: str, got) -> dict:
    """|gpu - oracle| / (1e-5 + 1e-4 |oracle|) at its largest over the oracle
    sample's sequences (the first rows of `got`); a value above 1 ends the
    report with an error once the line is printed."""
    want = args.oracle_rates["_refs"][variant]
    g = got[:want.shape[0]].detach().cpu().numpy().astype(np.float64).reshape(want.shape)
    ratio = float(np.max(np.abs(g - want) / (1e-5 + 1e-4 * np.abs(want))))
    if not ratio <= 1.0:
        args.parity_failures.append(variant)
    return {"parity_max_err_over_bound": round(ratio, 4), "parity_sequences": int(want.shape[0])}


def run_configs(args) -> None:
    """Decode throughput of every workload (single query: tensor-core and
    CUDA-core families; 4 and 8 query rows per sequence on the batches that
    fill the GPU: mma.sync and tcgen05 families), one JSON line per
    (workload, rows, family) -- a report next to the bench line, not a bench
    line itself."""
    import torch

    import int8_paged_kv_gb300 as pk
    from int8_paged_kv_gb300 import build as pkbuild

    pkbuild.build()
    dev = torch.device("cuda", 0)
    peaks = measured_peaks()
    flush = torch.ones(l2_flush_bytes(dev) // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    args.parity_failures = []
    for name in wl.CONFIGS:
        w = wl.build(name, with_append=False)
        cfg = w.cfg
        ora = oracle_rates(w, {"tiny": 2, "llama8b": 4, "long": 1, "large": 8, "edge": 8}[name])
        args.oracle_rates = ora
        print(json.dumps({"kind": "cpu oracle sample", "workload": name,
                          **{k: v for k, v in ora.items() if k != "_refs"}}), flush=True)
        S, H, Hk, D, B = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size

        def u32(x):
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to(dev)

        W = D // 4 + 1
        kc = torch.empty((w.num_blocks, Hk, B, W), dtype=torch.int32, device=dev)
        vc = torch.empty_like(kc)
        T = w.key.shape[0]
        for i in range(0, T, 1 << 18):
            pk.pa_q8_reshape_and_cache(torch.from_numpy(w.key[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                       torch.from_numpy(w.value[i:i + (1 << 18)].reshape(-1, Hk * D)).to(dev),
                                       kc, vc, u32(w.slot_mapping[i:i + (1 << 18)]), num_kv_heads=Hk,
                                       head_size=D, block_size=B)
        q = torch.from_numpy(w.q).to(dev)
        bt, cl, out = u32(w.block_tables), u32(w.context_lens), torch.empty_like(q)
        if name in ("llama8b", "long", "large"):
            run_f32_line(args, name, w, bt, cl, q, flush, sink, peaks)
        if name in ("llama8b", "large"):
            run_contig_line(args, name, w, cl, q, flush, sink, peaks)
        w.key = w.value = None
        # R > 1: causal decode of R query rows per sequence (pa_q8_decode_rows),
        # on the workloads whose batches fill the GPU
        runs = [(1, pk.PA_Q8_KERNEL_TENSOR_CORE), (1, pk.PA_Q8_KERNEL_CUDA_CORE)]
        if name in ("llama8b", "long", "large"):
            runs += [(R, k) for R in (4, 8) for k in (pk.PA_Q8_KERNEL_TENSOR_CORE, pk.PA_Q8_KERNEL_TCGEN05)]
        for R, kernel in runs:
            nbytes = wl.algorithmic_decode_bytes(cfg, w.context_lens, R)
            if R == 1:
                plan = pk.pa_q8_decode_plan(S, H, Hk, D, B, cfg.max_blocks_per_seq, kernel=kernel)
                ws = torch.empty(pk.pa_q8_decode_workspace_size(S, H, Hk, D, B, cfg.max_blocks_per_seq,
                                                                kernel=kernel), dtype=torch.uint8, device=dev)

                def run():
                    pk.pa_q8_decode(out, q, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B, scale=w.scale,
                                    workspace=ws, kernel=kernel)
            else:
                plan = {"partition_tokens": None}
                qr = torch.from_numpy(wl.query_rows(w, R)).to(dev)
                outr = torch.empty_like(qr)
                ws = torch.empty(pk.pa_q8_decode_rows_workspace_size(S, R, H, Hk, D, B, cfg.max_blocks_per_seq,
                                                                     kernel=kernel),
                                 dtype=torch.uint8, device=dev)

                def run():
                    pk.pa_q8_decode_rows(outr, qr, kc, vc, bt, cl, num_kv_heads=Hk, block_size=B,
                                         scale=w.scale, workspace=ws, kernel=kernel)
            for _ in range(max(3, args.warmup)):
                torch.sum(flush, dim=0, out=sink)
                run()
            ts = []
            for _ in range(args.steps):
                torch.sum(flush, dim=0, out=sink)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                run()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            ms = float(np.median(ts))
            par = parity_fields(args, "q8" if R == 1 else f"rows{R}", out if R == 1 else outr)
            print(json.dumps({"kind": "decode per workload", "workload": name, "description": cfg.description,
                              "query_rows": R,
                              "kernel": {1: "cuda-core", 2: "tensor-core", 3: "tcgen05"}[kernel],
                              "cpu_oracle_gbps": ora["q8" if R == 1 else f"rows{R}"],
                              "partition_tokens": plan["partition_tokens"], "ms": round(ms, 4),
                              "algorithmic_bytes": int(nbytes), "gbps": round(nbytes / ms / 1e6, 1),
                              "pct_of_hbm_peak": round(100 * nbytes / ms / 1e6 / peaks["hbm_gbs"], 1),
                              "pct_of_nominal_hbm": round(100 * nbytes / ms / 1e6 / NOMINAL_HBM_GBS, 1),
                              "seqs_per_s": round(S / (ms * 1e-3), 1), **par}), flush=True)
        if name in ("llama8b", "large"):
            run_append_lines(args, name, w, kc, vc, bt, cl, q, flush, sink, peaks)
        del kc, vc, q, out
        torch.cuda.empty_cache()
    if args.parity_failures:
        raise SystemExit(f"bench --configs: results outside the oracle tolerance: {args.parity_failures}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--configs", action="store_true",
                    help="print decode throughput of every workload instead of the bench line")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core")
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--profile-rows", type=int, default=0,
                    help="profiler case: multi-row decode with this many query rows (not a bench line)")
    ap.add_argument("--profile-f32", action="store_true", help="profiler case: f32-cache decode")
    ap.add_argument("--profile-workload", choices=["tiny", "llama8b", "long", "large", "edge"], default=None,
                    help="profiler case: pa_q8_decode on one workload")
    ap.add_argument("--profile-contig", action="store_true", help="profiler case: contiguous-cache decode")
    ap.add_argument("--seqs", type=int, default=0,
                    help="profile-size case: only the first N sequences (not a bench number)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=2, help="copy streams of the end-to-end step")
    ap.add_argument("--e2e-chunks", type=int, default=4, help="chunks the appended rows are copied in")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other four workloads' decode timings in the bench line")
    ap.add_argument("--sustain-seconds", type=float, default=1.5,
                    help="untimed back-to-back steps before the timed ones (clock sampler running)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.0,
                    help="oracle seconds per reference step (0: fit the run into ~2.5 minutes)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)          # timing rule: at least 3 warm-up steps
    if args.ref_step_seconds <= 0:
        args.ref_step_seconds = min(4.0, max(0.05, 150.0 / (args.steps + args.warmup)))
    if args.configs:
        run_configs(args)
    elif args.profile_rows:
        run_profile_rows(args)
    elif args.profile_workload:
        run_profile_workload(args)
    elif args.profile_f32 or args.profile_contig:
        run_profile_variant(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
