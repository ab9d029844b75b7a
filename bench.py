"""MiTA forward throughput on GB300 (queries/s), with per-stage roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long_1m]
    python bench.py --impl reference ...     # the fp64 CPU oracle, timed on host cores

One step = one full forward pass (pool, landmark experts + shared values,
route, bucket, expert attention) over one batch of the workload, inputs
already resident in HBM.  Inputs are larger than L2 for both long workloads,
so no flush is needed between steps.  N > 1 runs one independent replica per
GPU (the forward does not shard); `value` counts the queries of all ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sparse_top_landmark_gb300 import workloads as W  # noqa: E402

METRIC = "MiTA fwd queries/sec at N=64K and 1M on 1 GB300; % of per-stage roofline"
UNIT = "queries/s"
L2_BYTES = 129 * 2 ** 20
# DRAM traffic of the expert stage's kernels from an ncu capture, with the
# hash of the kernel source it was taken on (stale counters are not reported)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "expert_long_1m_dram.txt")
EXPERT_SOURCE = os.path.join(ROOT, "sparse_top_landmark_gb300", "csrc", "expert_tc.cu")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], tc=d["bf16_tflops"], tc_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sus=1700.0, src="fallback")


# ---------------------------------------------------------------------------
# Algorithmic work per stage (flops, bytes) for the whole batch
# ---------------------------------------------------------------------------
def stage_work(w):
    """s routes per query: s route entries, bucket entries and expert pairs per query (the
    shared branch's 2Nmd output flops are counted with the expert stage either way)."""
    BH, N, d, m, k, s = w.B * w.H, w.N, w.d, w.m, w.topk, w.s
    e = 2 if w.dtype == "bf16" else 4
    return {
        "pool": (0.0, BH * (N * d * e + m * d * e)),
        "landmark": (BH * 4.0 * m * N * d, BH * (2 * N * d * e + m * d * e + m * k * 4 + m * d * 4)),
        "route": (BH * 2.0 * N * m * d, BH * (N * d * e + m * d * e + 4 * N * s)),
        "bucket": (0.0, BH * (12 * N * s + 4 * (m + 1))),
        "expert": (BH * (4.0 * N * s * k * d + 2.0 * N * m * d),
                   BH * (2 * N * d * e + 2 * m * k * d * e + 4 * m * k + 4 * N * s
                         + m * d * (e + 4))),
    }


def roofline_s(flops, nbytes, pk, sustained=False):
    tc = (pk["tc_sus"] if sustained else pk["tc"]) * 1e12
    return max(flops / tc, nbytes / (pk["hbm"] * 1e9))


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples (every 20 ms, each with its own timestamp); summary()
    keeps the samples taken inside a given host-time window."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        """Start sampling and wait (up to 10 s) for the first sample."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        import threading
        first = threading.Event()

        def reader():
            for ln in self.proc.stdout:
                if ln.strip():
                    self.lines.append(ln)
                    first.set()
        self._t = threading.Thread(target=reader, daemon=True)
        self._t.start()
        first.wait(timeout=10.0)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=5)

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self, t0, t1):
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            ts = self._stamp(f[0])
            try:
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if r[0] is not None and t0 - 0.005 <= r[0] <= t1 + 0.005]
        used = inside
        if not used and rows:   # window shorter than the sampling period: the nearest sample
            used = [min(rows, key=lambda r: abs((r[0] or t0) - 0.5 * (t0 + t1)))]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in used:
            for nm, val in zip(names, r[3]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[1] for r in used),
                "sm_max_mhz": max(r[2] for r in used), "reasons": sorted(reasons),
                "samples": len(inside), "window_ms": round((t1 - t0) * 1e3, 1)}


class NvmlClockSampler(ClockSampler):
    """The same summary from NVML read in-process (every ~2 ms, so even a window of a few
    tens of milliseconds holds many samples).  Reads only: SM clock, its maximum and the
    clock-event reason bits.  start() returns False when NVML cannot be loaded."""
    # clock-event reason bits (nvml.h): sw power cap, hw slowdown, sw thermal, hw thermal
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index, period_s=0.002):
        super().__init__(gpu_index)
        self.period = period_s
        self.samples = []          # (time, sm_mhz, max_mhz, reason bits)
        self._stop = False

    def start(self):
        import ctypes
        import threading
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                return False
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            return False
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

        def read():
            lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))        # 1 = SM clock
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            reasons_fn(h, ctypes.byref(rs))
            return (time.time(), float(clk.value), float(mx.value), int(rs.value))

        def loop():
            while not self._stop:
                self.samples.append(read())
                time.sleep(self.period)
        read()
        self._t = threading.Thread(target=loop, daemon=True)
        self._t.start()
        return True

    def stop(self):
        self._stop = True
        if getattr(self, "_t", None) is not None:
            self._t.join(timeout=5)

    def summary(self, t0, t1):
        self.lines = []
        for ts, sm, mx, bits in self.samples:
            stamp = __import__("datetime").datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")
            flags = ["Active" if bits & self.BITS[n] else "Not Active"
                     for n in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                               "sw_power_cap")]
            self.lines.append(", ".join([stamp, str(self.gpu), str(sm), str(mx), "0", hex(bits)]
                                        + flags))
        out = ClockSampler.summary(self, t0, t1)
        out["source"] = "nvml"
        return out


def clock_sampler(gpu_index):
    """NVML in-process sampling when available, else nvidia-smi."""
    s = NvmlClockSampler(gpu_index)
    if s.start():
        return s
    s = ClockSampler(gpu_index)
    s.start()
    return s


# ---------------------------------------------------------------------------
# CPU oracle timing on a bounded sample (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_time(w, q, k, v, budget=15.0, seed=0):
    """Time the oracle on a bounded sample of the workload: every pooling
    window, then batches of landmark rows (one per thread) for about 60% of
    `budget` seconds, then batches of queries (route + joint attention) for
    about 30%.  Returns (estimated seconds for the whole workload,
    description, threads, seconds spent)."""
    import oracle
    g = torch.Generator().manual_seed(seed)
    BH, N, m = w.B * w.H, w.N, w.m
    threads = oracle.num_threads()
    t0 = time.perf_counter()
    qt = oracle.pool(q, w.grid_h, w.grid_w, m)
    t_pool = time.perf_counter() - t0
    rows, t_rows = [], 0.0
    tis, vts = [], []
    while len(rows) < BH * m and (not rows or t_rows < 0.6 * budget):
        sel = torch.randint(0, BH * m, (min(threads, BH * m),), generator=g)
        t0 = time.perf_counter()
        ti, vt, _ = oracle.landmark(qt, k, v, w.topk, rows=sel)
        t_rows += time.perf_counter() - t0
        rows.append(sel)
        tis.append(ti)
        vts.append(vt)
    nrows = sum(r.numel() for r in rows)
    ti, vt = torch.cat(tis), torch.cat(vts)
    # per-query work does not depend on the values: every landmark reuses the
    # sampled rows' outputs
    full_ti = ti[torch.arange(BH * m) % ti.shape[0]].view(w.B, w.H, m, w.topk).contiguous()
    full_vt = vt[torch.arange(BH * m) % vt.shape[0]].view(w.B, w.H, m, w.d).contiguous()
    nq, t_q = 0, 0.0
    while nq < BH * N and (nq == 0 or t_q < 0.3 * budget):
        qsel = torch.randint(0, BH * N, (min(8192, BH * N),), generator=g)
        t0 = time.perf_counter()
        r, _ = oracle.route(q, qt, w.s, queries=qsel)
        oracle.attend(q, k, v, qt, full_vt, full_ti, r, queries=qsel)
        t_q += time.perf_counter() - t0
        nq += qsel.numel()
    est = t_pool + t_rows * (BH * m) / nrows + t_q * (BH * N) / nq
    desc = (f"oracle on {threads} threads: pool of all {BH * m} windows, "
            f"{nrows} of {BH * m} landmark rows (top-k + shared value), route + joint "
            f"attention of {nq} of {BH * N} queries; times scaled to the whole workload")
    return est, desc, threads, t_pool + t_rows + t_q


def expert_traffic(workload):
    """DRAM bytes per expert-stage launch from the committed ncu summary, or
    None when missing or taken on a different kernel source."""
    import hashlib
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    a, b = line.split(":", 1)
                    kv[a.strip()] = b.strip()
        with open(EXPERT_SOURCE, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if kv.get("source_sha256") != sha or kv.get("workload") != workload:
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def count_launches(mita, w, dq, dk, dv, out, stream):
    """Library kernels one forward launches (the library's own launch counter)."""
    n0 = mita.kernel_launches()
    mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, w.s, out=out, stream=stream)
    return mita.kernel_launches() - n0


# ---------------------------------------------------------------------------
def smi_index(local):
    """nvidia-smi index of this process's GPU."""
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in cvd.split(",") if p.strip()]
    if parts:
        p = parts[local] if local < len(parts) else parts[0]
        return int(p) if p.strip().isdigit() else local
    return local


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(secs, device, world):
    """The slowest rank's seconds, on every rank (replicas: one process per GPU, each timing
    its own copy of the workload; no data-path collective)."""
    if world <= 1:
        return secs
    t = torch.tensor([secs], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def replica_throughput(queries_per_rank, steps, secs, world):
    """Whole-job queries/s: every rank's queries over the slowest rank's time."""
    return world * queries_per_rank * steps / secs


def config_of(w, n_gpus):
    total = 3 * w.B * w.H * w.N * w.d * (2 if w.dtype == "bf16" else 4)
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m,
            "topk": w.topk, "s": w.s, "grid": [w.grid_h, w.grid_w],
            "qk": f"{w.clusters}-cluster Gaussian mixture sigma={w.sigma}" if w.qk == "mixture"
            else "iid N(0,1)",
            "l2": f"inputs larger than L2 ({total / 2**20:.0f} MiB of Q,K,V vs "
                  f"{L2_BYTES / 2**20:.0f} MiB), no flush",
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workload_of(args.workload, args.s)
    q, k, v = W.make_qkv(w, 0)
    per, spent_s = [], []
    budget = max(2.0, min(15.0, 150.0 / (args.warmup + args.steps)))
    for i in range(args.warmup + args.steps):
        est, desc, threads, spent = oracle_sample_time(w, q, k, v, budget=budget, seed=i)
        if i >= args.warmup:
            per.append(est)
            spent_s.append(spent)
    est = statistics.median(per)
    value = w.queries / est
    # one step is one bounded sample: ms_per_step is its measured wall time; the value is the
    # sample's rate (its time scaled to the whole workload gives workload_ms_estimate)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(spent_s) * 1e3,
            "ms_per_step_kind": "measured wall time of one bounded oracle sample",
            "workload_ms_estimate": est * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def time_forward(mita, w, dq, dk, dv, out, steps, stream):
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, w.s, out=out, stream=stream)
    ev1.record(stream)
    ev1.synchronize()
    return ev0.elapsed_time(ev1) / 1e3


def stage_times(mita, w, dq, dk, dv, reps, stream):
    """Average device time of each stage, run through the stage entry points."""
    BH = w.B * w.H
    qt = torch.empty((w.B, w.H, w.m, w.d), dtype=dq.dtype, device=dq.device)
    ti = torch.empty((w.B, w.H, w.m, w.topk), dtype=torch.int32, device=dq.device)
    vt = torch.empty((w.B, w.H, w.m, w.d), dtype=torch.float32, device=dq.device)
    r = torch.empty((w.B, w.H, w.N, w.s), dtype=torch.int32, device=dq.device)
    off = torch.empty((w.B, w.H, w.m + 1), dtype=torch.int32, device=dq.device)
    qi = torch.empty((w.B, w.H, w.N * w.s), dtype=torch.int32, device=dq.device)
    out = torch.empty_like(dq)
    calls = {
        "pool": lambda: mita.mita_pool(dq, w.grid_h, w.grid_w, w.m, q_tilde=qt, stream=stream),
        "landmark": lambda: mita.mita_landmark_topk_shared(qt, dk, dv, w.topk, topk_idx=ti,
                                                           v_tilde=vt, stream=stream),
        "route": lambda: mita.mita_route(dq, qt, s=w.s, route_idx=r, stream=stream),
        "bucket": lambda: mita.mita_bucket(r, w.m, bucket_off=off, bucket_qidx=qi, stream=stream),
        "expert": lambda: mita.mita_expert_attn(dq, dk, dv, qt, vt, ti, off, qi, s=w.s, out=out,
                                                stream=stream),
    }
    for fn in calls.values():     # warm, and fill every intermediate
        fn()
    res = {}
    for name, fn in calls.items():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
        for i in range(reps):
            evs[2 * i].record(stream)
            fn()
            evs[2 * i + 1].record(stream)
        evs[-1].synchronize()
        res[name] = sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(reps)) / reps / 1e3
    del BH
    return res


def bench_workload(mita, w, args, dev, stream, n_gpus, do_e2e=True, min_window_s=0.0,
                   stages=True):
    """Times `args.steps` forwards, or more when `min_window_s` asks for a longer window (the
    secondary workloads: their forwards are short, and the clock samples must fall inside)."""
    q, k, v = W.make_qkv(w, 0)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(dq)
    # clocks: sampling runs from before the warm-up, the timed window is cut out below
    sampler = clock_sampler(smi_index(dev.index))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, w.s, out=out,
                              stream=stream)
    torch.cuda.synchronize(dev)
    steps = args.steps
    if min_window_s > 0:
        probe = time_forward(mita, w, dq, dk, dv, out, 3, stream) / 3
        steps = max(steps, int(min_window_s / max(probe, 1e-6)) + 1)
        if n_gpus > 1:   # every rank times the same number of steps
            t = torch.tensor([steps], dtype=torch.int64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            steps = int(t.item())
    if n_gpus > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    secs = time_forward(mita, w, dq, dk, dv, out, steps, stream)
    t1 = time.time()
    sampler.stop()
    torch.cuda.synchronize(dev)
    secs = max_over_ranks(secs, dev, n_gpus)
    if n_gpus > 1:
        torch.distributed.barrier()
    res = {"secs": secs, "clocks": sampler.summary(t0, t1), "steps": steps}
    res["value"] = replica_throughput(w.queries, steps, secs, n_gpus)
    res["ms_per_step"] = secs / steps * 1e3
    if stages:
        res["stages"] = stage_times(mita, w, dq, dk, dv, max(3, min(args.steps, 10)), stream)
    res["launches"] = count_launches(mita, w, dq, dk, dv, out, stream)
    if do_e2e:
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        hout = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        for _ in range(max(1, args.warmup // 2)):
            mita.mita_forward(hq, hk, hv, w.grid_h, w.grid_w, w.m, w.topk, w.s, out=hout,
                              stream=stream, device=dev)
        if n_gpus > 1:
            torch.distributed.barrier()
        esteps = max(2, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(esteps):
            mita.mita_forward(hq, hk, hv, w.grid_h, w.grid_w, w.m, w.topk, w.s, out=hout,
                              stream=stream, device=dev)
        es = max_over_ranks(time.perf_counter() - t0, dev, n_gpus)
        e = q.element_size()
        res["e2e"] = {"value": replica_throughput(w.queries, esteps, es, n_gpus), "unit": UNIT,
                      "h2d_bytes_per_step": 3 * q.numel() * e,
                      "d2h_bytes_per_step": q.numel() * e}
    res["inputs"] = (q, k, v)
    return res


def roofline_entry(w, stages, pk):
    work = stage_work(w)
    name = max(stages, key=lambda s: stages[s])
    fl, by = work[name]
    t = stages[name]
    tc_time = fl / (pk["tc"] * 1e12)
    hbm_time = by / (pk["hbm"] * 1e9)
    if tc_time >= hbm_time:
        ach = fl / t / 1e12
        ent = {"bound": "tensor", "achieved": ach, "peak": pk["tc"], "unit": "TFLOP/s"}
    else:
        ach = by / t / 1e9
        ent = {"bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s"}
    ent["frac"] = ent["achieved"] / ent["peak"]
    ent["kernel"] = name
    ent["peak_source"] = pk["src"]
    ent["traffic"] = expert_traffic(w.name) if name == "expert" and w.s == 1 else None
    per = {}
    for s, tt in stages.items():
        rl = roofline_s(*work[s], pk)
        per[s] = {"ms": tt * 1e3, "roofline_ms": rl * 1e3, "frac": rl / tt if tt > 0 else None}
    return ent, per


def workload_of(name, s):
    """A named workload, with its routes per query replaced by `s` when given."""
    w = W.WORKLOADS[name]
    if s is not None and s != w.s:
        w = dataclasses.replace(w, s=s, name=f"{w.name}_s{s}")
    return w


def forward_only(args):
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    w = workload_of(args.workload, args.s)
    q, k, v = W.make_qkv(w, 0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(dq)
    for _ in range(args.forward_only):
        mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, w.s, out=out)
    torch.cuda.synchronize()
    print(json.dumps({"forward_only": w.name, "runs": args.forward_only,
                      "device_error": mita.get_last_device_error()}))
    return 0


# Reported throughput of MiTA over dense attention on the long synthetic sequences (MiTA
# tutorial ch. 7, figure 5: RTX 4090, a three-layer model, batch tuned per length, m*k ~ N/4).
PAGES_FIG5 = {1 << 14: 4.7, 1 << 16: 19.0, 1 << 18: 56.0, 1 << 20: 159.0}


def _time_calls(fn, reps, stream):
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(reps):
        fn()
    ev1.record(stream)
    ev1.synchronize()
    return ev0.elapsed_time(ev1) / reps


def fig5(args):
    """The long-sequence sweep of the throughput figure: MiTA (m = k = sqrt(N/4)), the
    routing-only model at the same entry count per query (topk = m + k, no shared branch) and
    dense attention, one attention layer each, bf16, d = 64, H = 2, B*N = 2^20 tokens."""
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    out_rows = []
    for i, N in enumerate(sorted(PAGES_FIG5)):
        m = k = int(round((N / 4) ** 0.5))
        B = max(1, (1 << 20) // N)
        w = W.custom(f"fig5_{N}", B, 2, N, 64, "bf16", 1, N, m, k, clusters=max(16, m // 2),
                     index=80 + i)
        q, kk, v = W.make_qkv(w, 0)
        dq, dk, dv = q.to(dev), kk.to(dev), v.to(dev)
        out = torch.empty_like(dq)
        with torch.cuda.stream(stream):
            f_mita = lambda: mita.mita_forward(dq, dk, dv, 1, N, m, k, 1, out=out, stream=stream)
            f_routed = lambda: mita.mita_forward_ex(dq, dk, dv, 1, N, m, m + k, 1,
                                                    branches="routed", out=out, stream=stream)
            f_dense = lambda: mita.mita_dense_attn(dq, dk, dv, out=out, stream=stream)
            res = {}
            for name, fn, reps in (("mita", f_mita, max(args.steps, 3)),
                                   ("routed_equal_entries", f_routed, max(args.steps, 3)),
                                   ("dense", f_dense, 1 if N >= (1 << 18) else 3)):
                for _ in range(1 if name == "dense" else args.warmup):
                    fn()
                res[name] = _time_calls(fn, reps, stream)
        assert mita.get_last_device_error(stream) == 0
        row = {"N": N, "B": B, "H": 2, "d": 64, "m": m, "topk": k,
               "mita_ms": res["mita"], "routed_equal_entries_ms": res["routed_equal_entries"],
               "dense_ms": res["dense"], "speedup_vs_dense": res["dense"] / res["mita"],
               "routed_over_mita": res["routed_equal_entries"] / res["mita"],
               "pages_speedup_rtx4090_model": PAGES_FIG5[N]}
        print(json.dumps(row), flush=True)
        out_rows.append(row)
        del dq, dk, dv, out
        torch.cuda.empty_cache()
    print(json.dumps({"fig5": out_rows}))
    return 0


def backward_bench(args):
    """Device time of mita_backward (selections held constant; SIMT gradient kernels) on
    --workload, next to the forward's, for one upstream gradient."""
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    w = workload_of(args.workload, args.s)
    q, k, v = W.make_qkv(w, 0)
    dq_, dk_, dv_ = q.to(dev), k.to(dev), v.to(dev)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(1)).to(q.dtype).to(dev)
    out = torch.empty_like(dq_)
    with torch.cuda.stream(stream):
        f_fwd = lambda: mita.mita_forward(dq_, dk_, dv_, w.grid_h, w.grid_w, w.m, w.topk, w.s,
                                          out=out, stream=stream)
        f_bwd = lambda: mita.mita_backward(dq_, dk_, dv_, dout, w.grid_h, w.grid_w, w.m, w.topk,
                                           w.s, stream=stream)
        for _ in range(args.warmup):
            f_fwd()
            f_bwd()
        fwd = _time_calls(f_fwd, args.steps, stream)
        bwd = _time_calls(f_bwd, args.steps, stream)
    assert mita.get_last_device_error(stream) == 0
    print(json.dumps({"backward": w.name, "config": config_of(w, 1), "forward_ms": fwd,
                      "backward_ms": bwd, "steps": args.steps, "warmup": args.warmup,
                      "grad_dtype": "f32"}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mita", choices=["mita", "reference"])
    ap.add_argument("--workload", default="long_1m", choices=list(W.WORKLOADS))
    ap.add_argument("--secondary", default="long_64k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-images", dest="images", action="store_false",
                    help="skip the image-grid workloads' lines")
    ap.add_argument("--backward", action="store_true",
                    help="time mita_backward on --workload next to the forward")
    ap.add_argument("--fig5", action="store_true",
                    help="sweep N = 16K..1M: MiTA, routing-only at equal entries, dense attention")
    ap.add_argument("--s", type=int, default=None,
                    help="routes per query (top-s); default: the workload's own (1)")
    ap.add_argument("--forward-only", type=int, default=0, metavar="R",
                    help="run R untimed forwards of --workload and exit (for profilers)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)
    if args.forward_only > 0:
        return forward_only(args)
    if args.fig5:
        return fig5(args)
    if args.backward:
        return backward_bench(args)

    ws, rank, local = dist_env()
    n_gpus = max(ws, 1)
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    from sparse_top_landmark_gb300 import build, mita
    if rank == 0 or ws == 1:
        build.build()
    if ws > 1:
        torch.distributed.barrier()
    mita.load()
    stream = torch.cuda.Stream(dev)
    pk = peaks()

    w = workload_of(args.workload, args.s)
    main_res = bench_workload(mita, w, args, dev, stream, n_gpus)
    roof, per_stage = roofline_entry(w, main_res["stages"], pk)
    sec = None
    if args.secondary and args.secondary not in ("none", args.workload):
        w2 = workload_of(args.secondary, args.s)
        r2 = bench_workload(mita, w2, args, dev, stream, n_gpus, do_e2e=False, min_window_s=1.0)
        roof2, per2 = roofline_entry(w2, r2["stages"], pk)
        total2 = sum(roofline_s(*wk, pk) for wk in stage_work(w2).values())
        sec = {"workload": w2.name, "value": r2["value"], "ms_per_step": r2["ms_per_step"],
               "steps": r2["steps"], "forward_roofline_frac": total2 / (r2["ms_per_step"] / 1e3),
               "roofline": roof2, "stages": per2, "clocks": r2["clocks"]}
    # the image-grid workloads (ViT-S 14x14 tokens, segmentation 32x32): whole forwards only,
    # each over a window of about a second
    images = []
    if args.images and args.s in (None, 1):
        for nm in ("vit_s_14x14", "seg_32x32"):
            wi = workload_of(nm, None)
            ri = bench_workload(mita, wi, args, dev, stream, n_gpus, do_e2e=False,
                                min_window_s=1.0, stages=False)
            tot = sum(roofline_s(*wk, pk) for wk in stage_work(wi).values())
            images.append({"workload": wi.name, "value": ri["value"], "unit": UNIT,
                           "ms_per_step": ri["ms_per_step"], "steps": ri["steps"],
                           "forward_roofline_frac": tot / (ri["ms_per_step"] / 1e3),
                           "roofline_ms": tot * 1e3, "clocks": ri["clocks"]})

    cpu = None
    if rank == 0 and n_gpus == 1 and not args.no_cpu_baseline:
        q, k, v = main_res["inputs"]
        est, desc, threads, spent = oracle_sample_time(w, q, k, v)
        cpu = {"value": w.queries / est, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": desc, "sample_seconds": spent}

    if rank == 0:
        total_rl = sum(roofline_s(*wk, pk) for wk in stage_work(w).values())
        line = {
            "metric": METRIC, "value": main_res["value"], "unit": UNIT, "n_gpus": n_gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": main_res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_of(w, n_gpus),
            "clocks": main_res["clocks"],
            "e2e": main_res["e2e"],
            "gpu_launches": (main_res["launches"] * args.steps
                             if main_res["launches"] is not None else None),
            "roofline": roof,
            "forward_roofline_frac": total_rl / (main_res["ms_per_step"] / 1e3),
            "stages": per_stage,
            "cpu_baseline": cpu,
            "secondary": sec,
            "image_workloads": images,
        }
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
