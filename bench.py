"""Benchmark: selected-token logp forward + backward, rows/s and HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bil|reference]
    python bench.py --workload linear [...]     # the fused LM-head + logp

Workload (one step = the whole operator path over one batch):
  training: N=16384 rows (B=8 x T=2048), V=151936 bf16 logits ~ 3*randn, tile
  4096, targets 70% from the row's top-5 columns, g ~ N(0, 1) fp32; forward
  (logp, lse) then backward (bf16 dlogits).  Inputs live in HBM before the
  timed region; each pass reads 4.98 GB, far more than the 129 MB L2, so no
  flush is needed between steps.

Prints one JSON line.  ``value`` is rows/s over all GPUs (each rank runs its
own batch: weak scaling, no collective on the data path).  ``e2e`` is the same
metric through the public API with the inputs in pinned host memory and the
host<->device copies inside the timed region.  ``roofline`` rates the
backward kernel (two thirds of the step's bytes) against the measured HBM
copy bandwidth.  ``cpu_baseline`` times the CPU oracle on a sample of the
same workload.  ``--impl reference`` times the CPU oracle alone (rank 0).

``--workload linear`` measures the fused LM-head + logp instead: hidden
[16384, 4096] bf16 times a Qwen3-8B-shaped LM head [151936, 4096] bf16, with
the tile partials taken from the tensor-core accumulator and the fixed-order
merge, then the backward (dZ from the recomputed projection, dhidden and
dweight): four tensor-core GEMMs of 2*N*H*V flops each per step.  Its
roofline is the forward partials kernel against the measured dense bf16
tensor throughput; the backward is reported as a whole.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "logp fwd+bwd rows/s and achieved HBM GB/s (% of GB300 peak) at V=151936"
WORKLOAD = ("training: N=16384 rows (B=8 x T=2048), V=151936 bf16 logits ~ 3*randn, tile 4096, "
            "targets 70% top-5 / 30% uniform, g ~ N(0,1) fp32, forward + backward, bf16 dlogits")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth, the denominator the 75% target is stated against
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
KERNEL_SOURCE = os.path.join(ROOT, "invariant_token_log_gb300", "csrc", "logp_device.cuh")
LINEAR_SOURCE = os.path.join(ROOT, "invariant_token_log_gb300", "csrc", "linear.cu")
LINEAR_METRIC = ("fused LM-head + logp fwd+bwd rows/s and achieved TFLOP/s (% of GB300 dense bf16) at H=4096, "
                 "V=151936")
LINEAR_WORKLOAD = ("linear: N=16384 rows (B=8 x T=2048) of bf16 hidden states ~ randn, H=4096, LM-head weight "
                   "[151936, 4096] bf16 ~ randn*3/64 (Qwen3-8B shape), uniform targets, 5% rows ignored, "
                   "g ~ N(0,1); forward logp + lse (256-column vocabulary tiles), then the backward: dhidden and "
                   "dweight in bf16 from the recomputed projection")
LINEAR_CPU_ROWS = 8
LINEAR_REFERENCE_ROWS = 8
FALLBACK_BF16_TFLOPS = 1900.0
# the reference arm runs the whole batch each step while (steps + warm-up) x batch
# stays within this many rows (about a minute of the oracle on 16 host cores),
# and an equal share of it per step beyond
REFERENCE_ROW_BUDGET = 25 * 16384
CPU_BASELINE_ROWS = 16384


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["bil", "reference"], default="bil")
    # The end-to-end steps stream 10 GB per step over the host link; on the GPU machine a step now and
    # then stalls for 100-200 ms with the host already queued far ahead (the GPU side waits), so
    # the end-to-end figure is taken over enough steps that one such stall does not dominate it.
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--rows", type=int, default=16384,
                    help="rows of the workload per GPU (smaller only for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["training", "linear"], default="training")
    ap.add_argument("--entropy", action="store_true",
                    help="training step with the entropy output and its gradient (for profiling; not the headline)")
    ap.add_argument("--temperature", type=float, default=1.0,
                    help="training step at this temperature (for profiling; not the headline)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the secondary measurements (entropy with a temperature, decode latency, prefill, "
                         "the exponential unit, the fused LM-head step)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; rows shard across ranks)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return dist if world > 1 else None


def max_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(rows_per_rank: int, world: int, steps: int, max_total_ms: float):
    """(ms per step, whole-job rows/s): every rank processed its own rows per
    step, and the job took as long as its slowest rank."""
    ms_step = max_total_ms / steps
    return ms_step, rows_per_rank * world * steps / (max_total_ms / 1e3)


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class NvmlClocks:
    """The SM clock and the clock-event reasons read through NVML (read-only queries) every
    couple of milliseconds, so that a timed region of a few tens of milliseconds still gets
    a dozen samples; nvidia-smi's own loop samples every 50 ms."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid: str, period_s: float = 0.002):
        import ctypes
        self.rows, self.period, self.lib, self.handle = [], period_s, None, None
        self.stop_flag = threading.Event()
        self.thread = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            u = uuid if uuid.upper().startswith("GPU-") else "GPU-" + uuid
            if lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) != 0:
                return
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.lib, self.handle, self.ctypes = lib, h, ctypes
        except (OSError, AttributeError):
            self.lib = None

    def start(self):
        if self.lib is None:
            return
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct, lib, h = self.ctypes, self.lib, self.handle
        clk, reasons = ct.c_uint(0), ct.c_ulonglong(0)
        while not self.stop_flag.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0  # 1: the SM clock domain
            ok = ok and self.reason_fn(h, ct.byref(reasons)) == 0
            if ok:
                self.rows.append((time.time(), clk.value, reasons.value))
            time.sleep(self.period)

    def stop(self):
        self.stop_flag.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        window = [(c, r) for (ts, c, r) in self.rows if t0 <= ts <= t1]
        if len(window) < 3:
            return None
        reasons = sorted({name for (_, r) in window for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in window), "sm_min_mhz": min(c for c, _ in window),
                "reasons": reasons, "samples": len(window), "scope": "timed region", "source": "NVML, every 2 ms"}


class ClockSampler:
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.rows = []
        self.proc = None
        self.thread = None
        self.nvml = NvmlClocks(self.uuid) if self.uuid else None

    def start(self):
        if self.nvml is not None:
            self.nvml.start()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 10:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.nvml is not None:
            self.nvml.stop()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        """nvidia-smi's samples in the timed region (the whole measured phase if it holds fewer
        than three); with NVML's faster samples of the timed region, their median clock and
        reasons lead, and nvidia-smi's figures stay under `nvidia_smi`."""
        smi = self._smi_summary(t0, t1)
        fast = self.nvml.summary(t0, t1) if self.nvml is not None else None
        if fast is None:
            return smi
        out = dict(fast)
        out["sm_max_mhz"] = smi.get("sm_max_mhz")
        out["power_w_max"] = smi.get("power_w_max")
        out["reasons"] = sorted(set(fast["reasons"]) | set(smi.get("reasons") or []))
        out["nvidia_smi"] = smi
        return out

    def _smi_summary(self, t0: float, t1: float):
        uuids = {p[1] for (_, p) in self.rows}
        mine = [p for (_, p) in self.rows
                if len(uuids) == 1 or (self.uuid and p[1].lower().replace("gpu-", "") == self.uuid)]
        window = [p for (ts, p) in self.rows if t0 <= ts <= t1 and p in mine]
        scope = "timed region"
        if len(window) < 3:  # a short timed region: widen to the whole measured phase
            window, scope = mine, "warm-up + timed region"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "scope": "unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(p[2]) for p in window) if v is not None]
        mx = [v for v in (num(p[3]) for p in window) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in window for i in range(4) if p[6 + i].lower() == "active"})
        pw = [v for v in (num(p[4]) for p in window) if v is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "power_w_max": max(pw) if pw else None, "samples": len(window),
                "scope": scope}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_rows_per_s(rows: int, passes: int = 1, w=None):
    """Time the CPU oracle's forward + backward over the first `rows` rows of the
    workload (`w`, the generated training workload, or generated here)."""
    import oracle
    import workloads as wl
    oracle.build()
    if w is None:
        chunks = list(range(-(-rows // wl.CHUNK_ROWS)))
        w = wl.training(n_rows=rows, chunks=chunks)
    g = w.grad_logp.astype(np.float64)
    batch = 256
    t0 = time.perf_counter()
    for _ in range(passes):
        for r0 in range(0, rows, batch):
            r1 = min(rows, r0 + batch)
            x = w.logits[r0:r1]
            oracle.logp_fwd(x, w.dtype, w.vocab, w.target_ids[r0:r1], w.ignore_index)
            oracle.logp_bwd(x, w.dtype, w.vocab, w.target_ids[r0:r1], g[r0:r1], w.ignore_index)
    dt = time.perf_counter() - t0
    return rows * passes / dt, dt, oracle.num_threads()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads as wl
    oracle.build()
    n = args.rows
    per_step = REFERENCE_ROW_BUDGET // max(1, args.steps + args.warmup)
    rows = max(wl.CHUNK_ROWS, min(n, per_step // wl.CHUNK_ROWS * wl.CHUNK_ROWS))
    w = wl.training(n_rows=rows, chunks=list(range(-(-rows // wl.CHUNK_ROWS))))
    g = w.grad_logp.astype(np.float64)
    batch = 256

    def step():
        for r0 in range(0, rows, batch):
            r1 = min(rows, r0 + batch)
            x = w.logits[r0:r1]
            oracle.logp_fwd(x, w.dtype, w.vocab, w.target_ids[r0:r1], w.ignore_index)
            oracle.logp_bwd(x, w.dtype, w.vocab, w.target_ids[r0:r1], g[r0:r1], w.ignore_index)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    what = "all" if rows == n else "the first"
    sample = f"{what} {rows} of the {n} rows of the workload per step, float64 oracle, forward + backward"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, host-generated)",
        "config": training_config(n, args.gpus), "rows_per_step": rows,
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def hbm_peak():
    try:
        peaks = json.load(open(PEAKS_FILE))
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """(burst, sustained, source) dense bf16 TFLOP/s."""
    try:
        peaks = json.load(open(PEAKS_FILE))
        return float(peaks["bf16_tflops"]), float(peaks["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def ncu_traffic(kernel: str, source: str = KERNEL_SOURCE, active_rows: int | None = None):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on this kernel source.

    A record with ``bytes_per_row`` comes from a capture of a smaller batch than the
    benchmark's (the traffic of these kernels grows in proportion to the rows they
    process); it is scaled to ``active_rows``.  A record with ``bytes_per_launch``
    was taken on the benchmark's own batch."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    sha = hashlib.sha256(open(source, "rb").read()).hexdigest()[:16]
    for line in lines:
        if line.lstrip().startswith("#"):
            continue
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") != kernel or f.get("source_sha") != sha:
            continue
        if "bytes_per_row" in f and active_rows is not None:
            return float(f["bytes_per_row"]) * active_rows
        if "bytes_per_launch" in f:
            return float(f["bytes_per_launch"])
    return None


def exp_rate_probe(dev, sms: int):
    """Results per clock per SM of ex2.approx, the exponential the kernels use
    (bil_probe_exp_rate: 8 blocks of 256 threads per SM, 8 independent chains per
    thread); median, min and max over the SMs, from each SM's own cycle counter."""
    import ctypes

    import torch

    from invariant_token_log_gb300 import _lib
    lib = _lib.load()
    blocks = 8 * sms
    rec = torch.zeros(3 * blocks, dtype=torch.int64, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    iters = 4096
    for it in (256, iters):  # a short warm-up launch, then the measured one
        _lib.check("bil_probe_exp_rate", lib.bil_probe_exp_rate(blocks, it, sink.data_ptr(), rec.data_ptr(), stream))
    torch.cuda.synchronize(dev)
    r = rec.cpu().numpy().reshape(blocks, 3)
    per_sm = {}
    for smid, t0, t1 in r:
        lo, hi, k = per_sm.get(int(smid), (t0, t1, 0))
        per_sm[int(smid)] = (min(lo, t0), max(hi, t1), k + 1)
    rates = sorted(k * 256 * 8 * iters / float(hi - lo) for lo, hi, k in per_sm.values())
    return {"ex2_per_clk_per_sm": statistics.median(rates), "min": rates[0], "max": rates[-1],
            "sms": len(rates), "blocks": blocks, "iters": iters,
            "how": "bil_probe_exp_rate: 256-thread blocks, 8 per SM, 8 independent ex2.approx chains per thread; "
                   "results / span of the SM's clock64"}


def exp_secondary(variants, n, v, fwd_ms, bwd_ms, clocks):
    """The exponential unit as the second roofline of the logits path: one ex2 per
    element in the forward and in the backward.  demand_frac = exps per second
    needed at the measured time / (probe rate x SMs x median SM clock)."""
    if not variants or "sfu_exp" not in variants or not clocks.get("sm_mhz"):
        return None
    pr = variants["sfu_exp"]
    cap = pr["ex2_per_clk_per_sm"] * pr["sms"] * clocks["sm_mhz"] * 1e6  # ex2 per second
    out = {"bound": "sfu", "unit": "ex2/clk/SM", "peak": pr["ex2_per_clk_per_sm"], "sm_mhz": clocks["sm_mhz"],
           "fwd_demand_frac": n * v / (fwd_ms / 1e3) / cap, "bwd_demand_frac": n * v / (bwd_ms / 1e3) / cap}
    ent = variants.get("entropy_temperature_0.7")
    if ent:
        out["entropy_fwd_demand_frac"] = n * v / (ent["fwd_ms"] / 1e3) / cap
    return out


def host_link_probe(x_host, x_dev, out_host, dev, rows_per_copy: int = 4096, reps: int = 3):
    """Pinned host <-> device copy rates over the links the end-to-end figure
    crosses: host to device alone, device to host alone, and both at once (on two
    streams), each of `rows_per_copy` rows of the logits per copy."""
    import torch
    r = min(rows_per_copy, x_host.shape[0] // 2)
    src_h, dst_d = x_host[:r], torch.empty_like(x_dev[:r])
    src_d, dst_h = x_dev[r:2 * r], out_host[r:2 * r]
    nbytes = src_h.numel() * src_h.element_size()
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return time.perf_counter() - t0

    def h2d():
        with torch.cuda.stream(s1):
            dst_d.copy_(src_h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            dst_h.copy_(src_d, non_blocking=True)

    def both():
        h2d()
        d2h()
    h2d()
    d2h()
    t_h2d, t_d2h, t_both = timed(h2d), timed(d2h), timed(both)
    del dst_d
    return {"h2d_gbs": reps * nbytes / t_h2d / 1e9, "d2h_gbs": reps * nbytes / t_d2h / 1e9,
            "both_gbs": 2 * reps * nbytes / t_both / 1e9, "bytes_per_copy": nbytes, "reps": reps,
            "how": "pinned host <-> device tensor copies on their own streams, host wall clock around "
                   "synchronised batches",
            "trace": host_link_trace(x_host, x_dev, out_host, dev)}


def host_link_trace(x_host, x_dev, out_host, dev, iters: int = 40):
    """The host link alone over about a second, without the library: each iteration copies the whole
    pinned host logits to the device and the whole device logits back (the end-to-end step's bytes,
    one copy per direction on its own stream), timed with CUDA events.  Iterations well above the
    median show stalls of the link itself, which the end-to-end steps meet as well."""
    import torch
    cur = torch.cuda.current_stream(dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def it():
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        with torch.cuda.stream(s1):
            x_dev.copy_(x_host, non_blocking=True)   # the same bytes the device copy already holds
        with torch.cuda.stream(s2):
            out_host.copy_(x_dev, non_blocking=True)
        cur.wait_stream(s1)
        cur.wait_stream(s2)
    it()
    torch.cuda.synchronize(dev)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    marks[0].record(cur)
    for i in range(iters):
        it()
        marks[i + 1].record(cur)
    torch.cuda.synchronize(dev)
    ms = [round(marks[i].elapsed_time(marks[i + 1]), 2) for i in range(iters)]
    med = statistics.median(ms)
    return {"iter_ms": ms, "median_ms": med, "mean_ms": statistics.mean(ms),
            "stalled_iters": sum(m > 1.5 * med for m in ms),
            "bytes_per_iter": 2 * x_host.numel() * x_host.element_size()}


def secondary_measurements(bil, x, t, g, w, logp, lse, d, n, fwd_bytes, bwd_bytes, stream, dev):
    """The entropy output with a temperature of 0.7 (forward with the entropy, backward with an
    entropy gradient) on the same batch, and the forward's latency on decode-sized batches (the
    first N rows).  Outside the timed region of the headline value."""
    import torch

    gh = torch.from_numpy(np.random.default_rng(7).standard_normal(n).astype(np.float32)).to(dev)
    ent = torch.empty(n, dtype=torch.float32, device=dev)

    def step_ent():
        bil.logp_fwd(x, t, w.ignore_index, w.tile_v, out=logp, lse=lse, temperature=0.7, entropy=ent)
        bil.logp_bwd(x, t, lse, g, w.ignore_index, out=d, temperature=0.7, entropy=ent, grad_entropy=gh)
    for _ in range(3):
        step_ent()
    KV = 20
    evv = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KV)]
    for i in range(KV):
        evv[i][0].record(stream)
        bil.logp_fwd(x, t, w.ignore_index, w.tile_v, out=logp, lse=lse, temperature=0.7, entropy=ent)
        evv[i][1].record(stream)
        bil.logp_bwd(x, t, lse, g, w.ignore_index, out=d, temperature=0.7, entropy=ent, grad_entropy=gh)
        evv[i][2].record(stream)
    torch.cuda.synchronize(dev)
    ef = statistics.mean(e[0].elapsed_time(e[1]) for e in evv)
    eb = statistics.mean(e[1].elapsed_time(e[2]) for e in evv)
    variants = {"entropy_temperature_0.7": {
        "fwd_ms": ef, "fwd_gbs": (fwd_bytes + 4 * n) / (ef / 1e3) / 1e9,
        "bwd_ms": eb, "bwd_gbs": (bwd_bytes + 8 * n) / (eb / 1e3) / 1e9, "steps": KV}}
    # decode-sized batches: device time per forward call on the first N rows,
    # from a CUDA graph of 20 calls (so the host's per-call cost does not count),
    # and the same 20 calls issued one by one from Python (host-bound)
    lat, eager, eager_pre, eager_nolse = {}, {}, {}, {}
    for nd in (1, 2, 3, 7, 64, 128, 256):
        xs, ts = x[:nd], t[:nd]
        os_, ls_ = logp[:nd], lse[:nd]
        for _ in range(5):
            bil.logp_fwd(xs, ts, w.ignore_index, w.tile_v)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for res, kw in ((eager, {}), (eager_pre, {"out": os_, "lse": ls_}), (eager_nolse, {"with_lse": False})):
            e0.record(stream)
            for _ in range(20):
                bil.logp_fwd(xs, ts, w.ignore_index, w.tile_v, **kw)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            res[str(nd)] = round(e0.elapsed_time(e1) / 20 * 1e3, 2)
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="thread_local"):
                for _ in range(20):
                    bil.logp_fwd(xs, ts, w.ignore_index, w.tile_v)
            graph.replay()
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for _ in range(5):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            lat[str(nd)] = round(e0.elapsed_time(e1) / 100 * 1e3, 2)
            del graph
        except RuntimeError as exc:  # no graph: report the host-bound figure only
            lat[str(nd)] = f"unavailable: {str(exc).splitlines()[0][:80]}"
    variants["decode_fwd_us_per_call_graph"] = lat
    variants["decode_fwd_us_per_call_python"] = eager
    variants["decode_fwd_us_per_call_python_preallocated"] = eager_pre
    variants["decode_fwd_us_per_call_python_logp_only"] = eager_nolse  # with_lse=False: one allocation
    variants["prefill_fwd"] = prefill_measurement(bil, stream, dev)
    variants["sfu_exp"] = exp_rate_probe(dev, torch.cuda.get_device_properties(dev).multi_processor_count)
    variants["linear"] = linear_measurement(bil, stream, dev)
    return variants


def linear_measurement(bil, stream, dev, steps: int = 5):
    """The fused LM-head + logp step at full size: hidden [16384, 4096] bf16 times a
    Qwen3-8B-shaped LM head [151936, 4096] bf16 (the `--workload linear` batch).
    Forward: tile partials from the tensor-core accumulator, then the merge.
    Backward, queued step by step through the public calls it is made of: dZ
    from the recomputed projection, dhidden = dZ . W and dweight = dZ^T . X (the
    products read dZ, W and X where they lie).  Each step is timed with CUDA events on the
    launching stream, `steps` steps after 2 warm-up steps, clocks sampled
    meanwhile.  Outside the timed region of the headline value."""
    import torch

    import workloads as wl

    lw = wl.linear(16384)
    n, h, v = lw.n_rows, lw.hidden_size, lw.vocab
    x = torch.from_numpy(lw.hidden.view(np.int16)).view(torch.bfloat16).to(dev)
    wt = torch.from_numpy(lw.weight.view(np.int16)).view(torch.bfloat16).to(dev)
    t = torch.from_numpy(lw.target_ids).to(dev)
    g = torch.from_numpy(lw.grad_logp).to(dev)
    nt = -(-v // bil.LINEAR_TILE_V)
    pm = torch.empty((n, nt), dtype=torch.float32, device=dev)
    ps = torch.empty((n, nt), dtype=torch.float32, device=dev)
    tl = torch.empty(n, dtype=torch.float32, device=dev)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)

    def parts():
        bil.linear_logp_partials(x, wt, t, v, 0, nt, pm, ps, tl)

    def merge():
        bil.logp_merge(pm, ps, nt, tl, t, v, out=logp, lse=lse)
    state = {}

    def grad():
        state["dz"] = bil.linear_logp_grad(x, wt, t, lse, g)

    def dhidden():
        state["dh"] = bil.matmul(state["dz"], wt, out_dtype=torch.bfloat16)

    def dweight():
        state["dw"] = bil.matmul(state["dz"].t(), x, out_dtype=torch.bfloat16)
    seq = [("partials", parts), ("merge", merge), ("grad", grad), ("dhidden", dhidden), ("dweight", dweight)]
    for _ in range(2):
        for _, f in seq:
            f()
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(seq) + 1)] for _ in range(steps)]
    host_t0 = time.time()
    for i in range(steps):
        ev[i][0].record(stream)
        for j, (_, f) in enumerate(seq):
            f()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    host_t1 = time.time()
    sampler.stop()
    ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j, (name, _) in enumerate(seq)}
    step_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in ev)
    flops = 2.0 * n * h * v
    _, sustained, kind = tensor_peak()
    bwd_ms = ms["grad"] + ms["dhidden"] + ms["dweight"]
    out = {"workload": LINEAR_WORKLOAD, "steps": steps, "step_ms": step_ms, "rows_per_s": n / (step_ms / 1e3),
           "tflops": 4 * flops / (step_ms / 1e3) / 1e12, "fwd_ms": ms["partials"] + ms["merge"],
           "fwd_tflops": flops / (ms["partials"] / 1e3) / 1e12, "bwd_ms": bwd_ms,
           "bwd_tflops": 3 * flops / (bwd_ms / 1e3) / 1e12, "peak_sustained_tflops": sustained,
           "peak_source": f"{kind} cuBLAS bf16, sustained", "clocks": sampler.summary(host_t0, host_t1)}
    out["bwd_frac_of_sustained"] = out["bwd_tflops"] / sustained
    out["fwd_frac_of_sustained"] = out["fwd_tflops"] / sustained
    for name in ("grad", "dhidden", "dweight"):
        out[f"{name}_ms"] = ms[name]
        out[f"{name}_tflops"] = flops / (ms[name] / 1e3) / 1e12
    out["merge_ms"] = ms["merge"]

    # The same step with the forward's float32 logits kept for the backward (keep_logits): dZ by the
    # logits path's backward from them instead of a recomputing GEMM; the same bits, 4 bytes per row
    # and vocabulary column held from the forward to the backward.
    ws = torch.empty(bil.linear.workspace_bytes(n, v), dtype=torch.uint8, device=dev)

    def fwd_keep():
        state["lp"], state["lse"], state["logits"] = bil.linear_logp(x, wt, t, workspace=ws, return_logits=True,
                                                                     logits_dtype=torch.float32)

    def bwd_keep():
        state["dh"], state["dw"] = bil.linear.linear_logp_bwd_from_logits(x, wt, t, state["logits"], state["lse"], g)
    keep_seq = [("forward", fwd_keep), ("backward", bwd_keep)]
    for _ in range(2):
        for _, f in keep_seq:
            f()
    torch.cuda.synchronize(dev)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        kev[i][0].record(stream)
        for j, (_, f) in enumerate(keep_seq):
            f()
            kev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    k_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in kev)
    k_bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in kev)
    out["keep_logits"] = {"step_ms": k_fwd + k_bwd, "rows_per_s": n / ((k_fwd + k_bwd) / 1e3), "fwd_ms": k_fwd,
                          "bwd_ms": k_bwd, "logits_bytes": n * v * 4, "gemms": 3,
                          "how": "linear_logp(return_logits=True, float32) + linear_logp_bwd_from_logits; the same "
                                 "bits as the recomputing backward"}
    del state, pm, ps, x, wt, ws
    return out


def prefill_measurement(bil, stream, dev):
    """Forward of the prefill batch: 4096 rows (B=4, T=1024) of V=151936 bf16 logits at a
    padded pitch of 155648 columns (-inf pads, never read), 5% of the rows ignored (their
    logits are not read either).  Device time per call over 20 calls after 3 warm-up calls,
    CUDA events on the launching stream; bytes are counted for the active rows, and also for
    all rows to compare with figures quoted on N * V."""
    import torch

    import workloads as wl

    w = wl.prefill()
    x = torch.from_numpy(np.ascontiguousarray(w.logits).view(np.int16)).view(torch.bfloat16).to(dev)
    t = torch.from_numpy(w.target_ids).to(dev)
    n, v = w.n_rows, w.vocab
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    for _ in range(3):
        bil.logp_fwd(x, t, w.ignore_index, w.tile_v, vocab=v, out=logp, lse=lse)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record(stream)
    for _ in range(reps):
        bil.logp_fwd(x, t, w.ignore_index, w.tile_v, vocab=v, out=logp, lse=lse)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / reps
    active = int((w.target_ids != w.ignore_index).sum())
    peak, _ = hbm_peak()
    gbs_active = (active * v * 2 + n * 16) / (ms / 1e3) / 1e9
    return {"ms": ms, "rows_per_s": n / (ms / 1e3), "rows": n, "active_rows": active, "ld": int(x.shape[1]),
            "gbs": gbs_active, "frac": gbs_active / peak,
            "gbs_on_all_rows": n * v * 2 / (ms / 1e3) / 1e9}


def training_config(rows_per_gpu: int, world: int) -> dict:
    """The workload's `config`, the same on the CUDA arm and the reference arm."""
    return {"workload": WORKLOAD, "rows_per_gpu": rows_per_gpu, "vocab": 151936, "tile_v": 4096,
            "storage": "bf16 logits, bf16 dlogits, fp32 logp/lse",
            "l2": "no flush: every pass reads 4.98 GB of logits, 38x the 129 MB L2",
            "parallelism": f"dp{world} (independent row batches per GPU)"}


def run_bil(args):
    import torch

    import invariant_token_log_gb300 as bil
    import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    bil.load()

    w = wl.training(n_rows=args.rows)
    n, v = w.n_rows, w.vocab
    stored = np.ascontiguousarray(w.logits).view(np.int16)
    x_host = torch.from_numpy(stored).view(torch.bfloat16).pin_memory()
    t_host = torch.from_numpy(w.target_ids).pin_memory()
    g_host = torch.from_numpy(w.grad_logp).pin_memory()
    x = x_host.to(dev)
    t = t_host.to(dev)
    g = g_host.to(dev)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    d = torch.empty(n, v, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    # --entropy / --temperature: the same step with the entropy output (and its
    # gradient) and a temperature, for profiling those kernels; not the headline
    ent = torch.empty(n, dtype=torch.float32, device=dev) if args.entropy else None
    gh = torch.from_numpy(np.random.default_rng(7).standard_normal(n).astype(np.float32)).to(dev) \
        if args.entropy else None
    temp = args.temperature

    def fwd():
        bil.logp_fwd(x, t, w.ignore_index, w.tile_v, out=logp, lse=lse, temperature=temp, entropy=ent)

    def bwd():
        bil.logp_bwd(x, t, lse, g, w.ignore_index, out=d, temperature=temp, entropy=ent, grad_entropy=gh)

    def step():
        fwd()
        bwd()

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    host_t0 = time.time()
    for i in range(K):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    host_t1 = time.time()
    barrier(dist, dev)
    total_ms = ev[0][0].elapsed_time(ev[-1][2])
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)

    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_step, value = aggregate(n, world, K, total_ms)
    rows_total = n * world

    active = int((w.target_ids != w.ignore_index).sum())
    fwd_bytes = active * v * 2 + n * (8 + 4 + 4)                 # logits read; targets, logp, lse
    bwd_bytes = active * v * 2 + n * v * 2 + n * (8 + 4 + 4)     # logits read, dlogits write; targets, lse, g
    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms)
    peak, peak_kind = hbm_peak()
    bwd_gbs = bwd_bytes / (bwd_avg / 1e3) / 1e9
    fwd_gbs = fwd_bytes / (fwd_avg / 1e3) / 1e9
    step_gbs = (fwd_bytes + bwd_bytes) / (ms_step / 1e3) / 1e9  # per GPU

    # ---- secondary measurements (outside the timed region of `value`) ----
    variants = None
    if not args.no_variants:
        variants = secondary_measurements(bil, x, t, g, w, logp, lse, d, n, fwd_bytes, bwd_bytes, stream, dev)

    # ---- end to end: pinned host inputs -> device -> kernels -> host results ----
    # Through the public API for host-resident batches (HostStreamedLogp):
    # row chunks stream in, are computed and stream out on three CUDA streams.
    e2e = None
    if args.e2e_steps > 0:
        del d  # the streamed path keeps its own chunk buffers
        d_host = torch.empty((n, v), dtype=torch.bfloat16).pin_memory()
        logp_host = torch.empty(n, dtype=torch.float32).pin_memory()
        pipe = bil.HostStreamedLogp(n, v, torch.bfloat16, torch.bfloat16, chunk_rows=2048, device=dev)

        def e2e_step():
            # the host inputs are written by the CPU once: no queued work produces them, so each
            # step's copies in may start while the step before is still copying out
            return pipe.run(x_host, t_host, g_host, logp_host, d_host, w.ignore_index, w.tile_v,
                            order_inputs=False)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
        launches = 0
        # The steps are queued ahead of the GPU; a long pause of the host thread
        # can still leave it idle.  Collect once before timing and keep the
        # benchmark's own (static) heap out of later collections' scans.
        gc.collect()
        gc.freeze()
        marks[0].record(stream)
        for i in range(args.e2e_steps):
            launches += e2e_step()
            marks[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        gc.unfreeze()
        e2e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), dist, dev)
        step_ms = [round(marks[i].elapsed_time(marks[i + 1]), 2) for i in range(args.e2e_steps)]
        h2d = x_host.numel() * 2 + t_host.numel() * 8 + g_host.numel() * 4
        d2h = d_host.numel() * 2 + logp_host.numel() * 4
        e2e = {"value": rows_total * args.e2e_steps / (e2e_ms / 1e3), "unit": "rows/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.e2e_steps, "steps": args.e2e_steps,
               "path": "HostStreamedLogp: pinned host -> 2048-row chunks over 3 streams -> pinned host; a "
                       "step's copies in overlap the step before's copies out",
               "host_link_gbs": (h2d + d2h) / (e2e_ms / args.e2e_steps / 1e3) / 1e9,
               "gpu_launches": launches, "step_ms": step_ms,
               "step_ms_median": statistics.median(step_ms),
               "host_link_probe": host_link_probe(x_host, x, d_host, dev)}
        del pipe, d_host

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows_cpu = min(n, CPU_BASELINE_ROWS)
        rps, dt, cores = oracle_rows_per_s(rows_cpu, w=w)
        what = "all" if rows_cpu == n else "the first"
        cpu = {"value": rps, "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"{what} {rows_cpu} rows of the workload, forward + backward, float64 oracle, "
                         f"{dt:.1f} s wall"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, host-generated)",
            "config": dict(training_config(n, world), **({"entropy": True} if args.entropy else {}),
                           **({"temperature": args.temperature} if args.temperature != 1.0 else {})),
            "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak, "hbm_frac_of": f"{peak_kind} HBM copy bandwidth",
            "hbm_frac_nominal": step_gbs / NOMINAL_HBM_GBS,
            "kernels": {
                "logp_fwd": {"ms": fwd_avg, "gbs": fwd_gbs, "bytes": fwd_bytes, "frac": fwd_gbs / peak,
                             "frac_nominal": fwd_gbs / NOMINAL_HBM_GBS},
                "logp_bwd": {"ms": bwd_avg, "gbs": bwd_gbs, "bytes": bwd_bytes, "frac": bwd_gbs / peak,
                             "frac_nominal": bwd_gbs / NOMINAL_HBM_GBS},
            },
            "roofline": {"kernel": "bwd_kernel (logp_bwd)", "bound": "hbm", "achieved": bwd_gbs, "peak": peak,
                         "peak_source": f"{peak_kind} HBM copy bandwidth", "unit": "GB/s",
                         "frac": bwd_gbs / peak, "frac_nominal": bwd_gbs / NOMINAL_HBM_GBS,
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "traffic": ncu_traffic("bwd_kernel", active_rows=active),
                         "algorithmic_bytes_per_launch": bwd_bytes,
                         "secondary": exp_secondary(variants, n, v, fwd_avg, bwd_avg, clocks)},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * K, "clocks": clocks,
            "variants": variants,
        }
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the fused LM-head + logp
# ---------------------------------------------------------------------------

def _linear_oracle_step(x, w, t, g):
    import oracle
    oracle.linear_logp_fwd(x, w, "bfloat16", t)
    oracle.linear_logp_bwd(x, w, "bfloat16", t, g)


def oracle_linear_rows_per_s(rows: int):
    """Time the CPU oracle's LM-head projection, forward and backward over `rows` rows."""
    import oracle
    import workloads as wl
    oracle.build()
    x = wl.linear_hidden(rows)
    w = wl.linear_weight()
    t = wl.rng(wl.SEEDS["linear"], 1).integers(0, w.shape[0], rows, dtype=np.int64)
    g = wl.rng(wl.SEEDS["linear"], 5).standard_normal(rows)
    t0 = time.perf_counter()
    _linear_oracle_step(x, w, t, g)
    dt = time.perf_counter() - t0
    return rows / dt, dt, oracle.num_threads()


def run_linear_reference(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads as wl
    oracle.build()
    rows = LINEAR_REFERENCE_ROWS
    x = wl.linear_hidden(rows)
    w = wl.linear_weight()
    t = wl.rng(wl.SEEDS["linear"], 1).integers(0, w.shape[0], rows, dtype=np.int64)
    g = wl.rng(wl.SEEDS["linear"], 5).standard_normal(rows)
    for _ in range(args.warmup):
        _linear_oracle_step(x, w, t, g)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _linear_oracle_step(x, w, t, g)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": LINEAR_METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, host-generated)",
        "config": {"workload": LINEAR_WORKLOAD, "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{rows} rows of the workload per step, float64 oracle, projection, forward "
                                   "and backward"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_linear(args):
    import torch

    import invariant_token_log_gb300 as bil
    import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    bil.load()

    lw = wl.linear(args.rows)
    n, h, v = lw.n_rows, lw.hidden_size, lw.vocab
    x_host = torch.from_numpy(lw.hidden.view(np.int16)).view(torch.bfloat16).pin_memory()
    t_host = torch.from_numpy(lw.target_ids).pin_memory()
    g_host = torch.from_numpy(lw.grad_logp).pin_memory()
    x = x_host.to(dev)
    t = t_host.to(dev)
    g = g_host.to(dev)
    wt = torch.from_numpy(lw.weight.view(np.int16)).view(torch.bfloat16).to(dev)
    nt = -(-v // bil.LINEAR_TILE_V)
    pm = torch.empty((n, nt), dtype=torch.float32, device=dev)
    ps = torch.empty((n, nt), dtype=torch.float32, device=dev)
    tl = torch.empty(n, dtype=torch.float32, device=dev)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        bil.linear_logp_partials(x, wt, t, v, 0, nt, pm, ps, tl)
        bil.logp_merge(pm, ps, nt, tl, t, v, out=logp, lse=lse)
        bil.linear_logp_bwd(x, wt, t, lse, g)

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    host_t0 = time.time()
    for i in range(K):
        ev[i][0].record(stream)
        bil.linear_logp_partials(x, wt, t, v, 0, nt, pm, ps, tl)
        ev[i][1].record(stream)
        bil.logp_merge(pm, ps, nt, tl, t, v, out=logp, lse=lse)
        ev[i][2].record(stream)
        bil.linear_logp_bwd(x, wt, t, lse, g)
        ev[i][3].record(stream)
    torch.cuda.synchronize(dev)
    host_t1 = time.time()
    barrier(dist, dev)
    total_ms = ev[0][0].elapsed_time(ev[-1][3])
    part_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    merge_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    scratch = n * v * 2  # the backward's scratch: dZ (bf16)
    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_step, value = aggregate(n, world, K, total_ms)
    flops = 2.0 * n * h * v           # one projection-sized GEMM
    step_flops = 4 * flops            # forward, recomputation, dhidden, dweight
    tflops = flops / (part_ms / 1e3) / 1e12
    burst, sustained, peak_kind = tensor_peak()
    # the kernel is timed inside a loop of K back-to-back launches (seconds under
    # the power cap), so the sustained figure is its denominator
    peak = sustained

    e2e = None
    if args.e2e_steps > 0:
        logp_host = torch.empty(n, dtype=torch.float32).pin_memory()
        lse_host = torch.empty(n, dtype=torch.float32).pin_memory()
        ws = torch.empty(bil.linear.workspace_bytes(n, v), dtype=torch.uint8, device=dev)
        xd = torch.empty_like(x)
        td = torch.empty_like(t)
        gd = torch.empty_like(g)

        def e2e_step():
            xd.copy_(x_host, non_blocking=True)
            td.copy_(t_host, non_blocking=True)
            gd.copy_(g_host, non_blocking=True)
            lp, ls = bil.linear_logp(xd, wt, td, workspace=ws)
            bil.linear_logp_bwd(xd, wt, td, ls, gd)
            logp_host.copy_(lp, non_blocking=True)
            lse_host.copy_(ls, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
        marks[0].record(stream)
        for i in range(args.e2e_steps):
            e2e_step()
            marks[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), dist, dev)
        h2d = x_host.numel() * 2 + t_host.numel() * 8 + g_host.numel() * 4
        d2h = logp_host.numel() * 4 + lse_host.numel() * 4
        e2e = {"value": n * world * args.e2e_steps / (e2e_ms / 1e3), "unit": "rows/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.e2e_steps,
               "steps": args.e2e_steps,
               "path": "linear_logp + linear_logp_bwd: pinned host hidden states, targets, g -> device (weight "
                       "resident; dhidden and dweight stay on the device for the optimizer) -> pinned host logp, lse"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rps, dt, cores = oracle_linear_rows_per_s(LINEAR_CPU_ROWS)
        cpu = {"value": rps, "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"first {LINEAR_CPU_ROWS} rows of the workload, float64 projection, forward and "
                         f"backward, {dt:.1f} s wall"}
    if rank == 0:
        print(json.dumps({
            "metric": LINEAR_METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, host-generated)",
            "config": {"workload": LINEAR_WORKLOAD, "rows_per_gpu": n, "hidden": h, "vocab": v,
                       "tile_v": bil.LINEAR_TILE_V,
                       "l2": "no flush: every pass reads the 1.25 GB LM-head weight, 9.6x the 129 MB L2",
                       "parallelism": f"dp{world} (independent row batches per GPU, weight replicated)"},
            "tflops": step_flops / (ms_step / 1e3) / 1e12,
            "kernels": {"linear_partials": {"ms": part_ms, "tflops": tflops},
                        "logp_merge": {"ms": merge_ms},
                        "linear_logp_bwd": {"ms": bwd_ms, "tflops": 3 * flops / (bwd_ms / 1e3) / 1e12,
                                            "launches": 3, "scratch_bytes": scratch}},
            "roofline": {"kernel": "linear_partials_kernel", "bound": "tensor", "achieved": tflops, "peak": peak,
                         "peak_source": f"{peak_kind} sustained dense bf16 (burst {burst})", "unit": "TFLOP/s",
                         "frac": tflops / peak, "frac_of_burst": tflops / burst,
                         "traffic": ncu_traffic("linear_partials_kernel", LINEAR_SOURCE, active_rows=n),
                         "algorithmic_flops_per_launch": flops},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 5 * K, "clocks": clocks,
        }), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.workload == "linear":
        run_linear_reference(args) if args.impl == "reference" else run_linear(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_bil(args)


if __name__ == "__main__":
    main()
