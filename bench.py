"""Benchmark of the OScaR INT2 decode path on GB300.

Headline line (the workload the metric is quoted on): one step = one decode
step of one attention layer for the batch-48, 128K-context workload (32 query
/ 8 KV heads, head_dim 128): rotate the queries, append the new token's key
and value (the full residual window is flushed to INT2 every 128 steps, and
the run is arranged so that at least one flush falls inside the timed
steps), then the fused INT2 dequant + inverse scaling + split-K attention
with the log-sum-exp combine in its last CTA per row.  The packed cache
(about 4.35 GB read per step) is far larger than L2, so no flush of L2 is
needed between steps.

Prints one JSON line: value = device time per step (us, CUDA events over the
timed steps, max over ranks); e2e = the same through the C ABI with the step's
inputs copied from pinned host memory and the output read back every step;
roofline = the fused decode call against the measured HBM copy bandwidth;
configs = the other workloads (decode with L2 flushed before every rep, and
the streaming ones' whole steps); cpu_baseline = the CPU oracle on a bounded
sample, single thread and on all cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import os

# the CPU oracle leg is timed per process single-threaded (its BLAS calls must
# not fan out; the all-core timing runs one process per core)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np

WORKLOAD = "batch48_128k"
METRIC = "INT2 decode-attn µs/step & HBM GB/s (% of GB300 peak) at 128K ctx, batch 48"
UNIT = "us/step"
HERE = os.path.dirname(os.path.abspath(__file__))
TRAFFIC_FILE = os.path.join(HERE, "profiles", "decode_int2_batch48_128k_traffic.json")
L2_BYTES = 129 * 10**6             # GB300 L2
L2_FLUSH_BYTES = 512 << 20          # written before every flushed rep (about 4x L2)
CONFIG_WORKLOADS = ("tiny_1k", "qwen3_8b_32k", "long_stream_128k", "omni_tni_64k")
ABLATION_WORKLOADS = ("tiny_1k", "qwen3_8b_32k", "omni_tni_64k")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1024)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-bf16", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=256)
    p.add_argument("--no-paged", action="store_true",
                   help="skip the paged-cache decode over a variable-length batch")
    p.add_argument("--no-int4", action="store_true",
                   help="skip the INT4-option decode of the same workload")
    p.add_argument("--no-ablation", action="store_true",
                   help="skip the accuracy report of the variants against bf16 attention")
    p.add_argument("--no-prefill", action="store_true",
                   help="skip the prefill timing (fused vs two-call) of the prompt")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads' decode and stream timings")
    p.add_argument("--num-splits", type=int, default=0,
                   help="split-K count of the INT2 decode (0: the library's planner)")
    p.add_argument("--workload", default=WORKLOAD,
                   help="workload name (the headline line uses the default; others are "
                        "for profiling small cases)")
    return p.parse_args()


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _metric(wl):
    if wl.name == WORKLOAD:
        return METRIC
    return (f"INT2 decode-attn µs/step & HBM GB/s (% of GB300 peak), {wl.name}: batch {wl.B}, "
            f"{wl.Hq} q / {wl.Hkv} KV heads, {wl.T0} tokens")


def _cache_bytes(wl):
    return wl.B * wl.Hkv * (wl.n_packed * 86 + wl.n_res * 514)


def _config(wl, S=None):
    gb = _cache_bytes(wl) / 1e9
    cfg = {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": 128,
           "context": wl.T0, "key_group": 32, "residual_window": 128,
           "step": "rotate_q + append_kv (flush every 128) + fused INT2 decode with the "
                   "LSE combine in its last CTA per row, as three calls (step_compare times "
                   "the same step as one oscar_decode_step launch)",
           "l2": (f"inputs larger than L2: ~{gb:.2f} GB packed cache read per step vs 129 MB L2"
                  if gb > 2 * 0.129 else
                  f"~{gb * 1e3:.0f} MB packed cache; L2 flushed ({L2_FLUSH_BYTES >> 20} MB "
                  f"written) before every timed rep"),
           "parallelism": "replicas (one independent layer cache per GPU)"}
    if S is not None:
        cfg["num_splits"] = S
    return cfg


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi polled every 50 ms in a child process; a reader thread
    collects the lines.  ``wait_first`` returns once the first sample arrived,
    so the tool's own start-up never overlaps the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import threading
        self.lines = []
        self.proc = None
        self.first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            self.first.set()
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)
            self.first.set()
        self.first.set()

    def wait_first(self, timeout=20.0):
        self.first.wait(timeout)

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)
        rows = []
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append({"t": ts, "sm": float(f[2]), "sm_max": float(f[3]),
                             "power": float(f[4]) if f[4] not in ("[N/A]", "") else None,
                             "hw_slowdown": f[6], "hw_thermal": f[7], "sw_thermal": f[8],
                             "sw_power_cap": f[9]})
            except (ValueError, IndexError):
                continue
        return rows


def _clock_summary(rows, t0, t1):
    inside = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05]
    window = "timed"
    if len(inside) < 3:
        inside, window = rows, "benchmark run (timed region shorter than the sampling period)"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    reasons = set()
    for r in inside:
        for k in ("hw_slowdown", "hw_thermal", "sw_thermal", "sw_power_cap"):
            if r[k].lower().startswith("active"):
                reasons.add(k)
    return {"sm_mhz": statistics.median(r["sm"] for r in inside),
            "sm_max_mhz": max(r["sm_max"] for r in inside),
            "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# CPU oracle (bounded sample)
# ---------------------------------------------------------------------------

def _oracle_row_cache(wl, b, h, T_hist, timing=None):
    """The oracle's cache of row (b, h) over the workload's prompt; with a
    list `timing`, the seconds of the oracle's prefix build (rotate, scale,
    quantise) are appended to it."""
    from oracle import oscar_oracle as O
    kb = wl.k_bits([b], [h], 0, T_hist)[0, 0]
    vb = wl.v_bits([b], [h], 0, T_hist)[0, 0]
    t = time.perf_counter()
    hc = O.build_head_cache(kb[:wl.T0], vb[:wl.T0], wl.n_packed)
    if timing is not None:
        timing.append(time.perf_counter() - t)
    return hc, kb, vb


def cpu_baseline_configs(names, steps=2):
    """The oracle on each other workload: single-threaded on one row (its
    prefix build, i.e. rotate, scale, quantise the prompt, and `steps` decode
    steps), then on all host cores (one spawned process per core, one row
    each, all at once); each extrapolated to all the workload's rows."""
    from int2_kv_cache_02_gb300 import workloads as W
    res = {}
    for name in names:
        wl = W.WORKLOADS[name]
        rows = wl.B * wl.Hkv
        tb = []
        hc, kb, vb = _oracle_row_cache(wl, 0, 0, wl.T0 + steps + 1, timing=tb)
        t = _oracle_steps(wl, hc, kb, vb, 0, 0, 0, steps)
        res[name] = {"decode_us_per_step": t / steps * rows * 1e6,
                     "prefix_quantize_us": tb[0] * rows * 1e6, "cores": 1, "kind": "oracle",
                     "sample": f"row (0, 0) of {rows}: its prompt's prefix build and {steps} "
                               f"decode steps, single thread; extrapolated x{rows} rows"}
    ncpu = os.cpu_count() or 1
    try:
        import multiprocessing as mp
        with mp.get_context("spawn").Pool(ncpu) as pool:
            for name in names:
                wl = W.WORKLOADS[name]
                rows = wl.B * wl.Hkv
                jobs = [(name, r // wl.Hkv % wl.B, r % wl.Hkv, steps)
                        for r in range(min(ncpu, rows))]
                # the processes build and step their rows at the same time:
                # the slowest sets the rate of len(jobs) rows
                times = pool.map(_oracle_worker_timed, jobs, chunksize=1)
                build, step = max(x[0] for x in times), max(x[1] for x in times)
                res[name]["all_cores"] = {
                    "decode_us_per_step": step / steps * rows / len(jobs) * 1e6,
                    "prefix_quantize_us": build * rows / len(jobs) * 1e6,
                    "cores": len(jobs), "kind": "oracle",
                    "sample": f"{len(jobs)} rows in {len(jobs)} single-threaded processes at "
                              f"once, each its prefix build and {steps} decode steps; "
                              f"extrapolated x{rows / len(jobs):.1f}"}
    except Exception as e:  # a host without room for the processes keeps the 1-thread figures
        for name in names:
            res[name]["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"}
    return res


def _truncate_packed(hc, keep):
    """Keep only the first ``keep`` packed tokens of an oracle HeadCache."""
    from oracle import oscar_oracle as O
    kq, vq = hc.packed_k(), hc.packed_v()
    hc.k_codes = [O.QuantK(kq.codes[:keep], kq.step16[:keep // 32], kq.zero16[:keep // 32])]
    hc.k_norm16 = [hc.packed_norm16()[:keep]]
    hc.v_q = [O.QuantV(vq.codes[:keep], vq.step16[:keep], vq.zero16[:keep])]


def _oracle_steps(wl, hc, kb, vb, b, h, i0, n):
    """n oracle decode steps of one row: rotate its queries, append the new
    token (flush-before-append), attend over the row's cache.  Returns seconds."""
    from oracle import oscar_oracle as O
    g, tau = wl.g, 1.0 / math.sqrt(128)
    qs = [wl.q_bits([b], range(h * g, (h + 1) * g), i)[0] for i in range(i0, i0 + n)]
    t = time.perf_counter()
    for j in range(n):
        hc.append(kb[wl.T0 + i0 + j], vb[wl.T0 + i0 + j])
        hc.decode(O.rotate_q(qs[j]), tau)
    return time.perf_counter() - t


def _oracle_worker(job):
    """One process of the all-core oracle timing: builds row (b, h)'s cache and
    times n decode steps of it (single-threaded).  Module-level so that a
    spawned pool can run it."""
    name, b, h, n = job
    sys.path.insert(0, HERE)
    from int2_kv_cache_02_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    hc, kb, vb = _oracle_row_cache(wl, b, h, wl.T0 + n + 1)
    return _oracle_steps(wl, hc, kb, vb, b, h, 0, n)


def _oracle_worker_timed(job):
    """One process of the all-core oracle timing of a workload: seconds of
    row (b, h)'s prefix build and of its n decode steps (single-threaded)."""
    name, b, h, n = job
    sys.path.insert(0, HERE)
    from int2_kv_cache_02_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    tb = []
    hc, kb, vb = _oracle_row_cache(wl, b, h, wl.T0 + n + 1, timing=tb)
    return tb[0], _oracle_steps(wl, hc, kb, vb, b, h, 0, n)


def cpu_baseline(wl, budget_s=20.0):
    """The oracle as it stands, timed on this host's cores: one thread on 2
    rows, then one process per core on as many rows in parallel."""
    rows = [(0, 0), (wl.B - 1, wl.Hkv - 1)]
    max_steps = 20
    tb = []
    built = [(b, h) + _oracle_row_cache(wl, b, h, wl.T0 + max_steps + 1, timing=tb)
             for (b, h) in rows]
    b, h, hc, kb, vb = built[0]
    t1 = _oracle_steps(wl, hc, kb, vb, b, h, 0, 1)           # calibration step (untimed)
    n = max(1, min(max_steps, int(budget_s / max(t1, 1e-3) / len(rows))))
    tot = 0.0
    for k, (b, h, hc, kb, vb) in enumerate(built):
        tot += _oracle_steps(wl, hc, kb, vb, b, h, 1 if k == 0 else 0, n)
    per = tot / (n * len(rows))
    total_rows = wl.B * wl.Hkv
    out = {"value": per * total_rows * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{len(rows)} of {total_rows} (sequence, KV head) rows x {n} decode steps "
                     f"at full context, single thread; extrapolated x{total_rows} rows",
           "host_cores": os.cpu_count(),
           "prefix_quantize": {"value": sum(tb) / len(tb) * total_rows * 1e6, "unit": "us",
                               "cores": 1, "kind": "oracle",
                               "sample": f"the prompt's prefix build (rotate, scale, quantise "
                                         f"{wl.n_packed} tokens) of {len(tb)} rows, single "
                                         f"thread; extrapolated x{total_rows} rows"}}
    # all cores: one spawned process per core, one row each (the pool starts
    # with `spawn`: a forked child of a CUDA process can hang)
    ncpu = os.cpu_count() or 1
    rows_all = [(wl.name, r // wl.Hkv % wl.B, r % wl.Hkv, n) for r in range(min(ncpu, total_rows))]
    try:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        t0 = time.perf_counter()
        with ctx.Pool(len(rows_all)) as pool:
            times = pool.map(_oracle_worker, rows_all)
        wall = time.perf_counter() - t0
        # the processes ran their n steps concurrently: the slowest sets the
        # rate of len(rows_all) rows per n steps
        per_all = max(times) / n
        out["all_cores"] = {
            "value": per_all * total_rows / len(rows_all) * 1e6, "unit": UNIT,
            "cores": len(rows_all), "kind": "oracle",
            "sample": f"{len(rows_all)} rows in {len(rows_all)} single-threaded processes, "
                      f"{n} decode steps each at full context (their cache builds untimed, "
                      f"{wall:.1f} s in all); extrapolated x{total_rows / len(rows_all):.1f}"}
    except Exception as e:  # a host without room for the processes keeps the 1-thread figure
        out["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"}
    return out


# ---------------------------------------------------------------------------
# reference arm: the oracle as the timed program
# ---------------------------------------------------------------------------

def kernel_code_sha256() -> str:
    """sha256 of the decode kernel's source with comments and blank lines
    removed: the key of the stored traffic record, which a change of code
    (not of comments) invalidates."""
    import hashlib
    import re
    with open(os.path.join(HERE, "int2_kv_cache_02_gb300", "csrc", "decode_int2.cu")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def run_reference(args, world, rank):
    from int2_kv_cache_02_gb300 import workloads as W
    if rank != 0:
        return 0
    wl = W.WORKLOADS[args.workload]
    total_rows = wl.B * wl.Hkv
    steps = args.steps + args.warmup
    hc, kb, vb = _oracle_row_cache(wl, 0, 0, wl.T0 + steps + 1)
    probe = _oracle_steps(wl, hc, kb, vb, 0, 0, 0, 1)       # untimed size probe
    # size each step so that the whole run stays within about two minutes
    frac = min(1.0, max(1.0 / 64, (120.0 / max(steps, 1)) / max(probe, 1e-6)))
    keep = max(32, int(hc.n_packed * frac) // 32 * 32)
    _truncate_packed(hc, keep)
    _oracle_steps(wl, hc, kb, vb, 0, 0, 1, args.warmup)
    t = _oracle_steps(wl, hc, kb, vb, 0, 0, 1 + args.warmup, args.steps)
    per = t / max(args.steps, 1)
    scale = total_rows * (wl.n_packed / keep)
    value = per * scale * 1e6
    sample = (f"1 of {total_rows} rows per step, {keep} packed tokens (+ residual) of the "
              f"row (the workload's prompt has {wl.n_packed}), single thread; extrapolated "
              f"x{scale:.1f} (rows x packed-token ratio)")
    line = {"impl": "reference", "metric": _metric(wl), "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": value / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": _config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "host_cores": os.cpu_count()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def _algorithmic_bytes(wl, n_packed, n_res, S):
    rows = wl.B * wl.Hkv
    cache = rows * (n_packed * 86 + n_res * 514)
    qo = 2 * wl.B * wl.Hq * 128 * 4                      # q' in, out
    ws = 2 * wl.B * wl.Hq * (S + 1) * 132 * 4             # partials written and read
    return cache + qo + ws


def _peaks():
    try:
        with open(os.path.join(HERE, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def _median_timed(fn, reps, flushbuf=None):
    """Median device time (us) of fn() over reps, each bracketed by CUDA
    events on the current stream; with flushbuf, the buffer is written
    before every rep, outside the events."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a, b in evs:
        if flushbuf is not None:
            flushbuf.zero_()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    return ts[len(ts) // 2], ts


def _read_only_peak(dev) -> float:
    """GB/s of a read-only stream on this GPU: a sum over 4 GiB of fp32, best
    of 5 (context for the roofline, whose peak is a copy: read + write)."""
    import torch
    x = torch.ones(1 << 30, dtype=torch.float32, device=dev)
    for _ in range(2):
        x.sum()
    best = float("inf")
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        x.sum()
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) * 1e-3)
    del x
    torch.cuda.empty_cache()
    return (1 << 30) * 4 / best / 1e9


def _flush_loop_timed(fn, reps, flushbuf):
    """Device time (us) of fn() with L2 flushed before it: reps of (flush,
    fn) back to back between two CUDA events, less reps of the flush alone.
    Event pairs around one short launch read in steps of about 1 us on this
    GPU, so the loop gives the finer figure."""
    import torch
    a, b, c, d = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    a.record()
    for _ in range(reps):
        flushbuf.zero_()
        fn()
    b.record()
    c.record()
    for _ in range(reps):
        flushbuf.zero_()
    d.record()
    torch.cuda.synchronize()
    return (a.elapsed_time(b) - c.elapsed_time(d)) * 1e3 / reps


def measure_config(L, W, name, dev, flushbuf, peak, reps=100):
    """One workload other than the headline one: the fused decode over its
    prompt (plus one appended token) with L2 flushed before every rep, and
    for the streaming workloads the whole decode step (oscar_decode_step: rotate_q, append with
    the flushes every 128 tokens, decode) over the workload's 256 steps, L2
    flushed before every step."""
    import torch
    wl = W.WORKLOADS[name]
    tau = 1.0 / math.sqrt(128)
    steps = max(wl.steps, 1)
    K, V = W.draw_kv_cuda(wl, 0, wl.T0, device=dev)
    cache = W.build_cache_cuda(wl, K, V, T_cap=wl.t_cap(steps - wl.steps + 1), device=dev)
    del K, V
    Kn, Vn = W.draw_kv_cuda(wl, wl.T0, steps + 1, device=dev)
    Kn = Kn.permute(2, 0, 1, 3).contiguous()
    Vn = Vn.permute(2, 0, 1, 3).contiguous()
    Q = torch.stack([W.draw_q_cuda(wl, i, device=dev) for i in range(steps + 1)])
    qr = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device=dev)
    out = torch.empty_like(qr)
    S_max = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, cache.T_cap)
    ws = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, cache.T_cap,
                                                    max(S_max, 64)), device=dev)
    res = {"B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "context": wl.T0}
    if wl.n_packed:
        # decode over the prompt + the first appended token
        L.append_kv(cache, Kn[0], Vn[0], n_tok=1)
        L.rotate_q(Q[0], qr)
        S = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, cache.n_packed)
        dec = lambda: L.decode_attention(cache, qr, wl.Hq, tau, out, ws, num_splits=S)
        for _ in range(3):
            dec()
        us = _flush_loop_timed(dec, reps, flushbuf)
        us_ev, _ = _median_timed(dec, 20, flushbuf)
        nbytes = _algorithmic_bytes(wl, cache.n_packed, cache.n_res, S)
        gbs = nbytes / (us * 1e-6) / 1e9
        res.update({"num_splits": S, "packed_tokens": cache.n_packed,
                    "residual_tokens": cache.n_res, "decode_us": us,
                    "decode_us_event_median": us_ev,
                    "algorithmic_bytes": nbytes, "GB/s": gbs, "frac": gbs / peak,
                    "l2": f"flushed ({L2_FLUSH_BYTES >> 20} MB written) before each of {reps} "
                          "back-to-back reps; decode_us = (flush + decode) loop less the "
                          "flush-only loop, per rep; decode_us_event_median = median of 20 "
                          "event pairs around single launches (coarser)"})
    if wl.steps > 1:
        # the workload's decode steps, one by one, from the next token on
        n_st = wl.steps - 1
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_st)]
        flushes, nbytes = 0, 0
        for i, (a, b) in enumerate(evs):
            flushbuf.zero_()
            if cache.n_res == 128:
                flushes += 1
            a.record()
            L.decode_step(cache, Q[i + 1], Kn[i + 1], Vn[i + 1], wl.Hq, tau, out, ws)
            b.record()
            S = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, cache.n_packed)
            nbytes += _algorithmic_bytes(wl, cache.n_packed, cache.n_res, S)
        torch.cuda.synchronize()
        st = [a.elapsed_time(b) * 1e3 for a, b in evs]
        us = float(np.mean(st))
        gbs = nbytes / n_st / (us * 1e-6) / 1e9
        res["stream"] = {"steps": n_st, "flushes": flushes, "us_per_step": us,
                         "us_per_step_median": float(np.median(st)), "GB/s": gbs,
                         "frac": gbs / peak,
                         "note": "whole decode step (oscar_decode_step: rotate_q + append + "
                                 "decode in one launch, the flush before it when the window "
                                 "is full), L2 flushed before every step; GB/s counts the "
                                 "decode's algorithmic bytes only"}
    if L.device_status() != 0:
        raise RuntimeError(f"{name}: a kernel recorded an error")
    del cache, ws, Kn, Vn, Q
    torch.cuda.empty_cache()
    return res


ABLATION_VARIANTS = (("oscar", 0, 2), ("no_rotate (scaling only)", 1, 2),
                     ("no_scale (rotation only)", 2, 2), ("neither (KIVI-style)", 3, 2),
                     ("all_heads_norm", 4, 2), ("oscar_int4", 0, 4))


def ablation_report(L, W, dev):
    """Accuracy of the method and its ablations against unquantised bf16
    attention, on inputs whose attention is concentrated so that the
    reference output is far from zero: tiny_1k and qwen3_8b_32k with needle
    keys (a few keys per row point at the row's queries with graded score
    margins), omni_tni_64k as it is (its x30 tokens and x10 segments already
    draw most of the attention).  GPU: every row of the workload, against the
    bf16 split-K kernel on the same raw keys and values.  Oracle, row (0, 0):
    its own quantised attention against its own exact bf16 attention, and the
    same with quantised keys but exact values (the part rotation and scaling
    act on).  Information only, not a gate."""
    import torch
    from oracle import oscar_oracle as O
    tau = 1.0 / math.sqrt(128)
    rep = {"inputs": {"tiny_1k": "needles", "qwen3_8b_32k": "needles",
                      "omni_tni_64k": "the workload's own keys (no needles)"},
           "needles": f"{W.N_NEEDLES} keys per (sequence, KV head) row at seeded positions in "
                      f"the packed prefix, along the mean of the row's query group (tilted by a "
                      f"seeded tenth), scoring ln(context) + {list(W.NEEDLE_MARGINS)} nats; "
                      f"values unchanged; decode step 0",
           "reference": "bf16 attention over the same raw keys and values",
           "metric": "relative L2 error of the whole output ('rel_l2'); median over the "
                     "(sequence, query head) vectors ('median'); oracle 'keys_only': "
                     "quantised keys with exact values",
           "workloads": {}}
    for name in ABLATION_WORKLOADS:
        wl = W.WORKLOADS[name]
        needles = name != "omni_tni_64k"
        K, V = W.draw_kv_cuda(wl, 0, wl.T0, device=dev)
        if needles:
            W.plant_needles_cuda(wl, K)
        q = W.draw_q_cuda(wl, 0, device=dev)
        ref = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device=dev)
        wsr = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, wl.T0, 512),
                                device=dev)
        L.bf16_decode_attention(q, K, V, wl.B, wl.Hq, wl.Hkv, wl.T0, wl.T0, tau, ref, wsr,
                                num_splits=0)
        qr = torch.empty_like(ref)
        gpu = {}
        for vname, fl, bits in ABLATION_VARIANTS:
            cv = L.KVCache(wl.B, wl.Hkv, wl.n_packed, flags=fl, device=dev, bits=bits)
            L.prefill_kv(cv, K, V, n_tok=wl.n_packed, in_T=wl.T0)
            if wl.n_res:
                L.append_kv(cv, K[:, :, wl.n_packed:wl.T0].contiguous(),
                            V[:, :, wl.n_packed:wl.T0].contiguous(), n_tok=wl.n_res)
            L.rotate_q(q, qr, flags=fl)
            wsv = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, cv.n_packed),
                                    device=dev)
            ov = torch.empty_like(ref)
            L.decode_attention(cv, qr, wl.Hq, tau, ov, wsv)
            torch.cuda.synchronize()
            if L.device_status() != 0:
                raise RuntimeError(f"ablation {name} / {vname}: a kernel recorded an error")
            d = (ov - ref).double()
            per = torch.linalg.vector_norm(d, dim=-1) / torch.linalg.vector_norm(ref.double(),
                                                                                 dim=-1)
            gpu[vname] = {"rel_l2": float(torch.linalg.vector_norm(d)
                                          / torch.linalg.vector_norm(ref.double())),
                          "median": float(per.median())}
            del cv, wsv, ov
        del K, V, wsr
        torch.cuda.empty_cache()
        # the oracle on row (0, 0), per-head norm variants
        kb = wl.k_bits([0], [0], 0, wl.T0)[0, 0]
        if needles:
            kb = W.plant_needles(wl, kb, 0, 0)
        vb = wl.v_bits([0], [0], 0, wl.T0)[0, 0]
        qb = wl.q_bits([0], range(wl.g), 0)[0]
        oref = O.bf16_attention(qb, kb, vb, tau)
        vexact = O.bf16_to_f64(vb)
        orc = {}
        for vname, fl, bits in ABLATION_VARIANTS:
            if fl & O.NORM_ALL_HEADS:
                continue                         # spans every head of the token: GPU only
            hc = O.build_head_cache(kb, vb, wl.n_packed, fl, bits=bits)
            qrot = O.rotate_q(qb, fl)
            o = hc.decode(qrot, tau)
            keys, _ = hc.keys_values()
            ok = O.attention(np.atleast_2d(qrot), keys, vexact, tau)
            orc[vname] = {"rel_l2": float(np.linalg.norm(o - oref) / np.linalg.norm(oref)),
                          "keys_only": float(np.linalg.norm(ok - oref) / np.linalg.norm(oref))}
        rep["workloads"][name] = {"gpu": gpu, "oracle_row_0_0": orc}
    return rep


def run_ours(args, world, rank, local):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sys.path.insert(0, HERE)
    import __graft_entry__
    __graft_entry__.build()
    from int2_kv_cache_02_gb300 import oscar as L
    from int2_kv_cache_02_gb300 import workloads as W

    wl = W.WORKLOADS[args.workload]
    tau = 1.0 / math.sqrt(128)
    W_, K_ = args.warmup, args.steps
    E_ = args.e2e_steps
    flush_at = min(max(K_ // 2, 0), 64)         # timed step at which a flush falls
    N3 = 130   # steps of the three-call comparison leg (one flush among them)
    total_steps = W_ + 128 + K_ + 2 + E_ + N3
    T_cap = wl.t_cap(total_steps - wl.steps)
    peaks = _peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "of measured" if peak else "of fallback"
    peak = peak or 6800.0

    # prompt: raw K, V drawn on the device, cache built through the library
    K, V = W.draw_kv_cuda(wl, 0, wl.T0, device=dev)
    cache = W.build_cache_cuda(wl, K, V, T_cap=T_cap, device=dev)
    # per-step inputs, one contiguous slice per step
    Kn, Vn = W.draw_kv_cuda(wl, wl.T0, total_steps, device=dev)
    Kn = Kn.permute(2, 0, 1, 3).contiguous()
    Vn = Vn.permute(2, 0, 1, 3).contiguous()
    Q = torch.stack([W.draw_q_cuda(wl, i, device=dev) for i in range(total_steps)])
    torch.cuda.synchronize()

    S = args.num_splits or L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, wl.n_packed)
    ws = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, T_cap, S), device=dev)
    qr = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device=dev)
    out = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        # one decode step as three calls: rotate_q, append (with the flush of
        # a full window), decode; ev brackets the decode
        L.rotate_q(Q[i], qr)
        L.append_kv(cache, Kn[i], Vn[i], n_tok=1)
        if ev is not None:
            ev[0].record(stream)
        L.decode_attention(cache, qr, wl.Hq, tau, out, ws, num_splits=S)
        if ev is not None:
            ev[1].record(stream)

    def step_fused(i):
        # the same step in one call (one launch; two on a flush step)
        L.decode_step(cache, Q[i], Kn[i], Vn[i], wl.Hq, tau, out, ws, num_splits=S)

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    vis = [v for v in vis.split(",") if v.strip().isdigit()]
    sampler = ClockSampler(int(vis[local]) if local < len(vis) else local)
    sampler.wait_first()
    i_step = 0
    for _ in range(W_):
        step(i_step)
        i_step += 1
    # untimed steps until the residual window fills at timed step flush_at, so
    # that the timed steps include a flush (one every 128 steps)
    while (cache.n_res + flush_at) % 128 != 0 and K_ > 0:
        step(i_step)
        i_step += 1
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ctx0 = (cache.n_packed, cache.n_res)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K_)]
    st_evs = [torch.cuda.Event(enable_timing=True) for _ in range(K_ + 1)]
    flush_steps = []
    launches0 = L.kernel_launches()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    bytes_sum = 0
    for j in range(K_):
        if cache.n_res == 128:
            flush_steps.append(j)
        st_evs[j].record(stream)
        step(i_step, evs[j])
        i_step += 1
        bytes_sum += _algorithmic_bytes(wl, cache.n_packed, cache.n_res, S)
    if K_:
        st_evs[K_].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    launches = L.kernel_launches() - launches0
    clock_rows = sampler.stop()
    if L.device_status() != 0:
        raise RuntimeError("a kernel recorded an error during the benchmark")

    step_us = [st_evs[j].elapsed_time(st_evs[j + 1]) * 1e3 for j in range(K_)]
    # the part of each step before the decode: rotate_q and append_kv, with
    # the flush when the window is full
    pre_us = [st_evs[j].elapsed_time(evs[j][0]) * 1e3 for j in range(K_)]
    flush_obj = None
    if flush_steps:
        plain = [t for j, t in enumerate(pre_us) if j not in flush_steps]
        base_us = float(np.median(plain)) if plain else float("nan")
        with_f = [pre_us[j] for j in flush_steps]
        rows_ = wl.B * wl.Hkv
        fb = rows_ * 128 * (256 + 2 + 256) + rows_ * 4 * 2752   # read the window, write 4 records
        extra = float(np.mean(with_f)) - base_us
        flush_obj = {"timed_steps_with_flush": flush_steps,
                     "step_us_with_flush": [step_us[j] for j in flush_steps],
                     "pre_decode_us_with_flush": with_f,
                     "median_pre_decode_us_without": base_us, "flush_us": extra,
                     "flush_GB/s": fb / (extra * 1e-6) / 1e9 if extra > 0.5 else None,
                     "algorithmic_bytes": fb,
                     "note": "a flush quantises the batch's full residual windows (128 tokens "
                             "per row: rotated keys, norms and values read, 4 records per row "
                             "written); its cost is the time of the step's rotate_q + append "
                             "with the flush minus the median of the other steps' (the whole "
                             "step is no measure: after a flush the decode's residual is one "
                             "token, so its decode is shorter)"}
    ms_total = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(b) for a, b in evs]
    ms_step = max_over_ranks(ms_total / max(K_, 1), world, dev)
    dec_avg_ms = float(np.mean(dec_ms)) if dec_ms else float("nan")
    achieved = (bytes_sum / max(K_, 1)) / (dec_avg_ms * 1e-3) / 1e9

    # ---- end to end through the C ABI with host buffers ----
    e2e_us, h2d, d2h = None, 0, 0
    if E_ > 0:
        pin = lambda t: t.cpu().pin_memory()
        base = i_step + 2
        Qh, Kh, Vh = pin(Q[base:base + E_]), pin(Kn[base:base + E_]), pin(Vn[base:base + E_])
        outh = torch.empty((E_,) + tuple(out.shape), dtype=torch.float32).pin_memory()
        # Copies run on their own stream, double-buffered, so that step i + 1's
        # inputs travel and step i - 1's output returns while step i computes;
        # every copy is still inside the timed region.
        cs = torch.cuda.Stream(device=dev)
        qd = [torch.empty_like(Q[0]) for _ in range(2)]
        kd = [torch.empty_like(Kn[0]) for _ in range(2)]
        vd = [torch.empty_like(Vn[0]) for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        filled = [torch.cuda.Event() for _ in range(2)]   # inputs of buffer b on the device
        used = [torch.cuda.Event() for _ in range(2)]     # step done with buffer b
        back = [torch.cuda.Event() for _ in range(2)]     # output of buffer b on the host
        for i in range(2):  # untimed: touch the copy paths
            qd[i].copy_(Qh[i], non_blocking=True)
        torch.cuda.synchronize()

        def h2d_(i):
            b = i % 2
            with torch.cuda.stream(cs):
                if i >= 2:
                    cs.wait_event(used[b])
                qd[b].copy_(Qh[i], non_blocking=True)
                kd[b].copy_(Kh[i], non_blocking=True)
                vd[b].copy_(Vh[i], non_blocking=True)
                filled[b].record(cs)

        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cs.wait_event(e0)
        h2d_(0)
        for i in range(E_):
            b = i % 2
            if i + 1 < E_:
                h2d_(i + 1)
            stream.wait_event(filled[b])
            if i >= 2:
                stream.wait_event(back[b])
            L.rotate_q(qd[b], qr)
            L.append_kv(cache, kd[b], vd[b], n_tok=1)
            L.decode_attention(cache, qr, wl.Hq, tau, outs[b], ws, num_splits=S)
            used[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(used[b])
                outh[i].copy_(outs[b], non_blocking=True)
                back[b].record(cs)
        stream.wait_event(back[(E_ - 1) % 2])
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_us = e0.elapsed_time(e1) / max(E_, 1) * 1e3
        h2d = (Qh[0].numel() * Qh.element_size() + Kh[0].numel() * Kh.element_size()
               + Vh[0].numel() * Vh.element_size())
        d2h = out.numel() * out.element_size()
        e2e_us = max_over_ranks(e2e_us, world, dev)

    # ---- the fused step (oscar_decode_step) against the three calls ----
    # alternating on the same cache, so that both see the same context
    i3 = (i_step + 2 + E_) if E_ > 0 else (i_step + 2)
    t_fused, t_three = [], []
    for j in range(N3):
        a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush_now = cache.n_res == 128
        a3.record(stream)
        if j % 2:
            step_fused(i3 + j)
        else:
            step(i3 + j)
        b3.record(stream)
        if not flush_now:
            (t_fused if j % 2 else t_three).append((a3, b3))
    torch.cuda.synchronize()
    if L.device_status() != 0:
        raise RuntimeError("a kernel recorded an error in the step comparison")
    step_compare = {"fused_step_us_median": float(np.median([a.elapsed_time(b) * 1e3
                                                              for a, b in t_fused])),
                    "three_call_step_us_median": float(np.median([a.elapsed_time(b) * 1e3
                                                                  for a, b in t_three])),
                    "steps": N3,
                    "note": "oscar_decode_step (one launch) against rotate_q + append_kv + "
                            "decode_attention (three launches), alternating on the same cache "
                            "(flush steps left out); the timed steps above use the three calls"}

    # ---- bf16 comparison kernel, same shape (context T0) ----
    bf16 = None
    if not args.no_bf16:
        qb = Q[0]
        ws16 = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, wl.T0, 512),
                                 device=dev)
        o16 = torch.empty_like(out)
        run16 = lambda: L.bf16_decode_attention(qb, K, V, wl.B, wl.Hq, wl.Hkv, wl.T0, wl.T0,
                                                tau, o16, ws16, num_splits=0)
        for _ in range(3):
            run16()
        torch.cuda.synchronize()
        reps = 20
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            run16()
        b.record(stream)
        torch.cuda.synchronize()
        bf_ms = a.elapsed_time(b) / reps
        bf_bytes = wl.B * wl.Hkv * wl.T0 * 512
        bf16 = {"us_per_call": bf_ms * 1e3, "GB/s": bf_bytes / (bf_ms * 1e-3) / 1e9,
                "frac": bf_bytes / (bf_ms * 1e-3) / 1e9 / peak,
                "int2_decode_speedup": bf_ms / dec_avg_ms,
                "note": f"equal-shape bf16 split-K decode (B{wl.B}, {wl.Hq}/{wl.Hkv}, "
                        f"{wl.T0} tokens), {bf_bytes / 1e9:.1f} GB of K,V per call"}
        del ws16

    # ---- prefill of the prompt's packed part: fused vs two-call path ----
    prefill = None
    if not args.no_prefill and wl.n_packed:
        def time_build(fused, reps=3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(reps):
                c = L.KVCache(wl.B, wl.Hkv, wl.n_packed, device=dev)
                torch.cuda.synchronize()
                a.record(stream)
                if fused:
                    L.prefill_kv(c, K, V, n_tok=wl.n_packed, in_T=wl.T0)
                else:
                    W.prefill_two_call(c, K, V, wl.n_packed, device=dev)
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
                del c
            return sorted(ts)[len(ts) // 2]
        f_ms = time_build(True)
        s_ms = time_build(False)
        th = wl.B * wl.Hkv * wl.n_packed
        f_bytes = th * (256 + 256 + 86)          # read k, v; write the records
        prefill = {"tokens": wl.n_packed, "fused_us": f_ms * 1e3,
                   "fused_GB/s": f_bytes / (f_ms * 1e-3) / 1e9,
                   "fused_frac": f_bytes / (f_ms * 1e-3) / 1e9 / peak,
                   "two_call_us": s_ms * 1e3, "speedup": s_ms / f_ms,
                   "note": "rotate + scale + quantise of the prompt's packed tokens; "
                           "algorithmic bytes 598 per token-head (fused)"}
    # ---- paged cache: the same prompt at variable lengths, shuffled pages ----
    paged = None
    if not args.no_paged and wl.n_packed >= 4 * 32:
        rng = np.random.default_rng(wl.seed_k + 17)
        lo = max(32, (wl.n_packed // 4) // 32 * 32)
        n_tok_h = [int(x) // 32 * 32 for x in rng.integers(lo, wl.n_packed + 1, size=wl.B)]
        max_tok = max(n_tok_h)
        blocks = [n // 32 + 4 for n in n_tok_h]
        pc = L.PagedKVCache(wl.B, wl.Hkv, max(blocks), n_pages=sum(blocks), device=dev)
        pc.map_blocks(0, 0, order=list(rng.permutation(sum(blocks))))
        for b in range(wl.B):
            pc.map_blocks(b, blocks[b])
        L.paged_prefill_kv(pc, K, V, torch.tensor(n_tok_h, dtype=torch.int32, device=dev),
                           max_tok, in_T=wl.T0)
        L.paged_append_kv(pc, Kn[0], Vn[0])
        Sp = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, max_tok)
        wsp = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, max_tok, Sp),
                                device=dev)
        L.rotate_q(Q[0], qr)
        run_p = lambda: L.paged_decode_attention(pc, qr, wl.Hq, tau, max_tok, out, wsp,
                                                 num_splits=Sp)
        for _ in range(3):
            run_p()
        torch.cuda.synchronize()
        reps = 20
        a = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            run_p()
        b_.record(stream)
        torch.cuda.synchronize()
        if L.device_status() != 0:
            raise RuntimeError("paged decode recorded a device error")
        p_ms = a.elapsed_time(b_) / reps
        p_bytes = (sum(wl.Hkv * (n * 86 + 1 * 514) for n in n_tok_h)
                   + 2 * wl.B * wl.Hq * 128 * 4 + 2 * wl.B * wl.Hq * (Sp + 1) * 132 * 4)
        p_gbs = p_bytes / (p_ms * 1e-3) / 1e9
        del pc, wsp
        torch.cuda.empty_cache()
        # the contiguous cache at the batch's mean length, timed the same way
        n_mean = int(round(float(np.mean(n_tok_h)) / 32)) * 32
        cm = L.KVCache(wl.B, wl.Hkv, n_mean + 128, device=dev)
        L.prefill_kv(cm, K, V, n_tok=n_mean, in_T=wl.T0)
        L.append_kv(cm, Kn[0], Vn[0], n_tok=1)
        Sm = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, n_mean)
        wsm = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, n_mean, Sm),
                                device=dev)
        run_m = lambda: L.decode_attention(cm, qr, wl.Hq, tau, out, wsm, num_splits=Sm)
        for _ in range(3):
            run_m()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            run_m()
        b_.record(stream)
        torch.cuda.synchronize()
        if L.device_status() != 0:
            raise RuntimeError("contiguous decode recorded a device error")
        m_ms = a.elapsed_time(b_) / reps
        m_bytes = (wl.B * wl.Hkv * (n_mean * 86 + 514)
                   + 2 * wl.B * wl.Hq * 128 * 4 + 2 * wl.B * wl.Hq * (Sm + 1) * 132 * 4)
        m_gbs = m_bytes / (m_ms * 1e-3) / 1e9
        del cm, wsm
        torch.cuda.empty_cache()
        paged = {"sequences": wl.B, "packed_tokens_min": min(n_tok_h),
                 "packed_tokens_max": max_tok, "packed_tokens_mean": float(np.mean(n_tok_h)),
                 "pages": sum(blocks), "num_splits": Sp, "decode_us": p_ms * 1e3,
                 "GB/s": p_gbs, "frac": p_gbs / peak,
                 "contiguous_at_mean": {"packed_tokens": n_mean, "num_splits": Sm,
                                        "decode_us": m_ms * 1e3, "GB/s": m_gbs,
                                        "frac": m_gbs / peak},
                 "frac_vs_contiguous": p_gbs / m_gbs,
                 "note": "oscar_paged_decode_attention over per-sequence lengths drawn "
                         "uniformly in [n_packed/4, n_packed] (+1 residual token), pages "
                         "handed out in a shuffled order; contiguous_at_mean: "
                         "oscar_decode_attention on a contiguous cache of the same batch with "
                         "every sequence at the mean length"}
    # ---- INT4 option: the same prompt in 4800-byte records, decode only ----
    int4 = None
    if not args.no_int4 and wl.n_packed:
        c4 = L.KVCache(wl.B, wl.Hkv, wl.n_packed, device=dev, bits=4)
        L.prefill_kv(c4, K, V, n_tok=wl.n_packed, in_T=wl.T0)
        if wl.n_res:
            L.append_kv(c4, K[:, :, wl.n_packed:wl.T0].contiguous(),
                        V[:, :, wl.n_packed:wl.T0].contiguous(), n_tok=wl.n_res)
        S4 = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, c4.n_packed)
        ws4 = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, c4.n_packed, S4),
                                device=dev)
        L.rotate_q(Q[0], qr)
        run4 = lambda: L.decode_attention(c4, qr, wl.Hq, tau, out, ws4, num_splits=S4)
        for _ in range(3):
            run4()
        torch.cuda.synchronize()
        reps = 20
        a = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            run4()
        b_.record(stream)
        torch.cuda.synchronize()
        if L.device_status() != 0:
            raise RuntimeError("INT4 decode recorded a device error")
        i_ms = a.elapsed_time(b_) / reps
        rows = wl.B * wl.Hkv
        i_bytes = (rows * (c4.n_packed * 150 + c4.n_res * 514)
                   + 2 * wl.B * wl.Hq * 128 * 4 + 2 * wl.B * wl.Hq * (S4 + 1) * 132 * 4)
        i_gbs = i_bytes / (i_ms * 1e-3) / 1e9
        int4 = {"packed_tokens": c4.n_packed, "residual_tokens": c4.n_res, "num_splits": S4,
                "decode_us": i_ms * 1e3, "GB/s": i_gbs, "frac": i_gbs / peak,
                "note": "INT4 option (16 levels, 150 B per packed token-head) over the same "
                        "prompt; %.2f GB of records, %s" % (
                            rows * c4.n_packed * 150 / 1e9,
                            "L2 not flushed between the 20 reps (records larger than L2)"
                            if rows * c4.n_packed * 150 > 2 * L2_BYTES else
                            "L2 not flushed between the 20 reps (records fit in L2: a warm figure)")}
        del c4, ws4
        torch.cuda.empty_cache()
    # the headline workload's big buffers are not needed any more
    del K, V, Kn, Vn, cache, ws
    torch.cuda.empty_cache()

    # ---- the other workloads, each on its own ----
    configs = None
    if not args.no_configs and args.workload == WORKLOAD:
        flushbuf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        configs = {name: measure_config(L, W, name, dev, flushbuf, peak)
                   for name in CONFIG_WORKLOADS}
        del flushbuf
        torch.cuda.empty_cache()
    # ---- accuracy of the variants against unquantised bf16 attention ----
    ablation = None
    if not args.no_ablation and args.workload == WORKLOAD:
        ablation = ablation_report(L, W, dev)

    read_peak = _read_only_peak(dev)

    traffic = None
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        # counters taken on another version of the kernel do not describe this one
        if rec.get("kernel_code_sha256") == kernel_code_sha256() and wl.name == WORKLOAD:
            traffic = rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        traffic = None

    line = {
        "metric": _metric(wl), "value": ms_step * 1e3, "unit": UNIT, "n_gpus": world,
        "steps": K_, "warmup": W_, "ms_per_step": ms_step, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int2 codes; f16 tensor-core MMA (hi+lo split), f32 accumulate",
        "data": "synthetic", "config": _config(wl, S),
        "decode_tokens_per_s": world * wl.B / (ms_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src, "traffic": traffic,
                     "peak_note": "the measured copy bandwidth (read + write); a read-only "
                                  "stream can exceed it slightly (this library's INT4 decode "
                                  "reads at 1.02-1.04 of it), while torch.sum's read stream "
                                  "(read_only_peak) stays just below it",
                     "read_only_peak": {"GB/s": read_peak, "frac": achieved / read_peak,
                                        "how": "torch.sum over 4 GiB of fp32 on this GPU, "
                                               "best of 5, measured in this run (context)"},
                     "kernel": "oscar_decode_attention (fused INT2 decode, LSE combine in "
                               "the last CTA of each row)",
                     "decode_us": dec_avg_ms * 1e3,
                     "algorithmic_bytes_per_launch": bytes_sum / max(K_, 1)},
        "e2e": ({"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h, "steps": E_} if E_ > 0 else None),
        "gpu_launches": int(launches),
        "clocks": _clock_summary(clock_rows, wall0, wall1),
        "context_tokens": {"start": ctx0[0] + ctx0[1],
                           "end": ctx0[0] + ctx0[1] + K_},
        "flushes_in_timed_region": len(flush_steps),
        "flush": flush_obj,
        "step_compare": step_compare,
        "configs": configs,
        "prefill": prefill,
        "paged": paged,
        "int4": int4,
        "ablation": ablation,
    }
    if bf16 is not None:
        line["bf16_decode"] = bf16
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == WORKLOAD:
        line["cpu_baseline"] = cpu_baseline(wl)
        if not args.no_configs:
            line["cpu_baseline"]["configs"] = cpu_baseline_configs(CONFIG_WORKLOADS)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = _args()
    world, rank, local = _dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
