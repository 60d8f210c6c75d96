#!/usr/bin/env python
"""SANTA++ decode-step attention benchmark on GB300 — prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--cpu-seconds S] [--no-e2e] [--no-extra]

Workload: the Qwen2.5-7B-shaped decode attention layer at 32K context (1 sequence, 28 query
/ 4 KV heads, d = 128, T = 128, M = 31 draws, bf16 K/V, mixture keys), seeded synthetic
data.  A step is one SANTA++ decode step through santa_decode: one launch of the fused kernel
(team scoring and sampling, then split-K Horvitz-Thompson attention over the sampled teams).

value      steps/s of whole decode steps with inputs resident in HBM, K steps in one CUDA
           graph (see timing); the K/V/representative buffers rotate over R copies so that the
           bytes touched between two uses of a copy exceed 6x the L2 size.
roofline   the fused decode kernel (one launch per step): algorithmic bytes per launch (the
           team representatives, K and V of the sampled teams, q, out) / its mean duration
           (CUDA events around the K launches), against the measured HBM copy bandwidth.
e2e        the same steps through the C ABI with pinned host buffers: per step one call of
           santa_decode_host copies the query, page table and lengths host->device
           (StepInputs), runs the decode, copies out, draw/sampled ids, pi, |S| and the
           status word back device->host (packed DecodeBuffers) and waits for the stream.
dense      the in-run dense split-K decode kernel on the same buffers (speed reference).
workloads  the other full-size workloads (Qwen B=8 M=64, Llama paged B=16, 128K B=4) timed
           the same way, each with its roofline fraction and dense kernel, and the 128K
           workload's sweep over M in {16, 31, 64, 128}.
timing     every entry point's K steps run in one CUDA graph after one untimed step of the
           same entry point; the start event waits only for that step, so the K steps are
           timed as K step periods (each graph replayed untimed first, then once behind a
           spin kernel, so the events time the device only).
cpu_baseline  the fp64 C oracle, single-threaded, on a bounded sample of steps.
--impl reference  times that oracle alone (the reference arm of this benchmark).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn steps/s and achieved HBM GB/s at 32K ctx, M=31/64 teams, 1 GB300"
DEFAULT_WORKLOAD = "qwen7b_32k_b1_m31"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")
KERNEL_SOURCES = ["sampled_sparse_decode_gb300/csrc/decode_kernel.cuh",
                  "sampled_sparse_decode_gb300/csrc/common.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time the headline workload only (not the other full-size ones)")
    ap.add_argument("--mode", choices=["bench", "profile", "accuracy", "loop"], default="bench",
                    help="profile: W + K plain santa_decode (or --dense) steps on one copy of "
                         "the inputs, for ncu captures; accuracy: error of every sampler "
                         "against dense attention over many seeds; loop: a generation of "
                         "--gen-tokens steps (append + decode), fresh vs held sampled sets")
    ap.add_argument("--sampler", choices=["iid_ht", "systematic", "iid_hh"], default="iid_ht",
                    help="team sampler of the timed decode steps")
    ap.add_argument("--mix-alpha", type=float, default=0.0,
                    help="defensive mixture weight of the timed decode steps")
    ap.add_argument("--seeds", type=int, default=256, help="accuracy mode: seeds per sampler")
    ap.add_argument("--draws", type=int, default=None,
                    help="override the workload's number of draws M (for M sweeps)")
    ap.add_argument("--dense", action="store_true", help="profile mode: the dense kernel")
    ap.add_argument("--gen-tokens", type=int, default=4096,
                    help="loop mode: tokens generated after the workload's context")
    ap.add_argument("--refresh", default="16,64,256",
                    help="loop mode: hold periods R of the sampled set (comma separated)")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="write the per-launch DRAM traffic of the decode kernel, read from an "
                         "ncu --csv log of dram__bytes_read.sum and dram__bytes_write.sum "
                         "(bytes), to --traffic-out with the hash of the current kernel "
                         "sources, and exit")
    ap.add_argument("--traffic-out", default=None, help="where --record-traffic writes")
    ap.add_argument("--traffic-command", default="", help="the ncu command, for the record")
    return ap.parse_args()


# ---------------------------------------------------------------------------- helpers

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_rate(seconds, steps, world, device):
    """Whole-job rate of `world` replicas that each ran `steps` steps: the slowest rank's time
    (max over ranks, any torch.distributed backend) and world * steps / that time.
    Returns (rate, slowest seconds)."""
    import torch
    if world > 1:
        t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        seconds = float(t.item())
    return world * steps / seconds, seconds


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_cores():
    """The host's logical cores and the cores this process may run on."""
    try:
        allowed = sorted(os.sched_getaffinity(0))
    except AttributeError:
        allowed = list(range(os.cpu_count() or 1))
    return {"host_cores": os.cpu_count(), "affinity_cores": len(allowed),
            "affinity": _ranges(allowed)}


def _ranges(cores):
    """[0, 1, 2, 5] -> "0-2,5"."""
    out, i = [], 0
    while i < len(cores):
        j = i
        while j + 1 < len(cores) and cores[j + 1] == cores[j] + 1:
            j += 1
        out.append(f"{cores[i]}-{cores[j]}" if j > i else f"{cores[i]}")
        i = j + 1
    return ",".join(out)


def host_cores_note():
    h = host_cores()
    return (f"1 thread on a host of {h['host_cores']} cores "
            f"(affinity mask: {h['affinity_cores']} cores, {h['affinity']})")


def kernel_source_sha():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current kernel source and this workload (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha") == kernel_source_sha() and rec.get("workload") == workload:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


_BYTE_UNITS = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12}


def parse_ncu_traffic(csv_path, kernel_regex="decode_kernel"):
    """Per captured launch of the matching kernel (in launch order): (name, DRAM bytes read,
    DRAM bytes written), from an `ncu --csv` log with one row per metric."""
    import csv
    import re
    launches = {}
    with open(csv_path, newline="") as f:
        lines = [l for l in f if l.startswith('"')]       # drop ncu's own log lines
    for row in csv.DictReader(lines):
        name = row.get("Kernel Name", "")
        metric = row.get("Metric Name", "")
        if not re.search(kernel_regex, name) or metric not in ("dram__bytes_read.sum",
                                                                "dram__bytes_write.sum"):
            continue
        unit = _BYTE_UNITS[row.get("Metric Unit", "byte").strip().lower()]
        val = float(row["Metric Value"].replace(",", "")) * unit
        rec = launches.setdefault(int(row["ID"]), {"name": name})
        rec["read" if metric.endswith("read.sum") else "write"] = val
    return [(r["name"], r["read"], r["write"]) for _, r in sorted(launches.items())
            if "read" in r and "write" in r]


def record_traffic_file(csv_path, out_path, workload, command):
    """The committed traffic record: mean DRAM bytes per decode launch, keyed by the hash of
    the kernel sources this script sees, so the bench uses it only for those sources."""
    launches = parse_ncu_traffic(csv_path)
    if not launches:
        raise SystemExit(f"no decode_kernel launches with DRAM metrics in {csv_path}")
    rd = [r for _, r, _ in launches]
    wr = [w for _, _, w in launches]
    rec = {"kernel": launches[0][0], "workload": workload,
           "kernel_source_sha": kernel_source_sha(),
           "dram_bytes_per_launch": (sum(rd) + sum(wr)) / len(launches),
           "dram_bytes_read_per_launch": rd, "dram_bytes_write_per_launch": wr,
           "command": command,
           "note": "cold caches (ncu flushes them before each launch); written by "
                   "bench.py --record-traffic from the ncu log"}
    with open(out_path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms (read-only queries)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 - 0.15 <= t <= t1 + 0.15] or \
               [s for (_, s) in self.samples]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- oracle (CPU)

def oracle_steps_per_s(wl, seconds, max_steps=None, sampler="iid_ht", alpha=0.0):
    """The fp64 oracle, single-threaded, timed per decode step (reps precomputed)."""
    import oracle
    pr = oracle.Problem(wl.q, wl.k_pool, wl.v_pool, wl.page_table, wl.seq_lens)
    reps = oracle.build_reps(pr, wl.page_fill)
    cfg = wl.cfg
    steps = 0
    t0 = time.perf_counter()
    while True:
        for b in range(cfg.batch):
            for h in range(cfg.kv_heads):
                oracle.decode_ex(pr, reps, cfg.draws, steps, b, h, sampler, alpha)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_steps and steps >= max_steps):
            return steps / el, steps, el


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, same workload and metric.  Each
    step decodes a bounded sample of the step's (sequence, KV head) units, sized so that the
    whole run takes about two minutes, and the time is scaled to whole steps."""
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    from sampled_sparse_decode_gb300 import workloads as W
    wl = W.generate(args.workload, **({'draws': args.draws} if args.draws else {}))
    cfg = wl.cfg
    pr = oracle.Problem(wl.q, wl.k_pool, wl.v_pool, wl.page_table, wl.seq_lens)
    reps = oracle.build_reps(pr, wl.page_fill)
    units = [(b, h) for b in range(cfg.batch) for h in range(cfg.kv_heads)]
    t0 = time.perf_counter()
    smp, alpha = args.sampler, args.mix_alpha
    oracle.decode_ex(pr, reps, cfg.draws, 0, *units[0], smp, alpha)
    t_unit = time.perf_counter() - t0
    budget = 120.0
    per_step = budget / max(1, args.steps + args.warmup)
    n_units = int(min(len(units), max(1, per_step // max(t_unit, 1e-9))))
    steps = args.steps
    note = ""
    if n_units * t_unit * (steps + args.warmup) > 2 * budget:     # even one unit is too slow
        steps = max(1, int(budget / t_unit) - args.warmup)
        note = f"; {args.steps} steps asked, {steps} fit the time budget"
    sample_units = units[:n_units]
    for s_ in range(args.warmup):
        for b, h in sample_units:
            oracle.decode_ex(pr, reps, cfg.draws, s_, b, h, smp, alpha)
    t0 = time.perf_counter()
    for s_ in range(steps):
        for b, h in sample_units:
            oracle.decode_ex(pr, reps, cfg.draws, args.warmup + s_, b, h, smp, alpha)
    el = (time.perf_counter() - t0) * len(units) / n_units
    v = steps / el
    sample = (f"{steps} steps, each decoding {n_units} of the {len(units)} (sequence, KV head) "
              f"units; time scaled to whole steps{note}")
    print(json.dumps({
        "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": config_of(cfg, world),
        "sampler": {"name": smp, "mix_alpha": alpha},
        "cpu_baseline": {"value": v, "unit": "steps/s", "cores": 1, "kind": "oracle",
                         "sample": f"{sample}; {host_cores_note()}", **host_cores()},
        "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------------------- GPU arm

# Full-size workloads timed beside the headline one, each the same way, and the draw counts
# of the long-context sweep (against the same dense kernel).
EXTRA_WORKLOADS = ("qwen7b_32k_b8_m64", "llama8b_paged_32k_b16_m32", "long_128k_b4_m64")
SWEEP_WORKLOAD = "long_128k_b4_m64"
SWEEP_DRAWS = (16, 31, 64, 128)
SPIN_CYCLES = 400_000          # ~0.2 ms at 2 GHz: the host enqueues the timed graphs meanwhile


def config_of(cfg, world):
    """The workload description shared by both arms of the bench line."""
    return {"workload": cfg.name, "batch": cfg.batch, "q_heads": cfg.q_heads,
            "kv_heads": cfg.kv_heads, "head_dim": cfg.head_dim, "seq_len": cfg.seq_len,
            "team_size": cfg.team_size, "draws": cfg.draws,
            "parallelism": "replicas" if world > 1 else "1gpu",
            "l2": "inputs larger than L2: K, V and the representatives rotate over copies, "
                  ">= 6x the L2 size touched between two uses of a copy",
            "timing": "one CUDA graph per entry point: one untimed step, then the K timed "
                      "steps; CUDA events (start after the untimed step, end after step K), "
                      "the graph replayed untimed first, then timed behind a spin kernel"}


def _dev_tensor(a, dev):
    import numpy as np
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


class Rig:
    """One workload resident in HBM: R rotating copies of K, V and the representatives, so
    that the bytes the decode touches between two uses of a copy, (R - 1) steps' worth at
    |S| = M for the smallest M timed on it, exceed 6x the L2 size."""

    def __init__(self, name, dev, draws=None, min_draws=None):
        import torch
        import sampled_sparse_decode_gb300 as santa
        from sampled_sparse_decode_gb300 import workloads as W
        wl = W.generate(name, **({"draws": draws} if draws else {}))
        cfg = wl.cfg
        self.wl, self.cfg, self.dev = wl, cfg, dev
        self.esize = 2 if cfg.dtype == "bf16" else 4
        self.units = cfg.batch * cfg.kv_heads
        self.n_teams = wl.max_teams
        d, T = cfg.head_dim, cfg.team_size
        self.q = _dev_tensor(wl.q, dev)
        self.pt, self.lens, self.fill = (_dev_tensor(x, dev) for x in
                                         (wl.page_table, wl.seq_lens, wl.page_fill))
        k0, v0 = _dev_tensor(wl.k_pool, dev), _dev_tensor(wl.v_pool, dev)
        reps0 = santa.santa_build_reps(k0, self.fill)
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        m_small = min(cfg.draws, min_draws or cfg.draws, self.n_teams)
        self.touched = self.units * (self.n_teams * d * 4 + m_small * T * 2 * d * self.esize)
        pool = 2 * k0.numel() * self.esize + reps0.numel() * 4
        free, _ = torch.cuda.mem_get_info(dev)
        R = 1 + math.ceil(6 * self.l2 / self.touched)
        self.R = max(2, min(R, int(0.4 * free // pool)))
        self.ks = [k0] + [k0.clone() for _ in range(self.R - 1)]
        self.vs = [v0] + [v0.clone() for _ in range(self.R - 1)]
        self.reps = [reps0] + [reps0.clone() for _ in range(self.R - 1)]
        self.dense_kv = self.units * cfg.seq_len * 2 * d * self.esize

    def bufs(self, M, dense=False, team_probs=False):
        from sampled_sparse_decode_gb300 import binding as Bn
        c = self.cfg
        return Bn.DecodeBuffers.allocate(self.q.dtype, c.batch, c.q_heads, c.kv_heads,
                                         c.head_dim, c.team_size, self.n_teams, M, self.dev,
                                         dense=dense, team_probs=team_probs)

    def args(self, M, bufs, sampler="iid_ht", alpha=0.0, dense=False):
        """One argument structure per rotation copy; rotation r decodes with seed r."""
        from sampled_sparse_decode_gb300 import binding as Bn
        return [Bn._args(self.q, self.ks[r], self.vs[r], None if dense else self.reps[r],
                         self.pt, self.lens, 1 if dense else M, 0 if dense else r, bufs,
                         sampler, alpha) for r in range(self.R)]

    def step_bytes(self, mean_sel):
        """Algorithmic bytes of one decode step at the realised mean |S|: the representatives
        of every team, K and V of the sampled teams, q and out."""
        c = self.cfg
        d, T = c.head_dim, c.team_size
        return (self.units * self.n_teams * d * 4 + mean_sel * self.units * T * 2 * d * self.esize
                + c.batch * c.q_heads * d * (self.esize + 4))

    def sampled(self, M, a_list, bufs, lib, stream, call):
        """Mean |S| over the R seeds the graphs replay, and the share of teams whose sampling
        probability p_i (and inclusion probability pi_i) is below 1%, from seed 0."""
        import torch
        sel_total = 0
        with torch.cuda.stream(stream):
            for r in range(self.R):
                call(lib.santa_sample, a_list[r])
                stream.synchronize()
                sel_total += int(bufs.sel_count.sum().item())
        assert int(bufs.device_status.item()) == 0
        mean_sel = sel_total / (self.R * self.units)
        tp = self.bufs(M, team_probs=True)
        a0 = self.args(M, tp)[0]
        with torch.cuda.stream(stream):
            call(lib.santa_sample, a0)
        stream.synchronize()
        assert int(tp.device_status.item()) == 0
        p = tp.team_probs.double()
        n_valid = torch.div(self.lens.long() + self.cfg.team_size - 1, self.cfg.team_size,
                            rounding_mode="floor")
        valid = (torch.arange(self.n_teams, device=p.device)[None, None, :] <
                 n_valid[:, None, None]).expand_as(p)
        pi = -torch.expm1(M * torch.log1p(-p.clamp(max=1.0)))
        nv = float(valid.sum()) or 1.0
        rejected = {"p_below_1pct": float(((p < 0.01) & valid).sum()) / nv,
                    "pi_below_1pct": float(((pi < 0.01) & valid).sum()) / nv,
                    "teams": int(nv), "seed": 0}
        return mean_sel, rejected


class Timer:
    """Exactly K steps of one entry point, timed inside one CUDA graph over a rig's rotation
    copies (step k uses copy k mod R, so a copy is reused R steps later).  The graph holds one
    untimed step (copy R - 1), then the K timed steps.  The start event is recorded on a
    branch that waits only for that untimed step, and the end event after step K, so the
    interval is K step periods: the first timed step overlaps the tail of its predecessor,
    as every later one does (programmatic dependent launch), and no graph boundary or launch
    of the first kernel falls inside it.  The graph is replayed untimed until at least W steps
    have run, then once more, enqueued behind a spin kernel, for the timing."""

    def __init__(self, dev, stream, world):
        self.dev, self.stream, self.world = dev, stream, world

    def call(self, fn, a):
        rc = fn(ctypes.byref(a), self.stream.cuda_stream)
        if rc:
            raise RuntimeError(f"{fn.__name__}: status {rc}")

    def barrier(self):
        import torch
        if self.world > 1:
            torch.distributed.barrier()

    def run(self, step, R, K, W_, label):
        """step(r) enqueues one step on rotation copy r.  Returns (device seconds for the K
        steps, (wall start, wall end))."""
        import torch
        e0, e1 = timing_event_pair()
        fork = torch.cuda.Event()
        side = torch.cuda.Stream(device=self.dev)

        def body(capturing):
            step(R - 1)                              # untimed: its tail overlaps step 0
            if capturing:
                fork.record(self.stream)
                side.wait_event(fork)
                e0.record(side)
            for k in range(K):
                step(k % R)
            if capturing:
                e1.record(self.stream)
                self.stream.wait_stream(side)

        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            body(False)                              # attribute set-up, lazy loading
            self.stream.synchronize()
            with torch.cuda.graph(g, stream=self.stream):
                body(True)
            for _ in range(max(1, math.ceil(W_ / (K + 1)))):
                g.replay()
        torch.cuda.synchronize(self.dev)
        self.barrier()
        torch.cuda.nvtx.range_push(label)
        t0 = time.time()
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(SPIN_CYCLES)
            g.replay()
        torch.cuda.synchronize(self.dev)
        t1 = time.time()
        torch.cuda.nvtx.range_pop()
        self.barrier()
        return e0.elapsed_time(e1) / 1e3, (t0, t1)

    def steps(self, fn, a_list, K, W_, label):
        """Seconds per step of `fn` (an entry point taking a santa_decode_args) over a_list."""
        sec, window = self.run(lambda r: self.call(fn, a_list[r]), len(a_list), K, W_, label)
        return sec / K, window


def timing_event_pair():
    """Two timing events that become event-record nodes when recorded inside a graph capture
    (torch.cuda.Event's `external` flag)."""
    import torch
    return (torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True))


def measure_workload(rig, timer, lib, K, W_, peak, draws=None, dense_s=None, sampler="iid_ht",
                     alpha=0.0):
    """Decode, sampling-only and dense steps of one rig, each K steps timed the same way."""
    from sampled_sparse_decode_gb300 import binding as Bn
    cfg = rig.cfg
    M = draws or cfg.draws
    bufs = rig.bufs(M)
    a_dec = rig.args(M, bufs, sampler, alpha)
    tag = f"{cfg.name} M={M}"
    step_s, window = timer.steps(lib.santa_decode, a_dec, K, W_, f"decode {tag}")
    smp_s, _ = timer.steps(lib.santa_sample, a_dec, K, W_, f"sample {tag}")
    mean_sel, rejected = rig.sampled(M, a_dec, bufs, lib, timer.stream, timer.call)
    if dense_s is None:
        dbufs = rig.bufs(1, dense=True)
        dense_s, _ = timer.steps(lib.santa_dense_decode, rig.args(1, dbufs, dense=True), K, W_,
                                 f"dense {cfg.name}")
    sbytes = rig.step_bytes(mean_sel)
    plan = Bn.santa_decode_plan(rig.q, rig.ks[0], rig.pt, M)
    dplan = Bn.santa_decode_plan(rig.q, rig.ks[0], rig.pt, 1, which="dense")
    res = {
        "draws": M, "step_us": step_s * 1e6, "steps_per_s": 1.0 / step_s,
        "bytes_per_step": sbytes, "hbm_gbs": sbytes / step_s / 1e9,
        "frac": sbytes / step_s / 1e9 / peak, "mean_sel": mean_sel,
        "kv_read_ratio": mean_sel * rig.units * cfg.team_size * 2 * cfg.head_dim * rig.esize /
                         rig.dense_kv,
        "sample_only_us": smp_s * 1e6,
        "dense_us": dense_s * 1e6, "dense_hbm_gbs": rig.dense_kv / dense_s / 1e9,
        "dense_frac": rig.dense_kv / dense_s / 1e9 / peak,
        "speedup_vs_dense": dense_s / step_s,
        "rejected_teams": rejected,
        "plan": {"decode": plan, "dense": dplan}, "rotations": rig.R, "steps": K,
    }
    return res, window, dense_s


def run_ours(args):
    import numpy as np
    import torch
    import sampled_sparse_decode_gb300 as santa
    from sampled_sparse_decode_gb300 import binding as Bn

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    lib = Bn.lib()
    stream = torch.cuda.Stream(device=dev)
    timer = Timer(dev, stream, world)
    K, W_ = args.steps, max(3, args.warmup)
    peak, peak_kind = measured_peak()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    # ---- headline workload: whole decode steps, the two halves alone, and the dense kernel
    rig = Rig(args.workload, dev, draws=args.draws)
    cfg = rig.cfg
    G, d, T, M = cfg.group, cfg.head_dim, cfg.team_size, cfg.draws
    units, n_teams = rig.units, rig.n_teams
    head, (c0, c1), dense_s = measure_workload(rig, timer, lib, K, W_, peak,
                                               sampler=args.sampler, alpha=args.mix_alpha)
    step_s = head["step_us"] / 1e6
    value, slowest = job_rate(step_s * K, K, world, dev)
    step_s = slowest / K
    bufs = rig.bufs(M)
    a_dec = rig.args(M, bufs, args.sampler, args.mix_alpha)
    att_s, _ = timer.steps(lib.santa_attend, a_dec, K, W_, "attend")  # sets of the last seed
    step_bytes = rig.step_bytes(head["mean_sel"])
    achieved = step_bytes / step_s / 1e9

    # ---- the step before the decode: one appended token per unit (santa_append_kv) at the
    # last slot of every sequence
    q = rig.q
    kn = torch.randn((cfg.batch, cfg.kv_heads, d), device=dev).to(q.dtype)
    vn = torch.randn((cfg.batch, cfg.kv_heads, d), device=dev).to(q.dtype)
    last = (rig.lens - 1).contiguous()
    nxt = torch.empty_like(rig.lens)

    def append_step(r):
        santa.santa_append_kv(kn, vn, rig.ks[r], rig.vs[r], rig.reps[r], rig.pt, last, nxt,
                              stream=stream)

    n_app = max(rig.R, min(K, 1000))
    sec_app, _ = timer.run(append_step, rig.R, n_app, W_, "append")
    append_us = sec_app / n_app * 1e6

    # ---- the representatives of the whole cache (santa_build_reps, once after prefill): a
    # rebuild of every rotation copy in place from its own keys (the same values again)
    def reps_step(r):
        santa.santa_build_reps(rig.ks[r], rig.fill, reps=rig.reps[r], stream=stream)

    n_rep = max(rig.R, min(K, 200))
    sec_rep, _ = timer.run(reps_step, rig.R, n_rep, W_, "build_reps")
    reps_us = sec_rep / n_rep * 1e6
    valid_tokens = int(rig.wl.page_fill.astype(np.int64).sum())
    reps_bytes = valid_tokens * cfg.kv_heads * d * rig.esize + rig.reps[0].numel() * 4

    # ---- accuracy proxy: relative L2 error of the estimate against dense attention, per
    # query head, over 32 seeds (no model or dataset here: retention cannot be measured)
    acc = accuracy_vs_dense(q, rig.ks[0], rig.vs[0], rig.reps[0], rig.pt, rig.lens, M,
                            args.sampler, args.mix_alpha, 32, santa)

    # ---- end to end through the Python API, host buffers: per step one call of
    # santa_decode_host (PreparedDecode.run_host over the rotation's buffers): one
    # host->device copy of the step's inputs (StepInputs), the decode, one device->host copy
    # of the outputs and status word (packed DecodeBuffers), and the wait for the stream
    e2e = None
    if not args.no_e2e:
        inp = santa.StepInputs.allocate(q.dtype, cfg.batch, cfg.q_heads, d, n_teams, dev)
        inp.host_q.copy_(q.cpu())
        inp.host_page_table.copy_(rig.pt.cpu())
        inp.host_seq_lens.copy_(rig.lens.cpu())
        pbufs = santa.DecodeBuffers.allocate(q.dtype, cfg.batch, cfg.q_heads, cfg.kv_heads, d,
                                             T, n_teams, M, dev, packed=True)
        host = pbufs.host_mirror()
        preps = [santa.santa_decode_prepared(inp.q, rig.ks[r], rig.vs[r], rig.reps[r],
                                             inp.page_table, inp.seq_lens, M, bufs=pbufs,
                                             sampler=args.sampler, mix_alpha=args.mix_alpha)
                 for r in range(rig.R)]
        h2d = inp.host_slab.numel()
        d2h = host.slab.numel()
        K_e = max(20, min(K, 2000))

        def e2e_step(s):
            preps[s % rig.R].run_host(s, inp, host, stream)

        for s in range(W_):
            e2e_step(s)
        timer.barrier()
        torch.cuda.nvtx.range_push("e2e")
        t0 = time.perf_counter()
        for s in range(K_e):
            e2e_step(W_ + s)
        el = time.perf_counter() - t0
        torch.cuda.nvtx.range_pop()
        e2e_rate, el = job_rate(el, K_e, world, dev)
        assert int(host.device_status[0]) == 0
        e2e = {"value": e2e_rate, "unit": "steps/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": K_e}
    head_rot = rig.R
    del rig, bufs, a_dec
    torch.cuda.empty_cache()

    # ---- the other full-size workloads, each timed like the headline (its own rotation
    # copies), and the long-context draw sweep against one dense measurement
    workloads = {}
    if not args.no_extra:
        for name in EXTRA_WORKLOADS:
            if name == cfg.name:
                continue
            sweep = name == SWEEP_WORKLOAD
            r_ = Rig(name, dev, min_draws=min(SWEEP_DRAWS) if sweep else None)
            res, _, d_s = measure_workload(r_, timer, lib, K, W_, peak)
            workloads[name] = res
            if sweep:
                rows = []
                for m in SWEEP_DRAWS:
                    row = res if m == r_.cfg.draws else \
                        measure_workload(r_, timer, lib, K, W_, peak, draws=m, dense_s=d_s)[0]
                    rows.append({k: row[k] for k in ("draws", "step_us", "bytes_per_step",
                                                     "hbm_gbs", "frac", "mean_sel",
                                                     "kv_read_ratio", "dense_us",
                                                     "speedup_vs_dense")})
                workloads[f"{name} draw sweep"] = rows
            del r_
            torch.cuda.empty_cache()
    clocks.stop()
    clk = clocks.summary(c0, c1)
    clk_all = clocks.summary(0.0, float("inf"))

    # ---- CPU baseline (rank 0, single GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        from sampled_sparse_decode_gb300 import workloads as W
        wl = W.generate(args.workload, **({'draws': args.draws} if args.draws else {}))
        v, n, el = oracle_steps_per_s(wl, args.cpu_seconds, sampler=args.sampler,
                                      alpha=args.mix_alpha)
        cpu = {"value": v, "unit": "steps/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} whole decode steps ({units} units each) in {el:.1f} s, "
                         f"fp64 C oracle, reps precomputed; {host_cores_note()}",
               **host_cores()}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": W_, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic",
        "config": config_of(cfg, world),
        "rotation": {"copies": head_rot, "bytes_touched_per_step": step_bytes,
                     "l2_bytes": torch.cuda.get_device_properties(dev).L2_cache_size},
        "step_latency_us": step_s * 1e6,
        "hbm_gbs_step": achieved,
        "bytes_per_step": step_bytes,
        "kv_read_ratio": head["kv_read_ratio"],
        "mean_sel": head["mean_sel"],
        "dense": {"steps_per_s": 1.0 / dense_s, "latency_us": dense_s * 1e6,
                  "hbm_gbs": head["dense_hbm_gbs"], "frac": head["dense_frac"],
                  "plan": head["plan"]["dense"]},
        "speedup_vs_dense": dense_s / step_s,
        "kernels_us": {"decode": step_s * 1e6, "sample_only": head["sample_only_us"],
                       "attend_only": att_s * 1e6, "dense": dense_s * 1e6,
                       "append_token": append_us, "build_reps": reps_us},
        "build_reps": {"us": reps_us, "bytes": reps_bytes,
                       "hbm_gbs": reps_bytes / reps_us / 1e3,
                       "frac": reps_bytes / reps_us / 1e3 / peak,
                       "note": "all valid keys read once, fp32 representatives written; "
                               "once per prefill, not per step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "decode_kernel (fused sampling + split-K HT attention), "
                               "one launch per step",
                     "bytes_per_launch": step_bytes,
                     "traffic": recorded_traffic(cfg.name)},
        "plan": head["plan"]["decode"],
        "rejected_teams": head["rejected_teams"],
        "workloads": workloads,
        "sampler": {"name": args.sampler, "mix_alpha": args.mix_alpha},
        "accuracy": acc,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K,
        "clocks": clk,
        "clocks_whole_run": clk_all,
    }
    print(json.dumps(line))


def accuracy_vs_dense(q, k, v, reps, pt, lens, M, sampler, alpha, seeds, santa):
    """Mean and 90th percentile over seeds and query heads of ||out - dense|| / ||dense||."""
    import torch
    dense = santa.santa_dense_decode(q, k, v, pt, lens).out.clone()
    bufs = None
    errs = []
    for s_ in range(seeds):
        bufs = santa.santa_decode(q, k, v, reps, pt, lens, M, 10_000 + s_, bufs=bufs,
                                  sampler=sampler, mix_alpha=alpha)
        e = (bufs.out - dense).norm(dim=-1) / dense.norm(dim=-1)
        errs.append(e.flatten())
    torch.cuda.synchronize()
    assert bufs.status() == 0
    e = torch.cat(errs).double()
    return {"rel_l2_vs_dense_mean": float(e.mean()), "rel_l2_vs_dense_p90": float(e.quantile(0.9)),
            "seeds": seeds, "metric": "||out - dense|| / ||dense|| per query head"}


def run_accuracy(args):
    """Every sampler (and a 5% defensive mixture) against dense attention on one workload."""
    import numpy as np
    import torch
    import sampled_sparse_decode_gb300 as santa
    from sampled_sparse_decode_gb300 import workloads as W
    wl = W.generate(args.workload, **({'draws': args.draws} if args.draws else {}))
    cfg = wl.cfg

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    q, k, v = t(wl.q), t(wl.k_pool), t(wl.v_pool)
    pt, lens, fill = t(wl.page_table), t(wl.seq_lens), t(wl.page_fill)
    reps = santa.santa_build_reps(k, fill)
    rows = []
    for sampler, alpha in [("iid_ht", 0.0), ("systematic", 0.0), ("iid_hh", 0.0),
                           ("iid_ht", 0.05), ("systematic", 0.05)]:
        a = accuracy_vs_dense(q, k, v, reps, pt, lens, cfg.draws, sampler, alpha, args.seeds,
                              santa)
        bufs = santa.santa_sample(q, k, v, reps, pt, lens, cfg.draws, 1, sampler=sampler,
                                  mix_alpha=alpha)
        torch.cuda.synchronize()
        rows.append({"sampler": sampler, "mix_alpha": alpha, **a,
                     "mean_sel": float(bufs.sel_count.double().mean())})
    # value-row sampling inside the teams, against the full P.V product on the same sets
    sb = santa.santa_sample(q, k, v, reps, pt, lens, cfg.draws, 1)
    dense = santa.santa_dense_decode(q, k, v, pt, lens).out.clone()

    stream = torch.cuda.Stream()

    def timed_us(fn, n=50, reps_=10):
        """Mean device time per call: a CUDA graph of n calls, replayed reps_ times."""
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    fn()
            g.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps_):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (n * reps_)

    full = santa.santa_attend(q, k, v, pt, lens, sb.sel_ids, sb.sel_count, sb.pi)
    vs_rows = [{"value_rows": 0, "name": "full P.V (santa_attend)",
                "attend_us": timed_us(lambda: santa.santa_attend(q, k, v, pt, lens, sb.sel_ids,
                                                                 sb.sel_count, sb.pi, bufs=full,
                                                                 stream=stream)),
                "rel_l2_vs_dense_mean": float(((full.out - dense).norm(dim=-1) /
                                               dense.norm(dim=-1)).mean())}]
    for S in (8, 16, 32, 64):
        errs = []
        for s_ in range(min(args.seeds, 64)):
            vb, _ = santa.santa_attend_vs(q, k, v, pt, lens, sb.sel_ids, sb.sel_count, sb.pi, S,
                                          20_000 + s_)
            errs.append(((vb.out - dense).norm(dim=-1) / dense.norm(dim=-1)).flatten())
        vb2 = vb
        vs_rows.append({"value_rows": S, "name": "value-row sampling (santa_attend_vs)",
                        "attend_us": timed_us(lambda: santa.santa_attend_vs(
                            q, k, v, pt, lens, sb.sel_ids, sb.sel_count, sb.pi, S, 3,
                            bufs=vb2, stream=stream)),
                        "rel_l2_vs_dense_mean": float(torch.cat(errs).double().mean())})
    print(json.dumps({"mode": "accuracy", "workload": cfg.name, "draws": cfg.draws,
                      "results": rows, "value_sampling": vs_rows,
                      "note": "attention only, on one sampled set per unit; CUDA graphs of 50 "
                              "calls (inputs L2-resident: a comparison of the two, not a "
                              "bandwidth figure)"}))


def _mean_ci(xs):
    """Mean and half-width of its 95% confidence interval (normal approximation)."""
    n = len(xs)
    m = sum(xs) / n
    sd = statistics.stdev(xs) if n > 1 else 0.0
    return m, 1.96 * sd / math.sqrt(n)


def _drop_host_stalls(us, factor=20.0):
    """Steps that took more than `factor` times the median: the host fell behind the spin
    kernel that precedes each step, and the device waited for the next launch inside the
    timed interval (a Python or OS pause of milliseconds against steps of microseconds).
    Returns the remaining steps and how many were dropped."""
    med = statistics.median(us)
    kept = [u for u in us if u <= factor * med]
    return kept, len(us) - len(kept)


def run_loop(args):
    """A generation at the workload's context (the explainer's pitfall 2: sampling variance
    over autoregressive steps).  Every step appends the next token's K/V (santa_append_kv)
    and decodes with that step's query.  The policies are:
      dense       santa_dense_decode every step (also the reference of the errors);
      fresh       santa_decode every step (a new sampled set per step);
      held R      santa_decode every R steps, santa_attend over the held set in between.
    Per policy: step latency (append + decode; mean and 95% CI over the steps), the relative
    L2 error of each step's output against dense, and the error of the outputs summed over
    the first t steps (how the per-step errors add up over a generation)."""
    import dataclasses
    import numpy as np
    import torch
    import sampled_sparse_decode_gb300 as santa
    from sampled_sparse_decode_gb300 import workloads as W
    cfg = W.CONFIGS[args.workload]
    if args.draws:
        cfg = dataclasses.replace(cfg, draws=args.draws)
    steps, L0, T = args.gen_tokens, cfg.seq_len, cfg.team_size
    B, Hkv, Hq, d = cfg.batch, cfg.kv_heads, cfg.q_heads, cfg.head_dim
    wl = W.generate(cfg, seq_lens=[L0 + steps] * B)
    # the generated tokens are the continuation of each sequence; their slots start as NaN
    pos = L0 + np.arange(steps)
    kn = np.empty((steps, B, Hkv, d), dtype=wl.k_pool.dtype)
    vn = np.empty_like(kn)
    nan_bits = np.array([0x7FC0], np.uint16)[0] if wl.k_pool.dtype == np.uint16 else np.nan
    for b in range(B):
        pages, slots = wl.page_table[b, pos // T], pos % T
        kn[:, b] = wl.k_pool[pages, :, slots]
        vn[:, b] = wl.v_pool[pages, :, slots]
        wl.k_pool[pages, :, slots] = nan_bits
        wl.v_pool[pages, :, slots] = nan_bits
    fill0 = np.zeros(wl.k_pool.shape[0], np.int32)
    for b in range(B):
        for i in range(-(-L0 // T)):
            fill0[wl.page_table[b, i]] = min(T, L0 - i * T)

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
                torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    k0, v0 = t(wl.k_pool), t(wl.v_pool)
    kp, vp = torch.empty_like(k0), torch.empty_like(v0)
    pt, fill = t(wl.page_table), t(fill0)
    knd, vnd, qs = t(kn), t(vn), t(W.loop_queries(cfg, steps))
    lens0 = torch.full((B,), L0, dtype=torch.int32, device="cuda")
    reps = torch.empty((wl.k_pool.shape[0], Hkv, d), dtype=torch.float32, device="cuda")
    flush = torch.empty(2 * torch.cuda.get_device_properties(0).L2_cache_size,
                        dtype=torch.uint8, device="cuda")
    dense_out = torch.empty((steps, B, Hq, d), dtype=torch.float32, device="cuda")
    periods = [int(r) for r in args.refresh.split(",") if r]
    policies = [("dense", None), ("fresh", 1)] + [(f"held {r}", r) for r in periods]
    results = []
    for name, R in policies:
        kp.copy_(k0)
        vp.copy_(v0)
        santa.santa_build_reps(kp, fill, reps=reps)
        lens = [lens0.clone(), torch.empty_like(lens0)]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs = torch.empty_like(dense_out)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        dec = att = None
        for s in range(steps):
            flush.zero_()                          # L2 holds nothing of this layer
            torch.cuda._sleep(1_000_000)           # the device runs behind the host
            ev[s][0].record()
            santa.santa_append_kv(knd[s], vnd[s], kp, vp, reps, pt, lens[s % 2],
                                  lens[(s + 1) % 2], status)
            cur = lens[(s + 1) % 2]
            if R is None:
                dec = santa.santa_dense_decode(qs[s], kp, vp, pt, cur, bufs=dec)
                res = dec
            elif s % R == 0:
                dec = santa.santa_decode(qs[s], kp, vp, reps, pt, cur, cfg.draws, s, bufs=dec)
                res = dec
            else:
                att = santa.santa_attend(qs[s], kp, vp, pt, cur, dec.sel_ids, dec.sel_count,
                                         dec.pi, bufs=att)
                res = att
            ev[s][1].record()
            outs[s].copy_(res.out)
        torch.cuda.synchronize()
        st = int(status.item()) | dec.status() | (att.status() if att is not None else 0)
        if st:
            raise SystemExit(f"{name}: device status {st}")
        if R is None:
            dense_out.copy_(outs)
        us = [a.elapsed_time(b) * 1e3 for a, b in ev]
        kept, stalls = _drop_host_stalls(us)
        m, ci = _mean_ci(kept)
        row = {"policy": name, "refresh": R, "step_us_mean": m, "step_us_ci95": ci,
               "step_us_p50": statistics.median(us), "host_stall_steps_dropped": stalls}
        if R is not None:
            diff = (outs - dense_out).double()
            ref = dense_out.double()
            per_step = (diff.norm(dim=-1) / ref.norm(dim=-1)).mean(dim=(1, 2))
            acc = (diff.cumsum(0).norm(dim=-1) / ref.cumsum(0).norm(dim=-1)).mean(dim=(1, 2))
            row["rel_l2_step_mean"] = float(per_step.mean())
            row["rel_l2_step_p90"] = float(per_step.quantile(0.9))
            row["rel_l2_accumulated"] = {str(n): float(acc[n - 1]) for n in
                                         (1, 16, 64, 256, 1024, steps) if n <= steps}
        results.append(row)
    dm, dci = results[0]["step_us_mean"], results[0]["step_us_ci95"]
    for row in results[1:]:
        m, ci = row["step_us_mean"], row["step_us_ci95"]
        r = dm / m
        row["speedup_vs_dense"] = r
        row["speedup_ci95"] = r * math.sqrt((dci / dm) ** 2 + (ci / m) ** 2)
    print(json.dumps({
        "mode": "loop", "workload": cfg.name, "context_start": L0, "generated": steps,
        "draws": cfg.draws, "results": results,
        "l2": "flushed before every step (a write of 2x the L2 size)",
        "timing": "CUDA events around each step's append + decode; a spin kernel before "
                  "every step keeps the device behind the host, so no launch gap is timed; "
                  "steps above 20x the median (the host fell behind the spin) are left out "
                  "of the mean and counted",
        "queries": "per step: each head's mixture part fixed, fresh 0.3 * N(0, I) noise",
        "error": "||out - dense|| / ||dense|| per query head, mean over heads; accumulated: "
                 "the same for the outputs summed over the first t steps"}))


def run_profile(args):
    """A short run for ncu: one copy of the inputs, W + K steps launched on the stream."""
    import numpy as np
    import torch
    import sampled_sparse_decode_gb300 as santa
    from sampled_sparse_decode_gb300 import workloads as W
    wl = W.generate(args.workload, **({'draws': args.draws} if args.draws else {}))
    cfg = wl.cfg

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    q, k, v = t(wl.q), t(wl.k_pool), t(wl.v_pool)
    pt, lens, fill = t(wl.page_table), t(wl.seq_lens), t(wl.page_fill)
    reps = santa.santa_build_reps(k, fill)
    bufs = None
    for s_ in range(args.warmup + args.steps):
        if args.dense:
            bufs = santa.santa_dense_decode(q, k, v, pt, lens, bufs=bufs)
        else:
            bufs = santa.santa_decode(q, k, v, reps, pt, lens, cfg.draws, s_, bufs=bufs)
    torch.cuda.synchronize()
    st = bufs.status()
    print(json.dumps({"mode": "profile", "workload": cfg.name, "dense": args.dense,
                      "steps": args.warmup + args.steps, "device_status": st,
                      "sel_count": None if args.dense else bufs.sel_count.sum().item()}))
    if st:
        raise SystemExit(1)


def main():
    args = parse()
    if args.record_traffic:
        rec = record_traffic_file(args.record_traffic, args.traffic_out or TRAFFIC_FILE,
                                  args.workload, args.traffic_command)
        print(json.dumps(rec))
        return
    if args.mode == "profile":
        run_profile(args)
    elif args.mode == "accuracy":
        run_accuracy(args)
    elif args.mode == "loop":
        run_loop(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
