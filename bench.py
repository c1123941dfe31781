#!/usr/bin/env python3
"""Benchmark of split-KV paged GQA decode attention on GB300.

One step = one ``attn_decode`` call (split kernel with the last-CTA merge)
over one synthetic workload.  Default workload: the sliding-window multi-row
decode (nh16 nkv8 hd256, ctx 8192, rows at qpos 8188..8191, window 1024).

Prints ONE JSON line (rank 0).  ``value`` is KV GB/s: the call's algorithmic
bytes (in-window KV + Q + O) over the device time per call, measured with CUDA
events around a CUDA graph of exactly ``--steps`` back-to-back calls that
rotate over enough pool copies that every call reads its KV from HBM.

``--impl reference`` times the f64 CPU oracle instead (the only other place
this file runs it is the ``cpu_baseline`` leg).

Multi-GPU (torchrun): every rank runs the same workload on its own GPU (weak
scaling, no collective on the data path); the job's value is all ranks' bytes
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention KV GB/s and fraction of GB300 HBM peak; µs/call"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["paged_gqa_decode_attn_gb300/csrc/pgqa_device.cuh",
                  "paged_gqa_decode_attn_gb300/csrc/pgqa_launch.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_split_kernel_traffic.json")
PREP_SOURCES = ["paged_gqa_decode_attn_gb300/csrc/pgqa_prep.cu"]
PREP_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "qk_norm_rope_kernel_traffic.json")
TILED_SOURCES = ["paged_gqa_decode_attn_gb300/csrc/pgqa_prefill_tc.cuh",
                 "paged_gqa_decode_attn_gb300/csrc/pgqa_prefill.cuh"]
TILED_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "prefill_tc_kernel_traffic.json")


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(world: int):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    """Max of a host float over all ranks (gloo; host-side only)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ measured peaks, traffic, clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s, burst: a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def l2_note(copies: int, what: str, rotation_bytes: int, claim: str) -> str:
    """The run's L2 policy: ``claim`` holds only when one rotation moves more than 3x L2."""
    head = f"rotating {copies} {what} ({rotation_bytes / 1e6:.0f} MB per rotation"
    if rotation_bytes >= 3 * L2_BYTES:
        return head + f" > 3x L2): {claim}"
    return head + " <= 3x L2): part of the data may come from L2 (a diagnostic run, not a bench value)"


def kernel_sources_sha(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, path: str = TRAFFIC_FILE, sources=KERNEL_SOURCES):
    """dram bytes per launch from the committed ncu summary, or None if it is stale or absent."""
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(workload)
    if not e or e.get("kernel_sources_sha256_16") != kernel_sources_sha(sources):
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the GPU works."""

    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            import torch
            ident = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = ident if ident.startswith("GPU-") else "GPU-" + ident
        except Exception:
            ident = str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [ln.split(", ") for ln in out.strip().splitlines() if ln.count(",") >= len(self.FIELDS) - 1]
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                mhz.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not mhz:
            return None
        busy = [m for m in mhz if m > 0.5 * max(mhz)]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz), "window": "warm-up and timed steps"}


# ------------------------------------------------------------------ workloads

def build_case(name: str):
    if name == "sliding":
        return wl.sliding()
    if name == "sliding_mapped":
        return wl.sliding(mapped=True)
    if name == "tiny":
        return wl.tiny()
    if name == "long":
        return wl.long_ctx()
    if name == "batched":
        return wl.batched()
    if name == "prefill_page":
        return wl.prefill_page()
    if name == "prefill_long":
        return wl.prefill_long()
    if name == "prefill_hd512":
        return wl.prefill_hd512()
    if name == "prep_long":
        return wl.prep_long()
    if name == "multirow":
        return wl.multirow()
    raise SystemExit(f"unknown workload {name}")


def prefill_flops(case) -> int:
    """Algorithmic FLOPs of one prefill call: 4 nh hd per (row, visible position)."""
    hi = case.qpos if case.kvpos is None else np.minimum(case.qpos, case.kvpos)
    lo = np.maximum(0, case.qpos + 1 - case.window) if case.window > 0 else np.zeros_like(case.qpos)
    return int(np.maximum(0, hi.astype(np.int64) - lo + 1).sum()) * 4 * case.nh * case.hd


def nseq_of(case) -> int:
    return len(set(int(x) for x in case.off))


# ------------------------------------------------------------------ the CPU oracle (baseline / reference arm)

def oracle_rate(case, budget_s: float, steps: int | None = None, warmup: int = 0):
    """Time the f64 oracle on ``case`` (all host cores).  With ``steps`` set,
    each step is a bounded sample of (row, head) pairs sized so the whole run
    takes about ``budget_s``; otherwise whole calls repeat for ``budget_s``.
    Returns (GB/s, seconds per step, sample description, cores, pairs per step)."""
    import oracle
    cores = oracle.default_threads()
    total_pairs = case.rows * case.nh
    all_pairs = [(r, h) for r in range(case.rows) for h in range(case.nh)]
    t0 = time.perf_counter()
    oracle.decode_case(case, pairs=all_pairs[:min(total_pairs, max(cores, 1))], want_f64=False)
    t_pair = max((time.perf_counter() - t0) / min(total_pairs, max(cores, 1)), 1e-7)
    bytes_per_pair = case.algorithmic_bytes() / total_pairs
    if steps is None:
        n_calls, t_tot = 0, 0.0
        while t_tot < budget_s or n_calls == 0:
            t0 = time.perf_counter()
            oracle.decode_case(case, want_f64=False)
            t_tot += time.perf_counter() - t0
            n_calls += 1
        per = t_tot / n_calls
        return (case.algorithmic_bytes() / per / 1e9, per,
                f"{n_calls} whole calls ({total_pairs} (row, head) pairs each), {t_tot:.1f} s", cores, total_pairs)
    per_step_budget = budget_s / max(steps + warmup, 1)
    k = int(min(total_pairs, max(1, per_step_budget / t_pair * cores)))
    k = max(1, min(k, total_pairs))
    cursor = 0

    def one():
        nonlocal cursor
        sel = [all_pairs[(cursor + i) % total_pairs] for i in range(k)]
        cursor = (cursor + k) % total_pairs
        oracle.decode_case(case, pairs=sel, want_f64=False)

    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    el = time.perf_counter() - t0
    per = el / steps
    return (bytes_per_pair * k / per / 1e9, per,
            f"{k} of {total_pairs} (row, head) pairs per step, cycling", cores, k)


PREP_METRIC = "QK-RMSNorm / RoPE / paged K-V write GB/s"


def prep_rows(case, idx):
    """The oracle's inputs for rows ``idx`` of a prep case (same block table and page map)."""
    def rows_of(a, width):
        return np.ascontiguousarray(np.asarray(a).reshape(case.rows, width)[idx]).reshape(-1)
    return (rows_of(case.q_in, case.nh * case.hd), rows_of(case.k_in, case.nkv * case.hd),
            rows_of(case.v_in, case.nkv * case.hd), case.q_weight, case.k_weight, np.asarray(case.pos)[idx],
            case.block_table, np.asarray(case.off)[idx], case.page_map, case.nh, case.nkv, case.hd,
            case.rotary_dim, case.theta, case.eps, case.norm_v)


def prep_oracle_rate(case, budget_s: float, steps: int = 1, warmup: int = 0):
    """Time the f64 prep oracle (one host thread) on bounded samples of rows sized
    so the whole run takes about ``budget_s``.  Returns (GB/s, s per step, sample, cores)."""
    from oracle import prep as op
    t0 = time.perf_counter()
    op.prep(*prep_rows(case, np.arange(min(8, case.rows))))
    t_row = max((time.perf_counter() - t0) / min(8, case.rows), 1e-7)
    k = int(max(1, min(case.rows, budget_s / max(steps + warmup, 1) / t_row)))
    cursor = 0

    def one():
        nonlocal cursor
        op.prep(*prep_rows(case, (cursor + np.arange(k)) % case.rows))
        cursor = (cursor + k) % case.rows

    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    per = (time.perf_counter() - t0) / steps
    return (case.bytes_moved() * k / case.rows / per / 1e9, per,
            f"{k} of {case.rows} rows per step, cycling", 1)


def run_reference(args, case, rank, world):
    if args.workload.startswith("prep"):
        gbs, per, sample, cores = prep_oracle_rate(case, args.ref_budget, args.steps, args.warmup)
        line = {
            "impl": "reference", "metric": PREP_METRIC, "value": round(gbs, 6), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prep_config(case),
            "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
        print(json.dumps(line), flush=True)
        return 0
    gbs, per, sample, cores, k = oracle_rate(case, budget_s=args.ref_budget, steps=args.steps, warmup=args.warmup)
    metric, unit = METRIC, "GB/s"
    if args.workload == "multirow":
        metric = "multi-row decode KV GB/s (tiled split-KV path)"
    if args.workload.startswith("prefill"):
        metric, unit = "paged causal prefill attention TFLOP/s", "TFLOP/s"
        gbs = prefill_flops(case) * k / (case.rows * case.nh) / per / 1e12
    cfg = prefill_config(case) if args.workload.startswith("prefill") else config_of(case)
    line = {
        "impl": "reference", "metric": metric, "value": round(gbs, 6), "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(gbs, 6), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(case):
    """The workload alone: the same keys and values in both arms' lines."""
    return {"workload": case.name, "nh": case.nh, "nkv": case.nkv, "hd": case.hd, "ctx": case.ctx,
            "rows": case.rows, "window": case.window,
            "pool": "page map + NaN null page" if case.page_map is not None else "identity",
            "algorithmic_bytes_per_call": case.algorithmic_bytes()}


def prefill_config(case):
    c = config_of(case)
    del c["algorithmic_bytes_per_call"]
    c["flops_per_call"] = prefill_flops(case)
    return c


def run_of(args, case, splits):
    """How this arm ran the workload (split count and merge path)."""
    r = {"splits": splits}
    if splits == 1:
        r["merge"] = "none (one split)"
    elif args.merge == "counters" and splits <= 8:
        r["merge"] = "in the split kernel (thread-block cluster or last CTA, through merge counters)"
    else:
        r["merge"] = "combine kernel" + (" (more than 8 splits)" if args.merge == "counters" else "")
    return r


# ------------------------------------------------------------------ our arm

class DecodeRig:
    """One decode workload resident on the device, ready to call: rotating pool
    copies (each copy's reads > 3x L2 apart, so every call reads KV from HBM; and
    more copies than the streams of the concurrent and end-to-end runs, so calls
    in flight at once read different copies), the per-step inputs in one pinned
    host buffer and one device buffer, scratch and counters."""

    def __init__(self, args, case, dev, splits=None, copies=None):
        import torch
        import paged_gqa_decode_attn_gb300 as pgqa
        self.case = case
        self.bpc = case.algorithmic_bytes()
        self.splits = splits or args.splits or pgqa.choose_splits(case.kv_len_eff(), case.rows, case.nkv,
                                                                   nseq_of(case), nh=case.nh, hd=case.hd)
        self.pool_bytes = case.k_pool.nbytes + case.v_pool.nbytes
        n = max(2, math.ceil(3 * L2_BYTES / max(self.bpc, 1)), getattr(args, "e2e_streams", 1) + 2)
        n = min(n, max(2, int(0.25 * torch.cuda.get_device_properties(dev).total_memory // self.pool_bytes)))
        self.copies = copies or args.copies or n

        def i16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))

        def i32(a):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))

        k_host, v_host = i16(case.k_pool), i16(case.v_pool)
        self.ks = [k_host.to(dev) for _ in range(self.copies)]
        self.vs = [v_host.to(dev) for _ in range(self.copies)]
        # q, qpos, off and the block table share one pinned host buffer and one
        # device buffer, so a step moves them with a single copy
        parts = [np.ascontiguousarray(case.q).view(np.uint8),
                 np.ascontiguousarray(case.qpos, np.int32).view(np.uint8),
                 np.ascontiguousarray(case.off, np.int32).view(np.uint8),
                 np.ascontiguousarray(case.block_table, np.int32).view(np.uint8)]
        offs, pos = [], 0
        for a in parts:
            offs.append(pos)
            pos += (a.size + 255) // 256 * 256
        self.host_in = torch.zeros(pos, dtype=torch.uint8).pin_memory()
        for a, o0 in zip(parts, offs):
            self.host_in[o0:o0 + a.size] = torch.from_numpy(a)
        self.dev_in = self.host_in.to(dev)
        self.q = self.dev_in[offs[0]:offs[0] + parts[0].size].view(torch.int16)
        self.qpos = self.dev_in[offs[1]:offs[1] + parts[1].size].view(torch.int32)
        self.off = self.dev_in[offs[2]:offs[2] + parts[2].size].view(torch.int32)
        self.bt = self.dev_in[offs[3]:offs[3] + parts[3].size].view(torch.int32)
        self.block_table_bytes = parts[3].size
        self.kvpos = None if case.kvpos is None else i32(case.kvpos).to(dev)
        self.pm = None if case.page_map is None else i32(case.page_map).to(dev)
        self.part = torch.empty(max(1, pgqa.decode_part_bytes(case.rows, case.nh, self.splits, case.hd)) // 4 + 4,
                                dtype=torch.float32, device=dev)
        self.cnt = torch.zeros(max(1, pgqa.decode_counter_count(case.rows, case.nh, case.nkv)), dtype=torch.int32,
                               device=dev)
        self.o = torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16, device=dev)
        self.o_h = torch.empty_like(self.o, device="cpu").pin_memory()
        self.counters = self.cnt if args.merge == "counters" else None
        self.launches_per_call = pgqa.decode_kernel_count(self.splits, self.counters is not None)
        self.graphs = {}

    def call(self, i, stream=None):
        import paged_gqa_decode_attn_gb300 as pgqa
        c = self.case
        pgqa.attn_decode(self.o, self.part, self.q, self.ks[i % self.copies], self.vs[i % self.copies], self.bt,
                         self.off, self.qpos, self.kvpos, c.rows, c.nh, c.nkv, c.hd, c.window, self.splits,
                         self.counters, self.pm, stream)

    def spot_check(self, npairs=16):
        """rel-RMS of a sample of (row, head) outputs against the oracle (raises above the page's 1e-2)."""
        import torch
        import oracle
        c = self.case
        self.call(0)
        torch.cuda.synchronize()
        got = self.o.cpu().numpy().view(np.uint16).reshape(c.rows, c.nh, c.hd)
        pairs = [(r, h) for r in range(c.rows) for h in range(c.nh)][:: max(1, c.rows * c.nh // npairs)]
        _, ref = oracle.decode_case(c, pairs=pairs, want_f64=False)
        e = oracle.rel_rms(np.stack([got[r, h] for r, h in pairs]), ref)
        if not e < 1e-2:
            raise SystemExit(f"{c.name}: spot check against the oracle failed: rel_rms {e}")
        return e

    def graph(self, n):
        import torch
        if n not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    self.call(i)
            self.graphs[n] = g
        return self.graphs[n]

    def time_steps(self, steps, warmup, chunk, dist=None, load_s=0.0):
        """Device time (ms) of exactly ``steps`` back-to-back calls: CUDA events on the
        launching stream around graph replays, after ``warmup`` eager calls.  A short
        GPU sleep is queued ahead of the start event, so the replays are already
        queued when the GPU reaches it: the region holds the calls, not the host's
        launch latency.  With ``load_s`` the graphs also replay for about that long
        before and after the region (the clock samples' window)."""
        import torch
        for i in range(warmup):
            self.call(i)
        torch.cuda.synchronize()
        chunk = max(1, min(steps, chunk))
        full, rem = divmod(steps, chunk)
        g_full = self.graph(chunk) if full else None
        g_rem = self.graph(rem) if rem else None
        (g_full or g_rem).replay()       # settles the graphs' first-launch cost
        torch.cuda.synchronize()
        self._load(g_full or g_rem, load_s)
        stream = torch.cuda.current_stream()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        torch.cuda._sleep(200000)        # ~0.1 ms: the replays below queue behind it
        ev0.record(stream)
        for _ in range(full):
            g_full.replay()
        if rem:
            g_rem.replay()
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        barrier(dist)
        self._load(g_full or g_rem, load_s / 3)
        return ev0.elapsed_time(ev1), chunk

    def time_single(self, n=30):
        """Latency of one call alone: CUDA events around a single eager call on an idle
        GPU (synchronised before and after), median over ``n`` calls on rotating pool
        copies, in us.  A short GPU sleep ahead of the start event lets the host
        enqueue the call first, so the region holds the call, not its host launch.
        The per-call period of back-to-back calls is what the line's value reports;
        this is the time one call takes from its first kernel's start to its last
        kernel's end."""
        import torch
        stream = torch.cuda.current_stream()
        ts = []
        for i in range(n):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            torch.cuda._sleep(100000)    # ~50 us
            ev0.record(stream)
            self.call(i)
            ev1.record(stream)
            ev1.synchronize()
            ts.append(ev0.elapsed_time(ev1) * 1e3)
        return statistics.median(ts)

    def time_streams(self, steps, nstreams, reps=3):
        """us per call of ``steps`` independent calls taken in turn by ``nstreams``
        streams, each with its own output, scratch and counters (inputs resident, the
        pool copies rotating as in time_steps): one CUDA graph forked from and joined
        back to the timing stream, CUDA events around its replay on that stream, the
        median of ``reps`` regions.  Calls on different streams do not wait for each
        other, so several run at once; the line's value is the one-stream period."""
        import torch
        sets = [(self.o, self.part, self.cnt)] + [
            (torch.empty_like(self.o), torch.empty_like(self.part), torch.zeros_like(self.cnt))
            for _ in range(nstreams - 1)]
        streams = [torch.cuda.Stream() for _ in range(nstreams)]
        c = self.case

        def call_on(i, b, s):
            import paged_gqa_decode_attn_gb300 as pgqa
            o, part, cnt = b
            pgqa.attn_decode(o, part, self.q, self.ks[i % self.copies], self.vs[i % self.copies], self.bt,
                             self.off, self.qpos, self.kvpos, c.rows, c.nh, c.nkv, c.hd, c.window, self.splits,
                             cnt if self.counters is not None else None, self.pm, s)

        cap = torch.cuda.Stream()
        for k, b in enumerate(sets):
            call_on(k, b, cap)
        cap.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for st in streams:
                st.wait_stream(cap)
            for i in range(steps):
                call_on(i, sets[i % nstreams], streams[i % nstreams])
            for st in streams:
                cap.wait_stream(st)
        g.replay()
        torch.cuda.synchronize()
        out = []
        for _ in range(reps):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(cap):
                torch.cuda._sleep(200000)
                ev0.record(cap)
                g.replay()
                ev1.record(cap)
            ev1.synchronize()
            out.append(ev0.elapsed_time(ev1) * 1e3 / steps)
        del g
        return statistics.median(out)

    def time_repeats(self, steps, chunk, reps=5):
        """us per call of ``reps`` more timed regions of ``steps`` calls each (the
        graphs of time_steps, already captured): their median and each value."""
        import torch
        chunk = max(1, min(steps, chunk))
        full, rem = divmod(steps, chunk)
        stream = torch.cuda.current_stream()
        out = []
        for _ in range(reps):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            torch.cuda._sleep(200000)
            ev0.record(stream)
            for _ in range(full):
                self.graph(chunk).replay()
            if rem:
                self.graph(rem).replay()
            ev1.record(stream)
            ev1.synchronize()
            out.append(round(ev0.elapsed_time(ev1) * 1e3 / steps, 3))
        return {"median": statistics.median(out), "each": out}

    @staticmethod
    def _load(g, seconds):
        import torch
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            for _ in range(8):
                g.replay()
            torch.cuda.synchronize()

    def _step_buffers(self):
        """A second set of per-step buffers (inputs, scratch, counters, output), so
        two steps can be in flight at once."""
        import torch
        b = {"dev_in": torch.empty_like(self.dev_in), "part": torch.empty_like(self.part),
             "cnt": torch.zeros_like(self.cnt), "o": torch.empty_like(self.o),
             "o_h": torch.empty_like(self.o_h).pin_memory()}
        n = [self.q.numel() * 2, self.qpos.numel() * 4, self.off.numel() * 4, self.block_table_bytes]
        offs, pos = [], 0
        for a in n:
            offs.append(pos)
            pos += (a + 255) // 256 * 256
        d = b["dev_in"]
        b["q"] = d[offs[0]:offs[0] + n[0]].view(torch.int16)
        b["qpos"] = d[offs[1]:offs[1] + n[1]].view(torch.int32)
        b["off"] = d[offs[2]:offs[2] + n[2]].view(torch.int32)
        b["bt"] = d[offs[3]:offs[3] + n[3]].view(torch.int32)
        return b

    def _call_on(self, b, i, stream):
        import paged_gqa_decode_attn_gb300 as pgqa
        c = self.case
        pgqa.attn_decode(b["o"], b["part"], b["q"], self.ks[i % self.copies], self.vs[i % self.copies], b["bt"],
                         b["off"], b["qpos"], self.kvpos, c.rows, c.nh, c.nkv, c.hd, c.window, self.splits,
                         b["cnt"] if self.counters is not None else None, self.pm, stream)

    def time_e2e(self, steps, dist=None, nstreams=2):
        """End to end through the public API from pinned host memory: per step one
        host->device copy of the step's inputs, the call, and one device->host copy of
        o.  The timed run is one CUDA graph of `steps` such steps, taken in turn by
        `nstreams` streams, each with its own set of buffers, so one step's copies
        overlap other steps' kernels (the steps are independent batches).  Also
        reported: the same steps issued eagerly one after another on one stream, and
        the host cost of each part enqueued alone."""
        import torch
        mine = {"dev_in": self.dev_in, "part": self.part, "cnt": self.cnt, "o": self.o, "o_h": self.o_h,
                "q": self.q, "qpos": self.qpos, "off": self.off, "bt": self.bt}
        sets = [mine] + [self._step_buffers() for _ in range(nstreams - 1)]
        streams = [torch.cuda.Stream() for _ in range(nstreams)]
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.stream(cap):
            for b in sets[1:]:
                b["dev_in"].copy_(self.host_in)         # warm the other sets once, outside the graph
                self._call_on(b, 0, cap)
        cap.synchronize()
        with torch.cuda.graph(g, stream=cap):
            for s in streams:
                s.wait_stream(cap)
            for i in range(steps):
                s, b = streams[i % nstreams], sets[i % nstreams]
                with torch.cuda.stream(s):
                    b["dev_in"].copy_(self.host_in, non_blocking=True)
                    self._call_on(b, i, s)
                    b["o_h"].copy_(b["o"], non_blocking=True)
            for s in streams:
                cap.wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        barrier(dist)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g.replay()
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(dist, time.perf_counter() - t0)
        del g
        # eagerly, one step after another on one stream
        n = min(steps, 500)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            self.dev_in.copy_(self.host_in, non_blocking=True)
            self.call(i)
            self.o_h.copy_(self.o, non_blocking=True)
        torch.cuda.synchronize()
        eager_us = (time.perf_counter() - t0) / n * 1e6
        m = min(steps, 200)
        parts = {}
        for name, fn in (("h2d_copy", lambda i: self.dev_in.copy_(self.host_in, non_blocking=True)),
                         ("attn_decode_call", self.call),
                         ("d2h_copy", lambda i: self.o_h.copy_(self.o, non_blocking=True))):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(m):
                fn(i)
            parts[name] = round((time.perf_counter() - t0) / m * 1e6, 2)
            torch.cuda.synchronize()
        return e2e_s, parts, eager_us


# independent calls per timed region of DecodeRig.time_streams
CONCURRENT_CALLS = 400


def concurrent(rig, us, nstreams, peak):
    """The record of DecodeRig.time_streams: independent calls on several streams, inputs resident."""
    gbs = rig.bpc / (us * 1e-6) / 1e9
    return {"streams": nstreams, "calls": CONCURRENT_CALLS, "us_per_call": round(us, 3), "value": round(gbs, 2),
            "frac": round(gbs / peak, 4),
            "what": "independent calls taken in turn by the streams, each stream with its own output and scratch, "
                    "inputs resident; calls on different streams run at once, so this is throughput, not one "
                    "call's duration; the line's value and roofline are the one-stream period"}


def decode_summary(rig, el_ms, steps, spot, peak, single_us=None, repeats=None, conc=None):
    """Per-workload record: device time per call, GB/s, roofline fraction, splits, parity, traffic; with
    them, the latency of one call alone, the per-call time of repeated timed regions and the throughput
    of independent calls on several streams."""
    c = rig.case
    us = el_ms * 1e3 / steps
    gbs = rig.bpc / (us * 1e-6) / 1e9
    r = {"workload": c.name, "us_per_call": round(us, 3), "value": round(gbs, 2), "unit": "GB/s",
         "frac": round(gbs / peak, 4), "splits": rig.splits, "kernels_per_call": rig.launches_per_call,
         "algorithmic_bytes_per_call": rig.bpc, "spot_check_rel_rms": spot,
         "traffic": recorded_traffic(c.name), "steps": steps}
    if single_us is not None:
        r["single_call_us"] = round(single_us, 3)
    if repeats is not None:
        r["us_per_call_repeats"] = repeats
    if conc is not None:
        r["concurrent_streams"] = conc
    return r


# The other decode configurations timed in the default run beside the headline
# (sliding): the 32K-context target, the batched shared-table case and the tiny
# latency case.  Each is timed with the headline's protocol.
EXTRA_DECODE = ["long", "batched", "tiny"]
# The tiled tcgen05 paths and the K/V write, timed in the default run too, each
# by its own workload's protocol (no CPU baseline there, two end-to-end steps).
EXTRA_OTHER = ["prefill_long", "prefill_hd512", "multirow", "prep_long"]


def line_summary(line):
    """The per-workload record of another workload's full line."""
    ro = line["roofline"]
    return {"workload": line["config"]["workload"], "metric": line["metric"],
            "us_per_call": round(line["ms_per_step"] * 1e3, 3), "value": line["value"], "unit": line["unit"],
            "frac": ro["frac"], "bound": ro["bound"], "kernel": ro["kernel"],
            "spot_check": {k: v for k, v in line["run"].items() if k.startswith("spot_check")} or None,
            "traffic": ro["traffic"],
            "steps": line["steps"], "kernels_per_call": line["gpu_launches"] // max(1, line["steps"])}


def run_ours(args, case, rank, world, dist):
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    if rank == 0:
        pgqa.build()
    barrier(dist)
    pgqa.load()
    sampler = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None

    rig = DecodeRig(args, case, dev)
    spot = rig.spot_check() if rank == 0 and not args.no_check else None
    el_ms, chunk = rig.time_steps(args.steps, args.warmup, args.graph_chunk, dist,
                                  load_s=0.0 if args.no_clocks else args.clock_window)
    clocks = sampler.stop() if sampler else None
    single_us = rig.time_single()
    repeats = rig.time_repeats(args.steps, chunk)
    conc_us = rig.time_streams(CONCURRENT_CALLS, args.e2e_streams)
    el_max = max_over_ranks(dist, el_ms)
    ms_per_step = el_max / args.steps
    value = sum_over_ranks(dist, float(rig.bpc) * args.steps) / (el_max * 1e-3) / 1e9
    # the step's device time: with two launches the combine kernel overlaps the
    # split kernel's tail (programmatic dependent launch), so they are timed together
    kernel_us = el_ms * 1e3 / args.steps
    e2e_steps = max(1, args.e2e_steps)
    e2e_s, host_parts, eager_us = rig.time_e2e(e2e_steps, dist, args.e2e_streams)
    e2e_value = sum_over_ranks(dist, float(rig.bpc) * e2e_steps) / e2e_s / 1e9

    # the other decode configurations, same protocol, reported inside the one line
    peak, peak_kind = measured_peaks()
    extra = []
    if args.workload == "sliding" and not args.no_extra:
        for name in EXTRA_DECODE:
            c2 = build_case(name)
            r2 = DecodeRig(args, c2, dev)
            sp2 = r2.spot_check() if rank == 0 and not args.no_check else None
            ms2, ch2 = r2.time_steps(args.steps, args.warmup, args.graph_chunk, dist)
            ms2 = max_over_ranks(dist, ms2)
            extra.append(decode_summary(r2, ms2, args.steps, sp2, peak, r2.time_single(),
                                        r2.time_repeats(args.steps, ch2),
                                        concurrent(r2, r2.time_streams(CONCURRENT_CALLS, args.e2e_streams),
                                                   args.e2e_streams, peak)))
            del r2
            torch.cuda.empty_cache()
        for name in EXTRA_OTHER:
            a2 = argparse.Namespace(**vars(args))
            a2.workload, a2.no_cpu_baseline, a2.no_clocks, a2.e2e_steps, a2.copies = name, True, True, 2, 0
            run = run_multirow if name == "multirow" else (run_prep if name.startswith("prep") else run_prefill)
            l2 = run(a2, build_case(name), rank, world, dist)
            if isinstance(l2, dict):
                extra.append(line_summary(l2))
            torch.cuda.empty_cache()

    if rank != 0:
        return 0
    achieved = rig.bpc / (kernel_us * 1e-6) / 1e9
    traffic = recorded_traffic(case.name)
    kernel = "decode_split_kernel" if rig.launches_per_call == 1 else \
        "decode_split_kernel with decode_combine_kernel (timed together: the combine overlaps the split's tail)"
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic, "peak_kind": peak_kind, "kernel": kernel,
                "algorithmic_bytes_per_launch": rig.bpc, "launch_us": round(kernel_us, 3)}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, per, sample, cores, _ = oracle_rate(case, budget_s=args.cpu_budget)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    run = run_of(args, case, rig.splits)
    run["l2"] = l2_note(rig.copies, f"pool copies of {rig.pool_bytes / 1e9:.3f} GB, reads",
                        rig.copies * rig.bpc, "every step reads KV from HBM")
    run["timing"] = (f"CUDA events around CUDA graphs of {chunk} back-to-back calls, queued behind a short "
                     f"GPU sleep so the region holds only the calls")
    run["single_call_us"] = round(single_us, 3)
    run["single_call"] = "one call alone on an idle GPU, CUDA events around it, median of 30"
    run["us_per_call_repeats"] = repeats
    run["concurrent_streams"] = concurrent(rig, conc_us, args.e2e_streams, peak)
    if spot is not None:
        run["spot_check_rel_rms"] = spot
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_call": round(ms_per_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(case), "run": run, "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": rig.host_in.numel(),
                "d2h_bytes_per_step": rig.o_h.numel() * rig.o_h.element_size(),
                "steps": e2e_steps, "us_per_step": round(e2e_s / e2e_steps * 1e6, 3),
                "mode": f"one CUDA graph of the steps taken in turn by {args.e2e_streams} streams, each with its "
                        "own buffer set: each step copies its inputs in, calls attn_decode and copies o out; one "
                        "step's copies overlap other steps' kernels",
                "streams": args.e2e_streams,
                "eager_us_per_step": round(eager_us, 3), "host_us_per_part": host_parts,
                "resident": "k_pool and v_pool stay in HBM (the KV cache); q, qpos, off and the block table come "
                            "from pinned host memory (one copy) and o goes back (one copy) every step"},
        "gpu_launches": args.steps * rig.launches_per_call
        + sum(e["steps"] * e["kernels_per_call"] for e in extra), "clocks": clocks,
    }
    if extra:
        line["workloads"] = extra
    print(json.dumps(line), flush=True)
    return 0


def run_prefill(args, case, rank, world, dist):
    """One step = one pgqa_attn_prefill call over every row of the case: TFLOP/s
    against the bf16 tensor peak.  Returns the line (rank 0) or 0."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    if rank == 0:
        pgqa.build()
    barrier(dist)
    pgqa.load()
    flops = prefill_flops(case)
    pool_bytes = case.k_pool.nbytes + case.v_pool.nbytes
    copies = args.copies or max(2, math.ceil(3 * L2_BYTES / pool_bytes))
    t0_h, tn_h = pgqa.make_tiles(case.off, pgqa.prefill_rows_per_tile(case.hd))
    ntiles = len(t0_h)

    def i16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))

    ks = [i16(case.k_pool).to(dev) for _ in range(copies)]
    vs = [i16(case.v_pool).to(dev) for _ in range(copies)]
    parts = [np.ascontiguousarray(a).view(np.uint8) for a in
             (case.q, np.asarray(case.qpos, np.int32), np.asarray(case.off, np.int32),
              np.asarray(case.block_table, np.int32), t0_h, tn_h)]
    offs, pos = [], 0
    for a in parts:
        offs.append(pos)
        pos += (a.size + 255) // 256 * 256
    host_in = torch.zeros(pos, dtype=torch.uint8).pin_memory()
    for a, o0 in zip(parts, offs):
        host_in[o0:o0 + a.size] = torch.from_numpy(a)
    dev_in = host_in.to(dev)
    views = [dev_in[o0:o0 + a.size] for a, o0 in zip(parts, offs)]
    q = views[0].view(torch.int16)
    qpos, off, bt, t0, tn = (v.view(torch.int32) for v in views[1:])
    o = torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16, device=dev)
    o_h = torch.empty_like(o, device="cpu").pin_memory()

    def call(i, stream=None):
        pgqa.attn_prefill(o, q, ks[i % copies], vs[i % copies], bt, off, qpos, None, t0, tn, ntiles, case.nh,
                          case.nkv, case.hd, case.window, None, stream)

    call(0)
    torch.cuda.synchronize()
    spot = None
    if rank == 0 and not args.no_check:
        import oracle
        got = o.cpu().numpy().view(np.uint16).reshape(case.rows, case.nh, case.hd)
        pairs = [(r, h) for r in range(case.rows) for h in range(case.nh)][:: max(1, case.rows * case.nh // 64)]
        _, ref = oracle.decode_case(case, pairs=pairs, want_f64=False)
        spot = oracle.rel_rms(np.stack([got[r, h] for r, h in pairs]), ref)
        if not spot < 1e-2:
            raise SystemExit(f"spot check against the oracle failed: rel_rms {spot}")
    sampler = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(args.steps):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    ev0.record(stream)
    g.replay()
    ev1.record(stream)
    ev1.synchronize()
    barrier(dist)
    el_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    el_max = max_over_ranks(dist, el_ms)
    value = sum_over_ranks(dist, float(flops) * args.steps) / (el_max * 1e-3) / 1e12
    kernel_us = el_ms * 1e3 / args.steps

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    barrier(dist)
    torch.cuda.synchronize()
    t_0 = time.perf_counter()
    for i in range(e2e_steps):
        dev_in.copy_(host_in, non_blocking=True)
        call(i)
        o_h.copy_(o, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t_0)
    e2e_value = sum_over_ranks(dist, float(flops) * e2e_steps) / e2e_s / 1e12
    if rank != 0:
        return 0
    peak, peak_kind = measured_bf16_peak()
    achieved = flops / (kernel_us * 1e-6) / 1e12
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, per, sample, cores, k = oracle_rate(case, budget_s=args.cpu_budget, steps=1)
        tflops_cpu = flops * k / (case.rows * case.nh) / per / 1e12
        cpu = {"value": round(tflops_cpu, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": sample}
    cfg = prefill_config(case)
    run = {"tiles": ntiles, "rows_per_tile": pgqa.prefill_rows_per_tile(case.hd),
           "l2": l2_note(copies, "pool copies", copies * pool_bytes, "K/V and Q come from HBM on every call"),
           "timing": f"CUDA events around one CUDA graph of {args.steps} back-to-back calls"}
    if spot is not None:
        run["spot_check_rel_rms"] = spot
    line = {
        "metric": "paged causal prefill attention TFLOP/s", "value": round(value, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": el_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg, "run": run,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(case.name, TILED_TRAFFIC_FILE, TILED_SOURCES),
                     "peak_kind": peak_kind,
                     "kernel": "prefill_tc_kernel<%d>%s" % (case.hd, " (CTA pairs)" if case.hd > 256 else ""),
                     "launch_us": round(kernel_us, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": host_in.numel(),
                "d2h_bytes_per_step": o_h.numel() * o_h.element_size(), "steps": e2e_steps,
                "us_per_step": round(e2e_s / e2e_steps * 1e6, 3)},
        "gpu_launches": args.steps, "clocks": clocks,
    }
    return line


def run_multirow(args, case, rank, world, dist):
    """One step = one pgqa_attn_prefill_split call (the tcgen05 tiled kernel with
    split-KV, then the combine kernel) serving a multi-token decode: KV GB/s
    against the HBM peak, as for the decode workloads.  Returns the line (rank 0) or 0."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    if rank == 0:
        pgqa.build()
    barrier(dist)
    pgqa.load()
    bpc = case.algorithmic_bytes()
    t0_h, tn_h = pgqa.make_tiles(np.asarray(case.off, np.int32), pgqa.prefill_rows_per_tile(case.hd))
    ntiles = len(t0_h)
    splits = args.splits or pgqa.prefill_split_count(case.kv_len_eff(), case.rows, ntiles, case.nh, case.nkv,
                                                     hd=case.hd)
    pool_bytes = case.k_pool.nbytes + case.v_pool.nbytes
    copies = args.copies or max(2, math.ceil(3 * L2_BYTES / max(bpc, 1)))
    copies = min(copies, max(2, int(0.25 * torch.cuda.get_device_properties(dev).total_memory // pool_bytes)))

    def i16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))

    ks = [i16(case.k_pool).to(dev) for _ in range(copies)]
    vs = [i16(case.v_pool).to(dev) for _ in range(copies)]
    parts = [np.ascontiguousarray(a).view(np.uint8) for a in
             (case.q, np.asarray(case.qpos, np.int32), np.asarray(case.off, np.int32),
              np.asarray(case.block_table, np.int32), t0_h, tn_h)]
    offs, pos = [], 0
    for a in parts:
        offs.append(pos)
        pos += (a.size + 255) // 256 * 256
    host_in = torch.zeros(pos, dtype=torch.uint8).pin_memory()
    for a, o0 in zip(parts, offs):
        host_in[o0:o0 + a.size] = torch.from_numpy(a)
    dev_in = host_in.to(dev)
    views = [dev_in[o0:o0 + a.size] for a, o0 in zip(parts, offs)]
    q = views[0].view(torch.int16)
    qpos, off, bt, t0, tn = (v.view(torch.int32) for v in views[1:])
    part = torch.empty(pgqa.decode_part_bytes(case.rows, case.nh, splits, case.hd) // 4 + 4, dtype=torch.float32,
                       device=dev)
    o = torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16, device=dev)
    o_h = torch.empty_like(o, device="cpu").pin_memory()

    def call(i, stream=None):
        pgqa.attn_prefill_split(o, part, q, ks[i % copies], vs[i % copies], bt, off, qpos, None, t0, tn, ntiles,
                                case.rows, case.nh, case.nkv, case.hd, case.window, splits, None, stream)

    call(0)
    torch.cuda.synchronize()
    spot = None
    if rank == 0 and not args.no_check:
        import oracle
        got = o.cpu().numpy().view(np.uint16).reshape(case.rows, case.nh, case.hd)
        pairs = [(r, h) for r in range(case.rows) for h in range(case.nh)][:: max(1, case.rows * case.nh // 32)]
        _, ref = oracle.decode_case(case, pairs=pairs, want_f64=False)
        spot = oracle.rel_rms(np.stack([got[r, h] for r, h in pairs]), ref)
        if not spot < 1e-2:
            raise SystemExit(f"spot check against the oracle failed: rel_rms {spot}")
    sampler = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(args.steps):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    ev0.record(stream)
    g.replay()
    ev1.record(stream)
    ev1.synchronize()
    barrier(dist)
    el_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    el_max = max_over_ranks(dist, el_ms)
    value = sum_over_ranks(dist, float(bpc) * args.steps) / (el_max * 1e-3) / 1e9
    call_us = el_ms * 1e3 / args.steps

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    barrier(dist)
    torch.cuda.synchronize()
    t_0 = time.perf_counter()
    for i in range(e2e_steps):
        dev_in.copy_(host_in, non_blocking=True)
        call(i)
        o_h.copy_(o, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t_0)
    e2e_value = sum_over_ranks(dist, float(bpc) * e2e_steps) / e2e_s / 1e9
    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, per, sample, cores, _ = oracle_rate(case, budget_s=args.cpu_budget)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    cfg = config_of(case)
    run = {"splits": splits, "tiles": ntiles, "path": "pgqa_attn_prefill_split (tcgen05 tiled, split-KV) "
           "+ the decode combine kernel",
           "l2": f"rotating {copies} pool copies", "timing": f"CUDA events around one CUDA graph of "
           f"{args.steps} back-to-back calls (two kernels each)"}
    if spot is not None:
        run["spot_check_rel_rms"] = spot
    line = {
        "metric": "multi-row decode KV GB/s (tiled split-KV path)", "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": el_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg, "run": run,
        "roofline": {"bound": "hbm", "achieved": round(value, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4),
                     "traffic": recorded_traffic(case.name, TILED_TRAFFIC_FILE, TILED_SOURCES),
                     "peak_kind": peak_kind,
                     "kernel": "prefill_tc_kernel<256> (split) + decode_combine_kernel<256>",
                     "call_us": round(call_us, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": host_in.numel(),
                "d2h_bytes_per_step": o_h.numel() * o_h.element_size(), "steps": e2e_steps,
                "us_per_step": round(e2e_s / e2e_steps * 1e6, 3)},
        "gpu_launches": 2 * args.steps, "clocks": clocks,
    }
    return line


def prep_config(case):
    return {"workload": case.name, "nh": case.nh, "nkv": case.nkv, "hd": case.hd, "rotary_dim": case.rotary_dim,
            "theta": case.theta, "norm_v": case.norm_v, "rows": case.rows,
            "bytes_per_call": case.bytes_moved()}


def run_prep(args, case, rank, world, dist):
    """One step = one pgqa_qk_norm_rope_write call over every row of the case:
    head-vector bytes read and written over the device time, against the measured
    HBM copy bandwidth.  Returns the line (rank 0) or 0."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    if rank == 0:
        pgqa.build()
    barrier(dist)
    pgqa.load()
    nbytes = case.bytes_moved()
    copies = args.copies or max(2, math.ceil(3 * L2_BYTES / nbytes))
    npool = max(int(case.block_table.max()) + 1, case.npg)

    def i16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))

    parts = [np.ascontiguousarray(a).view(np.uint8) for a in
             (case.q_in, case.k_in, case.v_in, np.asarray(case.pos, np.int32), np.asarray(case.off, np.int32))]
    offs, total = [], 0
    for a in parts:
        offs.append(total)
        total += (a.size + 255) // 256 * 256
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for a, o0 in zip(parts, offs):
        host_in[o0:o0 + a.size] = torch.from_numpy(a)
    ins = [host_in.to(dev) for _ in range(copies)]
    views = [[d[o0:o0 + a.size] for a, o0 in zip(parts, offs)] for d in ins]
    qw, kw = i16(case.q_weight).to(dev), i16(case.k_weight).to(dev)
    bt = torch.from_numpy(np.asarray(case.block_table, np.int32)).to(dev)
    q_out = [torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16, device=dev) for _ in range(copies)]
    k_pool = [torch.zeros(npool * case.nkv * 16 * case.hd, dtype=torch.int16, device=dev) for _ in range(copies)]
    v_pool = [torch.zeros_like(k_pool[0]) for _ in range(copies)]
    q_h = torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16).pin_memory()

    def call(i, stream=None):
        c = i % copies
        v = views[c]
        pgqa.qk_norm_rope_write(q_out[c], k_pool[c], v_pool[c], v[0].view(torch.int16), v[1].view(torch.int16),
                                v[2].view(torch.int16), qw, kw, v[3].view(torch.int32), bt,
                                v[4].view(torch.int32), None, case.rows, case.nh, case.nkv, case.hd,
                                case.rotary_dim, case.theta, case.eps, case.norm_v, stream)

    call(0)
    torch.cuda.synchronize()
    spot = None
    if rank == 0 and not args.no_check:
        from oracle import prep as op
        idx = np.arange(0, case.rows, max(1, case.rows // 64))
        q_ref, k_ref, v_ref, slot = op.prep(*prep_rows(case, idx))
        got_q = q_out[0].cpu().numpy().view(np.uint16).reshape(case.rows, case.nh, case.hd)[idx]
        kf = k_pool[0].cpu().numpy().view(np.uint16)
        vf = v_pool[0].cpu().numpy().view(np.uint16)
        worst = 0.0
        for got, ref in [(got_q, q_ref)] + [
                (f[slot[:, None] + kh * 16 * case.hd + np.arange(case.hd)[None, :]], r[:, kh])
                for kh in range(case.nkv) for f, r in ((kf, k_ref), (vf, v_ref))]:
            g = wl.bf16_to_f32(got).astype(np.float64)
            rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
            worst = max(worst, float(np.max(np.abs(g - ref) / (np.abs(ref) + rms))))
        if not worst <= 2.0 ** -8:
            raise SystemExit(f"spot check against the oracle failed: {worst}")
        spot = worst
    sampler = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(args.steps):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    ev0.record(stream)
    g.replay()
    ev1.record(stream)
    ev1.synchronize()
    barrier(dist)
    el_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    el_max = max_over_ranks(dist, el_ms)
    value = sum_over_ranks(dist, float(nbytes) * args.steps) / (el_max * 1e-3) / 1e9
    kernel_us = el_ms * 1e3 / args.steps

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    barrier(dist)
    torch.cuda.synchronize()
    t_0 = time.perf_counter()
    for i in range(e2e_steps):
        ins[i % copies].copy_(host_in, non_blocking=True)
        call(i)
        q_h.copy_(q_out[i % copies], non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t_0)
    e2e_value = sum_over_ranks(dist, float(nbytes) * e2e_steps) / e2e_s / 1e9
    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    achieved = nbytes / (kernel_us * 1e-6) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, per, sample, cores = prep_oracle_rate(case, args.cpu_budget)
        cpu = {"value": round(gbs, 6), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    cfg = prep_config(case)
    run = {"l2": l2_note(copies, "input/output copies, bytes moved", copies * nbytes,
                         "every call reads and writes HBM"),
           "timing": f"CUDA events around one CUDA graph of {args.steps} back-to-back calls"}
    if spot is not None:
        run["spot_check_worst_err_over_abs_plus_rms"] = spot
    line = {
        "metric": PREP_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in/out, f32 arithmetic", "data": "synthetic", "config": cfg,
        "run": run,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(case.name, PREP_TRAFFIC_FILE, PREP_SOURCES),
                     "peak_kind": peak_kind, "kernel": "qk_norm_rope_kernel", "launch_us": round(kernel_us, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": host_in.numel(),
                "d2h_bytes_per_step": q_h.numel() * q_h.element_size(), "steps": e2e_steps,
                "us_per_step": round(e2e_s / e2e_steps * 1e6, 3)},
        "gpu_launches": args.steps, "clocks": clocks,
    }
    return line


def sweep_bytes(hd, ctx, rows, window, nh=32, nkv=16):
    """Algorithmic bytes of one sweep call: the union window's K/V once, Q and O."""
    q0 = ctx - rows
    lo = max(0, q0 + 1 - window) if window > 0 else 0
    return (ctx - lo) * nkv * hd * 2 * 2 + 2 * rows * nh * hd * 2


def run_sweep(args, rank, world, dist):
    """Every point of the decode sweep (nh32 nkv16; hd x ctx x rows x window =
    3 x 4 x 3 x 3 = 108 points): rows at the last positions of one sequence, its
    pages in a seeded permuted order.  Points with more query rows per kv head
    than the decode kernel packs (rows x g > 8) go through the tiled tcgen05
    kernel with split-KV where it serves the head dimension.  Each point is timed with CUDA events around
    a graph of back-to-back calls over rotating pool copies; ``value`` is the
    geometric mean of the points' KV GB/s.  Pools are drawn once per (hd, ctx) on
    the device from a seeded generator (a timing run: the sweep's parity is the
    decode tests' business), so this line carries no end-to-end number."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    if rank == 0:
        pgqa.build()
    barrier(dist)
    pgqa.load()
    nh, nkv = 32, 16
    total_mem = torch.cuda.get_device_properties(dev).total_memory
    results = []
    sampler = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    t_all0 = time.perf_counter()
    for hd in wl.SWEEP_HD:
        for ctx in wl.SWEEP_CTX:
            npages = (ctx + 15) // 16
            pool_elems = npages * nkv * 16 * hd
            gen = torch.Generator(device=dev)
            gen.manual_seed(12345 + hd + ctx)
            pool_bytes = 2 * pool_elems * 2
            copies = max(2, math.ceil(3 * L2_BYTES / pool_bytes))
            copies = min(copies, 16, max(2, int(0.25 * total_mem // pool_bytes)))
            ks = [torch.randn(pool_elems, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                  for _ in range(copies)]
            vs = [torch.randn(pool_elems, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                  for _ in range(copies)]
            bt = torch.from_numpy(wl.lcg_permutation(npages, hd + ctx).astype(np.int32)).to(dev)
            for rows in wl.SWEEP_ROWS:
                for window in wl.SWEEP_WINDOW:
                    q = torch.randn(rows * nh * hd, generator=gen, device=dev).to(torch.bfloat16)
                    qpos = torch.arange(ctx - rows, ctx, dtype=torch.int32, device=dev)
                    off = torch.zeros(rows, dtype=torch.int32, device=dev)
                    kv_eff = min(ctx, window) if window > 0 else ctx
                    # more query rows per kv head than pgqa_attn_decode packs into a
                    # CTA (8): the rows are one sequence's last positions, served by the
                    # tiled tcgen05 kernel with split-KV
                    tiled = rows * (nh // nkv) > 8
                    if tiled:
                        t0_h, tn_h = pgqa.make_tiles(np.zeros(rows, np.int32), pgqa.prefill_rows_per_tile(hd))
                        t0 = torch.from_numpy(t0_h).to(dev)
                        tn = torch.from_numpy(tn_h).to(dev)
                        splits = pgqa.prefill_split_count(kv_eff, rows, len(t0_h), nh, nkv, hd=hd)
                    else:
                        splits = pgqa.choose_splits(kv_eff, rows, nkv, 1, nh=nh, hd=hd)
                    part = torch.empty(max(1, pgqa.decode_part_bytes(rows, nh, splits, hd)) // 4 + 4,
                                       dtype=torch.float32, device=dev)
                    cnt = torch.zeros(max(1, pgqa.decode_counter_count(rows, nh, nkv)), dtype=torch.int32,
                                      device=dev)
                    o = torch.empty(rows * nh * hd, dtype=torch.bfloat16, device=dev)
                    bpc = sweep_bytes(hd, ctx, rows, window, nh, nkv)

                    def call(i):
                        if tiled:
                            pgqa.attn_prefill_split(o, part, q, ks[i % copies], vs[i % copies], bt, off, qpos, None,
                                                    t0, tn, len(t0_h), rows, nh, nkv, hd, window, splits, None)
                        else:
                            pgqa.attn_decode(o, part, q, ks[i % copies], vs[i % copies], bt, off, qpos, None, rows,
                                             nh, nkv, hd, window, splits, cnt, None)

                    for i in range(3):
                        call(i)
                    torch.cuda.synchronize()
                    n = int(min(400, max(20, 2e-3 / max(bpc / 6e12, 5e-6))))
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        for i in range(n):
                            call(i)
                    g.replay()
                    torch.cuda.synchronize()
                    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    ev0.record()
                    g.replay()
                    ev1.record()
                    ev1.synchronize()
                    us = ev0.elapsed_time(ev1) * 1e3 / n
                    kernels = (1 + (splits > 1)) if tiled else pgqa.decode_kernel_count(splits, True)
                    results.append({"hd": hd, "ctx": ctx, "rows": rows, "window": window, "splits": splits,
                                    "path": "tiled split-KV" if tiled else "decode",
                                    "us": round(us, 3), "gbs": round(bpc / (us * 1e-6) / 1e9, 1),
                                    "bytes": bpc, "launches": n * kernels})
                    del g
            del ks, vs
            torch.cuda.empty_cache()
    clocks = sampler.stop() if sampler else None
    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    gm = math.exp(sum(math.log(r["gbs"]) for r in results) / len(results))
    by = sorted(results, key=lambda r: r["gbs"])
    if args.sweep_out:
        with open(args.sweep_out, "w") as f:
            json.dump(results, f, indent=0)
    line = {
        "metric": "paged decode attention KV GB/s, geometric mean over the sweep", "value": round(gm, 1),
        "unit": "GB/s", "n_gpus": world, "steps": len(results), "warmup": 3,
        "ms_per_step": round(sum(r["us"] for r in results) / len(results) / 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (device-drawn Gaussian pools)",
        "config": {"workload": "sweep_nh32_nkv16", "points": len(results),
                   "grid": "hd {128,256,512} x ctx {1K,4K,16K,64K} x rows {1,4,16} x window {0,1024,4096}",
                   "worst": by[:3], "best": by[-3:], "seconds": round(time.perf_counter() - t_all0, 1),
                   "paths": "pgqa_attn_decode; pgqa_attn_prefill_split for rows x g > 8",
                   "l2": "rotating pool copies per (hd, ctx)",
                   "timing": "per point: CUDA events around a graph of 20-400 back-to-back calls"},
        "roofline": {"bound": "hbm", "achieved": round(gm, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gm / peak, 4), "traffic": None, "peak_kind": peak_kind,
                     "kernel": "decode_split_kernel (geometric mean over the points)"},
        "cpu_baseline": None, "e2e": None, "gpu_launches": sum(r["launches"] for r in results), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sliding",
                    choices=["sliding", "sliding_mapped", "tiny", "long", "batched", "prefill_page", "prefill_long",
                             "prefill_hd512", "prep_long", "sweep", "multirow"])
    ap.add_argument("--splits", type=int, default=0, help="override choose_splits")
    ap.add_argument("--merge", choices=["counters", "combine"], default="counters")
    ap.add_argument("--graph-chunk", type=int, default=2000)
    ap.add_argument("--copies", type=int, default=0, help="override the number of rotated pool copies")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--e2e-streams", type=int, default=6,
                    help="decode e2e: streams (each with its own buffers) that take the steps in turn")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=60.0, help="seconds of oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--sweep-out", default="", help="--workload sweep: write every point's numbers here (JSON)")
    ap.add_argument("--no-extra", action="store_true",
                    help="sliding: skip timing the other workloads (long, batched, tiny, the tiled paths, the "
                         "K/V write) beside it")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of graph replays around the timed region while clocks are sampled")
    args = ap.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps >= 1 and --warmup >= 0")
    rank, world, _ = dist_env()
    if args.impl == "reference" and rank != 0:
        return 0            # the reference arm runs on rank 0 alone
    if args.workload == "sweep":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the sweep is a device timing of every point; "
                              "the oracle baseline is reported on the single workloads"}), flush=True)
            return 0
        dist = init_dist(world)
        try:
            return run_sweep(args, rank, world, dist)
        finally:
            if dist is not None:
                dist.destroy_process_group()
    case = build_case(args.workload)
    if args.impl == "reference":
        return run_reference(args, case, rank, world)
    dist = init_dist(world)
    try:
        if args.workload.startswith("prefill"):
            line = run_prefill(args, case, rank, world, dist)
        elif args.workload.startswith("prep"):
            line = run_prep(args, case, rank, world, dist)
        elif args.workload == "multirow":
            line = run_multirow(args, case, rank, world, dist)
        else:
            return run_ours(args, case, rank, world, dist)
        if isinstance(line, dict):
            print(json.dumps(line), flush=True)
        return 0
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
