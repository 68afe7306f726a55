"""Benchmark: paged decode on the Llama-3-8B-shaped GQA workload.

One step = one decode step of the whole hot path for 256 sequences:
  host block allocation of the step's new token (done before the timed region
  for the device-resident figure, inside it for the end-to-end figure),
  copy-on-write block copies (none arise in this workload),
  pa_reshape_and_cache of the new K/V, pa_decode (schedule, attention,
  partition merge).
Inputs: 256 sequences, lengths lognormal (median 1000, sigma 1.0, cap 8192),
32 query / 8 KV heads, D 128, B 16, bf16 N(0,1), shuffled physical blocks
(1.50 GB of K/V per step at the seeded lengths: larger than L2, so no flush
is needed).

Output: one JSON line (rank 0).  `value` is KV-read GB/s over whole steps;
`roofline` is the attention kernel alone against the measured HBM copy rate;
`cpu_baseline` / `--impl reference` time the fp64 oracle on host cores.
The same line carries, under `workloads`, the other decode workloads (OPT-13B,
the copy-on-write parallel-sampling step, the 32K Yi-34B context paged at three
block sizes and in the contiguous layout), the cache write and the block copy
timed on their own (`cache_ops`), the tensor-core prefill, the block swap to
and from pinned host memory (`swap`) and the virtually contiguous KV buffers
(`vmm`: page mapping cost, decode over the mapped pages); about a second each,
`--no-workloads` skips them.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged decode KV-read GB/s (% of HBM peak), seq-steps/s at Llama-3-8B GQA"
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attend_llama3_8b.json")
DECODE_SRC = os.path.join(ROOT, "paged_kv_cache_302_gb300", "csrc", "decode.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--seqs", type=int, default=256,
                    help="sequences (256 is the benchmarked workload; fewer for small profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads, cache ops and prefill in the default run")
    ap.add_argument("--clock-window", type=float, default=1.5,
                    help="seconds of the same decode steps replayed right after the timed region under the clock "
                         "sampler (not part of value)")
    ap.add_argument("--measure", choices=["decode", "swap", "prefill", "configs", "vmm"], default="decode",
                    help="swap: pa_swap_blocks device<->pinned host; prefill: chunked paged prefill (tcgen05)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def whole_job(t_local: float, bytes_local: float, device):
    """Whole-job figures of independent replicas: the slowest rank's time and the sum of all ranks' bytes
    (a plain pass-through on one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(t_local), float(bytes_local)
    t = torch.tensor([float(t_local)], dtype=torch.float64, device=device)
    b = torch.tensor([float(bytes_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def workload(steps: int, warmup: int, seqs: int = 256) -> W.Workload:
    # room for every decode step of the device and end-to-end phases
    return W.llama3_8b(n_seqs=seqs, grow=2 * (steps + warmup) + 16)


def config_dict(w: W.Workload, pt: int) -> dict:
    return {
        "workload": "llama3_8b_gqa_paged_decode",
        "seqs": w.N, "H_q": w.H_q, "H_kv": w.H_kv, "D": w.D, "block_size": w.B, "kv_dtype": w.dtype,
        "ctx": "lognormal(median 1000, sigma 1.0), capped at 8192",
        "ctx_tokens_first_step": int(w.ctx.sum()),
        "partition_tokens": 512 if pt == 0 else pt,
        "l2": "inputs larger than L2 (1.50 GB of K/V per step at the seeded lengths), no flush",
    }


# ----------------------------------------------------------------------------- oracle timing

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the architecture)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def oracle_sample_rate(w: W.Workload, host_pool, tables, ctx, q, target_s: float, nthreads: int = 0):
    """Time the oracle over whole sequences (every query head) until ~target_s of CPU work
    (nthreads 0: every host core)."""
    import oracle

    order = np.random.default_rng(9).permutation(w.N)
    nthreads = nthreads or oracle.num_threads()
    done_bytes, t_total, seqs = 0, 0.0, 0
    per_tok = 2 * w.H_kv * w.D * w.elem_bytes
    for chunk in np.array_split(order, 16):
        pairs = np.array([(s, h) for s in chunk for h in range(w.H_q)], dtype=np.int32)
        t0 = time.perf_counter()
        oracle.paged_decode(q, host_pool, tables, ctx, w.dtype, pairs=pairs, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        done_bytes += int(ctx[chunk].astype(np.int64).sum()) * per_tok
        seqs += len(chunk)
        if t_total * nthreads >= target_s or t_total >= target_s:
            break
    return done_bytes / t_total / 1e9, nthreads, seqs, t_total


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    w = workload(args.steps, args.warmup, args.seqs)
    host_pool, tables, ctx, slots = host_state(w)
    q = W.queries(w)
    nthreads = oracle.num_threads()
    per_tok = 2 * w.H_kv * w.D * w.elem_bytes
    # each step: the oracle over a fixed seeded subset of whole sequences
    rng = np.random.default_rng(11)
    subset = np.sort(rng.choice(w.N, size=8, replace=False))
    pairs = np.array([(s, h) for s in subset for h in range(w.H_q)], dtype=np.int32)
    step_bytes = int(ctx[subset].astype(np.int64).sum()) * per_tok
    for _ in range(args.warmup):
        oracle.paged_decode(q, host_pool, tables, ctx, w.dtype, pairs=pairs, nthreads=nthreads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.paged_decode(q, host_pool, tables, ctx, w.dtype, pairs=pairs, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = step_bytes / t / 1e9
    sample = (f"fp64 oracle over all {w.H_q} query heads of 8 seeded sequences "
              f"({int(ctx[subset].sum())} context tokens) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, args.partition_tokens),
        "seq_steps_per_s": len(subset) / t,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- shared setup

def host_state(w: W.Workload):
    """Host-side pool, tables and lengths of the workload (oracle layout), used by the CPU legs."""
    import oracle
    from oracle.alloc_model import AllocModel

    m = AllocModel(w.NB, w.B, w.free_order)
    slots = []
    for s in range(w.N):
        m.add_seq(s)
        slots += m.append_slots(s, int(w.ctx[s]))[0]
    slots = np.asarray(slots, dtype=np.int64)
    MB = w.max_blocks_per_seq()
    tables = np.full((w.N, MB), -1, dtype=np.int32)
    for s in range(w.N):
        t = m.block_table(s)
        tables[s, : len(t)] = t
    k, v = W.token_kv(w, slots.size)
    pool = np.zeros((w.NB, w.B, 2, w.H_kv, w.D), dtype=np.uint16)
    oracle.reshape_and_cache(k, v, pool, slots)
    return pool, tables, w.ctx.copy(), slots


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which: str):
        setattr(self, which, time.time())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        """Samples taken from mark('t0') (start of the timed region) to mark('t2') (end of the clock window that
        replays the same steps right after it; mark('t1') when there is none), and how many fell inside the timed
        region itself."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", 0.0), getattr(self, "t1", float("inf"))
        t_end = getattr(self, "t2", t1)
        in_timed = 0
        for t, ln in self.lines:
            if not (t0 <= t <= t_end + 0.025):
                continue
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            in_timed += t <= t1 + 0.025
            for name, val in zip(names, p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": int(in_timed),
                "window_s": round(t_end - t0, 3),
                "note": "nvidia-smi every 20 ms over the timed region and the same decode steps replayed right "
                        "after it (not part of value)"}


DEVICE_HDR = os.path.join(ROOT, "paged_kv_cache_302_gb300", "csrc", "pa_device.cuh")


def attend_source_sha256() -> str:
    """Hash of the attention kernel's source: its template in decode.cu plus the device helpers."""
    src = open(DECODE_SRC).read()
    a = src.index("// ============================================================================= 2. attention")
    b = src.index("// ============================================================================= 3. partition merge")
    return hashlib.sha256((src[a:b] + open(DEVICE_HDR).read()).encode()).hexdigest()


def profile_traffic(bytes_per_launch: float):
    """DRAM bytes per attention launch: the committed ncu capture's DRAM bytes per algorithmic byte, scaled to
    this launch (traffic grows with the context tokens), if the kernel is unchanged since the capture."""
    try:
        d = json.load(open(PROFILE_SUMMARY))
        if d.get("attend_source_sha256") != attend_source_sha256():
            return None, "attention kernel changed since the ncu capture"
        return float(d["dram_bytes_per_algorithmic_byte"]) * bytes_per_launch, d.get("note", "")
    except Exception:
        return None, "no ncu summary"


# ----------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch

    import paged_kv_cache_302_gb300 as pa

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pa.load()
    w = workload(args.steps, args.warmup, args.seqs)
    nsteps = args.steps + args.warmup
    pt = args.partition_tokens

    # ---- build the cache state: allocate every context, write all K/V through slot_mapping
    alloc = pa.BlockAllocator(w.NB, w.B, w.free_order)
    prompt_len = w.ctx - 1                      # the decode step adds the last token
    slots = []
    for s in range(w.N):
        alloc.add_seq(s)
        if prompt_len[s] > 0:
            slots.append(alloc.append_slots(s, int(prompt_len[s]))[0])
    slots = np.concatenate(slots)
    k, v = W.token_kv(w, slots.size)
    dt = torch.bfloat16
    pool = torch.zeros((w.NB, w.B, 2, w.H_kv, w.D), dtype=dt, device=dev)

    def dev_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)

    for lo in range(0, slots.size, 1 << 20):
        hi = min(slots.size, lo + (1 << 20))
        pa.pa_reshape_and_cache(dev_bits(k[lo:hi]), dev_bits(v[lo:hi]), pool, torch.from_numpy(slots[lo:hi]).to(dev))
    del k, v
    MB = w.max_blocks_per_seq(grow=2 * nsteps + 16)
    seq_ids = list(range(w.N))
    ones = np.ones(w.N, dtype=np.int32)

    # ---- device-resident phase: allocation for every step done up front
    step_inputs = W.decode_steps(w, nsteps)
    slot_steps, ctx_steps = [], []
    for i in range(nsteps):
        sl, pairs = alloc.append_batch(seq_ids, ones)
        assert pairs.size == 0
        slot_steps.append(torch.from_numpy(sl).to(dev))
        ctx_steps.append(torch.from_numpy(np.array([alloc.seq_len(s) for s in seq_ids], dtype=np.int32)).to(dev))
    tables, _ = alloc.block_tables(seq_ids, MB)
    tab = torch.from_numpy(tables).to(dev)
    q_d = [dev_bits(x[0]) for x in step_inputs]
    k_d = [dev_bits(x[1]) for x in step_inputs]
    v_d = [dev_bits(x[2]) for x in step_inputs]
    max_ctx = int(w.ctx.max()) + 2 * nsteps + 16
    ws = torch.empty(pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, max_ctx, pt), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((w.N, w.H_q, w.D), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    per_tok = 2 * w.H_kv * w.D * w.elem_bytes
    step_bytes = [int(c.sum().item()) * per_tok for c in ctx_steps]
    stream = torch.cuda.current_stream()
    att_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(nsteps)]

    def step(i, events=None):
        pa.pa_reshape_and_cache(k_d[i], v_d[i], pool, slot_steps[i], dev_err=err)
        pa.pa_decode(out, q_d[i], pool, tab, ctx_steps[i], max_ctx, partition_tokens=pt, workspace=ws,
                     dev_err=err, attend_events=events)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.5)                      # let the sampler start (before the warm-up: no idle gap before timing)
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        launches0 = pa.launch_count()
        clk.mark("t0")
        e0.record(stream)
        for i in range(args.warmup, nsteps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark("t1")
        launches = pa.launch_count() - launches0
        # clock window: the timed region is a few milliseconds, shorter than the sampler's period, so the same
        # steps (each rewrites its own token and reads its own lengths: replaying them changes nothing) run again
        # for a second or so under the sampler
        t_end = time.time() + args.clock_window
        while time.time() < t_end:
            for i in range(args.warmup, nsteps):
                step(i)
            torch.cuda.synchronize()
        clk.mark("t2")
    t_dev = e0.elapsed_time(e1) * 1e-3
    # the attention kernel alone: the same steps again with events around it (an event between the
    # schedule and attention kernels stops their overlap, so these runs are not part of `value`)
    for i in range(args.warmup, nsteps):
        step(i, att_ev[i])
    torch.cuda.synchronize()
    attend_s = [att_ev[i][0].elapsed_time(att_ev[i][1]) * 1e-3 for i in range(args.warmup, nsteps)]
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    timed_bytes = sum(step_bytes[args.warmup:])
    t_dev, total_bytes = whole_job(t_dev, timed_bytes, dev)
    value = total_bytes / t_dev / 1e9
    ms_per_step = t_dev / args.steps * 1e3

    # ---- roofline of the attention kernel
    hbm, peak_src = peaks()
    att_mean = sum(attend_s) / len(attend_s)
    att_bytes = sum(step_bytes[args.warmup:]) / args.steps
    achieved = att_bytes / att_mean / 1e9
    traffic, traffic_note = profile_traffic(att_bytes)

    # ---- end-to-end through the public API with host buffers
    e2e_value, h2d, d2h, e2e_parts = None, 0, 0, None
    if not args.no_e2e:
        e2e_value, h2d, d2h, e2e_parts = run_e2e(args, w, alloc, pool, ws, out, err, MB, max_ctx, pt, dev, world,
                                                 tab)

    # ---- CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_pool, tables_h, ctx_h, _ = host_state(w)
        qh = W.queries(w)
        rate, cores, seqs, secs = oracle_sample_rate(w, host_pool, tables_h, ctx_h, qh, args.cpu_seconds)
        rate1, _, seqs1, secs1 = oracle_sample_rate(w, host_pool, tables_h, ctx_h, qh, min(args.cpu_seconds, 3.0), 1)
        cpu = {"value": rate, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"fp64 oracle, all {w.H_q} query heads of {seqs} of the {w.N} sequences "
                         f"(first decode step's contexts), {secs:.1f} s wall",
               "single_thread_value": rate1,
               "single_thread_sample": f"{seqs1} sequences, {secs1:.1f} s", "cpu_model": cpu_model()}

    # ---- the other workloads, the cache ops alone and the prefill (rank 0, N = 1 only; about a second each)
    extra = {}
    if rank == 0 and world == 1 and not args.no_workloads:
        extra = {"workloads": measure_workloads(hbm), "cache_ops": measure_cache_ops(hbm),
                 "prefill": measure_prefill(), "swap": measure_swap(), "vmm": measure_vmm()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(config_dict(w, pt), parallelism="independent replicas" if world > 1 else "1 GPU"),
            "seq_steps_per_s": w.N * world / (t_dev / args.steps),
            "pct_of_hbm_peak": 100.0 * value / world / hbm,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": traffic, "kernel": "attend_kernel<bf16,128,paged>",
                         "bytes_per_launch": att_bytes, "per_unit": f"{per_tok} B per context token",
                         "peak_source": peak_src, "traffic_note": traffic_note},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "breakdown": e2e_parts},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            **extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_e2e(args, w, alloc, pool, ws, out, err, MB, max_ctx, pt, dev, world, tab):
    """Decode steps through the public API from pinned host buffers.  Each step's inputs (q and the new K/V) sit in
    a pinned staging buffer of their own; the host block allocation of the step (slots, lengths and block-table
    updates, padded to a fixed count with skipped rows) is written into the same buffer.  Inside the timed region,
    per step i: the host allocation of step i+1 (it needs only the lengths, so it runs while the device works on
    step i), then the host->device copy of step i+1's staging buffer on a copy stream (into the device staging
    buffer step i-1 used: the host synchronised with step i-1 before), so that it overlaps step i's kernels as a
    serving loop's double-buffered inputs would; then one CUDA graph launch for step i (applies the table updates,
    writes the cache and runs the decode -- plan, attention, merge -- with its output in pinned host memory, so
    the kernels write the result rows across the host link themselves: the step's device->host bytes), after
    the main stream waits for step i's copy; then a synchronisation.  Every timed step still moves its own input
    and output bytes.  The graphs hold the same library calls a user would make eagerly, captured once per device
    staging buffer before the timed region: they remove the host launch latency, not device work.  Returns the
    e2e rate, the bytes in and out per step, and a breakdown of one step's costs measured after the timed region."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    e2e_steps = min(args.steps, 30)
    nsteps = e2e_steps + args.warmup
    per_tok = 2 * w.H_kv * w.D * w.elem_bytes
    seq_ids = list(range(w.N))
    ones = np.ones(w.N, dtype=np.int32)
    ctx = np.array([alloc.seq_len(s) for s in seq_ids], dtype=np.int32)
    cap_u = 2 * w.N + 1   # table updates per step: at most a new block and a copy-on-write replacement per sequence

    def al(x):
        return (x + 15) // 16 * 16

    # staging layout (bytes): q | k | v | slots int64 | ctx int32 | table updates int32[cap_u, 3]
    nq, nk = w.N * w.H_q * w.D * 2, w.N * w.H_kv * w.D * 2
    o_k = al(nq)
    o_v = o_k + al(nk)
    o_s = o_v + al(nk)
    o_c = o_s + al(w.N * 8)
    o_u = o_c + al(w.N * 4)
    total = o_u + al(cap_u * 12)
    stage = []
    for q, k, v in W.decode_steps(w, nsteps):
        h = torch.empty(total, dtype=torch.uint8).pin_memory()
        hb = h.numpy()
        hb[:nq] = q.view(np.uint8).reshape(-1)
        hb[o_k:o_k + nk] = k.view(np.uint8).reshape(-1)
        hb[o_v:o_v + nk] = v.view(np.uint8).reshape(-1)
        stage.append(h)
    main = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    d_stages = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_out = torch.empty((w.N, w.H_q, w.D), dtype=torch.float32).pin_memory()
    d2h = h_out.numel() * 4

    def views(d):
        return (d[:nq].view(torch.bfloat16).view(w.N, w.H_q, w.D),
                d[o_k:o_k + nk].view(torch.bfloat16).view(w.N, w.H_kv, w.D),
                d[o_v:o_v + nk].view(torch.bfloat16).view(w.N, w.H_kv, w.D),
                d[o_s:o_s + w.N * 8].view(torch.int64),
                d[o_c:o_c + w.N * 4].view(torch.int32),
                d[o_u:o_u + cap_u * 12].view(torch.int32).view(cap_u, 3))

    graphs = []
    for d in d_stages:
        d_q, d_k, d_v, d_slot, d_ctx, d_upd = views(d)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pa.pa_update_block_tables(tab, d_upd, dev_err=err)
            pa.pa_reshape_and_cache(d_k, d_v, pool, d_slot, dev_err=err)
            pa.pa_decode(h_out, d_q, pool, tab, d_ctx, max_ctx, partition_tokens=pt, workspace=ws, dev_err=err)
        graphs.append(g)
    torch.cuda.synchronize()
    copied = [torch.cuda.Event() for _ in range(2)]

    def prepare(i):
        """Host block allocation of step i into its staging buffer (it needs the lengths only)."""
        nonlocal ctx
        sl, pairs, upd = alloc.append_batch(seq_ids, ones, table_updates=True)
        ctx = ctx + 1
        hb = stage[i].numpy()
        hb[o_s:o_s + w.N * 8] = sl.view(np.uint8)
        hb[o_c:o_c + w.N * 4] = ctx.view(np.uint8)
        u = np.full((cap_u, 3), -1, dtype=np.int32)
        u[:upd.shape[0]] = upd
        hb[o_u:o_u + cap_u * 12] = u.view(np.uint8).reshape(-1)
        return pairs, int(ctx.astype(np.int64).sum()) * per_tok

    def copy_in(i):
        """Host->device copy of step i's staging buffer on the copy stream (device buffer i % 2)."""
        with torch.cuda.stream(copy_stream):
            d_stages[i % 2].copy_(stage[i], non_blocking=True)
            copied[i % 2].record(copy_stream)

    def e2e_step(i, prep, next_i):
        """Runs step i; the host prepares and copies in step next_i while the device works."""
        pairs, nbytes = prep
        main.wait_event(copied[i % 2])
        if pairs.size:   # copy-on-write before the step's cache write (none in this workload: no forks)
            pa.pa_copy_blocks(pool, torch.from_numpy(pairs).to(dev), dev_err=err)
        graphs[i % 2].replay()
        nxt = None
        if next_i is not None:
            nxt = prepare(next_i)
            copy_in(next_i)
        main.synchronize()
        return nbytes, nxt

    prep = prepare(0)
    copy_in(0)
    for i in range(args.warmup):
        _, prep = e2e_step(i, prep, i + 1)
    if world > 1:
        torch.distributed.barrier()
    e2e_bytes = []
    t0 = time.perf_counter()
    for i in range(args.warmup, nsteps):
        nbytes, prep = e2e_step(i, prep, i + 1 if i + 1 < nsteps else None)
        e2e_bytes.append(nbytes)
    t_e2e = time.perf_counter() - t0
    copy_stream.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    # the last step's result, as the kernels wrote it into host memory, against the same decode into device memory
    last = (nsteps - 1) % 2
    d_q, _, _, _, d_ctx, _ = views(d_stages[last])
    pa.pa_decode(out, d_q, pool, tab, d_ctx, max_ctx, partition_tokens=pt, workspace=ws, dev_err=err)
    assert torch.equal(out.cpu(), h_out), "decode output written to host memory differs from the device result"

    # breakdown of one step, measured apart (each piece alone, so they do not add up to the pipelined step):
    # the host allocation, the input copy and the step's graph (device time, output into host memory)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    reps = 10
    ev[0].record(main)
    for _ in range(reps):
        d_stages[last].copy_(stage[nsteps - 1], non_blocking=True)
    ev[1].record(main)
    for _ in range(reps):
        graphs[last].replay()     # replays the last step: it rewrites its own token and reads its own lengths
    ev[2].record(main)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), h_out), "replayed step differs"
    probe = pa.BlockAllocator.from_state(alloc.export_state())
    th = time.perf_counter()
    for _ in range(reps):
        probe.append_batch(seq_ids, ones, table_updates=True)
    t_host = (time.perf_counter() - th) / reps
    probe.close()
    breakdown = {"host_allocation_us": t_host * 1e6,
                 "input_copy_us": ev[0].elapsed_time(ev[1]) * 1e3 / reps,
                 "device_step_us": ev[1].elapsed_time(ev[2]) * 1e3 / reps,
                 "step_us": t_e2e / e2e_steps * 1e6,
                 "note": "each piece timed alone after the timed region; in the timed steps the host allocation and "
                         "the input copy of step i+1 overlap the device work of step i"}
    t_e2e, e2e_total = whole_job(t_e2e, sum(e2e_bytes), dev)
    e2e_value = e2e_total / t_e2e / 1e9
    return e2e_value, total, d2h, breakdown


def measure_swap(steps: int = 10, warmup: int = 3) -> dict:
    """Swap bandwidth: pa_swap_blocks moving whole Llama-3-8B-shaped blocks (16 tokens x 8 KV heads x 128, bf16:
    64 KB each) between the device pool and a pinned host pool, both directions, CUDA events; and one contiguous
    copy of the same bytes each way by the copy engine, for reference."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    B, H, D, nblk = 16, 8, 128, 4096            # 256 MB per direction
    dev_pool = torch.empty((nblk, B, 2, H, D), dtype=torch.bfloat16, device="cuda").normal_()
    host_pool = torch.empty((nblk, B, 2, H, D), dtype=torch.bfloat16).pin_memory()
    rng = np.random.default_rng(12)
    out_pairs = torch.from_numpy(np.stack([rng.permutation(nblk), rng.permutation(nblk)], 1).astype(np.int64)).cuda()
    in_pairs = torch.from_numpy(np.stack([rng.permutation(nblk), rng.permutation(nblk)], 1).astype(np.int64)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = {"unit": "GB/s", "blocks": nblk, "block_bytes": B * 2 * H * D * 2, "calls": steps}
    for name, dst, src, pairs in (("swap_out_d2h", host_pool, dev_pool, out_pairs),
                                  ("swap_in_h2d", dev_pool, host_pool, in_pairs)):
        for _ in range(warmup):
            pa.pa_swap_blocks(dst, src, pairs, dev_err=err)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            pa.pa_swap_blocks(dst, src, pairs, dev_err=err)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / steps
        res[name] = dev_pool.numel() * 2 / t / 1e9
    for name, dst, src in (("memcpy_d2h_contiguous", host_pool, dev_pool), ("memcpy_h2d_contiguous", dev_pool,
                                                                             host_pool)):
        dst.copy_(src, non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        res[name] = dev_pool.numel() * 2 / (e0.elapsed_time(e1) * 1e-3 / steps) / 1e9
    assert int(err.item()) == 0
    del dev_pool, host_pool
    return res


def run_swap(args):
    import torch

    torch.cuda.set_device(0)
    print(json.dumps({"measure": "pa_swap_blocks", **measure_swap(args.steps, args.warmup)}), flush=True)
    return 0


def measure_prefill(steps: int = 10, warmup: int = 3) -> list:
    """Chunked paged prefill on the tensor cores: Llama-3-8B shapes (32 q / 8 KV heads, D 128), 16 sequences whose
    last 2048 of 4096 tokens are the chunk (K/V already in the pool).  With 16-token blocks: bf16 with V staged,
    bf16 without a workspace (split P) and fp16; then bf16 staged and fp16 with 8- and 32-token blocks.  FLOPs
    count the causal score and value products actually needed: 4 * D * (position + 1) per query row and head.
    Calls back to back, CUDA events."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    N, ctx_len, chunk, H_q, H_kv, D = 16, 4096, 2048, 32, 8, 128
    ctx = torch.full((N,), ctx_len, dtype=torch.int32, device="cuda")
    q_start = torch.arange(0, (N + 1) * chunk, chunk, dtype=torch.int32, device="cuda")
    out = torch.empty((N * chunk, H_q, D), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = np.arange(ctx_len - chunk, ctx_len, dtype=np.float64)
    flops = N * H_q * 4.0 * D * float((pos + 1).sum())
    peak, peak_src = 1900.0, "fallback (1.9 PFLOP/s bf16, one earlier GB300 measurement)"
    try:
        peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
        peak_src = "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    except Exception:
        pass
    res = []
    cases = [(16, torch.bfloat16, "bf16", True), (16, torch.bfloat16, "bf16", False), (16, torch.float16, "f16", False),
             (8, torch.bfloat16, "bf16", True), (8, torch.float16, "f16", False),
             (32, torch.bfloat16, "bf16", True), (32, torch.float16, "f16", False)]
    for B, dt, name, stage_v in cases:
        nb = ctx_len // B
        NB = N * nb + 64
        perm = torch.from_numpy(np.random.default_rng(13).permutation(NB)[: N * nb].astype(np.int32))
        tables = perm.view(N, nb).cuda()
        ws = torch.empty(pa.pa_prefill_workspace_bytes(N, H_kv, D, B, nb), dtype=torch.uint8, device="cuda")
        pool = torch.empty((NB, B, 2, H_kv, D), dtype=dt, device="cuda").normal_()
        q = torch.empty((N * chunk, H_q, D), dtype=dt, device="cuda").normal_()

        def call():
            pa.pa_prefill(out, q, pool, tables, ctx, q_start, chunk, workspace=ws, stage_v=stage_v, dev_err=err)

        n = steps if B == 16 else max(3, steps // 2)
        for _ in range(warmup):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            call()
        e1.record()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        t = e0.elapsed_time(e1) * 1e-3 / n
        tf = flops / t / 1e12
        # the fp16 dense tensor rate equals the bf16 one on this GPU
        how = ("V staged as fp16 by a first kernel (included), one value product" if stage_v and name == "bf16"
               else "P split into two bf16 parts, two value products" if name == "bf16" else "fp16 P, one product")
        # the library's choice of kernel for these rows (prefill.cu: the wide kernel serves fp16 value products;
        # PA_PREFILL_KERNEL=narrow forces the two-tile kernel)
        wide = (name == "f16" or stage_v) and os.environ.get("PA_PREFILL_KERNEL", "") != "narrow"
        kernel = "prefill_wide_kernel" if wide else "prefill_kernel"
        res.append({"kv_dtype": name, "block_tokens": B, "value_product": how, "kernel": kernel, "unit": "TFLOP/s",
                    "value": tf, "ms_per_call": t * 1e3, "peak_bf16_tflops": peak, "peak_source": peak_src,
                    "frac": tf / peak, "seqs": N, "ctx": ctx_len, "chunk": chunk, "flops_per_call": flops,
                    "calls": n})
        del pool, q, ws
    return res


def run_prefill(args):
    import torch

    torch.cuda.set_device(0)
    for r in measure_prefill(args.steps, args.warmup):
        print(json.dumps({"measure": "pa_prefill", **r}), flush=True)
    return 0


def _time_decode(fn, att_ev, reps=20, warm=3):
    """(whole call, attention kernel) in seconds.  The whole call is timed over `reps` back-to-back calls
    between two events (the host enqueues ahead, as in a decode loop); the attention kernel is the median of
    per-call events around it, taken in a second pass (those events stop the schedule/attention overlap)."""
    import torch

    for _ in range(warm):
        fn(None)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn(None)
    e1.record()
    torch.cuda.synchronize()
    t_call = e0.elapsed_time(e1) * 1e-3 / reps
    ta = []
    for _ in range(reps):
        fn(att_ev)
        torch.cuda.synchronize()
        ta.append(att_ev[0].elapsed_time(att_ev[1]) * 1e-3)
    return t_call, float(np.median(ta))


def _time_cold(fn, reps=15, warm=3):
    """Median seconds of one call with L2 flushed before it (a 512 MB buffer is written between calls), CUDA
    events around the call alone."""
    import torch

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    del flush
    return float(np.median(ts))


def _paged_case(w, alloc_fn=None):
    """Allocator state, device tables and an N(0,1) pool / queries (drawn on the device) for a workload."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    a = pa.BlockAllocator(w.NB, w.B, w.free_order)
    extra = None
    if alloc_fn is None:
        for s in range(w.N):
            a.add_seq(s)
            a.append_slots(s, int(w.ctx[s]))
    else:
        extra = alloc_fn(a)
    tables, ctx = a.block_tables(list(range(w.N)), w.max_blocks_per_seq())
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    pool = torch.empty((w.NB, w.B, 2, w.H_kv, w.D), dtype=dt, device="cuda").normal_()
    q = torch.empty((w.N, w.H_q, w.D), dtype=dt, device="cuda").normal_()
    out = torch.empty((w.N, w.H_q, w.D), device="cuda")
    tab, cx = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
    ws = torch.empty(pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, int(ctx.max()), 0), dtype=torch.uint8,
                     device="cuda")
    return dict(a=a, tables=tables, ctx=ctx, pool=pool, q=q, out=out, tab=tab, cx=cx, ws=ws, extra=extra)


def measure_workloads(hbm: float) -> dict:
    """Decode throughput on the other workloads (whole pa_decode call back to back, and the attention kernel
    alone): OPT-13B MHA; the copy-on-write parallel-sampling batch, decode on logical and unique K/V bytes and a
    whole device step (the 224 copy-on-write block copies, the cache write of every sample's new tokens, the
    decode); the Yi-34B-shaped 32K context paged at B = 8 / 16 / 32 and in the contiguous per-request layout (the
    unpaged comparison).  Pools and queries are N(0,1) drawn on the device (throughput does not depend on the
    values; parity at these sizes is the test suite's)."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    res = {}

    def decode_fn(c):
        return lambda e: pa.pa_decode(c["out"], c["q"], c["pool"], c["tab"], c["cx"], int(c["ctx"].max()),
                                      workspace=c["ws"], dev_err=err, attend_events=e)

    def rates(nbytes, t, ta):
        return {"kv_bytes": nbytes, "step_gbs": nbytes / t / 1e9, "attend_gbs": nbytes / ta / 1e9,
                "attend_frac_of_hbm": nbytes / ta / 1e9 / hbm, "us_per_call": t * 1e6}

    # OPT-13B-shaped MHA
    w = W.opt13b()
    c = _paged_case(w)
    nbytes = int(c["ctx"].astype(np.int64).sum()) * 2 * w.H_kv * w.D * 2
    res["opt13b_mha_fp16"] = rates(nbytes, *_time_decode(decode_fn(c), ev))
    del c

    # parallel sampling with copy-on-write prefix sharing: prompts written, forked to 8 samples, then one batched
    # append of every sample's divergent tokens (host), the copy-on-write copies, the cache write and the decode
    w = W.cow()

    def cow_alloc(a):
        for pidx in range(w.prompts):
            base = pidx * w.samples
            a.add_seq(base)
            a.append_slots(base, w.prompt_len)
            for j in range(1, w.samples):
                a.fork(base, base + j)
        t0 = time.perf_counter()
        slots, pairs = a.append_batch(list(range(w.N)), w.extra)
        return slots, pairs, time.perf_counter() - t0

    c = _paged_case(w, cow_alloc)
    slots, pairs, t_host = c["extra"]
    per_tok = 2 * w.H_kv * w.D * 2
    logical = int(c["ctx"].astype(np.int64).sum()) * per_tok
    uniq = len(set(c["tables"][c["tables"] >= 0].tolist())) * w.B * per_tok
    t, ta = _time_decode(decode_fn(c), ev)
    r = rates(logical, t, ta)
    r.update(unique_kv_bytes=uniq, attend_unique_gbs=uniq / ta / 1e9, attend_unique_frac_of_hbm=uniq / ta / 1e9 / hbm)
    d_pairs = torch.from_numpy(np.ascontiguousarray(pairs)).cuda()
    d_slots = torch.from_numpy(slots).cuda()
    T = int(slots.size)
    k = torch.empty((T, w.H_kv, w.D), dtype=torch.bfloat16, device="cuda").normal_()
    v = torch.empty_like(k)

    def cow_step():
        pa.pa_copy_blocks(c["pool"], d_pairs, dev_err=err)
        pa.pa_reshape_and_cache(k, v, c["pool"], d_slots, dev_err=err)
        decode_fn(c)(None)

    for _ in range(3):
        cow_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record()
    for _ in range(reps):
        cow_step()
    e1.record()
    torch.cuda.synchronize()
    t_step = e0.elapsed_time(e1) * 1e-3 / reps
    blk = w.B * per_tok
    t_copy = _time_cold(lambda: pa.pa_copy_blocks(c["pool"], d_pairs, dev_err=err))
    r["cow_step"] = {
        "what": "device part of one step: pa_copy_blocks of the copy-on-write pairs, pa_reshape_and_cache of every "
                "sample's new tokens, pa_decode over all sequences; 20 steps back to back",
        "cow_pairs": int(pairs.shape[0]), "new_tokens": T, "us_per_step": t_step * 1e6,
        "logical_kv_gbs": logical / t_step / 1e9,
        "host_append_batch_us": t_host * 1e6,
        "copy_blocks_us": t_copy * 1e6,
        "copy_blocks_gbs": 2 * pairs.shape[0] * blk / t_copy / 1e9,
    }
    res["cow_parallel_sampling"] = r
    del c, k, v

    # Yi-34B-shaped long context, paged at three block sizes and contiguous
    for B in (8, 16, 32):
        w = W.yi34b_long(B=B)
        c = _paged_case(w)
        nbytes = int(c["ctx"].astype(np.int64).sum()) * 2 * w.H_kv * w.D * 2
        t, ta = _time_decode(decode_fn(c), ev)
        N_max, S_max = w.N, int(c["ctx"].max())
        req = torch.from_numpy(W.request_ids(w, N_max)).cuda()
        t_idx = torch.arange(S_max, device="cuda")
        kb = torch.empty((N_max, S_max, w.H_kv, w.D), dtype=torch.bfloat16, device="cuda")
        vb = torch.empty_like(kb)
        for si in range(w.N):
            phys = c["tab"][si, t_idx // B].long()
            kb[req[si]] = c["pool"][phys, t_idx % B, 0]
            vb[req[si]] = c["pool"][phys, t_idx % B, 1]
        out2 = torch.empty_like(c["out"])
        tc, tca = _time_decode(lambda e: pa.pa_decode_contiguous(out2, c["q"], kb, vb, req, c["cx"], S_max,
                                                                 workspace=c["ws"], dev_err=err, attend_events=e), ev)
        torch.cuda.synchronize()
        assert torch.equal(c["out"], out2), "paged and contiguous outputs differ"
        r = rates(nbytes, t, ta)
        r.update(contiguous_step_gbs=nbytes / tc / 1e9, contiguous_attend_gbs=nbytes / tca / 1e9,
                 paged_over_contiguous_step=tc / t, paged_over_contiguous_attend=tca / ta)
        res[f"yi34b_long_B{B}"] = r
        del kb, vb, c
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    return res


def measure_cache_ops(hbm: float) -> dict:
    """pa_reshape_and_cache and pa_copy_blocks timed on their own (L2 flushed before each call, CUDA events around
    the call, median), at Llama-3-8B shapes (one token = 8 KV heads x 128 x bf16 for K and for V: 4 KB; one block
    = 16 tokens: 64 KB): the cache write of one decode step (256 tokens) and of a 64K-token prefill, the block
    copy of 224 pairs (the copy-on-write step of the parallel-sampling workload) and of 8192 pairs.  GB/s count
    the bytes read plus the bytes written."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    H_kv, D, B = 8, 128, 16
    per_tok = 2 * H_kv * D * 2
    NB = 20000
    rng = np.random.default_rng(17)
    pool = torch.empty((NB, B, 2, H_kv, D), dtype=torch.bfloat16, device="cuda").normal_()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = {}
    for T in (256, 65536):
        slots = torch.from_numpy(rng.permutation(NB * B)[:T].astype(np.int64)).cuda()
        k = torch.empty((T, H_kv, D), dtype=torch.bfloat16, device="cuda").normal_()
        v = torch.empty_like(k)
        t = _time_cold(lambda: pa.pa_reshape_and_cache(k, v, pool, slots, dev_err=err))
        res[f"reshape_and_cache_{T}_tokens"] = {"us": t * 1e6, "gbs": 2 * T * per_tok / t / 1e9,
                                                "frac_of_hbm": 2 * T * per_tok / t / 1e9 / hbm}
    for n in (224, 8192):
        ids = rng.permutation(NB)[: 2 * n].astype(np.int64)
        pairs = torch.from_numpy(np.stack([ids[:n], ids[n:]], axis=1)).cuda()
        t = _time_cold(lambda: pa.pa_copy_blocks(pool, pairs, dev_err=err))
        res[f"copy_blocks_{n}_pairs"] = {"us": t * 1e6, "gbs": 2 * n * B * per_tok / t / 1e9,
                                         "frac_of_hbm": 2 * n * B * per_tok / t / 1e9 / hbm}
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    return res


def run_configs(args):
    """The other workloads, the cache ops, the prefill, the swap and the virtually contiguous KV, one JSON line each
    (the default run embeds the same figures in its line)."""
    import torch

    torch.cuda.set_device(0)
    hbm, _ = peaks()
    for name, r in measure_workloads(hbm).items():
        print(json.dumps({"measure": "decode_workload", "workload": name, "unit": "GB/s", **r}), flush=True)
    print(json.dumps({"measure": "cache_ops", **measure_cache_ops(hbm)}), flush=True)
    for r in measure_prefill():
        print(json.dumps({"measure": "pa_prefill", **r}), flush=True)
    print(json.dumps({"measure": "pa_swap_blocks", **measure_swap()}), flush=True)
    print(json.dumps({"measure": "vkv", **measure_vmm()}), flush=True)
    return 0


def measure_vmm() -> dict:
    """Virtually contiguous KV: time to map physical pages on demand (per 2 MB page, create + map + access) and
    decode over the mapped buffers, Yi-34B-shaped 8 x 32K context."""
    import torch

    import paged_kv_cache_302_gb300 as pa

    N, ctx_len, H_q, H_kv, D = 8, 32768, 56, 8, 128
    V = pa.VirtualKV(1, N, ctx_len, H_kv, D)
    reqs = [V.alloc_reqid() for _ in range(N)]
    t0 = time.perf_counter()
    V.step(reqs, [ctx_len] * N)
    t_map = time.perf_counter() - t0
    pages = sum(V.mapped_pages(r) for r in reqs) * 2        # K and V buffers
    # fill with N(0,1) through the contiguous cache write, then decode
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in reqs:
        k = torch.empty((ctx_len, H_kv, D), dtype=torch.bfloat16, device="cuda").normal_()
        pa.pa_write_contiguous(k, k, V.k_ptrs[0], V.v_ptrs[0], torch.full((ctx_len,), r, dtype=torch.int32,
                                                                            device="cuda"),
                               torch.arange(ctx_len, dtype=torch.int32, device="cuda"), N, V.S, dev_err=err)
    q = torch.empty((N, H_q, D), dtype=torch.bfloat16, device="cuda").normal_()
    out = torch.empty((N, H_q, D), device="cuda")
    req_t = torch.tensor(reqs, dtype=torch.int32, device="cuda")
    ctx_t = torch.full((N,), ctx_len, dtype=torch.int32, device="cuda")
    ws = torch.empty(pa.pa_decode_workspace_bytes(N, H_q, H_kv, D, ctx_len, 0), dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    t, ta = _time_decode(lambda e: pa.pa_decode_contiguous_raw(out, q, V.k_ptrs[0], V.v_ptrs[0], req_t, ctx_t, N, V.S,
                                                               H_kv, ctx_len, workspace=ws, dev_err=err,
                                                               attend_events=e), ev)
    assert int(err.item()) == 0
    nbytes = N * ctx_len * 2 * H_kv * D * 2
    hbm, _ = peaks()
    res = {"page_bytes": V.page_bytes, "pages_mapped": pages, "us_per_page_create_map_access": t_map / pages * 1e6,
           "decode_step_gbs": nbytes / t / 1e9, "decode_attend_gbs": nbytes / ta / 1e9,
           "decode_attend_frac_of_hbm": nbytes / ta / 1e9 / hbm,
           "tokens_per_page_per_buffer": V.page_bytes // (H_kv * D * 2)}
    V.close()
    return res


def run_vmm(args):
    import torch

    torch.cuda.set_device(0)
    print(json.dumps({"measure": "vkv", **measure_vmm()}), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.measure == "swap":
        return run_swap(args)
    if args.measure == "prefill":
        return run_prefill(args)
    if args.measure == "configs":
        return run_configs(args)
    if args.measure == "vmm":
        return run_vmm(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
