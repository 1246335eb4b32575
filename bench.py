"""Benchmark of one paged decode step on GB300.

A step = the whole hot path over one batch: copy-on-write block copies (when
the workload has any), the write of one new token per sequence and decode
attention (partition kernel + reduce kernel).  By default the write is fused
into the partition kernel (pkv_decode_step); --unfused runs pkv_write_cache
and pkv_decode_attention as separate calls.

Default line: the long-context layer (8 sequences, 32 query / 8 KV heads,
head_dim 128, bf16, context lengths uniform in [32768, 131072], split-K
partitions of 512 tokens) is the headline; the 8B-class layer (64 sequences,
lengths in [128, 2048]), the 70B-class layer (256 sequences, 64 query heads,
lognormal lengths) and the prefix-sharing step (128 sequences over one
2048-token prefix, copy-on-write tails) are measured the same way under
`per_config`.  `--config N` measures one recipe alone.  Blocks are scattered
over a pool 1.25x the need; inputs are synthetic, seeded, N(0,1).  The timed
steps are CUDA graph replays, so the device time is not paced by the host.

Metric: decode KV bytes per second (GB/s) over the step, its fraction of the
HBM peak, and sequences*layers per second.  `value` counts the algorithmic
bytes of the step (K+V history read, block-table entries, queries, outputs,
context lengths, new-token rows read and written, copy-on-write block bytes)
divided by the device time of exactly K steps.  Between timed steps the K/V
pools rotate over R device replicas whose total exceeds L2 several times.

`--kv fp8` runs the same step over FP8 (e4m3) pools with one float scale per
(block, KV head): copy-on-write, the quantising write kernel and decode
attention through the *_fp8 entry points (--fused: the write fused into the
partition kernel by pkv_decode_step_fp8, which measures no faster); bytes
count one byte per K/V element plus the scales.

`--impl reference` times the fp64 CPU oracle instead (a deliberately slow
statement of the same computation) on a bounded sample of the workload.

`--swap-gib X` times swapping X GiB of a preempted sequence's blocks out to
pinned host memory and back in (pkv_swap_blocks).

`--op write|copy` times pkv_write_cache (a bulk prefill of --op-tokens
tokens; --kv fp8: pkv_write_cache_fp8) or pkv_copy_blocks (--op-pairs pairs)
alone, in GB/s of algorithmic bytes.

`--layers N` times every layer of a decode step over an all-layer pool
[2][NB][N][16][H_kv][D], the step captured once as a CUDA graph and replayed
(eager time reported beside it).

Multi-GPU (torchrun): every rank runs the same per-GPU workload (replicas,
weak scaling); time is the max over ranks, value the sum of bytes / that time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode paged-attention KV GB/s and % of GB300 HBM peak; sequences·layers/sec"
E2E_BLOCK = 16  # end-to-end steps per captured graph
WARMUP_GRAPH_MS = 30.0  # graph replays after the eager warm-up steps, before the timed region
REPS = 5  # repetitions the timed steps are split into (rate of each, and their median, beside the total)
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------- multi-rank timing

def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the job is as slow as its slowest
    rank); identity when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, world: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time (weak scaling)."""
    return world * bytes_per_rank_step * steps / (elapsed_ms * 1e-3) / 1e9


# ----------------------------------------------------------- byte accounting

def workload_config(wl, fp8=False):
    """The keys of a JSON line's `config` that describe the workload, the same
    for the CUDA arm and the oracle's reference arm."""
    return {"workload": wl.name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "total_context_tokens": int(wl.context_lens.astype(np.int64).sum()), "num_blocks": wl.num_blocks,
            "cow_pairs": int(wl.copy_pairs.shape[0]),
            "kv_cache": "e4m3 + per-(block, KV head) f32 scales" if fp8 else wl.dtype}


def write_bytes(num_tokens, num_kv_heads, head_dim, fp8=False):
    """Algorithmic bytes of writing `num_tokens` new tokens: read their 16-bit
    K and V rows and write them into the pool (16-bit rows, or one e4m3 code
    per element plus the K and V scale read per (token, KV head)), and read
    the slot mapping."""
    T, Hkv, D = num_tokens, num_kv_heads, head_dim
    if fp8:
        return 2 * T * Hkv * D * (2 + 1) + T * Hkv * 2 * 4 + T * 4
    return 2 * T * Hkv * D * 2 * 2 + T * 4


def copy_bytes(num_pairs, block_size, num_kv_heads, head_dim, fp8=False):
    """Algorithmic bytes of `num_pairs` copy-on-write block copies: each reads
    and writes one K and one V block (16-bit, or e4m3 codes plus the block's
    K and V scales) and reads its (src, dst) pair."""
    P, B, Hkv, D = num_pairs, block_size, num_kv_heads, head_dim
    if fp8:
        return P * (2 * (B * Hkv * D + Hkv * 4) * 2 + 8)
    return P * (2 * B * Hkv * D * 2 * 2 + 8)


def step_bytes(wl, out_bytes_per_elem=4):
    """Algorithmic bytes of one step, split into the partition kernel's share and the rest."""
    S, Hq, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    L = wl.context_lens.astype(np.int64)
    kv = int(L.sum()) * Hkv * D * 2 * 2
    B = wl.block_size
    tables = int(np.sum((L + B - 1) // B)) * 4
    q = S * Hq * D * 2
    out = S * Hq * D * out_bytes_per_elem
    lens = S * 4
    attn = kv + tables + q + out + lens
    write = write_bytes(wl.slot_mapping.shape[0], Hkv, D)
    cow = copy_bytes(wl.copy_pairs.shape[0], B, Hkv, D)
    return {"attention": attn, "kv": kv, "write": write, "copy": cow, "step": attn + write + cow}


def step_bytes_fp8(wl, out_bytes_per_elem=4):
    """step_bytes over FP8 pools: one byte per K/V element plus the K and V
    scale (4 bytes each) of every (table entry, KV head) read; the write reads
    16-bit rows and a scale pair and writes codes; a copy moves codes and scales."""
    S, Hq, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    L = wl.context_lens.astype(np.int64)
    blocks = int(np.sum((L + 15) // 16))
    kv = int(L.sum()) * Hkv * D * 2 + blocks * Hkv * 2 * 4
    attn = kv + blocks * 4 + S * Hq * D * 2 + S * Hq * D * out_bytes_per_elem + S * 4
    write = write_bytes(wl.slot_mapping.shape[0], Hkv, D, fp8=True)
    cow = copy_bytes(wl.copy_pairs.shape[0], 16, Hkv, D, fp8=True)
    return {"attention": attn, "kv": kv, "write": write, "copy": cow, "step": attn + write + cow}


# -------------------------------------------------------------- clock sampler

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile

        fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- GPU arm

def unique_kv_bytes(wl, elem_bytes=2, scale_bytes=0):
    """K+V bytes of the distinct pool slots a step reads: a slot referenced by
    several sequences (a shared prefix) counts once.  With `scale_bytes`, each
    distinct block also contributes its K and V scale per KV head (FP8 pools)."""
    B = wl.block_size
    slots = []
    for s in range(wl.num_seqs):
        L = int(wl.context_lens[s])
        t = np.arange(L, dtype=np.int64)
        slots.append(wl.block_tables[s, t // B].astype(np.int64) * B + t % B)
    uniq = np.unique(np.concatenate(slots)) if slots else np.zeros(0, np.int64)
    n_blocks = int(np.unique(uniq // B).size)
    return (int(uniq.size) * wl.num_kv_heads * wl.head_dim * 2 * elem_bytes
            + n_blocks * wl.num_kv_heads * 2 * scale_bytes)


def graph_blocks(K, replicas):
    """Steps per captured graph for a timed region of exactly K steps: a
    multiple of the pool replica count (so replays continue the rotation),
    about K / REPS so the region splits into REPS repetitions.  Returns
    (steps per graph, full replays, remainder steps)."""
    b = max(replicas, (max(1, K // REPS) // replicas) * replicas)
    b = min(b, max(replicas, 64 // replicas * replicas))
    return b, K // b, K % b


def measure_workload(args, cfg, ctx, want_cpu_baseline):
    """One workload's bench line (rank 0; None on other ranks).

    Timed region A (value): exactly K steps, captured as CUDA graphs of a
    fixed number of steps and replayed back to back between two events, so
    the host's launch rate cannot pace the device.  Region B: the same steps
    launched eagerly with events around every partition-kernel launch (its
    average duration: the roofline's `achieved`).  e2e: the same step through
    the public API with every step's inputs copied up from pinned host memory
    and its output copied back."""
    import torch

    import paged_kv_cache_112_gb300 as pkv
    import pkv_inputs as P

    dist, dev, rank, world, local = ctx["dist"], ctx["dev"], ctx["rank"], ctx["world"], ctx["local"]
    wl = P.make_workload(cfg, poison=False, block_size=args.block_size)
    if args.partition_size is not None:
        ps = args.partition_size
    else:
        ps = P.fp8_partition_size(cfg) if args.kv == "fp8" else wl.partition_size
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]

    # Per-step inputs live in one device staging buffer (16-byte aligned
    # slices) mirrored by one pinned host buffer, so the end-to-end leg moves
    # them with a single host-to-device copy per step.
    step_inputs = [("q", wl.q.view(np.int16), dt), ("k_new", wl.k_new.view(np.int16), dt),
                   ("v_new", wl.v_new.view(np.int16), dt), ("bt", wl.block_tables, torch.int32),
                   ("cl", wl.context_lens, torch.int32), ("sm", wl.slot_mapping, torch.int32),
                   ("pairs", np.ascontiguousarray(wl.copy_pairs, dtype=np.int32), torch.int32)]
    offs, total = {}, 0
    for name, arr, _ in step_inputs:
        offs[name] = total
        total += (arr.nbytes + 255) // 256 * 256
    host_stage = torch.empty(max(total, 256), dtype=torch.uint8).pin_memory()
    for name, arr, _ in step_inputs:
        host_stage[offs[name]:offs[name] + arr.nbytes].copy_(
            torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
    dev_stage = host_stage.to(dev)

    def views(stage):
        """The step's inputs as views of one device staging buffer."""
        def view(name):
            arr, tdt = next((a, t) for n, a, t in step_inputs if n == name)
            t = stage[offs[name]:offs[name] + arr.nbytes].view(tdt if tdt in (torch.int32,) else torch.int16)
            t = t.view(arr.shape)
            return t.view(dt) if tdt is dt else t
        return {name: view(name) for name in ("q", "k_new", "v_new", "bt", "cl", "sm", "pairs")}

    io0 = views(dev_stage)
    pairs = io0["pairs"]
    fp8 = args.kv == "fp8"
    f8 = None
    if fp8:  # e4m3 codes + per-(block, KV head) scales; the write path quantises the new rows
        f8 = P.make_fp8_pools(wl, poison=False)
        k0, v0 = torch.from_numpy(f8.k8).to(dev), torch.from_numpy(f8.v8).to(dev)
        ks0, vs0 = torch.from_numpy(f8.k_scale).to(dev), torch.from_numpy(f8.v_scale).to(dev)
    else:
        k0 = torch.from_numpy(wl.k_pool.view(np.int16)).to(dev).view(dt)
        v0 = torch.from_numpy(wl.v_pool.view(np.int16)).to(dev).view(dt)
        ks0 = vs0 = None
    io0["out"] = torch.empty(io0["q"].shape, dtype=torch.float32, device=dev)
    ws_bytes = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, wl.max_context_len, ps)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = 2 * k0.numel() * k0.element_size()
    replicas = args.replicas or max(1, math.ceil(4 * l2 / pool_bytes))
    clone = lambda t: None if t is None else t.clone()
    pools = [(k0, v0, ks0, vs0)] + [(k0.clone(), v0.clone(), clone(ks0), clone(vs0)) for _ in range(replicas - 1)]
    max_len = wl.max_context_len
    separate_write = (not args.fused) if fp8 else args.unfused
    n_launch = (1 if separate_write else 0) + 1 + (1 if ws_bytes else 0) + (1 if pairs.shape[0] else 0)

    def step_fp8(i, ev, io):
        kp, vp, ksp, vsp = pools[i % replicas]
        q, k_new, v_new, bt, cl, sm, out = (io[k] for k in ("q", "k_new", "v_new", "bt", "cl", "sm", "out"))
        if io["pairs"].shape[0]:
            pkv.copy_blocks_fp8(kp, vp, ksp, vsp, io["pairs"], status=status)
        if not args.fused:
            pkv.write_cache_fp8(k_new, v_new, kp, vp, ksp, vsp, sm, status=status)
        if ev is not None:
            ev[0].record()
        if not args.fused:
            pkv.decode_partitions_fp8(out, q, kp, vp, ksp, vsp, bt, cl, wl.scale, partition_size=ps,
                                      max_context_len=max_len, workspace=ws, status=status)
        else:  # the quantising write of the new token fused into the partition kernel
            pkv.decode_step_partitions_fp8(out, q, k_new, v_new, kp, vp, ksp, vsp, bt, cl, sm, wl.scale,
                                           partition_size=ps, max_context_len=max_len, workspace=ws,
                                           status=status)
        if ev is not None:
            ev[1].record()
        if ws is not None:
            pkv.decode_reduce(out, cl, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                              head_dim=wl.head_dim, partition_size=ps, max_context_len=max_len, workspace=ws,
                              status=status)

    def step(i, ev=None, io=io0):
        if fp8:
            return step_fp8(i, ev, io)
        kp, vp = pools[i % replicas][:2]
        q, k_new, v_new, bt, cl, sm, out = (io[k] for k in ("q", "k_new", "v_new", "bt", "cl", "sm", "out"))
        if io["pairs"].shape[0]:
            pkv.copy_blocks(kp, vp, io["pairs"], status=status)
        if not args.unfused:  # the new token's write fused into the partition kernel
            if ev is not None:
                ev[0].record()
            pkv.decode_step_partitions(out, q, k_new, v_new, kp, vp, bt, cl, sm, wl.scale, partition_size=ps,
                                       max_context_len=max_len, workspace=ws, status=status)
        else:
            pkv.write_cache(k_new, v_new, kp, vp, sm, status=status)
            if ev is not None:
                ev[0].record()
            pkv.decode_partitions(out, q, kp, vp, bt, cl, wl.scale, partition_size=ps, max_context_len=max_len,
                                  workspace=ws, status=status)
        if ev is not None:
            ev[1].record()
        if ws is not None:
            pkv.decode_reduce(out, cl, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                              head_dim=wl.head_dim, partition_size=ps, max_context_len=max_len, workspace=ws,
                              status=status)

    nb = step_bytes_fp8(wl) if fp8 else step_bytes(wl)
    K, W = args.steps, args.warmup

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def capture(n):
        """A CUDA graph of steps 0..n-1 (pool replica i % replicas for step i)."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(n):
                step(i)  # eager run of the same work on the capture stream first
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(g):
            for i in range(n):
                step(i)
        return g

    def graph_warmup(g):
        """Replays g until at least WARMUP_GRAPH_MS of replays have run (one
        at least); returns the number of replays."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        more = max(0, math.ceil(WARMUP_GRAPH_MS / max(e0.elapsed_time(e1), 1e-3)) - 1)
        for _ in range(more):
            g.replay()
        torch.cuda.synchronize()
        return 1 + more

    def timed_launches(n_steps, per_graph):
        """Durations (ms) of the partition-kernel launches of steps 0..n_steps-1
        and how they were timed."""
        try:
            evs = [(torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True)) for _ in range(per_graph)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(per_graph):
                    step(i, evs[i])
        except (TypeError, RuntimeError):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_steps)]
            barrier()
            for i in range(n_steps):
                step(i, evs[i])
            barrier()
            return [x.elapsed_time(y) for x, y in evs], "eager launches, events around each"
        g.replay()  # warm-up replay, not timed
        barrier()
        out = []
        while len(out) < n_steps:
            g.replay()
            torch.cuda.synchronize()
            out += [x.elapsed_time(y) for x, y in evs][:n_steps - len(out)]
        del g
        if not all(t > 0 for t in out):
            raise RuntimeError("non-positive kernel duration from graph-recorded events")
        return out, f"CUDA graph replays of {per_graph} steps, event nodes around each launch"

    b, n_full, rem = graph_blocks(K, replicas)
    g_full = capture(b)
    g_rem = capture(rem) if rem else None
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()  # sampling starts before the warm-up: no idle gap before the timed region
    for i in range(W):
        step(i)
    warm_replays = graph_warmup(g_full)

    # Timed region A: exactly K steps (n_full replays of b steps, then the
    # remainder), nothing else on the stream.  Events between replays split it
    # into repetitions.
    groups = min(n_full, REPS)
    bounds = [n_full * r // groups for r in range(groups + 1)] if groups else [0]
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(len(bounds) + (1 if g_rem else 0))]
    barrier()
    # One untimed replay is already running when the first event is recorded,
    # so the timed replays queue behind it: the region starts on a busy GPU,
    # as every step of a serving loop does, not with a launch from idle.
    g_full.replay()
    marks[0].record()
    for r in range(groups):
        for _ in range(bounds[r + 1] - bounds[r]):
            g_full.replay()
        marks[r + 1].record()
    if g_rem is not None:
        g_rem.replay()
        marks[-1].record()
    barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = marks[0].elapsed_time(marks[-1])
    rep_gbs = [round(nb["step"] * b * (bounds[r + 1] - bounds[r]) / (marks[r].elapsed_time(marks[r + 1]) * 1e-3)
                     / 1e9, 2) for r in range(groups)]
    # Timed region B: the same K steps with CUDA events around every launch of
    # the partition kernel (its average launch duration; the events stop
    # consecutive kernels from overlapping, so region A alone gives the step
    # time).  The events are recorded by nodes of a captured graph where torch
    # can capture them, so the host's launch rate does not stretch the short
    # launches; otherwise the steps are launched eagerly.
    kern_ms, kern_timing = timed_launches(K, b)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")

    # End to end through the public API: every step uploads its inputs from pinned host memory
    # (one copy) and reads its output back, double-buffered as a serving loop runs it: step i's
    # inputs go up on one copy stream while step i-1 computes, and step i's output comes down on
    # another while step i+1 computes.  A block of E2E_BLOCK such steps is captured once as a
    # CUDA graph and replayed, so the host's per-call cost does not pace the loop.
    up_stream, down_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dev_stages = [dev_stage, torch.empty_like(dev_stage)]
    ios = [io0, views(dev_stages[1])]
    ios[1]["out"] = torch.empty_like(io0["out"])
    host_outs = [torch.empty(io0["out"].shape, dtype=io0["out"].dtype).pin_memory() for _ in range(2)]
    h2d = int(total)
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    block = E2E_BLOCK
    Ke = max(block, min(K, args.e2e_steps) // block * block)

    def e2e_block(n):
        comp = torch.cuda.current_stream()
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        down = [torch.cuda.Event() for _ in range(2)]
        up_stream.wait_stream(comp)
        down_stream.wait_stream(comp)
        for i in range(n):
            bb = i % 2
            if i >= 2:
                up_stream.wait_event(done[bb])    # step i-2 has finished reading this staging buffer
                comp.wait_event(down[bb])         # and its output has been read back
            with torch.cuda.stream(up_stream):
                dev_stages[bb].copy_(host_stage, non_blocking=True)
                up[bb].record(up_stream)
            comp.wait_event(up[bb])
            step(i, io=ios[bb])
            done[bb].record(comp)
            down_stream.wait_event(done[bb])
            with torch.cuda.stream(down_stream):
                host_outs[bb].copy_(ios[bb]["out"], non_blocking=True)
                down[bb].record(down_stream)
        comp.wait_stream(up_stream)
        comp.wait_stream(down_stream)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        e2e_block(block)  # eager warm-up of the same work
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        e2e_block(block)
    for _ in range(2):
        graph.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph.replay()  # untimed, in flight when the region starts (as in region A)
    e0.record()
    for _ in range(Ke // block):
        graph.replay()
    e1.record()
    barrier()
    e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the end-to-end steps")
    e2e = {"value": round(job_gbs(nb["step"], world, Ke, e_ms), 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": Ke,
           "ms_per_step": round(e_ms / Ke, 5),
           "overlap": f"double-buffered (inputs up / outputs down on two copy streams beside the step), "
                      f"{block} steps per CUDA graph replay"}
    del graph, g_full, g_rem
    if rank != 0:
        return None

    peak, peak_kind = _peaks()
    ms = elapsed_ms / K
    value = job_gbs(nb["step"], world, K, elapsed_ms)
    kern_avg_ms = statistics.mean(kern_ms)
    kernel_name = partition_kernel_name(wl.num_seqs, wl.num_kv_heads, ps, args.block_size, fp8, bool(args.fused),
                                        torch.cuda.get_device_properties(dev).multi_processor_count)
    traffic = _recorded_traffic(cfg, kernel_name)
    achieved = nb["attention"] / (kern_avg_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 2), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "bytes_per_launch": nb["attention"], "avg_launch_ms": round(kern_avg_ms, 5),
                "launch_timing": kern_timing}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"e4m3 KV, {wl.dtype} q" if fp8 else wl.dtype, "data": "synthetic",
        "config": {**workload_config(wl, fp8), "partition_size": ps, "max_context_len": max_len,
                   "out_dtype": "f32",
                   "entry": (("pkv_decode_step_fp8" if args.fused else
                              "pkv_write_cache_fp8 + pkv_decode_attention_fp8") if fp8 else
                             "pkv_write_cache + pkv_decode_attention" if args.unfused else "pkv_decode_step"),
                   "l2": f"inputs larger than L2: {replicas} pool replicas of {pool_bytes / 1e6:.0f} MB rotated "
                         f"(L2 {l2 / 1e6:.0f} MB)", "parallelism": f"replicas x{world}",
                   "timed_region": f"{n_full} CUDA graph replays of {b} steps" +
                                   (f" + one of {rem}" if rem else "") + " between two events",
                   "warmup_graph_replays": warm_replays + 1},
        "pct_of_hbm_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_hbm_measured": round(100 * value / world / peak, 2),
        "seq_layers_per_s": round(world * wl.num_seqs / (ms * 1e-3), 1),
        "repetitions": {"n": len(rep_gbs), "gbs_rank0": rep_gbs,
                        "median_gbs_rank0": statistics.median(rep_gbs) if rep_gbs else None,
                        "note": "the K timed steps in equal runs of graph replays, one GPU's rate each; "
                                "value is their total"},
        "kv_bytes_per_step": nb["kv"], "step_bytes": nb["step"],
        "roofline": roofline,
        "gpu_launches": n_launch * K,
        "clocks": clocks,
        "e2e": e2e,
    }
    if wl.copy_pairs.shape[0]:
        # A shared prefix is read by every sequence but sits in HBM once (and
        # stays in L2): the HBM roofline counts each distinct slot once.
        ukv = unique_kv_bytes(wl, 1, 4) if fp8 else unique_kv_bytes(wl)
        uniq = ukv + (nb["attention"] - nb["kv"])
        line["unique_bytes"] = {
            "note": "the logical bytes above count a shared prefix once per sequence; these count each distinct "
                    "pool slot once (the HBM roofline of this workload)",
            "attention_bytes_per_launch": uniq, "kv_bytes_per_step": ukv,
            "step_gbs": round(job_gbs(uniq + nb["write"] + nb["copy"], world, K, elapsed_ms), 2)}
        roofline["achieved_logical"] = roofline["achieved"]
        roofline["frac_logical"] = roofline["frac"]
        roofline["achieved"] = round(uniq / (kern_avg_ms * 1e-3) / 1e9, 2)
        roofline["frac"] = round(roofline["achieved"] / peak, 4)
        roofline["bytes_per_launch"] = uniq
        roofline["bytes_counted"] = "unique (each distinct pool slot once)"
    if want_cpu_baseline:  # the oracle's host-core baseline: one GPU runs only
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, f8)
    del pools, k0, v0, ws, dev_stage, dev_stages, ios, io0
    return line


# Workloads of the default line: the largest single-GPU configuration (long
# context, split-K) is the headline; the 8B- and 70B-class layers and the
# prefix-sharing step ride along under per_config.
HEADLINE_CONFIG = 4
PER_CONFIG = (2, 3, 5)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_112_gb300 as pkv

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    pkv.load()
    ctx = {"dist": dist, "dev": dev, "rank": rank, "world": world, "local": local}
    cpu_on = not args.no_cpu_baseline and world == 1
    if args.config is not None:
        line = measure_workload(args, args.config, ctx, cpu_on)
    else:
        line = measure_workload(args, HEADLINE_CONFIG, ctx, cpu_on)
        per = {}
        for cfg in PER_CONFIG:
            torch.cuda.empty_cache()
            per[str(cfg)] = measure_workload(args, cfg, ctx, False)
        if line is not None:
            keep = ("value", "unit", "ms_per_step", "pct_of_hbm_nominal_8tbs", "pct_of_hbm_measured",
                    "seq_layers_per_s", "repetitions", "roofline", "unique_bytes", "clocks", "e2e", "config",
                    "step_bytes", "gpu_launches")
            line["per_config"] = {k: {f: v[f] for f in keep if f in v} for k, v in per.items()}
            line["gpu_launches"] += sum(v["gpu_launches"] for v in per.values())
            line["config"]["per_config_workloads"] = [per[str(c)]["config"]["workload"] for c in PER_CONFIG]
    if world > 1:
        dist.destroy_process_group()
    return line


def run_layers(args):
    """Every layer of one decode step (--layers N) over an all-layer pool
    [2][NB][N][16][H_kv][D] ("KV Cache & PagedAttention" section 4), the
    step captured once as a CUDA graph and replayed.  Copy-on-write moves
    whole blocks (all layers); each layer runs the fused write + attention
    and the reduce on its view of the pool.  Values are seeded N(0,1) drawn
    on the device; tables, lengths and slots are the recipe's."""
    import torch
    import torch.distributed as dist

    import paged_kv_cache_112_gb300 as pkv
    import pkv_inputs as P

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    pkv.load()
    wl = P.make_workload(args.config, poison=False)
    ps = wl.partition_size if args.partition_size is None else args.partition_size
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
    n_layers = args.layers
    S, Hq, Hkv, D, NB = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.num_blocks
    gen = torch.Generator(device=dev).manual_seed(7919 * args.config + n_layers)
    pool = torch.empty((2, NB, n_layers, 16, Hkv, D), dtype=dt, device=dev)
    for kv in range(2):
        for layer in range(n_layers):
            pool[kv, :, layer].normal_(generator=gen)
    q = torch.randn((n_layers, S, Hq, D), generator=gen, device=dev).to(dt)
    k_new = torch.randn((n_layers, S, Hkv, D), generator=gen, device=dev).to(dt)
    v_new = torch.randn((n_layers, S, Hkv, D), generator=gen, device=dev).to(dt)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cl = torch.from_numpy(wl.context_lens).to(dev)
    sm = torch.from_numpy(wl.slot_mapping).to(dev)
    pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, dtype=np.int32)).to(dev)
    out = torch.empty((n_layers, S, Hq, D), dtype=torch.float32, device=dev)
    max_len = wl.max_context_len
    ws_bytes = pkv.decode_workspace_bytes(S, Hq, D, max_len, ps)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(evs=None):
        if pairs.shape[0]:
            pkv.copy_blocks(pool[0], pool[1], pairs, status=status)
        for layer in range(n_layers):
            kp, vp = pool[0, :, layer], pool[1, :, layer]
            if evs is not None:
                evs[layer][0].record()
            pkv.decode_step_partitions(out[layer], q[layer], k_new[layer], v_new[layer], kp, vp, bt, cl, sm, wl.scale,
                                       partition_size=ps, max_context_len=max_len, workspace=ws, status=status)
            if evs is not None:
                evs[layer][1].record()
            if ws is not None:
                pkv.decode_reduce(out[layer], cl, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, partition_size=ps,
                                  max_context_len=max_len, workspace=ws, status=status)

    K, W = args.steps, args.warmup

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def timed(fn, k):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        a.record()
        for _ in range(k):
            fn()
        b.record()
        barrier()
        return a.elapsed_time(b)

    for _ in range(W):
        step()
    eager_ms = timed(step, K)
    # the partition kernels' own durations (events between launches stop PDL overlap; eager)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_layers)]
    kern = []
    for _ in range(min(K, 20)):
        step(evs)
        torch.cuda.synchronize()
        kern += [x.elapsed_time(y) for x, y in evs]
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        step()
    for _ in range(W):
        graph.replay()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    graph_ms = timed(graph.replay, K)
    clocks = sampler.stop() if sampler else None
    graph_ms = max_over_ranks(graph_ms, dev)
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")

    # end to end: every layer's queries and new rows from pinned host memory, outputs back, each step
    h_q, h_k, h_v = q.cpu().pin_memory(), k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        q.copy_(h_q, non_blocking=True)
        k_new.copy_(h_k, non_blocking=True)
        v_new.copy_(h_v, non_blocking=True)
        graph.replay()
        h_out.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    Ke = max(1, min(K, args.e2e_steps))
    e_ms = max_over_ranks(timed(e2e_step, Ke), dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    peak, peak_kind = _peaks()
    nb = step_bytes(wl)
    per_step = n_layers * nb["step"]
    value = job_gbs(per_step, world, K, graph_ms)
    kern_avg_ms = statistics.mean(kern)
    achieved = nb["attention"] / (kern_avg_ms * 1e-3) / 1e9
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(graph_ms / K, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "layers": n_layers, "pool": "all-layer [2, NB, layers, 16, H_kv, D]",
                   "graph": "one CUDA graph per step, replayed", "num_seqs": S, "num_q_heads": Hq,
                   "num_kv_heads": Hkv, "head_dim": D, "partition_size": ps, "max_context_len": max_len,
                   "cow_pairs": int(wl.copy_pairs.shape[0]), "entry": "pkv_copy_blocks + pkv_decode_step per layer",
                   "l2": f"inputs larger than L2: {n_layers} layers x {2 * pool[0, :, 0].numel() * 2 / 1e6:.0f} MB",
                   "parallelism": f"replicas x{world}"},
        "pct_of_hbm_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_hbm_measured": round(100 * value / world / peak, 2),
        "seq_layers_per_s": round(world * S * n_layers / (graph_ms / K * 1e-3), 1),
        "eager_ms_per_step": round(eager_ms / K, 5), "graph_ms_per_step": round(graph_ms / K, 5),
        "step_bytes": per_step,
        "roofline": {"bound": "hbm",
                     "kernel": partition_kernel_name(S, Hkv, ps, 16, False, True,
                                                     torch.cuda.get_device_properties(dev).multi_processor_count),
                     "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "bytes_per_launch": nb["attention"], "avg_launch_ms": round(kern_avg_ms, 5)},
        "gpu_launches": ((1 if pairs.shape[0] else 0) + n_layers * (1 + (1 if ws_bytes else 0))) * K,
        "clocks": clocks,
        "e2e": {"value": round(job_gbs(per_step, world, Ke, e_ms), 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(h_out.numel() * h_out.element_size()), "steps": Ke,
                "ms_per_step": round(e_ms / Ke, 5)},
    }
    if world > 1:
        dist.destroy_process_group()
    return line


def run_swap(args):
    """Swap out / in of a preempted victim's blocks (--swap-gib X): the pages'
    example of 1.25 GiB of an 8B-class model's KV ("PagedAttention internals"
    section 05: 32 layers, 8 KV heads, head_dim 128, fp16, 16-token blocks of
    2 MiB over all layers, ~50 ms each way over PCIe 4.0 at ~25 GB/s).  The
    victim's blocks are scattered over an all-layer device pool; the host
    pool is pinned memory, reached by the kernel over NVLink-C2C."""
    import torch

    import paged_kv_cache_112_gb300 as pkv

    _, _, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load()
    layers, hkv, d = 32, 8, 128
    block_bytes = 2 * layers * 16 * hkv * d * 2  # K + V, all layers
    n = max(1, int(round(args.swap_gib * 2 ** 30 / block_bytes)))
    nb_dev = max(4 * n, 1024)
    gen = torch.Generator(device=dev).manual_seed(1250)
    pool = torch.empty((2, nb_dev, layers, 16, hkv, d), dtype=torch.float16, device=dev)
    pool.normal_(generator=gen)
    host = torch.empty((2, n, layers, 16, hkv, d), dtype=torch.float16).pin_memory()
    rng = np.random.default_rng(1250)
    victim = rng.permutation(nb_dev)[:n].astype(np.int32)
    target = rng.permutation(nb_dev)[:n].astype(np.int32)
    out_pairs = torch.from_numpy(np.stack([victim, np.arange(n, dtype=np.int32)], 1)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), target], 1)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def swap_out():
        pkv.swap_blocks(host[0], host[1], pool[0], pool[1], out_pairs, status=status)

    def swap_in():
        pkv.swap_blocks(pool[0], pool[1], host[0], host[1], in_pairs, status=status)

    res = {}
    for name, fn in (("out", swap_out), ("in", swap_in)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        res[name] = {"ms": round(ms, 4), "GB/s": round(n * block_bytes / (ms * 1e-3) / 1e9, 2)}
    # the link's bulk rate for comparison: one contiguous copy of the same bytes each way (copy engine)
    flat_dev = pool.view(-1)[: host.numel()]
    flat_host = host.view(-1)
    for name, fn in (("bulk_d2h", lambda: flat_host.copy_(flat_dev, non_blocking=True)),
                     ("bulk_h2d", lambda: flat_dev.copy_(flat_host, non_blocking=True))):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        res[name] = {"ms": round(ms, 4), "GB/s": round(n * block_bytes / (ms * 1e-3) / 1e9, 2)}
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    moved = n * block_bytes
    value = 2 * moved / ((res["out"]["ms"] + res["in"]["ms"]) * 1e-3) / 1e9
    return {"metric": "swap out + in of a preempted sequence's blocks, GB/s (device <-> pinned host)",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(res["out"]["ms"] + res["in"]["ms"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": "8B-class all-layer blocks (32 layers, 8 KV heads, head_dim 128, fp16), "
                                   f"{n} blocks of 2 MiB scattered over {nb_dev}",
                       "bytes_each_way": moved, "entry": "pkv_swap_blocks"},
            "swap_out": res["out"], "swap_in": res["in"],
            "contiguous_copy_engine": {"d2h": res["bulk_d2h"], "h2d": res["bulk_h2d"]},
            "pages_figure": "1.25 GiB over PCIe 4.0 x16 at ~25 GB/s: ~50 ms each way"}


def cache_op_sets(op, n, block_size, sets, rng):
    """Disjoint inputs for `sets` calls of write_cache or copy_blocks.
    write: n tokens per set filling whole blocks in order, the blocks a random
    permutation of the pool: slots int32 [sets, n].  copy: n (src, dst) pairs
    per set, every src and dst block distinct across all sets: pairs int32
    [sets, n, 2].  Returns (array, blocks the pool needs)."""
    B = block_size
    if op == "write":
        per = -(-n // B)
        nb = sets * per
        perm = rng.permutation(nb).astype(np.int64)
        t = np.arange(n, dtype=np.int64)
        slots = np.stack([perm[r * per + t // B] * B + t % B for r in range(sets)])
        return slots.astype(np.int32), nb
    nb = sets * 2 * n
    perm = rng.permutation(nb).astype(np.int32).reshape(sets, 2, n)
    return np.ascontiguousarray(np.stack([perm[:, 0], perm[:, 1]], axis=2)), nb


def run_cache_op(args):
    """pkv_write_cache or pkv_copy_blocks timed alone (--op write | copy), on
    the recipe's row shape (H_kv, head_dim, dtype; --kv fp8 for the FP8 entry
    points): a bulk write of --op-tokens new tokens (a prefill fills whole
    blocks, scattered over the pool; --op-tokens = the batch size gives the
    decode step's write), or --op-pairs copy-on-write block copies.  GB/s of
    algorithmic bytes (write_bytes / copy_bytes).  Call i works on input set
    i mod R, the R sets disjoint in inputs and blocks and together larger
    than 3x L2."""
    import torch

    import paged_kv_cache_112_gb300 as pkv
    import pkv_inputs as P

    _, _, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load()
    spec = P.CONFIGS[args.config]
    Hkv, D, dtype = spec["num_kv_heads"], spec["head_dim"], spec["dtype"]
    fp8 = args.kv == "fp8"
    B = args.block_size
    n = args.op_tokens if args.op == "write" else args.op_pairs
    if n <= 0:
        raise SystemExit("--op-tokens / --op-pairs must be positive")
    per_call = write_bytes(n, Hkv, D, fp8) if args.op == "write" else copy_bytes(n, B, Hkv, D, fp8)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    R = max(2, min(4096, math.ceil(3 * l2 / per_call)))
    sets, NB = cache_op_sets(args.op, n, B, R, np.random.default_rng(args.config))
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    gen = torch.Generator(device=dev).manual_seed(args.config)
    shape = (NB, B, Hkv, D)
    if fp8:
        k_pool = torch.randint(0, 0x7F, shape, generator=gen, dtype=torch.uint8, device=dev)
        v_pool = torch.randint(0, 0x7F, shape, generator=gen, dtype=torch.uint8, device=dev)
        k_scale = torch.rand((NB, Hkv), generator=gen, device=dev) + 0.5
        v_scale = torch.rand((NB, Hkv), generator=gen, device=dev) + 0.5
    else:
        k_pool = torch.randn(shape, generator=gen, device=dev).to(tdt)
        v_pool = torch.randn(shape, generator=gen, device=dev).to(tdt)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.op == "write":
        k_new = torch.randn((R, n, Hkv, D), generator=gen, device=dev).to(tdt)
        v_new = torch.randn((R, n, Hkv, D), generator=gen, device=dev).to(tdt)
        slots = torch.from_numpy(sets).to(dev)

        def call(i):
            r = i % R
            if fp8:
                pkv.write_cache_fp8(k_new[r], v_new[r], k_pool, v_pool, k_scale, v_scale, slots[r], status=status)
            else:
                pkv.write_cache(k_new[r], v_new[r], k_pool, v_pool, slots[r], status=status)
        entry = "pkv_write_cache_fp8" if fp8 else "pkv_write_cache"
        kernel = "write_cache_fp8_kernel" if fp8 else "write_cache_kernel"
        what = f"{n} new tokens filling whole {B}-token blocks scattered over a {NB}-block pool"
    else:
        pairs = torch.from_numpy(sets).to(dev)

        def call(i):
            r = i % R
            if fp8:
                pkv.copy_blocks_fp8(k_pool, v_pool, k_scale, v_scale, pairs[r], status=status)
            else:
                pkv.copy_blocks(k_pool, v_pool, pairs[r], status=status)
        entry = "pkv_copy_blocks_fp8" if fp8 else "pkv_copy_blocks"
        kernel = "copy_blocks_kernel"
        what = f"{n} copy-on-write pairs of {B}-token blocks, distinct blocks of a {NB}-block pool"
    K, W = args.steps, args.warmup
    for i in range(W):
        call(i)
    torch.cuda.synchronize()

    # The K timed calls are replays of captured graphs (calls 0..G-1, G <= R,
    # so a replay walks the disjoint input sets once), so the host's launch
    # rate does not pace short calls.
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                call(i)
        return g

    G = min(K, R)
    g_full = capture(G)
    g_rem = capture(K % G) if K % G else None
    sampler = ClockSampler(local)
    sampler.start()
    g_full.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g_full.replay()  # untimed, in flight when the region starts
    a.record()
    for _ in range(K // G):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    b.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    del g_full, g_rem
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = a.elapsed_time(b) / K
    gbs = per_call / (ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    return {"metric": f"{entry} alone, GB/s of algorithmic bytes", "value": round(gbs, 2), "unit": "GB/s",
            "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": f"e4m3 KV, {dtype} new rows" if fp8 else dtype, "data": "synthetic",
            "config": {"workload": f"{spec['name']}: {what}", "num_kv_heads": Hkv, "head_dim": D,
                       "block_size": B, "entry": entry, "bytes_per_call": per_call,
                       "l2": f"inputs larger than L2: {R} disjoint input sets of {per_call / 1e6:.2f} MB rotated "
                             f"(L2 {l2 / 1e6:.0f} MB)",
                       "timed_region": f"{K // G} CUDA graph replays of {G} calls" +
                                       (f" + one of {K % G}" if K % G else "") + " between two events"},
            "us_per_call": round(ms * 1e3, 3),
            "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 2), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None},
            "clocks": clocks, "gpu_launches": K}


def kernel_source_hash(paths) -> str:
    """First 16 hex digits of a sha256 over the given sources with comments
    and whitespace removed: any change to the code changes it, a change to a
    comment does not."""
    import hashlib
    import re

    h = hashlib.sha256()
    for p in paths:
        with open(p, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


def partition_kernel_name(num_seqs, num_kv_heads, partition_size, block_size, fp8, fused, sm_count):
    """The first kernel of a decode call, by the library's rule.  FP8 pools:
    write-then-attend over fixed partitions with H_kv % 4 == 0 runs the
    head-group grid.  16-bit pools: blocks of >= 16 tokens, an even H_kv and
    sequences x KV heads within one wave of the partition kernel's warp slots
    (six two-warp CTAs per SM) run the head-group kernel (2 or 4 heads a CTA)."""
    balanced = partition_size == -1
    if fp8:
        if balanced:
            return "decode_balanced_fp8_kernel"
        return "decode_partitions_fp8_hg_kernel" if not fused and num_kv_heads % 4 == 0 else \
            "decode_partitions_fp8_kernel"
    if balanced:
        return "decode_balanced_kernel"
    hg = block_size >= 16 and num_kv_heads % 2 == 0 and num_kv_heads * num_seqs <= 12 * sm_count
    return "decode_partitions_hg_kernel" if hg else "decode_partitions_kernel"


# short names of the workload recipes, as the profile summaries are named
WORKLOAD_SLUGS = {1: "tiny", 2: "8b_class", 3: "70b_class", 4: "long_context", 5: "prefix_sharing"}


def _recorded_traffic(cfg, kernel):
    """DRAM bytes per launch of the partition kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""

    sources = {"decode_partitions_kernel": ("decode_partitions", "pkv_decode.cu"),
               "decode_partitions_hg_kernel": ("decode_partitions_hg", "pkv_decode_hg.cu"),
               "decode_partitions_fp8_kernel": ("decode_partitions_fp8", "pkv_decode_fp8.cu"),
               "decode_partitions_fp8_hg_kernel": ("decode_partitions_fp8", "pkv_decode_fp8.cu")}
    if kernel not in sources:
        return None
    stem, src = sources[kernel]
    summ = os.path.join(ROOT, "profiles", f"{stem}_{WORKLOAD_SLUGS[cfg]}_traffic.txt")
    srcs = [os.path.join(ROOT, "paged_kv_cache_112_gb300", "csrc", f) for f in (src, "pkv_device.cuh")]
    if not os.path.exists(summ):
        return None
    vals = {}
    with open(summ) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash(srcs):
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------ CPU oracle arm

def _oracle_pass(wl, seqs, pools, threads):
    import oracle

    rows = [(s, h) for s in seqs for h in range(wl.num_q_heads)]
    if len(pools) == 4:  # FP8 codes and scales
        oracle.decode_attention_fp8(wl.q, *pools, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, rows=rows,
                                    num_threads=threads)
    else:
        oracle.decode_attention(wl.q, *pools, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, rows=rows,
                                num_threads=threads)


def _sample_bytes(wl, seqs, elem_bytes=2):
    L = wl.context_lens.astype(np.int64)[list(seqs)]
    return int(L.sum()) * wl.num_kv_heads * wl.head_dim * 2 * elem_bytes


def cpu_baseline(wl, seconds, fp8_pools=None):
    """The oracle, as it stands, on whole sequences of the workload, repeated
    for about `seconds` of wall time on all host cores (over FP8 pools when
    given)."""
    import oracle

    threads = oracle.hardware_threads()
    if fp8_pools is not None:
        pools = oracle.apply_step_fp8(wl, fp8_pools, attention=False)[:4]
        eb = 1
    else:
        pools = oracle.apply_step(wl, attention=False)[:2]
        eb = 2
    order = list(range(wl.num_seqs))
    t0 = time.perf_counter()
    _oracle_pass(wl, order[:1], pools, threads)
    per_seq = max(time.perf_counter() - t0, 1e-4)
    n = max(1, min(wl.num_seqs, int(seconds / 3 / per_seq)))
    seqs = order[:n]
    done_bytes, t0, reps = 0, time.perf_counter(), 0
    while True:
        _oracle_pass(wl, seqs, pools, threads)
        done_bytes += _sample_bytes(wl, seqs, eb)
        reps += 1
        if time.perf_counter() - t0 >= seconds or reps >= 1000:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle{' (FP8 pools)' if eb == 1 else ''} over the first {n} of {wl.num_seqs} "
                      f"sequences (all query heads), "
                      f"{reps} passes, {dt:.1f} s wall"}


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return None
    import oracle
    import pkv_inputs as P

    wl = P.make_workload(args.config, poison=False, block_size=args.block_size)
    threads = oracle.hardware_threads()
    fp8 = args.kv == "fp8"
    if fp8:
        pools = oracle.apply_step_fp8(wl, P.make_fp8_pools(wl, poison=False), attention=False)[:4]
        attend = oracle.decode_attention_fp8
    else:
        pools = oracle.apply_step(wl, attention=False)[:2]
        attend = oracle.decode_attention
    K, W = args.steps, args.warmup
    # size one step's sample so that W + K steps take about args.ref_seconds
    rows_all = [(s, h) for s in range(wl.num_seqs) for h in range(wl.num_q_heads)]
    t0 = time.perf_counter()
    attend(wl.q, *pools, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, rows=rows_all[: wl.num_q_heads],
           num_threads=threads)
    per_row = max((time.perf_counter() - t0) / wl.num_q_heads, 1e-6)
    budget = args.ref_seconds / max(1, K + W)
    n_rows = int(max(1, min(len(rows_all), budget / per_row)))
    rows = rows_all[:n_rows]
    G = wl.num_q_heads // wl.num_kv_heads
    L = wl.context_lens.astype(np.int64)
    # KV bytes the sampled rows account for (a row reads 1/G of its KV head's bytes)
    eb = 1 if fp8 else 2
    sample_bytes = sum(int(L[s]) * wl.head_dim * 2 * eb for s, _ in rows) / G

    def one():
        attend(wl.q, *pools, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, rows=rows, num_threads=threads)

    for _ in range(W):
        one()
    t0 = time.perf_counter()
    for _ in range(K):
        one()
    dt = time.perf_counter() - t0
    ms = dt / K * 1e3
    value = sample_bytes / (ms * 1e-3) / 1e9
    sample = (f"fp64 oracle{' (FP8 pools)' if fp8 else ''}, {n_rows} (sequence, query head) rows of "
              f"{len(rows_all)} per step, {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**workload_config(wl, fp8), "entry": "oracle.decode_attention" +
                       ("_fp8" if fp8 else ""), "sample_rows": n_rows},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="one workload recipe; default: the long-context layer (4) as the headline with the 8B-class "
                         "(2), 70B-class (3) and prefix-sharing (5) layers under per_config")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--partition-size", type=int, default=None)
    ap.add_argument("--replicas", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="run write_cache and decode attention as separate calls instead of pkv_decode_step")
    ap.add_argument("--block-size", type=int, default=16, choices=[8, 16, 32, 64],
                    help="tokens per KV block (16-bit pools; the recipes use 16)")
    ap.add_argument("--swap-gib", type=float, default=0.0,
                    help="time swapping this many GiB of a victim's blocks out to pinned host memory and back")
    ap.add_argument("--layers", type=int, default=0,
                    help="time every layer of a decode step (this many) over an all-layer pool, as a CUDA graph")
    ap.add_argument("--fused", action="store_true",
                    help="with --kv fp8: fuse the quantising write into the partition kernel (pkv_decode_step_fp8)")
    ap.add_argument("--op", default=None, choices=["write", "copy"],
                    help="time pkv_write_cache (--op-tokens new tokens) or pkv_copy_blocks (--op-pairs pairs) alone")
    ap.add_argument("--op-tokens", type=int, default=65536,
                    help="with --op write: tokens per call (default: a 64K-token bulk prefill)")
    ap.add_argument("--op-pairs", type=int, default=128,
                    help="with --op copy: copy-on-write pairs per call (default 128, about the prefix-sharing "
                         "recipe's per-step count)")
    ap.add_argument("--kv", default="16bit", choices=["16bit", "fp8"],
                    help="KV pool format: the workload's 16-bit type, or e4m3 codes with per-(block, KV head) "
                         "scales (copy, write and attention through the *_fp8 entry points)")
    args = ap.parse_args(argv)
    if args.steps is None:
        args.steps = 5000 if args.impl == "ours" else 20
    if args.warmup is None:
        args.warmup = 20 if args.impl == "ours" else 3
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.config is None and (args.impl == "reference" or args.layers > 0 or args.op is not None):
        # the reference arm times the headline workload; the single-purpose modes default to the 8B-class layer
        args.config = HEADLINE_CONFIG if args.impl == "reference" else 2
    if args.kv == "fp8" and args.block_size != 16:
        ap.error("FP8 pools use 16-token blocks")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.swap_gib > 0:
        line = run_swap(args)
    elif args.op is not None:
        line = run_cache_op(args)
    elif args.layers > 0:
        line = run_layers(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
