"""Benchmark of the paged-decode step on GB300.

A step is one pass of the whole hot path over one batch: copy_blocks (if the
workload has copy-on-write pairs), reshape_and_cache (if it appends a token)
and the decode (with its split-K merge).  The default run measures the GQA
batch-128 decode (128 sequences, 32 query / 8 kv heads, head_dim 128, bf16,
lognormal lengths) as the headline, and the other four decode workloads
(long-context split-K, MHA 7B-shaped, parallel sampling, tiny) the same way,
nested under "workloads" in the same line, and the pool-maintenance kernels
(copy_blocks, reshape_and_cache) alone under "pool_kernels".  ``--workload``
runs one workload alone (also the chunked-prefill, swap and cache lines).

Prints ONE JSON line (rank 0):
  value      effective KV-read GB/s of the whole job: sum over ranks of the
             K/V bytes a step must read (every live token, every kv head)
             divided by the step time (max over ranks); steps run back to
             back with no event node between them
  e2e        the same metric through the public API with host buffers: each
             step copies its inputs from pinned host memory and reads the
             output back inside the timed region, the copies on their own
             streams and double-buffered so that they overlap the
             neighbouring steps' compute, as a serving loop runs
  roofline   one decode call (decode + merge kernels) against the measured
             HBM peak, on the bytes that must leave HBM (a block shared by
             several sequences counts once); the call's duration is the
             timed region's average where a step is that call alone, else
             the mean of event pairs around single calls
  cpu_baseline  the fp64 oracle's step on the host cores, sized and timed
             the same way as ``--impl reference``
  parity_vs_oracle  the timed step's output, every sequence, against the
             oracle's

``--impl reference`` times the oracle instead (the only reference this
method has), on the same workload, metric and unit.

Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU (sequences are independent; there is no exchange step), so per-GPU
work is fixed as N grows (weak scaling).  Only the timing is reduced across
ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged decode attn: effective KV-read HBM GB/s, % of GB300 peak; seqs/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DEFAULT_PARTITION = {"tiny": 0, "mha7b": 0, "gqa8b": 0, "long": 512, "parsamp": 0, "batch20k": 0,
                     "parsamp8k": 0}
DESCRIPTION = {
    "tiny": "tiny decode: 4 seqs, 8/8 heads, head_dim 64, fp16, lens U[1,100], 64-block pool, +1 token",
    "mha7b": "MHA 7B-shaped decode: 64 seqs, 32/32 heads, head_dim 128, fp16, lens U[512,2048]",
    "gqa8b": ("GQA 8B-shaped decode: 128 seqs, 32/8 heads, head_dim 128, bf16, lens "
              "lognormal(median 600, sigma 1) clipped [16,4096], +1 token per seq via slot_mapping"),
    "long": ("long-context split-K decode: 4 seqs, 32/8 heads, head_dim 128, bf16, lens "
             "{32768,65536,98304,131072}, 512-token partitions + log-sum-exp merge"),
    "parsamp": ("parallel sampling: 16 prompts x 8 samples, 40/8 heads, head_dim 128, fp16, "
                "1024 shared prompt tokens + U[0,256] + 1, 112 copy-on-write pairs per step"),
    "batch20k": ("large continuous batch: 20000 seqs, 32/2 heads (group 16), head_dim 128, bf16, "
                 "lens U[1,256], +1 token per seq; per-sequence arrays in the workspace"),
    "parsamp8k": ("parallel sampling with a long prompt: 16 prompts x 8 samples, 40/8 heads, "
                  "head_dim 128, fp16, 8192 shared prompt tokens + U[0,256] + 1, 112 "
                  "copy-on-write pairs per step"),
}
# parallel-sampling workloads that run pa_decode_shared_prefix by default
SHARED_DEFAULT = {"parsamp": True, "parsamp8k": True}


# ---------------------------------------------------------------------------
# distributed plumbing (timing only)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend, rank=rank, world_size=world)
    return rank, world


def barrier(device=None):
    import torch
    import torch.distributed as dist
    if dist.is_initialized():
        if dist.get_backend() == "nccl" and device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()
    if device is not None and torch.cuda.is_available():
        torch.cuda.synchronize(device)


def dist_max(x: float, device=None) -> float:
    """Max of a scalar over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        return float(x)
    dev = device if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        return float(x)
    dev = device if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (independent sequences, same sizes)."""
    return base_seed + 7919 * rank


# ---------------------------------------------------------------------------
# workload, peaks, clocks
# ---------------------------------------------------------------------------
def make_workload(name: str, seed_offset: int = 0):
    import synth
    base = {"tiny": 1001, "mha7b": 1002, "gqa8b": 1003, "long": 1004, "parsamp": 1005,
            "batch20k": 1008, "parsamp8k": 1009}[name]
    return synth.by_name(name, seed=replica_seed(base, seed_offset))


def measured_hbm_peak():
    """(GB/s, source) from MEASURED_PEAKS.json, else the recipe's fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
            return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the decode, and the shared-prefix decode's prefix attention and helpers
DECODE_SOURCES = ("pa_decode_mma.cuh", "pa_schedule.cuh", "pa_device.cuh", "pa_internal.h",
                  "pa_prefix.cu", "pa_shared.cu", "pa_shared.h")
PREFILL_SOURCES = ("pa_prefill.cuh", "pa_prefill_abi.h", "pa_tcgen05.cuh", "pa_device.cuh")


def source_hash(names=DECODE_SOURCES) -> str:
    """Hash of a kernel's sources: ncu counters apply only to this build."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_260_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_source_hash() -> str:
    return source_hash(DECODE_SOURCES)


def ncu_traffic(workload: str, table: str = "decode_dram_traffic.txt", names=DECODE_SOURCES):
    """DRAM bytes per launch of the workload's dominant kernel (for the
    shared-prefix decode, its prefix attention and its suffix decode
    together) from the committed ncu summary, if it was taken on the current
    kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", table)
    if not os.path.exists(path):
        return None
    src = source_hash(names)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == src:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clock samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def physical_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if local_rank < len(ids) and ids[local_rank].isdigit():
        return int(ids[local_rank])
    return local_rank


# ---------------------------------------------------------------------------
# our arm: the CUDA path through the C ABI
# ---------------------------------------------------------------------------
class Step:
    """Device state of one replica and its decode step (graph-captured)."""

    def __init__(self, w, device, partition_size, shared=None):
        import torch
        import paged_kv_cache_260_gb300 as pa
        self.pa, self.w, self.dev, self.ps = pa, w, device, partition_size
        tdt = torch.float16 if w.dtype == "f16" else torch.bfloat16
        self.tdt = tdt

        def bits(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)

        self.q = bits(w.q)
        self.k = bits(w.k_cache)
        self.v = bits(w.v_cache)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.out = torch.empty_like(self.q)
        self.k_new = None if w.k_new is None else bits(w.k_new)
        self.v_new = None if w.v_new is None else bits(w.v_new)
        self.slots = None if w.slot_mapping is None else torch.from_numpy(w.slot_mapping).to(device)
        self.pairs = (None if w.block_mapping is None or len(w.block_mapping) == 0
                      else torch.from_numpy(w.block_mapping).to(device))
        # parallel samples with a long shared prompt: the shared-prefix decode
        # reads each prompt's shared blocks once per group of samples (with a
        # short prompt its second decode pass costs more than it saves)
        self.shared = (shared if shared is not None else SHARED_DEFAULT.get(w.name, False)) \
            and "samples" in w.meta and partition_size == 0
        if self.shared:
            self.group = int(w.meta["samples"])
            self.prefix_len = (-(-int(w.meta["prompt_len"]) // 16) - 1) * 16
            n, hq, d = self.q.shape
            nbytes = pa.decode_shared_prefix_workspace_size(n, self.group, self.prefix_len, hq,
                                                            self.k.shape[1], d,
                                                            self.tables.shape[1])
            self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        else:
            self.ws = pa.workspace_for(self.q, self.k, self.tables, partition_size)
        self.launches_per_step = self._count_launches()

    def _count_launches(self):
        n = int(self.pairs is not None)                 # copy_blocks
        # above 2048 sequences two kernels build the decode's per-sequence
        # arrays in the workspace
        n += 2 if self.w.num_seqs > 2048 else 0
        if self.shared:
            # prefix attention, suffix decode, final merge (which also folds
            # the suffix runs the decode cut)
            return n + 3
        n += 1                                          # decode (append fused in)
        # the library decodes short runs whole when each gets a warp of its
        # own (tables at most 8 blocks wide, at most four runs per SM)
        import torch
        sms = torch.cuda.get_device_properties(self.dev).multi_processor_count
        whole = self.ps < 0 or (self.ps == 0 and self.tables.shape[1] <= 8 and
                                self.w.num_seqs * self.k.shape[1] <= 4 * sms)
        if not whole:
            n += 1                                      # merge of cut runs / partitions
        if self.ps > 0 and self.tables.shape[1] * 16 > self.ps:
            n += 1                                      # merge of partitions per run
        return n

    def run(self, ev_pair=None):
        """Enqueue one step on the current stream; ev_pair brackets the decode call."""
        pa = self.pa
        if self.pairs is not None:
            pa.copy_blocks(self.k, self.v, self.pairs)
        if ev_pair is not None:
            ev_pair[0].record()
        if self.shared:
            pa.decode_shared_prefix(self.out, self.q, self.k, self.v, self.tables, self.lens,
                                    self.group, self.prefix_len, self.w.scale, k_new=self.k_new,
                                    v_new=self.v_new, slot_mapping=self.slots, workspace=self.ws)
        elif self.slots is not None:
            # reshape_and_cache of the newest token fused into the decode launch
            pa.decode_append(self.out, self.q, self.k, self.v, self.tables, self.lens, self.k_new,
                             self.v_new, self.slots, self.w.scale, partition_size=self.ps,
                             workspace=self.ws)
        else:
            pa.decode(self.out, self.q, self.k, self.v, self.tables, self.lens, self.w.scale,
                      partition_size=self.ps, workspace=self.ws)
        if ev_pair is not None:
            ev_pair[1].record()


def timing_event():
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:                      # torch without external events
        return None


def capture(fns, device):
    """A CUDA graph of the enqueued work of `fns`, called in order (after two
    eager warm-up passes on a side stream)."""
    import torch
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for _ in range(2):
            for f in fns:
                f()
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    return g


def pick_steps_per_graph(steps: int, cap: int = 32) -> int:
    """Largest divisor of `steps` not above `cap`, so K steps are replayed exactly."""
    for d in range(min(cap, max(1, steps)), 0, -1):
        if steps % d == 0:
            return d
    return 1


def pool_utilisation(w):
    """Slots of the pool holding a live token (shared blocks counted once)."""
    per_token = w.num_kv_heads * w.head_dim * 2 * 2
    unique = w.unique_kv_read_bytes() // per_token
    return {"live_tokens": int(unique), "pool_slots": int(w.num_blocks * 16),
            "frac_slots_live": float(unique) / (w.num_blocks * 16),
            "table_tokens": int(w.seq_lens.sum())}


# ---------------------------------------------------------------------------
# the oracle's timed step (cpu_baseline and --impl reference use the same one)
# ---------------------------------------------------------------------------
def oracle_pool_after_step(w):
    """Host copies of the pool after the step's copy_blocks and
    reshape_and_cache, applied by the oracle (not timed: the timed oracle step
    is the decode, which is where the step's work is)."""
    import oracle
    k, v = w.k_cache.copy(), w.v_cache.copy()
    if w.block_mapping is not None and len(w.block_mapping):
        oracle.copy_blocks(k, v, w.block_mapping)
    if w.slot_mapping is not None:
        oracle.reshape_and_cache(k, v, w.k_new, w.v_new, w.slot_mapping)
    return k, v


def oracle_step_budget(steps: int, warmup: int) -> float:
    """Seconds one oracle step may take: the whole --steps/--warmup run of the
    reference arm then ends within about two minutes."""
    return min(2.0, 120.0 / max(1, steps + warmup))


def oracle_sample(w, k, v, budget_s: float):
    """The oracle's step on the host cores: one fp64 decode call over the
    first n sequences of the workload (every host thread), n the largest prefix
    whose call fits `budget_s` (timed: doubling, then bisection); when one
    sequence alone exceeds it, a prefix of that sequence's tokens.

    Returns (run, bytes per step, threads, text); run() performs one step and
    returns the oracle's rows {sequence: fp64 [Hq, D]}."""
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    per_tok = 2 * w.num_kv_heads * w.head_dim * 2
    lens = w.seq_lens.copy()

    def call(n):
        sel = list(range(n))
        out = oracle.decode(w.q, k, v, w.block_tables, lens, w.scale, w.dtype, seqs=sel,
                            threads=threads)
        return {s: out[s] for s in sel}

    def timed(n):
        t0 = time.perf_counter()
        call(n)
        return time.perf_counter() - t0

    call(1)                                              # first call: library and pages
    one = timed(1)
    if one > budget_s:
        lens[0] = max(1, int(int(w.seq_lens[0]) * budget_s / one))
        n = 1
        what = f"the first {int(lens[0])} tokens of sequence 0"
    else:
        lo, hi = 1, 1
        while hi < w.num_seqs:
            hi = min(w.num_seqs, 2 * hi)
            if timed(hi) > budget_s:
                break
            lo = hi
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if timed(mid) > budget_s:
                hi = mid
            else:
                lo = mid
        n = lo
        what = ("all %d sequences" % n if n == w.num_seqs
                else f"sequences 0..{n - 1} of {w.num_seqs}")
    nbytes = int(sum(int(lens[s]) for s in range(n))) * per_tok
    text = (f"fp64 oracle decode of {what} per step, one call on {threads} host threads "
            f"(copy_blocks / reshape_and_cache applied once beforehand, untimed)")
    return (lambda: call(n)), nbytes, threads, text


def cpu_baseline(w, steps: int, warmup: int, budget_s: float = 10.0):
    """The oracle's step (oracle_sample, sized exactly as --impl reference
    sizes it for the same --steps/--warmup) repeated for ~budget_s."""
    k, v = oracle_pool_after_step(w)
    run, nbytes, threads, text = oracle_sample(w, k, v, oracle_step_budget(steps, warmup))
    run()
    reps = 0
    t0 = time.perf_counter()
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": nbytes * reps / dt / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "sample": f"{text}; {reps} steps in {dt:.1f} s"}


def parity_vs_oracle(w, out):
    """The timed step's output (every sequence) against the oracle's step."""
    import oracle
    oracle.build()
    k, v = oracle_pool_after_step(w)
    t0 = time.perf_counter()
    ref = oracle.decode(w.q, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype)
    dt = time.perf_counter() - t0
    got = out.float().cpu().numpy().astype(np.float64)
    err = float(np.abs(got - ref).max())
    tol = 4e-3 if w.dtype == "f16" else 1.6e-2
    return {"max_abs_err": err, "sequences": int(w.num_seqs), "tolerance": tol,
            "ok": bool(np.isfinite(got).all() and err <= tol), "oracle_s": dt}


# ---------------------------------------------------------------------------
# pipelined end-to-end steps through the public API
# ---------------------------------------------------------------------------
def pipelined_e2e(inputs, out, bind, step, steps: int, device, before=None):
    """End-to-end steps through the public API with host buffers, pipelined
    the way a serving loop runs them.

    Every step copies its inputs in from one packed, pinned host buffer (H2D,
    on a copy stream) and its output back to pinned host memory (D2H, on a
    second copy stream); the step itself runs on the current stream.  The
    device inputs and the output are double-buffered, so step i's H2D
    overlaps step i-1's compute and step i's D2H overlaps step i+1's; events
    order every reuse of a buffer.

    inputs: the device tensors a step reads (their contents fill the host
    buffer); out: the tensor it writes; bind(views, out_buf) points the step
    at one buffer set; step() enqueues the step; before(), if given, is
    enqueued on the compute stream ahead of each step (an L2 flush).
    Returns (ms per step, H2D bytes, D2H bytes, the last step's host output).
    """
    import torch
    offs, total = [], 0
    for t in inputs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(inputs, offs):
        host[o:o + t.numel() * t.element_size()].copy_(t.reshape(-1).view(torch.uint8).cpu())
    devs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [[d[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
              for t, o in zip(inputs, offs)] for d in devs]
    outs = [torch.empty_like(out) for _ in range(2)]
    outs_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    comp = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_ready, in_free, out_ready, out_free = ([torch.cuda.Event(), torch.cuda.Event()]
                                              for _ in range(4))
    count = [0]

    def one():
        i = count[0]
        count[0] += 1
        b = i % 2
        if i >= 2:                       # the step that last read set b is done
            s_in.wait_event(in_free[b])
        with torch.cuda.stream(s_in):
            devs[b].copy_(host, non_blocking=True)
        in_ready[b].record(s_in)
        if before is not None:
            before()
        comp.wait_event(in_ready[b])
        if i >= 2:                       # output buffer b has been read back
            comp.wait_event(out_free[b])
        bind(views[b], outs[b])
        step()
        in_free[b].record(comp)
        out_ready[b].record(comp)
        s_out.wait_event(out_ready[b])
        with torch.cuda.stream(s_out):
            outs_h[b].copy_(outs[b], non_blocking=True)
        out_free[b].record(s_out)

    for _ in range(3):
        one()
    torch.cuda.synchronize(device)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    s_in.wait_stream(comp)               # the first copy starts inside the timed region
    for _ in range(steps):
        one()
    comp.wait_stream(s_out)              # ... and the last read-back ends inside it
    z.record(comp)
    torch.cuda.synchronize(device)
    h2d = total
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    return a.elapsed_time(z) / steps, h2d, d2h, outs_h[(count[0] - 1) % 2].clone()


def e2e_measure(st, steps: int, device, rotate_pools: bool = False):
    """The decode step end to end (pipelined_e2e): q, tables, lengths, the new
    tokens, their slots and the copy-on-write pairs come in from one packed
    pinned host buffer, the output goes back.  With `rotate_pools` (working
    sets that L2 could hold) the steps cycle through copies of the pool whose
    sizes add up to at least twice L2, so that no step finds the K/V it reads
    left in L2 by an earlier step -- the end-to-end counterpart of the L2
    flush before every device-timed step, without a flush inside the timed
    region.  The last step's host output must equal the device-resident
    step's, bit for bit.  Returns (ms per step, h2d bytes, d2h bytes, pool
    copies)."""
    import torch
    names = [n for n in ["q", "tables", "lens", "k_new", "v_new", "slots", "pairs"]
             if getattr(st, n) is not None]
    saved = [getattr(st, n) for n in names]
    saved_out = st.out
    saved_pool = (st.k, st.v)
    pools = [saved_pool]
    if rotate_pools:
        pool_bytes = 2 * st.k.numel() * st.k.element_size()
        copies = min(64, max(2, -(-2 * L2_BYTES // pool_bytes)))
        pools += [(st.k.clone(), st.v.clone()) for _ in range(copies - 1)]
    turn = [0]

    def bind(views, out_buf):
        for n, v in zip(names, views):
            setattr(st, n, v)
        st.out = out_buf
        st.k, st.v = pools[turn[0] % len(pools)]
        turn[0] += 1

    try:
        ms, h2d, d2h, last = pipelined_e2e(saved, saved_out, bind, st.run, steps, device)
    finally:
        for n, v in zip(names, saved):
            setattr(st, n, v)
        st.out = saved_out
        st.k, st.v = saved_pool
    copies = len(pools)
    del pools
    st.run()
    torch.cuda.synchronize(device)
    if not torch.equal(st.out.cpu(), last):
        raise RuntimeError("the pipelined end-to-end step's output differs from the "
                           "device-resident step's")
    return ms, h2d, d2h, copies


# ---------------------------------------------------------------------------
# one decode workload, measured
# ---------------------------------------------------------------------------
def time_decode(st, w, args, device, big: bool, use_graph: bool):
    """Device time of K steps, and the mean duration of one decode call.

    big (K/V per step above twice L2): K steps run back to back, as a CUDA
    graph of `spg` steps replayed K/spg times with no event node inside it
    (an event-record node between two kernels would cut their programmatic
    dependency), CUDA events around the replays.  After the timed region one
    more replay of a second graph, with an event pair around every decode
    call, gives the durations of single calls.
    Otherwise: L2 flushed (2 x L2 write) before every step; each step timed
    alone with events around it and around its decode call.
    Returns (elapsed ms over K steps, mean ms of a single call between its
    own events, timing text)."""
    import torch
    K = args.steps
    if big and use_graph:
        spg = pick_steps_per_graph(K)
        g = capture([st.run] * spg, device)
        ev = [(timing_event(), timing_event()) for _ in range(spg)]
        g_ev = capture([lambda e=e: st.run(e) for e in ev], device)
        for _ in range(max(1, -(-args.warmup // spg))):
            g.replay()
        torch.cuda.synchronize(device)
        barrier(device)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(K // spg):
            g.replay()
        t1.record()
        torch.cuda.synchronize(device)
        elapsed = t0.elapsed_time(t1)
        g_ev.replay()
        torch.cuda.synchronize(device)
        call_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
        text = (f"CUDA graph of {spg} steps back to back (no event nodes), replayed {K // spg} "
                f"times, CUDA events around the replays; call durations from one more replay "
                f"of the same steps with an event pair around each decode call, after the "
                f"timed region")
        return elapsed, call_ms, text
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    if big:
        for _ in range(args.warmup):
            st.run()
        torch.cuda.synchronize(device)
        barrier(device)
        t0.record()
        for _ in range(K):
            st.run()
        t1.record()
        torch.cuda.synchronize(device)
        elapsed = t0.elapsed_time(t1)
        calls = []
        for _ in range(min(K, 32)):
            st.run(e)
            torch.cuda.synchronize(device)
            calls.append(e[0].elapsed_time(e[1]))
        return elapsed, float(np.mean(calls)), "eager steps back to back, CUDA events around them"
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    # a step timed alone would otherwise wait for the host between launches:
    # each step is one CUDA-graph replay (or, without graphs, eager launches)
    if use_graph:
        e = (timing_event(), timing_event())      # recorded inside a graph: external
        g1 = capture([st.run], device)
        g1_ev = capture([lambda: st.run(e)], device)
        one, one_ev = g1.replay, g1_ev.replay
    else:
        one, one_ev = st.run, (lambda: st.run(e))
    for _ in range(args.warmup):
        flush.zero_()
        one()
    torch.cuda.synchronize(device)
    barrier(device)
    elapsed, calls = 0.0, []
    for _ in range(K):
        flush.zero_()
        t0.record()
        one()
        t1.record()
        torch.cuda.synchronize(device)
        elapsed += t0.elapsed_time(t1)
    for _ in range(min(K, 32)):
        flush.zero_()
        one_ev()
        torch.cuda.synchronize(device)
        calls.append(e[0].elapsed_time(e[1]))
    return (elapsed, float(np.mean(calls)),
            "L2 flushed (2 x 129 MB write) before every step; each step timed alone with "
            "CUDA events" + (", replayed as a CUDA graph of the step" if use_graph else "")
            + "; call durations from separate replays with an event pair around the decode call")


def l2_carryover(w, st, args, device):
    """Steps alternating between two copies of the workload in separate
    buffers, so that no step finds the previous step's K/V in L2.  Returns the
    alternating step time, to set against the repeated step's."""
    import torch
    st2 = Step(w, device, st.ps)
    spg = 16
    g = capture([st.run, st2.run] * (spg // 2), device)
    for _ in range(max(1, -(-args.warmup // spg))):
        g.replay()
    torch.cuda.synchronize(device)
    reps = max(1, args.steps // spg)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        g.replay()
    t1.record()
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / (reps * spg)
    del st2, g
    return ms, reps * spg


def measure_decode(name: str, args, device, rank: int, world: int, partition=None,
                   headline: bool = False) -> dict:
    """One decode workload on this rank's GPU: device-resident rate, end-to-end
    rate through the public API, the decode call's roofline, the timed step's
    output against the oracle (rank 0, N=1) and the clocks seen."""
    import torch
    import paged_kv_cache_260_gb300 as pa
    ps = DEFAULT_PARTITION[name] if partition is None else partition
    w = make_workload(name, rank)
    st = Step(w, device, ps, shared={"auto": None, "on": True, "off": False}[args.shared_prefix])
    kv_bytes = w.kv_read_bytes()
    # blocks that sequences share (parallel sampling) need leaving HBM once
    # per step: the L2 decision and the HBM roofline count them once
    unique_bytes = w.unique_kv_read_bytes()
    big = unique_bytes > 2 * L2_BYTES
    use_graph = timing_event() is not None and not args.no_graph
    pa.get_device_error()
    with ClockSampler(physical_gpu_index(dist_env()[2])) as clk:
        elapsed, call_ms, timing_text = time_decode(st, w, args, device, big, use_graph)
        barrier(device)
    assert pa.get_device_error() == 0, f"{name}: a kernel recorded an error in the timed region"
    t_max = dist_max(elapsed, device)
    ms_per_step = t_max / args.steps
    total_bytes = dist_sum(kv_bytes, device)
    value = total_bytes / (ms_per_step * 1e-3) / 1e9
    e2e_ms, h2d, d2h, copies = e2e_measure(st, max(20, min(args.steps, 300)), device,
                                           rotate_pools=not big)
    e2e_ms = dist_max(e2e_ms, device)
    peak, peak_src = measured_hbm_peak()
    # The roofline's duration of one decode call: where a step is that call
    # alone and steps run back to back, the timed region's average (the
    # region's events over its calls); otherwise the mean of the event pairs
    # around single calls, which also keep a call from overlapping the one
    # before it.
    call_isolated = call_ms
    region_avg = big and st.pairs is None
    if region_avg:
        call_ms = t_max / args.steps
    achieved = unique_bytes / (call_ms * 1e-3) / 1e9
    # the other bytes a call must move, beside the K/V: q and the output,
    # the tables and lengths read, and the new tokens read and written
    el = 2
    io_bytes = (2 * w.num_seqs * w.num_heads * w.head_dim * el
                + w.block_tables.size * 4 + w.num_seqs * 4
                + (4 * w.num_seqs * w.num_kv_heads * w.head_dim * el
                   if w.slot_mapping is not None else 0))
    carry = None
    if headline and big and use_graph and not args.no_l2_check:
        alt_ms, alt_steps = l2_carryover(w, st, args, device)
        carry = {"ms_per_step_alternating": alt_ms, "steps": alt_steps,
                 "ms_per_step_repeated": ms_per_step,
                 "ratio": alt_ms / ms_per_step,
                 "how": "the same steps alternating between two copies of the workload in "
                        "separate buffers (no step finds the previous step's K/V in L2), "
                        "against the same step repeated"}
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        parity = parity_vs_oracle(w, st.out)
    shared = unique_bytes != kv_bytes
    other = None
    if "samples" in w.meta and ps == 0 and not args.no_other_decode:
        # the same step with the other decode of a parallel-sampling batch,
        # timed the same way, for comparison
        st_o = Step(w, device, ps, shared=not st.shared)
        o_elapsed, o_call, _ = time_decode(st_o, w, args, device, big, use_graph)
        other = {"ms_per_step": o_elapsed / args.steps, "call_ms": o_call,
                 "value": kv_bytes / (o_elapsed / args.steps * 1e-3) / 1e9,
                 "decode": ("pa_decode_shared_prefix (the shared prompt blocks read once per "
                            "group)" if st_o.shared else
                            "pa_decode_append (every sample reads the shared prompt blocks)")}
        del st_o
    res = {
        "value": value,
        "unit": "GB/s",
        "ms_per_step": ms_per_step,
        "pct_of_hbm_peak": 100.0 * unique_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
        "unique_gbps": dist_sum(unique_bytes, device) / (ms_per_step * 1e-3) / 1e9,
        "seqs_per_s": dist_sum(w.num_seqs, device) / (ms_per_step * 1e-3),
        "dtype": w.dtype,
        "config": {
            "workload": DESCRIPTION[name],
            "name": name,
            "num_seqs": w.num_seqs, "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": 16, "partition_size": ps,
            "kv_bytes_per_step": kv_bytes,
            "unique_kv_bytes_per_step": unique_bytes,
            "step": ("copy_blocks + " if w.block_mapping is not None else "")
                    + ("shared-prefix decode (pa_decode_shared_prefix, groups of %d samples, "
                       "%d shared tokens) with reshape_and_cache fused"
                       % (st.group, st.prefix_len) if st.shared else
                       "decode with reshape_and_cache fused (pa_decode_append)"
                       if w.slot_mapping is not None else "decode") + " + merge",
            "l2": ("inputs larger than L2 (K/V read per step %.0f MB vs 129 MB L2)"
                   % (unique_bytes / 1e6) if big else
                   "L2 flushed (2 x 129 MB write) before every step"),
            "timing": timing_text,
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "l2": ("inputs larger than L2" if big else
                       f"steps cycle through {copies} copies of the pool (>= 2 x L2 in all), "
                       f"no flush in the timed region")},
        "roofline": {"bound": "hbm",
                     "kernel": ("one pa_decode_shared_prefix call: prefix_attn_kernel (each "
                                "shared prefix block read once for all of its group's query "
                                "columns), the suffix decode (decode_mma_kernel + merge), the "
                                "final merge"
                                if st.shared else
                                "decode_mma_kernel + merge kernel(s): one pa_decode / "
                                "pa_decode_append call"),
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "peak_source": (peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy burst)"
                                     if peak_src == "measured" else "fallback 6.8 TB/s"),
                     "algorithmic_bytes_per_launch": unique_bytes,
                     "bytes_basis": ("unique blocks: a block that several sequences share "
                                     "counts once" if shared else
                                     "K and V of every live token and kv head"),
                     "call_ms": call_ms,
                     "call_ms_from": ("the timed region: its CUDA events over the decode "
                                      "calls it ran back to back" if region_avg else
                                      "an event pair around each decode call"),
                     "call_ms_isolated": call_isolated,
                     "io_bytes_per_launch": io_bytes,
                     "io_basis": ("q and the output, the tables and lengths, the new "
                                  "tokens read and written: bytes the call must move "
                                  "beside the K/V, left out of achieved"),
                     "all_bytes_gbps": (unique_bytes + io_bytes) / (call_ms * 1e-3) / 1e9,
                     "traffic": ncu_traffic(name)},
        "parity_vs_oracle": parity,
        "pool_utilisation": pool_utilisation(w),
        "gpu_launches": st.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if shared:
        res["logical_kv_gbps"] = value
    if other is not None:
        res["shared_prefix_decode" if not st.shared else "plain_decode"] = other
    if carry is not None:
        res["l2_carryover"] = carry
    res["_w"] = w
    return res


NESTED = ("long", "mha7b", "parsamp", "tiny", "batch20k", "parsamp8k")


def run_ours(args):
    import torch
    rank, world = dist_init("nccl" if torch.cuda.is_available() else "gloo")
    local = dist_env()[2]
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    from paged_kv_cache_260_gb300 import _build
    _build.build()
    import paged_kv_cache_260_gb300 as pa
    pa.load()

    head_name = args.workload or "gqa8b"
    head = measure_decode(head_name, args, device, rank, world, args.partition, headline=True)
    w = head.pop("_w")
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.steps, args.warmup)
    nested = {}
    cache = None
    if args.workload is None and not args.only_headline:
        for name in NESTED:
            r = measure_decode(name, args, device, rank, world)
            r.pop("_w")
            nested[name] = r
        # the pool-maintenance kernels alone (each rank on its own GPU)
        cases = measure_cache(args, device)
        cache = {"metric": CACHE_METRIC, "unit": "GB/s",
                 "bit_exact": all(c["bit_exact"] for c in cases.values()),
                 "cases": {k: {f: c[f] for f in ("us_per_launch", "bytes_per_launch", "gbps",
                                                  "frac", "bit_exact", "traffic")}
                           for k, c in cases.items()},
                 "peak": measured_hbm_peak()[0],
                 "timing": "bulk cases back to back, step-size cases one launch after an L2 "
                           "flush (`--workload cache` describes each case)"}
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V, random block permutation)",
    }
    line.update({k: v for k, v in head.items() if k not in ("value", "unit", "ms_per_step", "dtype")})
    line["cpu_baseline"] = cpu
    if nested:
        line["workloads"] = nested
    if cache is not None:
        line["pool_kernels"] = cache
    print(json.dumps(line), flush=True)


def run_swap(args):
    """Swap half the GQA batch's blocks out to a page-locked host pool and back
    (pa_swap_blocks), timed with CUDA events; the denominator is the plain
    pinned-memory copy rate of the same bytes measured in the same run."""
    import torch
    from paged_kv_cache_260_gb300 import _build
    _build.build()
    import paged_kv_cache_260_gb300 as pa
    pa.load()
    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    w = make_workload("gqa8b")
    st = Step(w, device, 0)
    seqs = range(0, w.num_seqs, 2)
    blocks = np.concatenate([w.block_tables[s, :(int(w.seq_lens[s]) + 15) // 16] for s in seqs])
    nb = len(blocks)
    host_k = torch.empty((nb,) + tuple(st.k.shape[1:]), dtype=st.k.dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    out_pairs = torch.from_numpy(np.stack([blocks, np.arange(nb)], 1).astype(np.int64)).to(device)
    in_pairs = torch.from_numpy(np.stack([np.arange(nb), blocks], 1).astype(np.int64)).to(device)
    moved = 2 * nb * st.k[0].numel() * st.k.element_size()      # K and V, one direction
    for _ in range(args.warmup):
        pa.swap_blocks(host_k, host_v, st.k, st.v, out_pairs)
        pa.swap_blocks(st.k, st.v, host_k, host_v, in_pairs)
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t_out = t_in = 0.0
    steps = max(1, min(args.steps, 50))
    for _ in range(steps):
        ev[0].record()
        pa.swap_blocks(host_k, host_v, st.k, st.v, out_pairs)
        ev[1].record()
        pa.swap_blocks(st.k, st.v, host_k, host_v, in_pairs)
        ev[2].record()
        torch.cuda.synchronize(device)
        t_out += ev[0].elapsed_time(ev[1])
        t_in += ev[1].elapsed_time(ev[2])
    assert pa.get_device_error() == 0
    # plain copies of the same bytes between device and page-locked host memory
    dev_buf = torch.empty(moved, dtype=torch.uint8, device=device)
    host_buf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    for _ in range(3):
        host_buf.copy_(dev_buf, non_blocking=True)
        dev_buf.copy_(host_buf, non_blocking=True)
    torch.cuda.synchronize(device)
    c_out = c_in = 0.0
    for _ in range(steps):
        ev[0].record()
        host_buf.copy_(dev_buf, non_blocking=True)
        ev[1].record()
        dev_buf.copy_(host_buf, non_blocking=True)
        ev[2].record()
        torch.cuda.synchronize(device)
        c_out += ev[0].elapsed_time(ev[1])
        c_in += ev[1].elapsed_time(ev[2])
    gbs = lambda t: moved * steps / (t * 1e-3) / 1e9
    value = 2 * moved * steps / ((t_out + t_in) * 1e-3) / 1e9
    peak = 2 * moved * steps / ((c_out + c_in) * 1e-3) / 1e9
    print(json.dumps({
        "metric": "swap_blocks: GB/s moved between the GPU pool and a page-locked host pool",
        "value": value, "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": (t_out + t_in) / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"swap out and back in {nb} blocks ({moved / 1e6:.0f} MB of K+V) "
                               "of 64 of the 128 GQA-8B sequences, random block ids"},
        "swap_out_gbs": gbs(t_out), "swap_in_gbs": gbs(t_in),
        "roofline": {"bound": "host link", "achieved": value, "peak": peak, "unit": "GB/s",
                     "frac": value / peak,
                     "peak_source": "pinned-memory cudaMemcpy of the same bytes, same run",
                     "copy_out_gbs": gbs(c_out), "copy_in_gbs": gbs(c_in)},
        "gpu_launches": 2 * steps,
    }), flush=True)


CACHE_METRIC = "KV-cache maintenance kernels: HBM GB/s moved (bytes read + written)"
CACHE_SOURCES = ("pa_cache.cu", "pa_cache.h", "pa_device.cuh")
CACHE_CASES = {
    "copy_cow": "copy_blocks, the parallel-sampling step's 112 copy-on-write pairs from 16 "
                "source blocks (K and V of 8 kv heads, 64 KB a pair), L2 flushed before every "
                "launch",
    "copy_bulk": "copy_blocks, 4096 pairs of random distinct blocks of an 8192-block pool "
                 "(8 kv heads, head_dim 128, bf16), back to back",
    "reshape_step": "reshape_and_cache, the GQA batch-128 step's 128 new tokens (8 kv heads, "
                    "head_dim 128, bf16), L2 flushed before every launch",
    "reshape_blocks": "reshape_and_cache, a prefill's 65536 tokens filling 4096 whole blocks "
                      "at random distinct ids of the same 8192-block pool, back to back",
    "reshape_scatter": "reshape_and_cache, 65536 tokens into random distinct slots of the same "
                       "8192-block pool (the decode's pattern at prefill size), back to back",
}


def measure_cache(args, device, only=None):
    """The two kernels that maintain the pool, timed alone: copy_blocks (the
    copy-on-write of whole blocks) and reshape_and_cache (each new token's K/V
    into its slot), at a config step's size and at a size large enough to be
    bound by HBM.  GB/s counts the bytes read and written.  The step-size
    pools are compared bit for bit with the oracle's; the bulk copies with
    their sources.  Returns {case: result}."""
    import torch
    import paged_kv_cache_260_gb300 as pa
    peak, _ = measured_hbm_peak()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    rng = np.random.default_rng(1010)
    steps = max(1, min(args.steps, 100))

    def timed(fn, big):
        g = capture([fn], device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize(device)
        if big:                            # back to back, events around the replays
            e0.record()
            for _ in range(steps):
                g.replay()
            e1.record()
            torch.cuda.synchronize(device)
            return e0.elapsed_time(e1) / steps, "back to back (one-launch graph replays)"
        total = 0.0                        # each launch alone after an L2 flush
        for _ in range(steps):
            flush.zero_()
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize(device)
            total += e0.elapsed_time(e1)
        return total / steps, "L2 flushed before each launch, events around a one-launch graph replay"

    def bits(t):
        return t.view(torch.int16)

    def host_bits(t):
        return bits(t).cpu().numpy().view(np.uint16).copy()

    def record(name, ms, timing, moved, exact):
        gbs = moved / (ms * 1e-3) / 1e9
        cases[name] = {"description": CACHE_CASES[name], "us_per_launch": ms * 1e3,
                       "bytes_per_launch": moved, "gbps": gbs, "frac": gbs / peak,
                       "bit_exact": exact, "timing": timing,
                       "traffic": ncu_traffic(name, "cache_dram_traffic.txt", CACHE_SOURCES)}

    cases = {}
    import oracle
    if only in (None, "copy_cow"):
        w = make_workload("parsamp")
        st = Step(w, device, 0, shared=False)
        pairs = st.pairs
        kh, vh = host_bits(st.k), host_bits(st.v)
        oracle.copy_blocks(kh, vh, pairs.cpu().numpy())
        pa.copy_blocks(st.k, st.v, pairs)
        torch.cuda.synchronize(device)
        exact = bool(np.array_equal(host_bits(st.k), kh) and np.array_equal(host_bits(st.v), vh))
        ms, timing = timed(lambda: pa.copy_blocks(st.k, st.v, pairs), big=False)
        # each distinct source block is read once (the samples of a group
        # copy the same partly filled block), every destination written
        nsrc = len(np.unique(pairs[:, 0].cpu().numpy()))
        moved = 2 * (nsrc + pairs.shape[0]) * st.k[0].numel() * st.k.element_size()
        record("copy_cow", ms, timing, moved, exact)
        del st
    nb, hkv, d = 8192, 8, 128
    kp = vp = None
    if only in (None, "copy_bulk", "reshape_blocks", "reshape_scatter"):
        kp = torch.randint(-32768, 32767, (nb, hkv, 16, d), dtype=torch.int16, device=device)
        vp = torch.randint(-32768, 32767, (nb, hkv, 16, d), dtype=torch.int16, device=device)
        kp = kp.view(torch.bfloat16)
        vp = vp.view(torch.bfloat16)
    if only in (None, "copy_bulk"):
        perm = rng.permutation(nb)
        src, dst = perm[:nb // 2], perm[nb // 2:]
        pairs = torch.from_numpy(np.stack([src, dst], 1).astype(np.int64)).to(device)
        pa.copy_blocks(kp, vp, pairs)
        torch.cuda.synchronize(device)
        s_t, d_t = torch.from_numpy(src).to(device), torch.from_numpy(dst).to(device)
        exact = bool(torch.equal(bits(kp)[d_t], bits(kp)[s_t]) and
                     torch.equal(bits(vp)[d_t], bits(vp)[s_t]))
        ms, timing = timed(lambda: pa.copy_blocks(kp, vp, pairs), big=True)
        moved = 2 * 2 * len(src) * kp[0].numel() * kp.element_size()
        record("copy_bulk", ms, timing, moved, exact)
    if only in (None, "reshape_step"):
        w = make_workload("gqa8b")
        st = Step(w, device, 0)
        kh, vh = host_bits(st.k), host_bits(st.v)
        oracle.reshape_and_cache(kh, vh, host_bits(st.k_new), host_bits(st.v_new),
                                 st.slots.cpu().numpy())
        pa.reshape_and_cache(st.k_new, st.v_new, st.k, st.v, st.slots)
        torch.cuda.synchronize(device)
        exact = bool(np.array_equal(host_bits(st.k), kh) and np.array_equal(host_bits(st.v), vh))
        ms, timing = timed(lambda: pa.reshape_and_cache(st.k_new, st.v_new, st.k, st.v, st.slots),
                           big=False)
        moved = 2 * 2 * st.k_new.numel() * st.k_new.element_size()
        record("reshape_step", ms, timing, moved, exact)
        del st
    for name in ("reshape_blocks", "reshape_scatter"):
        if only not in (None, name):
            continue
        ntok = 65536
        if name == "reshape_blocks":
            blocks = rng.choice(nb, ntok // 16, replace=False).astype(np.int64)
            slots_np = (blocks[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)
        else:
            slots_np = rng.choice(nb * 16, ntok, replace=False).astype(np.int64)
        slots = torch.from_numpy(slots_np).to(device)
        kn = torch.randint(-32768, 32767, (ntok, hkv, d), dtype=torch.int16,
                           device=device).view(torch.bfloat16)
        vn = torch.randint(-32768, 32767, (ntok, hkv, d), dtype=torch.int16,
                           device=device).view(torch.bfloat16)
        pa.reshape_and_cache(kn, vn, kp, vp, slots)
        torch.cuda.synchronize(device)
        blk, off = slots // 16, slots % 16
        exact = bool(torch.equal(bits(kp)[blk, :, off, :], bits(kn)) and
                     torch.equal(bits(vp)[blk, :, off, :], bits(vn)))
        ms, timing = timed(lambda: pa.reshape_and_cache(kn, vn, kp, vp, slots), big=True)
        moved = 2 * 2 * kn.numel() * kn.element_size()
        record(name, ms, timing, moved, exact)
        del kn, vn
    del kp, vp, flush
    torch.cuda.empty_cache()
    assert pa.get_device_error() == 0
    return cases


def run_cache(args):
    """`--workload cache`: measure_cache's cases as one line whose value is
    the bulk copy's."""
    import torch
    from paged_kv_cache_260_gb300 import _build
    _build.build()
    import paged_kv_cache_260_gb300 as pa
    pa.load()
    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    peak, peak_src = measured_hbm_peak()
    steps = max(1, min(args.steps, 100))
    cases = measure_cache(args, device, args.cache_case)
    head = "copy_bulk" if "copy_bulk" in cases else next(iter(cases))
    c = cases[head]
    print(json.dumps({
        "metric": CACHE_METRIC, "value": c["gbps"], "unit": "GB/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": c["us_per_launch"] * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": CACHE_CASES[head], "case": head},
        "roofline": {"bound": "hbm", "achieved": c["gbps"], "peak": peak, "unit": "GB/s",
                     "frac": c["frac"],
                     "peak_source": (peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy burst)"
                                     if peak_src == "measured" else "fallback 6.8 TB/s"),
                     "bytes_basis": "bytes read + written per launch",
                     "traffic": c["traffic"]},
        "cases": cases,
        "parity_vs_oracle": {"bit_exact": all(x["bit_exact"] for x in cases.values())},
        "gpu_launches": steps * len(cases),
    }), flush=True)


def run_reference_cache(args):
    """The oracle's copy_blocks on the bulk case, on the host: the same
    4096 pairs of an 8192-block pool, bytes read + written over time."""
    import oracle
    nb, hkv, d = 8192, 8, 128
    rng = np.random.default_rng(1010)
    k = rng.integers(0, 65536, (nb, hkv, 16, d), dtype=np.uint16)
    v = rng.integers(0, 65536, (nb, hkv, 16, d), dtype=np.uint16)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:nb // 2], perm[nb // 2:]], 1).astype(np.int64)
    moved = 2 * 2 * (nb // 2) * hkv * 16 * d * 2
    steps = max(1, min(args.steps, 20))
    for _ in range(min(args.warmup, 2)):
        oracle.copy_blocks(k, v, pairs)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.copy_blocks(k, v, pairs)
    dt = (time.perf_counter() - t0) / steps
    value = moved / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": CACHE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
        "data": "synthetic", "config": {"workload": CACHE_CASES["copy_bulk"], "case": "copy_bulk"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "the oracle's copy_blocks, one host thread, the whole case"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


PREFILL_METRIC = ("paged chunked prefill: causal attention TFLOP/s on tcgen05 tensor cores, "
                  "% of GB300 dense bf16 peak")
PREFILL_DESCRIPTION = {
    "prefill": ("chunked prefill: 8 seqs, 32/8 heads, head_dim 128, bf16, contexts "
                "U[512,4096] ending in a 512-token chunk (4096 query rows)"),
    "prefill_long": ("chunked prefill deep into long prompts: 16 seqs, 32/8 heads, head_dim 128, "
                     "bf16, 16384-token contexts ending in a 2048-token chunk (32768 query rows)"),
}


def measured_bf16_peak(sustained: bool):
    """(TFLOP/s, source) from MEASURED_PEAKS.json: the cuBLAS bf16 burst figure
    for a kernel timed alone, the sustained one (seconds under the power cap)
    for a long timed region; else the fallbacks (1.9 / 1.7 PFLOP/s)."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), f"measured (MEASURED_PEAKS.json {key})"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def prefill_flops(w, rows=None):
    """Algorithmic flops of a causal chunked prefill (2 for q.k and 2 for p.v per
    visible key, channel and head); rows: only the last `rows` rows of each chunk."""
    total = 0
    for s in range(w.num_seqs):
        c = int(w.query_start[s + 1] - w.query_start[s])
        L = int(w.seq_lens[s])
        r = c if rows is None else min(rows, c)
        # rows i = c-r .. c-1 see L-c+i+1 keys
        total += sum(L - c + i + 1 for i in range(c - r, c))
    return 4 * w.head_dim * w.num_heads * total


def prefill_oracle_rows(w, rows):
    """The query rows of a prefill sample: the last `rows` rows of every chunk
    (a prefill whose chunks are those rows, over the same contexts).
    Returns (row indices, query starts of the sample)."""
    idx, qs = [], [0]
    for s in range(w.num_seqs):
        a, b = int(w.query_start[s]), int(w.query_start[s + 1])
        r = min(rows, b - a)
        idx.extend(range(b - r, b))
        qs.append(qs[-1] + r)
    return idx, np.array(qs, np.int32)


def prefill_oracle_sample(w, budget_s: float):
    """The oracle's prefill step on the host cores: the fp64 oracle on the last
    r rows of every chunk, r the most rows whose call fits `budget_s` (one
    row timed first).  cpu_baseline and --impl reference use this same step.
    Returns (run, flops per step, threads, text, row indices)."""
    import oracle
    oracle.build()
    threads = min(oracle.num_threads(), w.num_seqs)

    def make(rows):
        idx, qs = prefill_oracle_rows(w, rows)
        q = np.ascontiguousarray(w.q[idx])
        return (lambda: oracle.prefill(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, qs,
                                       w.scale, w.dtype, threads=threads)), idx

    run1, _ = make(1)
    run1()
    t0 = time.perf_counter()
    run1()
    one = max(1e-4, time.perf_counter() - t0)
    max_chunk = int(np.diff(w.query_start).max())
    rows = int(max(1, min(max_chunk, budget_s / one)))
    run, idx = make(rows)
    text = (f"fp64 oracle prefill of the last {rows} rows of each of the {w.num_seqs} chunks "
            f"per step ({len(idx)} rows x {w.num_heads} heads), {threads} host threads")
    return run, prefill_flops(w, rows), threads, text, idx


def prefill_cpu_baseline(w, steps: int, warmup: int, budget_s: float = 10.0):
    """The oracle's prefill step (prefill_oracle_sample, sized as --impl
    reference sizes it) repeated for ~budget_s."""
    run, flops, threads, text, _ = prefill_oracle_sample(
        w, max(0.05, min(2.0, 90.0 / max(1, steps + warmup))))
    reps = 0
    t0 = time.perf_counter()
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": flops * reps / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": f"{text}; {reps} steps in {dt:.1f} s"}


def prefill_parity(w, out, rows=32):
    """The last `rows` rows of every chunk of the timed prefill's output
    against the oracle's."""
    import oracle
    oracle.build()
    idx, qs = prefill_oracle_rows(w, rows)
    ref = oracle.prefill(np.ascontiguousarray(w.q[idx]), w.k_cache, w.v_cache, w.block_tables,
                         w.seq_lens, qs, w.scale, w.dtype,
                         threads=min(oracle.num_threads(), w.num_seqs))
    got = out.float().cpu().numpy().astype(np.float64)[idx]
    err = float(np.abs(got - ref).max())
    tol = 4e-3 if w.dtype == "f16" else 1.6e-2
    return {"max_abs_err": err, "rows": len(idx), "tolerance": tol,
            "ok": bool(np.isfinite(got).all() and err <= tol)}


def run_prefill(args):
    """One pa_prefill (plan + kernel) per step on the chunked-prefill workload,
    each launch timed with CUDA events and L2 flushed between launches."""
    import torch
    from paged_kv_cache_260_gb300 import _build
    _build.build()
    import paged_kv_cache_260_gb300 as pa
    import synth
    pa.load()
    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    w = synth.by_name(args.workload)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)

    q, k, v = dev(w.q), dev(w.k_cache), dev(w.v_cache)
    tables = torch.from_numpy(w.block_tables).to(device)
    lens = torch.from_numpy(w.seq_lens).to(device)
    qs = torch.from_numpy(w.query_start).to(device)
    out = torch.empty_like(q)
    mq = int(np.diff(w.query_start).max())
    ws = torch.empty(pa.prefill_workspace_size(w.num_seqs, mq, w.num_heads, w.num_kv_heads),
                     dtype=torch.uint8, device=device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    flops = prefill_flops(w)

    def call():
        pa.prefill(out, q, k, v, tables, lens, qs, mq, w.scale, workspace=ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(device)
    assert pa.get_device_error() == 0
    steps = max(3, min(args.steps, 200))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        for e0, e1 in ev:
            flush.zero_()                      # K/V (90 MB) would otherwise stay in L2
            e0.record()
            call()
            e1.record()
        torch.cuda.synchronize(device)
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    assert pa.get_device_error() == 0
    value = flops / (ms * 1e-3) / 1e12
    # a timed region of seconds runs under the power cap: compare it with the
    # sustained peak, a short one with the burst peak
    peak, peak_src = measured_bf16_peak(sustained=ms * steps > 500.0)

    # end to end through the public API (pipelined_e2e): q, tables, lengths
    # and query starts from pinned host memory, the output back to it, every
    # step, with the L2 flush ahead of each step as above
    cur = {}

    def bind(views, out_buf):
        cur["q"], cur["tables"], cur["lens"], cur["qs"] = views
        cur["out"] = out_buf

    def e2e_step():
        pa.prefill(cur["out"], cur["q"], k, v, cur["tables"], cur["lens"], cur["qs"], mq,
                   w.scale, workspace=ws)

    e2e_steps = max(3, min(steps, 50))
    e2e_ms, h2d, d2h, last = pipelined_e2e([q, tables, lens, qs], out, bind, e2e_step, e2e_steps,
                                           device, before=flush.zero_)
    call()
    torch.cuda.synchronize(device)
    if not torch.equal(out.cpu(), last):
        raise RuntimeError("the pipelined end-to-end prefill's output differs from the "
                           "device-resident one's")
    cpu = None
    parity = None
    if not args.no_cpu_baseline:
        cpu = prefill_cpu_baseline(w, args.steps, args.warmup)
        parity = prefill_parity(w, out)
    print(json.dumps({
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": PREFILL_DESCRIPTION[args.workload], "name": args.workload,
                   "l2": "flushed (256 MB write) before every timed launch",
                   "flops": "causal: 4 * head_dim * heads * visible keys per row"},
        "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / peak,
                     "traffic": ncu_traffic(args.workload, "prefill_dram_traffic.txt",
                                            PREFILL_SOURCES),
                     "peak_source": peak_src + ", cuBLAS bf16 GEMM",
                     "timed_device_ms": ms * steps},
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "cpu_baseline": cpu,
        "parity_vs_oracle": parity,
        "clocks": clk.summary(),
        "gpu_launches": 2 * steps,
    }), flush=True)


def run_reference(args):
    """The oracle as the reference arm: W untimed and K timed steps of the
    oracle's step (oracle_sample: one fp64 decode call over the first n
    sequences, sized so that the whole run takes about two minutes), the same
    step cpu_baseline times in our arm's line."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = make_workload(args.workload or "gqa8b", 0)
    k, v = oracle_pool_after_step(w)
    run, nbytes, threads, text = oracle_sample(w, k, v,
                                               oracle_step_budget(args.steps, args.warmup))
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    name = args.workload or "gqa8b"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTION[name], "name": name},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": text},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference_prefill(args):
    """The oracle as the reference arm of the prefill line: W untimed and K
    timed steps of the oracle's prefill step (prefill_oracle_sample), sized so
    that the whole run takes about 90 s."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth
    w = synth.by_name(args.workload)
    run, flops, threads, text, _ = prefill_oracle_sample(
        w, max(0.05, min(2.0, 90.0 / max(1, args.steps + args.warmup))))
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = flops * args.steps / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL_DESCRIPTION[args.workload], "name": args.workload},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": text},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(DESCRIPTION) + ["swap", "cache", "prefill",
                                                              "prefill_long"],
                    default=None,
                    help="one workload alone (default: the GQA batch-128 headline, with the "
                         "other decode workloads nested in the same line)")
    ap.add_argument("--partition", type=int, default=None,
                    help="-1 no split, 0 balanced split, >0 fixed partition tokens")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle legs (cpu_baseline and parity)")
    ap.add_argument("--no-l2-check", action="store_true")
    ap.add_argument("--no-other-decode", action="store_true",
                    help="parallel sampling: skip timing the other decode beside it")
    ap.add_argument("--shared-prefix", choices=["auto", "on", "off"], default="auto",
                    help="parallel sampling: pa_decode_shared_prefix (on) or pa_decode_append "
                         "(off); auto: on for the long-prompt workload")
    ap.add_argument("--only-headline", action="store_true")
    ap.add_argument("--cache-case", choices=list(CACHE_CASES), default=None,
                    help="--workload cache: one case alone (for a profiler)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if args.workload and args.workload.startswith("prefill"):
            run_reference_prefill(args)
        elif args.workload == "swap":
            print(json.dumps({"impl": "reference", "unavailable": "swap_blocks moves bytes "
                              "between memories; the oracle has no timed counterpart"}))
        elif args.workload == "cache":
            run_reference_cache(args)
        else:
            run_reference(args)
    elif args.workload == "swap":
        run_swap(args)
    elif args.workload == "cache":
        run_cache(args)
    elif args.workload and args.workload.startswith("prefill"):
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
