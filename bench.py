"""Benchmark of one paged-decode step on GB300.

A step is one pass of the whole hot path over one batch: copy_blocks (if the
workload has copy-on-write pairs), reshape_and_cache (if it appends a token)
and the decode (with its split-K merge).  The default workload is the GQA
batch-128 decode (128 sequences, 32 query / 8 kv heads, head_dim 128, bf16,
lognormal lengths); ``--workload`` picks another.

Prints ONE JSON line (rank 0):
  value      effective KV-read GB/s of the whole job: sum over ranks of the
             K/V bytes a step must read (every live token, every kv head)
             divided by the step time (max over ranks)
  e2e        the same metric through the public API with host buffers: each
             step copies its inputs from pinned host memory and reads the
             output back inside the timed region, the copies on their own
             streams and double-buffered so that they overlap the
             neighbouring steps' compute, as a serving loop runs
  roofline   the decode kernel's achieved bytes/s against measured HBM peak
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample

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
DEFAULT_PARTITION = {"tiny": 0, "mha7b": 0, "gqa8b": 0, "long": 512, "parsamp": 0}
DESCRIPTION = {
    "tiny": "tiny decode: 4 seqs, 8/8 heads, head_dim 64, fp16, lens U[1,100], 64-block pool, +1 token",
    "mha7b": "MHA 7B-shaped decode: 64 seqs, 32/32 heads, head_dim 128, fp16, lens U[512,2048]",
    "gqa8b": ("GQA 8B-shaped decode: 128 seqs, 32/8 heads, head_dim 128, bf16, lens "
              "lognormal(median 600, sigma 1) clipped [16,4096], +1 token per seq via slot_mapping"),
    "long": ("long-context split-K decode: 4 seqs, 32/8 heads, head_dim 128, bf16, lens "
             "{32768,65536,98304,131072}, 512-token partitions + log-sum-exp merge"),
    "parsamp": ("parallel sampling: 16 prompts x 8 samples, 40/8 heads, head_dim 128, fp16, "
                "1024 shared prompt tokens + U[0,256] + 1, 112 copy-on-write pairs per step"),
}


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
    base = {"tiny": 1001, "mha7b": 1002, "gqa8b": 1003, "long": 1004, "parsamp": 1005}[name]
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


DECODE_SOURCES = ("pa_decode_mma.cuh", "pa_schedule.cuh", "pa_device.cuh", "pa_internal.h")
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
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu summary, if it was taken on the current kernel sources
    (else None)."""
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

    def __init__(self, w, device, partition_size):
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
        self.ws = pa.workspace_for(self.q, self.k, self.tables, partition_size)
        self.launches_per_step = self._count_launches()
        self.graph = None
        self.ev = None

    def _count_launches(self):
        n = 1                                           # decode (append fused in)
        n += int(self.pairs is not None)                # copy_blocks
        if self.ps >= 0:
            n += 1                                      # merge of cut runs / partitions
        if self.ps > 0 and self.tables.shape[1] * 16 > self.ps:
            n += 1                                      # merge of partitions per run
        return n

    def run(self, ev_pair=None):
        """Enqueue one step on the current stream; ev_pair brackets the decode."""
        pa = self.pa
        if self.pairs is not None:
            pa.copy_blocks(self.k, self.v, self.pairs)
        if ev_pair is not None:
            ev_pair[0].record()
        if self.slots is not None:
            # reshape_and_cache of the newest token fused into the decode launch
            pa.decode_append(self.out, self.q, self.k, self.v, self.tables, self.lens, self.k_new,
                             self.v_new, self.slots, self.w.scale, partition_size=self.ps,
                             workspace=self.ws)
        else:
            pa.decode(self.out, self.q, self.k, self.v, self.tables, self.lens, self.w.scale,
                      partition_size=self.ps, workspace=self.ws)
        if ev_pair is not None:
            ev_pair[1].record()

    def capture(self, steps_per_graph: int):
        """Capture `steps_per_graph` steps twice: `graph` runs them back to
        back, `graph_ev` with an event pair around each decode call.

        External events become event-record nodes of a graph, so each replay
        of `graph_ev` timestamps every decode.  A record node between two
        kernels also cuts the programmatic dependency between them (the next
        step's decode could otherwise be scheduled while this step's merge
        drains), so the timed steps replay `graph`, save for one replay of
        `graph_ev` at the end."""
        import torch
        self.ev = [(timing_event(), timing_event()) for _ in range(steps_per_graph)]
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            for _ in range(2):
                self.run()
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps_per_graph):
                self.run()
        self.graph = g
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps_per_graph):
                self.run(self.ev[i])
        self.graph_ev = g

    def decode_ms(self):
        """Mean decode duration (ms) over the events of the last graph replay."""
        return float(np.mean([a.elapsed_time(b) for a, b in self.ev]))


def timing_event():
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:                      # torch without external events
        return None


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


def cpu_baseline(w, budget_s: float = 12.0, threads: int = 0):
    """The fp64 oracle on a bounded sample: whole sequences in order, repeated
    until ~budget_s of CPU work, on `threads` host threads (0: all cores);
    returns (GB/s of KV processed, sample text, cores, {sequence: oracle
    output row} of the first pass)."""
    import oracle
    oracle.build()
    threads = threads or oracle.num_threads()
    k, v = w.k_cache.copy(), w.v_cache.copy()
    t0 = time.perf_counter()
    if w.block_mapping is not None and len(w.block_mapping):
        oracle.copy_blocks(k, v, w.block_mapping)
    if w.slot_mapping is not None:
        oracle.reshape_and_cache(k, v, w.k_new, w.v_new, w.slot_mapping)
    per_seq = 2 * w.num_kv_heads * w.head_dim * 2
    done_bytes, seqs, reps = 0, 0, 0
    chunk = max(1, threads // 2)
    rows = {}
    while True:
        for s0 in range(0, w.num_seqs, chunk):
            sel = list(range(s0, min(w.num_seqs, s0 + chunk)))
            out = oracle.decode(w.q, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype,
                                seqs=sel, threads=threads)
            if reps == 0:
                for s in sel:
                    rows[s] = out[s]
            done_bytes += int(sum(int(w.seq_lens[s]) for s in sel)) * per_seq
            seqs += len(sel)
            if time.perf_counter() - t0 > budget_s:
                break
        else:
            reps += 1
            if time.perf_counter() - t0 < budget_s:
                continue
        break
    dt = time.perf_counter() - t0
    sample = (f"fp64 oracle step (copy/reshape once, then decode of {seqs} sequences in order, "
              f"{reps} full passes) in {dt:.1f} s")
    return done_bytes / dt / 1e9, sample, threads, rows


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


def e2e_measure(st, steps: int, device, flush=None):
    """The decode step end to end (pipelined_e2e): q, tables, lengths, the new
    tokens, their slots and the copy-on-write pairs come in from one packed
    pinned host buffer, the output goes back.  `flush`, when given, is
    zeroed ahead of every step, as the device-resident timing does for
    working sets that L2 could hold.  The last step's host output must equal
    the device-resident step's, bit for bit.  Returns (ms per step, h2d
    bytes, d2h bytes)."""
    import torch
    names = [n for n in ["q", "tables", "lens", "k_new", "v_new", "slots", "pairs"]
             if getattr(st, n) is not None]
    saved = [getattr(st, n) for n in names]
    saved_out = st.out

    def bind(views, out_buf):
        for n, v in zip(names, views):
            setattr(st, n, v)
        st.out = out_buf

    try:
        ms, h2d, d2h, last = pipelined_e2e(saved, saved_out, bind, st.run, steps, device,
                                           before=None if flush is None else flush.zero_)
    finally:
        bind(saved, saved_out)
    st.run()
    torch.cuda.synchronize(device)
    if not torch.equal(st.out.cpu(), last):
        raise RuntimeError("the pipelined end-to-end step's output differs from the "
                           "device-resident step's")
    return ms, h2d, d2h


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

    ps = DEFAULT_PARTITION[args.workload] if args.partition is None else args.partition
    w = make_workload(args.workload, rank)
    st = Step(w, device, ps)
    kv_bytes = w.kv_read_bytes()
    # blocks shared between sequences (parallel sampling) are read once per
    # step from HBM at best; the L2 decision and the HBM figure use them once
    unique_bytes = w.unique_kv_read_bytes()
    l2_ok = unique_bytes > 2 * L2_BYTES
    spg = pick_steps_per_graph(args.steps)
    use_graph = timing_event() is not None and not args.no_graph
    if use_graph:
        st.ev = None
        st.capture(spg)
        replays = args.steps // spg
        for _ in range(max(1, -(-args.warmup // spg))):
            st.graph.replay()
        st.graph_ev.replay()
    else:
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for _ in range(args.warmup):
            st.run()
    torch.cuda.synchronize(device)
    assert pa.get_device_error() == 0, "a kernel recorded an error during warm-up"

    flush = None if l2_ok else torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    dec_ms = []
    with ClockSampler(physical_gpu_index(local)) as clk:
        barrier(device)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if flush is None:
            t0.record()
            if use_graph:
                # the last replay is the graph with an event pair around each
                # call, whose timestamps give the roofline its call durations
                for _ in range(replays - 1):
                    st.graph.replay()
                st.graph_ev.replay()
            else:
                for _ in range(args.steps):
                    st.run(ev)
            t1.record()
            torch.cuda.synchronize(device)
            elapsed = t0.elapsed_time(t1)
            dec_ms.append(st.decode_ms() if use_graph else ev[0].elapsed_time(ev[1]))
        else:
            # small working set: flush L2 before every step, time the steps only
            elapsed = 0.0
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps):
                flush.zero_()
                t0.record()
                st.run(ev)
                t1.record()
                torch.cuda.synchronize(device)
                elapsed += t0.elapsed_time(t1)
                dec_ms.append(ev[0].elapsed_time(ev[1]))
        barrier(device)
    assert pa.get_device_error() == 0, "a kernel recorded an error in the timed region"
    t_max = dist_max(elapsed, device)
    ms_per_step = t_max / args.steps
    total_bytes = dist_sum(kv_bytes, device)
    total_seqs = dist_sum(w.num_seqs, device)
    value = total_bytes / (ms_per_step * 1e-3) / 1e9
    dec = float(np.mean(dec_ms))

    e2e_ms, h2d, d2h = e2e_measure(st, max(20, min(args.steps, 300)), device, flush)
    e2e_ms = dist_max(e2e_ms, device)
    peak, peak_src = measured_hbm_peak()
    achieved = kv_bytes / (dec * 1e-3) / 1e9
    traffic = ncu_traffic(args.workload)
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample, cores, rows = cpu_baseline(w)
        cpu = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        if args.workload == "tiny":
            v1, sample1, _, _ = cpu_baseline(w, budget_s=3.0, threads=1)
            cpu["single_core"] = {"value": v1, "unit": "GB/s", "cores": 1, "sample": sample1}
        # the timed step's own output against the oracle rows the sample computed
        got = st.out.float().cpu().numpy().astype(np.float64)
        err = max(float(np.abs(got[s] - r).max()) for s, r in rows.items())
        parity = {"max_abs_err": err, "sequences": len(rows),
                  "tolerance": 4e-3 if w.dtype == "f16" else 1.6e-2, "ok": err <= (4e-3 if w.dtype == "f16" else 1.6e-2)}
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V, random block permutation)",
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "unique_gbps": dist_sum(unique_bytes, device) / (ms_per_step * 1e-3) / 1e9,
        "seqs_per_s": total_seqs / (ms_per_step * 1e-3),
        "config": {
            "workload": DESCRIPTION[args.workload],
            "name": args.workload,
            "num_seqs": w.num_seqs, "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": 16, "partition_size": ps,
            "kv_bytes_per_step": kv_bytes,
            "unique_kv_bytes_per_step": unique_bytes,
            "step": ("copy_blocks + " if w.block_mapping is not None else "")
                    + ("decode with reshape_and_cache fused (pa_decode_append)"
                       if w.slot_mapping is not None else "decode") + " + merge",
            "l2": ("inputs larger than L2 (KV read per step %.0f MB vs 129 MB L2)" % (unique_bytes / 1e6)
                   if l2_ok else "L2 flushed (258 MB write) before every step; steps timed alone"),
            "timing": ("CUDA graph of %d steps back to back, replayed %d times, CUDA events around "
                       "the replays; the last replay has an event pair around each call, which "
                       "gives the roofline its call duration" % (spg, args.steps // spg)
                       if use_graph and l2_ok else "CUDA events per step"),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "roofline": {"bound": "hbm", "kernel": "decode_mma_kernel + merge kernel(s) (one pa_decode / pa_decode_append call)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy burst)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": kv_bytes, "decode_ms": dec,
                     "traffic": traffic},
        "cpu_baseline": cpu,
        "parity_vs_oracle": parity,
        "pool_utilisation": pool_utilisation(w),
        "gpu_launches": st.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
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


def prefill_cpu_baseline(w, rows=32):
    """The fp64 oracle on the last `rows` rows of every chunk (a prefill whose
    chunks are those rows, over the same contexts)."""
    import oracle
    oracle.build()
    threads = min(oracle.num_threads(), w.num_seqs)
    idx = []
    qs = [0]
    for s in range(w.num_seqs):
        a, b = int(w.query_start[s]), int(w.query_start[s + 1])
        r = min(rows, b - a)
        idx.extend(range(b - r, b))
        qs.append(qs[-1] + r)
    q = np.ascontiguousarray(w.q[idx])
    t0 = time.perf_counter()
    ref = oracle.prefill(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                         np.array(qs, np.int32), w.scale, w.dtype, threads=threads)
    dt = time.perf_counter() - t0
    sample = (f"fp64 oracle prefill of the last {rows} rows of each of the {w.num_seqs} chunks "
              f"({len(idx)} rows x {w.num_heads} heads) in {dt:.1f} s")
    return prefill_flops(w, rows) / dt / 1e12, sample, threads, (idx, ref)


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
        cv, sample, cores, (idx, ref) = prefill_cpu_baseline(w)
        cpu = {"value": cv, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
        got = out.float().cpu().numpy().astype(np.float64)[idx]
        err = float(np.abs(got - ref).max())
        tol = 4e-3 if w.dtype == "f16" else 1.6e-2
        parity = {"max_abs_err": err, "rows": len(idx), "tolerance": tol, "ok": err <= tol}
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
    """The oracle as the reference arm: W untimed and K timed steps, each a
    bounded sample of the workload (its first sequences in order, or a prefix
    of the first sequence when one sequence is more than a step's share),
    sized so that the whole run takes about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = make_workload(args.workload, 0)
    per_seq = 2 * w.num_kv_heads * w.head_dim * 2
    budget = 120.0 / max(1, args.steps + args.warmup)   # seconds per step
    # small samples run on one thread: starting threads would dominate them
    threads = 1 if budget < 0.05 else oracle.num_threads()

    def run(sel, lens):
        oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale, w.dtype,
                      seqs=sel, threads=threads)

    lens = w.seq_lens.copy()

    def timed(n):
        t0 = time.perf_counter()
        run(list(range(n)), lens)
        return time.perf_counter() - t0

    # the largest prefix of sequences whose sample fits a step's share
    # (timed, since lengths differ): doubling, then bisection
    run([0], lens)                                       # first call: library and pages
    one = timed(1)
    if one > budget:
        lens[0] = max(1, int(int(w.seq_lens[0]) * budget / one))
        n = 1
        sample = f"fp64 oracle decode of the first {int(lens[0])} tokens of sequence 0 per step"
    else:
        lo, hi = 1, 1
        while hi < w.num_seqs:
            hi = min(w.num_seqs, 2 * hi)
            if timed(hi) > budget:
                break
            lo = hi
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if timed(mid) > budget:
                hi = mid
            else:
                lo = mid
        n = lo
        sample = f"fp64 oracle decode of sequences 0..{n - 1} of the workload per step"
    sel = list(range(n))
    for _ in range(args.warmup):
        run(sel, lens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(sel, lens)
    dt = time.perf_counter() - t0
    b = sum(int(lens[s]) for s in sel) * per_seq
    value = b * args.steps / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTION[args.workload], "name": args.workload},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference_prefill(args):
    """The oracle as the reference arm of the prefill line: W untimed and K
    timed steps, each the fp64 oracle on the last r rows of every chunk, r
    sized so that the whole run takes about 90 s."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    oracle.build()
    w = synth.by_name(args.workload)
    threads = min(oracle.num_threads(), w.num_seqs)
    budget = max(0.05, 90.0 / max(1, args.steps + args.warmup))   # seconds per step

    def sample(rows):
        idx, qs = [], [0]
        for s in range(w.num_seqs):
            a, b = int(w.query_start[s]), int(w.query_start[s + 1])
            r = min(rows, b - a)
            idx.extend(range(b - r, b))
            qs.append(qs[-1] + r)
        q = np.ascontiguousarray(w.q[idx])
        qs = np.array(qs, np.int32)
        return lambda: oracle.prefill(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, qs,
                                      w.scale, w.dtype, threads=threads)

    t0 = time.perf_counter()
    sample(1)()
    one = max(1e-4, time.perf_counter() - t0)
    max_chunk = int(np.diff(w.query_start).max())
    rows = int(max(1, min(max_chunk, budget / one)))
    step = sample(rows)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = prefill_flops(w, rows) * args.steps / dt / 1e12
    text = (f"fp64 oracle prefill of the last {rows} rows of each of the {w.num_seqs} chunks "
            f"per step")
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
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(DESCRIPTION) + ["swap", "prefill", "prefill_long"],
                    default="gqa8b")
    ap.add_argument("--partition", type=int, default=None,
                    help="-1 no split, 0 balanced split, >0 fixed partition tokens")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if args.workload.startswith("prefill"):
            run_reference_prefill(args)
        elif args.workload == "swap":
            print(json.dumps({"impl": "reference", "unavailable": "swap_blocks moves bytes "
                              "between memories; the oracle has no timed counterpart"}))
        else:
            run_reference(args)
    elif args.workload == "swap":
        run_swap(args)
    elif args.workload.startswith("prefill"):
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
