"""The benchmark's multi-process path on CPU: world_size-2 gloo ranks.

Every rank runs its own replica (independent sequences, its own seed); only
timing and byte counts cross ranks: the step time is the max over ranks and
the bytes are summed.  No data-path collective exists.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    bench.dist_init("gloo")
    w = bench.make_workload("tiny", rank)
    t = 1.0 + rank                                  # rank 1 is "slower"
    q.put((rank, bench.dist_max(t), bench.dist_sum(w.kv_read_bytes()), w.kv_read_bytes(),
           bench.replica_seed(1001, rank), w.seq_lens.tolist()))
    bench.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, max0, sum0, b0, seed0, lens0), (r1, max1, sum1, b1, seed1, lens1) = res
    assert max0 == max1 == 2.0
    assert sum0 == sum1 == b0 + b1
    assert seed0 != seed1 and lens0 != lens1        # independent replicas


def test_steps_per_graph_divides_steps():
    sys.path.insert(0, ROOT)
    import bench
    for k in (1, 7, 10, 64, 20000, 97):
        d = bench.pick_steps_per_graph(k)
        assert k % d == 0 and 1 <= d <= 32


def _bench_line(*args):
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_reference_arm_lines_on_cpu():
    # the oracle's copy_blocks on the bulk pool case: the contract's keys,
    # its own e2e and cpu_baseline, no GPU needed
    d = _bench_line("--impl", "reference", "--workload", "cache", "--steps", "1",
                    "--warmup", "1")
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["case"] == "copy_bulk"
    # swapping has no oracle timing: an `unavailable` line, exit 0
    d = _bench_line("--impl", "reference", "--workload", "swap")
    assert d["impl"] == "reference" and "unavailable" in d
