"""The benchmark's N > 1 logic on CPU (gloo, world size 2): each rank holds an
independent replica (no data-path collective), the step time is the max over
ranks, and the reference arm runs on rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    assert dist.get_backend() == "gloo"
    got = bench.reduce_max(1.5 + rank, w)
    b = bench.barrier_fn(w)
    b()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny_verify", "--steps", "3",
                    "--warmup", "3", "--gpus", str(world)])
    dist.destroy_process_group()
    q.put((rank, got, buf.getvalue()))


def test_two_rank_timing_reduction_and_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, max0, out0), (r1, max1, out1) = res
    assert max0 == max1 == 2.5
    assert out1.strip() == ""                   # rank 1 does no reference work
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_algorithmic_counts_of_the_tiny_case():
    sys.path.insert(0, ROOT)
    import bench
    import synthetic
    wl = synthetic.make_workload("tiny_verify")
    alg = bench.algorithmic(wl)
    # kv tokens 42 + 75, 2 KV heads, d 64, bf16, K and V
    assert alg["kv_bytes"] == (42 + 75) * 2 * 64 * 2 * 2
    # visible pairs: each request 5 tokens x 37/70 prefix + 15 causal draft pairs, 4 heads
    assert alg["flops"] == 4 * 64 * 4 * (5 * 37 + 15 + 5 * 70 + 15)
    assert alg["tokens"] == 10
