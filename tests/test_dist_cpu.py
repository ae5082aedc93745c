"""Multi-process path of bench.py on CPU (gloo, world size 2): the barrier, the
max-over-ranks timing reduction (the only cross-rank operation: the data path has
no collective), distinct per-rank batches, and the reference arm running on rank 0
only."""
import io
import os
import socket
import contextlib

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r = bench.dist_init("gloo")
    bench.barrier()
    t = bench.max_over_ranks(1.0 + rank)       # each rank's "time"
    seeds = bench.rank_seed_offset(r)
    w = dict(bench.WORKLOADS["c1"])
    from attention_gemms_gb300 import synth
    x0 = synth.normal((4, 8), synth.seed_of(w["cfg"], "X") + seeds, 1.0, "f32")
    bench.barrier()
    q.put((r, ws, t, x0.tolist()))
    dist.destroy_process_group()


def test_two_rank_timing_and_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, t0, x0), (r1, w1, t1, x1) = out
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert t0 == t1 == 2.0                 # both ranks see the slowest rank's time
    assert not np.array_equal(x0, x1)       # each replica has its own batch


def test_reference_arm_only_on_rank0(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "c1", "--steps", "1", "--warmup", "0"])
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "c1", "--steps", "1", "--warmup", "0",
                    "--ref-rows", "8"])
    import json
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
