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


def _dropout_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), TP_DIST_TIMEOUT_S="10")
    import time
    bench.dist_init("gloo")
    bench.barrier()                     # step 1, both ranks
    bench.max_over_ranks(1.0)
    if rank == 1:                       # leaves between steps, nothing in flight
        q.put((1, "left", 0.0))
        q.close()
        q.join_thread()                 # the message is out before the process ends
        os._exit(0)
    time.sleep(0.5)
    for name, call in (("barrier", bench.barrier), ("max_over_ranks", lambda: bench.max_over_ranks(2.0))):
        t0 = time.monotonic()
        try:
            call()
            q.put((0, name + ": no error", time.monotonic() - t0))
        except Exception as e:         # noqa: BLE001 -- any error is the expected outcome
            q.put((0, name + ": " + type(e).__name__, time.monotonic() - t0))
    q.close()
    q.join_thread()
    os._exit(0)


def test_rank_leaving_between_steps_fails_the_survivor_in_bounded_time():
    """A rank leaves between two steps (the launch of `torchrun --nproc_per_node=2` on
    the pages); the other rank's next barrier and timing reduction must raise within
    the process-group timeout rather than wait forever."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dropout_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = [q.get(timeout=120) for _ in range(3)]
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    left = [g for g in got if g[0] == 1]
    surv = {g[1].split(":")[0]: g for g in got if g[0] == 0}
    assert left and left[0][1] == "left"
    for name in ("barrier", "max_over_ranks"):
        _, msg, dt = surv[name]
        assert "no error" not in msg, msg
        assert dt < 60.0, (name, dt)
