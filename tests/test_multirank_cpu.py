"""The benchmark's multi-process path on CPU: two gloo ranks (no GPU).

Each rank runs an independent replica of the step (the forward has no exchange step), so the
only cross-rank operations are the barrier and the maximum of the ranks' times; the whole-job
value is the work of all ranks over that maximum.  The reference arm prints from rank 0 only.
"""
import json
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r took 1 + r seconds: every rank must see the slowest, 2 s
        slowest = bench.max_over_ranks(dist, 1.0 + rank, "cpu")
        out[rank] = (slowest, bench.whole_job_tflops(1e12, 10, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # both ranks: max time 2 s; value = 2 ranks x 1 TFLOP x 10 steps / 2 s = 10 TFLOP/s
    assert res == {0: (2.0, 10.0), 1: (2.0, 10.0)}


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.whole_job_tflops(2e12, 5, 1, 2.0) == 5.0


def _reference_rank(rank, world, out):
    import contextlib
    import io
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.WORKLOAD = "tiny_double_f32"  # the same code path on the small workload
    args = bench.argparse.Namespace(steps=1, warmup=3, impl="reference", gpus=world)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)
    out[rank] = buf.getvalue()


def test_reference_arm_prints_from_rank_zero_only():
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_reference_rank, args=(2, out), nprocs=2, join=True)
        res = dict(out)
    assert res[1] == ""
    lines = [ln for ln in res[0].splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res[0]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
