"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The hot path does not shard: `bench.py --gpus N` runs N replicas of the
one-GPU workload with no data-path collective.  What the N > 1 launch adds
is host logic, tested here with two gloo ranks on 127.0.0.1:
  - the timed region's barrier, and the maximum (time) and sum (work) over
    ranks that the reported value is built from;
  - the reference arm under a multi-rank launch: rank 0 alone runs the
    oracle and prints one JSON line, the other rank exits without work.
"""
import contextlib
import io
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, case, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    try:
        if case == "reduce":
            bench.maybe_init_dist(ws, "gloo")
            bench.barrier(ws)
            mx = bench.max_over_ranks(1.5 + rank, ws, "cpu")
            sm = bench.sum_over_ranks(10.0 * (rank + 1), ws, "cpu")
            bench.barrier(ws)
            q.put((rank, mx, sm))
            dist.destroy_process_group()
        else:
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                bench.main(["--impl", "reference", "--gpus", str(ws), "--steps", "1",
                            "--warmup", "3"])
            q.put((rank, buf.getvalue()))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, f"error: {e!r}"))


def _run(case, ws=2, timeout=240):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, case, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(ws):
            item = q.get(timeout=timeout)
            out[item[0]] = item[1:]
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return out


def test_max_and_sum_over_two_gloo_ranks():
    out = _run("reduce")
    for rank in (0, 1):
        mx, sm = out[rank]
        assert mx == pytest.approx(2.5)   # max(1.5, 2.5): the slowest rank's time
        assert sm == pytest.approx(30.0)  # 10 + 20: the work of both replicas


def test_reference_arm_prints_on_rank_zero_only():
    out = _run("reference")
    lines0 = [l for l in out[0][0].splitlines() if l.strip().startswith("{")]
    assert len(lines0) == 1, out[0][0]
    rec = json.loads(lines0[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    assert out[1][0].strip() == "", out[1][0]
