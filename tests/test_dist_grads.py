"""The token-sharded backward reduction on two CPU ranks (gloo, 127.0.0.1).

The batch's tokens are split across ranks (bit_nf4_quantized_35_b300.dist):
each rank computes the backward of its own rows -- here the fp64 oracle is
the per-rank compute, standing in for a GPU -- and the partial dA, dB are
summed with one all-reduce.  The result must equal the full-batch oracle's
dA and dB within the parity tolerance, and every rank's dX rows must equal
the full-batch oracle's rows exactly (rows are independent)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SHAPE = dict(N=264, K=320, M=97, r=8, alpha=16.0)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from bit_nf4_quantized_35_b300 import inputs
    from oracle import oracle
    shape = inputs.LinearShape("shard", **SHAPE)
    d = {k: v.float().numpy() for k, v in inputs.linear_inputs(shape).items()}
    w_hat = oracle.dequant_f32(oracle.quantize_nf4(d["W"], 64, 256, want_idx=False))
    return d, w_hat


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from bit_nf4_quantized_35_b300 import dist as qdist
    from oracle import oracle
    try:
        dist.init_process_group("gloo", rank=rank, world_size=ws)
        d, w_hat = _inputs()
        m0, m1 = qdist.token_shard(SHAPE["M"], ws, rank)
        ref = oracle.linear_bwd(d["x"][m0:m1], d["dY"][m0:m1], w_hat, d["A"], d["B"],
                                SHAPE["alpha"])
        dA = torch.from_numpy(ref["dA"].astype(np.float32))
        dB = torch.from_numpy(ref["dB"].astype(np.float32))
        qdist.allreduce_lora_grads(dA, dB)
        q.put((rank, m0, m1, dA.numpy(), dB.numpy(), ref["dX"]))
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, f"error: {e!r}"))


def test_token_shards_cover_the_batch():
    from bit_nf4_quantized_35_b300.dist import token_shard
    for M in (0, 1, 7, 97, 2048):
        for world in (1, 2, 3, 8):
            spans = [token_shard(M, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == M
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_sharded_backward_allreduce_equals_full_batch():
    sys.path.insert(0, ROOT)
    from oracle import oracle
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(ws):
            item = q.get(timeout=240)
            assert not isinstance(item[1], str), item
            out[item[0]] = item[1:]
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    d, w_hat = _inputs()
    full = oracle.linear_bwd(d["x"], d["dY"], w_hat, d["A"], d["B"], SHAPE["alpha"])
    for rank in range(ws):
        m0, m1, dA, dB, dX = out[rank]
        # every rank ends with the same, full-batch gradients
        for got, ref, name in ((dA, full["dA"], "dA"), (dB, full["dB"], "dB")):
            err = np.abs(got - ref).max()
            rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
            assert err <= 2e-2 and rel <= 1e-2, (name, rank, err, rel)
        assert np.array_equal(dX, full["dX"][m0:m1])
    assert out[0][0] == 0 and out[0][1] == out[1][0] and out[1][1] == SHAPE["M"]
    assert np.array_equal(out[0][2], out[1][2]) and np.array_equal(out[0][3], out[1][3])
