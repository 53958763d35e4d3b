"""The data-parallel identity of the step, on CPU ranks (gloo, world size 2).

The step shards by batch rows: each rank runs the forward and the backward of
its rows with the loss gradient scaled by the GLOBAL batch size (dz = (softmax
- onehot) / B), so a plain sum all-reduce of the gradients reproduces the
unsharded gradient, and identical AdamW updates keep the replicas equal.  Both
sides are the fp64 oracle; the only difference is the order of the batch sum.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth
from oracle import mlp_oracle as om

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_grads(params, x, y, acts, B_global):
    fw = om.forward(params, x, acts)
    loss_rows, dz = om.softmax_ce(fw["z"], y)
    dz = dz * (x.shape[0] / B_global)          # the oracle scales by its own rows: use the global batch
    return loss_rows.sum(), om.backward(fw, dz, acts)


def _rank_main(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        w = synth.WORKLOADS["mnist_mlp_b64"]
        params = [p.numpy().astype(np.float64) for p in synth.make_params(w)]
        x, y = (t.numpy() for t in synth.make_batch(w, 7))
        x = x.astype(np.float64)
        B = x.shape[0]
        lo, hi = rank * B // WORLD, (rank + 1) * B // WORLD
        lsum, grads = _shard_grads(params, x[lo:hi], y[lo:hi], w.acts, B)
        flat = torch.from_numpy(np.concatenate([g.ravel() for g in grads] + [np.array([lsum])]))
        dist.all_reduce(flat, op=dist.ReduceOp.SUM)
        # every replica applies the same AdamW step to the reduced gradient
        sizes = [g.size for g in grads]
        red = np.split(flat.numpy()[:-1], np.cumsum(sizes)[:-1])
        new = []
        for p, g in zip(params, red):
            pn, _, _ = om.adamw(p, g.reshape(p.shape), np.zeros_like(p), np.zeros_like(p), 1, w.lr, w.beta1,
                                w.beta2, w.eps, w.wd)
            new.append(pn)
        pflat = torch.from_numpy(np.concatenate([p.ravel() for p in new]))
        gathered = [torch.empty_like(pflat) for _ in range(WORLD)]
        dist.all_gather(gathered, pflat)
        if rank == 0:
            q.put((flat.numpy(), [t.numpy() for t in gathered]))
    finally:
        dist.destroy_process_group()


def test_batch_sharded_step_equals_unsharded_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    try:
        red, gathered = q.get(timeout=120)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # unsharded reference
    w = synth.WORKLOADS["mnist_mlp_b64"]
    params = [p.numpy().astype(np.float64) for p in synth.make_params(w)]
    x, y = (t.numpy() for t in synth.make_batch(w, 7))
    fw = om.forward(params, x.astype(np.float64), w.acts)
    loss_rows, dz = om.softmax_ce(fw["z"], y)
    grads = om.backward(fw, dz, w.acts)
    ref = np.concatenate([g.ravel() for g in grads])
    # the all-reduced gradient equals the unsharded one up to the order of the batch sum
    scale = np.abs(ref).max()
    np.testing.assert_allclose(red[:-1], ref, rtol=0, atol=1e-13 * scale)
    assert abs(red[-1] / x.shape[0] - loss_rows.mean()) <= 1e-13 * abs(loss_rows.mean())
    # the replicas' parameters after the update are identical
    assert np.array_equal(gathered[0], gathered[1])
