"""The data-parallel identity of the step, on CPU ranks (gloo, world size 2).

The step shards by batch rows: each rank runs the forward and the backward of
its rows with the loss gradient scaled by the GLOBAL batch size (dz = (softmax
- onehot) / B, or 2 (z - t) / (B C) for MSE), so a plain sum all-reduce of the
gradients reproduces the unsharded gradient; clipping by the reduced
gradient's global norm and identical updates keep the replicas equal.  Both
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


def _shard_grads(params, x, y, acts, B_global, loss):
    fw = om.forward(params, x, acts)
    if loss == "mse":
        rows, dz = om.mse(fw["z"], y)
        dz = dz * (x.shape[0] / B_global)      # the oracle scales by its own rows: use the global batch
    else:
        rows, dz = om.softmax_ce(fw["z"], y)
        dz = dz * (x.shape[0] / B_global)
    return rows.sum(), om.backward(fw, dz, acts)


def _batch(w, loss):
    x, y = (t.numpy() for t in synth.make_batch(w, 7))
    if loss == "mse":
        y = synth.make_targets(w, 7).numpy().astype(np.float64)
    return x.astype(np.float64), y


def _rank_main(rank, port, q, loss, optim, max_norm):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        w = synth.WORKLOADS["mnist_mlp_b64"]
        params = [p.numpy().astype(np.float64) for p in synth.make_params(w)]
        x, y = _batch(w, loss)
        B = x.shape[0]
        lo, hi = rank * B // WORLD, (rank + 1) * B // WORLD
        lsum, grads = _shard_grads(params, x[lo:hi], y[lo:hi], w.acts, B, loss)
        flat = torch.from_numpy(np.concatenate([g.ravel() for g in grads] + [np.array([lsum])]))
        dist.all_reduce(flat, op=dist.ReduceOp.SUM)
        # every replica clips the reduced gradient by its global norm and
        # applies the same update
        sizes = [g.size for g in grads]
        red = [g.reshape(p.shape) for g, p in zip(np.split(flat.numpy()[:-1], np.cumsum(sizes)[:-1]), params)]
        c = om.clip_coef(red, max_norm)
        new = []
        for p, g in zip(params, red):
            pn, _, _ = om.update(optim, p, g * c, np.zeros_like(p), np.zeros_like(p), 1, w.lr, w.beta1, w.beta2,
                                 w.eps, w.wd)
            new.append(pn)
        pflat = torch.from_numpy(np.concatenate([p.ravel() for p in new]))
        gathered = [torch.empty_like(pflat) for _ in range(WORLD)]
        dist.all_gather(gathered, pflat)
        if rank == 0:
            q.put((flat.numpy(), [t.numpy() for t in gathered]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("loss,optim,max_norm", [("ce", "adamw", 0.0), ("mse", "sgd", 0.05), ("ce", "adam", 0.05)])
def test_batch_sharded_step_equals_unsharded_gloo(loss, optim, max_norm):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q, loss, optim, max_norm)) for r in range(WORLD)]
    for p in procs:
        p.start()
    try:
        red, gathered = q.get(timeout=120)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # unsharded reference: the oracle's whole step on the full batch
    w = synth.WORKLOADS["mnist_mlp_b64"]
    params = [p.numpy().astype(np.float64) for p in synth.make_params(w)]
    x, y = _batch(w, loss)
    L, newp, _, _, grads, ex = om.train_step(params, [0 * p for p in params], [0 * p for p in params], 1, x, y,
                                             w.acts, w.lr, w.beta1, w.beta2, w.eps, w.wd, optim=optim,
                                             max_norm=max_norm, loss=loss)
    if max_norm:
        assert ex["clip"] < 1.0
    ref = np.concatenate([g.ravel() for g in grads])
    # the all-reduced gradient equals the unsharded one up to the order of the batch sum
    scale = np.abs(ref).max()
    np.testing.assert_allclose(red[:-1], ref, rtol=0, atol=1e-13 * scale)
    count = x.shape[0] * (w.n_classes if loss == "mse" else 1)
    assert abs(red[-1] / count - L) <= 1e-13 * abs(L)
    # the replicas' parameters after the update are identical, and equal the
    # unsharded step's up to the order of the batch sum
    assert np.array_equal(gathered[0], gathered[1])
    pref = np.concatenate([p.ravel() for p in newp])
    np.testing.assert_allclose(gathered[0], pref, rtol=0, atol=1e-12 * np.abs(pref).max())
