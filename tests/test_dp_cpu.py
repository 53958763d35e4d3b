"""The data-parallel driver's host logic on CPU ranks (gloo, world size 2).

neural_net_step_gb300.dp splits a global batch into contiguous row ranges
(shard_rows) and runs a step as: the model's gradient step on the rank's
rows (loss gradient scaled by 1 / global batch), a SUM all-reduce of the flat
gradient buffer and of the loss, then the update.  Here the model is a small
numpy stand-in with the same methods (a linear least-squares model and an
SGD update; no GPU), so the test checks the driver itself: which rows each
rank takes, that the exchange happens between the two halves of the step,
that ranks end with identical parameters, and that those equal one process
stepping on the whole batch.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from neural_net_step_gb300.dp import DataParallel, shard_rows

WORLD = 2


@pytest.mark.parametrize("B,W", [(64, 2), (65, 2), (4096, 8), (7, 7), (1000, 3)])
def test_shard_rows_cover_the_batch_in_order(B, W):
    spans = [shard_rows(B, W, r) for r in range(W)]
    assert spans[0][0] == 0 and spans[-1][1] == B
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def test_shard_rows_rejects_bad_arguments():
    with pytest.raises(ValueError):
        shard_rows(3, 4, 0)
    with pytest.raises(ValueError):
        shard_rows(8, 2, 2)


class LinearStandIn:
    """y ~ x w (mean squared error over the GLOBAL batch), SGD update; the
    gradient lives in one flat tensor like the library's G plane."""

    def __init__(self, w0, batch):
        self.batch = batch
        self.w = np.array(w0, np.float64)
        self.g = torch.zeros(self.w.size, dtype=torch.float64)
        self.steps = 0
        self.calls = []

    def grad_tensor(self):
        return self.g

    def grad_step(self, x, y, global_batch, loss=None):
        x, y = np.asarray(x), np.asarray(y)
        r = x @ self.w - y
        self.g.copy_(torch.from_numpy(2.0 * x.T @ r / global_batch))
        self.steps += 1
        self.calls.append("grad")
        return torch.tensor(float((r * r).sum() / global_batch), dtype=torch.float64)

    def apply_update(self, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0):
        self.calls.append("update")
        self.w = self.w - lr * self.g.numpy()

    def read_flat(self):
        return self.w.astype(np.float32), self.steps

    def write_flat(self, flat, step=0):
        self.w = np.asarray(flat, np.float64)
        self.steps = step


def _data(B, K, steps):
    rng = np.random.default_rng(5)
    return [(rng.standard_normal((B, K)), rng.standard_normal(B)) for _ in range(steps)]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir, B, K, steps):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        lo, hi = shard_rows(B, WORLD, rank)
        # rank 1 starts from other parameters: the broadcast must replace them
        model = LinearStandIn(np.linspace(-1, 1, K) + rank, hi - lo)
        dp = DataParallel(model, B)
        dp.broadcast_params(0)
        losses = []
        for x, y in _data(B, K, steps):
            losses.append(float(dp.step(x[lo:hi], y[lo:hi], 0.05)))
        np.save(os.path.join(out_dir, f"rank{rank}.npy"), np.concatenate([model.w, losses]))
        assert model.calls == ["grad", "update"] * steps
    finally:
        dist.destroy_process_group()


def test_two_rank_steps_equal_one_process_on_the_whole_batch(tmp_path):
    B, K, steps = 37, 5, 4        # 19 + 18 rows
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path), B, K, steps), nprocs=WORLD,
                       start_method="spawn")
    r0, r1 = (np.load(tmp_path / f"rank{r}.npy") for r in range(WORLD))
    assert np.array_equal(r0, r1)                     # identical replicas and losses
    one = LinearStandIn(np.linspace(-1, 1, K), B)     # rank 0's initial parameters
    dp = DataParallel(one, B)                         # no process group: this process alone
    losses = [float(dp.step(x, y, 0.05)) for x, y in _data(B, K, steps)]
    np.testing.assert_allclose(r0[:K], one.w, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r0[K:], losses, rtol=1e-12)
