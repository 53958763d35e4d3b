"""The data-parallel step through the C ABI (mlp_grad_step, a sum over ranks
of the gradient buffer, mlp_apply_update) on the GPU.

* One process: the split step equals mlp_train_step bit for bit (CE and MSE,
  AdamW with and without clipping, fp32 on the tensor cores with the output
  layer's partial sums, bf16).
* Two processes on the one GPU, each its own half of the batch, the sum done
  by gloo (host-staged: no kernel waits on another process): the replicas end
  identical, and the step equals the oracle's step on the WHOLE batch within
  the fp32 one-step bounds (loss 1e-4 relative; every gradient and parameter
  element as in test_gpu_step.fp32_one_step).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import neural_net_step_gb300 as nn
import synth
from neural_net_step_gb300.dp import DataParallel, shard_rows
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
W = synth.WORKLOADS


def _model(w, B, params0, loss_kind="ce", max_norm=0.0):
    m = nn.Model(w.dims, w.acts, nn.ACT_RELU, w.dtype, seed=w.seed, batch=B)
    m.write_flat(P.flat([p.numpy() for p in params0]).astype(np.float32), nn.PLANE_P, 0)
    if loss_kind == "mse":
        m.set_loss(nn.LOSS_MSE)
    if max_norm:
        m.set_optimizer(nn.OPTIM_ADAMW, max_norm)
    return m


def _batches(w, n, B, loss_kind):
    out = []
    for s in range(n):
        x, y = synth.make_batch(w, s, B)
        if loss_kind == "mse":
            y = synth.make_targets(w, s, B)
        out.append((x.to(DEV), y.to(DEV)))
    return out


@pytest.mark.parametrize("name,batch,loss_kind,max_norm", [
    ("mnist_mlp_b4096", None, "ce", 0.0),       # fp32 planes, output layer folded into the layer-2 forward
    ("mnist_mlp_b4096", 333, "ce", 0.05),       # ragged batch, clipping
    ("mnist_mlp_b64", None, "mse", 0.0),
    ("cifar_mlp_b8192", 512, "ce", 0.0),        # bf16
    ("lm_block_t16384", 512, "ce", 0.5),        # bf16, GELU, clipping
])
def test_split_step_equals_train_step_bitwise(name, batch, loss_kind, max_norm):
    w = W[name]
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = _batches(w, 3, B, loss_kind)
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    res = []
    for split in (False, True):
        m = _model(w, B, params0, loss_kind, max_norm)
        losses = torch.zeros(len(bl), dtype=torch.float32, device=DEV)
        dp = DataParallel(m, B) if split else None
        for i, (x, y) in enumerate(bl):
            if split:
                dp.step(x, y, loss=losses[i], **hyper)
            else:
                m.train_step(x, y, loss=losses[i], **hyper)
        m.check_errors()
        p, step = m.read_flat(nn.PLANE_P)
        g, _ = m.read_flat(nn.PLANE_G)
        assert step == len(bl)
        res.append((losses.cpu().numpy(), p, g))
        m.close()
    for a, b in zip(res[0], res[1]):
        assert np.array_equal(a, b)


def test_grad_step_rejects_a_global_batch_below_its_own():
    w = W["mnist_mlp_b64"]
    m = _model(w, 64, synth.make_params(w))
    x, y = _batches(w, 1, 64, "ce")[0]
    with pytest.raises(nn.MlpError):
        m.grad_step(x, y, 63)
    m.close()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir, name):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        torch.cuda.set_device(0)
        w = W[name]
        B = w.batch
        lo, hi = shard_rows(B, 2, rank)
        m = _model(w, hi - lo, synth.make_params(w))
        dp = DataParallel(m, B)
        x, y = synth.make_batch(w, 0)
        loss = dp.step(x[lo:hi].to(DEV), y[lo:hi].to(DEV), w.lr, w.beta1, w.beta2, w.eps, w.wd)
        m.check_errors()
        p, step = m.read_flat(nn.PLANE_P)
        g, _ = m.read_flat(nn.PLANE_G)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.concatenate([[float(loss.item()), float(step)], p.astype(np.float64), g.astype(np.float64)]))
        m.close()
    finally:
        dist.destroy_process_group()


def test_two_ranks_on_halves_equal_the_oracle_on_the_whole_batch(tmp_path):
    name = "mnist_mlp_b4096"
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path), name), nprocs=2, start_method="spawn")
    r0, r1 = (np.load(tmp_path / f"rank{r}.npy") for r in range(2))
    assert np.array_equal(r0, r1)               # identical replicas
    w = W[name]
    params0 = synth.make_params(w)
    n = w.n_params()
    loss, step, p, g = r0[0], r0[1], r0[2:2 + n], r0[2 + n:]
    assert step == 1
    split = lambda a: [a[o:o + s].reshape(sh) for o, s, sh in _layout(w)]
    bl = P.batches(w, 1)
    o_losses, o_params, _, _, o_grads = P.oracle_run(w, params0, bl, "fp64")
    assert abs(loss - o_losses[0]) <= 1e-4 * abs(o_losses[0])
    kappa = P.oracle_abs_sums(w, params0, *bl[0], "fp64")
    lr, eps = P.hyper32(w)[0], P.hyper32(w)[3]
    for i, (gg, go, k, pp, po) in enumerate(zip(split(g), o_grads, kappa, split(p), o_params)):
        tg = P.fp32_grad_tol(k)
        assert np.all(np.abs(gg - go) <= tg), (i, np.max(np.abs(gg - go) / tg))
        tp = P.fp32_first_step_param_tol(po, go, tg, lr, eps)
        assert np.all(np.abs(pp - po) <= tp), (i, np.max(np.abs(pp - po) / tp))


def _layout(w):
    """(offset, size, shape) of W1, b1, ... in the dense flat vector."""
    out, pos = [], 0
    for (nn_, k), _ in w.param_shapes():
        out.append((pos, nn_ * k, (nn_, k)))
        pos += nn_ * k
        out.append((pos, nn_, (nn_,)))
        pos += nn_
    return out
