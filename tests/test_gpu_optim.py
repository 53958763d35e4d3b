"""Optimizer variants and global-norm clipping through the C ABI against the
oracle: the flat update kernel on its own (mlp_op_optim), one fp32 training
step element by element, and short trajectories against the oracle ensemble,
for AdamW, Adam with L2 and SGD with momentum, with clipping off and on."""
import math

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from oracle import mlp_oracle as om
from tests import parity as P
from tests.test_gpu_step import F32_MODES, gpu_run, make_model

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
W = synth.WORKLOADS
KINDS = {"adamw": nn.OPTIM_ADAMW, "adam": nn.OPTIM_ADAM, "sgd": nn.OPTIM_SGD}
f32 = lambda a: float(np.float32(a))


def _stream():
    return torch.cuda.current_stream().cuda_stream


def clip_rel_err(n: int) -> float:
    """Relative error bound of the fp32 clipping factor: the sum of n squares
    runs as per-thread sums over n / (1216 * 256) terms and two trees of
    depth <= 11 each, every addition off by at most 2^-24 relative; the
    square root halves it, the division adds an ulp."""
    depth = n / (1216 * 256) + 32
    return depth * 2.0 ** -25 + 2.0 ** -23


# ---------------------------------------------------------------------------
# The flat update kernel
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("optim", list(KINDS))
@pytest.mark.parametrize("n,t,clip", [(1000, 1, 0.0), (4099, 7, 0.0), (4099, 7, 0.05), (5256202, 3, 0.3),
                                      (5256202, 1, 1e9)])
def test_flat_update(optim, n, t, clip):
    kind = KINDS[optim]
    p = synth.make_normal((n,), 0.05, 71, n)
    g = synth.make_normal((n,), 1e-3, 72, n)
    m = synth.make_normal((n,), 1e-4, 73, n)
    v = synth.make_uniform((n,), 0.0, 1e-6, 74, n)
    if t == 1:
        m.zero_()
        v.zero_()
    pd, gd, md, vd = (a.to(DEV) for a in (p, g, m, v))
    w16 = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(nn.OPTIM_WS_FLOATS, dtype=torch.float32, device=DEV)
    norm = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.05
    nn.mlp_op_optim(kind, n, pd.data_ptr(), gd.data_ptr(), md.data_ptr(), vd.data_ptr(), w16.data_ptr(), t, lr, b1,
                    b2, eps, wd, clip, ws.data_ptr(), norm.data_ptr(), _stream())
    torch.cuda.synchronize()
    p64, g64, m64, v64 = P.to64(p), P.to64(g), P.to64(m), P.to64(v)
    c = om.clip_coef([g64], f32(clip))
    dc = clip_rel_err(n) if clip else 0.0
    gn = math.sqrt(float(np.sum(g64 ** 2)))
    if clip:
        assert abs(norm.item() - gn) <= 2 * clip_rel_err(n) * gn
        assert (c < 1.0) == (clip < gn)
    else:
        assert norm.item() == -1.0            # untouched without clipping
    assert torch.equal(gd.cpu(), g)            # the gradient itself is not scaled
    pr, mr, vr = om.update(optim, p64, g64 * c, m64, v64, t, f32(lr), f32(b1), f32(b2), f32(eps), f32(wd))
    # the gradient the update sees: c g (+ wd p), c off by dc relative
    gp = c * g64 + (f32(wd) * p64 if optim != "adamw" else 0.0)
    dg = (dc + 2.0 ** -24) * c * np.abs(g64) + (2.0 ** -24 * np.abs(gp) if optim != "adamw" else 0.0)
    pd64, md64, vd64 = P.to64(pd), P.to64(md), P.to64(vd)
    if optim == "sgd":
        tol_m = 2.0 ** -22 * (f32(b1) * np.abs(m64) + np.abs(gp)) + dg + 1e-30
        assert np.all(np.abs(md64 - mr) <= tol_m)
        assert torch.equal(vd.cpu(), v)        # SGD leaves the second plane alone
        tol_p = f32(lr) * tol_m + 2.0 ** -23 * np.abs(pr)
    else:
        tol_m = 2.0 ** -21 * (f32(b1) * np.abs(m64) + (1 - f32(b1)) * np.abs(gp)) + (1 - f32(b1)) * dg + 1e-30
        tol_v = 2.0 ** -21 * (f32(b2) * v64 + (1 - f32(b2)) * gp * gp) + (1 - f32(b2)) * 2 * np.abs(gp) * dg + 1e-38
        assert np.all(np.abs(md64 - mr) <= tol_m)
        assert np.all(np.abs(vd64 - vr) <= tol_v)
        # the update term has size ~lr: relative 1e-5 of lr plus the ulp of p,
        # plus how far the oracle's own step moves when its gradient moves by
        # dg (large only where g' nearly cancels at t = 1: the direction
        # g' / (|g'| + eps) is then decided by rounding)
        hyp = (t, f32(lr), f32(b1), f32(b2), f32(eps), f32(wd))
        sens = np.maximum(np.abs(om.update(optim, p64, g64 * c + dg, m64, v64, *hyp)[0] - pr),
                          np.abs(om.update(optim, p64, g64 * c - dg, m64, v64, *hyp)[0] - pr))
        tol_p = 1e-5 * lr + 4 * dc * lr + 2.0 ** -23 * np.abs(pr) + sens
    assert np.all(np.abs(pd64 - pr) <= tol_p), np.max(np.abs(pd64 - pr) / tol_p)
    assert torch.equal(w16.cpu(), pd.cpu().to(torch.bfloat16))


def test_flat_update_rejects_bad_arguments():
    n = 64
    a = [torch.zeros(n, device=DEV) for _ in range(4)]
    ptr = [x.data_ptr() for x in a]
    with pytest.raises(nn.MlpError):   # unknown kind
        nn.mlp_op_optim(3, n, *ptr, None, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 0.0, None, None, _stream())
    with pytest.raises(nn.MlpError):   # clipping without a workspace
        nn.mlp_op_optim(0, n, *ptr, None, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1.0, None, None, _stream())
    with pytest.raises(nn.MlpError):   # Adam rules need t >= 1
        nn.mlp_op_optim(1, n, *ptr, None, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 0.0, None, None, _stream())


# ---------------------------------------------------------------------------
# One fp32 step, element by element
# ---------------------------------------------------------------------------
def _first_norm(w, params0, bl):
    grads = P.oracle_run(w, params0, bl[:1], "fp64")[4]
    return math.sqrt(sum(float(np.sum(g ** 2)) for g in grads))


def fp32_one_step_optim(w, optim, clip_frac, f32_tc, batch=None):
    """One step from a shared state with optimizer `optim`; clipping at
    clip_frac times the oracle's gradient norm (0: off)."""
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, 1, B)
    norm_ref = _first_norm(w, params0, bl)
    max_norm = f32(clip_frac * norm_ref)
    m = make_model(w, B, params0, f32_tc=f32_tc)
    m.set_optimizer(KINDS[optim], max_norm)
    g_losses, g_params, g_grads = gpu_run(m, w, bl)
    gpu_norm = m.grad_norm()
    kps = m.kernels_per_step()
    m.close()
    o_losses, o_params, _, _, o_grads = P.oracle_run(w, params0, bl, "fp64", optim=optim, max_norm=max_norm)
    assert abs(g_losses[0] - o_losses[0]) <= 1e-4 * abs(o_losses[0])
    c = om.clip_coef(o_grads, max_norm)
    if clip_frac:
        assert c < 1.0
        assert abs(gpu_norm - norm_ref) <= 1e-5 * norm_ref, (gpu_norm, norm_ref)
    kappa = P.oracle_abs_sums(w, params0, *bl[0], "fp64")
    lr, _, _, eps, wd = P.hyper32(w)
    n_all = sum(g.size for g in o_grads)
    dc = (clip_rel_err(n_all) + 1e-5) if clip_frac else 0.0   # plus the norm's own gradient error
    p0 = [P.to64(p) for p in params0]
    for i, (g, go, k, p, po, q0) in enumerate(zip(g_grads, o_grads, kappa, g_params, o_params, p0)):
        tg = P.fp32_grad_tol(k)
        assert np.all(np.abs(g - go) <= tg), (i, np.max(np.abs(g - go) / tg))   # G holds the unclipped gradient
        dg = c * tg + dc * c * np.abs(go)
        if optim != "adamw":   # fp32 rounding of g' = c g + wd p
            dg = dg + 2.0 ** -23 * (c * np.abs(go) + wd * np.abs(q0))
        if optim == "adamw":
            tp = P.fp32_first_step_param_tol(po, c * go, dg, lr, eps)
        elif optim == "adam":
            tp = P.fp32_first_step_param_tol(po, c * go + wd * q0, dg, lr, eps)
        else:
            tp = 1e-4 * np.maximum(np.abs(po), lr) + lr * dg
        assert np.all(np.abs(p - po) <= tp), (i, np.max(np.abs(p - po) / tp))
    return kps


@pytest.mark.parametrize("f32_tc", F32_MODES)
@pytest.mark.parametrize("optim", list(KINDS))
@pytest.mark.parametrize("clip_frac", [0.0, 0.5])
def test_mnist_mlp_b64_one_step_optim(optim, clip_frac, f32_tc):
    fp32_one_step_optim(W["mnist_mlp_b64"], optim, clip_frac, f32_tc)


@pytest.mark.parametrize("optim", list(KINDS))
def test_mnist_mlp_b4096_one_step_optim_clipped(optim):
    # full size: the output layer's and the deferred split-K gradients reach
    # the norm as partial sums
    fp32_one_step_optim(W["mnist_mlp_b4096"], optim, 0.5, 1)


def test_clipping_adds_one_kernel_and_options_are_checked():
    w = W["mnist_mlp_b64"]
    m = make_model(w)
    base = m.kernels_per_step()
    m.set_optimizer(nn.OPTIM_SGD, 0.0)
    assert m.kernels_per_step() == base
    m.set_optimizer(nn.OPTIM_ADAM, 1.0)
    assert m.kernels_per_step() == base + 1
    for bad in ((3, 0.0), (-1, 0.0), (0, -1.0), (0, float("inf")), (0, float("nan"))):
        with pytest.raises(nn.MlpError):
            m.set_optimizer(*bad)
    m.close()


# ---------------------------------------------------------------------------
# Trajectories against the oracle ensemble
# ---------------------------------------------------------------------------
def _ensemble_optim(w, n_steps, optim, clip_frac, batch=None, one_graph=False, f32_tc=None):
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, n_steps, B)
    max_norm = f32(clip_frac * _first_norm(w, params0, bl)) if clip_frac else 0.0
    m = make_model(w, B, params0, f32_tc=f32_tc)
    m.set_optimizer(KINDS[optim], max_norm)
    g_losses, g_params, g_grads = gpu_run(m, w, bl, one_graph)
    m.close()
    mode = P.oracle_mode(w)
    kw = dict(optim=optim, max_norm=max_norm)
    ref = P.oracle_run(w, params0, bl, mode, **kw)
    ens = [P.oracle_run(w, params0, bl, mode, perturb_seed=s + 1, **kw) for s in range(P.ENSEMBLE_RUNS)]
    p0 = [P.to64(p) for p in params0]
    if w.dtype == synth.F32:
        P.loss_ensemble_check("loss", g_losses, ref[0], [e[0] for e in ens], 1e-4)
        lr = P.hyper32(w)[0]
        scale = [np.maximum(np.abs(r), lr) for r in ref[1]]
        P.ensemble_check("params", g_params, ref[1], [e[1] for e in ens], scale, 1e-4)
    else:
        P.loss_ensemble_check("loss", g_losses, ref[0], [e[0] for e in ens], 1e-3)
        scale = [np.max(np.abs(r - q)) for r, q in zip(ref[1], p0)]
        P.ensemble_check("params", g_params, ref[1], [e[1] for e in ens], scale, 3e-2)


@pytest.mark.parametrize("f32_tc", F32_MODES)
@pytest.mark.parametrize("optim,clip_frac", [("adam", 0.0), ("sgd", 0.0), ("adamw", 0.3), ("sgd", 0.3)])
def test_mnist_mlp_b64_three_steps_optim(optim, clip_frac, f32_tc):
    _ensemble_optim(W["mnist_mlp_b64"], 3, optim, clip_frac, f32_tc=f32_tc)


@pytest.mark.parametrize("optim,clip_frac", [("adam", 0.5), ("sgd", 0.5)])
def test_cifar_mlp_bf16_reduced_batch_optim(optim, clip_frac):
    _ensemble_optim(W["cifar_mlp_b8192"], 3, optim, clip_frac, batch=320)


def test_deep_narrow_bf16_one_graph_sgd_clipped():
    _ensemble_optim(W["deep_narrow_b65536"], 3, "sgd", 0.5, batch=300, one_graph=True)
