"""The MSE loss through the C ABI against the oracle: the row kernel on its
own (mlp_op_mse, fp32 and bf16, scalar and vector paths, ragged shapes and
the 16384 x 32000 output of the largest workload on sampled rows), one fp32
training step element by element, trajectories against the oracle ensemble,
a full-size closed form, and host-input steps."""

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from oracle import mlp_oracle as om
from tests import parity as P
from tests.test_gpu_step import make_model

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
W = synth.WORKLOADS


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _tdt(dtype):
    return torch.float32 if dtype == nn.F32 else torch.bfloat16


def mse_batches(w, n, batch=None):
    return [(synth.make_batch(w, s, batch)[0], synth.make_targets(w, s, batch)) for s in range(n)]


# ---------------------------------------------------------------------------
# The row kernel
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,B,C,pad", [(nn.F32, 64, 10, 0), (nn.F32, 333, 7, 3), (nn.BF16, 300, 100, 0),
                                           (nn.BF16, 4099, 1000, 8), (nn.F32, 1000, 1024, 0)])
def test_mse_rows(dtype, B, C, pad):
    ld = C + pad
    td = _tdt(dtype)
    z = synth.make_normal((B, ld), 1.5, 201, B, C, dtype=td)
    t = synth.make_normal((B, ld), 1.0, 202, B, C)
    dz = torch.full((B, ld), 7.0, dtype=td, device=DEV)
    rows = torch.empty(B, dtype=torch.float32, device=DEV)
    gs = 2.0 / (B * C)
    zd, tdv = z.to(DEV), t.to(DEV)
    nn.mlp_op_mse(dtype, B, C, zd.data_ptr(), ld, tdv.data_ptr(), ld, gs, dz.data_ptr(), ld, rows.data_ptr(),
                  _stream())
    torch.cuda.synchronize()
    r_ref, dz_ref = om.mse(P.to64(z)[:, :C], P.to64(t)[:, :C])
    # fp32: one rounding of d = z - t, of each square and of each addition
    # (C / 32 terms a lane, then a 5-level warp tree)
    tol_r = (C / 32 + 8) * 2.0 ** -23 * r_ref + 1e-30
    assert np.all(np.abs(P.to64(rows) - r_ref) <= tol_r)
    got = P.to64(dz)
    scale = float(np.float32(gs)) / gs
    tol = 2.0 ** -22 * np.abs(dz_ref) + (2.0 ** -8 * np.abs(dz_ref) if dtype == nn.BF16 else 0) + 1e-30
    assert np.all(np.abs(got[:, :C] - dz_ref * scale) <= tol)
    if pad:
        assert torch.all(dz[:, C:].cpu() == 7.0)   # the padding is not written


def test_mse_rows_full_size_lm_output_sampled():
    B, C = 16384, 32000
    z = synth.make_normal((B, C), 2.0, 211, dtype=torch.bfloat16).to(DEV)
    t = synth.make_normal((B, C), 1.0, 212).to(DEV)
    dz = torch.empty_like(z)
    rows = torch.empty(B, dtype=torch.float32, device=DEV)
    gs = 2.0 / (B * C)
    nn.mlp_op_mse(nn.BF16, B, C, z.data_ptr(), C, t.data_ptr(), C, gs, dz.data_ptr(), C, rows.data_ptr(), _stream())
    torch.cuda.synchronize()
    r = np.concatenate([[0, B - 1], np.random.default_rng(213).integers(0, B, 30)])
    rt = torch.as_tensor(r, device=DEV)
    r_ref, dz_ref = om.mse(P.to64(z[rt]), P.to64(t[rt]))
    dz_ref = dz_ref * (len(r) / B)   # the oracle scales by its own element count
    assert np.all(np.abs(P.to64(rows[rt]) - r_ref) <= (C / 32 + 8) * 2.0 ** -23 * r_ref)
    got = P.to64(dz[rt])
    assert np.all(np.abs(got - dz_ref * float(np.float32(gs)) / gs) <= (2.0 ** -8 + 2.0 ** -22) * np.abs(dz_ref)
                  + 1e-30)


# ---------------------------------------------------------------------------
# Whole steps
# ---------------------------------------------------------------------------
# the kernels an fp32 MNIST-shaped step runs: the fused output layer with
# tensor-core planes (default), the fused layer with FFMA GEMMs, or separate
# GEMM / row kernels
MODES = {"tc3planes": dict(f32_tc=1, fuse=1), "ffma": dict(f32_tc=0, fuse=1), "unfused": dict(f32_tc=0, fuse=0)}


def _mse_model(w, B, params0, graph=True, mode="tc3planes"):
    m = make_model(w, B, params0, graph=graph, f32_tc=MODES[mode]["f32_tc"])
    m.set_option(nn.OPT_FUSE_HEAD, MODES[mode]["fuse"])
    m.set_loss(nn.LOSS_MSE)
    return m


def _run(m, w, bl):
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    losses = torch.empty(len(bl), dtype=torch.float32, device=DEV)
    for i, (x, t) in enumerate(bl):
        m.train_step(x.to(DEV), t.to(DEV), loss=losses[i], **hyper)
    m.check_errors()
    p, step = m.read_flat(nn.PLANE_P)
    g, _ = m.read_flat(nn.PLANE_G)
    assert step == len(bl)
    return (losses.cpu().numpy().astype(np.float64), m.split(p.astype(np.float64)),
            m.split(g.astype(np.float64)))


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("name,batch", [("mnist_mlp_b64", None), ("mnist_mlp_b64", 333), ("mnist_mlp_b4096", None)])
def test_fp32_one_step_mse(name, batch, mode):
    w = W[name]
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = mse_batches(w, 1, B)
    m = _mse_model(w, B, params0, mode=mode)
    names = [n for n, _ in nn.mlp_profile_step(m.h, bl[0][0].to(DEV).data_ptr(), bl[0][1].to(DEV).data_ptr(), 0.0,
                                               0.9, 0.999, 1e-8, 0.0, None, m.stream())]
    assert ("head_mse" in names) == (mode != "unfused") and ("mse" in names) == (mode == "unfused")
    assert ("split3" in names) == (mode == "tc3planes")
    m.close()
    m = _mse_model(w, B, params0, mode=mode)
    g_losses, g_params, g_grads = _run(m, w, bl)
    m.close()
    o_losses, o_params, _, _, o_grads = P.oracle_run(w, params0, bl, "fp64", loss="mse")
    assert abs(g_losses[0] - o_losses[0]) <= 1e-5 * abs(o_losses[0])
    kappa = P.oracle_abs_sums(w, params0, *bl[0], "fp64", loss="mse")
    lr, eps = P.hyper32(w)[0], P.hyper32(w)[3]
    for i, (g, go, k, p, po) in enumerate(zip(g_grads, o_grads, kappa, g_params, o_params)):
        tg = P.fp32_grad_tol(k)
        assert np.all(np.abs(g - go) <= tg), (i, np.max(np.abs(g - go) / tg))
        tp = P.fp32_first_step_param_tol(po, go, tg, lr, eps)
        assert np.all(np.abs(p - po) <= tp), (i, np.max(np.abs(p - po) / tp))


def _ensemble_mse(w, n_steps, batch=None, optim="adamw", mode="tc3planes"):
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = mse_batches(w, n_steps, B)
    m = _mse_model(w, B, params0, mode=mode)
    if optim != "adamw":
        m.set_optimizer({"adam": nn.OPTIM_ADAM, "sgd": nn.OPTIM_SGD}[optim], 0.0)
    g_losses, g_params, _ = _run(m, w, bl)
    m.close()
    mode = P.oracle_mode(w)
    kw = dict(optim=optim, loss="mse")
    ref = P.oracle_run(w, params0, bl, mode, **kw)
    ens = [P.oracle_run(w, params0, bl, mode, perturb_seed=s + 1, **kw) for s in range(P.ENSEMBLE_RUNS)]
    p0 = [P.to64(p) for p in params0]
    if w.dtype == synth.F32:
        P.loss_ensemble_check("loss", g_losses, ref[0], [e[0] for e in ens], 1e-4)
        lr = P.hyper32(w)[0]
        P.ensemble_check("params", g_params, ref[1], [e[1] for e in ens],
                         [np.maximum(np.abs(r), lr) for r in ref[1]], 1e-4)
    else:
        P.loss_ensemble_check("loss", g_losses, ref[0], [e[0] for e in ens], 1e-3)
        P.ensemble_check("params", g_params, ref[1], [e[1] for e in ens],
                         [np.max(np.abs(r - q)) for r, q in zip(ref[1], p0)], 3e-2)


@pytest.mark.parametrize("mode", list(MODES))
def test_mnist_mlp_b64_three_steps_mse(mode):
    _ensemble_mse(W["mnist_mlp_b64"], 3, mode=mode)


def test_cifar_mlp_bf16_reduced_batch_mse_sgd():
    _ensemble_mse(W["cifar_mlp_b8192"], 3, batch=320, optim="sgd")


def test_deep_narrow_bf16_reduced_batch_mse():
    _ensemble_mse(W["deep_narrow_b65536"], 2, batch=300)


@pytest.mark.parametrize("name", ["mnist_mlp_b4096", "cifar_mlp_b8192", "deep_narrow_b65536"])
def test_zero_params_closed_form_full_size_mse(name):
    """W = b = 0 => z = 0, loss = mean(t^2), dz = -2 t / (B C); only the last
    bias has a gradient, db_c = -2 sum_i t_ic / (B C), so one AdamW step
    gives b_c = -lr g / (|g| + eps) and leaves every other parameter 0."""
    w = W[name]
    m = make_model(w)
    m.set_loss(nn.LOSS_MSE)
    m.write_flat(np.zeros(m.n_params, np.float32), nn.PLANE_P, 0)
    x, _ = synth.make_batch(w, 0)
    t = synth.make_targets(w, 0)
    loss = m.train_step(x.to(DEV), t.to(DEV), w.lr, w.beta1, w.beta2, w.eps, w.wd)
    m.check_errors()
    t64 = P.to64(t)
    want_loss = float(np.mean(t64 ** 2))
    assert abs(loss.item() - want_loss) <= 1e-5 * want_loss
    p, _ = m.read_flat(nn.PLANE_P)
    parts = m.split(p)
    for q in parts[:-1]:
        assert np.all(q == 0)
    B, C = t64.shape
    # dz as the kernel forms it: fp32 product -t * fp32(2 / (B C)), stored in
    # the model dtype (bf16: round to nearest even); then fp32 column sums
    dz = torch.from_numpy(-t.numpy() * np.float32(2.0 / (B * C)))
    dz = P.to64(dz.to(torch.bfloat16) if w.dtype == synth.BF16 else dz)
    g = dz.sum(axis=0)
    dg = 2.0 ** -20 * np.abs(dz).sum(axis=0)
    lr, eps = P.hyper32(w)[0], P.hyper32(w)[3]
    want = -lr * g / (np.abs(g) + eps)
    sure = np.abs(g) > 10 * dg
    np.testing.assert_allclose(parts[-1][sure], want[sure], rtol=1e-3, atol=1e-3 * lr)
    assert np.all(np.abs(parts[-1]) <= lr * (1 + 1e-3))
    assert sure.sum() >= C // 2
    m.close()


def test_mse_host_steps_match_device_and_switching_losses():
    """Host-input MSE steps equal device-input ones bit for bit; a model can
    alternate CE and MSE steps (the weight planes the CE step reads stay
    current through MSE steps)."""
    w = W["mnist_mlp_b4096"]
    params0 = synth.make_params(w)
    bl = mse_batches(w, 3)
    m = _mse_model(w, w.batch, params0)
    d_losses, d_params, _ = _run(m, w, bl)
    m.close()
    m = _mse_model(w, w.batch, params0)
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    hl = torch.zeros(len(bl), dtype=torch.float32).pin_memory()
    # the host buffers must outlive their asynchronous copies
    hx = [x.pin_memory() for x, _ in bl]
    ht = [t.pin_memory() for _, t in bl]
    for i in range(len(bl)):
        m.train_step_host(hx[i], ht[i], loss=hl[i:i + 1], **hyper)
    torch.cuda.synchronize()
    m.check_errors()
    p, _ = m.read_flat(nn.PLANE_P)
    assert np.array_equal(hl.numpy().astype(np.float64), d_losses)
    assert np.array_equal(P.flat(m.split(p.astype(np.float64))), P.flat(d_params))
    # then a CE step on the same model equals a CE step of a fresh model
    # given the same parameters, moments and step count
    x, y = synth.make_batch(w, 9)
    mv = [m.read_flat(k)[0] for k in (nn.PLANE_M, nn.PLANE_V)]
    m.set_loss(nn.LOSS_CE)
    l1 = m.train_step(x.to(DEV), y.to(DEV), **hyper)
    p1, _ = m.read_flat(nn.PLANE_P)
    m.close()
    m2 = make_model(w)
    m2.write_flat(p, nn.PLANE_P, len(bl))
    m2.write_flat(mv[0], nn.PLANE_M, len(bl))
    m2.write_flat(mv[1], nn.PLANE_V, len(bl))
    l2 = m2.train_step(x.to(DEV), y.to(DEV), **hyper)
    p2, _ = m2.read_flat(nn.PLANE_P)
    m2.close()
    assert l1.item() == l2.item()
    assert np.array_equal(p1, p2)


def test_mse_host_targets_too_large_for_the_input_slot():
    # B * C * 4 > 64 MiB: the host-input slot holds labels only
    m = nn.Model([8, 8, 4096], [nn.ACT_RELU], nn.ACT_RELU, nn.BF16, seed=1, batch=4097)
    m.set_loss(nn.LOSS_MSE)
    x = torch.zeros(4097, 8, dtype=torch.bfloat16).pin_memory()
    t = torch.zeros(4097, 4096, dtype=torch.float32).pin_memory()
    with pytest.raises(nn.MlpError) as e:
        m.train_step_host(x, t, lr=1e-3)
    assert e.value.status == 2
    m.close()


def test_set_loss_rejects_unknown():
    m = make_model(W["mnist_mlp_b64"])
    with pytest.raises(nn.MlpError):
        m.set_loss(2)
    m.close()
