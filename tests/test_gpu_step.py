"""Whole-step parity: mlp_train_step / mlp_train_steps / mlp_forward through
the C ABI against the CPU oracle on the same seeded batches and initial
parameters (drawn by synth, written into the model), plus closed forms and
properties that hold at the full sizes of the five workloads."""
import math

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from oracle import mlp_oracle as om
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
W = synth.WORKLOADS


def make_model(w: synth.Workload, batch=None, params=None, graph=True, f32_tc=None, head_gemm=None):
    B = w.batch if batch is None else batch
    m = nn.Model(w.dims, w.acts, nn.ACT_RELU, w.dtype, seed=w.seed, batch=B)
    m.set_graph_mode(graph)
    if f32_tc is not None:
        m.set_option(nn.OPT_F32_TENSOR_CORES, f32_tc)
    if head_gemm is not None:
        m.set_option(nn.OPT_HEAD_IN_GEMM, head_gemm)
    if params is not None:
        m.write_flat(P.flat([p.numpy() for p in params]).astype(np.float32), nn.PLANE_P, 0)
    return m


def gpu_run(m: nn.Model, w: synth.Workload, bl, one_graph=False):
    xs = [x.to(DEV) for x, _ in bl]
    ys = [y.to(DEV) for _, y in bl]
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    if one_graph:
        losses = m.train_steps(xs, ys, **hyper)
    else:
        losses = torch.empty(len(bl), dtype=torch.float32, device=DEV)
        for i in range(len(bl)):
            m.train_step(xs[i], ys[i], loss=losses[i], **hyper)
    m.check_errors()
    p, step = m.read_flat(nn.PLANE_P)
    g, _ = m.read_flat(nn.PLANE_G)
    assert step == len(bl)
    return (losses.cpu().numpy().astype(np.float64), m.split(p.astype(np.float64)),
            m.split(g.astype(np.float64)))


def fp32_one_step(w: synth.Workload, batch=None, f32_tc=None, head_gemm=None):
    """One fp32 step from a shared state: loss, every gradient element and
    every parameter element against the oracle with the arithmetic-derived
    bounds of tests/parity.py."""
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, 1, B)
    m = make_model(w, B, params0, f32_tc=f32_tc, head_gemm=head_gemm)
    g_losses, g_params, g_grads = gpu_run(m, w, bl)
    m.close()
    o_losses, o_params, _, _, o_grads = P.oracle_run(w, params0, bl, "fp64")
    assert abs(g_losses[0] - o_losses[0]) <= 1e-4 * abs(o_losses[0])
    kappa = P.oracle_abs_sums(w, params0, *bl[0], "fp64")
    lr, eps = P.hyper32(w)[0], P.hyper32(w)[3]
    for i, (g, go, k, p, po) in enumerate(zip(g_grads, o_grads, kappa, g_params, o_params)):
        tg = P.fp32_grad_tol(k)
        assert np.all(np.abs(g - go) <= tg), (i, np.max(np.abs(g - go) / tg))
        tp = P.fp32_first_step_param_tol(po, go, tg, lr, eps)
        assert np.all(np.abs(p - po) <= tp), (i, np.max(np.abs(p - po) / tp))
        # how many elements needed the eps-sensitivity term
        n_cond = int(np.sum(np.abs(p - po) > 1e-4 * np.maximum(np.abs(po), lr)))
        assert n_cond <= 1e-3 * p.size + 2, (i, n_cond)


def trajectory_ensemble(w: synth.Workload, n_steps: int, batch=None, one_graph=False, f32_tc=None):
    """Free-running trajectory against the oracle and its perturbed ensemble."""
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, n_steps, B)
    m = make_model(w, B, params0, f32_tc=f32_tc)
    g_losses, g_params, g_grads = gpu_run(m, w, bl, one_graph)
    m.close()
    p0 = [P.to64(p) for p in params0]
    mode = P.oracle_mode(w)
    ref = P.oracle_run(w, params0, bl, mode)
    ens = [P.oracle_run(w, params0, bl, mode, perturb_seed=s + 1) for s in range(P.ENSEMBLE_RUNS)]
    reports = []
    if w.dtype == synth.F32:
        reports.append(P.loss_ensemble_check("loss", g_losses, ref[0], [e[0] for e in ens], 1e-4))
        lr = P.hyper32(w)[0]
        scale = [np.maximum(np.abs(r), lr) for r in ref[1]]
        reports.append(P.ensemble_check("params", g_params, ref[1], [e[1] for e in ens], scale, 1e-4))
    else:
        exact = P.oracle_run(w, params0, bl, "bf16")
        rel = np.abs(g_losses - np.array(exact[0])) / np.abs(exact[0])
        assert rel.max() <= 2e-2, (rel.max(), g_losses, exact[0])          # stated, strict
        reports.append(P.loss_ensemble_check("loss", g_losses, ref[0], [e[0] for e in ens], 1e-3))
        scale = [np.max(np.abs(r - q)) for r, q in zip(ref[1], p0)]
        reports.append(P.ensemble_check("params", g_params, ref[1], [e[1] for e in ens], scale, 3e-2))
        if n_steps == 1:
            gs = [np.max(np.abs(g)) for g in ref[4]]
            reports.append(P.ensemble_check("grads", g_grads, ref[4], [e[4] for e in ens], gs, 3e-2))
    return reports


# --------------------------------------------------------------------------
# fp32: one step, element by element
# --------------------------------------------------------------------------
# f32_tc = 1: GEMMs on the tensor cores with fp32 operands as three bf16
# planes (the default); 0: FFMA.
F32_MODES = [pytest.param(1, id="tc3planes"), pytest.param(0, id="ffma")]


@pytest.mark.parametrize("f32_tc", F32_MODES)
def test_mnist_mlp_b64_one_step(f32_tc):
    fp32_one_step(W["mnist_mlp_b64"], f32_tc=f32_tc)


@pytest.mark.parametrize("f32_tc", F32_MODES)
def test_mnist_mlp_b4096_one_step_full_size(f32_tc):
    fp32_one_step(W["mnist_mlp_b4096"], f32_tc=f32_tc)


@pytest.mark.parametrize("f32_tc", F32_MODES)
def test_mnist_mlp_ragged_batch_one_step(f32_tc):
    fp32_one_step(W["mnist_mlp_b64"], batch=333, f32_tc=f32_tc)


def test_mnist_mlp_large_batch_one_step():
    """Batch 6000: 47 row tiles, too many for CTA pairs in the layer-1 forward
    (94 tiles of 128 x 128) but not in the layer-2 forward, so that forward
    runs one CTA per tile while the output layer is still folded into the
    layer-2 forward; element by element within the fp32 bounds."""
    w = W["mnist_mlp_b4096"]
    m = make_model(w, 6000, f32_tc=1)
    x, y = P.batches(w, 1, 6000)[0]
    prof = nn.mlp_profile_step(m.h, x.to(DEV).data_ptr(), y.to(DEV).data_ptr(), w.lr, w.beta1, w.beta2, w.eps,
                               w.wd, None, m.stream())
    m.close()
    names = [n for n, _ in prof]
    assert "tc_gemm_fwd_head" in names and "head_ce" not in names
    fp32_one_step(w, batch=6000, f32_tc=1)


@pytest.mark.parametrize("batch", [4096, 333, 64])
def test_mnist_mlp_separate_output_layer_kernel_one_step(batch):
    """With the output layer kept out of the forward GEMM's epilogue
    (MLP_OPT_HEAD_IN_GEMM 0) the step runs the separate fused output-layer
    kernel; element by element within the same fp32 bounds."""
    fp32_one_step(W["mnist_mlp_b4096"], batch=batch, f32_tc=1, head_gemm=0)


def test_mnist_mlp_output_layer_placement():
    """By default the fp32-plane step folds the output layer into the layer-2
    forward (one kernel fewer); the option restores the separate kernel."""
    w = W["mnist_mlp_b4096"]
    x, y = P.batches(w, 1)[0]
    names = {}
    for hg in (1, 0):
        m = make_model(w, f32_tc=1, head_gemm=hg)
        xd, yd = x.to(DEV), y.to(DEV)
        prof = nn.mlp_profile_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps, w.wd, None,
                                   m.stream())
        names[hg] = [n for n, _ in prof]
        m.close()
    assert "tc_gemm_fwd_head" in names[1] and "head_ce" not in names[1]
    assert "head_ce" in names[0] and "tc_gemm_fwd_head" not in names[0]
    assert len(names[1]) == len(names[0]) - 1


def test_f32_tensor_core_mode_runs_tensor_core_kernels():
    """The fp32 step's GEMMs run on the tcgen05 kernels in the default mode
    and on the FFMA kernels with the option off."""
    w = W["mnist_mlp_b4096"]
    x, y = P.batches(w, 1)[0]
    names = {}
    for tc in (1, 0):
        m = make_model(w, f32_tc=tc)
        xd, yd = x.to(DEV), y.to(DEV)
        prof = nn.mlp_profile_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps, w.wd, None,
                                   m.stream())
        names[tc] = [n for n, _ in prof]
        m.close()
    assert "split3" in names[1] and "tc_gemm_fwd" in names[1] and "tc_gemm_wgrad" in names[1]
    assert not any(n.startswith("simt") for n in names[1])
    assert "simt_gemm_fwd" in names[0] and "split3" not in names[0]


# --------------------------------------------------------------------------
# Trajectories against the oracle ensemble
# --------------------------------------------------------------------------
@pytest.mark.parametrize("f32_tc", F32_MODES)
def test_mnist_mlp_b64_three_steps(f32_tc):
    trajectory_ensemble(W["mnist_mlp_b64"], 3, f32_tc=f32_tc)


def test_cifar_mlp_reduced_batch_one_step():
    trajectory_ensemble(W["cifar_mlp_b8192"], 1, batch=320)


def test_cifar_mlp_reduced_batch():
    trajectory_ensemble(W["cifar_mlp_b8192"], 3, batch=320)


def test_lm_block_reduced_batch():
    trajectory_ensemble(W["lm_block_t16384"], 2, batch=200)


def test_deep_narrow_reduced_batch_one_step():
    trajectory_ensemble(W["deep_narrow_b65536"], 1, batch=300)


def test_deep_narrow_reduced_batch_one_graph():
    trajectory_ensemble(W["deep_narrow_b65536"], 4, batch=300, one_graph=True)


# --------------------------------------------------------------------------
# Full-size closed form: all-zero parameters
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_zero_params_closed_form_full_size(name):
    """W = b = 0 => h = 0, z = 0, loss = ln C; only the last bias has a
    gradient, db_c = 1/C - n_c/B, so after one AdamW step
    b_c = -lr g/(|g| + eps) and every other parameter stays exactly 0.
    This pins label indexing, CE, the fused bias-gradient and AdamW end to end
    at the workload's full size and launch configuration."""
    w = W[name]
    m = make_model(w)
    m.write_flat(np.zeros(m.n_params, np.float32), nn.PLANE_P, 0)
    x, y = synth.make_batch(w, 0)
    loss = m.train_step(x.to(DEV), y.to(DEV), w.lr, w.beta1, w.beta2, w.eps, w.wd)
    m.check_errors()
    C = w.n_classes
    assert abs(loss.item() - math.log(C)) <= 1e-6 * math.log(C)
    p, _ = m.read_flat(nn.PLANE_P)
    parts = m.split(p)
    for t in parts[:-1]:
        assert np.all(t == 0)
    n_c = np.bincount(y.numpy(), minlength=C)
    B = w.batch
    # dz_ic = (1/C - [y_i = c]) / B as the kernel forms it: fp32 products,
    # then stored in the model dtype (bf16: round to nearest even)
    f = np.float32
    gs, inv_s = f(1.0 / B), f(1.0) / f(C)
    a, b = f(inv_s * gs), f(f(inv_s - f(1.0)) * gs)
    if w.dtype == synth.BF16:
        a, b = (float(torch.tensor(float(v)).to(torch.bfloat16).float()) for v in (a, b))
    a, b = float(a), float(b)
    g = (B - n_c) * a + n_c * b
    dg = 2.0 ** -20 * ((B - n_c) * abs(a) + n_c * abs(b))   # fp32 summation error
    lr, eps = P.hyper32(w)[0], P.hyper32(w)[3]
    want = -lr * g / (np.abs(g) + eps)
    sure = np.abs(g) > 10 * dg
    np.testing.assert_allclose(parts[-1][sure], want[sure], rtol=1e-3, atol=1e-3 * lr)
    assert np.all(np.abs(parts[-1]) <= lr * (1 + 1e-3))
    assert sure.sum() >= C - 2
    m.close()


# --------------------------------------------------------------------------
# Full-size sampled forward: logits of sampled rows against the oracle
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_forward_sampled_rows_full_size(name):
    w = W[name]
    params0 = synth.make_params(w)
    m = make_model(w, params=params0)
    x, _ = synth.make_batch(w, 0)
    logits, am = m.forward(x.to(DEV))
    torch.cuda.synchronize()
    rows = np.unique(np.random.default_rng(7).integers(0, w.batch, 24))
    rows = np.concatenate([rows, [0, w.batch - 1]])
    p64 = [P.to64(p) for p in params0]
    mode = P.oracle_mode(w, exact=False)
    fw = om.forward(p64, P.to64(x[rows]), w.acts, mode)
    z_ref = fw["z"]
    z = P.to64(logits[rows])
    scale = np.max(np.abs(z_ref), axis=1, keepdims=True)
    tol = 1e-4 if w.dtype == synth.F32 else 3e-2
    assert np.all(np.abs(z - z_ref) <= tol * scale), np.max(np.abs(z - z_ref) / scale)
    # argmax: exact wherever the oracle's top-2 gap exceeds the tolerance
    amr = om.argmax_rows(z_ref)
    s = np.sort(z_ref, axis=1)
    gap = s[:, -1] - s[:, -2] if z_ref.shape[1] > 1 else np.full(len(rows), np.inf)
    clear = gap > 2 * tol * scale[:, 0]
    assert np.array_equal(am.cpu().numpy()[rows][clear], amr[clear])
    # and always consistent with the GPU's own logits (lowest index on ties)
    assert np.array_equal(am.cpu().numpy(), np.argmax(P.to64(logits), axis=1))
    m.close()


def test_fp32_forward_runs_on_the_plane_gemms():
    """mlp_forward of an fp32 model runs its hidden layers on the tensor
    cores as three bf16 planes (as the training step does; the small output
    layer on the FFMA pipes from the exactly joined fp32 activation), and on
    the FFMA pipes throughout with the option off; logits agree with the
    oracle within the fp32 bound either way and argmax is the same."""
    w = W["mnist_mlp_b4096"]
    params0 = synth.make_params(w)
    x, _ = synth.make_batch(w, 0)
    xd = x.to(DEV)
    out = {}
    for tc in (1, 0):
        m = make_model(w, params=params0, f32_tc=tc)
        logits = torch.empty((w.batch, w.n_classes), dtype=torch.float32, device=DEV)
        am = torch.empty(w.batch, dtype=torch.int32, device=DEV)
        prof = nn.mlp_profile_forward(m.h, xd.data_ptr(), logits.data_ptr(), am.data_ptr(), m.stream())
        out[tc] = ([n for n, _ in prof], P.to64(logits), am.cpu().numpy())
        m.close()
    names1, names0 = out[1][0], out[0][0]
    assert names1[:3] == ["split3", "tc_gemm_fwd", "tc_gemm_fwd"] and "join3" in names1, names1
    assert not any(n.startswith("tc") for n in names0) and "split3" not in names0, names0
    p64 = [P.to64(p) for p in params0]
    z_ref = om.forward(p64, P.to64(x), w.acts, "fp64")["z"]
    scale = np.max(np.abs(z_ref), axis=1, keepdims=True)
    for tc in (1, 0):
        assert np.all(np.abs(out[tc][1] - z_ref) <= 1e-4 * scale)
        s = np.sort(z_ref, axis=1)
        clear = (s[:, -1] - s[:, -2]) > 2e-4 * scale[:, 0]
        assert np.array_equal(out[tc][2][clear], om.argmax_rows(z_ref)[clear])


# --------------------------------------------------------------------------
# Determinism, graph vs eager, error reporting
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["mnist_mlp_b4096", "cifar_mlp_b8192"])
def test_bitwise_deterministic_and_graph_equals_eager(name):
    w = W[name]
    params0 = synth.make_params(w)
    bl = P.batches(w, 2)
    res = []
    # graph with early-launch edges (twice), graph with plain edges, eager
    for graph, pdl in ((True, 1), (True, 1), (True, 0), (False, 1)):
        m = make_model(w, params=params0, graph=graph)
        m.set_option(nn.OPT_PDL, pdl)
        losses, _, _ = gpu_run(m, w, bl)
        p, _ = m.read_flat(nn.PLANE_P)
        res.append((losses, p))
        m.close()
    for l_, p_ in res[1:]:
        assert np.array_equal(l_, res[0][0])
        assert np.array_equal(p_, res[0][1])


@pytest.mark.parametrize("head_gemm,bad", [(1, 10), (1, -1), (0, 10), (0, -3)])
def test_label_out_of_range_reported(head_gemm, bad):
    """A label outside [0, C) latches MLP_ERR_LABEL_RANGE, with the output
    layer folded into the layer-2 forward (default) and in its own kernel."""
    w = W["mnist_mlp_b64"]
    m = make_model(w, head_gemm=head_gemm)
    x, y = synth.make_batch(w, 0)
    y[5] = bad
    m.train_step(x.to(DEV), y.to(DEV), w.lr)
    with pytest.raises(nn.MlpError) as e:
        m.check_errors()
    assert e.value.status == 5
    m.check_errors()   # cleared
    m.close()


def test_kaiming_init_statistics():
    w = W["cifar_mlp_b8192"]
    m = make_model(w)
    p, step = m.read_flat(nn.PLANE_P)
    assert step == 0
    parts = m.split(p)
    for l in range(w.n_layers):
        Wl, bl = parts[2 * l], parts[2 * l + 1]
        std = math.sqrt(2.0 / w.dims[l])
        assert abs(Wl.std() / std - 1) < 0.02 + 3 / math.sqrt(Wl.size)
        assert abs(Wl.mean()) < 5 * std / math.sqrt(Wl.size)
        assert np.all(bl == 0)
    m.close()


def test_shape_mismatch_and_bad_args_fail_before_enqueue():
    with pytest.raises(nn.MlpError):
        nn.Model([100, 20, 10], None, nn.ACT_RELU, nn.BF16, batch=8)    # 100 % 8 != 0 in bf16
    w = W["mnist_mlp_b64"]
    m = make_model(w)
    x, y = synth.make_batch(w, 0)
    with pytest.raises(nn.MlpError):
        nn.mlp_train_step(m.h, x.to(DEV).data_ptr(), y.to(DEV).data_ptr(), -1.0, 0.9, 0.999, 1e-8, 0.0, None,
                          0)
    m.close()


# --------------------------------------------------------------------------
# Fused output layer (head + CE + its VJPs) against the unfused kernels
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,batch", [("mnist_mlp_b4096", None), ("mnist_mlp_b64", 333)])
def test_fused_head_matches_unfused_path(name, batch):
    """Same step with and without the fused output layer (GEMMs on the FFMA
    pipes in both): the arithmetic and rounding points are the same, only the
    order of fp32 additions differs, so loss and gradients agree to fp32
    accumulation error."""
    w = W[name]
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, 1, B)
    res = []
    for fuse in (1, 0):
        m = make_model(w, B, params0, f32_tc=0)
        m.set_option(nn.OPT_FUSE_HEAD, fuse)
        res.append(gpu_run(m, w, bl))
        m.close()
    (l1, p1, g1), (l0, p0_, g0) = res
    assert abs(l1[0] - l0[0]) <= 1e-6 * abs(l0[0])
    kappa = P.oracle_abs_sums(w, params0, *bl[0], "fp64")
    for a, b, k in zip(g1, g0, kappa):
        assert np.all(np.abs(a - b) <= P.fp32_grad_tol(k))


# --------------------------------------------------------------------------
# Host-input steps (copies on the library's copy stream, two input slots)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,batch", [("mnist_mlp_b4096", None), ("cifar_mlp_b8192", 512)])
def test_train_step_host_matches_device_inputs(name, batch):
    """mlp_train_step_host on pinned host batches gives bit-identical losses and
    parameters to mlp_train_step on the same batches already on the device,
    over more steps than input slots (the slots are reused)."""
    w = W[name]
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, 5, B)
    m = make_model(w, B, params0)
    d_losses, d_params, _ = gpu_run(m, w, bl)
    m.close()
    m = make_model(w, B, params0)
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    hl = torch.zeros(len(bl), dtype=torch.float32).pin_memory()
    hx = [x.contiguous().pin_memory() for x, _ in bl]
    hy = [y.contiguous().pin_memory() for _, y in bl]
    for i in range(len(bl)):
        m.train_step_host(hx[i], hy[i], loss=hl[i:i + 1], **hyper)
    torch.cuda.synchronize()
    m.check_errors()
    p, step = m.read_flat(nn.PLANE_P)
    m.close()
    assert step == len(bl)
    assert np.array_equal(hl.numpy().astype(np.float64), d_losses)
    assert np.array_equal(P.flat(m.split(p.astype(np.float64))), P.flat(d_params))


# --------------------------------------------------------------------------
# 2-SM GEMMs (CTA pairs, 256 x 256 tiles): the same sums as the one-SM kernels
# --------------------------------------------------------------------------
RAGGED_2SM = synth.Workload("ragged_2sm", (320, 264, 520, 100), (om.ACT_GELU_TANH, om.ACT_RELU), synth.BF16, 300, 2,
                            1e-3, 0.9, 0.999, 1e-8, 0.01, "normal", 12)
# enough pair tiles for the 2-SM forwards by default (8 x 11), so they also
# store their activations transposed and the weight gradients read them
# K-major: 2000 rows (a 208-row pair tile, a 16-row K tail), 2600 / 2520 columns
RAGGED_PAIRS = synth.Workload("ragged_pairs", (1024, 2600, 2520, 100), (om.ACT_GELU_TANH, om.ACT_RELU), synth.BF16,
                              2000, 2, 1e-3, 0.9, 0.999, 1e-8, 0.01, "normal", 13)


@pytest.mark.parametrize("w,batch", [(W["cifar_mlp_b8192"], None), (W["lm_block_t16384"], 2048),
                                     (W["deep_narrow_b65536"], 3000), (RAGGED_2SM, None), (RAGGED_PAIRS, None)],
                         ids=["cifar_full", "lm_block_2048", "deep_narrow_3000", "ragged", "ragged_pairs"])
def test_gemm_2sm_equals_one_sm(w, batch):
    """The step with the bf16 forward / dgrad GEMMs on CTA pairs with 2-SM
    MMAs (MLP_OPT_GEMM_2SM 1) and with every GEMM on one SM (0): each output
    element is the same sequence of 16-deep MMA accumulations, so losses,
    parameters and gradients agree bit for bit.  Ragged case: 300 rows (one
    full and one partial 256-row pair tile), 264 and 520 columns, GELU and
    ReLU layers (the ReLU bits and the GELU pre-activation on pair tiles)."""
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, 2, B)
    res, names = [], []
    for on in (1, 0):
        m = make_model(w, B, params0)
        m.set_option(nn.OPT_GEMM_2SM, on)
        x, y = bl[0]
        prof = nn.mlp_profile_step(m.h, x.to(DEV).data_ptr(), y.to(DEV).data_ptr(), w.lr, w.beta1, w.beta2, w.eps,
                                   w.wd, None, m.stream())
        names.append([n for n, _ in prof])
        m.close()
        m = make_model(w, B, params0)
        m.set_option(nn.OPT_GEMM_2SM, on)
        losses, p, g = gpu_run(m, w, bl)
        m.close()
        res.append((losses, P.flat(p), P.flat(g)))
    assert "tc2_gemm_fwd" in names[0] and "tc2_gemm_dgrad" in names[0]
    assert not any(n.startswith("tc2_") for n in names[1])
    for a, b in zip(res[0], res[1]):
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# ReLU masks as bits (bf16): identical to reading the stored activation
# --------------------------------------------------------------------------
RAGGED_BF16 = synth.Workload("bits_ragged", (64, 200, 72, 10), (om.ACT_RELU, om.ACT_RELU), synth.BF16, 300, 2,
                             1e-3, 0.9, 0.999, 1e-8, 0.01, "normal", 11)


@pytest.mark.parametrize("w,batch", [(W["cifar_mlp_b8192"], None), (W["deep_narrow_b65536"], 3000),
                                     (RAGGED_BF16, None)], ids=["cifar_full", "deep_narrow_3000", "ragged"])
def test_relu_bits_equal_stored_activation_mask(w, batch):
    B = w.batch if batch is None else batch
    params0 = synth.make_params(w)
    bl = P.batches(w, 2, B)
    res = []
    for bits in (1, 0):
        m = make_model(w, B, params0)
        m.set_option(nn.OPT_RELU_BITS, bits)
        losses, p, g = gpu_run(m, w, bl)
        m.close()
        res.append((losses, P.flat(p), P.flat(g)))
    for a, b in zip(res[0], res[1]):
        assert np.array_equal(a, b)
