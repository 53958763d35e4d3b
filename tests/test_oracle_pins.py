"""Pins of the CPU oracle to facts fixed outside it.

Each test checks the oracle against something other than itself: brute force
on tiny inputs, central finite differences, closed forms, exact special cases,
or a library routine that computes the same textbook definition (torch in
float64).  The planted-mistake tests at the end show that a plausible slip in
the oracle (a dropped mask, a wrong scale, a misplaced epsilon, a transposed
operand) fails at least one pin.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import mlp_oracle as om

RELU, GELU, NONE = om.ACT_RELU, om.ACT_GELU_TANH, om.ACT_NONE


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------
# bf16 rounding: exact special case of a library conversion (fp32 -> bf16 RNE)
# --------------------------------------------------------------------------
def test_rne_bf16_matches_torch_cast_on_fp32_values():
    rng = np.random.default_rng(0)
    a = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),    # fp32 subnormals
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
    ])
    # exact ties: bf16 value + half a bf16 ulp (both tie directions)
    base = torch.from_numpy(rng.standard_normal(4000).astype(np.float32)).to(torch.bfloat16)
    bits = base.view(torch.int16).to(torch.int32) & 0xFFFF
    tie = ((bits << 16) | 0x8000).to(torch.int32).view(torch.float32).numpy()
    a = np.concatenate([a, tie, np.float32([0.0, -0.0, 1.0, -1.0, 65504.0])])
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = om.rne_bf16(a.astype(np.float64))
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# Linear layer: brute-force triple loop on a tiny shape
# --------------------------------------------------------------------------
def test_rne_bf16_equals_its_definition_on_fp64_values():
    """The rounding on fp64 inputs (which torch's cast from fp32 cannot
    give) against the definition written out: quantum q = 2^max(e - 8, -133)
    for |a| in [2^(e-1), 2^e), a rounded to a multiple of q, half to even;
    ties at 8 significant bits of both parities, bf16 subnormals, overflow."""
    rng = np.random.default_rng(21)
    a = np.concatenate([rng.standard_normal(200000) * np.exp(rng.uniform(-200, 200, 200000)),
                        rng.standard_normal(50000) * 2.0 ** rng.integers(-140, -120, 50000),
                        (rng.integers(128, 256, 50000) * 2 + 1) / 2 * 2.0 ** rng.integers(-100, 100, 50000),
                        (rng.integers(0, 1024, 20000) + 0.5) * 2.0 ** -133,
                        [(2 - 2.0 ** -8) * 2.0 ** 127, (2 - 2.0 ** -9) * 2.0 ** 127, 2.0 ** -126, 2.0 ** -134]])
    a = np.concatenate([a, -a])
    _, e = np.frexp(a)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    want = np.rint(a / q) * q
    want[np.abs(want) > (2 - 2.0 ** -7) * 2.0 ** 127] = np.inf * np.sign(want[np.abs(want) > (2 - 2.0 ** -7) * 2.0 ** 127])
    got = om.rne_bf16(a)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_linear_bruteforce():
    X, W, b = _rand((3, 5), 1), _rand((4, 5), 2), _rand(4, 3)
    want = np.zeros((3, 4))
    for i in range(3):
        for n in range(4):
            s = b[n]
            for k in range(5):
                s += X[i, k] * W[n, k]
            want[i, n] = s
    assert np.allclose(om.linear(X, W, b), want, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# Activations
# --------------------------------------------------------------------------
def test_relu_and_mask():
    u = np.array([-2.0, -0.0, 0.0, 1e-30, 3.0])
    assert np.array_equal(om.act_forward(u, RELU), [0, 0, 0, 1e-30, 3.0])


def test_gelu_matches_torch_tanh_gelu_and_its_autograd():
    u = torch.linspace(-8, 8, 4001, dtype=torch.float64, requires_grad=True)
    y = F.gelu(u, approximate="tanh")
    (g,) = torch.autograd.grad(y.sum(), u)
    un = u.detach().numpy()
    assert np.allclose(om.act_forward(un, GELU), y.detach().numpy(), rtol=0, atol=1e-15)
    assert np.allclose(om.gelu_tanh_grad(un), g.numpy(), rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# Softmax cross-entropy
# --------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 10, 100, 32000])
def test_ce_zero_logits_closed_form(C):
    B = 7
    y = np.arange(B) % C
    loss, dz = om.softmax_ce(np.zeros((B, C)), y)
    assert np.allclose(loss, math.log(C), rtol=0, atol=1e-13)
    want = np.full((B, C), 1.0 / C)
    want[np.arange(B), y] -= 1.0
    assert np.allclose(dz, want / B, rtol=0, atol=1e-17)


def test_ce_matches_torch_cross_entropy_and_rows_sum_to_zero():
    B, C = 33, 17
    z = _rand((B, C), 5, 4.0)
    y = np.random.default_rng(6).integers(0, C, B)
    zt = torch.tensor(z, requires_grad=True)
    lt = F.cross_entropy(zt, torch.tensor(y), reduction="mean")
    (gt,) = torch.autograd.grad(lt, zt)
    loss, dz = om.softmax_ce(z, y)
    assert abs(loss.mean() - lt.item()) < 1e-13
    assert np.allclose(dz, gt.numpy(), rtol=0, atol=1e-15)
    assert np.allclose(dz.sum(axis=1), 0.0, atol=1e-16)
    p = dz * B
    p[np.arange(B), y] += 1.0
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)


def test_ce_huge_margin_and_shift_invariance():
    B, C = 4, 9
    y = np.array([0, 3, 8, 5])
    z = np.zeros((B, C))
    z[np.arange(B), y] = 80.0
    loss, dz = om.softmax_ce(z, y)
    assert np.all(loss < 1e-30) and np.all(np.abs(dz) < 1e-30)
    z2 = _rand((B, C), 7)
    l1, d1 = om.softmax_ce(z2, y)
    l2, d2 = om.softmax_ce(z2 + 1000.0, y)
    assert np.allclose(l1, l2, atol=1e-12) and np.allclose(d1, d2, atol=1e-15)


def test_ce_label_out_of_range_is_an_error():
    with pytest.raises(ValueError):
        om.softmax_ce(np.zeros((2, 3)), np.array([0, 3]))
    with pytest.raises(ValueError):
        om.softmax_ce(np.zeros((2, 3)), np.array([-1, 0]))


def test_argmax_lowest_index_on_ties_bruteforce():
    z = np.array([[1, 3, 3, 0], [5, 5, 5, 5], [-1, -2, -1, -3], [0, 0, 0, 7]], float)
    want = []
    for row in z:
        best = 0
        for j in range(len(row)):
            if row[j] > row[best]:
                best = j
        want.append(best)
    assert list(om.argmax_rows(z)) == want


# --------------------------------------------------------------------------
# Backward: central finite differences and torch autograd (float64)
# --------------------------------------------------------------------------
def _tiny_net(dims, seed):
    ps = []
    for l in range(len(dims) - 1):
        ps += [_rand((dims[l + 1], dims[l]), seed + l, 0.7), _rand(dims[l + 1], seed + 50 + l, 0.3)]
    return ps


def _loss(ps, x, y, acts):
    fw = om.forward(ps, x, acts, "fp64")
    l, _ = om.softmax_ce(fw["z"], y)
    return l.mean(), fw


@pytest.mark.parametrize("acts", [(RELU, RELU), (GELU, NONE), (GELU, RELU)])
def test_backward_central_finite_differences(acts):
    dims = [5, 4, 3, 3]
    B = 4
    x = _rand((B, dims[0]), 11)
    y = np.array([0, 2, 1, 2])
    ps = _tiny_net(dims, 20)
    _, fw = _loss(ps, x, y, acts)
    h = 1e-6
    # keep every ReLU pre-activation at least 10h away from the kink
    for l, a in enumerate(acts):
        if a == RELU:
            assert np.min(np.abs(fw["u"][l])) > 10 * h * 100
    _, dz = om.softmax_ce(fw["z"], y)
    grads = om.backward(fw, dz, acts, "fp64")
    for pi, P in enumerate(ps):
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            old = P[idx]
            P[idx] = old + h
            lp, _ = _loss(ps, x, y, acts)
            P[idx] = old - h
            lm, _ = _loss(ps, x, y, acts)
            P[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        assert np.allclose(grads[pi], fd, rtol=1e-6, atol=1e-8), (pi, grads[pi], fd)


def test_backward_matches_torch_autograd():
    dims = [12, 9, 7, 5]
    acts = (RELU, GELU)
    B = 6
    x = _rand((B, dims[0]), 31)
    y = np.array([0, 4, 1, 2, 3, 4])
    ps = _tiny_net(dims, 40)
    tp = [torch.tensor(p, requires_grad=True) for p in ps]
    h = torch.tensor(x)
    for l in range(3):
        h = F.linear(h, tp[2 * l], tp[2 * l + 1])
        if l < 2:
            h = F.relu(h) if acts[l] == RELU else F.gelu(h, approximate="tanh")
    lt = F.cross_entropy(h, torch.tensor(y))
    tg = torch.autograd.grad(lt, tp)
    loss, _ = _loss(ps, x, y, acts)
    assert abs(loss - lt.item()) < 1e-13
    fw = om.forward(ps, x, acts, "fp64")
    _, dz = om.softmax_ce(fw["z"], y)
    grads = om.backward(fw, dz, acts, "fp64")
    for g, t in zip(grads, tg):
        assert np.allclose(g, t.numpy(), rtol=1e-12, atol=1e-14)


def test_one_layer_net_is_logistic_regression():
    """L = 1: dW = (softmax(z) - Y)^T X / B and db = colsum(softmax - Y) / B."""
    B, K, C = 9, 6, 4
    x = _rand((B, K), 51)
    y = np.random.default_rng(52).integers(0, C, B)
    W, b = _rand((C, K), 53), _rand(C, 54)
    fw = om.forward([W, b], x, (), "fp64")
    _, dz = om.softmax_ce(fw["z"], y)
    gW, gb = om.backward(fw, dz, (), "fp64")
    z = x @ W.T + b
    P = np.exp(z - z.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    Y = np.eye(C)[y]
    assert np.allclose(gW, (P - Y).T @ x / B, atol=1e-15)
    assert np.allclose(gb, (P - Y).sum(0) / B, atol=1e-15)


# --------------------------------------------------------------------------
# AdamW: first-step closed form, zero gradient, torch.optim.AdamW (float64)
# --------------------------------------------------------------------------
def test_adamw_first_step_closed_form():
    p0, g = _rand(1000, 61), _rand(1000, 62, 1e-3)
    g[:5] = [0.0, 1e-9, -1e-9, 1e-8, -3e-8]
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    p1, m1, v1 = om.adamw(p0, g, 0 * p0, 0 * p0, 1, lr, b1, b2, eps, wd)
    want = p0 - lr * (g / (np.abs(g) + eps) + wd * p0)
    assert np.allclose(p1, want, rtol=0, atol=1e-16)
    assert np.allclose(m1, 0.1 * g) and np.allclose(v1, 0.001 * g * g)


def test_adamw_zero_gradient_is_pure_decay():
    p0 = _rand(100, 63)
    p, m, v = p0, 0 * p0, 0 * p0
    for t in range(1, 6):
        p, m, v = om.adamw(p, 0 * p0, m, v, t, 3e-4, 0.9, 0.999, 1e-8, 0.05)
    assert np.allclose(p, p0 * (1 - 3e-4 * 0.05) ** 5, rtol=1e-15, atol=0)


def test_adamw_matches_torch_optim_adamw_100_steps():
    rng = np.random.default_rng(64)
    p0 = rng.standard_normal(500)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.1
    tp = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(500), np.zeros(500)
    for t in range(1, 101):
        g = rng.standard_normal(500) * 10 ** rng.uniform(-6, 0)
        tp.grad = torch.tensor(g)
        opt.step()
        p, m, v = om.adamw(p, g, m, v, t, lr, b1, b2, eps, wd)
    assert np.allclose(p, tp.detach().numpy(), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# Adam with L2, SGD with momentum, global-norm clipping: closed forms and the
# torch.optim / torch.nn.utils routines of the same definitions (float64)
# --------------------------------------------------------------------------
def test_adam_l2_first_step_closed_form():
    p0, g = _rand(1000, 91), _rand(1000, 92, 1e-3)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    p1, m1, v1 = om.adam_l2(p0, g, 0 * p0, 0 * p0, 1, lr, b1, b2, eps, wd)
    gp = g + wd * p0          # the decay enters the moments, not the step
    assert np.allclose(p1, p0 - lr * gp / (np.abs(gp) + eps), rtol=0, atol=1e-15)
    assert np.allclose(m1, 0.1 * gp, rtol=1e-15) and np.allclose(v1, 0.001 * gp * gp, rtol=1e-15)


def test_adam_l2_matches_torch_optim_adam_100_steps():
    rng = np.random.default_rng(93)
    p0 = rng.standard_normal(500)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.1
    tp = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.Adam([tp], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(500), np.zeros(500)
    for t in range(1, 101):
        g = rng.standard_normal(500) * 10 ** rng.uniform(-6, 0)
        tp.grad = torch.tensor(g)
        opt.step()
        p, m, v = om.adam_l2(p, g, m, v, t, lr, b1, b2, eps, wd)
    assert np.allclose(p, tp.detach().numpy(), rtol=0, atol=1e-13)


@pytest.mark.parametrize("momentum,wd", [(0.0, 0.0), (0.9, 0.0), (0.9, 0.01), (0.5, 0.1)])
def test_sgd_matches_torch_optim_sgd_50_steps(momentum, wd):
    rng = np.random.default_rng(94)
    p0 = rng.standard_normal(300)
    lr = 0.03
    tp = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.SGD([tp], lr=lr, momentum=momentum, weight_decay=wd)
    p, buf = p0.copy(), np.zeros(300)
    for _ in range(50):
        g = rng.standard_normal(300) * 10 ** rng.uniform(-3, 0)
        tp.grad = torch.tensor(g)
        opt.step()
        p, buf = om.sgd(p, g, buf, lr, momentum, wd)
    assert np.allclose(p, tp.detach().numpy(), rtol=0, atol=1e-13)


def test_sgd_constant_gradient_closed_form():
    # buf_t = g (1 - mu^t) / (1 - mu), so p_T = p_0 - lr g sum_t (1 - mu^t) / (1 - mu)
    p0, g = _rand(64, 95), _rand(64, 96)
    lr, mu, T = 0.01, 0.9, 7
    p, buf = p0, 0 * p0
    for _ in range(T):
        p, buf = om.sgd(p, g, buf, lr, mu, 0.0)
    s = sum((1 - mu ** t) / (1 - mu) for t in range(1, T + 1))
    assert np.allclose(p, p0 - lr * g * s, rtol=0, atol=1e-14)
    assert np.allclose(buf, g * (1 - mu ** T) / (1 - mu), rtol=1e-14)


def test_clip_coef_closed_form():
    grads = [np.array([[3.0, 0.0]]), np.array([4.0])]           # ||G|| = 5
    assert om.clip_coef(grads, 1.0) == 1.0 / (5.0 + 1e-6)
    assert om.clip_coef(grads, 2.5) == 2.5 / (5.0 + 1e-6)
    assert om.clip_coef(grads, 10.0) == 1.0                        # below the threshold: unchanged
    assert om.clip_coef(grads, 0.0) == 1.0                         # off
    assert om.clip_coef([np.zeros(3)], 1.0) == 1.0                 # zero gradient: 1 / 1e-6 clamps to 1


def test_clip_matches_torch_clip_grad_norm():
    rng = np.random.default_rng(97)
    shapes = [(7, 5), (7,), (3, 7), (3,)]
    grads = [rng.standard_normal(s) * 0.3 for s in shapes]
    for max_norm in (0.1, 1.0, 100.0):
        ts = [torch.zeros(s, dtype=torch.float64, requires_grad=True) for s in shapes]
        for t_, g in zip(ts, grads):
            t_.grad = torch.tensor(g)
        total = torch.nn.utils.clip_grad_norm_(ts, max_norm)
        c = om.clip_coef(grads, max_norm)
        assert abs(float(total) - math.sqrt(sum(float((g ** 2).sum()) for g in grads))) < 1e-14
        for t_, g in zip(ts, grads):
            assert np.allclose(t_.grad.numpy(), g * c, rtol=1e-15, atol=0)


@pytest.mark.parametrize("optim", ["adamw", "adam", "sgd"])
@pytest.mark.parametrize("max_norm", [0.0, 0.05])
@pytest.mark.parametrize("loss_kind", ["ce", "mse"])
def test_whole_step_matches_torch_modules_and_optimizers(optim, max_norm, loss_kind):
    """One whole step of the oracle against torch (float64): nn.Linear + ReLU
    layers, F.cross_entropy or F.mse_loss (means), backward, clip_grad_norm_,
    the optimizer."""
    dims = [9, 7, 6, 5]
    acts = (RELU, RELU)
    B = 11
    ps = _tiny_net(dims, 98)
    x = _rand((B, dims[0]), 99)
    if loss_kind == "ce":
        y = np.random.default_rng(100).integers(0, dims[-1], B)
    else:
        y = _rand((B, dims[-1]), 100)
    lr, b1, b2, eps, wd = 1e-2, 0.9, 0.999, 1e-8, 0.05
    loss, newp, _, _, grads, ex = om.train_step(ps, [0 * p for p in ps], [0 * p for p in ps], 1, x, y, acts,
                                                lr, b1, b2, eps, wd, optim=optim, max_norm=max_norm,
                                                loss=loss_kind)
    tps = [torch.tensor(p, requires_grad=True) for p in ps]
    h = torch.tensor(x)
    for l in range(3):
        h = h @ tps[2 * l].T + tps[2 * l + 1]
        if l < 2:
            h = torch.relu(h)
    tl = F.cross_entropy(h, torch.tensor(y)) if loss_kind == "ce" else F.mse_loss(h, torch.tensor(y))
    tl.backward()
    if max_norm:
        torch.nn.utils.clip_grad_norm_(tps, max_norm)
        assert ex["clip"] < 1.0            # the threshold is below this gradient's norm
    opt = {"adamw": lambda: torch.optim.AdamW(tps, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd),
           "adam": lambda: torch.optim.Adam(tps, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd),
           "sgd": lambda: torch.optim.SGD(tps, lr=lr, momentum=b1, weight_decay=wd)}[optim]()
    opt.step()
    assert abs(loss - tl.item()) < 1e-13
    for a, b in zip(newp, tps):
        assert np.allclose(a, b.detach().numpy(), rtol=0, atol=1e-13)


@pytest.mark.parametrize("optim", ["adamw", "adam", "sgd"])
def test_run_steps_matches_torch_training_loop(optim):
    """The oracle's multi-step driver (run_steps: the step counter advancing
    from 1, moments carried from step to step, a fresh batch each step)
    against a torch training loop in float64 over six whole-network steps:
    nn.Linear + GELU / ReLU layers, F.cross_entropy, backward, the optimizer
    (noeira "A complete example": a loop of forward, loss, backward and an
    optimizer step over batches)."""
    dims = [9, 8, 7, 5]
    acts = (GELU, RELU)
    B, steps = 13, 6
    ps = _tiny_net(dims, 120)
    rng = np.random.default_rng(121)
    batches = [(rng.standard_normal((B, dims[0])), rng.integers(0, dims[-1], B)) for _ in range(steps)]
    lr, b1, b2, eps, wd = 3e-2, 0.8, 0.95, 1e-8, 0.05
    losses, p, m, v, _ = om.run_steps(ps, acts, batches, (lr, b1, b2, eps, wd), optim=optim)
    tps = [torch.tensor(q, requires_grad=True) for q in ps]
    opt = {"adamw": lambda: torch.optim.AdamW(tps, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd),
           "adam": lambda: torch.optim.Adam(tps, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd),
           "sgd": lambda: torch.optim.SGD(tps, lr=lr, momentum=b1, weight_decay=wd)}[optim]()
    t_losses = []
    for x, y in batches:
        opt.zero_grad()
        h = torch.tensor(x)
        for l in range(3):
            h = h @ tps[2 * l].T + tps[2 * l + 1]
            if l == 0:
                h = F.gelu(h, approximate="tanh")
            elif l == 1:
                h = torch.relu(h)
        tl = F.cross_entropy(h, torch.tensor(y))
        tl.backward()
        opt.step()
        t_losses.append(tl.item())
    assert np.allclose(losses, t_losses, rtol=0, atol=1e-12)
    for a, b in zip(p, tps):
        assert np.allclose(a, b.detach().numpy(), rtol=0, atol=1e-12)
    if optim != "sgd":   # the first moment against torch's optimizer state
        for a, b in zip(m, tps):
            assert np.allclose(a, opt.state[b]["exp_avg"].numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# MSE: brute force, torch mse_loss and its autograd (float64), closed forms
# --------------------------------------------------------------------------
def test_mse_bruteforce_and_torch():
    z, t = _rand((5, 3), 101), _rand((5, 3), 102)
    rows, dz = om.mse(z, t)
    for i in range(5):
        assert abs(rows[i] - sum((z[i, j] - t[i, j]) ** 2 for j in range(3))) < 1e-14
    tz = torch.tensor(z, requires_grad=True)
    tl = F.mse_loss(tz, torch.tensor(t))
    tl.backward()
    assert abs(rows.sum() / z.size - tl.item()) < 1e-15
    assert np.allclose(dz, tz.grad.numpy(), rtol=1e-15, atol=0)


def test_mse_closed_forms():
    z = _rand((4, 6), 103)
    rows, dz = om.mse(z, z)
    assert np.all(rows == 0) and np.all(dz == 0)              # perfect fit
    rows, dz = om.mse(z, z - 0.5)                             # constant offset a: loss a^2, dz 2a / (B C)
    assert np.allclose(rows, 6 * 0.25, rtol=1e-15) and np.allclose(dz, 1.0 / 24, rtol=1e-14)
    with pytest.raises(ValueError):
        om.mse(z, z[:, :5])


def test_mse_one_layer_net_is_least_squares():
    # one Linear layer under MSE: the gradient is (2 / (B C)) (XW^T + b - T)^T X,
    # the normal-equation residual of least squares
    B, K, C = 9, 4, 3
    W, b = _rand((C, K), 104), _rand(C, 105)
    x, t = _rand((B, K), 106), _rand((B, C), 107)
    loss, _, _, _, grads, _ = om.train_step([W, b], [0 * W, 0 * b], [0 * W, 0 * b], 1, x, t, (), 1e-3, 0.9, 0.999,
                                            1e-8, 0.0, loss="mse")
    r = x @ W.T + b - t
    assert abs(loss - np.mean(r ** 2)) < 1e-14
    assert np.allclose(grads[0], 2.0 / (B * C) * r.T @ x, rtol=1e-13, atol=1e-15)
    assert np.allclose(grads[1], 2.0 / (B * C) * r.sum(axis=0), rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------
# Whole step: all-zero parameters have a closed form
# --------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["fp64", "bf16", "bf16_mirror"])
def test_whole_step_zero_params_closed_form(mode):
    dims = [6, 5, 4, 7]
    acts = (RELU, GELU)
    B, C = 13, dims[-1]
    x = _rand((B, dims[0]), 71)
    y = np.random.default_rng(72).integers(0, C, B)
    ps = [np.zeros((dims[l + 1], dims[l])) if i == 0 else np.zeros(dims[l + 1])
          for l in range(3) for i in range(2)]
    lr, wd, eps = 1e-3, 0.01, 1e-8
    loss, newp, *_ = om.train_step(ps, [0 * p for p in ps], [0 * p for p in ps], 1,
                                   x, y, acts, lr, 0.9, 0.999, eps, wd, mode=mode)
    assert abs(loss - math.log(C)) < 1e-13
    n_c = np.bincount(y, minlength=C)
    g = 1.0 / C - n_c / B
    want_b = -lr * g / (np.abs(g) + eps)
    tol = 1e-6 if mode == "bf16_mirror" else 1e-15   # dz rounded to bf16 in mirror mode
    assert np.allclose(newp[-1], want_b, rtol=tol, atol=1e-18)
    for p in newp[:-1]:
        assert np.all(p == 0)


# --------------------------------------------------------------------------
# Declared bf16 rounding points
# --------------------------------------------------------------------------
def test_mirror_mode_rounds_at_declared_points_only():
    dims = [8, 6, 5]
    x = om.rne_bf16(_rand((4, 8), 81))
    ps = _tiny_net(dims, 82)
    fwm = om.forward(ps, x, (RELU,), "bf16_mirror")
    fwe = om.forward(ps, x, (RELU,), "bf16")
    W16 = om.rne_bf16(ps[0])
    u = x @ W16.T + ps[1]
    assert np.array_equal(fwm["X"][1], om.rne_bf16(np.maximum(u, 0)))
    assert np.allclose(fwe["X"][1], np.maximum(u, 0), rtol=0, atol=1e-15)
    assert np.array_equal(fwm["z"], om.rne_bf16(fwm["X"][1] @ om.rne_bf16(ps[2]).T + ps[3]))


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by a pin above.
# --------------------------------------------------------------------------
def test_planted_mistakes_are_caught(monkeypatch):
    # (1) backward without the ReLU mask -> finite differences disagree
    orig_backward = om.backward

    def no_mask(fw, dz, acts, mode="fp64"):
        return orig_backward(fw, dz, tuple(NONE for _ in acts), mode)

    monkeypatch.setattr(om, "backward", no_mask)
    with pytest.raises(AssertionError):
        test_backward_central_finite_differences((RELU, RELU))
    monkeypatch.setattr(om, "backward", orig_backward)

    # (2) CE gradient without the 1/B scale -> zero-logit closed form fails
    orig_ce = om.softmax_ce
    monkeypatch.setattr(om, "softmax_ce", lambda z, y: (orig_ce(z, y)[0], orig_ce(z, y)[1] * len(y)))
    with pytest.raises(AssertionError):
        test_ce_zero_logits_closed_form(10)
    monkeypatch.setattr(om, "softmax_ce", orig_ce)

    # (3) eps inside the square root -> AdamW first-step closed form fails
    def adamw_eps_inside(p, g, m, v, t, lr, b1, b2, eps, wd):
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        return p - lr * (m / (1 - b1 ** t) / np.sqrt(v / (1 - b2 ** t) + eps) + wd * p), m, v

    orig_adamw = om.adamw
    monkeypatch.setattr(om, "adamw", adamw_eps_inside)
    with pytest.raises(AssertionError):
        test_adamw_first_step_closed_form()
    monkeypatch.setattr(om, "adamw", orig_adamw)

    # (4) transposed weight gradient (X^T dY instead of dY^T X) on a
    #     non-square layer -> shape / autograd pin fails
    def backward_transposed(fw, dz, acts, mode="fp64"):
        g = orig_backward(fw, dz, acts, mode)
        return [gi.T if gi.ndim == 2 else gi for gi in g]

    monkeypatch.setattr(om, "backward", backward_transposed)
    with pytest.raises((AssertionError, ValueError)):
        test_backward_matches_torch_autograd()
    monkeypatch.setattr(om, "backward", orig_backward)

    # (5) Adam with the decay decoupled (an AdamW step) -> the L2 pins fail
    orig_adam = om.adam_l2
    monkeypatch.setattr(om, "adam_l2", om.adamw)
    with pytest.raises(AssertionError):
        test_adam_l2_first_step_closed_form()
    with pytest.raises(AssertionError):
        test_adam_l2_matches_torch_optim_adam_100_steps()
    monkeypatch.setattr(om, "adam_l2", orig_adam)

    # (6) SGD with dampening (buf = mu buf + (1 - mu) g) -> closed form fails
    orig_sgd = om.sgd

    def sgd_damped(p, g, buf, lr, mu, wd):
        g = g + wd * p
        buf = mu * buf + (1 - mu) * g
        return p - lr * buf, buf

    monkeypatch.setattr(om, "sgd", sgd_damped)
    with pytest.raises(AssertionError):
        test_sgd_constant_gradient_closed_form()
    monkeypatch.setattr(om, "sgd", orig_sgd)

    # (7) clipping by the squared norm, or per tensor -> closed form / torch fail
    orig_clip = om.clip_coef
    monkeypatch.setattr(om, "clip_coef", lambda g, c: orig_clip(g, c) ** 2 if c else 1.0)
    with pytest.raises(AssertionError):
        test_clip_coef_closed_form()
    monkeypatch.setattr(om, "clip_coef", lambda g, c: min(orig_clip([x], c) for x in g))
    with pytest.raises(AssertionError):
        test_clip_matches_torch_clip_grad_norm()
    monkeypatch.setattr(om, "clip_coef", orig_clip)

    # (9) a multi-step driver whose step counter does not advance, or whose
    #     moments restart every step -> the torch training-loop pin fails
    orig_step = om.train_step
    monkeypatch.setattr(om, "train_step", lambda p, m, v, t, *a, **k: orig_step(p, m, v, 1, *a, **k))
    with pytest.raises(AssertionError):
        test_run_steps_matches_torch_training_loop("adamw")
    monkeypatch.setattr(om, "train_step",
                        lambda p, m, v, t, *a, **k: orig_step(p, [0 * q for q in m], [0 * q for q in v], t, *a, **k))
    with pytest.raises(AssertionError):
        test_run_steps_matches_torch_training_loop("adamw")
    monkeypatch.setattr(om, "train_step", orig_step)

    # (8) MSE gradient scaled by 1/B instead of 1/(B C), or missing the 2
    orig_mse = om.mse
    monkeypatch.setattr(om, "mse", lambda z, t: (orig_mse(z, t)[0], orig_mse(z, t)[1] * z.shape[1]))
    with pytest.raises(AssertionError):
        test_mse_bruteforce_and_torch()
    monkeypatch.setattr(om, "mse", lambda z, t: (orig_mse(z, t)[0], orig_mse(z, t)[1] / 2))
    with pytest.raises(AssertionError):
        test_mse_closed_forms()
    monkeypatch.setattr(om, "mse", orig_mse)


# --------------------------------------------------------------------------
# Frozen worked examples (the oracle's own output; a regression guard)
# --------------------------------------------------------------------------
def test_oracle_matches_frozen_worked_examples():
    """tests/golden/tiny_step.json holds whole steps (CE / MSE; AdamW, Adam,
    SGD; clipping off and on) computed by this oracle when it was pinned; a
    change of its arithmetic must show here and be justified."""
    import json
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    try:
        import make_golden
    finally:
        sys.path.remove(here)
    with open(os.path.join(here, "tiny_step.json")) as f:
        frozen = json.load(f)
    now = make_golden.compute()
    assert frozen["dims"] == now["dims"] and frozen["batch"] == now["batch"]
    for name, case in frozen["cases"].items():
        got = now["cases"][name]
        assert abs(got["loss"] - case["loss"]) <= 1e-14 * abs(case["loss"]), name
        assert abs(got["clip"] - case["clip"]) <= 1e-14, name
        for a, b in zip(got["grads"] + got["params"], case["grads"] + case["params"]):
            np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-16)
