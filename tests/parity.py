"""Shared helpers for GPU-vs-oracle parity tests.

Tolerances (each derived from the arithmetic it bounds):

Single GEMM-shaped results (op tests):
    |c - c*| <= 8 sqrt(K) 2^-24 sum_k |a_k b_k|    (fp32 accumulation; 8x the
    rms growth of recursive fp32 summation), plus half a bf16 ulp of |c*|
    (2^-8 |c*|) when the output is stored as bf16.

fp32 step (no TF32), one step from a shared state:
    loss: |L - L*| <= 1e-4 |L*|.
    gradients: |g - g*| <= 2^-17 kappa, kappa = sum of |products| that make g
        (|dY|^T |X| for a weight, sum |dY| for a bias): 128 fp32 ulps of the
        absolute sum, covering accumulation over up to 4096 terms and the
        propagation of the same error through dY.
    parameters: |p - p*| <= 1e-4 max(|p*|, lr) + lr * S, where
        S = min(2, eps dg / (max(|g*| - dg, 0) + eps)^2) is the first-order
        change of AdamW's first-step direction g / (|g| + eps) under a gradient
        error dg (the bound above).  S only matters where |g*| is near eps:
        there the direction itself is decided by fp32 rounding.

Trajectories and every bf16 comparison ("oracle ensemble"):
    The bf16 mirror computation and multi-step AdamW are ill-conditioned:
    rounding decisions and ReLU masks that sit within fp32 accumulation noise
    of a threshold flip, and AdamW's sign-like steps turn a flipped gradient
    sign into a 2 lr change.  The oracle itself, re-run with every product
    perturbed by (1 + eta r), r ~ U(-1, 1), eta = sqrt(K) 2^-24 (the
    probabilistic size of fp32 accumulation error over K terms), moves by the
    same amount.  The GPU must be statistically indistinguishable from that
    ensemble: per tensor, rms and fraction of elements beyond the stated
    tolerance no larger than 3x the largest perturbed run (plus small floors);
    per step, |L - L*| <= max(stated |L*|, 3 max_j |L_j - L*|).  The stated
    element-wise tolerances (fp32: 1e-4; bf16: loss 2e-2 against the oracle's
    exact mode, parameters 3e-2 of the tensor's largest oracle update) are
    computed and reported alongside.
"""
from __future__ import annotations

import contextlib
import math
from typing import Dict, List, Sequence

import numpy as np
import torch

import synth
from oracle import mlp_oracle as om

ENSEMBLE_RUNS = 3
ENSEMBLE_FACTOR = 3.0


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def flat(params: Sequence[np.ndarray]) -> np.ndarray:
    return np.concatenate([np.asarray(p, np.float64).ravel() for p in params])


# ---------------------------------------------------------------------------
# GEMM-level tolerance
# ---------------------------------------------------------------------------
def gemm_tol(absum: np.ndarray, K: int, ref: np.ndarray, bf16_out: bool) -> np.ndarray:
    t = 8.0 * math.sqrt(max(K, 1)) * 2.0 ** -24 * absum
    if bf16_out:
        t = t + 2.0 ** -8 * np.abs(ref)
    return t + 1e-30


def assert_close_gemm(got: np.ndarray, ref: np.ndarray, absum: np.ndarray, K: int, bf16_out: bool, what="",
                      extra=None):
    """extra: an additional absolute tolerance (e.g. the fp32 evaluation
    error of an activation derivative applied to the GEMM result)."""
    tol = gemm_tol(absum, K, ref, bf16_out)
    if extra is not None:
        tol = tol + extra
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}")


# ---------------------------------------------------------------------------
# Oracle runs
# ---------------------------------------------------------------------------
def oracle_mode(w: synth.Workload, exact: bool = False) -> str:
    if w.dtype == synth.F32:
        return "fp64"
    return "bf16" if exact else "bf16_mirror"


def batches(w: synth.Workload, n: int, batch=None):
    return [synth.make_batch(w, s, batch) for s in range(n)]


def hyper32(w: synth.Workload):
    """The optimiser settings as the C ABI receives them (fp32)."""
    return tuple(float(np.float32(a)) for a in (w.lr, w.beta1, w.beta2, w.eps, w.wd))


@contextlib.contextmanager
def perturbed_products(seed: int):
    """Inside the block every product the oracle forms (linear, weight_grad,
    input_grad, bias_grad) is multiplied elementwise by (1 + eta r),
    r ~ U(-1, 1), eta = sqrt(K) 2^-24 for a reduction over K terms."""
    rng = np.random.default_rng(seed)
    orig = (om.linear, om.weight_grad, om.input_grad, om.bias_grad, om.softmax_ce, om.update, om.clip_coef, om.mse)

    def rel(a, e):
        return a * (1.0 + e * rng.uniform(-1.0, 1.0, np.shape(a)))

    def ce(z, y):
        # fp32 exp / log / division: a few ulps on each output
        lr_, dz_ = orig[4](z, y)
        return rel(lr_, 2.0 ** -22), rel(dz_, 2.0 ** -22)

    def update(optim, p, g, m, v, t, *hyper):
        # fp32 arithmetic and fp32 storage of p, m, v after every step
        p2, m2, v2 = orig[5](optim, p, g, m, v, t, *hyper)
        return rel(p2, 2.0 ** -23), rel(m2, 2.0 ** -22), rel(v2, 2.0 ** -22)

    def clip_coef(grads, max_norm):
        # an fp32 sum of squares over every gradient element
        c = orig[6](grads, max_norm)
        return c if c == 1.0 else rel(c, 2.0 ** -20)

    def mse(z, t):
        # fp32 difference, square and row sum; dz scaled in fp32
        r_, dz_ = orig[7](z, t)
        return rel(r_, 2.0 ** -22), rel(dz_, 2.0 ** -22)

    om.softmax_ce = ce
    om.update = update
    om.clip_coef = clip_coef
    om.mse = mse

    def noisy(a, absum, K):
        # fp32 accumulation error scales with the sum of |terms|, not with
        # the (possibly cancelled) result
        eta = math.sqrt(max(K, 1)) * 2.0 ** -24
        return a + eta * absum * rng.uniform(-1.0, 1.0, np.shape(a))

    om.linear = lambda X, W, b: noisy(orig[0](X, W, b), np.abs(X) @ np.abs(W).T + np.abs(b), X.shape[1])
    om.weight_grad = lambda dY, X: noisy(orig[1](dY, X), np.abs(dY).T @ np.abs(X), dY.shape[0])
    om.input_grad = lambda dY, W: noisy(orig[2](dY, W), np.abs(dY) @ np.abs(W), dY.shape[1])
    om.bias_grad = lambda dY: noisy(orig[3](dY), np.abs(dY).sum(axis=0), dY.shape[0])
    try:
        yield
    finally:
        (om.linear, om.weight_grad, om.input_grad, om.bias_grad, om.softmax_ce, om.update, om.clip_coef,
         om.mse) = orig


def oracle_run(w: synth.Workload, params0, bl, mode: str, perturb_seed: int = 0, optim: str = "adamw",
               max_norm: float = 0.0, loss: str = "ce"):
    """(losses, params, m, v, first-step grads) of len(bl) steps from params0.
    bl holds (x, labels) pairs, or (x, fp32 targets) for loss="mse"."""
    hyper = hyper32(w)
    xs = [(to64(x), to64(y) if loss == "mse" else y.numpy().astype(np.int64)) for x, y in bl]
    p0 = [to64(p) for p in params0]
    kw = dict(mode=mode, optim=optim, max_norm=float(np.float32(max_norm)), loss=loss)
    if perturb_seed:
        with perturbed_products(perturb_seed):
            return om.run_steps(p0, w.acts, xs, hyper, **kw)
    return om.run_steps(p0, w.acts, xs, hyper, **kw)


def oracle_abs_sums(w: synth.Workload, params0, x, y, mode: str, loss: str = "ce") -> List[np.ndarray]:
    """kappa for every first-step gradient element (a running error bound).

    Forward on absolute values, F_0 = |x|, F_l = (F_{l-1} |W_l|^T + |b_l|) *
    |act'(u_l)|, bounds every product behind the activations (an error in
    X_l is a multiple of u F_l, however much X_l itself cancels).  The
    softmax turns a logit error of u max_k F_L[i, k] into at most
    2 p_ij u max_k F_L[i, k] in p_ij.  Backward on absolute values,
    A_L = |dz| + 2 p max_k F_L / B, A_{l-1} = (A_l |W_l|) * |act'|.  Then
    kappa_W = A_l^T F_{l-1} and kappa_b = sum_rows A_l bound every product
    that feeds the gradient, including those that cancel inside dY or X.
    For MSE, dz = 2 (z - t) / (B C) moves by 2 u F_L / (B C) under the same
    logit error, so A_L = |dz| + 2 F_L / (B C)."""
    p0 = [to64(p) for p in params0]
    fw = om.forward(p0, to64(x), w.acts, mode)
    if loss == "mse":
        _, dz = om.mse(fw["z"], to64(y))
    else:
        _, dz = om.softmax_ce(fw["z"], y.numpy().astype(np.int64))
    L = w.n_layers

    def dact(l):   # |act'| of hidden layer l's pre-activation
        act = w.acts[l]
        if act == om.ACT_RELU:
            return (fw["X"][l + 1] > 0).astype(np.float64)
        if act == om.ACT_GELU_TANH:
            return np.abs(om.gelu_tanh_grad(fw["u"][l]))
        return np.ones_like(fw["X"][l + 1])

    F = [np.abs(fw["X"][0])]
    for l in range(L):
        Fl = F[-1] @ np.abs(fw["W"][l]).T + np.abs(p0[2 * l + 1])
        F.append(Fl * dact(l) if l < L - 1 else Fl)
    B = dz.shape[0]
    out = [None] * (2 * L)
    if loss == "mse":
        A = np.abs(dz) + 2.0 * F[L] / dz.size
    else:
        pz = dz * B                                   # softmax probabilities p
        pz[np.arange(B), y.numpy().astype(np.int64)] += 1.0
        A = np.abs(dz) + 2.0 * pz * F[L].max(axis=1, keepdims=True) / B
    for l in range(L - 1, -1, -1):
        X = F[l]
        out[2 * l] = A.T @ X
        out[2 * l + 1] = A.sum(axis=0)
        if l > 0:
            act = w.acts[l - 1]
            if act == om.ACT_RELU:
                d = (fw["X"][l] > 0).astype(np.float64)
            elif act == om.ACT_GELU_TANH:
                d = np.abs(om.gelu_tanh_grad(fw["u"][l - 1]))
            else:
                d = np.ones_like(fw["X"][l])
            A = (A @ np.abs(fw["W"][l])) * d
    return out


# ---------------------------------------------------------------------------
# Criteria
# ---------------------------------------------------------------------------
def fp32_grad_tol(kappa: np.ndarray) -> np.ndarray:
    return 2.0 ** -17 * kappa + 1e-30


def fp32_first_step_param_tol(p_ref, g_ref, dg, lr, eps):
    s = np.minimum(2.0, eps * dg / (np.maximum(np.abs(g_ref) - dg, 0.0) + eps) ** 2)
    return 1e-4 * np.maximum(np.abs(p_ref), lr) + lr * s


def ensemble_check(what: str, gpu: Sequence[np.ndarray], ref: Sequence[np.ndarray],
                   perts: Sequence[Sequence[np.ndarray]], scale: Sequence[float], stated: float) -> Dict:
    """Per tensor i: deviations |gpu - ref| against the ensemble's |pert_j - ref|.

    scale[i] is the tensor's reference magnitude (the largest oracle update
    for parameters, max |g*| for gradients); `stated` is the stated
    element-wise tolerance as a fraction of it."""
    report, bad = [], []
    for i, (g, r, sc) in enumerate(zip(gpu, ref, scale)):
        sc = np.maximum(np.asarray(sc, np.float64), 1e-30)   # scalar or per element
        nd = np.abs(np.asarray(g, np.float64) - r) / sc
        rms_g = float(np.sqrt(np.mean(nd ** 2)))
        frac_g = float(np.mean(nd > stated))
        max_g = float(nd.max())
        rms_p = frac_p = max_p = 0.0
        for pr in perts:
            d = np.abs(pr[i] - r) / sc
            rms_p = max(rms_p, float(np.sqrt(np.mean(d ** 2))))
            frac_p = max(frac_p, float(np.mean(d > stated)))
            max_p = max(max_p, float(d.max()))
        ok = (rms_g <= ENSEMBLE_FACTOR * rms_p + 0.1 * stated) and \
             (frac_g <= ENSEMBLE_FACTOR * frac_p + 1e-3)
        row = dict(tensor=i, rms=rms_g, rms_ens=rms_p, frac=frac_g, frac_ens=frac_p, max=max_g, max_ens=max_p,
                   stated_ok=max_g <= stated, ok=ok)
        report.append(row)
        if not ok:
            bad.append(row)
    if bad:
        raise AssertionError(f"{what}: outside the oracle ensemble: {bad}")
    return {"what": what, "tensors": report}


def loss_ensemble_check(what, gpu_losses, ref_losses, pert_losses, stated):
    gl, rl = np.asarray(gpu_losses, np.float64), np.asarray(ref_losses, np.float64)
    spread = np.zeros_like(rl)
    for pl in pert_losses:
        spread = np.maximum(spread, np.abs(np.asarray(pl) - rl))
    tol = np.maximum(stated * np.abs(rl), ENSEMBLE_FACTOR * spread)
    dev = np.abs(gl - rl)
    if np.any(dev > tol):
        i = int(np.argmax(dev / tol))
        raise AssertionError(f"{what}: step {i} loss {gl[i]} vs oracle {rl[i]} (ensemble spread {spread[i]}, "
                             f"tol {tol[i]})")
    return {"what": what, "max_rel": float(np.max(dev / np.abs(rl))), "stated_ok": bool(np.all(dev <= stated * np.abs(rl)))}
