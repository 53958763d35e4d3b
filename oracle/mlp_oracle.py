"""Plain, slow, fp64 CPU oracle of one supervised MLP training step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA path
and must never be used as a fallback for it.

What it computes, with the passage each step follows:

* Linear layer y = x W^T + b, W stored [out, in] (MuNet, pypi "munet-nn",
  section "Python training": `mu.nn.Linear(in, out)`; noeira.ai "Neural
  networks", section "A complete example": `LinearReLU[784, 256]`).
* Activation after every hidden Linear, none after the output Linear
  (noeira "A complete example": two LinearReLU layers then a plain Linear).
  ReLU is max(0, u); GELU is the tanh form 0.5 u (1 + tanh(sqrt(2/pi)(u +
  0.044715 u^3))) (textbook definition, Hendrycks & Gimpel; the pages do not
  define it).
* Softmax cross-entropy with integer labels, mean over the batch (Orthon,
  devpost "Orthon", sections "Core capabilities" and "Selected Orthon vs.
  PyTorch results"; integer labels are the one-hot rows of noeira "A complete
  example").
* Mean squared error against real targets, mean over all elements (MuNet
  "Python training": mse_loss in the example step; "Training swarm").
* Backward as the composition of per-layer vector-Jacobian products, no tape
  (noeira "The design in one page": "Forward and backward are explicit").
* AdamW with decoupled weight decay and moments m, v kept per parameter,
  zero before the first step (MuNet "What runs today": AdamW; noeira "The
  design in one page": a Param is four tensors, moments allocated lazily).
* Adam with L2 in the gradient, SGD with momentum, and global gradient-norm
  clipping (MuNet "What runs today"; noeira "What is in it"; Orthon "Core
  capabilities"), each in its PyTorch form.
* Mixed precision: matmul inputs rounded to nearest (even), fp32-or-better
  accumulation, fp32 master weights (MuNet "Configuration", precision="mixed";
  Orthon "Core capabilities", Mixed precision).  Here the low-precision type
  is bfloat16.

Readings of points the pages leave open (each stated here in full):
ReLU'(0) = 0 and the ReLU mask is taken from the stored activation h > 0;
AdamW follows the Loshchilov-Hutter / PyTorch form (eps added to sqrt(v_hat)
after bias correction, decay applied to the pre-step parameter, t starts at 1,
decay on every parameter including biases); argmax returns the lowest index
among equal maxima; a label outside [0, C) is an error.

Precision modes
  "fp64"      everything in float64 (used for the fp32 workloads, whose inputs
              are fp32 values).
  "bf16"      "exact" bf16 reading: only x and the bf16 weight copy
              W16 = rne_bf16(P) are rounded; all else float64.
  "bf16_mirror" rounds to bf16 at the points where a bf16 implementation
              stores tensors: W16, hidden activations h (and GELU
              pre-activations u), logits z, dz and every dY; bias, gradients,
              master params and moments stay unrounded.  Accumulation is
              float64 in between.

All functions take and return float64 numpy arrays unless stated.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

ACT_NONE, ACT_RELU, ACT_GELU_TANH = 0, 1, 2
_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_GELU_C = 0.044715


# ---------------------------------------------------------------------------
# bfloat16 round-to-nearest-even (definition: keep 8 significant bits; the
# smallest quantum is 2^-133, bf16's subnormal spacing; ties go to the even
# neighbour; beyond the largest bf16 value, infinity).  Mixed precision per
# MuNet "Configuration" (precision="mixed": inputs rounded to nearest), with
# bfloat16 in place of fp16.
# ---------------------------------------------------------------------------
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def rne_bf16(a: np.ndarray) -> np.ndarray:
    """Round every value to the nearest bfloat16, ties to even.

    From 2^-126 up (bf16's normal range) the quantum is 2^(e-8) for a value
    in [2^(e-1), 2^e): of the fp64 significand's 52 stored bits the top 7
    stay, and the 45 below are rounded away on the bit pattern -- add
    2^44 - 1 plus the lowest kept bit, then clear them (half rounds up only
    when the kept part is odd; a carry moves to the next binade, as it
    should).  Below 2^-126 the quantum is the fixed 2^-133: rint(a / q) q.
    Zeros, infinities and NaNs pass through."""
    a = np.asarray(a, dtype=np.float64)
    out = a.copy()
    fin = np.isfinite(a)
    mag = np.abs(a)
    normal = fin & (mag >= 2.0 ** -126)
    bits = a[normal].view(np.int64)
    lsb = (bits >> 45) & 1
    bits = (bits + ((1 << 44) - 1) + lsb) & ~np.int64((1 << 45) - 1)
    out[normal] = bits.view(np.float64)
    tiny = fin & (mag < 2.0 ** -126) & (a != 0)
    q = 2.0 ** -133
    out[tiny] = np.rint(a[tiny] / q) * q
    over = np.abs(out) > _BF16_MAX
    out[over] = np.copysign(np.inf, out[over])
    return out


# ---------------------------------------------------------------------------
# Activations and their derivatives.
# ---------------------------------------------------------------------------
def act_forward(u: np.ndarray, act: int) -> np.ndarray:
    if act == ACT_NONE:
        return u.copy()
    if act == ACT_RELU:
        return np.maximum(u, 0.0)
    if act == ACT_GELU_TANH:
        t = np.tanh(_SQRT_2_OVER_PI * (u + _GELU_C * u ** 3))
        return 0.5 * u * (1.0 + t)
    raise ValueError(f"unknown activation {act}")


def gelu_tanh_grad(u: np.ndarray) -> np.ndarray:
    """d/du of the tanh-form GELU (product and chain rule on the definition)."""
    inner = _SQRT_2_OVER_PI * (u + _GELU_C * u ** 3)
    t = np.tanh(inner)
    dinner = _SQRT_2_OVER_PI * (1.0 + 3.0 * _GELU_C * u ** 2)
    return 0.5 * (1.0 + t) + 0.5 * u * (1.0 - t * t) * dinner


# ---------------------------------------------------------------------------
# Steps of the path.
# ---------------------------------------------------------------------------
def linear(X: np.ndarray, W: np.ndarray, b: np.ndarray) -> np.ndarray:
    """u = X W^T + b  (W is [out, in])."""
    return X @ W.T + b[None, :]


def weight_grad(dY: np.ndarray, X: np.ndarray) -> np.ndarray:
    """dW = dY^T X: the VJP of u = X W^T + b with respect to W."""
    return dY.T @ X


def input_grad(dY: np.ndarray, W: np.ndarray) -> np.ndarray:
    """dX = dY W: the VJP of u = X W^T + b with respect to X."""
    return dY @ W


def bias_grad(dY: np.ndarray) -> np.ndarray:
    """db = sum over rows of dY: the VJP of u = X W^T + b with respect to b."""
    return dY.sum(axis=0)


def softmax_ce(z: np.ndarray, y: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-row loss l_i = logsumexp(z_i) - z_i[y_i] and dz = (softmax(z) -
    onehot(y)) / B, the gradient of the batch-mean loss."""
    B, C = z.shape
    y = np.asarray(y)
    if B and (y.min() < 0 or y.max() >= C):
        raise ValueError("label out of range")
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    s = e.sum(axis=1, keepdims=True)
    rows = np.arange(B)
    loss_rows = (m[:, 0] + np.log(s[:, 0])) - z[rows, y]
    p = e / s
    dz = p.copy()
    dz[rows, y] -= 1.0
    return loss_rows, dz / B


def mse(z: np.ndarray, t: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Mean squared error against real targets t [B, C] (MuNet "Python
    training": the example step calls mse_loss(model(x), target); "Training
    swarm": the current loss is MSE).  Reading: the PyTorch mse_loss default,
    the mean over all B C elements.  Returns the per-row sums of squares
    r_i = sum_j (z_ij - t_ij)^2 (loss = sum_i r_i / (B C)) and dz = 2 (z - t)
    / (B C), the gradient of that mean."""
    t = np.asarray(t, np.float64)
    if t.shape != z.shape:
        raise ValueError("targets must have the shape of the outputs")
    d = z - t
    return (d * d).sum(axis=1), 2.0 * d / max(d.size, 1)


def argmax_rows(z: np.ndarray) -> np.ndarray:
    """Index of the row maximum, lowest index among equal maxima."""
    return np.argmax(z, axis=1).astype(np.int32)   # numpy returns the first


def adamw(p, g, m, v, t: int, lr, beta1, beta2, eps, wd):
    """One AdamW update at step t (t >= 1); returns new (p, m, v).

    m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
    p <- p - lr (m_hat / (sqrt(v_hat) + eps) + wd p),  m_hat = m/(1-b1^t),
    v_hat = v/(1-b2^t), with p on the right the pre-step value."""
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p - lr * (m_hat / (np.sqrt(v_hat) + eps) + wd * p)
    return p, m, v


def adam_l2(p, g, m, v, t: int, lr, beta1, beta2, eps, wd):
    """One Adam update with L2 regularisation folded into the gradient
    (noeira "Neural networks", section "What is in it", optimizers: Adam next
    to AdamW; Orthon "Core capabilities", training stack: SGD and Adam).
    Reading (the pages give no formula): the PyTorch Adam form, decay coupled
    into the gradient, g' = g + wd p, then the AdamW moments and step without
    the decoupled term, p <- p - lr m_hat / (sqrt(v_hat) + eps).  Returns new
    (p, m, v)."""
    g = g + wd * p
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    return p - lr * m_hat / (np.sqrt(v_hat) + eps), m, v


def sgd(p, g, buf, lr, momentum, wd):
    """One SGD update (MuNet "What runs today" lists SGD and its "Python
    training" example steps `mu.optim.SGD(params, lr=0.03)`; noeira "What is in
    it"; Orthon "Core capabilities").  Reading: the PyTorch SGD form with
    heavy-ball momentum, no dampening and coupled L2: g' = g + wd p,
    buf <- momentum buf + g' (buf zero before the first step), p <- p - lr buf.
    momentum = 0 and wd = 0 give the plain p <- p - lr g of the example.
    Returns (p, buf)."""
    g = g + wd * p
    buf = momentum * buf + g
    return p - lr * buf, buf


def clip_coef(grads, max_norm) -> float:
    """Global gradient-norm clipping (MuNet "What runs today" and noeira "What
    is in it" list gradient clipping; neither gives the rule).  Reading: the
    PyTorch clip_grad_norm_ form, the factor min(1, max_norm / (||G||_2 +
    1e-6)) applied to every gradient, ||G|| the 2-norm over every element of
    every gradient; 1 when max_norm <= 0 (off)."""
    if not max_norm or max_norm <= 0:
        return 1.0
    total = math.sqrt(sum(float(np.sum(np.asarray(g, np.float64) ** 2)) for g in grads))
    return min(1.0, float(max_norm) / (total + 1e-6))


OPTIMIZERS = ("adamw", "adam", "sgd")


def update(optim: str, p, g, m, v, t: int, lr, beta1, beta2, eps, wd):
    """The parameter update of the step: AdamW (default), Adam with L2, or
    SGD whose momentum coefficient is beta1 (its buffer kept in m; v
    unchanged)."""
    if optim == "adamw":
        return adamw(p, g, m, v, t, lr, beta1, beta2, eps, wd)
    if optim == "adam":
        return adam_l2(p, g, m, v, t, lr, beta1, beta2, eps, wd)
    if optim == "sgd":
        pn, buf = sgd(p, g, m, lr, beta1, wd)
        return pn, buf, v
    raise ValueError(f"unknown optimizer {optim}")


# ---------------------------------------------------------------------------
# Whole network.
# ---------------------------------------------------------------------------
def _round(a, on: bool):
    return rne_bf16(a) if on else a


def forward(params: Sequence[np.ndarray], x: np.ndarray, acts: Sequence[int],
            mode: str = "fp64") -> Dict[str, list]:
    """Forward pass.  params = [W1, b1, ..., WL, bL] (float64 master values).

    Returns dict with the per-layer inputs X_l, pre-activations u_l (as stored:
    rounded in mirror mode), and the logits z."""
    L = len(params) // 2
    lowp = mode in ("bf16", "bf16_mirror")
    mirror = mode == "bf16_mirror"
    X = _round(np.asarray(x, np.float64), lowp)
    Xs, us, Ws = [], [], []
    for l in range(L):
        W = _round(params[2 * l], lowp)
        b = params[2 * l + 1]
        u = linear(X, W, b)
        Xs.append(X)
        Ws.append(W)
        if l < L - 1:
            act = acts[l]
            h = _round(act_forward(u, act), mirror)
            us.append(_round(u, mirror))
            X = h
        else:
            us.append(_round(u, mirror))
    return {"X": Xs, "u": us, "W": Ws, "z": us[-1]}


def backward(fw: Dict[str, list], dz: np.ndarray, acts: Sequence[int],
             mode: str = "fp64") -> List[np.ndarray]:
    """Gradients [dW1, db1, ..., dWL, dbL] by composing the layer VJPs:
    dW_l = dY_l^T X_l, db_l = sum_i dY_l[i], dY_{l-1} = (dY_l W_l) * act'."""
    mirror = mode == "bf16_mirror"
    L = len(fw["W"])
    grads: List[Optional[np.ndarray]] = [None] * (2 * L)
    dY = _round(dz, mirror)
    for l in range(L - 1, -1, -1):
        X = fw["X"][l]
        grads[2 * l] = weight_grad(dY, X)
        grads[2 * l + 1] = bias_grad(dY)
        if l > 0:
            dX = input_grad(dY, fw["W"][l])
            act = acts[l - 1]
            if act == ACT_RELU:
                d = dX * (fw["X"][l] > 0)            # mask from the stored h
            elif act == ACT_GELU_TANH:
                d = dX * gelu_tanh_grad(fw["u"][l - 1])
            else:
                d = dX
            dY = _round(d, mirror)
    return grads


def train_step(params: Sequence[np.ndarray], m: Sequence[np.ndarray],
               v: Sequence[np.ndarray], t: int, x: np.ndarray, y: np.ndarray,
               acts: Sequence[int], lr, beta1, beta2, eps, wd,
               mode: str = "fp64", optim: str = "adamw", max_norm: float = 0.0, loss: str = "ce"):
    """One step: forward, the loss (softmax CE with integer labels y, batch
    mean; or MSE with real targets y [B, C], element mean), backward, the
    update at step t (AdamW by default) of the gradient scaled by the
    clipping factor.

    Returns (loss, new_params, new_m, new_v, grads, extras); grads are the
    unclipped gradients."""
    fw = forward(params, x, acts, mode)
    if loss == "ce":
        loss_rows, dz = softmax_ce(fw["z"], y)
        loss = float(loss_rows.mean())
    elif loss == "mse":
        loss_rows, dz = mse(fw["z"], y)
        loss = float(loss_rows.sum() / max(dz.size, 1))
    else:
        raise ValueError(f"unknown loss {loss}")
    grads = backward(fw, dz, acts, mode)
    c = clip_coef(grads, max_norm)
    newp, newm, newv = [], [], []
    for p_, g_, m_, v_ in zip(params, grads, m, v):
        a, b, c_ = update(optim, p_, g_ * c, m_, v_, t, lr, beta1, beta2, eps, wd)
        newp.append(a)
        newm.append(b)
        newv.append(c_)
    return loss, newp, newm, newv, grads, {"fw": fw, "loss_rows": loss_rows, "dz": dz, "clip": c}


def run_steps(params, acts, batches, hyper, mode="fp64", t0: int = 0, optim: str = "adamw",
              max_norm: float = 0.0, loss: str = "ce"):
    """Run len(batches) consecutive steps from zero moments.  batches yields
    (x, y) pairs (y: labels, or targets for loss="mse").  hyper = (lr, beta1,
    beta2, eps, wd).  Returns (losses, params, m, v, first_step_grads)."""
    p = [np.asarray(a, np.float64) for a in params]
    m = [np.zeros_like(a) for a in p]
    v = [np.zeros_like(a) for a in p]
    losses, g1 = [], None
    for i, (x, y) in enumerate(batches):
        L, p, m, v, g, _ = train_step(p, m, v, t0 + i + 1, x, y, acts, *hyper, mode=mode, optim=optim,
                                      max_norm=max_norm, loss=loss)
        losses.append(L)
        if g1 is None:
            g1 = g
    return losses, p, m, v, g1
