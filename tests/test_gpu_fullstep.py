"""Whole training steps at the full sizes of the three bf16 workloads, checked
layer by layer, element by element, against the oracle.

The step runs through mlp_trace_step: the same kernels, launch
configurations and buffers as mlp_train_step (the test checks that the
parameters and gradients it leaves are bitwise those of the graph step), with
every stored intermediate tensor copied aside.  Each kernel's output is then
compared with the oracle's definition applied to the GPU's own inputs of that
kernel (the stored activations, logits, dz and dY the step actually read):

  forward l : h_l = rne(act(X_l W16_l^T + b_l)), u_l = rne(X_l W16_l^T + b_l)
  logits    : z = rne(h W16_L^T + b_L)
  softmax-CE: loss rows, dz = rne((softmax(z) - onehot(y)) / B), the mean loss
  dgrad l   : dY_{l-1} = rne((dY_l W16_l) * act'(stored h_{l-1} or u_{l-1}))
  wgrad l   : G[W_l] = dY_l^T X_l, G[b_l] = sum_rows dY_l (fp32)
  update    : p, m, v after AdamW at step t from the step's G and the state
              before the step

with W16 = rne(P) (noeira.ai "Neural networks", "The design in one page":
explicit forward and VJPs; MuNet "Configuration", precision="mixed": inputs
rounded to nearest, fp32 accumulation).  Because every comparison starts from
the same stored inputs, each bound is that of one kernel's own arithmetic --
fp32 accumulation (8 sqrt(K) 2^-24 sum|a b|), half a bf16 ulp where the
result is stored in bf16, ulps of the AdamW arithmetic -- and it is asserted
for every element, with no element excused.  Taken together the checks show
that the composed step, at full batch and in the launch configuration the
benchmark times (persistent multi-wave GEMMs, the full-batch split-K policy,
ReLU masks as bits), computes the oracle's step up to those roundings.

The free-running oracle (its own roundings from the start) is compared on
the loss: within 2e-2 of the oracle's exact-rounding mode, as stated for the
bf16 workloads.  Trajectories over the workloads' configured step counts are
in test_gpu_trajectory.py.
"""
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
BF16_FULL = ["cifar_mlp_b8192", "lm_block_t16384", "deep_narrow_b65536"]
CHUNK = 2048    # rows per oracle block (the LM head's fp64 logits stay ~0.5 GB a block)
ACC = 8.0 * 2.0 ** -24   # fp32 accumulation: ACC sqrt(K) sum|a b|
HALF_ULP = 2.0 ** -8     # bf16 storage (8 significant bits, round to nearest)
# The tensor cores' fp32 accumulation is not IEEE round-to-nearest: each
# 16-deep tcgen05.mma adds its products into the accumulator after aligning
# them to the largest exponent in play and dropping the bits below a few
# guard bits, so small addends lose low bits in one direction and the loss
# grows with the number of MMA steps, not as sqrt(K).  The LM head's weight
# gradient shows it: a class's row sum is one -1/B label term plus ~16000
# terms some 2^-15 smaller, and its fp32 result sits up to ~2.5 fp32 ulps of
# the running sum per MMA step from the exact sum.  Bound used for fp32
# results of the tensor cores: TC_ULPS ulps (2^-23 relative) of the running
# sum's magnitude per 16-deep step, on top of the rounding bound above.
MMA_K = 16
TC_ULPS = 6.0
PREFIX_ROWS = 512        # the running sum is tracked at this granularity


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


class Trace:
    """The traced tensors of one step, by (kind, layer), as fp64 [rows, cols]
    (planes summed)."""

    def __init__(self, entries):
        self.t = {}
        self.launch = {}
        for e, ten in entries:
            v = ten[:, :, :e.cols]
            self.t[(e.kind, e.layer)] = v
            self.launch[(e.kind, e.layer)] = e.launch

    def rows(self, kind, layer, r0, r1) -> np.ndarray:
        v = self.t[(kind, layer)][:, r0:r1]
        a = _f64(v[0])
        for k in range(1, v.shape[0]):
            a = a + _f64(v[k])
        return a

    def full(self, kind, layer) -> np.ndarray:
        return self.rows(kind, layer, 0, self.t[(kind, layer)].shape[1])


def _bad(got, ref, tol, what):
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of bounds; worst at {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r} bound {tol[i]!r}")


def _act_grad(act, stored):
    """act' from the stored tensor the dgrad reads (h for ReLU: h > 0; u for
    GELU)."""
    if act == om.ACT_RELU:
        return (stored > 0).astype(np.float64)
    if act == om.ACT_GELU_TANH:
        return om.gelu_tanh_grad(stored)
    return np.ones_like(stored)


def check_step(w, tr: Trace, x, y, p_before, m_before, v_before, t, p_after, m_after, v_after, g, loss):
    """Every kernel of one traced step against the oracle on the GPU's inputs.
    p_* / m_* / v_* / g: [W1, b1, ...] fp64.  Returns a small report."""
    L, B = w.n_layers, w.batch
    W16 = [om.rne_bf16(p_before[2 * l]) for l in range(L)]
    bias = [p_before[2 * l + 1] for l in range(L)]
    x64 = _f64(x)
    y64 = y.numpy().astype(np.int64)
    rep = {}

    def X_rows(l, r0, r1):   # the input of layer l as the step stored it
        return x64[r0:r1] if l == 0 else tr.rows(nn.TRACE_H, l - 1, r0, r1)

    # ---- forward ----
    for l in range(L):
        K = w.dims[l]
        Wa = np.abs(W16[l])
        for r0 in range(0, B, CHUNK):
            r1 = min(B, r0 + CHUNK)
            Xr = X_rows(l, r0, r1)
            u = Xr @ W16[l].T + bias[l]
            absum = np.abs(Xr) @ Wa.T + np.abs(bias[l])
            acc = ACC * math.sqrt(K) * absum
            if l == L - 1:
                z = tr.rows(nn.TRACE_Z, l, r0, r1)
                _bad(z, u, acc + HALF_ULP * np.abs(u) + 1e-30, f"{w.name} logits rows {r0}:{r1}")
                continue
            act = w.acts[l]
            h = om.act_forward(u, act)
            # ReLU is 1-Lipschitz, GELU-tanh 1.13-Lipschitz
            _bad(tr.rows(nn.TRACE_H, l, r0, r1), h, 1.13 * acc + HALF_ULP * np.abs(h) + 1e-30,
                 f"{w.name} h_{l} rows {r0}:{r1}")
            if act == om.ACT_GELU_TANH:
                _bad(tr.rows(nn.TRACE_U, l, r0, r1), u, acc + HALF_ULP * np.abs(u) + 1e-30,
                     f"{w.name} u_{l} rows {r0}:{r1}")
    rep["forward"] = "ok"

    # ---- softmax-CE and the loss mean ----
    C = w.n_classes
    loss_rows = _f64(tr.t[(nn.TRACE_LOSS_ROWS, L - 1)][0, :, 0])
    ref_rows = np.empty(B)
    for r0 in range(0, B, CHUNK):
        r1 = min(B, r0 + CHUNK)
        z = tr.rows(nn.TRACE_Z, L - 1, r0, r1)
        lr_, dz_ = om.softmax_ce(z, y64[r0:r1])
        dz_ = dz_ * (r1 - r0) / B          # the batch mean is over all B rows
        ref_rows[r0:r1] = lr_
        # fp32 exp / sum / division on the stored logits, then bf16 storage
        _bad(tr.rows(nn.TRACE_DZ, L - 1, r0, r1), dz_, HALF_ULP * np.abs(dz_) + 1e-6 / B / C,
             f"{w.name} dz rows {r0}:{r1}")
    np.testing.assert_allclose(loss_rows, ref_rows, rtol=1e-5, atol=1e-5)
    assert abs(loss - ref_rows.mean()) <= 1e-5 * abs(ref_rows.mean()), (loss, ref_rows.mean())
    rep["loss"] = loss

    # ---- backward: wgrad (fp32 into G) and dgrad with the activation VJP ----
    for l in range(L - 1, -1, -1):
        N, K = w.dims[l + 1], w.dims[l]
        dW = np.zeros((N, K))
        dWa = np.zeros((N, K))
        db = np.zeros(N)
        dba = np.zeros(N)
        # bound on the running sum's magnitude over the batch: at the start of
        # every PREFIX_ROWS interval |S| plus the interval's absolute sum
        dWm = np.zeros((N, K))
        dbm = np.zeros(N)
        dY_kind = nn.TRACE_DZ if l == L - 1 else nn.TRACE_DY
        for r0 in range(0, B, CHUNK):
            r1 = min(B, r0 + CHUNK)
            dY = tr.rows(dY_kind, l, r0, r1)
            Xr = X_rows(l, r0, r1)
            for s0 in range(0, r1 - r0, PREFIX_ROWS):
                s1 = min(r1 - r0, s0 + PREFIX_ROWS)
                a = np.abs(dY[s0:s1]).T @ np.abs(Xr[s0:s1])
                np.maximum(dWm, np.abs(dW) + a, out=dWm)
                dW += dY[s0:s1].T @ Xr[s0:s1]
                dWa += a
                ab = np.abs(dY[s0:s1]).sum(0)
                np.maximum(dbm, np.abs(db) + ab, out=dbm)
                db += dY[s0:s1].sum(0)
                dba += ab
            if l > 0:
                act = w.acts[l - 1]
                stored = tr.rows(nn.TRACE_U if act == om.ACT_GELU_TANH else nn.TRACE_H, l - 1, r0, r1)
                fac = _act_grad(act, stored)
                dX = dY @ W16[l]
                absum = np.abs(dY) @ np.abs(W16[l])
                ref = dX * fac
                # GELU' is evaluated in fp32 on the stored u: 2^-21 |dY||W| on top
                extra = 2.0 ** -21 * absum if act == om.ACT_GELU_TANH else 0.0
                tol = ACC * math.sqrt(N) * absum * np.abs(fac) * 1.001 + extra + HALF_ULP * np.abs(ref) + 1e-30
                _bad(tr.rows(nn.TRACE_DY, l - 1, r0, r1), ref, tol, f"{w.name} dY_{l - 1} rows {r0}:{r1}")
        sb = ACC * math.sqrt(B)
        # split-K sums prefixes of parts of the batch: twice the bound covers them
        tc = math.ceil(B / MMA_K) * TC_ULPS * 2.0 ** -23 * 2.0
        # observed loss in fp32 ulps of the running sum per MMA step (reported)
        steps = math.ceil(B / MMA_K)
        ulps = np.abs(g[2 * l] - dW) / (steps * 2.0 ** -23 * dWm + 1e-300)
        rep.setdefault("wgrad_ulps_per_mma_step", {})[l] = float(ulps.max())
        _bad(g[2 * l], dW, sb * dWa + tc * dWm + 1e-30, f"{w.name} G[W_{l}]")
        _bad(g[2 * l + 1], db, sb * dba + tc * dbm + 1e-30, f"{w.name} G[b_{l}]")
    rep["backward"] = "ok"

    # ---- the AdamW update from this step's gradient ----
    f = lambda a: float(np.float32(a))
    lr, b1, b2, eps, wd = (f(a) for a in (w.lr, w.beta1, w.beta2, w.eps, w.wd))
    for i in range(2 * L):
        pr, mr, vr = om.adamw(p_before[i], g[i], m_before[i], v_before[i], t, lr, b1, b2, eps, wd)
        tol_m = 2.0 ** -21 * (b1 * np.abs(m_before[i]) + (1 - b1) * np.abs(g[i])) + 1e-30
        tol_v = 2.0 ** -21 * (b2 * v_before[i] + (1 - b2) * g[i] * g[i]) + 1e-38
        _bad(m_after[i], mr, tol_m, f"{w.name} m[{i}]")
        _bad(v_after[i], vr, tol_v, f"{w.name} v[{i}]")
        _bad(p_after[i], pr, 1e-5 * lr + 2.0 ** -23 * np.abs(pr), f"{w.name} p[{i}]")
    rep["update"] = "ok"
    return rep


def make_model(w, params=None):
    m = nn.Model(w.dims, w.acts, nn.ACT_RELU, w.dtype, seed=w.seed, batch=w.batch)
    if params is not None:
        m.write_flat(P.flat([p.numpy() for p in params]).astype(np.float32), nn.PLANE_P, 0)
    return m


def read_state(m):
    out = {}
    for name, pl in (("p", nn.PLANE_P), ("g", nn.PLANE_G), ("m", nn.PLANE_M), ("v", nn.PLANE_V)):
        a, step = m.read_flat(pl)
        out[name] = m.split(a.astype(np.float64))
        out["step"] = step
    return out


def traced_step_check(w, m, step_index):
    """Trace the next step of model m on batch `step_index` and check it."""
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    before = read_state(m)
    x, y = synth.make_batch(w, step_index)
    loss, ents = m.trace_step(x.to(DEV), y.to(DEV), **hyper)
    m.check_errors()
    after = read_state(m)
    assert after["step"] == before["step"] + 1
    tr = Trace(ents)
    rep = check_step(w, tr, x, y, before["p"], before["m"], before["v"], after["step"], after["p"], after["m"],
                     after["v"], after["g"], float(loss.item()))
    return rep, before, after, (x, y)


@pytest.mark.parametrize("name", BF16_FULL)
def test_full_size_first_step_layer_by_layer(name):
    w = W[name]
    params0 = synth.make_params(w)
    m = make_model(w, params0)
    rep, before, after, (x, y) = traced_step_check(w, m, 0)
    print(f"{name}: {rep}")
    m.close()
    # the traced step is the product step: same kernels, same results bit for bit
    m2 = make_model(w, params0)
    loss2 = m2.train_step(x.to(DEV), y.to(DEV), w.lr, w.beta1, w.beta2, w.eps, w.wd)
    m2.check_errors()
    st2 = read_state(m2)
    m2.close()
    assert float(loss2.item()) == rep["loss"]
    for k in ("p", "g", "m", "v"):
        assert np.array_equal(P.flat(st2[k]), P.flat(after[k])), k
    # the free-running oracle's loss in its exact-rounding mode (x and W16
    # rounded, everything else fp64): within 2e-2, as stated for bf16
    # (that mode rounds x, already bf16, and W16 = rne(P) once: the same
    # arithmetic as om.forward(..., "bf16"), with the weights rounded up front)
    p_exact = [om.rne_bf16(P.to64(p)) if i % 2 == 0 else P.to64(p) for i, p in enumerate(params0)]
    zl = []
    for r0 in range(0, w.batch, CHUNK):
        fw = om.forward(p_exact, P.to64(x[r0:r0 + CHUNK]), w.acts, "fp64")
        zl.append(om.softmax_ce(fw["z"], y[r0:r0 + CHUNK].numpy().astype(np.int64))[0])
    exact = float(np.concatenate(zl).mean())
    assert abs(rep["loss"] - exact) <= 2e-2 * abs(exact), (rep["loss"], exact)


def test_ragged_pair_tiles_layer_by_layer():
    """A ragged bf16 net whose forwards run on CTA pairs by default (so they
    also store their activations transposed and the weight gradients read
    them K-major): 2000 rows, widths 2600 and 2520, GELU and ReLU; every
    kernel of a step checked element by element."""
    from tests.test_gpu_step import RAGGED_PAIRS as w
    m = make_model(w, synth.make_params(w))
    x, y = synth.make_batch(w, 0)
    xd, yd = x.to(DEV), y.to(DEV)
    names = [n for n, _ in nn.mlp_profile_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps,
                                                 w.wd, None, m.stream())]
    assert names.count("tc2_gemm_fwd") == 2 and names.count("tc2_gemm_wgrad") == 2, names
    m.close()
    m = make_model(w, synth.make_params(w))
    rep, _, _, _ = traced_step_check(w, m, 0)
    m.close()
    assert rep["backward"] == "ok"


# Ragged nets (widths that are multiples of 8, as the bf16 row pitches need)
# whose bf16 weight gradients run in one wave with 16, 5, 3 and 2 column
# tiles of 256, so that the bias-gradient sums of a row tile are
# shared among its column tiles in every arrangement the kernels use (parts
# over eight epilogue warps: 8 of 16 tiles, 5, 3, 2), on CTA pairs and on one
# SM.  Both kernels give the same sums, so only a check against the oracle
# shows that every row of db is summed once.
BIAS_PARTS = [
    synth.Workload("bias_parts_16_2", (4000, 512, 1096, 100), (om.ACT_GELU_TANH, om.ACT_RELU), synth.BF16, 1000, 2,
                   1e-3, 0.9, 0.999, 1e-8, 0.01, "normal", 21),
    synth.Workload("bias_parts_5_3", (1096, 704, 2200, 100), (om.ACT_RELU, om.ACT_GELU_TANH), synth.BF16, 1200, 2,
                   1e-3, 0.9, 0.999, 1e-8, 0.01, "normal", 22),
]


@pytest.mark.parametrize("two_sm", [1, 0])
@pytest.mark.parametrize("w", BIAS_PARTS, ids=[w.name for w in BIAS_PARTS])
def test_bias_gradient_parts_layer_by_layer(w, two_sm):
    m = make_model(w, synth.make_params(w))
    m.set_option(nn.OPT_GEMM_2SM, two_sm)
    x, y = synth.make_batch(w, 0)
    xd, yd = x.to(DEV), y.to(DEV)
    names = [n for n, _ in nn.mlp_profile_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps,
                                                 w.wd, None, m.stream())]
    assert (names.count("tc2_gemm_wgrad") == 2) == (two_sm == 1), names
    m.close()
    m = make_model(w, synth.make_params(w))
    m.set_option(nn.OPT_GEMM_2SM, two_sm)
    rep, _, _, _ = traced_step_check(w, m, 0)
    m.close()
    assert rep["backward"] == "ok"


def test_trace_entries_describe_the_step():
    """The trace lists each stored tensor once, written by the launch that the
    profiling pass names for it."""
    w = W["lm_block_t16384"].with_(batch=256)
    m = make_model(w)
    x, y = synth.make_batch(w, 0)
    xd, yd = x.to(DEV), y.to(DEV)
    names = [n for n, _ in nn.mlp_profile_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps,
                                                 w.wd, None, m.stream())]
    ents, need = nn.mlp_trace_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps, w.wd, None,
                                   None, 0, m.stream())
    # (forward / dgrad launches run on one SM or on CTA pairs: tc_ or tc2_)
    kinds = [(e.kind, e.layer, names[e.launch].replace("tc2_", "tc_")) for e in ents]
    assert kinds == [(nn.TRACE_H, 0, "tc_gemm_fwd"), (nn.TRACE_U, 0, "tc_gemm_fwd"), (nn.TRACE_H, 1, "tc_gemm_fwd"),
                     (nn.TRACE_Z, 2, "tc_gemm_fwd"), (nn.TRACE_DZ, 2, "softmax_ce"),
                     (nn.TRACE_LOSS_ROWS, 2, "softmax_ce"), (nn.TRACE_DY, 1, "tc_gemm_dgrad"),
                     (nn.TRACE_DY, 0, "tc_gemm_dgrad")]
    assert need >= sum(e.bytes for e in ents)
    # a buffer one byte short is refused before anything runs
    buf = torch.empty(need - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(nn.MlpError):
        nn.mlp_trace_step(m.h, xd.data_ptr(), yd.data_ptr(), w.lr, w.beta1, w.beta2, w.eps, w.wd, None,
                          buf.data_ptr(), buf.numel(), m.stream())
    _, step = m.read_flat(nn.PLANE_P)
    assert step == 1   # only the profiling pass stepped
    m.close()
