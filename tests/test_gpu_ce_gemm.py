"""Softmax cross-entropy inside the output layer's GEMMs (bf16): the forward's
epilogue statistics, the combine, and dz formed in shared memory by the dgrad
and the wgrad, through mlp_op_linear_ce against the oracle (element by
element on ragged shapes; sampled rows at the 16384 x 32000 x 1024 LM-head
size), and the training step with the option on against the separate
softmax-CE pass."""
import math

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from oracle import mlp_oracle as om
from tests import parity as P
from tests.parity import assert_close_gemm, gemm_tol, to64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _run_op(B, C, K, act, seed, bad_label=False):
    h = synth.make_normal((B, K), 1.0, seed, 1, dtype=torch.bfloat16)
    if act == nn.ACT_RELU:
        h = torch.relu(h)
    W = synth.make_normal((C, K), math.sqrt(2.0 / K), seed, 2, dtype=torch.bfloat16)
    b = synth.make_normal((C,), 0.5, seed, 3)
    y = synth.make_labels(B, C, seed, 4)
    if bad_label:
        y[B // 2] = C
    aux = None
    if act == nn.ACT_RELU:
        aux = h
    elif act == nn.ACT_GELU_TANH:
        aux = synth.make_normal((B, K), 1.0, seed, 5, dtype=torch.bfloat16)
    ldz = (C + 7) // 8 * 8
    hd, Wd, bd, yd = h.to(DEV), W.to(DEV), b.to(DEV), y.to(DEV)
    auxd = aux.to(DEV) if aux is not None else None
    z = torch.full((B, ldz), float("nan"), dtype=torch.bfloat16, device=DEV)
    rows = torch.full((B,), float("nan"), dtype=torch.float32, device=DEV)
    dX = torch.full((B, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dW = torch.full((C, K), float("nan"), dtype=torch.float32, device=DEV)
    db = torch.full((C,), float("nan"), dtype=torch.float32, device=DEV)
    wsb = nn.mlp_op_linear_ce_workspace_bytes(B, C, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nn.mlp_op_linear_ce(B, C, K, hd.data_ptr(), K, Wd.data_ptr(), bd.data_ptr(), yd.data_ptr(), act,
                        auxd.data_ptr() if auxd is not None else None, K, z.data_ptr(), ldz, rows.data_ptr(),
                        dX.data_ptr(), K, dW.data_ptr(), K, db.data_ptr(), ws.data_ptr(), wsb, err.data_ptr(),
                        _stream())
    torch.cuda.synchronize()
    return dict(h=h, W=W, b=b, y=y, aux=aux, z=z[:, :C], rows=rows, dX=dX, dW=dW, db=db, err=err.item())


def _act_fac(act, aux64):
    if act == nn.ACT_RELU:
        return (aux64 > 0).astype(np.float64)
    if act == nn.ACT_GELU_TANH:
        return om.gelu_tanh_grad(aux64)
    return 1.0


def _oracle_and_bounds(out, act, rows=None):
    """The oracle's mirror computation (logits and dz rounded to bf16) on rows
    `rows` (all by default), and the bound E on |dz - dz*| per element: one
    bf16 ulp of the rounding plus the softmax's response to the logits' own
    tolerance Dz (|d softmax_c| <= 2 p_c Dz)."""
    h64 = to64(out["h"]) if rows is None else to64(out["h"][rows])
    y = out["y"].numpy().astype(np.int64) if rows is None else out["y"].numpy().astype(np.int64)[rows]
    w64, b64 = to64(out["W"]), to64(out["b"])
    B_all = out["h"].shape[0]
    u = om.linear(h64, w64, b64)
    absum = np.abs(h64) @ np.abs(w64).T + np.abs(b64)
    z_star = om.rne_bf16(u)
    tol_z = gemm_tol(absum, h64.shape[1], u, True)
    loss_star, dz_exact = om.softmax_ce(z_star, y)
    dz_exact = dz_exact * (len(y) / B_all)          # the oracle scales by its own rows; the kernels by 1/B
    dz_star = om.rne_bf16(dz_exact)
    p = dz_exact * B_all
    p[np.arange(len(y)), y] += 1.0                  # softmax probabilities
    Dz = tol_z.max(axis=1, keepdims=True)
    E = 2.0 ** -7 * np.abs(dz_star) + (2.0 * p * Dz + 2.0 ** -20 * p) / B_all + 1e-30
    return dict(u=u, absum=absum, z_star=z_star, loss=loss_star, dz=dz_star, E=E, Dz=Dz[:, 0], h64=h64)


CASES = [
    # B, C, K, act
    (300, 1000, 256, nn.ACT_NONE),       # ragged batch, a partial 128-column group
    (129, 520, 128, nn.ACT_RELU),        # a group of 8 columns; ReLU VJP below
    (256, 4096, 512, nn.ACT_GELU_TANH),  # GELU VJP below
    (1000, 2056, 64, nn.ACT_NONE),       # a last tile with one partial group
]


@pytest.mark.parametrize("B,C,K,act", CASES)
def test_linear_ce_elementwise(B, C, K, act):
    out = _run_op(B, C, K, act, seed=B + C + K)
    assert out["err"] == 0
    o = _oracle_and_bounds(out, act)
    assert_close_gemm(to64(out["z"]), o["u"], o["absum"], K, True, "z")
    # loss rows from the stored logits: the logits' tolerance moves them by <= 2 Dz
    lr = to64(out["rows"])
    assert np.all(np.abs(lr - o["loss"]) <= 2 * o["Dz"] + 1e-5 * np.abs(o["loss"]) + 1e-6)
    w64 = to64(out["W"])
    fac = _act_fac(act, to64(out["aux"]) if out["aux"] is not None else None)
    ref = (o["dz"] @ w64) * fac
    extra = (o["E"] @ np.abs(w64)) * np.abs(fac)
    if act == nn.ACT_GELU_TANH:
        extra = extra + (np.abs(o["dz"]) @ np.abs(w64)) * 2.0 ** -21
    assert_close_gemm(to64(out["dX"]), ref, (np.abs(o["dz"]) @ np.abs(w64)) * np.abs(fac) * 1.001, C, True, "dX",
                      extra)
    h64 = o["h64"]
    assert_close_gemm(to64(out["dW"]), o["dz"].T @ h64, np.abs(o["dz"]).T @ np.abs(h64), B, False, "dW",
                      o["E"].T @ np.abs(h64))
    assert_close_gemm(to64(out["db"]), o["dz"].sum(0), np.abs(o["dz"]).sum(0), B, False, "db", o["E"].sum(0))


def test_linear_ce_label_out_of_range_sets_error_bit():
    out = _run_op(200, 1000, 128, nn.ACT_NONE, seed=7, bad_label=True)
    assert out["err"] & 1
    assert out["rows"][100].item() == 0.0


def test_linear_ce_full_size_lm_head_sampled_rows():
    """The 16384 x 32000 x 1024 LM head: loss rows and dX rows (which need
    only the oracle's logits of those rows) on sampled rows, including the
    first and the last; dW / db through the property sum_c db_c = sum_i
    sum_c dz_ic, which is 0 up to the rounding of dz."""
    B, C, K = 16384, 32000, 1024
    out = _run_op(B, C, K, nn.ACT_NONE, seed=99)
    assert out["err"] == 0
    r = np.unique(np.concatenate([[0, B - 1], np.random.default_rng(98).integers(0, B, 30)]))
    o = _oracle_and_bounds(out, nn.ACT_NONE, rows=r)
    assert_close_gemm(to64(out["z"][r]), o["u"], o["absum"], K, True, "z")
    lr = to64(out["rows"])[r]
    assert np.all(np.abs(lr - o["loss"]) <= 2 * o["Dz"] + 1e-5 * np.abs(o["loss"]) + 1e-6)
    w64 = to64(out["W"])
    assert_close_gemm(to64(out["dX"][r]), o["dz"] @ w64, np.abs(o["dz"]) @ np.abs(w64) * 1.001, C, True, "dX",
                      o["E"] @ np.abs(w64))
    db = to64(out["db"])
    assert np.all(np.isfinite(to64(out["dW"]))) and np.all(np.isfinite(db))
    # each row of dz sums to 0 before rounding; the rounding moves a row's sum
    # by at most 2^-9 sum_c |dz_ic| <= 2^-9 * 2 / B, and fp32 sums add little
    assert abs(db.sum()) <= 2.0 ** -9 * 2.0 + 1e-4


# ---------------------------------------------------------------------------
# The training step: CE in the GEMMs vs the separate softmax-CE pass
# ---------------------------------------------------------------------------
def _lm_step(w, ce_gemm, batch, names=False):
    params0 = synth.make_params(w)
    m = nn.Model(w.dims, w.acts, nn.ACT_RELU, w.dtype, seed=w.seed, batch=batch)
    m.set_option(nn.OPT_CE_GEMM, ce_gemm)
    m.write_flat(P.flat([p.numpy() for p in params0]).astype(np.float32), nn.PLANE_P, 0)
    x, y = synth.make_batch(w, 0, batch)
    xd, yd = x.to(DEV), y.to(DEV)
    kn = None
    if names:
        kn = [n for n, _ in nn.mlp_profile_step(m.h, xd.data_ptr(), yd.data_ptr(), 0.0, 0.9, 0.999, 1e-8, 0.0, None,
                                               m.stream())]
        m.write_flat(P.flat([p.numpy() for p in params0]).astype(np.float32), nn.PLANE_P, 0)
    loss = m.train_step(xd, yd, w.lr, w.beta1, w.beta2, w.eps, w.wd)
    m.check_errors()
    g, _ = m.read_flat(nn.PLANE_G)
    p, _ = m.read_flat(nn.PLANE_P)
    m.close()
    return loss.item(), g.astype(np.float64), p.astype(np.float64), kn


@pytest.mark.parametrize("batch", [200, 16384])
def test_lm_block_step_ce_in_gemms_matches_separate_pass(batch):
    """Same rounding points (logits, dz); the row sums differ in order only,
    so the loss agrees to fp32 accuracy and the gradients to the bf16 rounding
    of a few dz elements; the kernels that ran are the fused ones."""
    w = synth.WORKLOADS["lm_block_t16384"]
    l1, g1, p1, k1 = _lm_step(w, 1, batch, names=True)
    l0, g0, p0, k0 = _lm_step(w, 0, batch, names=True)
    assert "ce_combine" in k1 and "softmax_ce" not in k1
    assert "softmax_ce" in k0 and "ce_combine" not in k0
    assert abs(l1 - l0) <= 1e-5 * abs(l0)
    # per gradient tensor: the two agree up to a few bf16 ulps of dz
    pos = 0
    for l in range(w.n_layers):
        for size in (w.dims[l + 1] * w.dims[l], w.dims[l + 1]):
            a, b_ = g1[pos:pos + size], g0[pos:pos + size]
            assert np.max(np.abs(a - b_)) <= 2e-2 * (np.max(np.abs(b_)) + 1e-30), (l, size)
            pos += size
