"""Full-size parity in the launch configuration the benchmark times.

Every distinct GEMM of the five workloads (forward with its activation,
dgrad with the activation VJP, wgrad with the fused bias gradient) runs
through the C ABI at its full shape on seeded inputs; sampled outputs --
including the first and last row and column, so ragged tile edges are
covered -- are checked against the oracle's definition, each computed one by
one.  The 16384 x 32000 softmax-CE is checked on sampled rows, and AdamW on
all 41 M parameters of the largest model.
"""
import math

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from oracle import mlp_oracle as om
from tests.parity import gemm_tol, to64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _shapes():
    seen, out = set(), []
    for name in synth.WORKLOAD_ORDER:
        w = synth.WORKLOADS[name]
        B = w.batch
        for l in range(w.n_layers):
            K, N = w.dims[l], w.dims[l + 1]
            act = w.acts[l] if l < w.n_layers - 1 else nn.ACT_NONE
            below = w.acts[l - 1] if l > 0 else None
            cases = [("fwd", B, N, K, act), ("wgrad", N, K, B, None)]
            if l > 0:
                cases.append(("dgrad", B, N, K, below))
            for c in cases:
                key = (w.dtype,) + c
                if key not in seen:
                    seen.add(key)
                    out.append(pytest.param(w.dtype, *c, id=f"{name}-{c[0]}-L{l + 1}"))
    return out


def _samples(rows, cols, n, seed):
    rng = np.random.default_rng(seed)
    r = np.concatenate([[0, rows - 1], rng.integers(0, rows, n)])
    c = np.concatenate([[cols - 1, 0], rng.integers(0, cols, n)])
    return r, c


@pytest.mark.parametrize("dtype,kind,d0,d1,d2,act", _shapes())
def test_gemm_full_size_sampled(dtype, kind, d0, d1, d2, act):
    td = torch.float32 if dtype == nn.F32 else torch.bfloat16
    bf = dtype == nn.BF16
    s = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if kind == "fwd":
        M, N, K = d0, d1, d2
        X = synth.make_normal((M, K), 1.0, 301, M, N, K, dtype=td).to(DEV)
        W = synth.make_normal((N, K), math.sqrt(2.0 / K), 302, M, N, K, dtype=td).to(DEV)
        b = synth.make_normal((N,), 0.3, 303, M, N, K).to(DEV)
        ldh = (N + 7) // 8 * 8
        H = torch.empty((M, ldh), dtype=td, device=DEV)
        U = torch.empty((M, ldh), dtype=td, device=DEV) if act == nn.ACT_GELU_TANH else None
        nn.mlp_op_linear_act(dtype, act, M, N, K, X.data_ptr(), K, W.data_ptr(), K, b.data_ptr(), H.data_ptr(), ldh,
                             U.data_ptr() if U is not None else None, ldh, err.data_ptr(), s)
        torch.cuda.synchronize()
        r, c = _samples(M, N, 62, 304)
        xr, wc = to64(X[torch.as_tensor(r, device=DEV)]), to64(W[torch.as_tensor(c, device=DEV)])
        u = np.sum(xr * wc, axis=1) + to64(b)[c]
        ref = om.act_forward(u, act)
        absum = np.sum(np.abs(xr * wc), axis=1) + np.abs(to64(b)[c])
        got = to64(H[torch.as_tensor(r, device=DEV), torch.as_tensor(c, device=DEV)])
        tol = gemm_tol(1.13 * absum, K, ref, bf)
    elif kind == "dgrad":
        M, Nout, Kin = d0, d1, d2      # dX[M, Kin] = (dY[M, Nout] W[Nout, Kin]) * act'
        ldy = (Nout + 7) // 8 * 8
        dY = synth.make_normal((M, ldy), 1e-3, 311, M, Nout, Kin, dtype=td).to(DEV)
        W = synth.make_normal((Nout, Kin), math.sqrt(2.0 / Kin), 312, M, Nout, Kin, dtype=td).to(DEV)
        S = synth.make_normal((M, Kin), 1.0, 313, M, Nout, Kin, dtype=td).to(DEV)
        if act == nn.ACT_RELU:
            S = torch.relu(S)
        dX = torch.empty((M, Kin), dtype=td, device=DEV)
        nn.mlp_op_dgrad(dtype, act, M, Nout, Kin, dY.data_ptr(), ldy, W.data_ptr(), Kin, S.data_ptr(), Kin,
                        dX.data_ptr(), Kin, err.data_ptr(), s)
        torch.cuda.synchronize()
        r, c = _samples(M, Kin, 62, 314)
        dyr = to64(dY[torch.as_tensor(r, device=DEV), :Nout])
        wc = to64(W[:, torch.as_tensor(c, device=DEV)]).T
        sv = to64(S[torch.as_tensor(r, device=DEV), torch.as_tensor(c, device=DEV)])
        fac = (sv > 0).astype(float) if act == nn.ACT_RELU else (
            om.gelu_tanh_grad(sv) if act == nn.ACT_GELU_TANH else np.ones_like(sv))
        ref = np.sum(dyr * wc, axis=1) * fac
        absum = np.sum(np.abs(dyr * wc), axis=1) * (np.abs(fac) + 2.0 ** -12)
        got = to64(dX[torch.as_tensor(r, device=DEV), torch.as_tensor(c, device=DEV)])
        tol = gemm_tol(absum, Nout, ref, bf)
        K = Nout
    else:
        Nout, Kin, B = d0, d1, d2      # dW[Nout, Kin] = dY[B, Nout]^T X[B, Kin], db = colsum dY
        ldy = (Nout + 7) // 8 * 8
        dY = synth.make_normal((B, ldy), 1e-3, 321, Nout, Kin, B, dtype=td).to(DEV)
        X = synth.make_normal((B, Kin), 1.0, 322, Nout, Kin, B, dtype=td).to(DEV)
        dW = torch.empty((Nout, Kin), dtype=torch.float32, device=DEV)
        db = torch.empty(Nout, dtype=torch.float32, device=DEV)
        wsb = nn.mlp_op_wgrad_workspace_bytes(dtype, Nout, Kin, B)
        ws = torch.empty(max(wsb, 4), dtype=torch.uint8, device=DEV)
        nn.mlp_op_wgrad(dtype, Nout, Kin, B, dY.data_ptr(), ldy, X.data_ptr(), Kin, dW.data_ptr(), Kin, db.data_ptr(),
                        ws.data_ptr(), wsb, err.data_ptr(), s)
        torch.cuda.synchronize()
        r, c = _samples(Nout, Kin, 30, 324)
        dyc = to64(dY[:, torch.as_tensor(r, device=DEV)])       # [B, n]
        xc = to64(X[:, torch.as_tensor(c, device=DEV)])         # [B, n]
        ref = np.sum(dyc * xc, axis=0)
        absum = np.sum(np.abs(dyc * xc), axis=0)
        got = to64(dW[torch.as_tensor(r, device=DEV), torch.as_tensor(c, device=DEV)])
        tol = gemm_tol(absum, B, ref, False)
        rb = np.unique(r)
        dyb = to64(dY[:, torch.as_tensor(rb, device=DEV)])
        refb = dyb.sum(0)
        tolb = gemm_tol(np.abs(dyb).sum(0), B, refb, False)
        assert np.all(np.abs(to64(db)[rb] - refb) <= tolb)
        K = B
    assert err.item() == 0
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (kind, int(bad.sum()), np.max(np.abs(got - ref) / tol))


def test_softmax_ce_full_size_lm_head_sampled_rows():
    B, C = 16384, 32000
    z = synth.make_normal((B, C), 2.0, 331, dtype=torch.bfloat16).to(DEV)
    y = synth.make_labels(B, C, 332).to(DEV)
    dz = torch.empty_like(z)
    rows = torch.empty(B, dtype=torch.float32, device=DEV)
    nn.mlp_op_softmax_ce(nn.BF16, B, C, z.data_ptr(), C, y.data_ptr(), 1.0 / B, dz.data_ptr(), C, rows.data_ptr(),
                         None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    r = np.concatenate([[0, B - 1], np.random.default_rng(333).integers(0, B, 30)])
    rt = torch.as_tensor(r, device=DEV)
    lr_ref, dz_ref = om.softmax_ce(to64(z[rt]), y[rt].cpu().numpy())
    dz_ref = dz_ref * (len(r) / B)   # the oracle scales by 1/(rows it was given); the kernel by 1/B
    np.testing.assert_allclose(to64(rows[rt]), lr_ref, rtol=1e-5, atol=1e-5)
    got = to64(dz[rt])
    assert np.all(np.abs(got - dz_ref) <= 2.0 ** -8 * np.abs(dz_ref) + 1e-6 / B / C)


def test_adamw_full_size_lm_block_all_parameters():
    w = synth.WORKLOADS["lm_block_t16384"]
    n = w.n_params()
    p = synth.make_normal((n,), 0.02, 341)
    g = synth.make_normal((n,), 1e-4, 342)
    m = synth.make_normal((n,), 1e-5, 343)
    v = synth.make_uniform((n,), 0.0, 1e-8, 344)
    pd, gd, md, vd = (a.to(DEV) for a in (p, g, m, v))
    w16 = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    t = 7
    f = lambda a: float(np.float32(a))
    nn.mlp_op_adamw(n, pd.data_ptr(), gd.data_ptr(), md.data_ptr(), vd.data_ptr(), w16.data_ptr(), t, w.lr, w.beta1,
                    w.beta2, w.eps, w.wd, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    p64, g64, m64, v64 = to64(p), to64(g), to64(m), to64(v)
    pr, mr, vr = om.adamw(p64, g64, m64, v64, t, f(w.lr), f(w.beta1), f(w.beta2), f(w.eps), f(w.wd))
    assert np.all(np.abs(to64(md) - mr) <= 2.0 ** -21 * (f(w.beta1) * np.abs(m64) + (1 - f(w.beta1)) * np.abs(g64)) + 1e-30)
    assert np.all(np.abs(to64(vd) - vr) <= 2.0 ** -21 * (f(w.beta2) * v64 + (1 - f(w.beta2)) * g64 * g64) + 1e-38)
    assert np.all(np.abs(to64(pd) - pr) <= 1e-5 * w.lr + 2.0 ** -23 * np.abs(pr))
    assert torch.equal(w16.cpu(), pd.cpu().to(torch.bfloat16))
