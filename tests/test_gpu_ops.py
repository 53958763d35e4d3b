"""Op-level parity: each kernel of the step, called through the C ABI on
seeded inputs, against the CPU oracle element by element (small and ragged
shapes) or on sampled outputs (full-size shapes of the five workloads)."""
import math

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from oracle import mlp_oracle as om
from tests.parity import assert_close_gemm, to64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _tdt(dtype):
    return torch.float32 if dtype == nn.F32 else torch.bfloat16


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ---------------------------------------------------------------------------
# LinearAct forward
# ---------------------------------------------------------------------------
FWD_CASES = [
    # dtype, act, M, N, K
    (nn.F32, nn.ACT_RELU, 64, 256, 784),
    (nn.F32, nn.ACT_NONE, 77, 10, 128),
    (nn.F32, nn.ACT_GELU_TANH, 130, 72, 40),
    (nn.BF16, nn.ACT_RELU, 256, 256, 256),
    (nn.BF16, nn.ACT_RELU, 300, 384, 200),       # ragged M, K tail inside a 64-block
    (nn.BF16, nn.ACT_GELU_TANH, 200, 4096, 1024),
    (nn.BF16, nn.ACT_NONE, 300, 10, 1024),        # 10 outputs (16-wide tile)
    (nn.BF16, nn.ACT_NONE, 260, 100, 512),
    (nn.BF16, nn.ACT_NONE, 130, 1000, 64),
    (nn.BF16, nn.ACT_RELU, 4864, 1000, 320),      # 256-wide tiles (152 and more), ragged N
]


@pytest.mark.parametrize("dtype,act,M,N,K", FWD_CASES)
def test_linear_act_forward(dtype, act, M, N, K):
    td = _tdt(dtype)
    X = synth.make_normal((M, K), 1.0, 11, M, N, K, dtype=td)
    W = synth.make_normal((N, K), math.sqrt(2.0 / K), 12, M, N, K, dtype=td)
    b = synth.make_normal((N,), 0.5, 13, M, N, K)
    ldh = (N + 7) // 8 * 8
    Xd, Wd, bd = X.to(DEV), W.to(DEV), b.to(DEV)
    H = torch.full((M, ldh), float("nan"), dtype=td, device=DEV)
    U = torch.full((M, ldh), float("nan"), dtype=td, device=DEV) if act == nn.ACT_GELU_TANH else None
    err = _err()
    nn.mlp_op_linear_act(dtype, act, M, N, K, Xd.data_ptr(), K, Wd.data_ptr(), K, bd.data_ptr(), H.data_ptr(), ldh,
                         U.data_ptr() if U is not None else None, ldh, err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    x64, w64, b64 = to64(X), to64(W), to64(b)
    u = om.linear(x64, w64, b64)
    h = om.act_forward(u, act)
    absum = np.abs(x64) @ np.abs(w64).T + np.abs(b64)
    got = to64(H)[:, :N]
    # the activation is 1-Lipschitz (GELU-tanh: |gelu'| < 1.13), so the GEMM
    # bound carries through it with a factor 1.13
    assert_close_gemm(got, h, 1.13 * absum, K, dtype == nn.BF16, "H")
    if U is not None:
        assert_close_gemm(to64(U)[:, :N], u, absum, K, True, "U")


# ---------------------------------------------------------------------------
# dgrad with the activation VJP
# ---------------------------------------------------------------------------
DGRAD_CASES = [
    (nn.F32, nn.ACT_RELU, 64, 10, 128),
    (nn.F32, nn.ACT_RELU, 4096, 128, 256),
    (nn.BF16, nn.ACT_RELU, 300, 1024, 1024),
    (nn.BF16, nn.ACT_RELU, 260, 10, 1024),        # reduction over 10 classes
    (nn.BF16, nn.ACT_GELU_TANH, 200, 1024, 4096),
    (nn.BF16, nn.ACT_NONE, 130, 32000, 1024),
    (nn.BF16, nn.ACT_RELU, 250, 100, 512),
    (nn.BF16, nn.ACT_RELU, 4864, 200, 1000),      # MN-major W, ragged N, K tail
]


@pytest.mark.parametrize("dtype,act,M,N,K", DGRAD_CASES)
def test_dgrad(dtype, act, M, N, K):
    """dX[M,K] = (dY[M,N] W[N,K]) * act'(S[M,K])."""
    td = _tdt(dtype)
    ldy = (N + 7) // 8 * 8
    dY = synth.make_normal((M, ldy), 1e-3, 21, M, N, K, dtype=td)
    W = synth.make_normal((N, K), math.sqrt(2.0 / K), 22, M, N, K, dtype=td)
    S = synth.make_normal((M, K), 1.0, 23, M, N, K, dtype=td)
    if act == nn.ACT_RELU:
        S = torch.relu(S)
    dYd, Wd, Sd = dY.to(DEV), W.to(DEV), S.to(DEV)
    dX = torch.full((M, K), float("nan"), dtype=td, device=DEV)
    err = _err()
    nn.mlp_op_dgrad(dtype, act, M, N, K, dYd.data_ptr(), ldy, Wd.data_ptr(), K, Sd.data_ptr(), K, dX.data_ptr(), K,
                    err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    dy64, w64, s64 = to64(dY)[:, :N], to64(W), to64(S)
    if act == nn.ACT_RELU:
        fac = (s64 > 0).astype(np.float64)
    elif act == nn.ACT_GELU_TANH:
        fac = om.gelu_tanh_grad(s64)
    else:
        fac = np.ones_like(s64)
    ref = (dy64 @ w64) * fac
    absum = (np.abs(dy64) @ np.abs(w64)) * np.abs(fac) * 1.001
    # GELU' is evaluated in fp32 on the stored u: a few ulp(1) absolute error
    # near its root (u ~ -0.75), so allow 2^-21 |dY||W| on top
    extra = (np.abs(dy64) @ np.abs(w64)) * 2.0 ** -21 if act == nn.ACT_GELU_TANH else None
    assert_close_gemm(to64(dX), ref, absum, N, dtype == nn.BF16, "dX", extra)


# ---------------------------------------------------------------------------
# wgrad with the fused bias gradient
# ---------------------------------------------------------------------------
WGRAD_CASES = [
    (nn.F32, 256, 784, 64),
    (nn.F32, 10, 128, 4096),
    (nn.F32, 128, 256, 4096),
    (nn.BF16, 1024, 1024, 512),
    (nn.BF16, 10, 1024, 640),
    (nn.BF16, 100, 512, 1000),                    # ragged batch
    (nn.BF16, 512, 512, 4096),                    # split-K
    (nn.BF16, 4096, 1024, 256),
    (nn.BF16, 2000, 1000, 16384),                 # 256-wide tiles (long K per unit), ragged M and N
]


@pytest.mark.parametrize("dtype,N,K,B", WGRAD_CASES)
def test_wgrad(dtype, N, K, B):
    """dW[N,K] = dY[B,N]^T X[B,K] (fp32), db[N] = sum_rows dY."""
    td = _tdt(dtype)
    ldy = (N + 7) // 8 * 8
    dY = synth.make_normal((B, ldy), 1e-3, 31, N, K, B, dtype=td)
    X = synth.make_normal((B, K), 1.0, 32, N, K, B, dtype=td)
    dYd, Xd = dY.to(DEV), X.to(DEV)
    dW = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
    db = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    wsb = nn.mlp_op_wgrad_workspace_bytes(dtype, N, K, B)
    ws = torch.empty(max(wsb, 4), dtype=torch.uint8, device=DEV)
    err = _err()
    nn.mlp_op_wgrad(dtype, N, K, B, dYd.data_ptr(), ldy, Xd.data_ptr(), K, dW.data_ptr(), K, db.data_ptr(),
                    ws.data_ptr(), wsb, err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    dy64, x64 = to64(dY)[:, :N], to64(X)
    ref = dy64.T @ x64
    absum = np.abs(dy64).T @ np.abs(x64)
    assert_close_gemm(to64(dW), ref, absum, B, False, "dW")
    refb = dy64.sum(0)
    assert_close_gemm(to64(db), refb, np.abs(dy64).sum(0), B, False, "db")


# ---------------------------------------------------------------------------
# Softmax cross-entropy (+ loss mean)
# ---------------------------------------------------------------------------
CE_CASES = [
    (nn.F32, 64, 10), (nn.F32, 4096, 10), (nn.BF16, 8192, 10), (nn.BF16, 1000, 100),
    (nn.BF16, 256, 32000), (nn.F32, 33, 1003), (nn.BF16, 17, 777), (nn.F32, 5, 1),
    (nn.F32, 40, 8000), (nn.BF16, 64, 4096),
    # four elements a lane (C % 4 == 0): one and two 128-wide slots, ragged
    (nn.F32, 77, 12), (nn.F32, 300, 200), (nn.BF16, 129, 256), (nn.BF16, 65536, 100),
]


@pytest.mark.parametrize("dtype,B,C", CE_CASES)
def test_softmax_ce(dtype, B, C):
    td = _tdt(dtype)
    ld = (C + 7) // 8 * 8
    z = synth.make_normal((B, ld), 3.0, 41, B, C, dtype=td)
    y = synth.make_labels(B, C, 42, B, C)
    zd, yd = z.to(DEV), y.to(DEV)
    dz = torch.full((B, ld), float("nan"), dtype=td, device=DEV)
    rows = torch.full((B,), float("nan"), dtype=torch.float32, device=DEV)
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device=DEV)
    err = _err()
    nn.mlp_op_softmax_ce(dtype, B, C, zd.data_ptr(), ld, yd.data_ptr(), 1.0 / B, dz.data_ptr(), ld, rows.data_ptr(),
                         err.data_ptr(), _stream())
    nn.mlp_op_loss_mean(B, rows.data_ptr(), loss.data_ptr(), err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    z64 = to64(z)[:, :C]
    lr_ref, dz_ref = om.softmax_ce(z64, y.numpy())
    # fp32 math on exactly-representable inputs: relative 1e-5 on the loss
    # rows (log-sum-exp of up to 32000 terms), and for dz half a bf16 ulp
    # (bf16) or 1e-5 relative (fp32) plus a tiny absolute floor
    np.testing.assert_allclose(to64(rows), lr_ref, rtol=1e-5, atol=1e-5)
    got = to64(dz)[:, :C]
    rt = 2.0 ** -8 if dtype == nn.BF16 else 1e-5
    assert np.all(np.abs(got - dz_ref) <= rt * np.abs(dz_ref) + 1e-6 / B / C), np.max(np.abs(got - dz_ref))
    assert abs(loss.item() - lr_ref.mean()) <= 1e-5 * abs(lr_ref.mean()) + 1e-6


def test_softmax_ce_zero_logits_closed_form_and_label_gather():
    """Zero logits: loss = ln C, dz = (1/C - onehot)/B; a bias pattern z_c =
    c * delta picks out z[y] exactly: loss_i = lse - y_i * delta."""
    B, C = 300, 32000
    z = torch.zeros((B, C), dtype=torch.bfloat16, device=DEV)
    y = synth.make_labels(B, C, 43).to(DEV)
    dz = torch.empty_like(z)
    rows = torch.empty(B, dtype=torch.float32, device=DEV)
    nn.mlp_op_softmax_ce(nn.BF16, B, C, z.data_ptr(), C, y.data_ptr(), 1.0 / B, dz.data_ptr(), C, rows.data_ptr(),
                         None, _stream())
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(rows), math.log(C), rtol=1e-6)
    ref = np.full((B, C), 1.0 / C / B)
    ref[np.arange(B), y.cpu().numpy()] -= 1.0 / B
    np.testing.assert_allclose(to64(dz), ref, rtol=2.0 ** -8, atol=0)
    # label gather: z_c = c * 2^-6 is exact in bf16 for c < 256
    C2 = 200
    zc = (torch.arange(C2, dtype=torch.float32) * 2.0 ** -6).to(torch.bfloat16)
    z2 = zc.repeat(B, 1).to(DEV).contiguous()
    y2 = synth.make_labels(B, C2, 44)
    dz2 = torch.empty_like(z2)
    rows2 = torch.empty(B, dtype=torch.float32, device=DEV)
    nn.mlp_op_softmax_ce(nn.BF16, B, C2, z2.data_ptr(), C2, y2.to(DEV).data_ptr(), 1.0 / B, dz2.data_ptr(), C2,
                         rows2.data_ptr(), None, _stream())
    torch.cuda.synchronize()
    zz = to64(zc)
    lse = zz.max() + np.log(np.exp(zz - zz.max()).sum())
    want = lse - zz[y2.numpy()]
    np.testing.assert_allclose(to64(rows2), want, rtol=0, atol=2e-5)


@pytest.mark.parametrize("C", [10, 12])
def test_softmax_ce_label_out_of_range_sets_error_bit(C):
    B = 8
    z = torch.zeros((B, C), dtype=torch.float32, device=DEV)
    y = torch.tensor([0, 1, 2, C, 4, -1, 6, 7], dtype=torch.int32, device=DEV)
    dz = torch.empty_like(z)
    rows = torch.empty(B, dtype=torch.float32, device=DEV)
    err = _err()
    nn.mlp_op_softmax_ce(nn.F32, B, C, z.data_ptr(), C, y.data_ptr(), 1.0 / B, dz.data_ptr(), C, rows.data_ptr(),
                         err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() & 1
    r = rows.cpu().numpy()
    assert r[3] == 0.0 and r[5] == 0.0 and abs(r[0] - math.log(C)) < 1e-6


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,t,with_w16", [(1000, 1, False), (4099, 7, True), (5256202, 3, True)])
def test_adamw(n, t, with_w16):
    p = synth.make_normal((n,), 0.05, 51, n)
    g = synth.make_normal((n,), 1e-3, 52, n)
    m = synth.make_normal((n,), 1e-4, 53, n)
    v = synth.make_uniform((n,), 0.0, 1e-6, 54, n)
    if t == 1:
        m.zero_()
        v.zero_()
    pd, gd, md, vd = (a.to(DEV) for a in (p, g, m, v))
    w16 = torch.empty(n, dtype=torch.bfloat16, device=DEV) if with_w16 else None
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.05
    nn.mlp_op_adamw(n, pd.data_ptr(), gd.data_ptr(), md.data_ptr(), vd.data_ptr(),
                    w16.data_ptr() if w16 is not None else None, t, lr, b1, b2, eps, wd, _stream())
    torch.cuda.synchronize()
    # the C ABI takes fp32 hyper-parameters: give the oracle the same values
    f = lambda a: float(np.float32(a))
    p64, g64, m64, v64 = to64(p), to64(g), to64(m), to64(v)
    pr, mr, vr = om.adamw(p64, g64, m64, v64, t, f(lr), f(b1), f(b2), f(eps), f(wd))
    # fp32 arithmetic: a few ulp of the larger term of each moment update
    tol_m = 2.0 ** -21 * (f(b1) * np.abs(m64) + (1 - f(b1)) * np.abs(g64)) + 1e-30
    tol_v = 2.0 ** -21 * (f(b2) * v64 + (1 - f(b2)) * g64 * g64) + 1e-38
    assert np.all(np.abs(to64(md) - mr) <= tol_m)
    assert np.all(np.abs(to64(vd) - vr) <= tol_v)
    # the update term has size ~lr: relative 1e-5 of lr plus the ulp of p
    assert np.all(np.abs(to64(pd) - pr) <= 1e-5 * lr + 2.0 ** -23 * np.abs(pr))
    if w16 is not None:
        assert torch.equal(w16.cpu(), pd.cpu().to(torch.bfloat16))


# ---------------------------------------------------------------------------
# argmax
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,B,C", [(nn.F32, 64, 10), (nn.BF16, 300, 100), (nn.BF16, 50, 32000)])
def test_argmax_bit_exact_with_ties(dtype, B, C):
    td = _tdt(dtype)
    # coarse integer values make ties common
    z = torch.from_numpy(np.random.default_rng(61).integers(0, 5, (B, C)).astype(np.float32)).to(td)
    out = torch.empty(B, dtype=torch.int32, device=DEV)
    zd = z.to(DEV)
    nn.mlp_op_argmax(dtype, B, C, zd.data_ptr(), C, out.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), om.argmax_rows(to64(z)))


# ---------------------------------------------------------------------------
# The error path of the bounded device waits (no fault: the wait gives up)
# ---------------------------------------------------------------------------
def test_bounded_wait_gives_up_and_context_stays_usable():
    import time
    err = _err()
    t0 = time.perf_counter()
    nn.mlp_op_wait_timeout_check(50_000_000, err.data_ptr(), _stream())   # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert err.item() == 4                 # the timeout bit, nothing else
    assert 0.05 <= dt < 5.0
    # the context still runs kernels correctly afterwards
    test_linear_act_forward(nn.BF16, nn.ACT_RELU, 256, 256, 256)
    with pytest.raises(nn.MlpError):
        nn.mlp_op_wait_timeout_check(2_000_000_000, err.data_ptr(), _stream())   # over the 1 s cap
