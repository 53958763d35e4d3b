"""fp32 GEMMs on the tensor cores (MLP_F32X3 operands: three bf16 planes per
fp32 value) against the oracle's fp32 GEMMs in fp64, element by element.

The plane encoding is checked bit for bit against its definition
(hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid)), computed here
on the CPU with torch's round-to-nearest-even casts.  A GEMM result comes
back as planes too; their fp64 sum is the kernel's fp32 result exactly.

Tolerance: the fp32 accumulation bound of the other GEMM tests
(8 sqrt(K) 2^-24 sum|a b|) plus the plane products the kernel leaves out:
mid*lo, lo*mid and lo*lo are each below 2^-24 |a b| (|mid| <= 2^-8 |x|,
|lo| <= 2^-16 |x|), so 2^-22 sum|a b| covers them with room.
"""
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
DROPPED = 2.0 ** -22


def _stream():
    return torch.cuda.current_stream().cuda_stream


def planes_cpu(x: torch.Tensor, ld: int) -> torch.Tensor:
    """[3, rows, ld] bf16 planes of an fp32 [rows, cols] CPU tensor (columns
    beyond cols zero)."""
    rows, cols = x.shape
    hi = x.to(torch.bfloat16)
    r = x - hi.float()
    mid = r.to(torch.bfloat16)
    lo = (r - mid.float()).to(torch.bfloat16)
    out = torch.zeros((3, rows, ld), dtype=torch.bfloat16)
    out[0, :, :cols], out[1, :, :cols], out[2, :, :cols] = hi, mid, lo
    return out


def from_planes(p: torch.Tensor, cols: int) -> np.ndarray:
    q = to64(p)
    return (q[0] + q[1] + q[2])[:, :cols]


def test_split3_bit_exact_and_exact_sum():
    rows, cols, ld = 257, 300, 304
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-30, 30, (rows, cols)))).astype(np.float32)
    x[0, :10] = 0.0
    x[1, :10] = -x[2, :10]
    xt = torch.from_numpy(x)
    ref = planes_cpu(xt, ld)
    out = torch.full((3, rows, ld), float("nan"), dtype=torch.bfloat16, device=DEV)
    out[:, :, cols:] = 0
    nn.mlp_op_split3(rows, cols, xt.to(DEV).data_ptr(), cols, out.data_ptr(), ld, _stream())
    torch.cuda.synchronize()
    got = out.cpu()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert np.array_equal(from_planes(got, cols), x.astype(np.float64))


FWD = [
    (nn.ACT_RELU, 64, 256, 784),
    (nn.ACT_RELU, 4096, 256, 784),
    (nn.ACT_RELU, 4096, 128, 256),
    (nn.ACT_RELU, 300, 136, 200),       # ragged M, N and K
    (nn.ACT_NONE, 130, 24, 72),
    (nn.ACT_GELU_TANH, 200, 256, 128),  # forward only: GELU applied to the fp32 sum
]


@pytest.mark.parametrize("act,M,N,K", FWD)
def test_x3_linear_act(act, M, N, K):
    X = synth.make_normal((M, K), 1.0, 411, M, N, K)
    if act == nn.ACT_RELU:
        X = torch.relu(X)                 # a hidden layer's input: same-sign terms
    Wt = synth.make_normal((N, K), math.sqrt(2.0 / K), 412, M, N, K)
    b = synth.make_normal((N,), 0.3, 413, M, N, K)
    ldh = (N + 7) // 8 * 8
    Xp, Wp = planes_cpu(X, K).to(DEV), planes_cpu(Wt, K).to(DEV)
    H = torch.full((3, M, ldh), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nn.mlp_op_linear_act(nn.F32X3, act, M, N, K, Xp.data_ptr(), K, Wp.data_ptr(), K, b.to(DEV).data_ptr(),
                         H.data_ptr(), ldh, None, ldh, err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    x64, w64, b64 = to64(X), to64(Wt), to64(b)
    ref = om.act_forward(om.linear(x64, w64, b64), act)
    absum = np.abs(x64) @ np.abs(w64).T + np.abs(b64)
    assert_close_gemm(from_planes(H.cpu(), N), ref, 1.13 * absum, K, False, "H", DROPPED * 1.13 * absum)


DGRAD = [
    (nn.ACT_RELU, 64, 128, 256),
    (nn.ACT_RELU, 4096, 128, 256),      # CTA pairs (four K stages)
    (nn.ACT_RELU, 4096, 256, 128),      # two K stages: one CTA per tile
    (nn.ACT_RELU, 300, 40, 136),
    (nn.ACT_NONE, 130, 256, 784),
]


@pytest.mark.parametrize("act,M,N,K", DGRAD)
def test_x3_dgrad(act, M, N, K):
    """dX[M,K] = (dY[M,N] W[N,K]) * relu'(S), S read from its hi plane."""
    ldy = (N + 7) // 8 * 8
    dY = synth.make_normal((M, N), 1e-3, 421, M, N, K)
    Wt = synth.make_normal((N, K), math.sqrt(2.0 / K), 422, M, N, K)
    S = torch.relu(synth.make_normal((M, K), 1.0, 423, M, N, K))
    dYp, Wp, Sp = planes_cpu(dY, ldy).to(DEV), planes_cpu(Wt, K).to(DEV), planes_cpu(S, K).to(DEV)
    dX = torch.full((3, M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nn.mlp_op_dgrad(nn.F32X3, act, M, N, K, dYp.data_ptr(), ldy, Wp.data_ptr(), K, Sp.data_ptr(), K, dX.data_ptr(),
                    K, err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    dy64, w64, s64 = to64(dY), to64(Wt), to64(S)
    fac = (s64 > 0).astype(np.float64) if act == nn.ACT_RELU else np.ones_like(s64)
    ref = (dy64 @ w64) * fac
    absum = (np.abs(dy64) @ np.abs(w64)) * fac
    assert_close_gemm(from_planes(dX.cpu(), K), ref, absum, N, False, "dX", DROPPED * absum)


WGRAD = [
    (256, 784, 64),
    (256, 784, 4096),
    (128, 256, 4096),
    (40, 136, 1000),       # ragged M, N and batch
]


@pytest.mark.parametrize("N,K,B", WGRAD)
def test_x3_wgrad(N, K, B):
    """dW[N,K] = dY[B,N]^T X[B,K], db = column sums of dY, both fp32."""
    ldy = (N + 7) // 8 * 8
    dY = synth.make_normal((B, N), 1e-3, 431, N, K, B)
    X = torch.relu(synth.make_normal((B, K), 1.0, 432, N, K, B))
    dYp, Xp = planes_cpu(dY, ldy).to(DEV), planes_cpu(X, K).to(DEV)
    dW = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
    db = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    wsb = nn.mlp_op_wgrad_workspace_bytes(nn.F32X3, N, K, B)
    ws = torch.empty(max(wsb, 4), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nn.mlp_op_wgrad(nn.F32X3, N, K, B, dYp.data_ptr(), ldy, Xp.data_ptr(), K, dW.data_ptr(), K, db.data_ptr(),
                    ws.data_ptr(), wsb, err.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert err.item() == 0
    dy64, x64 = to64(dY), to64(X)
    absum = np.abs(dy64).T @ np.abs(x64)
    assert_close_gemm(to64(dW), dy64.T @ x64, absum, B, False, "dW", DROPPED * absum)
    absb = np.abs(dy64).sum(0)
    assert_close_gemm(to64(db), dy64.sum(0), absb, B, False, "db", DROPPED * absb)


def test_x3_rejects_gelu_vjp_and_stored_u():
    M, N, K = 128, 64, 64
    buf = torch.zeros(3 * M * 64, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(N, dtype=torch.float32, device=DEV)
    p = buf.data_ptr()
    with pytest.raises(nn.MlpError):
        nn.mlp_op_dgrad(nn.F32X3, nn.ACT_GELU_TANH, M, N, K, p, N, p, K, p, K, p, K, None, _stream())
    with pytest.raises(nn.MlpError):
        nn.mlp_op_linear_act(nn.F32X3, nn.ACT_GELU_TANH, M, N, K, p, K, p, K, b.data_ptr(), p, N, p, N, None,
                             _stream())
