"""mlp_op_wgrad_noalloc: the weight gradient for callers that cannot allocate.

Some callers cannot call cudaMalloc (their device memory belongs to another
allocator, or their loop must not allocate because cudaMalloc/cudaFree can
synchronise the device and fail under memory pressure).  mlp_op_wgrad_noalloc
serves them by keeping its split-K partial sums in a built-in 16 MiB device
array.  These tests call it through the C ABI and check that it gives the
same dW and db as mlp_op_wgrad with a caller-provided workspace, within the
GEMM tolerance the other tests use, on two calls in a row (the second call
reuses the array the first one wrote), and that a shape needing more scratch
than the array holds is refused before anything is enqueued.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from tests.parity import assert_close_gemm, to64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(dtype, N, K, B, seed):
    td = torch.float32 if dtype == nn.F32 else torch.bfloat16
    ldy = (N + 7) // 8 * 8
    dY = synth.make_normal((B, ldy), 1e-3, 91, seed, N, K, B, dtype=td).to(DEV)
    X = synth.make_normal((B, K), 1.0, 92, seed, N, K, B, dtype=td).to(DEV)
    return dY, ldy, X


def _reference(dtype, N, K, B, dY, ldy, X):
    """The existing entry point, with a workspace the test allocates."""
    dW = torch.empty((N, K), dtype=torch.float32, device=DEV)
    db = torch.empty(N, dtype=torch.float32, device=DEV)
    wsb = nn.mlp_op_wgrad_workspace_bytes(dtype, N, K, B)
    ws = torch.empty(max(wsb, 4), dtype=torch.uint8, device=DEV)
    nn.mlp_op_wgrad(dtype, N, K, B, dY.data_ptr(), ldy, X.data_ptr(), K, dW.data_ptr(), K, db.data_ptr(),
                    ws.data_ptr(), wsb, None, torch.cuda.current_stream().cuda_stream)
    return dW, db


@pytest.mark.parametrize("dtype,N,K,B", [
    (nn.BF16, 512, 512, 4096),    # tensor-core path, split over the batch
    (nn.F32, 256, 784, 4096),     # FFMA path, split over the batch
    (nn.BF16, 100, 512, 1000),    # ragged batch, small split
])
def test_noalloc_matches_wgrad_on_two_calls(dtype, N, K, B):
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dY, ldy, X = _inputs(dtype, N, K, B, call)
        want_dW, want_db = _reference(dtype, N, K, B, dY, ldy, X)
        dW = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
        db = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        nn.mlp_op_wgrad_noalloc(dtype, N, K, B, dY.data_ptr(), ldy, X.data_ptr(), K, dW.data_ptr(), K,
                                db.data_ptr(), err.data_ptr(), stream)
        torch.cuda.synchronize()
        assert err.item() == 0
        dy64, x64 = to64(dY)[:, :N], to64(X)
        absum = np.abs(dy64).T @ np.abs(x64)
        # against the existing entry point, within the GEMM tolerance
        assert_close_gemm(to64(dW), to64(want_dW), absum, B, False, f"dW call {call}")
        assert_close_gemm(to64(db), to64(want_db), np.abs(dy64).sum(0), B, False, f"db call {call}")
        # and against the oracle's definition dW = dY^T X
        assert_close_gemm(to64(dW), dy64.T @ x64, absum, B, False, f"dW vs definition, call {call}")


def _planes(x: torch.Tensor, ld: int) -> torch.Tensor:
    """[3, rows, ld] bf16 planes hi, mid, lo of an fp32 CPU matrix (the
    MLP_F32X3 operand encoding), columns beyond the matrix zero."""
    rows, cols = x.shape
    hi = x.to(torch.bfloat16)
    r = x - hi.float()
    mid = r.to(torch.bfloat16)
    out = torch.zeros((3, rows, ld), dtype=torch.bfloat16)
    out[0, :, :cols], out[1, :, :cols], out[2, :, :cols] = hi, mid, (r - mid.float()).to(torch.bfloat16)
    return out


def test_noalloc_fp32_planes_match_wgrad_on_two_calls():
    """fp32 operands given as three bf16 planes (MLP_F32X3), split over the
    batch: the same dW and db as mlp_op_wgrad on two calls in a row."""
    N, K, B = 256, 784, 4096
    ldy = N
    stream = torch.cuda.current_stream().cuda_stream
    assert nn.mlp_op_wgrad_workspace_bytes(nn.F32X3, N, K, B) > 0
    for call in range(2):
        dY = synth.make_normal((B, N), 1e-3, 93, call)
        X = torch.relu(synth.make_normal((B, K), 1.0, 94, call))
        dYp, Xp = _planes(dY, ldy).to(DEV), _planes(X, K).to(DEV)
        want_dW, want_db = _reference(nn.F32X3, N, K, B, dYp, ldy, Xp)
        dW = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
        db = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        nn.mlp_op_wgrad_noalloc(nn.F32X3, N, K, B, dYp.data_ptr(), ldy, Xp.data_ptr(), K, dW.data_ptr(), K,
                                db.data_ptr(), err.data_ptr(), stream)
        torch.cuda.synchronize()
        assert err.item() == 0
        dy64, x64 = to64(dY), to64(X)
        absum = np.abs(dy64).T @ np.abs(x64)
        # same kernels, same split policy: the results agree within the GEMM bound
        assert_close_gemm(to64(dW), to64(want_dW), absum, B, False, f"dW call {call}")
        assert_close_gemm(to64(db), to64(want_db), np.abs(dy64).sum(0), B, False, f"db call {call}")
        # against dY^T X, allowing the three plane products the kernels leave out
        assert_close_gemm(to64(dW), dy64.T @ x64, absum, B, False, f"dW vs definition, call {call}",
                          2.0 ** -22 * absum)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 1024 x 2048 over 65536 rows splits the batch in two: 16.8 MB > 16 MiB
    N, K, B = 1024, 2048, 65536
    need = nn.mlp_op_wgrad_workspace_bytes(nn.BF16, N, K, B)
    assert need > 16 << 20
    dY = torch.zeros((B, N), dtype=torch.bfloat16, device=DEV)
    X = torch.zeros((B, K), dtype=torch.bfloat16, device=DEV)
    dW = torch.empty((N, K), dtype=torch.float32, device=DEV)
    with pytest.raises(nn.MlpError) as e:
        nn.mlp_op_wgrad_noalloc(nn.BF16, N, K, B, dY.data_ptr(), N, X.data_ptr(), K, dW.data_ptr(), K, None, None,
                                torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 2 and "scratch" in str(e.value)
