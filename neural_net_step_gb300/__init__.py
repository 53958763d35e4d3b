"""Python binding of the GB300 MLP training-step library (libmlpstep.so).

The functions below carry the C ABI's names (include/mlp.h, include/mlp_ops.h)
and only marshal arguments: pointers are passed as integers (device addresses
from torch tensors' data_ptr()), streams as cudaStream_t integers.  Every
step of the path runs in the library's CUDA kernels; there is no CPU path.
`Model` is a small convenience wrapper that lets torch allocate the arena.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmlpstep.so")

MLP_OK = 0
STATUS_NAMES = {0: "MLP_OK", 1: "MLP_ERR_ARG", 2: "MLP_ERR_SHAPE", 3: "MLP_ERR_DTYPE", 4: "MLP_ERR_CUDA",
                5: "MLP_ERR_LABEL_RANGE", 6: "MLP_ERR_NONFINITE", 7: "MLP_ERR_STATE", 8: "MLP_ERR_TIMEOUT"}
ACT_NONE, ACT_RELU, ACT_GELU_TANH = 0, 1, 2
F32, BF16 = 0, 1
F32X3 = 2   # op-level GEMM operands: fp32 as three bf16 planes [3][rows][ld]
PLANE_P, PLANE_G, PLANE_M, PLANE_V = 0, 1, 2, 3
OPTIM_ADAMW, OPTIM_ADAM, OPTIM_SGD = 0, 1, 2
OPTIM_WS_FLOATS = 1216   # op-level clipping workspace (floats)
LOSS_CE, LOSS_MSE = 0, 1


class MlpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None
_c = ctypes
_P, _I64, _I32, _F, _SZ = _c.c_void_p, _c.c_int64, _c.c_int, _c.c_float, _c.c_size_t

_SIGS = {
    "mlp_arena_bytes": (_SZ, [_c.POINTER(_I64), _I32, _c.POINTER(_I32), _I32, _I32, _I64]),
    "mlp_create": (_I32, [_c.POINTER(_I64), _I32, _c.POINTER(_I32), _I32, _I32, _c.c_uint64, _I64, _P, _SZ, _I32,
                          _c.POINTER(_P)]),
    "mlp_forward": (_I32, [_P, _P, _P, _P, _P]),
    "mlp_train_step": (_I32, [_P, _P, _P, _F, _F, _F, _F, _F, _P, _P]),
    "mlp_train_step_host": (_I32, [_P, _P, _P, _F, _F, _F, _F, _F, _P, _P]),
    "mlp_train_steps": (_I32, [_P, _I32, _c.POINTER(_P), _c.POINTER(_P), _F, _F, _F, _F, _F, _P, _P]),
    "mlp_set_graph_mode": (_I32, [_P, _I32]),
    "mlp_set_option": (_I32, [_P, _I32, _I64]),
    "mlp_set_optimizer": (_I32, [_P, _I32, _F]),
    "mlp_read_grad_norm": (_I32, [_P, _c.POINTER(_F)]),
    "mlp_set_loss": (_I32, [_P, _I32]),
    "mlp_num_params": (_I64, [_P]),
    "mlp_num_layers": (_I32, [_P]),
    "mlp_read_params": (_I32, [_P, _I32, _P, _SZ, _c.POINTER(_I64)]),
    "mlp_write_params": (_I32, [_P, _I32, _P, _SZ, _I64]),
    "mlp_check_errors": (_I32, [_P, _P]),
    "mlp_kernels_per_step": (_I32, [_P]),
    "mlp_profile_step": (_I32, [_P, _P, _P, _F, _F, _F, _F, _F, _P, _P, _c.POINTER(_F), _c.POINTER(_c.c_char_p),
                                _I32, _c.POINTER(_I32)]),
    "mlp_profile_forward": (_I32, [_P, _P, _P, _P, _P, _c.POINTER(_F), _c.POINTER(_c.c_char_p), _I32,
                                   _c.POINTER(_I32)]),
    "mlp_grad_step": (_I32, [_P, _P, _P, _I64, _P, _P]),
    "mlp_apply_update": (_I32, [_P, _F, _F, _F, _F, _F, _P]),
    "mlp_grad_buffer": (_I32, [_P, _c.POINTER(_P), _c.POINTER(_I64)]),
    "mlp_trace_step": (_I32, [_P, _P, _P, _F, _F, _F, _F, _F, _P, _P, _SZ, _P, _I32, _c.POINTER(_I32),
                              _c.POINTER(_SZ), _P]),
    "mlp_last_error": (_c.c_char_p, []),
    "mlp_destroy": (None, [_P]),
    "mlp_op_linear_act": (_I32, [_I32, _I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _P, _P]),
    "mlp_op_dgrad": (_I32, [_I32, _I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _P]),
    "mlp_op_wgrad_workspace_bytes": (_SZ, [_I32, _I64, _I64, _I64]),
    "mlp_op_wgrad": (_I32, [_I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "mlp_op_wgrad_noalloc": (_I32, [_I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _P, _P]),
    "mlp_op_split3": (_I32, [_I64, _I64, _P, _I64, _P, _I64, _P]),
    "mlp_op_softmax_ce": (_I32, [_I32, _I64, _I64, _P, _I64, _P, _F, _P, _I64, _P, _P, _P]),
    "mlp_op_linear_ce_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "mlp_op_linear_ce": (_I32, [_I64, _I64, _I64, _P, _I64, _P, _P, _P, _I32, _P, _I64, _P, _I64, _P, _P, _I64, _P,
                                _I64, _P, _P, _SZ, _P, _P]),
    "mlp_op_mse": (_I32, [_I32, _I64, _I64, _P, _I64, _P, _I64, _F, _P, _I64, _P, _P]),
    "mlp_op_loss_mean": (_I32, [_I64, _P, _P, _P, _P]),
    "mlp_op_adamw": (_I32, [_I64, _P, _P, _P, _P, _P, _I64, _F, _F, _F, _F, _F, _P]),
    "mlp_op_optim": (_I32, [_I32, _I64, _P, _P, _P, _P, _P, _I64, _F, _F, _F, _F, _F, _F, _P, _P, _P]),
    "mlp_op_argmax": (_I32, [_I32, _I64, _I64, _P, _I64, _P, _P]),
    "mlp_op_wait_timeout_check": (_I32, [_c.c_uint64, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """Load libmlpstep.so (built by neural_net_step_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with neural_net_step_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def mlp_last_error() -> str:
    return (lib().mlp_last_error() or b"").decode()


def _check(st: int) -> None:
    if st != MLP_OK:
        raise MlpError(st, mlp_last_error())


def _i64arr(v: Sequence[int]):
    return (_I64 * len(v))(*v)


def _i32arr(v: Optional[Sequence[int]]):
    return None if v is None else (_I32 * len(v))(*v)


# ---- model ---------------------------------------------------------------
def mlp_arena_bytes(dims, acts, act, dtype, batch) -> int:
    n = lib().mlp_arena_bytes(_i64arr(dims), len(dims), _i32arr(acts), act, dtype, batch)
    if n == 0:
        raise MlpError(1, mlp_last_error())
    return n


def mlp_create(dims, acts, act, dtype, seed, batch, arena_ptr, arena_bytes, device) -> int:
    h = _P()
    _check(lib().mlp_create(_i64arr(dims), len(dims), _i32arr(acts), act, dtype, seed, batch, arena_ptr,
                            arena_bytes, device, ctypes.byref(h)))
    return h.value


def mlp_forward(h, x_ptr, logits_ptr, argmax_ptr, stream) -> None:
    _check(lib().mlp_forward(h, x_ptr, logits_ptr, argmax_ptr, stream))


def mlp_train_step(h, x_ptr, labels_ptr, lr, beta1, beta2, eps, wd, loss_ptr, stream) -> None:
    _check(lib().mlp_train_step(h, x_ptr, labels_ptr, lr, beta1, beta2, eps, wd, loss_ptr, stream))


def mlp_train_step_host(h, x_host_ptr, labels_host_ptr, lr, beta1, beta2, eps, wd, loss_host_ptr, stream) -> None:
    _check(lib().mlp_train_step_host(h, x_host_ptr, labels_host_ptr, lr, beta1, beta2, eps, wd, loss_host_ptr, stream))


def mlp_grad_step(h, x_ptr, y_ptr, global_batch, loss_ptr, stream) -> None:
    _check(lib().mlp_grad_step(h, x_ptr, y_ptr, global_batch, loss_ptr, stream))


def mlp_apply_update(h, lr, beta1, beta2, eps, wd, stream) -> None:
    _check(lib().mlp_apply_update(h, lr, beta1, beta2, eps, wd, stream))


def mlp_grad_buffer(h):
    """(device address, length in floats) of the gradient plane G."""
    ptr, n = _P(), _I64(0)
    _check(lib().mlp_grad_buffer(h, ctypes.byref(ptr), ctypes.byref(n)))
    return ptr.value, n.value


def mlp_train_steps(h, x_ptrs, label_ptrs, lr, beta1, beta2, eps, wd, losses_ptr, stream) -> None:
    n = len(x_ptrs)
    xs = (_P * n)(*x_ptrs)
    ys = (_P * n)(*label_ptrs)
    _check(lib().mlp_train_steps(h, n, xs, ys, lr, beta1, beta2, eps, wd, losses_ptr, stream))


def mlp_set_graph_mode(h, enable: bool) -> None:
    _check(lib().mlp_set_graph_mode(h, int(bool(enable))))


OPT_GRAPH, OPT_FUSE_HEAD, OPT_F32_TENSOR_CORES, OPT_PDL, OPT_CE_GEMM, OPT_RELU_BITS, OPT_HEAD_IN_GEMM = 0, 1, 2, 3, 4, 5, 6
OPT_GEMM_2SM = 7


def mlp_set_option(h, option: int, value: int) -> None:
    _check(lib().mlp_set_option(h, option, value))


def mlp_set_optimizer(h, kind: int, max_grad_norm: float = 0.0) -> None:
    _check(lib().mlp_set_optimizer(h, kind, max_grad_norm))


def mlp_set_loss(h, loss: int) -> None:
    _check(lib().mlp_set_loss(h, loss))


def mlp_read_grad_norm(h) -> float:
    out = _F(0.0)
    _check(lib().mlp_read_grad_norm(h, ctypes.byref(out)))
    return out.value


def mlp_num_params(h) -> int:
    return lib().mlp_num_params(h)


def mlp_num_layers(h) -> int:
    return lib().mlp_num_layers(h)


def mlp_kernels_per_step(h) -> int:
    return lib().mlp_kernels_per_step(h)


def mlp_profile_step(h, x_ptr, labels_ptr, lr, beta1, beta2, eps, wd, loss_ptr, stream, max_kernels=256):
    """Returns [(kernel name, device ms), ...] for one serialised step."""
    ms = (_F * max_kernels)()
    names = (_c.c_char_p * max_kernels)()
    n = _I32(0)
    _check(lib().mlp_profile_step(h, x_ptr, labels_ptr, lr, beta1, beta2, eps, wd, loss_ptr, stream, ms, names,
                                  max_kernels, ctypes.byref(n)))
    return [(names[i].decode(), ms[i]) for i in range(min(n.value, max_kernels))]


TRACE_H, TRACE_U, TRACE_Z, TRACE_DZ, TRACE_LOSS_ROWS, TRACE_DY = 0, 1, 2, 3, 4, 5


class TraceEntry(ctypes.Structure):
    """mlp_trace_entry (include/mlp.h)."""
    _fields_ = [("kind", _c.c_int32), ("layer", _c.c_int32), ("launch", _c.c_int32), ("planes", _c.c_int32),
                ("rows", _c.c_int64), ("cols", _c.c_int64), ("ld", _c.c_int64), ("plane_stride", _c.c_int64),
                ("elem_bytes", _c.c_int32), ("reserved", _c.c_int32), ("offset", _c.c_uint64),
                ("bytes", _c.c_uint64)]


def mlp_trace_step(h, x_ptr, y_ptr, lr, beta1, beta2, eps, wd, loss_ptr, trace_ptr, trace_bytes, stream,
                   max_entries=512):
    """Returns ([TraceEntry, ...], bytes needed); with trace_ptr None nothing runs."""
    ents = (TraceEntry * max_entries)()
    n = _I32(0)
    need = _SZ(0)
    _check(lib().mlp_trace_step(h, x_ptr, y_ptr, lr, beta1, beta2, eps, wd, loss_ptr, trace_ptr, trace_bytes, ents,
                                max_entries, ctypes.byref(n), ctypes.byref(need), stream))
    return [ents[i] for i in range(n.value)], need.value


def mlp_profile_forward(h, x_ptr, logits_ptr, argmax_ptr, stream, max_kernels=256):
    """Returns [(kernel name, device ms), ...] of one serialised mlp_forward."""
    ms = (_F * max_kernels)()
    names = (_c.c_char_p * max_kernels)()
    n = _I32(0)
    _check(lib().mlp_profile_forward(h, x_ptr, logits_ptr, argmax_ptr, stream, ms, names, max_kernels,
                                     ctypes.byref(n)))
    return [(names[i].decode(), ms[i]) for i in range(min(n.value, max_kernels))]


def mlp_read_params(h, plane, host_ptr, n) -> int:
    step = _I64(0)
    _check(lib().mlp_read_params(h, plane, host_ptr, n, ctypes.byref(step)))
    return step.value


def mlp_write_params(h, plane, host_ptr, n, step) -> None:
    _check(lib().mlp_write_params(h, plane, host_ptr, n, step))


def mlp_check_errors(h, stream) -> None:
    _check(lib().mlp_check_errors(h, stream))


def mlp_destroy(h) -> None:
    lib().mlp_destroy(h)


# ---- individual operations -------------------------------------------------
def mlp_op_linear_act(dtype, act, M, N, K, X, ldx, W, ldw, b, H, ldh, U, ldu, err, stream) -> None:
    _check(lib().mlp_op_linear_act(dtype, act, M, N, K, X, ldx, W, ldw, b, H, ldh, U, ldu, err, stream))


def mlp_op_dgrad(dtype, act, M, N, K, dY, ldy, W, ldw, S, lds, dX, ldx, err, stream) -> None:
    _check(lib().mlp_op_dgrad(dtype, act, M, N, K, dY, ldy, W, ldw, S, lds, dX, ldx, err, stream))


def mlp_op_wgrad_workspace_bytes(dtype, N, K, B) -> int:
    return lib().mlp_op_wgrad_workspace_bytes(dtype, N, K, B)


def mlp_op_wgrad(dtype, N, K, B, dY, ldy, X, ldx, dW, lddw, db, ws, ws_bytes, err, stream) -> None:
    _check(lib().mlp_op_wgrad(dtype, N, K, B, dY, ldy, X, ldx, dW, lddw, db, ws, ws_bytes, err, stream))


def mlp_op_wgrad_noalloc(dtype, N, K, B, dY, ldy, X, ldx, dW, lddw, db, err, stream) -> None:
    """mlp_op_wgrad for callers that cannot provide a workspace: the split-K
    partial sums live in the library's built-in 16 MiB device array."""
    _check(lib().mlp_op_wgrad_noalloc(dtype, N, K, B, dY, ldy, X, ldx, dW, lddw, db, err, stream))


def mlp_op_split3(rows, cols, X, ldx, P, ldp, stream) -> None:
    _check(lib().mlp_op_split3(rows, cols, X, ldx, P, ldp, stream))


def mlp_op_softmax_ce(dtype, B, C, z, ldz, labels, grad_scale, dz, lddz, loss_rows, err, stream) -> None:
    _check(lib().mlp_op_softmax_ce(dtype, B, C, z, ldz, labels, grad_scale, dz, lddz, loss_rows, err, stream))


def mlp_op_linear_ce_workspace_bytes(B, C, K) -> int:
    return lib().mlp_op_linear_ce_workspace_bytes(B, C, K)


def mlp_op_linear_ce(B, C, K, h, ldh, W, bias, labels, act, aux, ld_aux, z, ldz, loss_rows, dX, ldx, dW, lddw, db,
                     ws, ws_bytes, err, stream) -> None:
    _check(lib().mlp_op_linear_ce(B, C, K, h, ldh, W, bias, labels, act, aux, ld_aux, z, ldz, loss_rows, dX, ldx,
                                  dW, lddw, db, ws, ws_bytes, err, stream))


def mlp_op_mse(dtype, B, C, z, ldz, t, ldt, grad_scale, dz, lddz, loss_rows, stream) -> None:
    _check(lib().mlp_op_mse(dtype, B, C, z, ldz, t, ldt, grad_scale, dz, lddz, loss_rows, stream))


def mlp_op_loss_mean(B, loss_rows, loss, err, stream) -> None:
    _check(lib().mlp_op_loss_mean(B, loss_rows, loss, err, stream))


def mlp_op_adamw(n, p, g, m, v, w16, t, lr, beta1, beta2, eps, wd, stream) -> None:
    _check(lib().mlp_op_adamw(n, p, g, m, v, w16, t, lr, beta1, beta2, eps, wd, stream))


def mlp_op_optim(kind, n, p, g, m, v, w16, t, lr, beta1, beta2, eps, wd, max_norm, ws, norm, stream) -> None:
    _check(lib().mlp_op_optim(kind, n, p, g, m, v, w16, t, lr, beta1, beta2, eps, wd, max_norm, ws, norm, stream))


def mlp_op_wait_timeout_check(limit_ns, err, stream) -> None:
    _check(lib().mlp_op_wait_timeout_check(limit_ns, err, stream))


def mlp_op_argmax(dtype, B, C, z, ldz, out, stream) -> None:
    _check(lib().mlp_op_argmax(dtype, B, C, z, ldz, out, stream))


# ---- convenience wrapper ---------------------------------------------------
class Model:
    """An MLP whose arena is a torch uint8 CUDA tensor.  Inputs are torch CUDA
    tensors (x in the model dtype, labels int32); outputs are torch tensors."""

    def __init__(self, dims: Sequence[int], acts: Optional[Sequence[int]] = None, act: int = ACT_RELU,
                 dtype: int = F32, seed: int = 0, batch: int = 1, device: int = 0):
        import torch
        self.torch = torch
        self.dims = list(dims)
        self.acts = None if acts is None else list(acts)
        self.dtype = dtype
        self.batch = batch
        self.device = device
        nbytes = mlp_arena_bytes(self.dims, self.acts, act, dtype, batch)
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=f"cuda:{device}")
        self.h = mlp_create(self.dims, self.acts, act, dtype, seed, batch, self.arena.data_ptr(), nbytes, device)
        self.n_params = mlp_num_params(self.h)
        self.loss_kind = LOSS_CE

    @property
    def tdtype(self):
        return self.torch.float32 if self.dtype == F32 else self.torch.bfloat16

    def stream(self) -> int:
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def set_graph_mode(self, enable: bool) -> None:
        mlp_set_graph_mode(self.h, enable)

    def set_option(self, option: int, value: int) -> None:
        mlp_set_option(self.h, option, value)

    def set_optimizer(self, kind: int, max_grad_norm: float = 0.0) -> None:
        mlp_set_optimizer(self.h, kind, max_grad_norm)

    def grad_norm(self) -> float:
        return mlp_read_grad_norm(self.h)

    def set_loss(self, loss: int) -> None:
        mlp_set_loss(self.h, loss)
        self.loss_kind = loss

    def _check_y(self, y, on_device: bool) -> None:
        t = self.torch
        assert y.is_cuda == on_device and y.is_contiguous()
        if self.loss_kind == LOSS_MSE:
            assert y.dtype == t.float32 and tuple(y.shape) == (self.batch, self.dims[-1])
        else:
            assert y.dtype == t.int32 and y.numel() == self.batch

    def _check_x(self, x, labels=None):
        t = self.torch
        assert x.is_cuda and x.dtype == self.tdtype and x.is_contiguous() and tuple(x.shape) == (self.batch, self.dims[0])
        if labels is not None:
            self._check_y(labels, True)

    def train_step(self, x, labels, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, loss=None):
        self._check_x(x, labels)
        if loss is None:
            loss = self.torch.empty((), dtype=self.torch.float32, device=x.device)
        mlp_train_step(self.h, x.data_ptr(), labels.data_ptr(), lr, beta1, beta2, eps, wd, loss.data_ptr(),
                       self.stream())
        return loss

    def train_step_host(self, x, labels, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, loss=None):
        """One step on pinned host tensors (copies overlap the previous step);
        `loss` (optional) is a pinned float32 host tensor of one element."""
        t = self.torch
        assert not x.is_cuda and x.dtype == self.tdtype and x.is_contiguous() and tuple(x.shape) == (self.batch, self.dims[0])
        self._check_y(labels, False)
        mlp_train_step_host(self.h, x.data_ptr(), labels.data_ptr(), lr, beta1, beta2, eps, wd,
                            loss.data_ptr() if loss is not None else None, self.stream())

    def train_steps(self, xs, ys, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, losses=None):
        for x, y in zip(xs, ys):
            self._check_x(x, y)
        if losses is None:
            losses = self.torch.empty(len(xs), dtype=self.torch.float32, device=xs[0].device)
        mlp_train_steps(self.h, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], lr, beta1, beta2, eps, wd,
                        losses.data_ptr(), self.stream())
        return losses

    def forward(self, x, want_logits=True, want_argmax=True):
        self._check_x(x)
        t = self.torch
        logits = t.empty((self.batch, self.dims[-1]), dtype=self.tdtype, device=x.device) if want_logits else None
        am = t.empty(self.batch, dtype=t.int32, device=x.device) if want_argmax else None
        mlp_forward(self.h, x.data_ptr(), logits.data_ptr() if logits is not None else None,
                    am.data_ptr() if am is not None else None, self.stream())
        return logits, am

    def grad_step(self, x, labels, global_batch, loss=None):
        """Forward + backward of this shard of a global batch (mlp_grad_step);
        G then holds the shard's gradient of the global mean loss."""
        self._check_x(x, labels)
        if loss is None:
            loss = self.torch.empty((), dtype=self.torch.float32, device=x.device)
        mlp_grad_step(self.h, x.data_ptr(), labels.data_ptr(), global_batch, loss.data_ptr(), self.stream())
        return loss

    def apply_update(self, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0):
        mlp_apply_update(self.h, lr, beta1, beta2, eps, wd, self.stream())

    def grad_tensor(self):
        """G as a float32 CUDA tensor viewing the arena (the all-reduce buffer)."""
        ptr, n = mlp_grad_buffer(self.h)
        off = ptr - self.arena.data_ptr()
        assert 0 <= off and off + 4 * n <= self.arena.numel() and off % 4 == 0
        return self.arena[off:off + 4 * n].view(self.torch.float32)

    def trace_step(self, x, labels, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, loss=None):
        """One traced training step (mlp_trace_step).  Returns (loss, [(entry,
        tensor)]): each tensor a CPU torch tensor [planes, rows, ld] of the
        stored dtype (bf16, or fp32 for 4-byte elements), exactly as stored."""
        t = self.torch
        self._check_x(x, labels)
        if loss is None:
            loss = t.empty((), dtype=t.float32, device=x.device)
        args = (self.h, x.data_ptr(), labels.data_ptr(), lr, beta1, beta2, eps, wd, loss.data_ptr())
        _, need = mlp_trace_step(*args, None, 0, self.stream())
        buf = t.empty(max(need, 256), dtype=t.uint8, device=x.device)
        ents, _ = mlp_trace_step(*args, buf.data_ptr(), buf.numel(), self.stream())
        out = []
        for e in ents:
            raw = buf[e.offset:e.offset + e.bytes].cpu()
            td = t.bfloat16 if e.elem_bytes == 2 else t.float32
            v = raw.view(td)
            full = e.rows * e.ld
            planes = [v[k * e.plane_stride:k * e.plane_stride + full].view(e.rows, e.ld) for k in range(e.planes)]
            out.append((e, t.stack(planes)))
        del buf
        return loss, out

    def read_flat(self, plane: int = PLANE_P):
        import numpy as np
        out = np.empty(self.n_params, dtype=np.float32)
        step = mlp_read_params(self.h, plane, out.ctypes.data, self.n_params)
        return out, step

    def write_flat(self, flat, plane: int = PLANE_P, step: int = 0) -> None:
        import numpy as np
        a = np.ascontiguousarray(flat, dtype=np.float32)
        assert a.size == self.n_params
        mlp_write_params(self.h, plane, a.ctypes.data, self.n_params, step)

    def split(self, flat) -> List:
        """Cut a flat parameter vector into [W1, b1, ..., WL, bL] (views)."""
        out, pos = [], 0
        for l in range(len(self.dims) - 1):
            n, k = self.dims[l + 1], self.dims[l]
            out.append(flat[pos:pos + n * k].reshape(n, k))
            pos += n * k
            out.append(flat[pos:pos + n])
            pos += n
        return out

    def check_errors(self) -> None:
        mlp_check_errors(self.h, self.stream())

    def kernels_per_step(self) -> int:
        return mlp_kernels_per_step(self.h)

    def close(self) -> None:
        if getattr(self, "h", None):
            mlp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
