"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/*.h declares, sizes arenas, rejects
bad shapes, and refuses to compute without a GPU (no CPU fallback)."""
import ctypes
import os
import re

import pytest

import neural_net_step_gb300 as nn
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from neural_net_step_gb300 import build
    build.build()
    return nn.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(mlp_\w+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    for n in sorted(names):
        assert hasattr(lib, n), n
        assert n in nn._SIGS, f"{n} has no Python binding"


def test_arena_bytes_for_every_workload(lib):
    for name in synth.WORKLOAD_ORDER:
        w = synth.WORKLOADS[name]
        n = nn.mlp_arena_bytes(list(w.dims), list(w.acts), nn.ACT_RELU, w.dtype, w.batch)
        es = 4 if w.dtype == synth.F32 else 2
        # at least the four fp32 planes and the activations of the forward
        acts = sum(w.batch * d * es for d in w.dims[1:])
        assert n >= 16 * w.n_params() + acts
        assert n % 256 == 0


@pytest.mark.parametrize("dims,dtype", [([784], 0), ([100, 20, 10], 1), ([8, 0, 4], 0)])
def test_bad_shapes_rejected(lib, dims, dtype):
    with pytest.raises(nn.MlpError):
        nn.mlp_arena_bytes(dims, None, nn.ACT_RELU, dtype, 4)


def test_bad_dtype_and_activation_rejected(lib):
    with pytest.raises(nn.MlpError):
        nn.mlp_arena_bytes([8, 8, 4], None, nn.ACT_RELU, 7, 4)
    with pytest.raises(nn.MlpError):
        nn.mlp_arena_bytes([8, 8, 4], [9], nn.ACT_RELU, 0, 4)


def test_no_gpu_means_no_compute(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    dims = (ctypes.c_int64 * 3)(8, 8, 4)
    st = lib.mlp_create(dims, 3, None, 1, 0, 0, 4, ctypes.c_void_p(256), 1 << 20, 0, ctypes.byref(h))
    assert st != 0 and not h.value
    assert nn.mlp_last_error()


def test_every_kernel_takes_one_parameter_block():
    """Launches pass one argument pointer (a kernel's parameter block), so a
    kernel with any other parameter list would read past it: every
    __global__ function takes exactly one `const __grid_constant__` struct."""
    csrc = os.path.join(ROOT, "neural_net_step_gb300", "csrc")
    n = 0
    for f in sorted(os.listdir(csrc)):
        if not f.endswith(".cu"):
            continue
        txt = re.sub(r"//[^\n]*", "", open(os.path.join(csrc, f)).read())
        for m in re.finditer(r"__global__", txt):
            seg = txt[m.end():txt.index("{", m.end())]
            params = seg[seg.rindex("(") + 1:seg.rindex(")")].strip()
            assert re.fullmatch(r"const __grid_constant__ \w+ \w+", params), (f, params)
            n += 1
    assert n >= 15


def test_binding_constants_match_the_headers():
    """Every enumerator the headers declare (activations, dtypes, planes,
    options, update rules, losses, status codes, workspace sizes) has the
    same value in the Python binding."""
    found = {}
    for f in ("mlp.h", "mlp_ops.h"):
        txt = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", f)).read(), flags=re.S)
        for body in re.findall(r"enum\s*\{(.*?)\}", txt, flags=re.S):
            for name, val in re.findall(r"\b(MLP_\w+)\s*=\s*(-?\d+)", body):
                found[name] = int(val)
    assert len(found) >= 30
    for name, val in found.items():
        if name.startswith("MLP_ERR_") or name == "MLP_OK":
            assert nn.STATUS_NAMES[val] == name, name
            continue
        py = name[len("MLP_"):]
        assert getattr(nn, py) == val, (name, val, getattr(nn, py, None))


@pytest.mark.parametrize("M,N,K", [(256, 784, 4096), (128, 256, 4096), (10, 128, 4096), (256, 784, 333),
                                   (1024, 3072, 8192), (512, 512, 65536), (100, 512, 1000)])
def test_plane_wgrad_split_policy(lib, M, N, K):
    """The K splits of a plane-mode (fp32 as bf16 planes) weight gradient,
    read back from the workspace it asks for: at most 16 (the optimizer adds
    16 partials per batch of loads), chunks of 32-row stages that come out
    even, and for layer 1 of the 4096-row MNIST-shaped step ten splits (140
    work units: one wave of 152 SMs)."""
    ws = nn.mlp_op_wgrad_workspace_bytes(nn.F32X3, M, N, K)
    s = 1 if ws == 0 else ws // ((M * N + M) * 4)
    assert ws in (0, s * (M * N + M) * 4)
    kbs = -(-K // 32)
    assert 1 <= s <= 16
    assert -(-kbs // -(-kbs // s)) == s
    if (M, N, K) == (256, 784, 4096):
        assert s == 10
