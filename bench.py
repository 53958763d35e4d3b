"""Benchmark of the GB300 MLP training step (one JSON line on rank 0).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole hot path -- LinearAct forward GEMMs,
softmax-CE forward+backward, loss mean, wgrad (+ fused bias gradient) and
dgrad (+ fused activation VJP) GEMMs, one flat AdamW update -- over one batch
of synthetic data, launched as one CUDA-graph replay through the C ABI.
Default workload: the token-level LM block (1024 -> 4096 GELU-tanh -> 1024 ->
32000-way softmax-CE head, bf16 with fp32 master weights, 16384 tokens), the
largest of the five workloads.  `--graph-steps G` launches G consecutive
steps as one CUDA graph (the deep narrow net's configuration captures 50).

Timing: W untimed warm-up steps, then K steps between CUDA events on the
launching stream, bracketed by a barrier and a device synchronize; the step
reads a fresh batch each time from a device-resident pool larger than L2
(129 MB), so no step finds its input in L2.  Under torchrun (N ranks, one
GPU each) the default is data parallelism at the workload's fixed global
batch (strong scaling): each rank steps on its rows, the flat fp32 gradient
plane is summed over the ranks with an NCCL all-reduce between the gradient
step and the update (neural_net_step_gb300.dp), and `value` is the global
batch per step time; `--parallel replicas` runs N independent replicas
instead (weak scaling).  The slowest rank's time counts.

Also reported: `e2e` (the same metric through the C ABI with pinned host
buffers: every step copies its batch host->device and reads the loss back),
`roofline` for the kernel with the largest device time (per-kernel times
from the library's serialised profiling pass, mlp_profile_step), a
per-kernel table, `cpu_baseline` (the CPU oracle timed on a bounded sample
of the same workload on this host), and SM clocks sampled during the timed
region.  `--impl reference` times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train samples/sec per MLP step (fwd+bwd+AdamW), 1 GB300; % of step roofline"
L2_BYTES = 129 * 1024 * 1024
SMS, FP32_LANES, SM_MAX_GHZ = 152, 128, 2.07
FP32_FFMA_PEAK_TFLOPS = SMS * FP32_LANES * 2 * SM_MAX_GHZ / 1e3   # 80.5 TFLOP/s, derived


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# Algorithmic work of each kernel of the step (the order the library plans it)
# ---------------------------------------------------------------------------
def layer_work(w, kind, l, x3=False):
    """(flops, algorithmic bytes) of one kernel of the step.  x3: the fp32
    model keeps its weights as three bf16 planes, which the update writes."""
    B, es = w.batch, (4 if w.dtype == 0 else 2)
    d, L = w.dims, w.n_layers
    if kind in ("fwd", "wgrad", "dgrad"):
        K, N = d[l], d[l + 1]
        if kind == "fwd":
            gelu_u = es * B * N if (l < L - 1 and w.acts[l] == 2) else 0
            return 2 * B * K * N, es * (B * K + N * K + B * N) + 4 * N + gelu_u
        if kind == "wgrad":
            return 2 * B * K * N, es * (B * N + B * K) + 4 * (N * K + N)
        return 2 * B * K * N, es * (B * N + N * K + 2 * B * K)
    C = d[L]
    if kind == "fwd_head":   # the forward GEMM (writing dY in place of h) + the output layer's FFMA work
        K, N, C = d[l], d[l + 1], d[L]
        return 2 * B * K * N + 3 * 2 * B * N * C, es * (B * K + N * K + B * N) + 4 * N + 4 * (C * N + C)
    if kind == "head":   # output layer fwd + CE + dgrad + wgrad in one pass over h
        K = d[L - 1]
        return 3 * 2 * B * K * C, es * 3 * B * K + 4 * B + 4 * (C * K + C)
    if kind == "ce":
        return 0, 2 * es * B * C + 8 * B
    if kind == "mse":   # read z and fp32 targets, write dz and the row sums
        return 0, 2 * es * B * C + 4 * B * C + 4 * B
    if kind == "loss_mean":
        return 0, 4 * B
    w16 = 2 if w.dtype == 1 else (6 if x3 else 0)   # bf16 weight copy (planes) written by the update
    if kind in ("adamw", "adam_l2"):   # read p, g, m, v; write p, m, v
        return 0, w.n_params() * (28 + w16)
    if kind == "sgd":                  # read p, g, m; write p, m
        return 0, w.n_params() * (20 + w16)
    if kind == "grad_norm":            # read g
        return 0, w.n_params() * 4
    if kind == "split3":   # fp32 input -> three bf16 planes (read 4 B, write 6 B per element)
        return 0, 10 * B * d[0]
    return 0, 0


# fp32 GEMMs on the tensor cores run six bf16 plane products per fp32
# product: their ceiling is the bf16 peak / 6.
X3_PRODUCTS = 6


def peak_source(peaks, top, w):
    if top["bound"] == "alu":
        how = "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz"
    elif top["bound"] == "tensor" and w.dtype == 0:
        how = "MEASURED_PEAKS.json bf16 burst / 6: fp32 operands as three bf16 planes, six products"
    else:
        how = "MEASURED_PEAKS.json burst"
    return f"{peaks['source']} ({how})"


def attach_work(w, prof):
    """Pair each profiled launch (in plan order) with its algorithmic work."""
    rows, fwd_l, bwd_l = [], 0, w.n_layers - 1
    x3 = any(name == "split3" for name, _ in prof)
    for name, ms in prof:
        if name.endswith("_fwd"):
            kind, l = "fwd", fwd_l
            fwd_l += 1
        elif name.endswith("_fwd_head"):   # last hidden layer's forward with the output layer in its epilogue
            kind, l = "fwd_head", fwd_l
            fwd_l += 1
            bwd_l = w.n_layers - 2
        elif name == "head_ce":
            kind, l = "head", w.n_layers - 1
            bwd_l = w.n_layers - 2
        elif name == "softmax_ce":
            kind, l = "ce", -1
        elif name == "mse":
            kind, l = "mse", -1
        elif name == "loss_mean":
            kind, l = "loss_mean", -1
        elif name.endswith("_wgrad"):
            kind, l = "wgrad", bwd_l
        elif name.endswith("_dgrad"):
            kind, l = "dgrad", bwd_l
            bwd_l -= 1
        elif name == "split_reduce":
            kind, l = "split_reduce", rows[-1]["layer"]
        elif name.endswith("_flat"):   # adamw_flat, adam_l2_flat, sgd_flat
            kind, l = name[:-len("_flat")], -1
        else:
            kind, l = name, -1
        fl, by = layer_work(w, kind, l, x3)
        rows.append({"kernel": name, "kind": kind, "layer": l, "ms": ms, "flops": fl, "bytes": by})
    return rows


def roofline_rows(w, rows, peaks):
    """Per kernel: bound, achieved, peak, fraction; and the step roofline."""
    t_roof = 0.0
    for r in rows:
        sec = max(r["ms"], 1e-9) / 1e3
        if r["flops"] and r["kind"] != "head":
            if w.dtype == 0 and r["kernel"].startswith("tc_"):
                bound, peak, unit = "tensor", peaks["bf16_tflops"] / X3_PRODUCTS, "TFLOP/s"
            elif w.dtype == 0:
                bound, peak, unit = "alu", FP32_FFMA_PEAK_TFLOPS, "TFLOP/s"
            else:
                bound, peak, unit = "tensor", peaks["bf16_tflops"], "TFLOP/s"
            ach = r["flops"] / sec / 1e12
            t = max(r["flops"] / (peak * 1e12), r["bytes"] / (peaks["hbm_gbs"] * 1e9))
        else:
            bound, peak, unit = "hbm", peaks["hbm_gbs"], "GB/s"
            ach = r["bytes"] / sec / 1e9
            t = r["bytes"] / (peaks["hbm_gbs"] * 1e9)
        r.update(bound=bound, achieved=ach, peak=peak, unit=unit, frac=ach / peak, t_roof_ms=t * 1e3)
        t_roof += t
    return t_roof * 1e3


# Sources of the kernels and of their launch planning; the model runtime
# (graph building, host-input copies) does not change what a kernel does.
HOST_ONLY_SOURCES = ("model.cu", "noalloc.cu")


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and whitespace: what a kernel is
    made of (a comment edit leaves the counters taken on it valid)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "neural_net_step_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f in HOST_ONLY_SOURCES:
            continue
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update((f + _code_only(fh.read())).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` (name and layer, e.g.
    "tc_gemm_fwd:L1") on `workload` from the committed ncu summary, or None
    when absent or when the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("source_hash") != source_hash():
        return None
    return t.get("kernels", {}).get(f"{workload}:{kernel}")


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.file:
            return None
        try:
            with open(self.file.name) as f:
                lines = [l.strip().split(",") for l in f if l.strip()]
            os.unlink(self.file.name)
        except Exception:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in lines:
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
                for n, v in zip(names, p[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_rows(w, budget_s=1.0):
    """Rows per oracle step so that one step costs about budget_s of CPU
    (fp64 at an assumed ~50 GFLOP/s, refined by measurement)."""
    flops_per_row = w.gemm_flops() / w.batch
    return int(max(64, min(w.batch, budget_s * 50e9 / flops_per_row)))


class OracleRunner:
    """The CPU oracle, as it stands, stepping on a bounded row sample."""

    def __init__(self, w, optim="adamw", max_norm=0.0, loss="ce"):
        import numpy as np
        import synth
        from oracle import mlp_oracle as om
        self.np, self.om, self.w = np, om, w
        self.rows = oracle_sample_rows(w)
        self.params = [p.numpy().astype(np.float64) for p in synth.make_params(w)]
        self.m = [np.zeros_like(p) for p in self.params]
        self.v = [np.zeros_like(p) for p in self.params]
        self.mode = "fp64" if w.dtype == 0 else "bf16_mirror"
        self.hyper = tuple(float(np.float32(a)) for a in (w.lr, w.beta1, w.beta2, w.eps, w.wd))
        self.optim, self.max_norm, self.loss = optim, float(np.float32(max_norm)), loss
        self.batches = []
        for s in range(4):
            x, y = synth.make_batch(w, s)
            y = (synth.make_targets(w, s)[:self.rows].numpy().astype(np.float64) if loss == "mse"
                 else y[:self.rows].numpy().astype(np.int64))
            self.batches.append((x[:self.rows].float().numpy().astype(np.float64), y))
        self.t = 0

    def step(self) -> float:
        x, y = self.batches[self.t % 4]
        t0 = time.perf_counter()
        _, self.params, self.m, self.v, _, _ = self.om.train_step(self.params, self.m, self.v, self.t + 1, x, y,
                                                                  self.w.acts, *self.hyper, mode=self.mode,
                                                                  optim=self.optim, max_norm=self.max_norm,
                                                                  loss=self.loss)
        self.t += 1
        return time.perf_counter() - t0

    def sample(self) -> str:
        return (f"oracle steps (numpy fp64, {self.mode} mode) on {self.rows} of {self.w.batch} rows of the "
                f"{self.w.name} workload; {blas_threads()} BLAS threads on {os.cpu_count()} host cores")


def blas_threads() -> int:
    """Threads the oracle's BLAS actually uses: threadpoolctl where installed,
    else the thread-count variables OpenBLAS reads (torchrun sets
    OMP_NUM_THREADS=1 for its ranks), else every host core."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit() and int(v) > 0:
            return int(v)
    return os.cpu_count() or 1


def time_oracle(w, target_s=10.0, optim="adamw", max_norm=0.0, loss="ce"):
    r = OracleRunner(w, optim, max_norm, loss)
    el, steps = 0.0, 0
    while el < target_s:
        el += r.step()
        steps += 1
    return {"value": r.rows * steps / el, "unit": "samples/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{steps} " + r.sample()}


# ---------------------------------------------------------------------------
# Main
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    r = OracleRunner(w, args.optim, args.max_grad_norm, args.loss)
    for _ in range(args.warmup):
        r.step()
    t_all = sum(r.step() for _ in range(args.steps))
    value = r.rows * args.steps / t_all
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "samples/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_all / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_of(w, None, args),
            "cpu_baseline": {"value": round(value, 2), "unit": "samples/s", "cores": blas_threads(),
                             "kind": "oracle", "sample": f"each step: one of {args.steps} " + r.sample()},
            "e2e": {"value": round(value, 2), "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


OPTIM_NAMES = {"adamw": "AdamW", "adam": "Adam (L2 in the gradient)", "sgd": "SGD (momentum = beta1, L2)"}


def config_of(w, extra=None, args=None):
    optim = args.optim if args else "adamw"
    opt = (f"{OPTIM_NAMES[optim]} lr={w.lr} momentum={w.beta1} wd={w.wd}" if optim == "sgd" else
           f"{OPTIM_NAMES[optim]} lr={w.lr} betas=({w.beta1},{w.beta2}) eps={w.eps} wd={w.wd}")
    if args and args.max_grad_norm > 0:
        opt += f", global grad-norm clipping at {args.max_grad_norm}"
    mse = bool(args and args.loss == "mse")
    c = {"workload": f"{w.name}: MLP {'-'.join(map(str, w.dims))}, "
                     f"{'fp32' if w.dtype == 0 else 'bf16 + fp32 master'}, batch {w.batch}"
                     + (", MSE loss on fp32 targets" if mse else ""),
         "dims": list(w.dims), "acts": [["none", "relu", "gelu_tanh"][a] for a in w.acts], "global_batch": w.batch,
         "loss": "MSE (element mean, fp32 N(0,1) targets)" if mse else "softmax CE (batch mean)",
         "optimizer": opt,
         "parallelism": "replicas"}
    if extra:
        c.update(extra)
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="lm_block_t16384")
    ap.add_argument("--graph-steps", type=int, default=0,
                    help="steps per CUDA-graph launch (default: the workload's own, 50 for deep_narrow_b65536)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernels", action="store_true", help="include the per-kernel table")
    ap.add_argument("--f32-ffma", action="store_true",
                    help="fp32 models: GEMMs on the FFMA pipes instead of the tensor cores")
    ap.add_argument("--optim", default="adamw", choices=["adamw", "adam", "sgd"],
                    help="update rule (default AdamW)")
    ap.add_argument("--max-grad-norm", type=float, default=0.0, help="> 0: global gradient-norm clipping")
    ap.add_argument("--loss", default="ce", choices=["ce", "mse"], help="softmax CE (default) or MSE")
    ap.add_argument("--parallel", default="dp", choices=["dp", "replicas"],
                    help="N > 1: data parallelism at the fixed global batch (default) or independent replicas")
    ap.add_argument("--gemm-2sm", type=int, default=-1, choices=[-1, 0, 1],
                    help="bf16 forward / dgrad GEMMs on CTA pairs with 2-SM MMAs: -1 library policy, 0 off, 1 on")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (small cases for profiling; not a bench line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import synth
    w = synth.WORKLOADS[args.workload]
    if args.batch > 0:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, w, world, rank)

    import torch
    import neural_net_step_gb300 as nn
    from neural_net_step_gb300 import build as nbuild
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    if not os.path.exists(nn.LIB_PATH):
        nbuild.build()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))
        pg = dist

    peaks = load_peaks()
    dp_mode = world > 1 and args.parallel == "dp"
    from neural_net_step_gb300.dp import DataParallel, shard_rows
    lo, hi = shard_rows(w.batch, world, rank) if dp_mode else (0, w.batch)
    B_local = hi - lo
    # data parallel: every rank starts from the same parameters (same seed,
    # then rank 0's broadcast); replicas: one seed per rank
    model = nn.Model(w.dims, w.acts, nn.ACT_RELU, w.dtype, seed=w.seed + (0 if dp_mode else rank), batch=B_local,
                     device=local)
    if w.dtype == 0:
        model.set_option(nn.OPT_F32_TENSOR_CORES, 0 if args.f32_ffma else 1)
    model.set_optimizer({"adamw": nn.OPTIM_ADAMW, "adam": nn.OPTIM_ADAM, "sgd": nn.OPTIM_SGD}[args.optim],
                        args.max_grad_norm)
    model.set_option(nn.OPT_GEMM_2SM, args.gemm_2sm)
    mse = args.loss == "mse"
    if mse:
        model.set_loss(nn.LOSS_MSE)
    gemm_mode = None if w.dtype != 0 else (
        "FFMA" if args.f32_ffma or mse else
        "tensor cores, fp32 operands as three bf16 planes (6 products, fp32 accumulate)")
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    dp = None
    if dp_mode:
        dp = DataParallel(model, w.batch)
        dp.broadcast_params(0)

    # device-resident batch pool larger than L2 (data parallel: every rank
    # draws the same global batches and keeps its own rows)
    x0, y0 = synth.make_batch(w, 0)
    per = x0.numel() * x0.element_size() + (w.batch * w.n_classes if args.loss == "mse" else y0.numel()) * 4
    n_pool = max(4, min(64, math.ceil(1.5 * L2_BYTES / per)))
    n_gen = min(n_pool, 8)
    seed_off = 0 if dp_mode else 1000 * rank
    gen = [synth.make_batch(w, s + seed_off) for s in range(n_gen)]
    if mse:   # regression targets in place of the labels
        gen = [(x, synth.make_targets(w, s + seed_off)) for s, (x, _) in enumerate(gen)]
    if dp_mode:
        gen = [(x[lo:hi].contiguous(), y[lo:hi].contiguous()) for x, y in gen]
    xs, ys = [], []
    for i in range(n_pool):
        x, y = gen[i % n_gen]
        if i >= n_gen:   # distinct bytes for every pool slot: roll the rows
            x, y = torch.roll(x, i, 0), torch.roll(y, i, 0)
        xs.append(x.to(dev))
        ys.append(y.to(dev))
    stream = torch.cuda.current_stream()
    losses = torch.empty(args.steps + args.warmup, dtype=torch.float32, device=dev)

    # (data parallel: one exchange per step, so one step per launch)
    G = 1 if dp_mode else (args.graph_steps if args.graph_steps > 0 else w.graph_steps)

    def step(i, loss_slot):
        if dp_mode:
            dp.step(xs[i % n_pool], ys[i % n_pool], loss=loss_slot, **hyper)
        else:
            model.train_step(xs[i % n_pool], ys[i % n_pool], loss=loss_slot, **hyper)

    def steps(i0, n, loss_slots):
        """Steps i0 .. i0+n-1: one graph launch of n steps (G > 1), else n
        single-step launches."""
        if G > 1:
            model.train_steps([xs[(i0 + j) % n_pool] for j in range(n)], [ys[(i0 + j) % n_pool] for j in range(n)],
                              losses=loss_slots, **hyper)
        else:
            for j in range(n):
                step(i0 + j, loss_slots[j])

    def chunks(n):
        return [G] * (n // G) + ([n % G] if n % G else []) if G > 1 else [n]

    warm_losses = torch.empty(max(G, args.warmup), dtype=torch.float32, device=dev)
    if G > 1:   # every graph shape the timed region launches is built and run at least once
        for c in sorted(set(chunks(args.steps)) | {G}):
            steps(0, c, warm_losses[:c])
    for i in range(args.warmup):
        step(i, warm_losses[i])
    model.check_errors()
    torch.cuda.synchronize()

    # ---- timed region (clocks sampled from ~1 s before it, under the same
    # continuous load, until it ends) ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_end = time.perf_counter() + 1.0
        i = 0
        while time.perf_counter() < t_end:
            steps(i, G, warm_losses[:G])
            i += G
            if i % (16 * G) == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        ev0.record(stream)
        i = 0
        for c in chunks(args.steps):
            steps(args.warmup + i, c, losses[args.warmup + i:args.warmup + i + c])
            i += c
        ev1.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms = ev0.elapsed_time(ev1)
    model.check_errors()
    if pg:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / args.steps
    samples_per_step = w.batch if dp_mode else w.batch * world   # the whole job's rows a step
    value = samples_per_step * args.steps / (ms / 1e3)
    kernels_per_step = model.kernels_per_step()
    clocks = clk.summary()

    # ---- end to end through the C ABI with pinned host buffers: every step
    # copies its batch host->device (mlp_train_step_host: the library's copy
    # stream and two input slots overlap the copies of step i+1 with step i)
    # and reads its loss back device->host ----
    hx = [gen[i % n_gen][0].pin_memory() for i in range(n_gen)]
    hy = [gen[i % n_gen][1].pin_memory() for i in range(n_gen)]
    hl = torch.empty(args.steps + 3, dtype=torch.float32).pin_memory()

    def host_step(i, slot):
        if dp_mode:   # this rank's rows up, the data-parallel step, the global loss down
            xd = hx[i % n_gen].to(dev, non_blocking=True)
            yd = hy[i % n_gen].to(dev, non_blocking=True)
            hl[slot].copy_(dp.step(xd, yd, **hyper), non_blocking=True)
        else:
            model.train_step_host(hx[i % n_gen], hy[i % n_gen], loss=hl[slot:slot + 1], **hyper)

    for i in range(3):
        host_step(i, i)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        host_step(i, 3 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if pg:
        t = torch.tensor([e2e_ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_ms = float(t.item())
    x_bytes = hx[0].numel() * hx[0].element_size()
    e2e = {"value": samples_per_step * args.steps / (e2e_ms / 1e3), "unit": "samples/s",
           "h2d_bytes_per_step": int(x_bytes + hy[0].numel() * hy[0].element_size()), "d2h_bytes_per_step": 4}

    # ---- per-kernel times (serialised profiling pass, same stream) ----
    n_prof = 10
    acc = None
    for i in range(n_prof):
        prof = nn.mlp_profile_step(model.h, xs[i % n_pool].data_ptr(), ys[i % n_pool].data_ptr(), w.lr, w.beta1,
                                   w.beta2, w.eps, w.wd, None, stream.cuda_stream)
        if acc is None:
            acc = [[n, 0.0] for n, _ in prof]
        for a, (_, t) in zip(acc, prof):
            a[1] += t / n_prof
    rows = attach_work(w, [(n, t) for n, t in acc])
    t_roof_ms = roofline_rows(w, rows, peaks)
    top = max(rows, key=lambda r: r["ms"])
    rf = {"bound": top["bound"], "achieved": round(top["achieved"], 3), "peak": top["peak"], "unit": top["unit"],
          "frac": round(top["frac"], 4),
          "traffic": ncu_traffic(f"{top['kernel']}:L{top['layer'] + 1}" if top["layer"] >= 0 else top["kernel"], w.name),
          "kernel": f"{top['kernel']} (layer {top['layer'] + 1})" if top["layer"] >= 0 else top["kernel"],
          "launch_ms": round(top["ms"], 5),
          "peak_source": peak_source(peaks, top, w)}

    line = {"metric": METRIC, "value": round(value, 1), "unit": "samples/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "strong" if dp_mode else "weak", "vs_baseline": None,
            "dtype": "f32" if w.dtype == 0 else "bf16",
            "data": "synthetic",
            "config": config_of(w, {"l2": f"fresh batch per step from a {n_pool}-batch device pool "
                                          f"({n_pool * per / 2**20:.0f} MiB > 129 MB L2)",
                                    "graph": (f"{G} steps per CUDA-graph launch" if G > 1 else
                                              "one CUDA-graph replay per step"),
                                    **({"f32_gemm": gemm_mode} if gemm_mode else {}),
                                    **({"parallelism": f"dp{world}: {B_local} of {w.batch} rows a rank, NCCL sum "
                                                       f"all-reduce of the fp32 gradient plane each step"}
                                       if dp_mode else {})}, args),
            "roofline": rf,
            "step_roofline": {"t_roof_ms": round(t_roof_ms, 5), "measured_ms": round(ms_per_step, 5),
                              "frac": round(t_roof_ms / ms_per_step, 4),
                              "kernels_serial_ms": round(sum(r["ms"] for r in rows), 5)},
            "e2e": {k: (round(v, 1) if isinstance(v, float) else v) for k, v in e2e.items()},
            "gpu_launches": kernels_per_step * args.steps,
            "clocks": clocks}
    if args.kernels:
        line["kernels"] = [{k: (round(v, 5) if isinstance(v, float) else v) for k, v in r.items()} for r in rows]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = time_oracle(w, target_s=10.0, optim=args.optim, max_norm=args.max_grad_norm, loss=args.loss)
        line["cpu_baseline"] = {k: (round(v, 2) if isinstance(v, float) else v) for k, v in cb.items()}
    if rank == 0:
        print(json.dumps(line))
    model.close()
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
