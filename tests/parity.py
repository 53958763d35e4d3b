"""Shared helpers for GPU-vs-oracle parity tests.

Tolerances (derived from the arithmetic; each is also stated in the design doc):
  * fp32 step (no TF32): loss |L - L*| / |L*| <= 1e-4; every parameter
    |p - p*| / max(|p*|, lr) <= 1e-4 (lr is the scale one AdamW step moves a
    parameter, so the bound stays meaningful where p* crosses zero).
  * bf16 step with fp32 master weights: loss relative error <= 2e-2 against
    the oracle's "bf16" (exact) mode; per tensor, max |p - p*| <= 3e-2 *
    max |p* - p0| against the oracle's "bf16_mirror" mode (the update
    magnitude is the tensor's largest oracle update over the run).
  * single GEMMs: |c - c*| <= 8 sqrt(K) 2^-24 sum_k |a_k b_k| (fp32
    accumulation; a statistical bound, 8x the rms growth of recursive fp32
    summation) plus, for bf16 outputs, half a bf16 ulp of |c*| (2^-8 |c*|).
"""
from __future__ import annotations

import math
from typing import List, Sequence

import numpy as np
import torch

import synth
from oracle import mlp_oracle as om


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def flat(params: Sequence[np.ndarray]) -> np.ndarray:
    return np.concatenate([np.asarray(p, np.float64).ravel() for p in params])


def gemm_tol(absum: np.ndarray, K: int, ref: np.ndarray, bf16_out: bool) -> np.ndarray:
    t = 8.0 * math.sqrt(max(K, 1)) * 2.0 ** -24 * absum
    if bf16_out:
        t = t + 2.0 ** -8 * np.abs(ref)
    return t + 1e-30


def assert_close_gemm(got: np.ndarray, ref: np.ndarray, absum: np.ndarray, K: int, bf16_out: bool, what=""):
    tol = gemm_tol(absum, K, ref, bf16_out)
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}")


def f32_param_error(p: np.ndarray, pref: np.ndarray, lr: float) -> float:
    return float(np.max(np.abs(p - pref) / np.maximum(np.abs(pref), lr)))


def bf16_param_errors(p_list, pref_list, p0_list) -> List[float]:
    """Per tensor: max|p - p*| / max|p* - p0|."""
    out = []
    for p, pr, p0 in zip(p_list, pref_list, p0_list):
        upd = float(np.max(np.abs(pr - p0)))
        out.append(float(np.max(np.abs(p - pr))) / max(upd, 1e-30))
    return out


def oracle_mode(w: synth.Workload, exact: bool = False) -> str:
    if w.dtype == synth.F32:
        return "fp64"
    return "bf16" if exact else "bf16_mirror"


def batches(w: synth.Workload, n: int, batch=None):
    return [synth.make_batch(w, s, batch) for s in range(n)]


def oracle_run(w: synth.Workload, params0, bl, mode: str):
    hyper = (w.lr, w.beta1, w.beta2, w.eps, w.wd)
    xs = [(to64(x), y.numpy().astype(np.int64)) for x, y in bl]
    p0 = [to64(p) for p in params0]
    return om.run_steps(p0, w.acts, xs, hyper, mode=mode)
