"""Free-running trajectories over each workload's configured number of steps,
at full batch, against the oracle's stored trajectories
(tests/golden/trajectories_<workload>.npz, written by make_trajectories.py
from the CPU oracle alone).  Every trajectory runs as ONE CUDA-graph launch
of all its steps (mlp_train_steps), as the deep narrow net's configuration
asks (50 steps in one graph).

What is asserted, per step and per tensor:
  * bf16 workloads: every step's loss within 2e-2 of the oracle's
    exact-rounding mode (the stated bound), strictly.
  * the loss within max(stated |L*|, 3 x the spread of the oracle's own
    perturbed runs) of the oracle (fp32 stated: 1e-4 relative).
  * parameters after the last step, on each tensor's sampled elements: the
    rms deviation and the fraction of elements beyond the stated bound
    (bf16: 3e-2 of the tensor's largest oracle update; fp32: 1e-4 of
    max(|p|, lr)) no more than 3x those of the oracle's perturbed runs on the
    same elements, plus small floors.
The stated element-wise parameter bound itself is reported, not asserted,
for trajectories: the oracle re-run with every product perturbed at fp32
accumulation size misses it on a sizeable fraction of elements
(ens_frac in the stored files), because AdamW's sign-like early steps turn a
gradient whose sign rounding decides into a 2 lr difference that later steps
do not undo.  Each kernel's own arithmetic is instead checked tightly and
without exemptions by a traced step taken right after the trajectory, at
step count + 1 (bias corrections and moments of a late step), layer by
layer as in test_gpu_fullstep.py.

Set MLP_PARITY_REPORT_DIR to a directory to receive one JSON report per
workload (losses, per-tensor deviations, stated-bound results).
"""
import json
import os

import numpy as np
import pytest
import torch

import neural_net_step_gb300 as nn
import synth
from tests import parity as P
from tests.golden import make_trajectories as mk
from tests.test_gpu_fullstep import make_model, traced_step_check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
W = synth.WORKLOADS
CASES = ["mnist_mlp_b4096", "cifar_mlp_b8192", "lm_block_t16384", "deep_narrow_b65536"]


def load(name):
    path = os.path.join(os.path.dirname(mk.__file__), f"trajectories_{name}.npz")
    if not os.path.exists(path):
        pytest.fail(f"{path} is missing: run python tests/golden/make_trajectories.py {name}")
    d = np.load(path)
    if str(d["source_hash"]) != mk.source_hash():
        pytest.fail(f"{path} was written by another version of the oracle or the input generators: "
                    f"rerun python tests/golden/make_trajectories.py {name}")
    return d


def write_report(name, rep):
    out = os.environ.get("MLP_PARITY_REPORT_DIR")
    if not out:
        return
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(out, f"parity_{name}.json"), "w") as f:
        json.dump(rep, f, indent=1)


@pytest.mark.parametrize("name", CASES)
def test_configured_trajectory_in_one_graph(name):
    w = W[name]
    d = load(name)
    bf16 = w.dtype == synth.BF16
    stated = mk.stated(w)
    params0 = synth.make_params(w)
    p0 = [P.to64(p) for p in params0]
    bl = P.batches(w, w.steps)
    m = make_model(w, params0)
    hyper = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.wd)
    losses = m.train_steps([x.to(DEV) for x, _ in bl], [y.to(DEV) for _, y in bl], **hyper)
    m.check_errors()
    p, step = m.read_flat(nn.PLANE_P)
    assert step == w.steps
    parts = m.split(p.astype(np.float64))
    gl = losses.cpu().numpy().astype(np.float64)
    rep = {"workload": name, "steps": w.steps, "graph_launches": 1, "oracle_mode": str(d["mode"])}

    # ---- losses ----
    rl = d["losses_ref"]
    spread = np.max(np.abs(d["losses_ens"] - rl), axis=0)
    dev = np.abs(gl - rl)
    rep["loss"] = {"gpu": gl.tolist(), "oracle": rl.tolist(), "ensemble_spread": spread.tolist(),
                   "max_rel_vs_oracle": float(np.max(dev / np.abs(rl)))}
    if bf16:
        ex = d["losses_exact"]
        rel = np.abs(gl - ex) / np.abs(ex)
        rep["loss"]["max_rel_vs_exact_mode"] = float(rel.max())
        rep["loss"]["stated_ok"] = bool(rel.max() <= 2e-2)
    else:
        rep["loss"]["stated_ok"] = bool(np.all(dev <= 1e-4 * np.abs(rl)))
    loss_stated = 2e-2 if bf16 else 1e-4
    tol = np.maximum((1e-3 if bf16 else 1e-4) * np.abs(rl), P.ENSEMBLE_FACTOR * spread)

    # ---- parameters after the last step, sampled ----
    rows, bad = [], []
    lr = P.hyper32(w)[0]
    for i, t in enumerate(parts):
        idx, ref, ens = d[f"idx_{i}"], d[f"ref_{i}"], d[f"ens_{i}"]
        got = t.ravel()[idx]
        sc = np.maximum(np.abs(ref), lr) if not bf16 else np.full(ref.shape, max(float(d["U"][i]), 1e-30))
        dg = np.abs(got - ref) / sc
        de = np.abs(ens - ref[None, :]) / sc[None, :]
        rms_g, frac_g, max_g = float(np.sqrt(np.mean(dg ** 2))), float(np.mean(dg > stated)), float(dg.max())
        rms_e = float(np.max(np.sqrt(np.mean(de ** 2, axis=1))))
        frac_e = float(np.max(np.mean(de > stated, axis=1)))
        ok = rms_g <= P.ENSEMBLE_FACTOR * rms_e + 0.1 * stated and frac_g <= P.ENSEMBLE_FACTOR * frac_e + 1e-3
        row = {"tensor": i, "elements": int(t.size), "sampled": int(idx.size), "U": float(d["U"][i]),
               "gpu_rms": rms_g, "gpu_frac_over_stated": frac_g, "gpu_max_over_stated": max_g / stated,
               "ens_rms_sampled": rms_e, "ens_frac_sampled": frac_e,
               "ens_frac_all_elements": float(np.max(d["ens_frac"][:, i])),
               "ens_max_over_stated_all_elements": float(np.max(d["ens_max"][:, i])) / stated,
               "stated_ok_sampled": bool(max_g <= stated), "ensemble_ok": bool(ok)}
        rows.append(row)
        if not ok:
            bad.append(row)
    rep["params"] = rows
    rep["stated_params_ok"] = all(r["stated_ok_sampled"] for r in rows)
    write_report(name, rep)
    # asserted after the report is written, so that a failure still leaves it
    if bf16:
        assert rep["loss"]["stated_ok"], ("loss vs exact mode", rep["loss"]["max_rel_vs_exact_mode"])
    i = int(np.argmax(dev / tol))
    assert np.all(dev <= tol), (f"step {i}: loss {gl[i]} vs oracle {rl[i]}, spread {spread[i]}, "
                                f"stated {loss_stated}")
    assert not bad, f"parameters outside the oracle ensemble: {bad}"

    # ---- one more step, traced and checked kernel by kernel ----
    if bf16:
        trep, _, _, _ = traced_step_check(w, m, w.steps)
        rep["traced_step"] = {"t": w.steps + 1, **{k: v for k, v in trep.items() if k != "loss"}}
        write_report(name, rep)
    m.close()
