"""Write trajectories_<workload>.npz: the oracle's training trajectories over
each workload's configured number of steps (100 for the 4096-row fp32 MNIST
net, 20 for the CIFAR net, 10 for the LM block, 50 for the deep narrow net),
computed by the CPU oracle alone (no GPU code) from the seeded initial
parameters and batches of synth/.

Each file holds, for the oracle (fp64 for the fp32 workload, the bf16
mirror-rounding mode for the others):
  losses_ref[t]         the batch loss of every step
  losses_exact[t]       bf16 workloads: the loss in the exact-rounding mode
  losses_ens[j, t]      the same run with every product perturbed at fp32
                        accumulation size (tests/parity.py, perturbed_products),
                        j = 0..2: how far rounding alone moves the trajectory
  U[i]                  max |p_T - p_0| of tensor i over all its elements (the
                        "update magnitude" of the stated bf16 bound)
  idx_<i>, ref_<i>, ens_<i>   sampled elements of tensor i after the last
                        step: every element of tensors of at most 4096
                        elements, else 4096 seeded random ones
  ens_rms[j, i], ens_frac[j, i], ens_max[j, i]   member j's deviation from
                        the oracle over ALL elements of tensor i, in units of
                        the stated tolerance scale (bf16: U[i]; fp32:
                        max(|p|, lr) per element): rms, fraction above the
                        stated bound (3e-2 / 1e-4), and max
  source_hash           of the oracle, the input generators and the
                        perturbation model; a test refuses a stale file

The GPU tests compare the library's trajectory with these values; nothing
here comes from the CUDA path.

Run:  python tests/golden/make_trajectories.py [workload ...]   (about two
hours on 8 cores for all four; the LM block needs ~30 GB of host memory)
"""
import hashlib
import inspect
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import mlp_oracle as om  # noqa: E402
from tests import parity as P  # noqa: E402

WORKLOADS = ["mnist_mlp_b4096", "cifar_mlp_b8192", "deep_narrow_b65536", "lm_block_t16384"]
SAMPLES = 4096
# perturbed oracle runs per workload (MLP_TRAJ_ENSEMBLE overrides; the test
# takes the spread over however many the file holds)
ENSEMBLE = int(os.environ.get("MLP_TRAJ_ENSEMBLE", "3"))


def source_hash() -> str:
    h = hashlib.sha256()
    for f in (os.path.join(ROOT, "oracle", "mlp_oracle.py"), os.path.join(ROOT, "synth", "__init__.py")):
        with open(f, encoding="utf-8") as fh:
            h.update(fh.read().encode())
    h.update(inspect.getsource(P.perturbed_products).encode())
    h.update(inspect.getsource(P.oracle_run).encode())
    return h.hexdigest()[:16]


def stated(w) -> float:
    return 1e-4 if w.dtype == synth.F32 else 3e-2


def scale_of(w, ref, p0, U):
    """The tolerance scale per element: bf16, the tensor's largest oracle
    update; fp32, max(|p|, lr) (a parameter moves by about lr a step)."""
    if w.dtype == synth.F32:
        return np.maximum(np.abs(ref), P.hyper32(w)[0])
    return np.full(ref.shape, max(U, 1e-30))


def run(name: str) -> str:
    w = synth.WORKLOADS[name]
    t0 = time.time()
    params0 = synth.make_params(w)
    bl = P.batches(w, w.steps)
    mode = P.oracle_mode(w)
    ref = P.oracle_run(w, params0, bl, mode)
    print(f"{name}: reference run {time.time() - t0:.0f} s", flush=True)
    out = {"workload": name, "steps": w.steps, "mode": mode, "source_hash": source_hash(),
           "losses_ref": np.array(ref[0])}
    if w.dtype != synth.F32:
        ex = P.oracle_run(w, params0, bl, "bf16")
        out["losses_exact"] = np.array(ex[0])
        del ex
        print(f"{name}: exact-mode run {time.time() - t0:.0f} s", flush=True)
    p0 = [P.to64(p) for p in params0]
    pref = [np.asarray(a, np.float64) for a in ref[1]]
    del ref
    n_t = len(pref)
    U = np.array([float(np.max(np.abs(r - q))) for r, q in zip(pref, p0)])
    out["U"] = U
    rng = np.random.default_rng(20261202)
    idx = []
    for i, r in enumerate(pref):
        n = r.size
        ii = np.arange(n) if n <= SAMPLES else np.sort(rng.choice(n, SAMPLES, replace=False))
        idx.append(ii)
        out[f"idx_{i}"] = ii.astype(np.int64)
        out[f"ref_{i}"] = r.ravel()[ii]
    ens_l, ens_s = [], [[] for _ in range(n_t)]
    rms = np.zeros((ENSEMBLE, n_t))
    frac = np.zeros((ENSEMBLE, n_t))
    mx = np.zeros((ENSEMBLE, n_t))
    for j in range(ENSEMBLE):
        e = P.oracle_run(w, params0, bl, mode, perturb_seed=j + 1)
        ens_l.append(np.array(e[0]))
        for i in range(n_t):
            pe = np.asarray(e[1][i], np.float64)
            sc = scale_of(w, pref[i], p0[i], U[i])
            d = np.abs(pe - pref[i]) / sc
            rms[j, i] = float(np.sqrt(np.mean(d ** 2)))
            frac[j, i] = float(np.mean(d > stated(w)))
            mx[j, i] = float(d.max())
            ens_s[i].append(pe.ravel()[idx[i]])
        del e
        print(f"{name}: ensemble member {j} {time.time() - t0:.0f} s", flush=True)
    out["losses_ens"] = np.stack(ens_l)
    for i in range(n_t):
        out[f"ens_{i}"] = np.stack(ens_s[i])
    out["ens_rms"], out["ens_frac"], out["ens_max"] = rms, frac, mx
    path = os.path.join(HERE, f"trajectories_{name}.npz")
    np.savez_compressed(path, **out)
    print(f"{name}: wrote {path} ({os.path.getsize(path) / 1e6:.2f} MB) in {time.time() - t0:.0f} s", flush=True)
    return path


if __name__ == "__main__":
    for name in (sys.argv[1:] or WORKLOADS):
        run(name)
