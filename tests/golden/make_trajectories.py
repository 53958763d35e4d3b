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

Run:  python tests/golden/make_trajectories.py [--jobs N] [workload ...]
(one after another: hours for the deep narrow net and the LM block on 8
cores, and the LM block holds about 40 GB; --jobs runs the reference, exact
and perturbed runs as N processes at a time where memory allows)
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


def _piece(name: str, kind: str, j: int = 0):
    """One oracle run of workload `name`: kind "ref" (the reference mode),
    "exact" (bf16 workloads: the exact-rounding mode) or "ens" (perturbed
    run j + 1).  Returns (losses, final parameters or None)."""
    w = synth.WORKLOADS[name]
    params0 = synth.make_params(w)
    bl = P.batches(w, w.steps)
    mode = P.oracle_mode(w)
    if kind == "exact":
        e = P.oracle_run(w, params0, bl, "bf16")
        return np.array(e[0]), None
    r = P.oracle_run(w, params0, bl, mode, perturb_seed=(j + 1) if kind == "ens" else 0)
    return np.array(r[0]), [np.asarray(a, np.float64) for a in r[1]]


def _assemble(name: str, ref, exact, ens, t0: float) -> str:
    """The stored file from the pieces: ref = (losses, params), exact =
    losses or None, ens = [(losses, params)] in member order."""
    w = synth.WORKLOADS[name]
    out = {"workload": name, "steps": w.steps, "mode": P.oracle_mode(w), "source_hash": source_hash(),
           "losses_ref": ref[0]}
    if exact is not None:
        out["losses_exact"] = exact
    p0 = [P.to64(p) for p in synth.make_params(w)]
    pref = ref[1]
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
    m = len(ens)
    rms, frac, mx = np.zeros((m, n_t)), np.zeros((m, n_t)), np.zeros((m, n_t))
    ens_s = [[] for _ in range(n_t)]
    for jj, (_, pe_all) in enumerate(ens):
        for i in range(n_t):
            pe = pe_all[i]
            sc = scale_of(w, pref[i], p0[i], U[i])
            d = np.abs(pe - pref[i]) / sc
            rms[jj, i] = float(np.sqrt(np.mean(d ** 2)))
            frac[jj, i] = float(np.mean(d > stated(w)))
            mx[jj, i] = float(d.max())
            ens_s[i].append(pe.ravel()[idx[i]])
    out["losses_ens"] = np.stack([e[0] for e in ens])
    for i in range(n_t):
        out[f"ens_{i}"] = np.stack(ens_s[i])
    out["ens_rms"], out["ens_frac"], out["ens_max"] = rms, frac, mx
    path = os.path.join(HERE, f"trajectories_{name}.npz")
    np.savez_compressed(path, **out)
    print(f"{name}: wrote {path} ({os.path.getsize(path) / 1e6:.2f} MB) in {time.time() - t0:.0f} s", flush=True)
    return path


def run(name: str) -> str:
    """The oracle runs one after another in this process."""
    w = synth.WORKLOADS[name]
    t0 = time.time()
    ref = _piece(name, "ref")
    print(f"{name}: reference run {time.time() - t0:.0f} s", flush=True)
    exact = None
    if w.dtype != synth.F32:
        exact = _piece(name, "exact")[0]
        print(f"{name}: exact-mode run {time.time() - t0:.0f} s", flush=True)
    ens = []
    for j in range(ENSEMBLE):
        ens.append(_piece(name, "ens", j))
        print(f"{name}: ensemble member {j} {time.time() - t0:.0f} s", flush=True)
    return _assemble(name, ref, exact, ens, t0)


def _mem_available() -> float:
    """Bytes of host memory available (Linux)."""
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                return float(line.split()[1]) * 1024.0
    return 0.0


def _piece_to_file(name, kind, j, path):
    losses, params = _piece(name, kind, j)
    arrs = {"losses": losses}
    if params is not None:
        for i, a in enumerate(params):
            arrs[f"p_{i}"] = a
    np.savez(path, **arrs)


def run_parallel(name: str, jobs: int, min_free_gb: float) -> str:
    """The same oracle runs as separate processes, at most `jobs` at a time
    and a new one only while more than `min_free_gb` of host memory is
    free (each full-batch run of the LM block holds about 40 GB)."""
    import multiprocessing as mp
    import tempfile
    w = synth.WORKLOADS[name]
    t0 = time.time()
    kinds = [("ref", 0)] + ([("exact", 0)] if w.dtype != synth.F32 else []) + [("ens", j) for j in range(ENSEMBLE)]
    ctx = mp.get_context("spawn")
    tmp = tempfile.mkdtemp(prefix="traj_")
    files = {k: os.path.join(tmp, f"{k[0]}_{k[1]}.npz") for k in kinds}
    todo, running = list(kinds), {}
    while todo or running:
        for k, pr in list(running.items()):
            if not pr.is_alive():
                pr.join()
                if pr.exitcode != 0:
                    raise RuntimeError(f"{name}: oracle run {k} failed ({pr.exitcode})")
                print(f"{name}: {k[0]} {k[1]} done at {time.time() - t0:.0f} s", flush=True)
                del running[k]
        if todo and len(running) < jobs and (not running or _mem_available() > min_free_gb * 2 ** 30):
            k = todo.pop(0)
            pr = ctx.Process(target=_piece_to_file, args=(name, k[0], k[1], files[k]))
            pr.start()
            running[k] = pr
            time.sleep(60)   # let its memory grow before the next check
        else:
            time.sleep(5)

    def load(k):
        d = np.load(files[k])
        n = len([f for f in d.files if f.startswith("p_")])
        return d["losses"], ([d[f"p_{i}"] for i in range(n)] if n else None)
    ref = load(("ref", 0))
    exact = load(("exact", 0))[0] if ("exact", 0) in files else None
    ens = [load(("ens", j)) for j in range(ENSEMBLE)]
    return _assemble(name, ref, exact, ens, t0)


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("workloads", nargs="*", default=WORKLOADS)
    ap.add_argument("--jobs", type=int, default=1, help="oracle runs at a time, each in its own process")
    ap.add_argument("--min-free-gb", type=float, default=60.0)
    a = ap.parse_args()
    for name in a.workloads:
        if a.jobs > 1:
            run_parallel(name, a.jobs, a.min_free_gb)
        else:
            run(name)
