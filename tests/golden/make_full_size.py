"""Writes tests/golden/full_size/<workload>.npz: the float64 oracle's results
for sampled matrices of the full-size workloads, for the GPU parity tests
(tests/test_configs_gpu.py).  Calls only the oracle (oracle/rot_oracle.py)
and the seeded input generator; nothing here comes from the CUDA path.

For each sampled matrix i of a workload, after the workload's steps:
  idx      S flat indices into W (m x n, row-major), drawn once from a
           seeded generator and stored (so the test does not depend on the
           generator's stream)
  w        the oracle's final W at those indices (float64)
  norm     ||W||_F of the oracle's whole final W
  wsamp    ||W[idx]||  (the sample's own norm, for the relative error)
  floor    the method's float32 floor: the largest relative change of the
           final W over five runs whose stored quantities are perturbed at
           2^-24 (oracle.floor)
  f32      the relative error, on the same sampled entries, of the same run
           computed in plain float32 arithmetic (oracle.run(dtype=float32)):
           what an actual float32 implementation of the method gives
  floor22  the spread at 2^-22: the largest relative change, on the sampled
           entries, over five runs whose stored quantities are perturbed at
           2^-22, the precision of the 22-bit operands (hi + lo, 11 bits
           each) that three-term tensor-core products read
  rank_u, rank_v   the numerical ranks at the last refresh

The matrices are independent, so each sampled one is run on its own.  The
samples cover every distinct shape of each Qwen3-shaped workload (one
matrix per shape, spread over the layers) and one matrix per distinct
(m, n) of the ragged workload.

    python tests/golden/make_full_size.py [workload ...]   # default: all four
    python tests/golden/make_full_size.py --add-f32 [workload ...]  # add f32 to existing files
    python tests/golden/make_full_size.py --add-floor22 [workload ...]  # add floor22
    python tests/golden/make_full_size.py slice8b --items 4 27 --seeds 3  # some matrices
    python tests/golden/make_full_size.py slice8b --merge a.npz b.npz  # join partial files

Each matrix's record is merged into the workload's file as soon as it is
computed (so a long run can be split over processes: --items, --out).  The
floor and the 2^-22 spread take the largest change over --seeds oracle runs
(default five).  The Qwen3-8B-shaped slice samples one matrix per distinct
shape (k, q, gate, down) and the second matrix of the k/v and q/o pairs.
"""

import argparse
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from matrix_optimizer_step_rot_gb300 import inputs  # noqa: E402
from oracle import rot_oracle as orc  # noqa: E402

OUT = os.path.join(HERE, "full_size")

# (workload, sampled items, samples per matrix)
PLAN = {
    # every matrix of the block
    "block": (list(range(7)), 8192),
    # one per shape kind, spread over the 28 layers: L0.k, L13.v, L27.q,
    # L5.o, L20.gate, L9.up, L14.down
    "full": ([1, 7 * 13 + 2, 7 * 27 + 0, 7 * 5 + 3, 7 * 20 + 4, 7 * 9 + 5, 7 * 14 + 6], 8192),
    # L0.k, L1.v, L3.q, L2.o, L0.gate, L3.down (up has gate's shape and path)
    "slice8b": ([1, 7 + 2, 21 + 0, 14 + 3, 4, 21 + 6], 8192),
    # filled in by ragged_items(): first matrix of each distinct (m, n)
    "ragged": (None, 1024),
}


def ragged_items(wl):
    seen, items = set(), []
    for i, shp in enumerate(wl.shapes):
        if shp not in seen:
            seen.add(shp)
            items.append(i)
    return items


class CachedInputs:
    """The workload with its gradients memoised, so the six runs of a matrix
    (reference + five floor seeds) draw them once."""

    def __init__(self, wl):
        self._wl = wl
        self._g = {}

    def __getattr__(self, name):
        return getattr(self._wl, name)

    def grad(self, i, t):
        if (i, t) not in self._g:
            self._g[(i, t)] = self._wl.grad(i, t)
        return self._g[(i, t)]

    def forget(self):
        self._g.clear()


def one(wl, i, samples, seeds=orc.FLOOR_SEEDS, with_floor22=True):
    m, n = wl.shapes[i]
    W, st = orc.run(wl, [i])[i]
    fl = orc.floor(wl, i, W, seeds=seeds)
    rng = np.random.default_rng([20260, wl.seed, i])
    s = min(samples, m * n)
    idx = np.sort(rng.choice(m * n, size=s, replace=False)).astype(np.uint32)
    w = W.ravel()[idx]
    r = dict(idx=idx, w=w, norm=float(np.linalg.norm(W)), wsamp=float(np.linalg.norm(w)),
             floor=fl, f32=f32_error(wl, i, idx, w),
             rank_u=int(st.rank_u), rank_v=int(st.rank_v))
    if with_floor22:
        r["floor22"] = floor22(wl, i, idx, w, seeds)
    return r


def f32_error(wl, i, idx, w):
    """The float32 run's relative error on the sampled entries."""
    W32, _ = orc.run(wl, [i], dtype=np.float32)[i]
    x = W32.ravel()[idx]
    return float(np.linalg.norm(x - w) / np.linalg.norm(w))


def floor22(wl, i, idx, w, seeds=orc.FLOOR_SEEDS):
    """The spread at 2^-22 on the sampled entries (see the module docstring)."""
    worst = 0.0
    for s in seeds:
        Wp, _ = orc.run(wl, [i], perturb_seed=s, perturb_rel=2.0 ** -22)[i]
        worst = max(worst, float(np.linalg.norm(Wp.ravel()[idx] - w) / np.linalg.norm(w)))
    return worst


def add_floor22(name):
    path = os.path.join(OUT, f"{name}.npz")
    z = dict(np.load(path))
    wl = CachedInputs(inputs.workload(name))
    t0 = time.time()
    for i in [int(i) for i in z["items"]]:
        z[f"{i}.floor22"] = floor22(wl, i, z[f"{i}.idx"], z[f"{i}.w"])
        wl.forget()
        print(f"{name}[{i}]: spread at 2^-22 {float(z[f'{i}.floor22']):.2e}  "
              f"[{time.time() - t0:.0f} s]", flush=True)
    np.savez_compressed(path, **z)


def add_f32(name):
    path = os.path.join(OUT, f"{name}.npz")
    z = dict(np.load(path))
    wl = CachedInputs(inputs.workload(name))
    t0 = time.time()
    for i in [int(i) for i in z["items"]]:
        z[f"{i}.f32"] = f32_error(wl, i, z[f"{i}.idx"], z[f"{i}.w"])
        wl.forget()
        print(f"{name}[{i}]: float32 run error {float(z[f'{i}.f32']):.2e}, floor "
              f"{float(z[f'{i}.floor']):.2e}  [{time.time() - t0:.0f} s]", flush=True)
    np.savez_compressed(path, **z)


def merge(path, wl0, i, r):
    """Add matrix i's record to the file (created if absent)."""
    z = dict(np.load(path)) if os.path.exists(path) else {
        "items": np.zeros(0, dtype=np.int32), "steps": wl0.steps,
        "refresh_every": wl0.refresh_every, "seed": wl0.seed}
    z["items"] = np.array(sorted(set(int(k) for k in z["items"]) | {i}), dtype=np.int32)
    for key, val in r.items():
        z[f"{i}.{key}"] = val
    np.savez_compressed(path + ".tmp.npz", **z)
    os.replace(path + ".tmp.npz", path)


def make(name, items=None, seeds=orc.FLOOR_SEEDS, out=None, with_floor22=True):
    wl0 = inputs.workload(name)
    planned, samples = PLAN[name]
    if items is None:
        items = planned if planned is not None else ragged_items(wl0)
    wl = CachedInputs(wl0)
    os.makedirs(OUT, exist_ok=True)
    path = out or os.path.join(OUT, f"{name}.npz")
    t0 = time.time()
    for k, i in enumerate(items):
        r = one(wl, i, samples, seeds, with_floor22)
        wl.forget()
        merge(path, wl0, i, r)
        print(f"{name}[{i}] {wl0.shapes[i]}: floor {r['floor']:.2e}, float32 run "
              f"{r['f32']:.2e}, spread at 2^-22 {r.get('floor22', float('nan')):.2e}, ranks "
              f"({r['rank_u']}, {r['rank_v']})  [{k + 1}/{len(items)}, "
              f"{time.time() - t0:.0f} s]", flush=True)


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("names", nargs="*", default=["ragged", "block", "full", "slice8b"])
    ap.add_argument("--add-f32", action="store_true",
                    help="add the float32 run's error to existing files")
    ap.add_argument("--add-floor22", action="store_true",
                    help="add the spread at 2^-22 to existing files")
    ap.add_argument("--items", type=int, nargs="*", help="these matrices only")
    ap.add_argument("--seeds", type=int, default=len(orc.FLOOR_SEEDS),
                    help="oracle runs for the floor and the 2^-22 spread")
    ap.add_argument("--out", help="write to this file instead of the workload's")
    ap.add_argument("--merge", nargs="*", help="merge these files' records into the workload's")
    ap.add_argument("--no-floor22", action="store_true",
                    help="skip the spread at 2^-22 (the test then bounds by 4 x float32's)")
    args = ap.parse_args()
    seeds = tuple(range(1, args.seeds + 1))
    for nm in args.names:
        if args.merge:
            wl0 = inputs.workload(nm)
            for f in args.merge:
                z = np.load(f)
                for i in (int(k) for k in z["items"]):
                    merge(os.path.join(OUT, f"{nm}.npz"), wl0, i,
                          {k.split(".", 1)[1]: z[k] for k in z.files if k.startswith(f"{i}.")})
        elif args.add_f32:
            add_f32(nm)
        elif args.add_floor22:
            add_floor22(nm)
        else:
            make(nm, args.items, seeds, args.out, not args.no_floor22)
