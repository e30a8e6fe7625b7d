"""CPU oracle for the rotated-Adam matrix-optimizer step (float64, numpy).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA path
(no kernels, headers, helpers or tables); the two meet only in the seeded input
generator, which holds none of the method's arithmetic.

Sources (page titles as published):
* Canzona page ("Canzona" matrix-optimizer framework, aitangshan.cn), section
  3.2.2 "微组调度算法": global LPT sort by compute cost, then greedy grouping
  with rollback, a min-heap load simulation and a byte cap per micro-group
  (section 6.1 / the 3.2.2 tip give 512 MB as a typical cap); section 3.2.1
  (the α-balanced greedy LPT partition of data-parallel buckets) and 3.1.1
  (static ownership by parameter start).
* "分布式训练中的流水线并行与梯度陈旧性优化", section 2.1 (the per-coordinate
  Adam update m/(sqrt(v)+eps), no bias correction) and section 2.2 (momentum
  kept as an m x n matrix; power iteration plus QR every K iterations; the
  two-sided rotation U^T W V).
* "大模型分布式优化：通信、内存、计算三层解耦实战", section 2.1 (second moment
  v_t = beta2 v_{t-1} + (1 - beta2) g_t^2).

Readings taken where the pages are silent or garbled (each is listed with its
reason in the design notes of this repository):
* the power iteration is taken to a full basis, one subspace-iteration step per
  refresh: U <- QR(M M^T U), V <- QR(M^T M V), starting from U = I, V = I;
* QR is Householder with beta = -sgn(x1)*||x|| (sgn(0) = +1), stopped at the
  numerical rank (||x|| <= rank_rtol * max_j ||a_j||), Q = H_1 ... H_r I, and the
  first r columns of Q multiplied by sgn(R_kk) so R's diagonal is positive;
* the rotated update W <- W - lr * U D V^T, D = M~ / (sqrt(v) + eps);
* v is kept as is across a refresh; no bias correction, no weight decay;
* an item's bytes are 4*m*n; one GPU is one rank for the heap.

Every function here is a plain restatement of those steps.  No blocking, no
fusion, no reordering beyond what the definitions allow.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np
import scipy.linalg
import scipy.linalg.lapack


# ---------------------------------------------------------------------------
# Micro-group planner (Canzona page, section 3.2.2)
# ---------------------------------------------------------------------------

def item_cost(m: int, n: int) -> int:
    """Compute-cost proxy of one matrix: m^2 n + m n^2 + m^3 + n^3 (exact int)."""
    return m * m * n + m * n * n + m ** 3 + n ** 3


def item_bytes(m: int, n: int) -> int:
    """Bytes of one float32 m x n matrix."""
    return 4 * m * n


@dataclasses.dataclass
class Plan:
    groups: List[List[int]]       # input indices, in LPT order, per group
    owners: List[int]             # rank assigned to each input index
    group_bytes: List[int]        # total bytes per group
    group_cost: List[int]         # total cost per group


def plan(shapes: Sequence[Tuple[int, int]], c_max: int, ranks: int = 1) -> Plan:
    """Global LPT sort, then greedy grouping with rollback under a byte cap.

    1. Sort all items by cost, descending; equal costs keep input order.
    2. Walk the sorted list.  Tentatively put the item into the current group:
       the load simulation gives it to the rank with the smallest accumulated
       cost in this group (ties: lowest rank id), as a min-heap would.
    3. If that leaves some rank of the group holding more than c_max bytes and
       the group already had items, undo the tentative step, close the group,
       and place the item in a fresh group (where it is alone at first).  An
       item larger than c_max therefore ends up in a group of its own.
    """
    count = len(shapes)
    cost = [item_cost(m, n) for m, n in shapes]
    nbytes = [item_bytes(m, n) for m, n in shapes]
    order = sorted(range(count), key=lambda i: (-cost[i], i))

    groups: List[List[int]] = []
    owners = [-1] * count
    current: List[int] = []
    load = [0] * ranks      # accumulated cost per rank, current group
    held = [0] * ranks      # accumulated bytes per rank, current group

    for i in order:
        r = min(range(ranks), key=lambda q: (load[q], q))
        trial = list(held)
        trial[r] += nbytes[i]
        if current and max(trial) > c_max:
            groups.append(current)          # roll back: close the group
            current, load, held = [], [0] * ranks, [0] * ranks
            r = 0
            trial = list(held)
            trial[r] += nbytes[i]
        current.append(i)
        load[r] += cost[i]
        held = trial
        owners[i] = r
    if current:
        groups.append(current)

    return Plan(groups=groups, owners=owners,
                group_bytes=[sum(nbytes[i] for i in g) for g in groups],
                group_cost=[sum(cost[i] for i in g) for g in groups])


# ---------------------------------------------------------------------------
# Data-parallel partition (Canzona page, section 3.2.1 "α平衡贪心LPT算法",
# and section 3.1.1 for the static baseline)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Partition:
    owners: List[int]   # rank of every item (input order)
    loads: List[int]    # total work per rank


def static_partition(elems: Sequence[int], bucket_sizes: Sequence[int], ranks: int) -> List[int]:
    """Ownership by parameter start (section 3.1.1), bucket by bucket as a
    ZeRO-1 flat buffer is sharded: bucket b's items lie back to back in E_b =
    sum of their elements, cut into `ranks` equal shards of S_b = ceil(E_b /
    ranks) elements; an item belongs to the shard holding its first element."""
    if sum(bucket_sizes) != len(elems):
        raise ValueError("bucket sizes must cover the items")
    owners, i = [], 0
    for c in bucket_sizes:
        total = sum(elems[i:i + c])
        shard = max(1, -(-total // ranks))
        start = 0
        for e in elems[i:i + c]:
            owners.append(min(ranks - 1, start // shard))
            start += e
        i += c
    return owners


IDEAL_BEFORE = "before"  # the page's printed ideal load: sum(L) / R
IDEAL_AFTER = "after"    # the even share once the bucket is placed: (sum(L) + W_b) / R


def alpha_partition(work: Sequence[int], bucket_sizes: Sequence[int], ranks: int,
                    alpha: float, ideal: str = IDEAL_BEFORE) -> Partition:
    """α-balanced greedy LPT partition of buckets of items (section 3.2.1).

    Items lie in physical order; bucket b is the next bucket_sizes[b] of them
    and its work W_b is the sum of its items' work.
    1. Visit the buckets by W_b, largest first (equal W_b: lower index first).
    2. For the bucket at hand, with per-rank loads L so far: the ideal load A
       is sum(L) / R, the mean load before the bucket, as the page's code
       prints it (ideal="before"), or (sum(L) + W_b) / R, the mean once the
       bucket is placed (ideal="after", this library's alternative reading);
       deficit d_r = max(0, A - L_r); fill shares v_fill = d / sum(d) (1/R each
       if every deficit is zero); even shares 1/R; mixed shares
       v*_r = (1 - alpha) / R + alpha * v_fill_r.
    3. The bucket is cut into R consecutive pieces, rank r taking piece r.  Cut
       r (after rank r's piece) is the item boundary j whose prefix work P_j is
       nearest to W_b * (v*_0 + ... + v*_r); on a tie the earlier boundary.
       Cuts therefore fall on item boundaries only (no item is split).
    4. Each rank's load grows by the work of its piece.
    Floating-point steps are done in float64 in exactly this order; prefix
    work and loads are exact integers.
    """
    if ranks < 1:
        raise ValueError("ranks must be >= 1")
    if ideal not in (IDEAL_BEFORE, IDEAL_AFTER):
        raise ValueError("ideal must be 'before' or 'after'")
    if sum(bucket_sizes) != len(work):
        raise ValueError("bucket sizes must cover the items")
    starts, s = [], 0
    for c in bucket_sizes:
        starts.append(s)
        s += c
    bwork = [sum(work[starts[b]:starts[b] + bucket_sizes[b]]) for b in range(len(bucket_sizes))]
    order = sorted(range(len(bucket_sizes)), key=lambda b: (-bwork[b], b))
    owners = [-1] * len(work)
    loads = [0] * ranks
    for b in order:
        items = list(range(starts[b], starts[b] + bucket_sizes[b]))
        placed = sum(loads) + (bwork[b] if ideal == IDEAL_AFTER else 0)
        target_load = float(placed) / float(ranks)
        deficit = [max(0.0, target_load - float(l)) for l in loads]
        dsum = 0.0
        for d in deficit:
            dsum += d
        if dsum > 0.0:
            fill = [d / dsum for d in deficit]
        else:
            fill = [1.0 / float(ranks)] * ranks
        share = [(1.0 - alpha) / float(ranks) + alpha * f for f in fill]
        prefix = [0]
        for i in items:
            prefix.append(prefix[-1] + work[i])
        cuts, cum = [], 0.0
        for r in range(ranks - 1):
            cum += share[r]
            target = float(bwork[b]) * cum
            best = 0
            for j in range(len(prefix)):
                if abs(float(prefix[j]) - target) < abs(float(prefix[best]) - target):
                    best = j
            cuts.append(best)
        cuts.append(len(items))
        lo = 0
        for r in range(ranks):
            hi = max(lo, cuts[r])
            for j in range(lo, hi):
                owners[items[j]] = r
            loads[r] += prefix[hi] - prefix[lo]
            lo = hi
    return Partition(owners=owners, loads=loads)


def imbalance(values: Sequence[float]) -> float:
    """max / mean of per-rank totals (1.0 = perfectly even)."""
    mean = sum(values) / len(values)
    return max(values) / mean if mean > 0 else 1.0


# ---------------------------------------------------------------------------
# Householder QR with positive R diagonal and numerical-rank stop
# ---------------------------------------------------------------------------

def hqr_plus(A: np.ndarray, rank_rtol: float) -> Tuple[np.ndarray, int, np.ndarray]:
    """Q factor of a square matrix by Householder reflections.

    tau = rank_rtol * max_j ||a_j||.  For k = 0, 1, ...: x = (H_{k-1}..H_0 A)[k:, k];
    stop when ||x|| <= tau (r = k).  Otherwise beta_k = -sgn(x_0) ||x|| with
    sgn(0) = +1, w = x - beta_k e_0, H_k = I - 2 w w^T / (w^T w) on rows k...
    Q = H_0 H_1 ... H_{r-1} I (accumulated backwards), then column k of Q for
    k < r is multiplied by sgn(beta_k), which makes R's diagonal positive.
    Columns r.. are left as the reflectors make them.

    Returns (Q, r, beta[0:r]).
    """
    A = np.array(A, dtype=np.float64, copy=True)
    p, q = A.shape
    assert p == q, "square input expected"
    tau = rank_rtol * max(float(np.linalg.norm(A[:, j])) for j in range(q)) if q else 0.0

    reflectors: List[Tuple[int, np.ndarray]] = []
    betas: List[float] = []
    for k in range(q):
        x = A[k:, k]
        nx = float(np.linalg.norm(x))
        if nx <= tau:
            break
        beta = -nx if x[0] >= 0.0 else nx
        w = x.copy()
        w[0] -= beta
        ww = float(w @ w)
        # apply H_k to the trailing block (columns k.. of rows k..)
        A[k:, k:] -= np.outer(w, (2.0 / ww) * (w @ A[k:, k:]))
        reflectors.append((k, w))
        betas.append(beta)
    r = len(reflectors)

    # Backward accumulation: Q = H_0 (H_1 (... (H_{r-1} I))).  When H_k is
    # applied, columns 0..k-1 of the partial product are still the unit vectors
    # e_j (j < k), whose rows k.. are zero, so only Q[k:, k:] changes.
    Q = np.eye(p)
    for k, w in reversed(reflectors):
        ww = float(w @ w)
        Q[k:, k:] -= np.outer(w, (2.0 / ww) * (w @ Q[k:, k:]))
    for k in range(r):
        if betas[k] < 0.0:
            Q[:, k] = -Q[:, k]
    return Q, r, np.array(betas)


_C = None


def _c_lib():
    """The C build of the same QR+ (oracle/hqr.c), or None if not built."""
    global _C
    if _C is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhqr.so")
        if not os.path.exists(path):
            return None
        lib = ctypes.CDLL(path)
        lib.hqr_plus_f64.restype = ctypes.c_long
        lib.hqr_plus_f64.argtypes = [ctypes.c_long, ctypes.c_void_p, ctypes.c_double,
                                     ctypes.c_void_p, ctypes.c_void_p]
        _C = lib
    return _C


def hqr_plus_c(A: np.ndarray, rank_rtol: float) -> Tuple[np.ndarray, int, np.ndarray]:
    """hqr_plus() computed by oracle/hqr.c (same steps, column-major C loops)."""
    lib = _c_lib()
    if lib is None:
        raise RuntimeError("oracle/libhqr.so is not built (oracle/build_oracle.py)")
    p = A.shape[0]
    a = np.array(A, dtype=np.float64, order="F", copy=True)
    Q = np.empty((p, p), dtype=np.float64, order="F")
    beta = np.zeros(max(p, 1), dtype=np.float64)
    r = lib.hqr_plus_f64(p, a.ctypes.data, float(rank_rtol), Q.ctypes.data, beta.ctypes.data)
    if r < 0:
        raise MemoryError("hqr_plus_f64")
    return np.ascontiguousarray(Q), int(r), beta[:r].copy()


def hqr_plus_lapack(A: np.ndarray, rank_rtol: float,
                    ncols: Optional[int] = None) -> Tuple[np.ndarray, int, np.ndarray]:
    """hqr_plus() with LAPACK's Householder routines as its two library steps:
    dgeqrf finds the reflectors of A's columns, dorgqr multiplies them out,
    Q = H_0 H_1 ... H_{r-1} I.

    The same definition as hqr_plus: LAPACK's reflector generator (dlarfg)
    takes beta = -sgn(x_0) ||x|| as well, and |R_kk| = ||x|| at step k, so
    the rank r is the first k with |R_kk| <= tau.  One case differs: when the
    part of x below x_0 is exactly zero, dlarfg takes H_k = I (tau_k = 0,
    R_kk = x_0) where hqr_plus reflects with w = 2 x_0 e_0 (beta_k = -x_0).
    That reflector is put back here (tau_k = 2, v = e_k, beta_k = -R_kk), so
    the completion columns match too.

    ncols: only the first ncols columns are factored (the reflectors of the
    first k columns do not depend on later ones, so the result is the same
    whenever the stop comes by column ncols - 1, as it does when
    ncols > rank(A)); default: all.  Returns (Q, r, beta[0:r]).
    """
    dt = np.float32 if np.asarray(A).dtype == np.float32 else np.float64  # float32 runs
    A = np.asarray(A, dtype=dt)
    p, q = A.shape
    assert p == q, "square input expected"
    if p == 0:
        return np.eye(0, dtype=dt), 0, np.zeros(0, dtype=dt)
    tau_abs = rank_rtol * float(np.max(np.linalg.norm(A, axis=0)))
    c = p if ncols is None else max(1, min(p, int(ncols)))
    (qr, tau), R = scipy.linalg.qr(A[:, :c], mode="raw")
    diag = np.diag(R)
    r = c
    for k in range(c):
        if abs(float(diag[k])) <= tau_abs:
            r = k
            break
    beta = np.array(diag[:r], dtype=dt)
    t = np.array(tau[:r], dtype=dt)
    flat = t == 0.0  # zero sub-column: restore the reflection hqr_plus makes
    t[flat] = 2.0
    beta[flat] = -beta[flat]
    if r == 0:
        return np.eye(p, dtype=dt), 0, beta
    a = np.zeros((p, p), dtype=dt, order="F")
    a[:, :r] = qr[:, :r]
    orgqr = scipy.linalg.lapack.sorgqr if dt == np.float32 else scipy.linalg.lapack.dorgqr
    Q, _, info = orgqr(a, t, lwork=max(1, 64 * p))
    if info != 0:
        raise RuntimeError(f"dorgqr failed ({info})")
    Q = np.array(Q)
    Q[:, :r][:, beta < 0.0] *= -1.0
    return Q, r, beta


def default_qr():
    """The QR+ the oracle's runs use: the LAPACK-step version (fast at the
    12288-sized bases); hqr_plus and hqr_plus_c are its hand-written checks."""
    return hqr_plus_lapack


# ---------------------------------------------------------------------------
# One optimizer step for one matrix
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class MatrixState:
    M: np.ndarray   # momentum, m x n, original coordinates
    v: np.ndarray   # second moment, m x n, rotated coordinates
    U: np.ndarray   # left basis, m x m
    V: np.ndarray   # right basis, n x n
    rank_u: int = -1
    rank_v: int = -1


def init_state(m: int, n: int, dtype=np.float64) -> MatrixState:
    """M = 0, v = 0, U = I_m, V = I_n."""
    return MatrixState(M=np.zeros((m, n), dtype=dtype), v=np.zeros((m, n), dtype=dtype),
                       U=np.eye(m, dtype=dtype), V=np.eye(n, dtype=dtype))


def refresh_basis(M: np.ndarray, U: np.ndarray, V: np.ndarray, rank_rtol: float,
                  qr: Optional[Callable] = None, perturb: Optional[Callable] = None):
    """One subspace-iteration step on each side: U <- QR+(M M^T U), V <- QR+(M^T M V).

    `qr` picks the QR+ implementation (default: default_qr()); `perturb`, used
    only to measure the method's sensitivity, maps (name, array) to a
    perturbed copy of each stored quantity (see run())."""
    qr = qr or default_qr()
    m, n = M.shape
    A_U = M @ (M.T @ U)
    A_V = M.T @ (M @ V)
    if perturb is not None:
        A_U, A_V = perturb("A_U", A_U), perturb("A_V", A_V)
    if qr is hqr_plus_lapack:
        # rank(A_U), rank(A_V) <= min(m, n): the stop comes by column min(m, n)
        U_new, r_u, _ = qr(A_U, rank_rtol, ncols=min(m, n) + 1)
        V_new, r_v, _ = qr(A_V, rank_rtol, ncols=min(m, n) + 1)
    else:
        U_new, r_u, _ = qr(A_U, rank_rtol)
        V_new, r_v, _ = qr(A_V, rank_rtol)
    if perturb is not None:
        U_new, V_new = perturb("U", U_new), perturb("V", V_new)
    return U_new, V_new, r_u, r_v


def step(W: np.ndarray, G: np.ndarray, st: MatrixState, beta1: float, beta2: float,
         eps: float, lr: float, refresh: bool, rank_rtol: float,
         perturb: Optional[Callable] = None) -> np.ndarray:
    """One rotated-Adam step; updates `st` in place and returns the new W (float64).

    (1) M <- beta1 M + (1 - beta1) G
    (2) if refresh: U, V <- subspace-iteration step + QR+
    (3) G~ = U^T G V, M~ = U^T M V, v <- beta2 v + (1 - beta2) G~^2, D = M~ / (sqrt(v) + eps)
    (4) W <- W - lr U D V^T

    `perturb` (sensitivity runs only) maps (name, array) to a perturbed copy of
    each quantity a float32 implementation stores: M, the QR inputs A_U and
    A_V, the new U and V, G~, M~, v and D.
    """
    p = perturb or (lambda name, X: X)
    dt = st.M.dtype  # float64; float32 in the float32 runs (see run())
    G = np.asarray(G, dtype=dt)
    beta1, beta2, eps, lr = dt.type(beta1), dt.type(beta2), dt.type(eps), dt.type(lr)
    one = dt.type(1.0)
    st.M = p("M", beta1 * st.M + (one - beta1) * G)
    if refresh:
        st.U, st.V, st.rank_u, st.rank_v = refresh_basis(st.M, st.U, st.V, rank_rtol,
                                                         perturb=perturb)
    Gt = p("Gt", (st.U.T @ G) @ st.V)
    Mt = p("Mt", (st.U.T @ st.M) @ st.V)
    st.v = p("v", beta2 * st.v + (one - beta2) * (Gt * Gt))
    D = p("D", Mt / (np.sqrt(st.v) + eps))
    return np.asarray(W, dtype=dt) - lr * ((st.U @ D) @ st.V.T)


# ---------------------------------------------------------------------------
# A whole run of a workload (matrices are independent, so any subset can run)
# ---------------------------------------------------------------------------

FLOOR_REL = 2.0 ** -24  # float32 unit roundoff
FLOOR_SEEDS = (1, 2, 3, 4, 5)
# The reduced-precision state the pages describe: rotation matrices stored in
# float16 (the rotation page, section 3.1; unit roundoff 2^-11) and the first
# moment in BF16 (the ZeRO essay, section 3.3; unit roundoff 2^-8), v and
# everything else as before.
COMPACT_RELS = {"U": 2.0 ** -11, "V": 2.0 ** -11, "M": 2.0 ** -8, "Mt": 2.0 ** -8}


def run(wl, items: Optional[Sequence[int]] = None, steps: Optional[int] = None,
        first_step: int = 1, perturb_seed: Optional[int] = None,
        perturb_rel: float = FLOOR_REL,
        perturb_rels: Optional[Dict[str, float]] = None,
        dtype=np.float64) -> Dict[int, Tuple[np.ndarray, MatrixState]]:
    """Run `steps` steps (default: the workload's) for the chosen matrices.

    `wl` is a workload object exposing shapes, hyper, refresh(t), w0(i) and
    grad(i, t).  Returns {i: (W, state)} with W in float64.

    With perturb_seed set, every quantity a float32 implementation stores (see
    step()) is multiplied element-wise by (1 + perturb_rel * xi), xi ~ N(0, 1),
    each time it is formed: the same method on values that differ at float32
    rounding level.  How far that moves the final W is the method's own
    sensitivity, the floor any float32 implementation faces.  perturb_rels
    gives some quantities (by the names step() uses) another size: the
    rounding of a lower-precision storage format (COMPACT_RELS).

    dtype=np.float32 runs the same steps in float32 arithmetic (float32
    arrays, float32 BLAS products and LAPACK's float32 Householder routines)
    and returns its W in float64: what a plain float32 implementation of the
    method gives, a sensitivity reference.  The oracle proper is float64.
    """
    items = list(range(wl.count)) if items is None else list(items)
    steps = wl.steps if steps is None else steps
    h = wl.hyper
    out = {}
    for i in items:
        m, n = wl.shapes[i]
        W = wl.w0(i).astype(dtype)
        st = init_state(m, n, dtype)
        perturb = None
        if perturb_seed is not None:
            rng = np.random.default_rng([perturb_seed, i])
            rels = dict(perturb_rels or {})
            perturb = (lambda name, X, rng=rng, rels=rels:
                       X * (1.0 + rels.get(name, perturb_rel) * rng.standard_normal(X.shape)))
        for t in range(first_step, first_step + steps):
            W = step(W, wl.grad(i, t), st, h.beta1, h.beta2, h.eps, h.lr, wl.refresh(t),
                     h.rank_rtol, perturb=perturb)
        out[i] = (np.asarray(W, dtype=np.float64), st)
    return out


def floor(wl, item: int, W_ref: np.ndarray, seeds: Sequence[int] = FLOOR_SEEDS,
          steps: Optional[int] = None, rel: float = FLOOR_REL,
          rels: Optional[Dict[str, float]] = None) -> float:
    """The method's float32 floor for one matrix: the largest relative change
    of the final W over runs (one per seed) whose stored quantities are
    perturbed at relative size `rel` (float32 unit roundoff by default;
    `rels` overrides it per quantity, see run())."""
    worst = 0.0
    for s in seeds:
        Wp, _ = run(wl, [item], steps=steps, perturb_seed=s, perturb_rel=rel,
                    perturb_rels=rels)[item]
        worst = max(worst, float(np.linalg.norm(Wp - W_ref) / np.linalg.norm(W_ref)))
    return worst


def float32_error(wl, item: int, W_ref: np.ndarray, steps: Optional[int] = None) -> float:
    """Relative Frobenius distance between the float64 oracle's final W and
    the same run computed in plain float32 arithmetic (see run())."""
    W32, _ = run(wl, [item], steps=steps, dtype=np.float32)[item]
    return float(np.linalg.norm(W32 - W_ref) / np.linalg.norm(W_ref))


def orthogonality_error(Q: np.ndarray) -> float:
    """||Q^T Q - I||_F."""
    return float(np.linalg.norm(Q.T @ Q - np.eye(Q.shape[1])))
