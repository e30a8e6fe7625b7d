"""Pins for the fp64 oracle: each test checks it against something other than
itself (closed forms, a library routine, brute force, hand-worked values)."""

import itertools

import numpy as np
import pytest

from oracle import build_oracle
from oracle import rot_oracle as orc
from matrix_optimizer_step_rot_gb300 import inputs

build_oracle.build()
QR_IMPLS = [orc.hqr_plus, orc.hqr_plus_c, orc.hqr_plus_lapack]

H = inputs.Hyper()
B1, B2, EPS, LR = H.beta1, H.beta2, H.eps, H.lr


def rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# P1: with U = V = I and no refresh the step is plain Adam, bit for bit
# --------------------------------------------------------------------------

def test_reduces_to_plain_adam_bit_exact():
    r = rng(1)
    m, n = 24, 40
    W = r.normal(0, 0.02, (m, n)).astype(np.float32).astype(np.float64)
    st = orc.init_state(m, n)
    W_ref = W.copy()
    mom = np.zeros((m, n))
    var = np.zeros((m, n))
    for t in range(1, 8):
        g = r.normal(0, 1e-2, (m, n)).astype(np.float32).astype(np.float64)
        W = orc.step(W, g, st, B1, B2, EPS, LR, False, H.rank_rtol)
        # plain Adam without bias correction
        mom = B1 * mom + (1.0 - B1) * g
        var = B2 * var + (1.0 - B2) * g * g
        W_ref = W_ref - LR * (mom / (np.sqrt(var) + EPS))
        assert np.array_equal(W, W_ref), f"step {t}"
        assert np.array_equal(st.M, mom) and np.array_equal(st.v, var)


# --------------------------------------------------------------------------
# P2: closed form of the first step without refresh
# --------------------------------------------------------------------------

def test_step_one_closed_form():
    r = rng(2)
    m, n = 16, 12
    g = r.normal(0, 1e-2, (m, n))
    W0 = r.normal(0, 0.02, (m, n))
    st = orc.init_state(m, n)
    W1 = orc.step(W0, g, st, B1, B2, EPS, LR, False, H.rank_rtol)
    D = (1.0 - B1) * g / (np.sqrt(1.0 - B2) * np.abs(g) + EPS)
    np.testing.assert_allclose((W0 - W1) / LR, D, rtol=1e-12, atol=0)
    # with |g| >> eps the first update is (1-b1)/sqrt(1-b2) * sign(g) ~ 3.1623
    big = np.abs(g) > 1e-3      # eps / (sqrt(1-b2) |g|) < 3.2e-4 there
    np.testing.assert_allclose(np.abs(D[big]), (1.0 - B1) / np.sqrt(1.0 - B2), rtol=4e-4)


# --------------------------------------------------------------------------
# Rotation direction: U^T G V forward and U D V^T back, with known bases
# --------------------------------------------------------------------------

def _signed_perm(p, seed):
    r = rng(seed)
    P = np.zeros((p, p))
    P[np.arange(p), (np.arange(p) + 1) % p] = r.choice([-1.0, 1.0], size=p)  # signed cycle
    return P


def test_rotation_directions_closed_form():
    m, n = 7, 5
    U0, V0 = _signed_perm(m, 3), _signed_perm(n, 4)
    assert not np.allclose(U0, U0.T) and not np.allclose(V0, V0.T)
    r = rng(5)
    S = r.normal(0, 1e-2, (m, n))      # rotated-coordinate gradient
    S2 = r.normal(0, 1e-2, (m, n))     # rotated-coordinate old momentum
    G = U0 @ S @ V0.T
    st = orc.init_state(m, n)
    st.U, st.V = U0.copy(), V0.copy()
    st.M = U0 @ S2 @ V0.T
    W0 = r.normal(0, 0.02, (m, n))
    W1 = orc.step(W0, G, st, B1, B2, EPS, LR, False, H.rank_rtol)
    Mt = B1 * S2 + (1.0 - B1) * S
    v = (1.0 - B2) * S * S
    D = Mt / (np.sqrt(v) + EPS)
    np.testing.assert_allclose(W1, W0 - LR * U0 @ D @ V0.T, rtol=0, atol=1e-15)
    np.testing.assert_allclose(st.v, v, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# P4: Householder QR+ against LAPACK (numpy.linalg.qr)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("qr", QR_IMPLS)
@pytest.mark.parametrize("p", [1, 2, 8, 33, 64])
def test_hqr_full_rank_matches_lapack_with_sign_fix(p, qr):
    A = rng(10 + p).normal(size=(p, p))
    Q, r, beta = qr(A, 1e-3)
    assert r == p
    Qn, Rn = np.linalg.qr(A)
    Qn = Qn * np.sign(np.diag(Rn))[None, :]
    np.testing.assert_allclose(Q, Qn, rtol=0, atol=1e-12)
    assert orc.orthogonality_error(Q) <= 1e-12
    # R = Q^T A is upper triangular with a positive diagonal
    R = Q.T @ A
    assert np.all(np.diag(R) > 0)
    assert np.abs(np.tril(R, -1)).max() <= 1e-12 * np.abs(A).max() * p


@pytest.mark.parametrize("qr", QR_IMPLS)
@pytest.mark.parametrize("p,rk", [(6, 2), (17, 5), (40, 39)])
def test_hqr_rank_deficient_completion_matches_lapack(p, rk, qr):
    """A = [B | 0]: LAPACK's reflectors for the zero columns are identities, so
    its complete Q is H_0..H_{r-1} I, the completion the numerical-rank stop uses.
    The opposite reflector sign convention would give a different completion."""
    B = rng(20 + p).normal(size=(p, rk))
    A = np.hstack([B, np.zeros((p, p - rk))])
    Q, r, beta = qr(A, 1e-3)
    assert r == rk
    Qn, Rn = np.linalg.qr(A, mode="complete")
    signs = np.ones(p)
    signs[:rk] = np.sign(np.diag(Rn)[:rk])
    np.testing.assert_allclose(Q, Qn * signs[None, :], rtol=0, atol=1e-12)
    assert orc.orthogonality_error(Q) <= 1e-12


@pytest.mark.parametrize("qr", QR_IMPLS)
def test_hqr_rank_one_closed_form_completion(qr):
    """Rank one: a single reflector; every column is written out by hand."""
    p = 9
    a = rng(30).normal(size=p)
    a[0] = -abs(a[0])                       # exercise the negative-x0 branch
    c = rng(31).normal(size=p)
    A = np.outer(a, c)
    Q, r, beta = qr(A, 1e-6)
    assert r == 1
    x = A[:, 0]
    nx = np.linalg.norm(x)
    b = -np.sign(x[0]) * nx
    w = x.copy()
    w[0] -= b
    H0 = np.eye(p) - 2.0 * np.outer(w, w) / (w @ w)
    expect = H0.copy()
    expect[:, 0] *= np.sign(b)
    np.testing.assert_allclose(Q, expect, rtol=0, atol=1e-13)
    # first column is the unit vector along the column space, positive R
    # H_0 e_0 = x / beta, so the sign-fixed first column is sgn(c_0) a / ||a||
    np.testing.assert_allclose(Q[:, 0], np.sign(c[0]) * a / np.linalg.norm(a), atol=1e-13)


@pytest.mark.parametrize("qr", QR_IMPLS)
def test_hqr_zero_matrix_is_identity(qr):
    Q, r, _ = qr(np.zeros((5, 5)), 1e-3)
    assert r == 0 and np.array_equal(Q, np.eye(5))


def test_c_qr_matches_numpy_definition_on_refresh_inputs():
    """The C build follows the numpy definition step for step (rounding order
    aside) on Gram-type inputs with a rank stop inside, as the refresh makes."""
    for m, n, seed in [(70, 40, 1), (40, 70, 2), (96, 96, 3)]:
        M = rng(seed).normal(size=(m, n))
        for A in (M @ M.T, M.T @ M):
            Qn, rn, bn = orc.hqr_plus(A, 1e-3)
            Qc, rc, bc = orc.hqr_plus_c(A, 1e-3)
            assert rn == rc
            np.testing.assert_allclose(Qc, Qn, rtol=0, atol=1e-11)
            np.testing.assert_allclose(bc, bn, rtol=1e-12, atol=0)


def test_lapack_qr_matches_hand_written_householder_on_refresh_inputs():
    """The oracle's runs take QR+ through LAPACK's Householder routines; the
    plain Householder loop (hqr_plus) checks it, completion columns included,
    on Gram-type inputs with a rank stop inside, with and without the column
    limit the refresh passes."""
    for m, n, seed in [(70, 40, 1), (40, 70, 2), (96, 96, 3), (130, 9, 4)]:
        M = rng(seed).normal(size=(m, n))
        for A in (M @ M.T, M.T @ M):
            Qn, rn, bn = orc.hqr_plus(A, 1e-3)
            for ncols in (None, min(m, n) + 1):
                Ql, rl, bl = orc.hqr_plus_lapack(A, 1e-3, ncols=ncols)
                assert rl == rn
                np.testing.assert_allclose(Ql, Qn, rtol=0, atol=1e-11)
                np.testing.assert_allclose(bl, bn, rtol=1e-12, atol=0)


@pytest.mark.parametrize("qr", QR_IMPLS)
def test_hqr_zero_subcolumns_hand_worked(qr):
    """A = diag(3, -2, 0, 0): each factored column has nothing below its
    diagonal, so x = x_0 e_0.  By the definition beta = -sgn(x_0)|x_0| and
    w = 2 x_0 e_0, H_k = I - 2 e_k e_k^T: H_0 = diag(-1, 1, 1, 1) (beta_0 = -3),
    H_1 = diag(1, -1, 1, 1) (beta_1 = 2), then the stop (r = 2).  Q = H_0 H_1 I
    = diag(-1, -1, 1, 1); the sign fix negates column 0: diag(1, -1, 1, 1).
    (LAPACK's generator takes H = I here; the LAPACK-step version restores the
    reflection.)"""
    A = np.diag([3.0, -2.0, 0.0, 0.0])
    Q, r, beta = qr(A, 1e-3)
    assert r == 2
    np.testing.assert_array_equal(beta, [-3.0, 2.0])
    np.testing.assert_array_equal(Q, np.diag([1.0, -1.0, 1.0, 1.0]))


# --------------------------------------------------------------------------
# P3: subspace iteration against a full eigendecomposition
# --------------------------------------------------------------------------

def _principal_cosines(A, B):
    return np.linalg.svd(A.T @ B, compute_uv=False)


@pytest.mark.parametrize("m,n", [(64, 16), (12, 30), (128, 64), (32, 96)])
def test_one_refresh_spans_top_eigenvectors(m, n):
    M = rng(40 + m + n).normal(size=(m, n))
    U, V, ru, rv = orc.refresh_basis(M, np.eye(m), np.eye(n), 1e-3)
    k = min(m, n)
    assert ru == k and rv == k
    wu, Eu = np.linalg.eigh(M @ M.T)
    wv, Ev = np.linalg.eigh(M.T @ M)
    cu = _principal_cosines(U[:, :k], Eu[:, -k:])
    cv = _principal_cosines(V[:, :k], Ev[:, -k:])
    assert np.all(np.arccos(np.clip(cu, -1, 1)) < 1e-7)
    assert np.all(np.arccos(np.clip(cv, -1, 1)) < 1e-7)
    # cos -> angle loses half the digits; the projector difference is exact-ish
    Pu = U[:, :k] @ U[:, :k].T - Eu[:, -k:] @ Eu[:, -k:].T
    assert np.linalg.norm(Pu) < 1e-10
    assert orc.orthogonality_error(U) <= 1e-12 and orc.orthogonality_error(V) <= 1e-12


def test_repeated_refresh_converges_to_eigenvectors():
    m, n = 10, 6
    r = rng(50)
    Uo, _ = np.linalg.qr(r.normal(size=(m, m)))
    Vo, _ = np.linalg.qr(r.normal(size=(n, n)))
    s = np.array([10.0, 6.0, 3.0, 1.5, 0.7, 0.3])
    M = Uo[:, :n] @ np.diag(s) @ Vo.T
    U, V = np.eye(m), np.eye(n)
    for _ in range(40):
        U, V, _, _ = orc.refresh_basis(M, U, V, 1e-6)
    for j in range(3):
        assert abs(abs(U[:, j] @ Uo[:, j]) - 1.0) < 1e-12
        assert abs(abs(V[:, j] @ Vo[:, j]) - 1.0) < 1e-12


# --------------------------------------------------------------------------
# P5: special cases
# --------------------------------------------------------------------------

def test_diagonal_momentum_gives_identity_bases():
    d = np.array([3.0, 1.0, 2.5, 0.5, 4.0])
    M = np.diag(d)
    U, V, ru, rv = orc.refresh_basis(M, np.eye(5), np.eye(5), 1e-3)
    assert np.array_equal(U, np.eye(5)) and np.array_equal(V, np.eye(5))


def test_rank_one_momentum_bases():
    a = rng(60).normal(size=8)
    b = rng(61).normal(size=5)
    M = np.outer(a, b)
    U, V, ru, rv = orc.refresh_basis(M, np.eye(8), np.eye(5), 1e-3)
    assert ru == 1 and rv == 1
    np.testing.assert_allclose(U[:, 0], np.sign(a[0]) * a / np.linalg.norm(a), atol=1e-14)
    np.testing.assert_allclose(V[:, 0], np.sign(b[0]) * b / np.linalg.norm(b), atol=1e-14)


# --------------------------------------------------------------------------
# P6: planner
# --------------------------------------------------------------------------

def test_cost_and_bytes_literals():
    assert orc.item_cost(2, 3) == 65          # 12 + 18 + 8 + 27
    assert orc.item_cost(2048, 2048) == 4 * 2048 ** 3
    assert orc.item_bytes(6144, 2048) == 50331648


def test_planner_hand_worked_two_ranks():
    # costs: (4,4)=256, (3,3)=108, (2,2)=32, (2,1)=15, (1,1)=4
    shapes = [(1, 1), (3, 3), (2, 1), (4, 4), (2, 2)]
    p = orc.plan(shapes, c_max=10 ** 9, ranks=2)
    assert p.groups == [[3, 1, 4, 2, 0]]
    # LPT heap: 256 -> r0; 108 -> r1; 32 -> r1 (108 < 256); 15 -> r1; 4 -> r1
    assert p.owners == [1, 1, 1, 0, 1]
    # byte cap 64 B per rank: (4,4)=64 B on r0, (3,3)=36 B on r1, (2,2)=16 B on r1
    # -> 52 B; (2,1)=8 B on r1 -> 60 B; (1,1)=4 B on r1 -> 64 B: one group
    p = orc.plan(shapes, c_max=64, ranks=2)
    assert p.groups == [[3, 1, 4, 2, 0]]
    # cap 63 B: (4,4) alone holds 64 B, so the next item rolls back and opens
    # group 2, where the heap starts afresh: (3,3) -> r0; (2,2), (2,1), (1,1) -> r1
    p = orc.plan(shapes, c_max=63, ranks=2)
    assert p.groups == [[3], [1, 4, 2, 0]]
    assert p.owners == [1, 0, 1, 0, 1]
    # one rank, cap 60 B: 36 + 16 + 8 = 60 fits, adding 4 B more rolls back
    p = orc.plan(shapes, c_max=60, ranks=1)
    assert p.groups == [[3], [1, 4, 2], [0]]
    assert p.group_bytes == [64, 60, 4] and p.group_cost == [256, 155, 4]


def test_planner_ties_keep_input_order_and_oversize_singletons():
    shapes = [(8, 8), (2, 2), (8, 8), (2, 2), (16, 16)]
    # (16,16) = 1024 B > cap: alone.  (8,8) = 256 B twice exceeds 300 B, so the
    # tied pair splits in input order; 256 + 16 + 16 = 288 B fits.
    p = orc.plan(shapes, c_max=300)
    assert p.groups == [[4], [0], [2, 1, 3]]
    assert orc.plan([], 100).groups == []


def _contiguous_splits(n):
    for mask in range(1 << max(n - 1, 0)):
        cuts = [j + 1 for j in range(n - 1) if mask >> j & 1]
        yield [0] + cuts + [n]


@pytest.mark.parametrize("seed", range(12))
def test_planner_matches_exhaustive_search(seed):
    r = rng(100 + seed)
    count = int(r.integers(1, 9))
    shapes = [(int(r.integers(1, 9)) * 8, int(r.integers(1, 9)) * 8) for _ in range(count)]
    nb = [4 * m * n for m, n in shapes]
    c_max = int(r.integers(min(nb), 2 * sum(nb) // max(1, count // 2) + 1))
    p = orc.plan(shapes, c_max)
    cost = [orc.item_cost(m, n) for m, n in shapes]
    order = sorted(range(count), key=lambda i: (-cost[i], i))
    # LPT order: cost descending, index ascending on ties
    assert [i for g in p.groups for i in g] == order
    # (i) fewest groups among all contiguous splits of the LPT order that obey
    # the cap (a lone item may exceed it) ...
    best = None
    for cuts in _contiguous_splits(count):
        segs = [order[a:b] for a, b in zip(cuts[:-1], cuts[1:])]
        if all(len(s) == 1 or sum(nb[i] for i in s) <= c_max for s in segs):
            if best is None or len(segs) < best:
                best = len(segs)
    assert len(p.groups) == best
    # ... and the split is the maximal-prefix one
    k = 0
    for g in p.groups:
        j = k + 1
        while j < count and sum(nb[i] for i in order[k:j + 1]) <= c_max:
            j += 1
        assert g == order[k:j]
        k = j


@pytest.mark.parametrize("seed", range(6))
def test_lpt_owner_makespan_within_graham_bound(seed):
    r = rng(200 + seed)
    count, R = int(r.integers(3, 9)), int(r.integers(2, 4))
    shapes = [(int(r.integers(1, 7)) * 4, int(r.integers(1, 7)) * 4) for _ in range(count)]
    p = orc.plan(shapes, 10 ** 12, ranks=R)
    cost = [orc.item_cost(m, n) for m, n in shapes]
    loads = [0] * R
    for i, o in enumerate(p.owners):
        loads[o] += cost[i]
    opt = min(max(sum(cost[i] for i in range(count) if a[i] == q) for q in range(R))
              for a in itertools.product(range(R), repeat=count))
    assert max(loads) * 3 * R <= (4 * R - 1) * opt


# --------------------------------------------------------------------------
# Generator sanity (shared inputs): determinism, independence, moments
# --------------------------------------------------------------------------

def test_generator_deterministic_and_keyed():
    wl = inputs.workload("tiny")
    a, b = wl.grad(1, 3), wl.grad(1, 3)
    assert a.dtype == np.float32 and a.shape == (64, 128) and np.array_equal(a, b)
    assert not np.array_equal(wl.grad(1, 4), a) and not np.array_equal(wl.grad(2, 3)[:64, :64], a[:, :64])
    z = inputs.normals(7, 2, 1, 0, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    t = inputs.student_t3(7, 2, 1, 0, 200000)
    assert abs(np.median(t)) < 0.01 and 1.5 < t.std() < 2.0


def test_ragged_shapes():
    wl = inputs.workload("ragged")
    dims = {d for s in wl.shapes for d in s}
    assert wl.count == 256 and dims <= set(range(64, 1025, 64)) and len(dims) == 16


# --------------------------------------------------------------------------
# P9: the float32 floor (oracle against itself, perturbed)
# --------------------------------------------------------------------------

def _small_workload(steps, K, shapes=((24, 16), (16, 24))):
    return inputs.Workload("floorpin", shapes, ("a", "b"), 0.02, 1e-2, "normal", steps, K,
                           1 << 20, 11)


def test_floor_is_zero_without_perturbation():
    wl = _small_workload(4, 2)
    W, _ = orc.run(wl, [0])[0]
    assert orc.floor(wl, 0, W, rel=0.0) == 0.0


def test_floor_is_first_order_in_the_perturbation_where_the_step_is_smooth():
    """No refresh (Adam's D is smooth in its inputs away from G~ = 0, and the
    identity bases rotate nothing): the change of W is linear in the
    perturbation size, so 16 times the size gives 16 times the floor (to
    first order).  Its size: W_T = W_0 - lr sum_t D_t, and each D_t moves by
    about 1.5 u relative (D itself, M~, and half of v's perturbation;
    u = 2^-24), so |dW| ~ lr |D| 1.5 u sqrt(T), with |D| ~ 4.5 over the first
    five steps of Adam without bias correction: relative to |W| = 0.02, about
    0.75 u."""
    wl = _small_workload(5, 100)  # K > steps: plain Adam, U = V = I
    W, _ = orc.run(wl, [1])[1]
    u = 2.0 ** -24
    f24 = orc.floor(wl, 1, W, rel=u)
    f20 = orc.floor(wl, 1, W, rel=16 * u)
    assert 0.25 * u < f24 < 4.0 * u
    assert 14.0 < f20 / f24 < 18.0


def test_floor_large_when_the_first_step_refreshes():
    """Refresh on step 1 (K = 1): v = 0 before the step, so D = M~ / (|G~|
    sqrt(1 - beta2) + eps) ~ 3.16 sgn(G~) is discontinuous in G~ and the rotated
    G~ has entries near zero; rounding-level changes flip some signs and move
    W by far more than the perturbation (the survey's measured 5e-4 .. 2e-3 at
    larger sizes)."""
    wl = _small_workload(3, 1)
    W, _ = orc.run(wl, [0])[0]
    assert orc.floor(wl, 0, W) > 1e3 * 2.0 ** -24


def test_per_quantity_perturbation_sizes():
    """perturb_rels reaches only the named quantities: a size for a name the
    step never forms changes nothing; the compact format's sizes (fp16 bases,
    bf16 moments) move W by much more than float32 rounding; perturbing only
    M at 16 times the size moves W 16 times as far (first order, smooth case)."""
    wl = _small_workload(5, 100)
    W, _ = orc.run(wl, [1])[1]
    u = 2.0 ** -24
    base = orc.floor(wl, 1, W, rel=u)
    assert orc.floor(wl, 1, W, rel=u, rels={"no such quantity": 1.0}) == base
    assert orc.floor(wl, 1, W, rel=u, rels=orc.COMPACT_RELS) > 100 * base
    only_m = orc.floor(wl, 1, W, rel=0.0, rels={"M": 2.0 ** -12})
    only_m16 = orc.floor(wl, 1, W, rel=0.0, rels={"M": 2.0 ** -8})
    assert 14.0 < only_m16 / only_m < 18.0


def test_float32_run_is_a_float32_execution_of_the_same_steps():
    """run(dtype=float32) keeps every array in float32 and lands within a few
    units of float32 rounding of the float64 run where the steps are smooth
    (plain Adam, no refresh: each step adds one rounding of W's size); with
    refreshes it stays close but not exact."""
    u = 2.0 ** -24
    wl = _small_workload(5, 100)
    W, _ = orc.run(wl, [1])[1]
    W32, st = orc.run(wl, [1], dtype=np.float32)[1]
    assert st.M.dtype == np.float32 and st.U.dtype == np.float32
    e = np.linalg.norm(W32 - W) / np.linalg.norm(W)
    assert 0 < e < 8 * u
    wl = _small_workload(6, 2)
    W, st64 = orc.run(wl, [0])[0]
    W32, st32 = orc.run(wl, [0], dtype=np.float32)[0]
    assert (st32.rank_u, st32.rank_v) == (st64.rank_u, st64.rank_v)
    assert 0 < orc.float32_error(wl, 0, W) < 1e-3
    assert orc.orthogonality_error(st32.U.astype(np.float64)) < 1e-5
