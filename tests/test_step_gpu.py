"""GPU parity of rot_step against the fp64 oracle (tiny and ragged-small
workloads), through the C ABI."""

import numpy as np
import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs
from matrix_optimizer_step_rot_gb300.optimizer import RotatedAdam
from oracle import rot_oracle as orc

pytestmark = pytest.mark.gpu

F16 = B.ROT_PREC_3XF16
TOL_W = {B.ROT_PREC_3XTF32: 1e-4, B.ROT_PREC_TF32: 2e-3, F16: 1e-4}
FULL = [B.ROT_PREC_3XTF32, F16]  # the float32-accuracy modes
TOL_ORTH = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    B.lib()


def run_gpu(wl, precision, steps=None, items=None):
    h = wl.hyper
    opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr, h.rank_rtol,
                      precision)
    W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
    for t in range(1, (steps or wl.steps) + 1):
        G = [torch.from_numpy(wl.grad(i, t)).cuda() for i in range(wl.count)]
        opt.step(W, G, wl.refresh(t))
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK
    return W, opt


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def orth(Q):
    Q = Q.astype(np.float64)
    return float(np.linalg.norm(Q.T @ Q - np.eye(Q.shape[1])))


@pytest.mark.parametrize("precision", [B.ROT_PREC_3XTF32, B.ROT_PREC_TF32, F16])
def test_tiny_parity(precision):
    wl = inputs.workload("tiny")
    W, opt = run_gpu(wl, precision)
    ref = orc.run(wl)
    for i in range(wl.count):
        Wo, st = ref[i]
        e = rel(W[i].cpu().numpy().astype(np.float64), Wo)
        assert e <= TOL_W[precision], (i, e)
        U = opt.export(i, B.ROT_WHICH_U).cpu().numpy()
        V = opt.export(i, B.ROT_WHICH_V).cpu().numpy()
        assert orth(U) <= TOL_ORTH and orth(V) <= TOL_ORTH
        assert opt.ranks(i) == (st.rank_u, st.rank_v)
        if precision in FULL:
            M = opt.export(i, B.ROT_WHICH_M).cpu().numpy()
            assert rel(M, st.M) <= 1e-6
            np.testing.assert_allclose(U, st.U, atol=1e-4)
            np.testing.assert_allclose(V, st.V, atol=1e-4)


@pytest.mark.parametrize("precision", FULL)
def test_plain_adam_steps_match_closed_form(precision):
    """Before the first refresh (U = V = I) the GPU step is plain Adam."""
    wl = inputs.workload("tiny")
    W, opt = run_gpu(wl, precision, steps=3)
    h = wl.hyper
    for i in range(wl.count):
        w = wl.w0(i).astype(np.float64)
        m = np.zeros_like(w)
        v = np.zeros_like(w)
        for t in range(1, 4):
            g = wl.grad(i, t).astype(np.float64)
            m = h.beta1 * m + (1 - h.beta1) * g
            v = h.beta2 * v + (1 - h.beta2) * g * g
            w = w - h.lr * m / (np.sqrt(v) + h.eps)
        assert rel(W[i].cpu().numpy().astype(np.float64), w) <= 1e-6


@pytest.mark.parametrize("precision", FULL)
def test_item_larger_than_c_max_runs_in_its_own_group(precision):
    """A matrix above the byte cap (130 x 90: 46800 bytes, C_max 40000) forms a
    group of one (the planner's oversize rule) and steps like the others."""
    shapes = ((130, 90), (60, 40), (40, 60))
    wl = inputs.Workload("oversize", shapes, ("big", "a", "b"), 0.02, 1e-3, "normal", 6, 3,
                         40000, 13)
    W, opt = run_gpu(wl, precision)
    groups = opt.plan.groups()
    assert [0] in groups, groups
    ref = orc.run(wl)
    for i in range(wl.count):
        Wo, st = ref[i]
        e = rel(W[i].cpu().numpy().astype(np.float64), Wo)
        assert e <= TOL_W[precision], (i, shapes[i], e)
        assert opt.ranks(i) == (st.rank_u, st.rank_v), (i, shapes[i])


@pytest.mark.parametrize("precision", FULL)
def test_ragged_small_parity(precision):
    """Shapes that are not multiples of the tile sizes, several groups."""
    shapes = ((100, 36), (36, 100), (97, 97), (1, 40), (40, 1), (130, 70), (33, 65))
    wl = inputs.Workload("ragged_small", shapes, tuple(map(str, range(len(shapes)))), 0.02,
                         1e-3, "t3", 6, 3, 40000, 11)
    W, opt = run_gpu(wl, precision)
    ref = orc.run(wl)
    for i in range(wl.count):
        Wo, st = ref[i]
        e = rel(W[i].cpu().numpy().astype(np.float64), Wo)
        assert e <= TOL_W[precision], (i, shapes[i], e)
        assert opt.ranks(i) == (st.rank_u, st.rank_v), (i, shapes[i])


@pytest.mark.parametrize("precision", FULL)
def test_medium_multi_block_parity(precision):
    """QR inputs wider than one 256-column block (several block reflectors,
    multi-CTA panel clusters), rectangular both ways and square."""
    shapes = ((520, 300), (300, 520), (384, 384), (1030, 260))
    wl = inputs.Workload("medium", shapes, tuple(map(str, range(len(shapes)))), 0.02, 1e-3,
                         "normal", 4, 2, 1 << 30, 21)
    W, opt = run_gpu(wl, precision)
    ref = orc.run(wl)
    for i in range(wl.count):
        Wo, st = ref[i]
        e = rel(W[i].cpu().numpy().astype(np.float64), Wo)
        assert e <= TOL_W[precision], (i, shapes[i], e)
        assert opt.ranks(i) == (st.rank_u, st.rank_v), (i, shapes[i])
        U = opt.export(i, B.ROT_WHICH_U).cpu().numpy()
        V = opt.export(i, B.ROT_WHICH_V).cpu().numpy()
        assert orth(U) <= TOL_ORTH and orth(V) <= TOL_ORTH, (i, orth(U), orth(V))


def scaled_workload(scale):
    hyper = inputs.Hyper(eps=float(np.float32(1e-8 * scale)))
    return inputs.Workload("scaled", ((96, 64), (64, 160)), ("a", "b"), 0.02, 1e-3 * scale,
                           "normal", 4, 2, 1 << 30, 31, hyper)


def arithmetic_allowance(wl, i):
    """What 22-bit product operands allow for matrix i of wl, relative to its
    update (the full-size parity tests' criterion, tests/test_configs_gpu.py):
    A = max(4 F, the spread at 2^-22), F the larger of the float32 run's error
    and the perturbation floor at 2^-24 (five oracle runs each)."""
    w0 = wl.w0(i).astype(np.float64)
    d0 = orc.run(wl, items=[i])[i][0] - w0
    f32 = rel(orc.run(wl, items=[i], dtype=np.float32)[i][0] - w0, d0)
    floor = max(rel(orc.run(wl, items=[i], perturb_seed=s)[i][0] - w0, d0) for s in range(5))
    spread = max(rel(orc.run(wl, items=[i], perturb_seed=s, perturb_rel=2.0 ** -22)[i][0] - w0,
                     d0) for s in range(5))
    return max(4.0 * max(f32, floor), spread)


@pytest.mark.parametrize("precision", FULL)
def test_gradients_of_any_scale(precision):
    """Gradients of order 1e-15 and 1e9 -- far outside fp16's range (its
    smallest subnormal is 6e-8, its largest value 65504), and squared (M M^T U,
    then the QR's column norms) far outside float32's -- with eps scaled alike
    so that Adam's step is the same, match the oracle as at the usual scale:
    3xF16 scales its operands, and the QR its input, by powers of two.  Each
    matrix is held to the bar or, where the method's own sensitivity exceeds
    it, to what 22-bit product operands allow at the usual scale (the 64 x 160
    matrix: float32 run 6.7e-5, spread at 2^-22 2.7e-4).  The sensitivity is
    the same at every scale; the float32 run is taken at the usual scale,
    where plain float32 does not underflow.  A zero gradient leaves W
    unchanged."""
    usual = scaled_workload(1.0)
    allowed = [max(TOL_W[precision], arithmetic_allowance(usual, i)) for i in range(usual.count)]
    for scale in (1e-12, 1e12):
        wl = scaled_workload(scale)
        Wg, _ = run_gpu(wl, precision)
        ref = orc.run(wl)
        for i in range(wl.count):
            w0 = wl.w0(i).astype(np.float64)
            e = rel(Wg[i].cpu().numpy().astype(np.float64) - w0, ref[i][0] - w0)
            print(f"scale {scale:g} matrix {i}: update rel err {e:.3e} (allowed {allowed[i]:.3e})")
            assert e <= allowed[i], (scale, i, e, allowed[i])
    wl = inputs.Workload("zero", usual.shapes, ("a", "b"), 0.02, 0.0, "normal", 3, 2, 1 << 30, 32)
    Wg, opt = run_gpu(wl, precision)
    for i in range(wl.count):
        np.testing.assert_array_equal(Wg[i].cpu().numpy(), wl.w0(i))


@pytest.mark.parametrize("precision", FULL)
def test_non_finite_gradient_stays_in_its_matrix(precision):
    """A NaN in one matrix's gradient (on a refresh step) propagates into that
    matrix's W (IEEE; nothing is reported) and leaves the other matrices of the
    same micro-group equal to the oracle's."""
    wl = inputs.workload("tiny")
    h = wl.hyper
    opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr, h.rank_rtol,
                      precision)
    W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
    for t in range(1, wl.steps + 1):
        G = [torch.from_numpy(wl.grad(i, t)).cuda() for i in range(wl.count)]
        if t == wl.refresh_every:
            G[1][3, 5] = float("nan")
        opt.step(W, G, wl.refresh(t))
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK
    assert torch.isnan(W[1]).any()
    ref = orc.run(wl, [0, 2, 3])
    for i in (0, 2, 3):
        assert torch.isfinite(W[i]).all()
        e = rel(W[i].cpu().numpy().astype(np.float64), ref[i][0])
        assert e <= TOL_W[precision], (i, e)


@pytest.mark.parametrize("precision", FULL)
def test_resume_from_saved_state_is_bit_identical(precision):
    """Checkpoint/resume: the state blob is caller-owned device memory holding
    no pointers, so saving it (and W) after step 3 and resuming in a fresh
    optimizer reproduces the uninterrupted run bit for bit, through a basis
    refresh (t = 5) and plain steps after it."""
    wl = inputs.workload("tiny")
    h = wl.hyper

    def make():
        return RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr,
                           h.rank_rtol, precision)

    def grads(t):
        return [torch.from_numpy(wl.grad(i, t)).cuda() for i in range(wl.count)]

    opt = make()
    W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
    for t in range(1, 4):
        opt.step(W, grads(t), wl.refresh(t))
    saved_state = opt.state.clone()
    saved_W = [w.clone() for w in W]
    for t in range(4, 8):
        opt.step(W, grads(t), wl.refresh(t))

    resumed = make()
    resumed.state.copy_(saved_state)
    W2 = [w.clone() for w in saved_W]
    for t in range(4, 8):
        resumed.step(W2, grads(t), wl.refresh(t))
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK and resumed.status() == B.ROT_OK
    for a, b in zip(W, W2):
        assert torch.equal(a, b)
    for i in range(wl.count):
        for which in (B.ROT_WHICH_M, B.ROT_WHICH_V2, B.ROT_WHICH_U, B.ROT_WHICH_V):
            assert torch.equal(opt.export(i, which), resumed.export(i, which))
