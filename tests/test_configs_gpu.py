"""Parity on the five workloads at their full sizes, in the launch
configuration the benchmark uses (the real plan: same micro-groups, same
grouped launches), in both float32-accuracy modes (3xTF32 and 3xF16).

Matrices are independent, so the oracle runs on a sample of each workload's
matrices (their inputs come from the shared seeded generator); the other
matrices get device-random inputs.  Every matrix's bases are checked for
orthogonality.  W is held to the 1e-4 bar (3xTF32); where a matrix misses it,
the method's own floor for that matrix is measured with the oracle (the same
run with its QR inputs perturbed at float32 rounding level, five seeds, the
largest change kept) and the GPU's error must stay within the bar plus three
times that floor.
Every number is printed and appended to parity_results.txt in the directory
named by ROT_PARITY_LOG (if set).
"""

import os

import numpy as np
import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs
from matrix_optimizer_step_rot_gb300.optimizer import RotatedAdam
from oracle import build_oracle
from oracle import rot_oracle as orc

pytestmark = pytest.mark.gpu

BAR_W = 1e-4
BAR_ORTH = 1e-4
FLOOR_FACTOR = 3.0
FULL = [B.ROT_PREC_3XTF32, B.ROT_PREC_3XF16]  # float32-accuracy modes, 1e-4 bar

# the oracle's results and floors do not depend on the GPU's precision mode:
# computed once per workload and shared by the modes' tests
_ORACLE = {}
_FLOOR = {}


def oracle_run(wl, sampled, steps):
    key = (wl.name, tuple(sampled), steps)
    if key not in _ORACLE:
        _ORACLE[key] = orc.run(wl, sampled, steps=steps)
    return _ORACLE[key]


def oracle_floor(wl, i, Wo, steps):
    key = (wl.name, i, steps)
    if key not in _FLOOR:
        _FLOOR[key] = orc.floor(wl, i, Wo, seeds=(1, 2, 3, 4, 5), steps=steps)
    return _FLOOR[key]


def orth_bound(p):
    """||Q^T Q - I||_F bound for a p x p basis.  1e-4 up to p = 8192.  Beyond,
    the float32 floor of the blocked Householder Q formation itself takes over:
    a CPU emulation of the same 128-wide backward accumulation in float32, with
    exact partial sums, grows linearly in p (2.1e-5 at 2048, 4.1e-5 at 4096,
    ~1.2e-4 at 12288), so the bound there is 1.5x that growth, 1.5e-8 * p."""
    return max(BAR_ORTH, 1.5e-8 * p)


def log(line):
    print(line)
    d = os.environ.get("ROT_PARITY_LOG")
    if d:
        with open(os.path.join(d, "parity_results.txt"), "a") as f:
            f.write(line + "\n")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    build_oracle.build()
    B.lib()


def run_gpu(wl, sampled, precision=B.ROT_PREC_3XTF32, steps=None):
    h = wl.hyper
    opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr, h.rank_rtol,
                      precision)
    gen = torch.Generator(device="cuda").manual_seed(12345)
    W = []
    for i, (m, n) in enumerate(wl.shapes):
        if i in sampled:
            W.append(torch.from_numpy(wl.w0(i)).cuda())
        else:
            W.append(torch.randn(m, n, device="cuda", generator=gen) * wl.w_std)
    for t in range(1, (steps or wl.steps) + 1):
        G = []
        for i, (m, n) in enumerate(wl.shapes):
            if i in sampled:
                G.append(torch.from_numpy(wl.grad(i, t)).cuda())
            else:
                G.append(torch.randn(m, n, device="cuda", generator=gen) * wl.g_std)
        opt.step(W, G, wl.refresh(t))
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK
    return W, opt


def orth_gpu(opt, item, which):
    Q = opt.export(item, which).double()
    eye = torch.eye(Q.shape[0], dtype=torch.float64, device=Q.device)
    return float(torch.linalg.norm(Q.T @ Q - eye))


def check(wl, sampled, precision=B.ROT_PREC_3XTF32, bar=BAR_W, steps=None):
    W, opt = run_gpu(wl, set(sampled), precision, steps)
    refreshed = any(wl.refresh(t) for t in range(1, (steps or wl.steps) + 1))
    if refreshed:
        worst, excess = 0.0, 0.0
        for i, (m, n) in enumerate(wl.shapes):
            for which, pdim in ((B.ROT_WHICH_U, m), (B.ROT_WHICH_V, n)):
                o = orth_gpu(opt, i, which)
                worst = max(worst, o)
                excess = max(excess, o / orth_bound(pdim))
        log(f"{wl.name}: max ||Q^T Q - I||_F over {wl.count} matrices = {worst:.2e} "
            f"(largest ratio to its bound {excess:.2f})")
        assert excess <= 1.0
    ref = oracle_run(wl, sampled, steps)
    for i in sampled:
        Wo, st = ref[i]
        e = float(np.linalg.norm(W[i].cpu().numpy().astype(np.float64) - Wo) / np.linalg.norm(Wo))
        if refreshed:
            assert opt.ranks(i) == (st.rank_u, st.rank_v), (i, wl.shapes[i])
        if e <= bar:
            log(f"{wl.name}[{i}] {wl.shapes[i]} prec {precision}: W rel err {e:.2e} <= {bar:.0e}")
            continue
        fl = oracle_floor(wl, i, Wo, steps)
        log(f"{wl.name}[{i}] {wl.shapes[i]} prec {precision}: W rel err {e:.2e} > {bar:.0e}; "
            f"method floor (oracle, float32-level QR-input perturbation) {fl:.2e}")
        assert e <= bar + FLOOR_FACTOR * fl, (i, e, fl)


@pytest.mark.parametrize("precision", FULL)
def test_block_parity(precision):
    wl = inputs.workload("block")
    check(wl, [0, 1, 4], precision)  # q_proj, k_proj, gate


def test_block_parity_tf32():
    wl = inputs.workload("block")
    check(wl, [1], precision=B.ROT_PREC_TF32, bar=2e-3)


@pytest.mark.parametrize("precision", FULL)
def test_full_stack_sampled(precision):
    wl = inputs.workload("full")
    check(wl, [1, 7 * 13 + 2, 7 * 27], precision)  # L0.k_proj, L13.v_proj, L27.q_proj


@pytest.mark.parametrize("precision", FULL)
def test_slice8b_sampled(precision):
    wl = inputs.workload("slice8b")
    check(wl, [1], precision)  # L0.k_proj 1024 x 4096, refresh on every step


@pytest.mark.parametrize("precision", FULL)
def test_ragged_sampled(precision):
    wl = inputs.workload("ragged")
    check(wl, list(range(0, 256, 11)), precision)
