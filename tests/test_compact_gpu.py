"""Reduced-precision state (ROT_STATE_COMPACT): the first moments M and M~ in
bf16, v in float32 (the ZeRO essay, section 3.3) and every basis as a single
fp16 (the rotation page, section 3.1).

Its tolerance is the method's own spread at those precisions: the largest
relative change of W over five oracle runs whose stored quantities are
perturbed at the format's rounding (2^-11 for U and V, 2^-8 for M and M~,
2^-24 for the rest; oracle.COMPACT_RELS).  A GPU run in this format must stay
within that spread.  The bases' orthogonality is held to what fp16 storage
of an orthogonal matrix gives: sqrt(2) 2^-11 sqrt(p) (rounding each of the
p^2 entries by up to 2^-11 relative), not to the float32 bar."""

import math

import numpy as np
import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs
from matrix_optimizer_step_rot_gb300.optimizer import RotatedAdam
from oracle import rot_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    B.lib()


def run_gpu(wl, sampled, precision):
    h = wl.hyper
    opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr, h.rank_rtol,
                      precision, state_format=B.ROT_STATE_COMPACT)
    gen = torch.Generator(device="cuda").manual_seed(777)
    W = [torch.from_numpy(wl.w0(i)).cuda() if i in sampled
         else torch.randn(m, n, device="cuda", generator=gen) * wl.w_std
         for i, (m, n) in enumerate(wl.shapes)]
    for t in range(1, wl.steps + 1):
        G = [torch.from_numpy(wl.grad(i, t)).cuda() if i in sampled
             else torch.randn(m, n, device="cuda", generator=gen) * wl.g_std
             for i, (m, n) in enumerate(wl.shapes)]
        opt.step(W, G, wl.refresh(t))
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK
    return W, opt


def check(wl, items, precision):
    W, opt = run_gpu(wl, set(items), precision)
    ref = orc.run(wl, items)
    for i in items:
        Wo, st = ref[i]
        e = float(np.linalg.norm(W[i].cpu().numpy().astype(np.float64) - Wo) / np.linalg.norm(Wo))
        fl = orc.floor(wl, i, Wo, rels=orc.COMPACT_RELS)
        print(f"compact {wl.name}[{i}] {wl.shapes[i]} prec {precision}: W rel err {e:.2e}, "
              f"spread at the compact format's precision {fl:.2e}")
        assert e <= fl, (i, e, fl)
        for which, p in ((B.ROT_WHICH_U, wl.shapes[i][0]), (B.ROT_WHICH_V, wl.shapes[i][1])):
            Q = opt.export(i, which).double()
            o = float(torch.linalg.norm(Q.T @ Q - torch.eye(p, dtype=torch.float64,
                                                             device=Q.device)))
            assert o <= math.sqrt(2.0) * 2.0 ** -11 * math.sqrt(p), (i, which, o)
        # the exported momentum is the bf16 state, within bf16 rounding of the oracle's
        Mg = opt.export(i, B.ROT_WHICH_M).double().cpu().numpy()
        assert np.linalg.norm(Mg - st.M) <= 2.0 ** -7 * np.linalg.norm(st.M)


@pytest.mark.parametrize("precision", [B.ROT_PREC_3XF16, B.ROT_PREC_3XTF32])
def test_compact_tiny_within_its_spread(precision):
    check(inputs.workload("tiny"), [0, 1, 2, 3], precision)


def test_compact_block_k_proj_within_its_spread():
    check(inputs.workload("block"), [1], B.ROT_PREC_3XF16)  # k_proj 1024 x 2048
