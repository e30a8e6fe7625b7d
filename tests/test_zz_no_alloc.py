"""rot_step_noalloc: the step for callers that cannot allocate device memory
(its temporaries live in a static device array inside the library instead of
a caller-provided workspace).  Checked against rot_step, the entry point that
takes a workspace, on two calls in a row, through the C ABI.  This file is
named to be collected last."""

import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    B.lib()


def test_empty_plan_is_a_no_op_without_a_device():
    """An empty plan returns ROT_OK before any device query, as rot_step does."""
    plan = B.Plan([], 1 << 20)
    rc = B.lib().rot_step_noalloc(plan.handle, None, None, None, 0.9, 0.999, 1e-8, 1e-3, 0,
                                  B.ROT_PREC_3XTF32, 1e-3, None)
    assert rc == B.ROT_OK


def test_argument_errors_come_before_device_work():
    """Bad arguments are refused as rot_step refuses them, with no GPU needed."""
    plan = B.Plan([(64, 64)], 1 << 20)
    rc = B.lib().rot_step_noalloc(plan.handle, None, None, None, 0.9, 0.999, 1e-8, 1e-3, 0,
                                  B.ROT_PREC_3XTF32, 1e-3, None)
    assert rc == B.ROT_EINVAL
    W = (B._vp * 1)(B._vp(256))
    rc = B.lib().rot_step_noalloc(plan.handle, W, W, B._vp(256), 0.9, 0.999, 1e-8, 1e-3, 0,
                                  99, 1e-3, None)
    assert rc == B.ROT_EINVAL


def test_rejects_plans_beyond_the_static_scratch():
    """A plan whose workspace exceeds the array is refused before device work."""
    plan = B.Plan([(4096, 4096)], 1 << 30)
    assert plan.state_bytes()[1] > B.ROT_NOALLOC_MAX_BYTES
    W = (B._vp * 1)(B._vp(256))
    rc = B.lib().rot_step_noalloc(plan.handle, W, W, B._vp(256), 0.9, 0.999, 1e-8, 1e-3, 0,
                                  B.ROT_PREC_3XTF32, 1e-3, None)
    assert rc == B.ROT_ETOOLARGE
    assert "no-allocation" in B.strerror(rc)


@pytest.mark.gpu
def test_noalloc_step_matches_workspace_step_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = inputs.workload("tiny")
    h = wl.hyper
    plan = B.Plan(wl.shapes, wl.c_max)
    sb, wb = plan.state_bytes()
    assert wb <= B.ROT_NOALLOC_MAX_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    states = [torch.empty(sb, dtype=torch.uint8, device="cuda") for _ in range(2)]
    work = torch.empty(wb, dtype=torch.uint8, device="cuda")
    for s in states:
        B.rot_state_init(plan, s.data_ptr(), stream)
    W = [[torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)] for _ in range(2)]
    # two calls in a row: a plain step, then a step with the basis refresh, so
    # both the rotation's and the QR's temporaries pass through the array
    for t, refresh in ((1, False), (2, True)):
        G = [torch.from_numpy(wl.grad(i, t)).cuda() for i in range(wl.count)]
        B.rot_step(plan, [w.data_ptr() for w in W[0]], [g.data_ptr() for g in G],
                   states[0].data_ptr(), work.data_ptr(), h.beta1, h.beta2, h.eps, h.lr,
                   refresh, B.ROT_PREC_3XTF32, h.rank_rtol, stream)
        B.rot_step_noalloc(plan, [w.data_ptr() for w in W[1]], [g.data_ptr() for g in G],
                           states[1].data_ptr(), h.beta1, h.beta2, h.eps, h.lr, refresh,
                           B.ROT_PREC_3XTF32, h.rank_rtol, stream)
        torch.cuda.synchronize()
        assert B.rot_status(plan, states[1].data_ptr(), stream) == B.ROT_OK
        # the two calls differ only in where the temporaries live; every kernel
        # accumulates in a fixed order, so the results agree bit for bit (a
        # read of stale scratch left by the previous call would break this)
        for i in range(wl.count):
            assert torch.equal(W[0][i], W[1][i]), (t, i)
        for i in range(wl.count):
            for which in (B.ROT_WHICH_U, B.ROT_WHICH_V):
                m, n = wl.shapes[i]
                p = m if which == B.ROT_WHICH_U else n
                outs = []
                for s in states:
                    o = torch.empty(p, p, device="cuda")
                    B.rot_state_export(plan, s.data_ptr(), i, which, o.data_ptr(), stream)
                    outs.append(o)
                torch.cuda.synchronize()
                assert torch.equal(outs[0], outs[1]), (t, i, which)
