"""Failure detection without a GPU fault: a device-side wait that can never be
satisfied gives up after its limit and reports ROT_ETIMEOUT; the context
stays usable afterwards.  Host-side argument errors are covered in
test_capi_cpu.py."""

import time

import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs
from matrix_optimizer_step_rot_gb300.optimizer import RotatedAdam

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    B.lib()


def test_bounded_wait_times_out_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    assert B.lib().rot_test_wait_timeout(50_000_000, B._vp(status.data_ptr()),
                                         B._vp(stream)) == B.ROT_OK
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert int(status.item()) == B.ROT_ETIMEOUT
    assert 0.04 <= took < 5.0
    # the context is still usable: a normal step runs and reports no error
    wl = inputs.workload("tiny")
    h = wl.hyper
    opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr, h.rank_rtol)
    W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
    G = [torch.from_numpy(wl.grad(i, 1)).cuda() for i in range(wl.count)]
    opt.step(W, G, False)
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK
    assert all(torch.isfinite(w).all() for w in W)


def test_wait_limit_argument_checks():
    assert B.lib().rot_test_wait_timeout(1000, None, None) == B.ROT_EINVAL
    old = B.rot_set_wait_timeout_ns(1_500_000_000)
    assert B.rot_set_wait_timeout_ns(old) == 1_500_000_000


@pytest.mark.parametrize("precision", [B.ROT_PREC_3XF16, B.ROT_PREC_3XTF32])
def test_nonfinite_check_reports_a_nan_gradient(precision):
    """With the check on, a NaN in one gradient makes rot_status report
    ROT_ENONFINITE once (the read clears it); with the check off, the same
    step reports ROT_OK.  The values propagate either way (IEEE)."""
    wl = inputs.workload("tiny")
    h = wl.hyper
    old = B.lib().rot_set_nonfinite_check(0)
    try:
        for on in (1, 0):
            B.lib().rot_set_nonfinite_check(on)
            opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr,
                              h.rank_rtol, precision)
            W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
            G = [torch.from_numpy(wl.grad(i, 1)).cuda() for i in range(wl.count)]
            opt.step(W, G, False)  # clean step first
            assert opt.status() == B.ROT_OK
            G[2][1, 3] = float("nan")
            opt.step(W, G, False)
            torch.cuda.synchronize()
            assert opt.status() == (B.ROT_ENONFINITE if on else B.ROT_OK)
            assert opt.status() == B.ROT_OK  # cleared by the read
            assert torch.isnan(W[2]).any()
            assert all(torch.isfinite(W[i]).all() for i in (0, 1, 3))
            G2 = [torch.from_numpy(wl.grad(i, 2)).cuda() for i in range(wl.count)]
            G2[0][0, 0] = float("inf")  # an infinity is reported too
            opt.step(W, G2, False)
            assert opt.status() == (B.ROT_ENONFINITE if on else B.ROT_OK)
    finally:
        B.lib().rot_set_nonfinite_check(old)


def test_nonfinite_check_silent_on_large_finite_gradients():
    """Gradients of 1e30 square to infinity in the row norms, but are finite:
    no report."""
    wl = inputs.workload("tiny")
    h = wl.hyper
    old = B.lib().rot_set_nonfinite_check(1)
    try:
        opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr,
                          h.rank_rtol, B.ROT_PREC_3XF16)
        W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
        G = [torch.from_numpy(wl.grad(i, 1)).cuda() * 1e30 for i in range(wl.count)]
        opt.step(W, G, False)
        assert opt.status() == B.ROT_OK
    finally:
        B.lib().rot_set_nonfinite_check(old)


def test_step_reports_host_allocation_failure_before_device_work():
    """The step's first host allocation fails: ROT_ENOMEM, no kernel launched,
    W and the state untouched; the next step runs normally."""
    wl = inputs.workload("tiny")
    h = wl.hyper
    opt = RotatedAdam(wl.shapes, wl.c_max, "cuda", h.beta1, h.beta2, h.eps, h.lr, h.rank_rtol)
    W = [torch.from_numpy(wl.w0(i)).cuda() for i in range(wl.count)]
    W0 = [w.clone() for w in W]
    G = [torch.from_numpy(wl.grad(i, 1)).cuda() for i in range(wl.count)]
    torch.cuda.synchronize()
    launches = B.lib().rot_launch_count()
    B.lib().rot_test_fail_host_alloc(0)
    try:
        with pytest.raises(B.RotError) as e:
            opt.step(W, G, False)
    finally:
        B.lib().rot_test_fail_host_alloc(-1)
    assert e.value.code == B.ROT_ENOMEM
    torch.cuda.synchronize()
    assert B.lib().rot_launch_count() == launches
    assert all(torch.equal(a, b) for a, b in zip(W, W0))
    opt.step(W, G, False)
    torch.cuda.synchronize()
    assert opt.status() == B.ROT_OK
    assert not all(torch.equal(a, b) for a, b in zip(W, W0))
