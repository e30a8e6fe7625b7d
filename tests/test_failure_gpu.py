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
