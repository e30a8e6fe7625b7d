"""Runs steps through whichever library build ROT_LIB names (for
tests/test_check_build_gpu.py, one process per build).

    python tests/check_build_worker.py steps OUT.npz   # seeded steps, W and status to OUT
    python tests/check_build_worker.py corrupt         # overwrite a guard, print the status
"""

import ctypes
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from matrix_optimizer_step_rot_gb300 import binding as B  # noqa: E402
from matrix_optimizer_step_rot_gb300.optimizer import RotatedAdam  # noqa: E402

# several micro-groups (C_max 4 MB), bases of one to three 256-column blocks
SHAPES = [(64, 96), (600, 700), (300, 520), (520, 300), (128, 1000), (700, 600)]


def optimizer():
    return RotatedAdam(SHAPES, 4 << 20, "cuda", 0.9, 0.999, 1e-8, 1e-3, 1e-3, B.ROT_PREC_3XF16)


def steps(out):
    opt = optimizer()
    g = torch.Generator(device="cuda").manual_seed(5)
    W = [torch.randn(m, n, device="cuda", generator=g) * 0.02 for m, n in SHAPES]
    for t in range(1, 5):
        G = [torch.randn(m, n, device="cuda", generator=g) * 1e-2 for m, n in SHAPES]
        opt.step(W, G, t % 2 == 0)  # refreshes on steps 2 and 4
    torch.cuda.synchronize()
    np.savez(out, status=opt.status(), **{f"w{i}": w.cpu().numpy() for i, w in enumerate(W)})


def corrupt():
    opt = optimizer()
    g = torch.Generator(device="cuda").manual_seed(5)
    W = [torch.randn(m, n, device="cuda", generator=g) * 0.02 for m, n in SHAPES]
    G = [torch.randn(m, n, device="cuda", generator=g) * 1e-2 for m, n in SHAPES]
    opt.step(W, G, True)
    torch.cuda.synchronize()
    before = opt.status()
    n = ctypes.c_int32()
    L = B.lib()
    assert L.rot_test_guard_offsets(opt.plan.handle, 0, None, 0, ctypes.byref(n)) == B.ROT_OK
    buf = (ctypes.c_uint64 * n.value)()
    assert L.rot_test_guard_offsets(opt.plan.handle, 0, buf, n.value, ctypes.byref(n)) == B.ROT_OK
    off = int(buf[n.value // 2])
    opt.work[off:off + 4] = 0  # a write past the end of a slice
    stream = torch.cuda.current_stream().cuda_stream
    assert L.rot_test_check_guards(opt.plan.handle, 0, ctypes.c_void_p(opt.state.data_ptr()),
                                   ctypes.c_void_p(opt.work.data_ptr()),
                                   ctypes.c_void_p(stream)) == B.ROT_OK
    torch.cuda.synchronize()
    print(before, opt.status())


if __name__ == "__main__":
    if sys.argv[1] == "steps":
        steps(sys.argv[2])
    else:
        corrupt()
