"""The bounds-checked build (librot_check.so, compiled with ROT_CHECK): the
plan's guard regions, host-side (the survey's test strategy: canary words
around every workspace slice).  Its device checks run in
tests/test_check_build_gpu.py."""

import ctypes

import pytest

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs


@pytest.fixture(scope="module")
def libs():
    plain = B.load_library(build.build())
    checked = B.load_library(build.build(check=True))
    return plain, checked


def plan_of(L, shapes, c_max):
    arr = (B.rot_shape * len(shapes))(*[B.rot_shape(m, n) for m, n in shapes])
    handle = ctypes.c_void_p()
    assert L.rot_plan_create(arr, len(shapes), c_max, ctypes.byref(handle)) == B.ROT_OK
    sb, wb = ctypes.c_uint64(), ctypes.c_uint64()
    assert L.rot_state_bytes(handle, ctypes.byref(sb), ctypes.byref(wb)) == B.ROT_OK
    ng = ctypes.c_int32()
    assert L.rot_plan_groups(handle, ctypes.byref(ng)) == B.ROT_OK
    return handle, sb.value, wb.value, ng.value


def guards(L, handle, group):
    n = ctypes.c_int32()
    assert L.rot_test_guard_offsets(handle, group, None, 0, ctypes.byref(n)) == B.ROT_OK
    buf = (ctypes.c_uint64 * max(n.value, 1))()
    assert L.rot_test_guard_offsets(handle, group, buf, n.value, ctypes.byref(n)) == B.ROT_OK
    return list(buf[:n.value])


@pytest.mark.parametrize("name", ["tiny", "block"])
def test_every_workspace_slice_is_followed_by_a_guard(libs, name):
    plain, checked = libs
    wl = inputs.workload(name)
    hp, sb_p, wb_p, ng_p = plan_of(plain, wl.shapes, wl.c_max)
    hc, sb_c, wb_c, ng_c = plan_of(checked, wl.shapes, wl.c_max)
    try:
        # the same grouping and state; the workspace grows by the guards
        assert (ng_c, sb_c) == (ng_p, sb_p)
        assert wb_c > wb_p
        n = ctypes.c_int32()
        assert plain.rot_test_guard_offsets(hp, 0, None, 0, ctypes.byref(n)) == B.ROT_ENOTSUP
        for g in range(ng_c):
            offs = guards(checked, hc, g)
            assert offs, g
            # ascending, 256-byte aligned, 256 bytes each, inside the workspace,
            # and never adjacent: a slice lies between consecutive guards
            assert all(o % 256 == 0 for o in offs)
            assert all(b - a > 256 for a, b in zip(offs, offs[1:]))
            assert offs[-1] + 256 <= wb_c
        assert checked.rot_test_guard_offsets(hc, ng_c, None, 0, ctypes.byref(n)) == B.ROT_EINVAL
    finally:
        plain.rot_plan_destroy(hp)
        checked.rot_plan_destroy(hc)
