"""Thin ctypes binding of librot.so (include/rot.h).

Argument marshalling only: every step of the optimizer runs in the library's
CUDA kernels.  Device memory comes from the caller (PyTorch tensors are used
for it in the tests and the benchmark); pointers are passed as integers.
The library must have been built (build.build()); there is no other path.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Sequence, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
# the library to load: librot.so, or the file ROT_LIB names (the bounds-checked
# build, librot_check.so, in its tests)
LIB_PATH = os.environ.get("ROT_LIB") or os.path.join(PKG, "librot.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
HEADERS = [os.path.join(INCLUDE, "rot.h"), os.path.join(INCLUDE, "rot_testing.h")]

ROT_OK = 0
ROT_EINVAL = -1
ROT_ENOMEM = -2
ROT_ECUDA = -3
ROT_ETIMEOUT = -4
ROT_ENONFINITE = -5
ROT_ENOTSUP = -6
ROT_ETOOLARGE = -7
ROT_ECORRUPT = -8
ROT_NOALLOC_MAX_BYTES = 64 << 20
ROT_PREC_TF32 = 1
ROT_PREC_3XTF32 = 3
ROT_PREC_3XTF32_PRECISE = 4
ROT_PREC_3XF16 = 5
ROT_TEST_PREC_3XF16_PRECISE = 16  # rot_test_gemm only: the precise kernel on fp16 splits
ROT_WHICH_M, ROT_WHICH_V2, ROT_WHICH_U, ROT_WHICH_V = 0, 1, 2, 3
ROT_STATE_FULL, ROT_STATE_COMPACT = 0, 1


class RotError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class rot_shape(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_u64 = ctypes.c_uint64
_f32 = ctypes.c_float

_SIGS = {
    "rot_plan_create": (_i32, [ctypes.POINTER(rot_shape), _i32, _u64, ctypes.POINTER(_vp)]),
    "rot_plan_create_ex": (_i32, [ctypes.POINTER(rot_shape), _i32, _u64, _i32,
                                  ctypes.POINTER(_vp)]),
    "rot_plan_destroy": (None, [_vp]),
    "rot_plan_groups": (_i32, [_vp, ctypes.POINTER(_i32)]),
    "rot_plan_group": (_i32, [_vp, _i32, ctypes.POINTER(ctypes.POINTER(_i32)),
                              ctypes.POINTER(_i32), ctypes.POINTER(_u64), ctypes.POINTER(_u64)]),
    "rot_plan_owners": (_i32, [_vp, ctypes.POINTER(ctypes.POINTER(_i32))]),
    "rot_state_bytes": (_i32, [_vp, ctypes.POINTER(_u64), ctypes.POINTER(_u64)]),
    "rot_state_init": (_i32, [_vp, _vp, _vp]),
    "rot_step": (_i32, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _vp, _f32, _f32,
                        _f32, _f32, _i32, _i32, _f32, _vp]),
    "rot_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32), _vp]),
    "rot_state_export": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp]),
    "rot_state_ranks": (_i32, [_vp, _vp, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32), _vp]),
    "rot_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "rot_set_wait_timeout_ns": (_u64, [_u64]),
    "rot_set_nonfinite_check": (_i32, [_i32]),
    "rot_launch_count": (_u64, []),
    "rot_plan_set_state_format": (_i32, [_vp, _i32]),
    "rot_profile_enable": (_i32, [_i32]),
    "rot_profile_reset": (_i32, []),
    "rot_profile_read": (_i32, [_i32, ctypes.POINTER(_u64), ctypes.POINTER(ctypes.c_double),
                                ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "rot_step_noalloc": (_i32, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _f32, _f32,
                                _f32, _f32, _i32, _i32, _f32, _vp]),
    "rot_test_gemm": (_i32, [_i32, _i32, _i32, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _f32, _i32,
                             _vp, _u64, _vp, _vp]),
    "rot_test_gemm_work_bytes": (_u64, [_i32, _i32, _i32]),
    "rot_test_guard_offsets": (_i32, [_vp, _i32, ctypes.POINTER(_u64), _i32,
                                      ctypes.POINTER(_i32)]),
    "rot_test_check_guards": (_i32, [_vp, _i32, _vp, _vp, _vp]),
    "rot_test_wait_timeout": (_i32, [_u64, _vp, _vp]),
    "rot_test_fail_host_alloc": (_i32, [ctypes.c_int64]),
    "rot_item_work": (_i32, [ctypes.POINTER(rot_shape), _i32, ctypes.POINTER(_u64)]),
    "rot_partition_static": (_i32, [ctypes.POINTER(_u64), _i32, ctypes.POINTER(_i32), _i32, _i32,
                                    ctypes.POINTER(_i32)]),
    "rot_partition_alpha": (_i32, [ctypes.POINTER(_u64), _i32, ctypes.POINTER(_i32), _i32, _i32,
                                   ctypes.c_double, ctypes.POINTER(_i32), ctypes.POINTER(_u64)]),
    "rot_partition_alpha_ex": (_i32, [ctypes.POINTER(_u64), _i32, ctypes.POINTER(_i32), _i32,
                                      _i32, ctypes.c_double, _i32, ctypes.POINTER(_i32),
                                      ctypes.POINTER(_u64)]),
}


def load_library(path: str) -> ctypes.CDLL:
    """A build of the library at `path` with every entry point's signature set
    (the default build is lib()'s; this also opens the bounds-checked one)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "matrix_optimizer_step_rot_gb300.build.build()")
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    """Load librot.so, or the library ROT_LIB names (raises if it has not been
    built)."""
    global _lib
    if _lib is None:
        _lib = load_library(LIB_PATH)
    return _lib


def header_symbols() -> List[str]:
    """Names of the functions the headers under include/ declare."""
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(rot_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def strerror(code: int) -> str:
    try:
        return lib().rot_strerror(code).decode()
    except Exception:
        return f"error {code}"


def _check(code: int, where: str) -> None:
    if code != ROT_OK:
        raise RotError(code, where)


class Plan:
    """Owns a rot_plan handle."""

    def __init__(self, shapes: Sequence[Tuple[int, int]], c_max: int, ranks: int = 1,
                 state_format: int = 0):
        self.shapes = [(int(m), int(n)) for m, n in shapes]
        arr = (rot_shape * max(1, len(self.shapes)))(*[rot_shape(m, n) for m, n in self.shapes])
        h = _vp()
        _check(lib().rot_plan_create_ex(arr, len(self.shapes), int(c_max), int(ranks),
                                        ctypes.byref(h)), "rot_plan_create_ex")
        self.handle = h
        if state_format:
            _check(lib().rot_plan_set_state_format(h, int(state_format)),
                   "rot_plan_set_state_format")

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.rot_plan_destroy(h)
            self.handle = None

    @property
    def count(self) -> int:
        return len(self.shapes)

    def groups(self) -> List[List[int]]:
        n = _i32()
        _check(lib().rot_plan_groups(self.handle, ctypes.byref(n)), "rot_plan_groups")
        out = []
        for g in range(n.value):
            items = ctypes.POINTER(_i32)()
            k = _i32()
            _check(lib().rot_plan_group(self.handle, g, ctypes.byref(items), ctypes.byref(k),
                                        None, None), "rot_plan_group")
            out.append([items[j] for j in range(k.value)])
        return out

    def group_totals(self, g: int) -> Tuple[int, int]:
        b, c = _u64(), _u64()
        _check(lib().rot_plan_group(self.handle, g, None, None, ctypes.byref(b),
                                    ctypes.byref(c)), "rot_plan_group")
        return b.value, c.value

    def owners(self) -> List[int]:
        o = ctypes.POINTER(_i32)()
        _check(lib().rot_plan_owners(self.handle, ctypes.byref(o)), "rot_plan_owners")
        return [o[i] for i in range(self.count)]

    def state_bytes(self) -> Tuple[int, int]:
        s, w = _u64(), _u64()
        _check(lib().rot_state_bytes(self.handle, ctypes.byref(s), ctypes.byref(w)),
               "rot_state_bytes")
        return s.value, w.value


def item_work(shapes: Sequence[Tuple[int, int]]) -> List[int]:
    """rot_item_work: the planner's cost of each m x n matrix."""
    n = len(shapes)
    arr = (rot_shape * max(n, 1))(*[rot_shape(m, k) for m, k in shapes])
    out = (_u64 * max(n, 1))()
    _check(lib().rot_item_work(arr, n, out), "rot_item_work")
    return [out[i] for i in range(n)]


def partition_static(elems: Sequence[int], bucket_sizes: Sequence[int], ranks: int) -> List[int]:
    """rot_partition_static: owner of every item by its start in its bucket."""
    n, nb = len(elems), len(bucket_sizes)
    e = (_u64 * max(n, 1))(*elems)
    b = (_i32 * max(nb, 1))(*bucket_sizes)
    out = (_i32 * max(n, 1))()
    _check(lib().rot_partition_static(e, n, b, nb, ranks, out), "rot_partition_static")
    return [out[i] for i in range(n)]


ROT_ALPHA_IDEAL_BEFORE, ROT_ALPHA_IDEAL_AFTER = 0, 1


def partition_alpha(work: Sequence[int], bucket_sizes: Sequence[int], ranks: int,
                    alpha: float, ideal: str = "before") -> Tuple[List[int], List[int]]:
    """rot_partition_alpha (ideal "before", the page's rule) or
    rot_partition_alpha_ex with ROT_ALPHA_IDEAL_AFTER (ideal "after"):
    (owner of every item, total work per rank)."""
    n, nb = len(work), len(bucket_sizes)
    w = (_u64 * max(n, 1))(*work)
    b = (_i32 * max(nb, 1))(*bucket_sizes)
    out = (_i32 * max(n, 1))()
    loads = (_u64 * max(ranks, 1))()
    if ideal == "before":
        rc = lib().rot_partition_alpha(w, n, b, nb, ranks, float(alpha), out, loads)
    else:
        code = {"after": ROT_ALPHA_IDEAL_AFTER}.get(ideal, -1)
        rc = lib().rot_partition_alpha_ex(w, n, b, nb, ranks, float(alpha), code, out, loads)
    _check(rc, "rot_partition_alpha")
    return [out[i] for i in range(n)], [loads[r] for r in range(ranks)]


def rot_set_wait_timeout_ns(ns: int) -> int:
    return int(lib().rot_set_wait_timeout_ns(int(ns)))


def rot_test_gemm(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, epi, alpha, precision, work_ptr,
                  work_bytes, status_ptr, stream) -> None:
    _check(lib().rot_test_gemm(M, N, K, _vp(a_ptr), lda, _vp(b_ptr), ldb, _vp(c_ptr), ldc, epi,
                               alpha, precision, _vp(work_ptr), work_bytes, _vp(status_ptr),
                               _vp(stream)), "rot_test_gemm")


def rot_test_gemm_work_bytes(M, N, K) -> int:
    return int(lib().rot_test_gemm_work_bytes(M, N, K))


def rot_state_init(plan: Plan, state_ptr: int, stream: int) -> None:
    _check(lib().rot_state_init(plan.handle, _vp(state_ptr), _vp(stream)), "rot_state_init")


def rot_step(plan: Plan, w_ptrs: Sequence[int], g_ptrs: Sequence[int], state_ptr: int,
             work_ptr: int, beta1: float, beta2: float, eps: float, lr: float, refresh: bool,
             precision: int, rank_rtol: float, stream: int) -> None:
    n = max(1, plan.count)
    W = (_vp * n)(*[_vp(p) for p in w_ptrs])
    G = (_vp * n)(*[_vp(p) for p in g_ptrs])
    _check(lib().rot_step(plan.handle, W, G, _vp(state_ptr), _vp(work_ptr), beta1, beta2, eps,
                          lr, 1 if refresh else 0, precision, rank_rtol, _vp(stream)),
           "rot_step")


def rot_step_noalloc(plan: Plan, w_ptrs: Sequence[int], g_ptrs: Sequence[int], state_ptr: int,
                     beta1: float, beta2: float, eps: float, lr: float, refresh: bool,
                     precision: int, rank_rtol: float, stream: int) -> None:
    """rot_step with its temporaries in the library's static device array."""
    n = max(1, plan.count)
    W = (_vp * n)(*[_vp(p) for p in w_ptrs])
    G = (_vp * n)(*[_vp(p) for p in g_ptrs])
    _check(lib().rot_step_noalloc(plan.handle, W, G, _vp(state_ptr), beta1, beta2, eps, lr,
                                  1 if refresh else 0, precision, rank_rtol, _vp(stream)),
           "rot_step_noalloc")


def rot_status(plan: Plan, state_ptr: int, stream: int) -> int:
    st = _i32()
    _check(lib().rot_status(plan.handle, _vp(state_ptr), ctypes.byref(st), _vp(stream)),
           "rot_status")
    return st.value


def rot_state_export(plan: Plan, state_ptr: int, item: int, which: int, dst_ptr: int,
                     stream: int) -> None:
    _check(lib().rot_state_export(plan.handle, _vp(state_ptr), item, which, _vp(dst_ptr),
                                  _vp(stream)), "rot_state_export")


def rot_state_ranks(plan: Plan, state_ptr: int, item: int, stream: int) -> Tuple[int, int]:
    ru, rv = _i32(), _i32()
    _check(lib().rot_state_ranks(plan.handle, _vp(state_ptr), item, ctypes.byref(ru),
                                 ctypes.byref(rv), _vp(stream)), "rot_state_ranks")
    return ru.value, rv.value
