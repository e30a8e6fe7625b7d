"""CPU checks of the C-ABI library: it loads, exports every declared symbol,
and its host planner matches the oracle's plan bit for bit."""

import ctypes
import importlib.util
import os
import re

import numpy as np
import pytest

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs
from oracle import rot_oracle as orc


@pytest.fixture(scope="module", autouse=True)
def built_library():
    build.build()
    B.lib()


def test_exports_every_declared_symbol():
    names = B.header_symbols()
    assert len(names) >= 12
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n


@pytest.mark.parametrize("name", inputs.WORKLOADS)
def test_plan_bit_exact_against_oracle(name):
    wl = inputs.workload(name)
    p = B.Plan(wl.shapes, wl.c_max)
    o = orc.plan(wl.shapes, wl.c_max)
    assert p.groups() == o.groups
    assert p.owners() == o.owners
    for g in range(len(o.groups)):
        assert p.group_totals(g) == (o.group_bytes[g], o.group_cost[g])


@pytest.mark.parametrize("seed", range(40))
def test_plan_fuzz_against_oracle(seed):
    r = np.random.default_rng(1000 + seed)
    count = int(r.integers(0, 60))
    shapes = [(int(r.integers(1, 300)), int(r.integers(1, 300))) for _ in range(count)]
    if seed % 5 == 0:  # many ties
        shapes = [shapes[j % 3] for j in range(count)] if count >= 3 else shapes
    ranks = int(r.integers(1, 5))
    c_max = int(r.integers(1, 400000))
    p = B.Plan(shapes, c_max, ranks=ranks)
    o = orc.plan(shapes, c_max, ranks=ranks)
    assert p.groups() == o.groups and p.owners() == o.owners


def test_large_dims_cost_is_exact():
    shapes = [(65536, 65536), (65536, 1), (1, 65536), (12288, 4096)]
    p = B.Plan(shapes, 1 << 40)
    o = orc.plan(shapes, 1 << 40)
    assert p.groups() == o.groups and p.group_totals(0) == (o.group_bytes[0], o.group_cost[0])


def test_argument_errors():
    L = B.lib()
    h = ctypes.c_void_p()
    good = (B.rot_shape * 1)(B.rot_shape(4, 4))
    assert L.rot_plan_create(good, 1, 0, ctypes.byref(h)) == B.ROT_EINVAL       # c_max = 0
    assert L.rot_plan_create(good, -1, 10, ctypes.byref(h)) == B.ROT_EINVAL
    assert L.rot_plan_create(None, 1, 10, ctypes.byref(h)) == B.ROT_EINVAL
    assert L.rot_plan_create(good, 1, 10, None) == B.ROT_EINVAL
    for bad in [(0, 4), (4, 0), (-3, 4), (65537, 2)]:
        arr = (B.rot_shape * 1)(B.rot_shape(*bad))
        assert L.rot_plan_create(arr, 1, 10, ctypes.byref(h)) == B.ROT_EINVAL
        assert h.value is None
    assert L.rot_plan_create_ex(good, 1, 10, 0, ctypes.byref(h)) == B.ROT_EINVAL
    n = ctypes.c_int32()
    assert L.rot_plan_groups(None, ctypes.byref(n)) == B.ROT_EINVAL
    p = B.Plan([(4, 4)], 10)
    assert L.rot_plan_group(p.handle, 5, None, None, None, None) == B.ROT_EINVAL
    assert L.rot_plan_group(p.handle, -1, None, None, None, None) == B.ROT_EINVAL
    # the step validates its arguments before touching the device
    W = (ctypes.c_void_p * 1)(ctypes.c_void_p(256))
    assert L.rot_step(p.handle, W, W, ctypes.c_void_p(256), ctypes.c_void_p(512), 0.9, 0.999,
                      1e-8, 1e-3, 0, 2, 1e-3, None) == B.ROT_EINVAL          # precision
    assert L.rot_step(p.handle, W, W, ctypes.c_void_p(256), ctypes.c_void_p(512), 0.9, 0.999,
                      1e-8, 1e-3, 0, 3, 0.0, None) == B.ROT_EINVAL           # rank_rtol
    assert L.rot_step(p.handle, W, W, ctypes.c_void_p(100), ctypes.c_void_p(512), 0.9, 0.999,
                      1e-8, 1e-3, 0, 3, 1e-3, None) == B.ROT_EINVAL          # alignment
    assert L.rot_step(p.handle, None, W, ctypes.c_void_p(256), ctypes.c_void_p(512), 0.9,
                      0.999, 1e-8, 1e-3, 0, 3, 1e-3, None) == B.ROT_EINVAL
    assert L.rot_state_export(p.handle, ctypes.c_void_p(256), 1, 0, ctypes.c_void_p(256),
                              None) == B.ROT_EINVAL
    assert L.rot_state_export(p.handle, ctypes.c_void_p(256), 0, 7, ctypes.c_void_p(256),
                              None) == B.ROT_EINVAL
    # the test GEMM validates before any device work: unknown precision, and
    # the untransposed split outputs, which have no fp16 form
    vp = ctypes.c_void_p
    for prec, epi in [(2, 2), (B.ROT_PREC_3XF16, 0), (B.ROT_PREC_3XF16, 5)]:
        assert L.rot_test_gemm(32, 32, 32, vp(256), 32, vp(256), 32, vp(256), 32, epi, 1.0, prec,
                               vp(256), 1 << 20, None, None) == B.ROT_EINVAL
    assert B.strerror(B.ROT_EINVAL) == "invalid argument"


def test_empty_plan_and_state_sizes():
    p = B.Plan([], 100)
    assert p.groups() == []
    wl = inputs.workload("tiny")
    p = B.Plan(wl.shapes, wl.c_max)
    sb, wb = p.state_bytes()
    # state: M, v, M~ in float32 and fp16 splits of U, U^T, V, V^T per matrix
    # (rows padded to 32 elements), a 256-byte status header, the ranks
    need = sum(4 * 3 * m * n + 8 * (m * m + n * n) for m, n in wl.shapes)
    pad = lambda x: (x + 31) // 32 * 32
    most = 256 + 256 + sum(4 * 3 * m * pad(n) + 8 * (m * pad(m) + n * pad(n)) + 7 * 256
                           for m, n in wl.shapes)
    assert need <= sb <= most and sb % 256 == 0 and wb > 0


def test_state_is_within_twice_the_algorithmic_state():
    """M, v, U, V in float32 is the method's own state; this layout keeps M~
    (the incremental rotated momentum) beside it and each basis in two
    orientations at 4 bytes per element: at most twice the algorithmic bytes
    on the Qwen3-shaped workloads."""
    for name in ("full", "slice8b", "block"):
        wl = inputs.workload(name)
        algorithmic = sum(4 * (2 * m * n + m * m + n * n) for m, n in wl.shapes)
        sb, _ = B.Plan(wl.shapes, wl.c_max).state_bytes()
        assert sb <= 2 * algorithmic, (name, sb / algorithmic)


def test_host_checked_edge_cases():
    """Cases the step settles on the host, before any device work."""
    L = B.lib()
    vp = ctypes.c_void_p
    # an empty plan: nothing to do
    p = B.Plan([], 100)
    assert L.rot_step(p.handle, None, None, None, None, 0.9, 0.999, 1e-8, 1e-3, 1, 3, 1e-3,
                      None) == B.ROT_OK
    # a refresh of a basis larger than the QR takes (16 x 1536 = 24576 rows)
    p = B.Plan([(24577, 8)], 1 << 40)
    W = (vp * 1)(vp(256))
    assert L.rot_step(p.handle, W, W, vp(256), vp(512), 0.9, 0.999, 1e-8, 1e-3, 1, 3, 1e-3,
                      None) == B.ROT_ENOTSUP
    # the same matrix without a refresh is not refused on the host (the check
    # that follows needs a device, so it is not called here)


def test_plan_bit_exact_at_scale():
    """100 000 matrices, many ties and groups, four simulated ranks."""
    r = np.random.default_rng(77)
    dims = [64 * k for k in range(1, 33)]
    shapes = [(int(r.choice(dims)), int(r.choice(dims))) for _ in range(100_000)]
    p = B.Plan(shapes, 64 << 20, ranks=4)
    o = orc.plan(shapes, 64 << 20, ranks=4)
    assert len(o.groups) > 100
    assert p.groups() == o.groups and p.owners() == o.owners


def _fail_each_allocation_in_turn(call, cleanup=None, limit=400):
    """Make the k-th host allocation of `call` fail for k = 0, 1, ... until the
    call gets through; every failing run must return ROT_ENOMEM (no exception
    across the C ABI, no crash).  Returns how many allocations were failed."""
    L = B.lib()
    for k in range(limit):
        L.rot_test_fail_host_alloc(k)
        try:
            rc, res = call()
        finally:
            L.rot_test_fail_host_alloc(-1)
        if rc == B.ROT_OK:
            if cleanup:
                cleanup(res)
            return k
        assert rc == B.ROT_ENOMEM, (k, rc)
    raise AssertionError("the call never succeeded")


def test_plan_create_reports_host_allocation_failure():
    wl = inputs.workload("block")
    arr = (B.rot_shape * wl.count)(*[B.rot_shape(m, n) for m, n in wl.shapes])

    def call():
        out = ctypes.c_void_p()
        rc = B.lib().rot_plan_create_ex(arr, wl.count, 64 << 20, 2, ctypes.byref(out))
        if rc != B.ROT_OK:
            assert not out.value  # *out is NULL on error
        return rc, out

    failed = _fail_each_allocation_in_turn(call, lambda out: B.lib().rot_plan_destroy(out))
    assert failed >= 5  # shapes, groups, owners, layouts: each failed in turn


def test_partitions_report_host_allocation_failure():
    work = [int(x) for x in np.random.default_rng(5).integers(1, 1000, 30)]
    sizes = [7, 8, 15]
    w = (ctypes.c_uint64 * 30)(*work)
    b = (ctypes.c_int32 * 3)(*sizes)
    owners = (ctypes.c_int32 * 30)()
    loads = (ctypes.c_uint64 * 4)()
    for fn in ("rot_partition_alpha", "rot_partition_static"):
        def call():
            if fn == "rot_partition_alpha":
                return B.lib().rot_partition_alpha(w, 30, b, 3, 4, 1.0, owners, loads), None
            return B.lib().rot_partition_static(w, 30, b, 3, 4, owners), None
        assert _fail_each_allocation_in_turn(call) >= 1, fn
    # and the results are unaffected by the earlier failures
    o = orc.alpha_partition(work, sizes, 4, 1.0)
    assert B.partition_alpha(work, sizes, 4, 1.0) == (o.owners, o.loads)


def test_compact_state_bytes():
    """The reduced-precision format (bf16 moments, fp16 bases) takes about the
    algorithmic float32 state (M, v, U, V) and less than 0.6 of the full
    format; switching back restores the full layout."""
    wl = inputs.workload("full")
    p = B.Plan(wl.shapes, wl.c_max)
    full = p.state_bytes()[0]
    assert B.lib().rot_plan_set_state_format(p.handle, B.ROT_STATE_COMPACT) == B.ROT_OK
    compact = p.state_bytes()[0]
    algorithmic = sum(4 * (2 * m * n + m * m + n * n) for m, n in wl.shapes)
    assert compact <= 1.05 * algorithmic and compact < 0.6 * full
    assert B.lib().rot_plan_set_state_format(p.handle, B.ROT_STATE_FULL) == B.ROT_OK
    assert p.state_bytes()[0] == full
    assert B.lib().rot_plan_set_state_format(p.handle, 7) == B.ROT_EINVAL


def test_profile_classes_match_the_header_and_the_bench():
    """Every kernel class the header declares can be read, the next id is
    refused, and the benchmark names exactly those classes."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "rot.h")) as f:
        header = f.read()
    count = int(re.search(r"#define ROT_PROF_CLASSES (\d+)", header).group(1))
    ids = sorted(int(v) for v in re.findall(r"#define ROT_PROF_\w+ (\d+)", header))
    assert ids == list(range(count)) + [count]  # the classes, then ROT_PROF_CLASSES
    L = B.lib()
    n, tot, mx, work = ctypes.c_uint64(), ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    args = (ctypes.byref(n), ctypes.byref(tot), ctypes.byref(mx), ctypes.byref(work))
    for c in range(count):
        assert L.rot_profile_read(c, *args) == B.ROT_OK, c
    assert L.rot_profile_read(count, *args) == B.ROT_EINVAL
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert len(bench.PROF_CLASSES) == count
