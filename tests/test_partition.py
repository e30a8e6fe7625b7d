"""Data-parallel partition of matrices over ranks (Canzona page, section 3.2.1
α-balanced greedy LPT; section 3.1.1 static ownership by parameter start).

First the oracle is pinned by hand-worked examples, closed forms, invariants
and brute force; then the C-ABI host implementation is held to the oracle bit
for bit (owners and loads)."""

import itertools

import numpy as np
import pytest

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build, inputs
from oracle import rot_oracle as orc


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.lib()


# ---------------------------------------------------------------- oracle pins

def test_hand_worked_alpha_mix():
    """Two buckets on two ranks: [7] then seven items of work 1 (both W = 7,
    so the lower index goes first).

    Bucket [7]: loads 0, even targets 3.5; boundaries 0 and 7 are equally near,
    the earlier wins: rank 0 takes nothing, rank 1 takes the 7.  Loads (0, 7).
    Bucket of ones: ideal 7 / 2 (printed rule) or (7 + 7) / 2 (after the
    bucket), deficits (3.5, 0) or (7, 0): fill (1, 0) either way.
      alpha = 1: share (1, 0), cut at 7: loads (7, 7).
      alpha = 0: share (0.5, 0.5), target 3.5, boundaries 3 and 4 tie -> 3: (3, 11).
      alpha = 0.5: share (0.75, 0.25), target 5.25 -> 5: (5, 9)."""
    work = [7, 1, 1, 1, 1, 1, 1, 1]
    for alpha, owners, loads in [
        (1.0, [1, 0, 0, 0, 0, 0, 0, 0], [7, 7]),
        (0.0, [1, 0, 0, 0, 1, 1, 1, 1], [3, 11]),
        (0.5, [1, 0, 0, 0, 0, 0, 1, 1], [5, 9]),
    ]:
        for ideal in ("before", "after"):  # fill (1, 0) under either ideal here
            p = orc.alpha_partition(work, [1, 7], 2, alpha, ideal)
            assert p.owners == owners and p.loads == loads, (alpha, ideal)


def test_bucket_order_is_by_work_not_position():
    """Buckets [1, 1] (W = 2) then [6] (W = 6) on two ranks: the 6 is placed
    first (tie at 3 between boundaries 0 and 6 -> rank 1 gets it), then the
    ones fill rank 0 under alpha = 1."""
    for ideal in ("before", "after"):
        p = orc.alpha_partition([1, 1, 6], [2, 1], 2, 1.0, ideal)
        assert p.owners == [0, 0, 1] and p.loads == [2, 6]


def test_printed_ideal_against_the_post_bucket_ideal():
    """Buckets [100], [98], fifty ones; two ranks; alpha = 1.

    [100] from zero loads: fill 1/2 under both readings, target 50, boundaries
    0 and 100 tie, the earlier wins: rank 1 takes it, loads (0, 100).
    [98]: printed ideal 100 / 2 = 50, deficits (50, 0); post-bucket ideal
    (100 + 98) / 2 = 99, deficits (99, 0): fill (1, 0) either way, loads
    (98, 100).
    Ones: printed ideal 198 / 2 = 99, deficits (1, 0), fill (1, 0): rank 0
    takes all fifty, loads (148, 100).  Post-bucket ideal 248 / 2 = 124,
    deficits (26, 24), fill (26/50, 24/50), target 26: loads (124, 124)."""
    work = [100, 98] + [1] * 50
    before = orc.alpha_partition(work, [1, 1, 50], 2, 1.0, "before")
    assert before.owners == [1, 0] + [0] * 50 and before.loads == [148, 100]
    assert orc.alpha_partition(work, [1, 1, 50], 2, 1.0) == before  # the default
    after = orc.alpha_partition(work, [1, 1, 50], 2, 1.0, "after")
    assert after.owners == [1, 0] + [0] * 26 + [1] * 24 and after.loads == [124, 124]


@pytest.mark.parametrize("seed", range(10))
def test_printed_ideal_alpha_one_skips_ranks_at_or_above_the_mean(seed):
    """Printed rule, alpha = 1: a rank whose load is at or above the mean before
    the bucket has no deficit, hence share 0, and its piece lies between two
    cuts aimed at the same target: it receives nothing from that bucket
    (unless no rank is below the mean, when the shares are even)."""
    r = np.random.default_rng(70 + seed)
    R = int(r.integers(2, 6))
    sizes = [int(x) for x in r.integers(1, 12, 7)]
    work = [int(x) for x in r.integers(1, 50, sum(sizes))]
    starts = [sum(sizes[:b]) for b in range(len(sizes))]
    bwork = [sum(work[starts[b]:starts[b] + sizes[b]]) for b in range(len(sizes))]
    order = sorted(range(len(sizes)), key=lambda b: (-bwork[b], b))
    loads = [0] * R
    for k, b in enumerate(order):
        # the partition of the first k + 1 buckets visited is the state after them
        keep = set(order[:k + 1])
        sub_sizes = [sizes[c] if c in keep else 0 for c in range(len(sizes))]
        sub_work = [work[i] for c in range(len(sizes)) if c in keep
                    for i in range(starts[c], starts[c] + sizes[c])]
        p = orc.alpha_partition(sub_work, sub_sizes, R, 1.0, "before")
        mean = sum(loads) / R
        if any(l < mean for l in loads):
            got = [0] * R
            at = sum(sub_sizes[c] for c in range(b))
            for j in range(sizes[b]):
                got[p.owners[at + j]] += work[starts[b] + j]
            for q in range(R):
                if loads[q] >= mean:
                    assert got[q] == 0, (k, q, loads, got)
        loads = p.loads


def test_single_rank_owns_everything():
    r = np.random.default_rng(3)
    work = [int(x) for x in r.integers(0, 1000, 40)]
    p = orc.alpha_partition(work, [10, 0, 25, 5], 1, 0.7)
    assert p.owners == [0] * 40 and p.loads == [sum(work)]
    assert orc.static_partition(work, [10, 0, 25, 5], 1) == [0] * 40


def test_alpha_zero_splits_divisible_buckets_evenly():
    """Unit-work items, every bucket a multiple of R: the even targets land on
    boundaries, so each rank takes an equal consecutive run of every bucket."""
    R = 4
    sizes = [12, 8, 20, 4]
    p = orc.alpha_partition([1] * sum(sizes), sizes, R, 0.0)
    at = 0
    for c in sizes:
        assert p.owners[at:at + c] == [r for r in range(R) for _ in range(c // R)]
        at += c
    assert p.loads == [sum(sizes) // R] * R


@pytest.mark.parametrize("seed", range(6))
def test_alpha_one_keeps_unit_loads_within_one_of_ideal(seed):
    """Post-bucket ideal, alpha = 1, with unit-work items and every bucket holding >= 2R items:
    every load stays within 1 of the ideal after every bucket.  (The loads stay
    within 2 of each other, so each bucket's ideal is above every load; the
    fill targets are then the exact deficits and rounding each cut moves a
    load by at most 1/2 at either end.)  Buckets are given largest first, so
    the partition of the first k buckets is the state after k buckets."""
    r = np.random.default_rng(50 + seed)
    R = int(r.integers(2, 7))
    sizes = sorted((int(x) for x in r.integers(2 * R, 12 * R, 8)), reverse=True)
    for k in range(1, len(sizes) + 1):
        p = orc.alpha_partition([1] * sum(sizes[:k]), sizes[:k], R, 1.0, "after")
        ideal = sum(sizes[:k]) / R
        assert max(abs(l - ideal) for l in p.loads) <= 1.0, (k, p.loads, ideal)


@pytest.mark.parametrize("seed", range(20))
def test_single_bucket_cuts_are_nearest_boundaries_by_brute_force(seed):
    """One bucket from zero loads: every share is 1/R for any alpha, so cut r
    targets W (r + 1) / R.  Brute force over every non-decreasing cut vector:
    the oracle's cuts reach the least total distance to the targets, and the
    earliest such vector on ties."""
    r = np.random.default_rng(100 + seed)
    n = int(r.integers(1, 7))
    R = int(r.integers(2, 5))
    work = [int(x) for x in r.integers(0, 9, n)]
    W = sum(work)
    prefix = [0] + list(itertools.accumulate(work))
    p = orc.alpha_partition(work, [n], R, float(r.uniform(0, 1)), ["before", "after"][seed % 2])
    cuts, at = [], 0
    for q in range(R - 1):
        while at < n and p.owners[at] <= q:
            at += 1
        cuts.append(at)
    best = None
    for cand in itertools.combinations_with_replacement(range(n + 1), R - 1):
        cost = sum(abs(prefix[c] - W * (q + 1) / R) for q, c in enumerate(cand))
        if best is None or cost < best[0] - 1e-12:
            best = (cost, list(cand))
    got = sum(abs(prefix[c] - W * (q + 1) / R) for q, c in enumerate(cuts))
    assert got == pytest.approx(best[0], abs=1e-9)
    if W > 0 and len(set(prefix)) == len(prefix):
        assert cuts == best[1]


@pytest.mark.parametrize("seed", range(15))
def test_partition_invariants(seed):
    """Every item owned once; owners non-decreasing inside a bucket (R
    consecutive pieces in rank order); loads are the owned work."""
    r = np.random.default_rng(200 + seed)
    sizes = [int(x) for x in r.integers(0, 9, int(r.integers(1, 10)))]
    work = [int(x) for x in r.integers(0, 10 ** 6, sum(sizes))]
    R = int(r.integers(1, 9))
    p = orc.alpha_partition(work, sizes, R, float(r.uniform(0, 1)), ["before", "after"][seed % 2])
    assert all(0 <= o < R for o in p.owners)
    at = 0
    for c in sizes:
        assert p.owners[at:at + c] == sorted(p.owners[at:at + c])
        at += c
    got = [0] * R
    for i, o in enumerate(p.owners):
        got[o] += work[i]
    assert got == p.loads


def test_static_by_start_hand_worked():
    """Shards of ceil(E / R) elements; the owner holds the item's first element."""
    assert orc.static_partition([4, 4, 4, 4], [4], 2) == [0, 0, 1, 1]
    assert orc.static_partition([10, 1, 1], [3], 2) == [0, 1, 1]       # S = 6: starts 0, 10, 11
    assert orc.static_partition([1, 1, 10], [3], 2) == [0, 0, 0]       # starts 0, 1, 2 < 6
    assert orc.static_partition([3, 3, 3], [1, 2], 2) == [0, 0, 1]     # per bucket: [3] | [3, 3]
    assert orc.static_partition([5, 5, 5], [3], 4) == [0, 1, 2]        # S = 4: starts 0, 5, 10


def test_alpha_one_beats_static_on_the_qwen_stack():
    """The page's claim in kind (section 5.2.1: FLOPs imbalance falls under
    the α-balanced partition): on the 28-block stack, one bucket per block,
    8 ranks."""
    wl = inputs.workload("full")
    work = [orc.item_cost(m, n) for m, n in wl.shapes]
    elems = [m * n for m, n in wl.shapes]
    st = orc.static_partition(elems, [7] * 28, 8)
    static_loads = [0] * 8
    for i, o in enumerate(st):
        static_loads[o] += work[i]
    for ideal in ("before", "after"):
        p = orc.alpha_partition(work, [7] * 28, 8, 1.0, ideal)
        assert orc.imbalance(p.loads) < 1.1 < 2.0 < orc.imbalance(static_loads), ideal


# ---------------------------------------------------- C ABI against the oracle

def test_item_work_matches_oracle(lib):
    shapes = [(1, 1), (65536, 65536), (6144, 2048), (3, 7)]
    assert B.item_work(shapes) == [orc.item_cost(m, n) for m, n in shapes]


@pytest.mark.parametrize("seed", range(60))
def test_alpha_partition_bit_exact(lib, seed):
    r = np.random.default_rng(1000 + seed)
    nb = int(r.integers(0, 12))
    sizes = [int(x) for x in r.integers(0, 10, nb)]
    hi = [10, 1000, 10 ** 9][seed % 3]
    work = [int(x) for x in r.integers(0, hi, sum(sizes))]
    if seed % 4 == 0 and work:  # many equal buckets
        work = [work[0]] * len(work)
    R = int(r.integers(1, 12))
    alpha = [0.0, 1.0, float(r.uniform(0, 1)), 0.8][seed % 4]
    for ideal in ("before", "after"):
        o = orc.alpha_partition(work, sizes, R, alpha, ideal)
        owners, loads = B.partition_alpha(work, sizes, R, alpha, ideal)
        assert owners == o.owners and loads == o.loads, ideal


@pytest.mark.parametrize("name", ["full", "ragged", "slice8b"])
@pytest.mark.parametrize("ranks", [2, 8, 64])
def test_workload_partitions_bit_exact(lib, name, ranks):
    wl = inputs.workload(name)
    per = 7 if name != "ragged" else 16
    sizes = [per] * (len(wl.shapes) // per)
    work = B.item_work(wl.shapes)
    elems = [m * n for m, n in wl.shapes]
    for alpha in (0.0, 0.8, 1.0):
        for ideal in ("before", "after"):
            o = orc.alpha_partition(work, sizes, ranks, alpha, ideal)
            assert B.partition_alpha(work, sizes, ranks, alpha, ideal) == (o.owners, o.loads)
    assert B.partition_static(elems, sizes, ranks) == orc.static_partition(elems, sizes, ranks)


@pytest.mark.parametrize("seed", range(30))
def test_static_partition_bit_exact(lib, seed):
    r = np.random.default_rng(3000 + seed)
    sizes = [int(x) for x in r.integers(0, 9, int(r.integers(0, 8)))]
    elems = [int(x) for x in r.integers(0, 10 ** 8, sum(sizes))]
    R = int(r.integers(1, 10))
    assert B.partition_static(elems, sizes, R) == orc.static_partition(elems, sizes, R)


def test_partition_argument_errors(lib):
    E = B.ROT_EINVAL
    for call in [
        lambda: B.partition_alpha([1, 2], [1], 2, 0.5),           # sizes do not cover
        lambda: B.partition_alpha([1, 2], [3, -1], 2, 0.5),       # negative size
        lambda: B.partition_alpha([1, 2], [2], 0, 0.5),           # ranks
        lambda: B.partition_alpha([1, 2], [2], 2, 1.5),           # alpha
        lambda: B.partition_alpha([1, 2], [2], 2, float("nan")),
        lambda: B.partition_alpha([2 ** 52, 2 ** 52], [2], 2, 1.0),  # total >= 2^53
        lambda: B.partition_alpha([1, 2], [2], 2, 0.5, "sideways"),  # unknown ideal
        lambda: B.partition_static([1, 2], [1], 2),
        lambda: B.partition_static([2 ** 63, 2 ** 63], [2], 2),   # bucket total overflows
        lambda: B.item_work([(0, 4)]),
    ]:
        with pytest.raises(B.RotError) as e:
            call()
        assert e.value.code == E
    assert B.partition_alpha([], [], 3, 1.0) == ([], [0, 0, 0])
    assert B.partition_static([], [0, 0], 3) == []


def test_partitions_bit_exact_at_scale(lib):
    """20 000 items in 2 500 buckets on 64 ranks, several alphas."""
    r = np.random.default_rng(4242)
    sizes = [int(x) for x in r.integers(1, 15, 2500)]
    n = sum(sizes)
    work = [int(x) for x in r.integers(1, 10 ** 9, n)]
    elems = [int(x) for x in r.integers(1, 10 ** 7, n)]
    for alpha in (0.0, 0.8, 1.0):
        for ideal in ("before", "after"):
            o = orc.alpha_partition(work, sizes, 64, alpha, ideal)
            assert B.partition_alpha(work, sizes, 64, alpha, ideal) == (o.owners, o.loads)
    assert B.partition_static(elems, sizes, 64) == orc.static_partition(elems, sizes, 64)
