"""Seeded synthetic inputs and workload definitions.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.  It
holds none of the optimizer's arithmetic: only a counter-based random number
generator, the distributions drawn from it, and the five workload definitions
(shapes, hyper-parameters, step counts, refresh period, micro-group byte cap).

Generator
---------
A counter-based SplitMix64 stream (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; finalizer constants as published
by Vigna).  Every value is a pure function of (seed, kind, t, i, element), so
any single matrix of a large workload can be regenerated on its own:

* key   = mix(mix(mix(mix(seed + G) ^ kind*G) + t*G) ^ i*G)  (uint64, wrapping)
* u(c)  = ((mix(key + (c+1)*G) >> 11) + 0.5) * 2**-53          uniform in (0, 1)
* normal(e)   = sqrt(-2 ln u(2e)) * cos(2*pi*u(2e+1))          (Box-Muller)
* student3(e) = z0 / sqrt((z1^2+z2^2+z3^2)/3), z_j = normal(4e+j)

All of it in float64; the value handed to either side is rounded to float32
once, and both sides consume those float32 values.
"""

from __future__ import annotations

import dataclasses
from typing import List, Tuple

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

KIND_W = 1      # initial parameter matrix W
KIND_G = 2      # gradient G at step t
KIND_SHAPE = 3  # shape draws of the ragged workload


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finalizer on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, kind: int, t: int, i: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = _mix(np.array([seed], dtype=np.uint64) + _G)
        k = _mix(k ^ (np.uint64(kind) * _G))
        k = _mix(k + np.uint64(t) * _G)
        k = _mix(k ^ (np.uint64(i) * _G))
    return k[0]


def uniforms(seed: int, kind: int, t: int, i: int, count: int, offset: int = 0) -> np.ndarray:
    """`count` float64 uniforms in (0, 1) at counters offset .. offset+count-1."""
    key = _key(seed, kind, t, i)
    c = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix(key + c * _G)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(seed: int, kind: int, t: int, i: int, count: int) -> np.ndarray:
    """`count` standard normals (float64) by Box-Muller, two uniforms each."""
    u = uniforms(seed, kind, t, i, 2 * count)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def student_t3(seed: int, kind: int, t: int, i: int, count: int) -> np.ndarray:
    """`count` Student-t draws with 3 degrees of freedom (float64)."""
    z = normals(seed, kind, t, i, 4 * count).reshape(count, 4)
    chi2 = z[:, 1] ** 2 + z[:, 2] ** 2 + z[:, 3] ** 2
    return z[:, 0] / np.sqrt(chi2 / 3.0)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

BLOCK_1P7B = [  # Qwen3-1.7B-shaped transformer block, rows x cols (out x in)
    ("q_proj", 2048, 2048), ("k_proj", 1024, 2048), ("v_proj", 1024, 2048),
    ("o_proj", 2048, 2048), ("gate", 6144, 2048), ("up", 6144, 2048),
    ("down", 2048, 6144),
]
BLOCK_8B = [  # Qwen3-8B-shaped block
    ("q_proj", 4096, 4096), ("k_proj", 1024, 4096), ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096), ("gate", 12288, 4096), ("up", 12288, 4096),
    ("down", 4096, 12288),
]

MB = 1 << 20
GB = 1 << 30


@dataclasses.dataclass(frozen=True)
class Hyper:
    """Optimizer hyper-parameters, held as the float32 values both sides use."""
    beta1: float = float(np.float32(0.9))
    beta2: float = float(np.float32(0.999))
    eps: float = float(np.float32(1e-8))
    lr: float = float(np.float32(1e-3))
    rank_rtol: float = float(np.float32(1e-3))


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shapes: Tuple[Tuple[int, int], ...]
    names: Tuple[str, ...]
    w_std: float
    g_std: float          # normal std, or the Student-t scale when g_dist == "t3"
    g_dist: str           # "normal" | "t3"
    steps: int
    refresh_every: int    # K: refresh on steps t with t % K == 0 (t is 1-based)
    c_max: int            # micro-group byte cap
    seed: int
    hyper: Hyper = Hyper()

    @property
    def count(self) -> int:
        return len(self.shapes)

    def refresh(self, t: int) -> bool:
        """Refresh schedule: steps K, 2K, ... (t counts from 1)."""
        return t % self.refresh_every == 0

    def w0(self, i: int) -> np.ndarray:
        m, n = self.shapes[i]
        return (self.w_std * normals(self.seed, KIND_W, 0, i, m * n)).astype(np.float32).reshape(m, n)

    def grad(self, i: int, t: int) -> np.ndarray:
        m, n = self.shapes[i]
        if self.g_dist == "t3":
            z = student_t3(self.seed, KIND_G, t, i, m * n)
        else:
            z = normals(self.seed, KIND_G, t, i, m * n)
        return (self.g_std * z).astype(np.float32).reshape(m, n)


def _ragged_shapes(seed: int, count: int = 256) -> List[Tuple[int, int]]:
    u = uniforms(seed, KIND_SHAPE, 0, 0, 2 * count)
    dims = 64 * (1 + np.minimum(np.floor(u * 16.0), 15.0).astype(np.int64))
    return [(int(dims[2 * j]), int(dims[2 * j + 1])) for j in range(count)]


def workload(name: str) -> Workload:
    """The five workloads: tiny, block, full, slice8b, ragged."""
    if name == "tiny":
        shapes = ((64, 64), (64, 128), (128, 64), (32, 96))
        return Workload("tiny", shapes, tuple(f"m{j}" for j in range(4)), 0.02, 1e-2,
                        "normal", 10, 5, 1 * MB, 0)
    if name == "block":
        return Workload("block", tuple((m, n) for _, m, n in BLOCK_1P7B),
                        tuple(nm for nm, _, _ in BLOCK_1P7B), 0.02, 1e-3, "normal", 20, 10,
                        512 * MB, 1)
    if name == "full":
        shapes = tuple((m, n) for _ in range(28) for _, m, n in BLOCK_1P7B)
        names = tuple(f"L{b}.{nm}" for b in range(28) for nm, _, _ in BLOCK_1P7B)
        return Workload("full", shapes, names, 0.02, 1e-3, "normal", 10, 5, 512 * MB, 2)
    if name == "slice8b":
        shapes = tuple((m, n) for _ in range(4) for _, m, n in BLOCK_8B)
        names = tuple(f"L{b}.{nm}" for b in range(4) for nm, _, _ in BLOCK_8B)
        return Workload("slice8b", shapes, names, 0.02, 1e-3, "normal", 5, 1, 1 * GB, 3)
    if name == "ragged":
        shapes = tuple(_ragged_shapes(4))
        return Workload("ragged", shapes, tuple(f"r{j}" for j in range(256)), 0.02, 1e-3,
                        "t3", 10, 2, 64 * MB, 4)
    raise KeyError(name)


WORKLOADS = ("tiny", "block", "full", "slice8b", "ragged")
