"""Analytic work of the rotated-Adam step (what the method itself needs).

Per matrix W (m x n):
  rotation   G~ = U^T G V and U D V^T every step: two two-sided products,
             4 (m^2 n + m n^2) flops; M~ = U^T M V, a third, only when the
             bases change (refresh steps; in between M~ follows
             beta1 M~ + (1 - beta1) G~ element-wise, the same quantity).
On refresh steps, in addition:
  products   A_U = M (M^T U) when n < m (4 m^2 n), else (M M^T) U
             (2 m^2 n + 2 m^3); the same with m and n exchanged for A_V.
  QR+        Householder QR of a p x p input whose rank is at most
             r = min(m, n): the first r columns are factored (each reflector
             k updates the r - k columns after it, rows k.., 4 flops an
             element) and Q = H_0 .. H_{r-1} I is accumulated (4 flops an
             element of the (p - k)^2 block per reflector):
             sum_{k<r} 4 (p - k)(r - k) + 4 (p - k)^2.
             Square full rank gives (8/3) p^3.
Element-wise work (momentum, v, D) is counted in bytes, not flops.
"""

from __future__ import annotations


def rotation_flops(m: int, n: int, refresh: bool = True) -> float:
    return (6.0 if refresh else 4.0) * (m * m * n + m * n * n)


def product_flops(m: int, n: int) -> float:
    a_u = 4.0 * m * m * n if n < m else 2.0 * m * m * n + 2.0 * m ** 3
    a_v = 4.0 * m * n * n if m < n else 2.0 * m * n * n + 2.0 * n ** 3
    return a_u + a_v


def _sum_sq(a: int, b: int) -> float:
    """sum_{j=a+1}^{b} j^2 (0 <= a <= b)."""
    f = lambda x: x * (x + 1) * (2 * x + 1) / 6.0
    return f(b) - f(a)


def qr_flops(p: int, r: int) -> float:
    """sum_{k<r} 4 (p-k)(r-k) + 4 (p-k)^2, in closed form."""
    # with j = p - k running over p-r+1 .. p:  (p-k)(r-k) = j (j - (p - r))
    d = p - r
    s2 = _sum_sq(p - r, p)
    s1 = (p * (p + 1) - (p - r) * (p - r + 1)) / 2.0
    return 4.0 * (s2 - d * s1) + 4.0 * s2


def refresh_flops(m: int, n: int) -> float:
    r = min(m, n)
    return product_flops(m, n) + qr_flops(m, r) + qr_flops(n, r)


def matrix_step_flops(m: int, n: int, refresh: bool) -> float:
    return rotation_flops(m, n, refresh) + (refresh_flops(m, n) if refresh else 0.0)


def step_flops(shapes, refresh: bool) -> float:
    return sum(matrix_step_flops(m, n, refresh) for m, n in shapes)


def step_bytes(shapes) -> float:
    """Minimum HBM traffic of one step: read W, G, M, v and write W, M, v
    (float32, 28 B an element) plus one read of U and V."""
    return sum(28.0 * m * n + 4.0 * (m * m + n * n) for m, n in shapes)
