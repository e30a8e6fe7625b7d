"""The analytic work counts behind the benchmark's TFLOP/s and roofline
figures, checked against their literal definitions on small sizes."""

import itertools

from matrix_optimizer_step_rot_gb300 import flops as FL


def test_qr_closed_form_equals_the_sum():
    for p, r in itertools.product(range(1, 40), range(0, 40)):
        if r > p:
            continue
        literal = sum(4 * (p - k) * (r - k) + 4 * (p - k) ** 2 for k in range(r))
        assert FL.qr_flops(p, r) == literal, (p, r)


def test_square_full_rank_qr_is_eight_thirds_p_cubed():
    p = 3000
    assert abs(FL.qr_flops(p, p) / (8.0 / 3.0 * p ** 3) - 1.0) < 2e-3


def test_products_take_the_cheaper_association():
    """A_U = M (M^T U) costs 4 m^2 n, (M M^T) U costs 2 m^2 n + 2 m^3; the
    count (and the GPU path) takes the cheaper one, and likewise for A_V."""
    for m, n in [(6144, 2048), (2048, 6144), (2048, 2048), (1, 7), (7, 1), (300, 299)]:
        a_u = min(4 * m * m * n, 2 * m * m * n + 2 * m ** 3)
        a_v = min(4 * m * n * n, 2 * m * n * n + 2 * n ** 3)
        assert FL.product_flops(m, n) == a_u + a_v, (m, n)


def test_rotation_counts_two_or_three_two_sided_products():
    m, n = 300, 500
    two_sided = 2 * m * m * n + 2 * m * n * n  # U^T X V, one product pair
    assert FL.rotation_flops(m, n, refresh=False) == 2 * two_sided   # G~ and U D V^T
    assert FL.rotation_flops(m, n, refresh=True) == 3 * two_sided    # + M~ = U^T M V
    assert FL.matrix_step_flops(m, n, False) == 2 * two_sided
    assert FL.matrix_step_flops(m, n, True) == (3 * two_sided + FL.product_flops(m, n)
                                                + FL.qr_flops(m, m if m < n else n)
                                                + FL.qr_flops(n, m if m < n else n))
