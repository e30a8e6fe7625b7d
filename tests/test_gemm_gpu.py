"""The tensor-core grouped GEMM in isolation (rot_test_gemm) against a float64
matmul, for every output mode, ragged sizes and both precisions."""

import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 32), (64, 64, 64), (300, 520, 100), (1, 40, 7), (33, 1, 65),
          (1000, 1000, 1000), (2048, 256, 4096), (130, 300, 2000)]
PRECISE = B.ROT_PREC_3XTF32_PRECISE
F16 = B.ROT_PREC_3XF16
PRECISE16 = B.ROT_TEST_PREC_3XF16_PRECISE  # the precise kernel on fp16 splits
TOL = {B.ROT_PREC_3XTF32: 3e-6, B.ROT_PREC_TF32: 2e-3, PRECISE: 1.5e-6, F16: 3e-6,
       PRECISE16: 1.5e-6}


def tol(precision, K):
    """Relative Frobenius bound.  The tensor cores accumulate in float32 but
    truncate each partial sum, an error that grows with the number of K steps
    (about 2^-24 per step relative to the running sum); 3xTF32 is therefore
    bounded by a K-proportional term on top of the split's own error."""
    if precision in (B.ROT_PREC_3XTF32, F16):
        return TOL[precision] + 2.5e-8 * K
    return TOL[precision]  # TF32: input rounding dominates; precise: K-independent


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    B.lib()


def run(M, N, K, epi, precision, alpha=0.5, seed=0, row_spread=False):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.rand(M, K, device="cuda", generator=g) * 2 - 1
    Bm = torch.rand(N, K, device="cuda", generator=g) * 2 - 1
    if row_spread:  # rows of very different magnitude (exercises the fp16 scales)
        A = A * torch.logspace(-12, 6, M, device="cuda")[:, None]
        Bm = Bm * torch.logspace(-3, 3, N, device="cuda")[:, None]
    ref = A.double() @ Bm.double().T
    transposed = epi in (1, 3)
    rows, ldc = (N, M) if transposed else (M, N)
    if epi in (0, 1):
        C = torch.zeros(2 * rows * ldc, device="cuda")
    elif epi == 5:
        C = torch.cat([torch.rand(rows * ldc, device="cuda", generator=g),
                       torch.zeros(rows * ldc, device="cuda")])
    else:
        C = torch.rand(rows * ldc, device="cuda", generator=g)
    C0 = C.clone()
    wb = B.rot_test_gemm_work_bytes(M, N, K)
    work = torch.empty(wb, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.rot_test_gemm(M, N, K, A.data_ptr(), K, Bm.data_ptr(), K, C.data_ptr(), ldc, epi, alpha,
                    precision, work.data_ptr(), wb, status.data_ptr(),
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if epi == 1 and precision in (F16, PRECISE16):
        halves = C.view(torch.float16)
        out = (halves[:rows * ldc].double() + halves[rows * ldc:2 * rows * ldc].double())
        out = out.view(rows, ldc)
    elif epi in (0, 1):
        out = (C[:rows * ldc].double() + C[rows * ldc:].double()).view(rows, ldc)
        # the split is exact: hi has 10 explicit mantissa bits
        hi = C[:rows * ldc]
        assert torch.equal(hi.view(torch.int32) & 0x1FFF, torch.zeros_like(hi, dtype=torch.int32))
    elif epi == 4:
        out = (C0.double() - C.double()).view(rows, ldc) / alpha
    elif epi == 5:
        before = C0[:rows * ldc].double() + C0[rows * ldc:].double()
        after = C[:rows * ldc].double() + C[rows * ldc:].double()
        out = (before - after).view(rows, ldc) / alpha
    else:
        out = C.double().view(rows, ldc)
    if transposed:
        out = out.T
    return out, ref


@pytest.mark.parametrize("precision", [B.ROT_PREC_3XTF32, B.ROT_PREC_TF32, PRECISE, F16, PRECISE16])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_store_f32(M, N, K, precision):
    out, ref = run(M, N, K, 2, precision)
    err = float((out - ref).norm() / ref.norm())
    print(f"gemm {M}x{N}x{K} prec {precision}: rel err {err:.3e}")
    assert err <= tol(precision, K), err


@pytest.mark.parametrize("precision", [PRECISE, PRECISE16])
@pytest.mark.parametrize("K", [6144, 12288])
def test_gemm_precise_error_does_not_grow_with_k(K, precision):
    """The precise product sums its K-block partials (32 TF32 or 64 fp16
    elements) with compensation: its error stays near the split's own (1.3e-7
    measured) at long K, where a plain float32 running sum of the blocks gives
    2.8e-7 (K = 6144) and 3.8e-7 (K = 12288)."""
    out, ref = run(256, 256, K, 2, precision, seed=K)
    err = float((out - ref).norm() / ref.norm())
    print(f"precise 256x256x{K}: rel err {err:.3e}")
    assert err <= 2e-7, err


@pytest.mark.parametrize("epi", [0, 1, 2, 4, 5])
@pytest.mark.parametrize("M,N,K", [(300, 520, 300), (256, 384, 512), (130, 260, 513)])
def test_gemm_precise_around_the_short_k_limit(M, N, K, epi):
    """K up to 512 runs the short-K variant (the whole sum in registers, four
    TMEM buffers), K = 513 the long one: both in every output mode."""
    out, ref = run(M, N, K, epi, PRECISE, seed=K + epi)
    err = float((out - ref).norm() / ref.norm())
    assert err <= (1e-5 if epi in (4, 5) else TOL[PRECISE]), err


@pytest.mark.parametrize("epi", [1, 2, 3, 4])
@pytest.mark.parametrize("M,N,K", [(300, 520, 300), (256, 384, 512), (130, 260, 513),
                                   (200, 72, 1000)])
def test_gemm_precise16_output_modes(M, N, K, epi):
    """The precise kernel on fp16 splits: the short-K variant (K <= 512, up to
    eight blocks of 64) and the long one; the transposed fp16-split store
    (unscaled here), the float32 stores and the apply mode."""
    out, ref = run(M, N, K, epi, PRECISE16, seed=K + epi)
    err = float((out - ref).norm() / ref.norm())
    bound = {1: 2e-6, 2: TOL[PRECISE16], 3: TOL[PRECISE16], 4: 1e-5}[epi]
    assert err <= bound, err


@pytest.mark.parametrize("precision", [B.ROT_PREC_3XTF32, PRECISE])
@pytest.mark.parametrize("epi", [0, 1, 3, 4, 5])
@pytest.mark.parametrize("M,N,K", [(300, 520, 100), (64, 64, 64), (1, 40, 7)])
def test_gemm_output_modes(M, N, K, epi, precision):
    out, ref = run(M, N, K, epi, precision)
    err = (out - ref).norm() / ref.norm()
    # the apply modes recover the product from a difference of float32 values
    assert err <= (1e-5 if epi in (4, 5) else tol(precision, K)), float(err)


@pytest.mark.parametrize("epi", [1, 3, 4])
@pytest.mark.parametrize("M,N,K", [(300, 520, 100), (64, 64, 64), (1, 40, 7), (257, 129, 4100)])
def test_gemm_f16_output_modes(M, N, K, epi):
    """3xF16: the transposed fp16-split store (unscaled, values of order 1),
    the transposed float32 store and the apply mode."""
    out, ref = run(M, N, K, epi, F16)
    err = float((out - ref).norm() / ref.norm())
    bound = {1: 2e-6 + 2.5e-8 * K, 3: tol(F16, K), 4: 1e-5 + tol(F16, K)}[epi]
    assert err <= bound, err


@pytest.mark.parametrize("precision", [B.ROT_PREC_3XTF32, F16, PRECISE16])
def test_gemm_rows_of_very_different_magnitude(precision):
    """Rows of A spanning 18 decades and of B 6: per-row scaling keeps every
    row's product at float32-level relative accuracy in 3xF16, as 3xTF32
    (checked row by row, so the small rows are not hidden by the large)."""
    out, ref = run(384, 200, 1000, 2, precision, row_spread=True)
    row_err = (out - ref).norm(dim=1) / ref.norm(dim=1)
    print(f"prec {precision}: worst row rel err {float(row_err.max()):.3e}")
    assert float(row_err.max()) <= 5e-5, float(row_err.max())


def test_gemm_f16_rejects_untransposed_split_modes():
    M = N = K = 32
    A = torch.zeros(M, K, device="cuda")
    C = torch.zeros(2 * M * N, device="cuda")
    wb = B.rot_test_gemm_work_bytes(M, N, K)
    work = torch.empty(wb, dtype=torch.uint8, device="cuda")
    for precision in (F16, PRECISE16):
        for epi in (0, 5):
            with pytest.raises(B.RotError):
                B.rot_test_gemm(M, N, K, A.data_ptr(), K, A.data_ptr(), K, C.data_ptr(), N, epi,
                                1.0, precision, work.data_ptr(), wb, 0,
                                torch.cuda.current_stream().cuda_stream)
