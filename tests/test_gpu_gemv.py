"""GPU: fused dequantize-GEMV through nt_gemv_q against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import ensure_built, rel_l2, torch_cuda
from inputs import activation

pytestmark = pytest.mark.gpu
FORMATS = ["q8_0", "q4_0", "q4_k", "q6_k", "q5_k"]
TOL = 2e-3   # relative L2 against fp64 accumulation of the same dequantized weights


@pytest.fixture(scope="module")
def nt():
    torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt as _nt
    return _nt


def _gemv(nt, t, x, rows):
    torch = torch_cuda()
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    yd = torch.full((rows,), float("nan"), device="cuda")
    nt.nt_gemv_q(t, xd.data_ptr(), yd.data_ptr(), torch.cuda.current_stream())
    torch.cuda.synchronize()
    return yd.cpu().numpy()


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 512), (37, 1536), (1000, 4096), (77, 8192), (45, 14336),
                                       (19, 28672), (5, 32768), (2, 31744)])
def test_gemv_matches_oracle(nt, fmt, rows, cols):
    t = nt.nt_qtensor_create(fmt, rows, cols, 3, 55, 0.02)
    try:
        x = activation(cols, seed=1)
        got = _gemv(nt, t, x, rows)
        want = oracle.gemv(fmt, oracle.qtensor_rows(fmt, rows, cols, 3, 55, 0.02, nthreads=8), rows, cols, x,
                           nthreads=8)
        assert np.isfinite(got).all()
        err = rel_l2(got, want)
        assert err < TOL, err
        # activations are carried as 16-bit fixed point per 32-column block (error <= 2^-16 of the
        # block's largest |x|): expected relative L2 ~2e-5, far inside the tolerance
        assert err < 1e-4, f"should be far inside the tolerance: {err}"
        # determinism: a second launch gives the same bits
        np.testing.assert_array_equal(_gemv(nt, t, x, rows), got)
    finally:
        nt.nt_qtensor_destroy(t)


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_wider_than_one_launch_in_column_windows(nt, fmt):
    """More than 32768 columns: launches over column windows of at most 32768 add
    their products in window order; against the oracle as any GEMV.  A width past
    32768 that is not a multiple of 1024 is refused."""
    rows, cols = 37, 2 * 32768 + 4096
    t = nt.nt_qtensor_create(fmt, rows, cols, 3, 57, 0.02)
    try:
        x = activation(cols, seed=2)
        got = _gemv(nt, t, x, rows)
        want = oracle.gemv(fmt, oracle.qtensor_rows(fmt, rows, cols, 3, 57, 0.02, nthreads=8), rows, cols, x,
                           nthreads=8)
        assert np.isfinite(got).all()
        err = rel_l2(got, want)
        assert err < TOL and err < 1e-4, err
        np.testing.assert_array_equal(_gemv(nt, t, x, rows), got)
    finally:
        nt.nt_qtensor_destroy(t)
    t = nt.nt_qtensor_create(fmt, 4, 33024, 3, 58, 0.02)
    try:
        with pytest.raises(nt.NtError) as ei:
            _gemv(nt, t, np.zeros(33024, np.float32), 4)
        assert ei.value.status == nt.NT_E_UNSUPPORTED
    finally:
        nt.nt_qtensor_destroy(t)


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_degenerate_inputs(nt, fmt):
    rows, cols = 9, 768 if fmt in ("q8_0", "q4_0") else 1024
    t = nt.nt_qtensor_create(fmt, rows, cols, 3, 56, 0.02)
    try:
        assert not _gemv(nt, t, np.zeros(cols, np.float32), rows).any()
        W = oracle.dequant_rows(fmt, oracle.qtensor_rows(fmt, rows, cols, 3, 56, 0.02), cols)
        for c in (0, 33, cols - 1):
            e = np.zeros(cols, np.float32)
            e[c] = 1.0
            np.testing.assert_allclose(_gemv(nt, t, e, rows), W[:, c], rtol=1e-6, atol=1e-9)
    finally:
        nt.nt_qtensor_destroy(t)


SHAPES = [(8192, 8192), (1024, 8192), (28672, 8192), (8192, 28672), (128256, 8192)]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_gemv_full_size_sampled_rows(nt, fmt, rows, cols):
    """70B layer shapes in the benchmark's launch configuration; the oracle recomputes sampled rows."""
    t = nt.nt_qtensor_create(fmt, rows, cols, 0, 9, 0.02)
    try:
        x = activation(cols, seed=1)
        got = _gemv(nt, t, x, rows)
        assert np.isfinite(got).all()
        sample = sorted({0, 1, 2, 3, rows // 3, rows // 2 + 1, rows - 2, rows - 1})
        want = np.array([oracle.gemv(fmt, oracle.qtensor_rows(fmt, rows, cols, 0, 9, 0.02, row0=r, nrows=1), 1,
                                     cols, x)[0] for r in sample])
        assert rel_l2(got[sample], want) < TOL
        # property at any size: |y| is bounded by sum |w| |x| <= max|w| * ||x||_1
        assert np.abs(got).max() < 0.2 * np.abs(x).sum()
    finally:
        nt.nt_qtensor_destroy(t)


def test_gemv_argument_checks(nt):
    torch = torch_cuda()
    t = nt.nt_qtensor_create("q8_0", 8, 256, 0, 1, 0.02)
    try:
        xd = torch.zeros(256 + 4, device="cuda")
        yd = torch.zeros(16, device="cuda")
        with pytest.raises(nt.NtError) as ei:
            nt.nt_gemv_q(t, xd.data_ptr() + 4, yd.data_ptr())
        assert ei.value.status == nt.NT_E_INVAL
        with pytest.raises(nt.NtError):
            nt.nt_gemv_q(t, 0, yd.data_ptr())
    finally:
        nt.nt_qtensor_destroy(t)
