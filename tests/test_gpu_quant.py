"""GPU: generated block bytes and dequantization against the oracle (bit-exact)."""
import numpy as np
import pytest

import oracle
from gpu_util import blocks, ensure_built, torch_cuda

pytestmark = pytest.mark.gpu
FORMATS = ["q8_0", "q4_0", "q4_k", "q6_k", "q5_k"]


@pytest.fixture(scope="module")
def nt():
    torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt as _nt
    return _nt


def _export(nt, t, fmt, rows, cols, row0=0, nrows=None):
    qk, bb = blocks(fmt)
    return nt.nt_qtensor_export(t, row0, rows - row0 if nrows is None else nrows, qk, bb, cols)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 512), (64, 1536), (5, 8192), (3, 28672)])
def test_generated_blocks_bytewise_equal_oracle(nt, fmt, rows, cols):
    t = nt.nt_qtensor_create(fmt, rows, cols, 11, 321, 0.02)
    try:
        got = _export(nt, t, fmt, rows, cols)
        want = oracle.qtensor_rows(fmt, rows, cols, 11, 321, 0.02)
        assert got.shape == want.shape
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:5].tolist()}"
        name, r, c, nbytes = nt.nt_qtensor_info(t)
        qk, bb = blocks(fmt)
        assert (name, r, c, nbytes) == (fmt, rows, cols, rows * cols // qk * bb)
    finally:
        nt.nt_qtensor_destroy(t)


@pytest.mark.parametrize("fmt", FORMATS)
def test_zero_std_tensor_is_all_neutral(nt, fmt):
    rows, cols = 4, 512
    t = nt.nt_qtensor_create(fmt, rows, cols, 0, 1, 0.0)
    try:
        np.testing.assert_array_equal(_export(nt, t, fmt, rows, cols),
                                      oracle.qtensor_rows(fmt, rows, cols, 0, 1, 0.0))
    finally:
        nt.nt_qtensor_destroy(t)


@pytest.mark.parametrize("fmt", FORMATS)
def test_dequant_bit_exact(nt, fmt):
    torch = torch_cuda()
    rows, cols = 19, 1024
    t = nt.nt_qtensor_create(fmt, rows, cols, 5, 77, 0.02)
    try:
        out = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
        nt.nt_dequant(t, 0, rows, out.data_ptr(), torch.cuda.current_stream())
        part = torch.empty(3 * cols, dtype=torch.float32, device="cuda")
        nt.nt_dequant(t, 7, 3, part.data_ptr(), torch.cuda.current_stream())
        torch.cuda.synchronize()
        want = oracle.dequant_rows(fmt, oracle.qtensor_rows(fmt, rows, cols, 5, 77, 0.02), cols)
        got = out.cpu().numpy().reshape(rows, cols)
        np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
        np.testing.assert_array_equal(part.cpu().numpy().reshape(3, cols).view(np.uint32),
                                      want[7:10].view(np.uint32))
    finally:
        nt.nt_qtensor_destroy(t)


@pytest.mark.parametrize("fmt", FORMATS)
def test_full_size_output_matrix_sampled_rows(nt, fmt):
    """The 128256 x 8192 output matrix at full size: sampled rows bytewise equal."""
    rows, cols = 128256, 8192
    t = nt.nt_qtensor_create(fmt, rows, cols, 0, 0x100001, 0.02)
    try:
        for r in (0, 1, 4097, 64127, rows - 1):
            got = _export(nt, t, fmt, rows, cols, row0=r, nrows=1)
            want = oracle.qtensor_rows(fmt, rows, cols, 0, 0x100001, 0.02, row0=r, nrows=1)
            np.testing.assert_array_equal(got, want)
    finally:
        nt.nt_qtensor_destroy(t)
