"""GPU: the allocation-free entry point (nt_gemv_argmax_noalloc) against nt_gemv_q.

For callers that cannot allocate device memory on this path: its scratch is a
file-scope device array, so two calls in a row share it.  Both calls are
checked against the allocating GEMV entry point.  Collected last on purpose.
"""
import numpy as np
import pytest

from gpu_util import ensure_built, rel_l2, torch_cuda
from inputs import activation

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.mark.parametrize("fmt,rows,cols", [("q6_k", 128256, 8192), ("q8_0", 4099, 4096), ("q4_k", 1000, 28672)])
def test_noalloc_matches_gemv_entry_point_two_calls(fmt, rows, cols):
    torch = torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt
    t = nt.nt_qtensor_create(fmt, rows, cols, 0, 0x100001, 0.02)
    try:
        s = torch.cuda.current_stream()
        y_ref = torch.empty(rows, device="cuda")
        y = torch.full((rows,), float("nan"), device="cuda")
        idx = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        margin = torch.full((1,), float("nan"), device="cuda")
        for call in range(2):                      # the second call reuses the static scratch
            x = torch.from_numpy(activation(cols, seed=20 + call)).cuda()
            nt.nt_gemv_q(t, x.data_ptr(), y_ref.data_ptr(), s)
            nt.nt_gemv_argmax_noalloc(t, x.data_ptr(), y.data_ptr(), idx.data_ptr(), margin.data_ptr(), s)
            torch.cuda.synchronize()
            yr, yn = y_ref.cpu().numpy(), y.cpu().numpy()
            assert rel_l2(yn, yr) < TOL
            top = np.sort(yr.astype(np.float64))[::-1]
            assert int(idx.item()) == int(np.argmax(yr))
            assert abs(float(margin.item()) - (top[0] - top[1])) <= 1e-6 * max(1.0, abs(top[0]))
    finally:
        nt.nt_qtensor_destroy(t)


def test_noalloc_one_row_and_ties():
    """One row: index 0 and an infinite margin.  x = 0 makes every y equal: the
    lowest row wins the tie with margin 0 (on two calls in a row)."""
    torch = torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt
    s = torch.cuda.current_stream()
    for rows, cols, x_zero in ((1, 1024, False), (300, 1024, True), (5, 96, True)):
        t = nt.nt_qtensor_create("q8_0", rows, cols, 0, 5, 0.02)
        try:
            x = torch.zeros(cols, device="cuda") if x_zero else torch.from_numpy(activation(cols, seed=3)).cuda()
            y = torch.empty(rows, device="cuda")
            idx = torch.full((1,), -7, dtype=torch.int32, device="cuda")
            margin = torch.full((1,), float("nan"), device="cuda")
            for _ in range(2):
                nt.nt_gemv_argmax_noalloc(t, x.data_ptr(), y.data_ptr(), idx.data_ptr(), margin.data_ptr(), s)
                torch.cuda.synchronize()
                assert int(idx.item()) == 0
                if rows == 1:
                    assert float(margin.item()) == float("inf")
                else:
                    assert float(margin.item()) == 0.0 and float(y.abs().max().item()) == 0.0
        finally:
            nt.nt_qtensor_destroy(t)


def test_noalloc_rejects_bad_arguments():
    torch = torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt
    t = nt.nt_qtensor_create("q8_0", 64, 256, 0, 1, 0.02)
    try:
        x = torch.zeros(256, device="cuda")
        y = torch.zeros(64, device="cuda")
        idx = torch.zeros(1, dtype=torch.int32, device="cuda")
        with pytest.raises(nt.NtError) as ei:
            nt.nt_gemv_argmax_noalloc(t, x.data_ptr(), y.data_ptr(), 0, idx.data_ptr())
        assert ei.value.status == nt.NT_E_INVAL
    finally:
        nt.nt_qtensor_destroy(t)
