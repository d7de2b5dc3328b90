"""GPU: the multi-token GEMV (nt_gemv_q_batch, the verification GEMV of
self-speculative decoding) against single-token nt_gemv_q, bit for bit, and
against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import ensure_built, rel_l2, torch_cuda
from inputs import activation

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def nt():
    torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt as _nt
    return _nt


# (format, rows, cols, tokens per launch when the x of several fit): four rows
# per warp (Q4_K, 28672 rows), the 70B down projection's width (two x of 28672
# columns fit), pipeline shapes with four per launch, and widths the pipeline does
# not take (one launch per vector).
CASES = [("q4_k", 28672, 8192, 4), ("q6_k", 1024, 28672, 2), ("q8_0", 1000, 4096, 4), ("q4_0", 300, 2048, 4),
         ("q5_k", 8192, 1024, 4), ("q6_k", 77, 8192, 4), ("q8_0", 37, 1536, 1), ("q4_k", 5, 512, 1)]


@pytest.mark.parametrize("fmt,rows,cols,per_launch", CASES)
@pytest.mark.parametrize("k", [1, 3, 8])
def test_batch_equals_single_token_gemv_and_the_oracle(nt, fmt, rows, cols, per_launch, k):
    torch = torch_cuda()
    t = nt.nt_qtensor_create(fmt, rows, cols, 5, 77, 0.02)
    try:
        xs = [activation(cols, seed=40 + i) for i in range(k)]
        xd = [torch.from_numpy(x).cuda() for x in xs]
        yb = [torch.full((rows,), float("nan"), device="cuda") for _ in range(k)]
        ys = [torch.full((rows,), float("nan"), device="cuda") for _ in range(k)]
        s = torch.cuda.current_stream()
        launches = nt.nt_gemv_q_batch(t, [x.data_ptr() for x in xd], [y.data_ptr() for y in yb], s)
        for x, y in zip(xd, ys):
            nt.nt_gemv_q(t, x.data_ptr(), y.data_ptr(), s)
        torch.cuda.synchronize()
        assert launches == (k + per_launch - 1) // per_launch
        blocks = oracle.qtensor_rows(fmt, rows, cols, 5, 77, 0.02, nthreads=8)
        for i in range(k):
            got, single = yb[i].cpu().numpy(), ys[i].cpu().numpy()
            np.testing.assert_array_equal(got.view(np.uint32), single.view(np.uint32))
            if i in (0, k - 1):
                want = oracle.gemv(fmt, blocks, rows, cols, xs[i], nthreads=8)
                assert rel_l2(got, want) < TOL
    finally:
        nt.nt_qtensor_destroy(t)


def test_batch_argument_checks(nt):
    torch = torch_cuda()
    t = nt.nt_qtensor_create("q8_0", 64, 1024, 0, 1, 0.02)
    try:
        x = torch.zeros(1024, device="cuda")
        ys = [torch.zeros(64, device="cuda") for _ in range(9)]
        with pytest.raises(nt.NtError) as ei:        # more than 8 vectors
            nt.nt_gemv_q_batch(t, [x.data_ptr()] * 9, [y.data_ptr() for y in ys])
        assert ei.value.status == nt.NT_E_INVAL
        with pytest.raises(nt.NtError) as ei:        # two outputs in the same place
            nt.nt_gemv_q_batch(t, [x.data_ptr()] * 2, [ys[0].data_ptr()] * 2)
        assert ei.value.status == nt.NT_E_INVAL
        with pytest.raises(nt.NtError) as ei:        # misaligned output
            nt.nt_gemv_q_batch(t, [x.data_ptr()], [ys[0].data_ptr() + 4])
        assert ei.value.status == nt.NT_E_INVAL
    finally:
        nt.nt_qtensor_destroy(t)
