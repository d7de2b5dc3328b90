"""Helpers for the GPU tests: device buffers through torch, error metrics."""
import numpy as np
import pytest


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def ensure_built():
    import __graft_entry__
    __graft_entry__.build()


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def blocks(fmt):
    from quantized_decode_dequant_gb300 import workloads as W
    return W.BLOCK_ELEMS[fmt], W.BLOCK_BYTES[fmt]
