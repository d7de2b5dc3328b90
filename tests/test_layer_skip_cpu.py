"""Layer-skip plan (nt_plan_layer_skip): host arithmetic checked against the oracle's plan."""
import numpy as np
import pytest

import oracle
from quantized_decode_dequant_gb300 import nt


@pytest.fixture(scope="module")
def lib():
    try:
        nt.lib()
    except nt.NtLibraryMissing:
        import __graft_entry__
        __graft_entry__.build()
    return nt


def test_plan_matches_the_oracle_plan(lib):
    rng = np.random.default_rng(5)
    for n in (0, 1, 7, 80):
        cos = np.round(rng.uniform(0.9, 1.0, n), 3)   # rounded so that ties occur
        for thr in (0.9, 0.95, 0.98, 1.0):
            for cap in (0, 1, 5, 20, 200):
                got = lib.nt_plan_layer_skip(cos, thr, cap)
                np.testing.assert_array_equal(got, oracle.plan_layer_skip(cos, thr, cap))


def test_plan_cases(lib):
    cos = [0.5, 0.99, 0.97, 0.98, 0.995, 0.99]
    np.testing.assert_array_equal(lib.nt_plan_layer_skip(cos, 0.98), [0, 1, 0, 1, 1, 1])
    np.testing.assert_array_equal(lib.nt_plan_layer_skip(cos, 0.98, 2), [0, 1, 0, 0, 1, 0])
    np.testing.assert_array_equal(lib.nt_plan_layer_skip(cos, 2.0), [0] * 6)
    assert lib.lib().nt_plan_layer_skip(None, 3, 0.5, 0, None, None) == lib.NT_E_INVAL
    assert lib.lib().nt_plan_layer_skip(None, 0, 0.5, 0, None, None) == lib.NT_OK
