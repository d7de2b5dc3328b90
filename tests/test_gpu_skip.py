"""GPU: layer skip and the per-layer similarity step, against the oracle and
against the unskipped paths.

Cosine tolerance: for residuals a, b with relative L2 errors e_a, e_b the
cosine moves by at most 2 (e_a + e_b); the residual stream of these small
models stays within 2.5e-4 of the oracle's, so |cos_gpu - cos_oracle| <= 1e-3.
"""
import os

import numpy as np
import pytest

import oracle
from gpu_util import ensure_built, rel_l2, torch_cuda

pytestmark = pytest.mark.gpu
MAX_ABS, REL_L2, MARGIN, COS_TOL = 1e-2, 5e-3, 1e-2, 1e-3
SPEC = dict(n_layers=4, hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1536, vocab=4096, max_ctx=96)


@pytest.fixture(scope="module")
def nt():
    torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt as _nt
    return _nt


@pytest.fixture(scope="module")
def W():
    from quantized_decode_dequant_gb300 import workloads
    return workloads


def _bits(a):
    return a.view(np.uint32)


def test_skipping_the_last_layers_equals_a_shallower_model(nt):
    deep = nt.nt_model_create(nt.make_config(**dict(SPEC, n_layers=3), seed=4))
    shallow = nt.nt_model_create(nt.make_config(**dict(SPEC, n_layers=1), seed=4))
    try:
        nt.nt_set_layer_skip(deep, [0, 1, 1])
        ld, ls = np.empty(SPEC["vocab"], np.float32), np.empty(SPEC["vocab"], np.float32)
        t = 12
        for _ in range(5):
            nd, ns = nt.nt_decode_step(deep, t, ld), nt.nt_decode_step(shallow, t, ls)
            np.testing.assert_array_equal(_bits(ld), _bits(ls))
            assert nd == ns
            t = nd
        # the skipped layers wrote no K/V rows
        hd = SPEC["head_dim"]
        assert not nt.nt_kv_export(deep, 2, 0, 1, 0, 5, hd).any()
        # device loop and launch profile follow the mask too
        nt.nt_decode_run(deep, t, 3)
        nt.nt_decode_run(shallow, t, 3)
        np.testing.assert_array_equal(nt.nt_get_tokens(deep, 0, 8), nt.nt_get_tokens(shallow, 0, 8))
        kt = nt.nt_profile_steps(deep, 3, 1)
        assert kt.launches[nt.KC_ATTN] == 1
    finally:
        nt.nt_model_destroy(deep)
        nt.nt_model_destroy(shallow)


@pytest.mark.parametrize("mix", ["q8_0", "q4_k_m"])
def test_skip_teacher_forced_vs_oracle(nt, W, mix):
    spec = dict(SPEC) if mix == "q8_0" else dict(SPEC, **W.Q4_K_M)
    mask = [0, 1, 0, 1]
    m = nt.nt_model_create(nt.make_config(**spec, seed=6))
    om = oracle.Model(oracle.ModelSpec(**spec, seed=6), nthreads=os.cpu_count() or 8)
    try:
        nt.nt_kv_prefill(m, 40, W.SEED_KV)
        om.kv_prefill(40, W.SEED_KV)
        nt.nt_set_layer_skip(m, mask)
        om.set_layer_skip(mask)
        gl = np.empty(spec["vocab"], np.float32)
        for i, tok in enumerate(oracle.tokens(8, 6, spec["vocab"])):
            gnx = nt.nt_decode_step(m, int(tok), gl)
            ol, onx, omg = om.decode_step(int(tok))
            err_abs, err_rel = float(np.abs(gl - ol).max()), rel_l2(gl, ol)
            assert err_abs <= MAX_ABS and err_rel <= REL_L2, (i, err_abs, err_rel)
            if omg > MARGIN:
                assert gnx == onx
    finally:
        om.close()
        nt.nt_model_destroy(m)


def test_layer_similarity_vs_oracle_and_same_step(nt, W):
    spec = SPEC
    a = nt.nt_model_create(nt.make_config(**spec, seed=7))
    b = nt.nt_model_create(nt.make_config(**spec, seed=7))
    om = oracle.Model(oracle.ModelSpec(**spec, seed=7), nthreads=os.cpu_count() or 8)
    try:
        for m in (a, b):
            nt.nt_kv_prefill(m, 33, W.SEED_KV)
        om.kv_prefill(33, W.SEED_KV)
        t = 21
        for i in range(3):
            na, cos = nt.nt_layer_similarity(a, t)
            nb = nt.nt_decode_step(b, t)
            _, onx, _ = om.decode_step(t)
            assert na == nb
            ocos = om.layer_cos()
            assert cos.shape == (spec["n_layers"],)
            np.testing.assert_allclose(cos, ocos, rtol=0, atol=COS_TOL)
            assert np.all(np.abs(cos) <= 1.0 + 1e-12)
            t = na
        # the similarity step left the same cache and position as the plain step
        assert nt.nt_get_stats(a).pos == nt.nt_get_stats(b).pos
        hd = spec["head_dim"]
        for layer in range(spec["n_layers"]):
            np.testing.assert_array_equal(nt.nt_kv_export(a, layer, 1, 0, 33, 3, hd),
                                          nt.nt_kv_export(b, layer, 1, 0, 33, 3, hd))
    finally:
        om.close()
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


def test_streamed_skip_equals_resident_skip_and_copies_fewer_bytes(nt, W):
    spec = dict(SPEC, n_layers=6)
    cfg = nt.make_config(**spec, seed=3)
    res, stm, full = nt.nt_model_create(cfg), nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        nt.nt_stream_layers(stm, 1, 2)
        nt.nt_stream_layers(full, 1, 2)
        # calibrate on the streamed model, then plan and apply the same mask to both
        _, cos = nt.nt_layer_similarity(stm, 5)
        mask = nt.nt_plan_layer_skip(cos, -1.0, 3)          # the three most similar layers
        assert mask.sum() == 3
        for m in (res, stm, full):
            nt.nt_kv_reset(m)
        nt.nt_set_layer_skip(res, mask)
        nt.nt_set_layer_skip(stm, mask)
        lr, ls = np.empty(spec["vocab"], np.float32), np.empty(spec["vocab"], np.float32)
        t = 5
        for _ in range(4):
            nr, ns = nt.nt_decode_step(res, t, lr), nt.nt_decode_step(stm, t, ls)
            nt.nt_decode_step(full, t)
            np.testing.assert_array_equal(_bits(lr), _bits(ls))
            assert nr == ns
            t = nr
        st, sf = nt.nt_get_stats(stm), nt.nt_get_stats(full)
        lay = sf.h2d_bytes / (spec["n_layers"] - 1)
        streamed_skipped = int(mask[1:].sum())
        assert st.h2d_bytes == pytest.approx(sf.h2d_bytes - streamed_skipped * lay, rel=1e-12)
        # clearing the mask brings back the full model
        nt.nt_set_layer_skip(stm, None)
        nt.nt_decode_step(stm, t)
        assert nt.nt_get_stats(stm).h2d_bytes == sf.h2d_bytes
    finally:
        for m in (res, stm, full):
            nt.nt_model_destroy(m)


def test_skipping_every_layer_is_the_zero_layer_model(nt):
    every = nt.nt_model_create(nt.make_config(**dict(SPEC, n_layers=2), seed=5))
    none = nt.nt_model_create(nt.make_config(**dict(SPEC, n_layers=0), seed=5))
    try:
        nt.nt_set_layer_skip(every, [1, 1])
        le, ln = np.empty(SPEC["vocab"], np.float32), np.empty(SPEC["vocab"], np.float32)
        t = 3
        for _ in range(3):
            ne, nn = nt.nt_decode_step(every, t, le), nt.nt_decode_step(none, t, ln)
            np.testing.assert_array_equal(_bits(le), _bits(ln))
            assert ne == nn
            t = ne
        # a speculative cycle whose draft is the whole (empty) remaining model accepts everything
        e, j = nt.nt_speculative_step(every, t, 2, 3)
        assert j == 3 and len(e) == 3
    finally:
        nt.nt_model_destroy(every)
        nt.nt_model_destroy(none)
