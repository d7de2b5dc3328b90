"""GPU: the persistent step kernel (one cooperative launch per decode step).

Small models shaped for it (GEMV widths multiples of 1024; the two format plans
it is built for: Q8_0 throughout with four query heads per kv head, and the
Q4_K_M mix with eight), checked against the oracle and bit for bit against the
per-kernel launch path and the layer-streamed path, which share its arithmetic.
"""
import os

import numpy as np
import pytest

import oracle
from gpu_util import ensure_built, rel_l2, torch_cuda

pytestmark = pytest.mark.gpu
MAX_ABS, REL_L2, MARGIN = 1e-2, 5e-3, 1e-2

STEP_Q8_0 = dict(n_layers=3, hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=4096,
                 max_ctx=384)


@pytest.fixture(scope="module")
def nt():
    torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt as _nt
    return _nt


@pytest.fixture(autouse=True)
def step_kernel_on(monkeypatch):
    """The step kernel is opt-in; a model decides at its first step."""
    monkeypatch.setenv("NT_STEP_KERNEL", "1")


@pytest.fixture(scope="module")
def W():
    from quantized_decode_dequant_gb300 import workloads
    return workloads


def step_q4_k_m(W):
    return dict(n_layers=2, hidden=1024, n_heads=8, n_kv_heads=1, head_dim=128, ffn_dim=2048, vocab=4096,
                max_ctx=384, **W.Q4_K_M)


def _uses_step_kernel(nt, m, tok):
    """One profiled step; the step kernel is a single launch split into phases."""
    kt = nt.nt_profile_steps(m, tok, 1)
    return kt.kernel_launches == 1, kt


def test_step_kernel_runs_one_launch_per_step(nt, W):
    spec = STEP_Q8_0
    m = nt.nt_model_create(nt.make_config(**spec, seed=1))
    try:
        nt.nt_kv_prefill(m, 70, 2)
        kt = nt.nt_profile_steps(m, 11, 3)
        assert kt.kernel_launches == 3
        L = spec["n_layers"]
        assert kt.launches[nt.KC_GEMV] == 3 * (4 * L + 1)
        assert kt.launches[nt.KC_ATTN] == 3 * L
        assert kt.launches[nt.KC_OTHER] == 3 * 2
        assert kt.ms[nt.KC_GEMV] > 0 and kt.ms[nt.KC_ATTN] > 0 and kt.step_ms > 0
        total = kt.ms[nt.KC_GEMV] + kt.ms[nt.KC_ATTN] + kt.ms[nt.KC_OTHER]
        assert total == pytest.approx(3 * kt.step_ms, rel=0.05)
    finally:
        nt.nt_model_destroy(m)


@pytest.mark.parametrize("plan", ["q8_0", "q4_k_m"])
def test_step_kernel_teacher_forced_vs_oracle(nt, W, plan):
    spec = STEP_Q8_0 if plan == "q8_0" else step_q4_k_m(W)
    seed, n_ctx = 5, 190       # three full chunks and a ragged one; steps cross no boundary
    m = nt.nt_model_create(nt.make_config(**spec, seed=seed))
    om = oracle.Model(oracle.ModelSpec(**spec, seed=seed), nthreads=os.cpu_count() or 8)
    try:
        nt.nt_kv_prefill(m, n_ctx, W.SEED_KV)
        om.kv_prefill(n_ctx, W.SEED_KV)
        assert _uses_step_kernel(nt, m, 0)[0]
        nt.nt_kv_prefill(m, n_ctx, W.SEED_KV)   # the profiled step advanced the position
        gl = np.empty(spec["vocab"], np.float32)
        for i, tok in enumerate(oracle.tokens(7, 6, spec["vocab"])):
            gnx = nt.nt_decode_step(m, int(tok), gl)
            ol, onx, omg = om.decode_step(int(tok))
            err_abs = float(np.abs(gl.astype(np.float64) - ol).max())
            err_rel = rel_l2(gl, ol)
            assert err_abs <= MAX_ABS and err_rel <= REL_L2, (i, err_abs, err_rel)
            if omg > MARGIN:
                assert gnx == onx, (i, gnx, onx, omg)
        # the cache row the kernel appended at the last position matches the oracle's
        hd = spec["head_dim"]
        for layer in range(spec["n_layers"]):
            for kv in (0, 1):
                got = nt.nt_kv_export(m, layer, kv, 0, n_ctx + 5, 1, hd)[0].view(np.float16).astype(np.float64)
                want = np.array([oracle.f16_to_double(om.kv_get(layer, kv, 0, n_ctx + 5, d)) for d in range(hd)])
                np.testing.assert_allclose(got, want, rtol=2e-3, atol=2e-3 * np.abs(want).max())
    finally:
        om.close()
        nt.nt_model_destroy(m)


@pytest.mark.parametrize("plan", ["q8_0", "q4_k_m"])
def test_step_kernel_bitwise_equals_per_kernel_and_streamed_paths(nt, W, plan, monkeypatch):
    spec = STEP_Q8_0 if plan == "q8_0" else step_q4_k_m(W)
    cfg = nt.make_config(**spec, seed=9)
    a = nt.nt_model_create(cfg)
    monkeypatch.setenv("NT_STEP_KERNEL", "0")
    b = nt.nt_model_create(cfg)
    c = nt.nt_model_create(cfg)
    try:
        for m in (a, b, c):
            nt.nt_kv_prefill(m, 61, W.SEED_KV)   # steps cross the 64-position chunk boundary
        nt.nt_stream_layers(c, 1, 2)
        assert nt.nt_profile_steps(b, 3, 1).kernel_launches > 1
        monkeypatch.setenv("NT_STEP_KERNEL", "1")
        assert _uses_step_kernel(nt, a, 3)[0]
        for m in (a, b, c):
            nt.nt_kv_prefill(m, 61, W.SEED_KV)
        la, lb, lc = (np.empty(spec["vocab"], np.float32) for _ in range(3))
        t = 3
        for _ in range(7):
            na = nt.nt_decode_step(a, t, la)
            nb = nt.nt_decode_step(b, t, lb)
            nc = nt.nt_decode_step(c, t, lc)
            np.testing.assert_array_equal(la.view(np.uint32), lb.view(np.uint32))
            np.testing.assert_array_equal(la.view(np.uint32), lc.view(np.uint32))
            assert na == nb == nc
            t = na
        hd = spec["head_dim"]
        for layer in range(spec["n_layers"]):
            ka = nt.nt_kv_export(a, layer, 0, 0, 0, 68, hd)
            kb = nt.nt_kv_export(b, layer, 0, 0, 0, 68, hd)
            np.testing.assert_array_equal(ka, kb)
    finally:
        for m in (a, b, c):
            nt.nt_model_destroy(m)


def test_step_kernel_device_loop_matches_host_loop(nt, W):
    cfg = nt.make_config(**STEP_Q8_0, seed=2)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        seq, t = [], 17
        for _ in range(12):
            t = nt.nt_decode_step(a, t)
            seq.append(t)
        nt.nt_decode_run(b, 17, 12)
        np.testing.assert_array_equal(nt.nt_get_tokens(b, 0, 12), seq)
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


def test_step_kernel_barrier_timeout_is_reported_and_recovers(nt, W, monkeypatch):
    """A barrier base that the arrivals never reach: every CTA's first wait runs
    into its one-second limit, the step is abandoned with NT_E_TIMEOUT and the
    next step runs normally."""
    cfg = nt.make_config(**STEP_Q8_0, seed=3)
    ref = nt.nt_model_create(cfg)
    monkeypatch.setenv("NT_STEP_BARRIER_OFFSET", "100000")
    m = nt.nt_model_create(cfg)
    try:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_decode_step(m, 5)
        assert ei.value.status == nt.NT_E_TIMEOUT
        assert nt.nt_get_stats(m).pos == 0
        monkeypatch.delenv("NT_STEP_BARRIER_OFFSET")
        lm, lr = np.empty(STEP_Q8_0["vocab"], np.float32), np.empty(STEP_Q8_0["vocab"], np.float32)
        t = 5
        for _ in range(3):
            n1 = nt.nt_decode_step(m, t, lm)
            n2 = nt.nt_decode_step(ref, t, lr)
            np.testing.assert_array_equal(lm.view(np.uint32), lr.view(np.uint32))
            assert n1 == n2
            t = n1
    finally:
        nt.nt_model_destroy(m)
        nt.nt_model_destroy(ref)
