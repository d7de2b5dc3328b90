"""GPU: the decode step through nt_decode_step against the oracle (teacher-forced)."""
import os

import numpy as np
import pytest

import oracle
from gpu_util import ensure_built, rel_l2, torch_cuda

pytestmark = pytest.mark.gpu
MAX_ABS, REL_L2, MARGIN = 1e-2, 5e-3, 1e-2


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


def _check_step(gl, gnx, ol, onx, omg, where):
    err_abs = float(np.abs(gl.astype(np.float64) - ol).max())
    err_rel = rel_l2(gl, ol)
    assert err_abs <= MAX_ABS and err_rel <= REL_L2, (where, err_abs, err_rel)
    if omg > MARGIN:
        assert gnx == onx, (where, gnx, onx, omg)
    return err_abs, err_rel


def test_tiny_teacher_forced_64_steps(nt, W):
    m = nt.nt_model_create(nt.make_config(**W.TINY, seed=0))
    om = oracle.Model(oracle.ModelSpec(**W.TINY, seed=0))
    try:
        toks = oracle.tokens(0, W.TINY_STEPS, W.TINY["vocab"])
        gl = np.empty(W.TINY["vocab"], np.float32)
        worst = 0.0
        for i, t in enumerate(toks):
            gnx = nt.nt_decode_step(m, t, gl)
            ol, onx, omg = om.decode_step(t)
            worst = max(worst, _check_step(gl, gnx, ol, onx, omg, i)[0])
        # the cache holds every step's K and V, RoPE'd, in f16
        hd = W.TINY["head_dim"]
        for (l, kv, g, t) in [(0, 0, 0, 0), (1, 1, 1, 63), (0, 0, 1, 31), (1, 1, 0, 5)]:
            got = nt.nt_kv_export(m, l, kv, g, t, 1, hd)[0].view(np.float16).astype(np.float64)
            want = np.array([om.kv_get(l, kv, g, t, d) for d in range(hd)], np.uint16).view(np.float16)
            np.testing.assert_allclose(got, want.astype(np.float64), rtol=2e-3, atol=1e-4)
        st = nt.nt_get_stats(m)
        assert st.pos == W.TINY_STEPS and st.steps == W.TINY_STEPS
        with pytest.raises(nt.NtError) as ei:
            nt.nt_decode_step(m, 0)
        assert ei.value.status == nt.NT_E_INVAL    # position reached max_ctx
    finally:
        nt.nt_model_destroy(m)


WIDE = dict(n_layers=2, hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=2048, vocab=4096, max_ctx=64)


@pytest.mark.parametrize("mix,shape", [("q4_k_m", "tiny"), ("q5_k_m", "tiny"), ("q5_k_m", "wide"),
                                       ("q4_k_m", "wide")])
def test_tiny_mixed_formats_teacher_forced(nt, W, mix, shape):
    """Mixed K-quant formats; 'wide' widths (multiples of 1024) take the shared-memory pipeline everywhere."""
    spec = dict(W.TINY if shape == "tiny" else WIDE, **(W.Q4_K_M if mix == "q4_k_m" else W.Q5_K_M))
    m = nt.nt_model_create(nt.make_config(**spec, seed=4))
    om = oracle.Model(oracle.ModelSpec(**spec, seed=4))
    try:
        gl = np.empty(spec["vocab"], np.float32)
        for i, t in enumerate(oracle.tokens(4, 12, spec["vocab"])):
            gnx = nt.nt_decode_step(m, t, gl)
            ol, onx, omg = om.decode_step(t)
            _check_step(gl, gnx, ol, onx, omg, i)
    finally:
        nt.nt_model_destroy(m)


def test_kv_prefill_bit_exact(nt, W):
    m = nt.nt_model_create(nt.make_config(**W.TINY, seed=0))
    om = oracle.Model(oracle.ModelSpec(**W.TINY, seed=0))
    try:
        nt.nt_kv_prefill(m, 40, 2)
        om.kv_prefill(40, 2)
        hd = W.TINY["head_dim"]
        for (l, kv, g) in [(0, 0, 0), (1, 1, 1), (0, 1, 1)]:
            got = nt.nt_kv_export(m, l, kv, g, 0, 40, hd)
            want = np.array([[om.kv_get(l, kv, g, t, d) for d in range(hd)] for t in range(40)], np.uint16)
            np.testing.assert_array_equal(got, want)
        # decoding on top of the prefilled cache
        gl = np.empty(W.TINY["vocab"], np.float32)
        for i, t in enumerate(oracle.tokens(3, 5, W.TINY["vocab"])):
            gnx = nt.nt_decode_step(m, t, gl)
            ol, onx, omg = om.decode_step(t)
            _check_step(gl, gnx, ol, onx, omg, i)
    finally:
        nt.nt_model_destroy(m)


def test_device_loop_matches_host_loop_and_profile(nt, W):
    cfg = nt.make_config(**W.TINY, seed=0)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        tok = 17
        seq = []
        t = tok
        for _ in range(10):
            t = nt.nt_decode_step(a, t)
            seq.append(t)
        nt.nt_decode_run(b, tok, 10)
        np.testing.assert_array_equal(nt.nt_get_tokens(b, 0, 10), seq)
        nt.nt_kv_reset(b)
        kt = nt.nt_profile_steps(b, tok, 3)
        assert kt.launches[nt.KC_GEMV] == 3 * (4 * W.TINY["n_layers"] + 1)
        assert kt.launches[nt.KC_ATTN] == 3 * W.TINY["n_layers"]
        assert kt.kernel_launches == 3 * (5 * W.TINY["n_layers"] + 3)
        assert kt.ms[nt.KC_GEMV] > 0 and kt.step_ms > 0
        np.testing.assert_array_equal(nt.nt_get_tokens(b, 0, 3), seq[:3])
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


@pytest.mark.parametrize("nr", [2, 0])   # 0: every layer in the page-locked host tier
def test_streamed_layers_bitwise_equal_resident(nt, W, nr):
    spec = dict(W.TINY, n_layers=5)
    cfg = nt.make_config(**spec, seed=6)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        nt.nt_stream_layers(b, nr, 2)
        la = np.empty(spec["vocab"], np.float32)
        lb = np.empty(spec["vocab"], np.float32)
        t = 5
        for _ in range(6):
            na = nt.nt_decode_step(a, t, la)
            nb = nt.nt_decode_step(b, t, lb)
            np.testing.assert_array_equal(la.view(np.uint32), lb.view(np.uint32))
            assert na == nb
            t = na
        st = nt.nt_get_stats(b)
        assert st.n_resident == nr and st.h2d_bytes > 0 and st.h2d_ms > 0
        assert 0.0 <= st.overlap <= 1.0
        # per-layer copy rates: the slowest copied layer is a streamed one
        assert 0 < st.h2d_layer_min_GBs <= st.h2d_layer_max_GBs
        assert nr <= st.h2d_layer_min_idx < spec["n_layers"]
        assert nt.nt_get_stats(a).h2d_layer_min_idx == -1
        # a streamed tensor still exports, but cannot be used in place
        tq = nt.nt_model_tensor(b, 4, "q")
        from gpu_util import blocks
        qk, bb = blocks("q8_0")
        got = nt.nt_qtensor_export(tq, 0, 2, qk, bb, spec["hidden"])
        want = oracle.qtensor_rows("q8_0", 512, 512, 6, oracle.uid_layer(4, "q"), 0.02, row0=0, nrows=2)
        np.testing.assert_array_equal(got, want)
        with pytest.raises(nt.NtError) as ei:
            nt.nt_gemv_q(tq, 0, 0)
        assert ei.value.status in (nt.NT_E_STATE, nt.NT_E_INVAL)
        # back to fully resident
        nt.nt_stream_layers(b, spec["n_layers"], 2)
        na = nt.nt_decode_step(a, t, la)
        nb = nt.nt_decode_step(b, t, lb)
        np.testing.assert_array_equal(la.view(np.uint32), lb.view(np.uint32))
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


def test_argument_and_resource_errors(nt, W):
    with pytest.raises(nt.NtError) as ei:
        nt.nt_model_create(nt.make_config(**dict(W.TINY, n_kv_heads=3)))
    assert ei.value.status == nt.NT_E_INVAL
    m = nt.nt_model_create(nt.make_config(**W.TINY))
    try:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_decode_step(m, W.TINY["vocab"])
        assert ei.value.status == nt.NT_E_INVAL
        with pytest.raises(nt.NtError):
            nt.nt_kv_prefill(m, W.TINY["max_ctx"] + 1, 0)
        with pytest.raises(nt.NtError) as ei:
            nt.nt_stream_layers(m, 1, 3)
        assert ei.value.status == nt.NT_E_UNSUPPORTED
    finally:
        nt.nt_model_destroy(m)
    os.environ["NT_DEVICE_BYTES_LIMIT"] = str(1 << 20)
    try:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_model_create(nt.make_config(**W.TINY))
        assert ei.value.status == nt.NT_E_NOMEM
    finally:
        del os.environ["NT_DEVICE_BYTES_LIMIT"]


@pytest.mark.parametrize("nr", [1, 0])
def test_streamed_q4_k_m_layers_bitwise_equal_resident(nt, W, nr):
    """The Q4_K_M mix at whole-tile widths, layers streamed through the staging
    buffers: the two-format Q/K/V launch (Q4_K Q/K, Q6_K V rows one per warp),
    the Q4_K O and gate/up and the Q6_K down read staging buffers, and every
    step's logits equal the resident model's bit for bit."""
    spec = dict(WIDE, n_layers=3, **W.Q4_K_M)
    cfg = nt.make_config(**spec, seed=8)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        for m in (a, b):
            nt.nt_kv_prefill(m, 17, 2)
        nt.nt_stream_layers(b, nr, 2)
        la = np.empty(spec["vocab"], np.float32)
        lb = np.empty(spec["vocab"], np.float32)
        t = 11
        for _ in range(5):
            na = nt.nt_decode_step(a, t, la)
            nb = nt.nt_decode_step(b, t, lb)
            np.testing.assert_array_equal(la.view(np.uint32), lb.view(np.uint32))
            assert na == nb
            t = na
        st = nt.nt_get_stats(b)
        assert st.n_resident == nr and st.h2d_bytes > 0
        hd = spec["head_dim"]
        for layer in range(spec["n_layers"]):
            for kv in (0, 1):
                np.testing.assert_array_equal(nt.nt_kv_export(a, layer, kv, 1, 0, 22, hd),
                                              nt.nt_kv_export(b, layer, kv, 1, 0, 22, hd))
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


def test_llama8b_q8_0_teacher_forced(nt, W):
    """8B shape at full size: prefilled context 512, prompt token, GPU's own greedy tokens fed to both."""
    spec = W.LLAMA_8B_Q8_0
    nthreads = os.cpu_count() or 8
    m = nt.nt_model_create(nt.make_config(**spec, seed=W.SEED_WEIGHTS))
    try:
        nt.nt_kv_prefill(m, W.LLAMA_8B_CTX, W.SEED_KV)
        om = oracle.Model(oracle.ModelSpec(**spec, seed=W.SEED_WEIGHTS), nthreads=nthreads)
        om.kv_prefill(W.LLAMA_8B_CTX, W.SEED_KV)
        gl = np.empty(spec["vocab"], np.float32)
        tok = oracle.token(W.SEED_PROMPT, oracle.UID_TOKENS, 0, spec["vocab"])
        worst = (0.0, 0.0)
        for i in range(int(os.environ.get("NT_8B_STEPS", "16"))):
            gnx = nt.nt_decode_step(m, tok, gl)
            ol, onx, omg = om.decode_step(tok)
            e = _check_step(gl, gnx, ol, onx, omg, i)
            worst = (max(worst[0], e[0]), max(worst[1], e[1]))
            tok = gnx
        print(f"8B worst over {i + 1} steps: max-abs {worst[0]:.3e} rel-L2 {worst[1]:.3e}")
    finally:
        nt.nt_model_destroy(m)


def _teacher_forced(nt, m, om, spec, ctx, steps, W, where, also=None):
    """Prefilled context ctx on both sides, the prompt token, then the GPU's own
    greedy tokens fed to both; logits checked at every step.  also(m2): a second
    device model stepped alongside that must give bit-identical logits."""
    nt.nt_kv_prefill(m, ctx, W.SEED_KV)
    om.kv_prefill(ctx, W.SEED_KV)
    if also is not None:
        nt.nt_kv_prefill(also, ctx, W.SEED_KV)
    gl = np.empty(spec["vocab"], np.float32)
    al = np.empty(spec["vocab"], np.float32)
    tok = oracle.token(W.SEED_PROMPT, oracle.UID_TOKENS, 0, spec["vocab"])
    worst = (0.0, 0.0)
    for i in range(steps):
        gnx = nt.nt_decode_step(m, tok, gl)
        if also is not None:
            anx = nt.nt_decode_step(also, tok, al)
            np.testing.assert_array_equal(gl.view(np.uint32), al.view(np.uint32))
            assert anx == gnx
        ol, onx, omg = om.decode_step(tok)
        e = _check_step(gl, gnx, ol, onx, omg, (where, i))
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
        tok = gnx
    print(f"{where}: worst over {steps} steps max-abs {worst[0]:.3e} rel-L2 {worst[1]:.3e}")
    return worst


def test_llama70b_widths_q4_k_m_4_layers_ctx4096(nt, W):
    """The 70B Q4_K_M workload's kernels at full width with 4 layers: 8192-wide
    two-format Q/K/V launch (Q4_K q/k, Q6_K v), 64/8 heads attended over 4097+
    cached positions in 256-position items, four-rows-per-warp Q4_K O and
    gate/up, Q6_K down and 128256-row Q6_K head; ctx 4096, 4 teacher-forced steps."""
    spec = dict(W.LLAMA_70B_Q4_K_M, n_layers=4)
    m = nt.nt_model_create(nt.make_config(**spec, seed=W.SEED_WEIGHTS))
    om = oracle.Model(oracle.ModelSpec(**spec, seed=W.SEED_WEIGHTS), nthreads=os.cpu_count() or 8)
    try:
        _teacher_forced(nt, m, om, spec, W.LLAMA_70B_Q4_K_M_CTX, 4, W, "70B-width Q4_K_M 4 layers")
    finally:
        om.close()
        nt.nt_model_destroy(m)


def test_llama70b_widths_q6_k_2_resident_2_streamed_ctx1024(nt, W):
    """The streamed 70B Q6_K workload's path at full width with 4 layers, 2 of
    them copied from page-locked host memory into the staging buffers every step
    (so the pipeline GEMVs read staging buffers): against the oracle, and bit for
    bit against the same model held resident; ctx 1024, 3 teacher-forced steps."""
    spec = dict(W.LLAMA_70B_Q6_K, n_layers=4)
    cfg = nt.make_config(**spec, seed=W.SEED_WEIGHTS)
    stm, res = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    om = oracle.Model(oracle.ModelSpec(**spec, seed=W.SEED_WEIGHTS), nthreads=os.cpu_count() or 8)
    try:
        nt.nt_stream_layers(stm, 2, 2)
        _teacher_forced(nt, stm, om, spec, W.LLAMA_70B_Q6_K_CTX, 3, W, "70B-width Q6_K 2+2 streamed", also=res)
        st = nt.nt_get_stats(stm)
        assert st.n_resident == 2 and st.h2d_bytes > 0
    finally:
        om.close()
        nt.nt_model_destroy(stm)
        nt.nt_model_destroy(res)


@pytest.mark.slow
@pytest.mark.skipif(os.environ.get("NT_RUN_SLOW") != "1", reason="70B oracle takes minutes per step; NT_RUN_SLOW=1")
def test_llama70b_q4_k_m_teacher_forced(nt, W):
    spec = W.LLAMA_70B_Q4_K_M
    m = nt.nt_model_create(nt.make_config(**spec, seed=W.SEED_WEIGHTS))
    try:
        nt.nt_kv_prefill(m, W.LLAMA_70B_Q4_K_M_CTX, W.SEED_KV)
        om = oracle.Model(oracle.ModelSpec(**spec, seed=W.SEED_WEIGHTS), lazy=True, nthreads=os.cpu_count() or 8)
        om.kv_prefill(W.LLAMA_70B_Q4_K_M_CTX, W.SEED_KV)
        gl = np.empty(spec["vocab"], np.float32)
        tok = oracle.token(W.SEED_PROMPT, oracle.UID_TOKENS, 0, spec["vocab"])
        for i in range(int(os.environ.get("NT_70B_STEPS", "2"))):
            gnx = nt.nt_decode_step(m, tok, gl)
            ol, onx, omg = om.decode_step(tok)
            e = _check_step(gl, gnx, ol, onx, omg, i)
            print(f"70B step {i}: max-abs {e[0]:.3e} rel-L2 {e[1]:.3e} margin {omg:.3e}")
            tok = gnx
    finally:
        nt.nt_model_destroy(m)


@pytest.mark.slow
@pytest.mark.skipif(os.environ.get("NT_RUN_SLOW") != "1", reason="70B oracle takes minutes per step; NT_RUN_SLOW=1")
def test_llama70b_q6_k_streamed_teacher_forced_and_equal_to_resident(nt, W):
    """70B all-Q6_K, 26 layers resident and 54 streamed: against the oracle, and bit for bit
    against the same model held entirely in device memory."""
    spec = W.LLAMA_70B_Q6_K
    cfg = nt.make_config(**spec, seed=W.SEED_WEIGHTS)
    stm, res = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        nt.nt_stream_layers(stm, W.LLAMA_70B_Q6_K_RESIDENT, 2)
        for m in (stm, res):
            nt.nt_kv_prefill(m, W.LLAMA_70B_Q6_K_CTX, W.SEED_KV)
        om = oracle.Model(oracle.ModelSpec(**spec, seed=W.SEED_WEIGHTS), lazy=True, nthreads=os.cpu_count() or 8)
        om.kv_prefill(W.LLAMA_70B_Q6_K_CTX, W.SEED_KV)
        gl, rl = np.empty(spec["vocab"], np.float32), np.empty(spec["vocab"], np.float32)
        tok = oracle.token(W.SEED_PROMPT, oracle.UID_TOKENS, 0, spec["vocab"])
        for i in range(int(os.environ.get("NT_70B_STEPS", "2"))):
            gnx = nt.nt_decode_step(stm, tok, gl)
            rnx = nt.nt_decode_step(res, tok, rl)
            np.testing.assert_array_equal(gl.view(np.uint32), rl.view(np.uint32))
            assert gnx == rnx
            assert nt.nt_get_stats(stm).h2d_bytes > 0
            ol, onx, omg = om.decode_step(tok)
            e = _check_step(gl, gnx, ol, onx, omg, i)
            print(f"70B Q6_K streamed step {i}: max-abs {e[0]:.3e} rel-L2 {e[1]:.3e} margin {omg:.3e}")
            tok = gnx
        om.close()
    finally:
        nt.nt_model_destroy(stm)
        nt.nt_model_destroy(res)


def test_auto_residency_places_layers_and_decodes_the_same(nt, W):
    """nt_auto_residency keeps a model that fits resident; with a margin that
    leaves room for only a few layers it streams the rest, bit for bit the same."""
    import torch
    spec = dict(W.TINY, n_layers=6)
    cfg = nt.make_config(**spec, seed=8)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        assert nt.nt_auto_residency(a, 1 << 30) == spec["n_layers"]
        _, dev_all, lay = nt.nt_plan_residency(cfg, 1 << 50)
        fixed = dev_all - spec["n_layers"] * lay
        free, _ = torch.cuda.mem_get_info()
        margin = free + dev_all - (fixed + 5 * lay)          # about three layers resident
        n = nt.nt_auto_residency(b, margin)
        assert 1 <= n < spec["n_layers"]
        assert nt.nt_get_stats(b).n_resident == n
        la, lb = np.empty(spec["vocab"], np.float32), np.empty(spec["vocab"], np.float32)
        t = 9
        for _ in range(4):
            na, nb = nt.nt_decode_step(a, t, la), nt.nt_decode_step(b, t, lb)
            np.testing.assert_array_equal(la.view(np.uint32), lb.view(np.uint32))
            assert na == nb
            t = na
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


def test_two_models_in_two_threads_match_sequential_runs(nt, W):
    """One model per host thread: concurrent steps (first launches included) give
    the same logits as the same models stepped one after the other."""
    import threading
    specs = [dict(WIDE, **W.Q4_K_M), dict(WIDE, n_layers=3)]

    def run(spec, seed, out):
        m = nt.nt_model_create(nt.make_config(**spec, seed=seed))
        try:
            lg = np.empty(spec["vocab"], np.float32)
            t, logs = 7, []
            for _ in range(6):
                t = nt.nt_decode_step(m, t, lg)
                logs.append(lg.copy())
            out.extend(logs)
        finally:
            nt.nt_model_destroy(m)

    seq = [[], []]
    for i, sp in enumerate(specs):
        run(sp, 20 + i, seq[i])
    par = [[], []]
    th = [threading.Thread(target=run, args=(sp, 20 + i, par[i])) for i, sp in enumerate(specs)]
    for x in th:
        x.start()
    for x in th:
        x.join()
    for i in range(2):
        assert len(par[i]) == 6
        for a, b in zip(seq[i], par[i]):
            np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
