"""GPU: self-speculative decoding (resident layers as the draft) against plain
greedy decoding on the device and against the oracle's cycle reference."""
import os

import numpy as np
import pytest

import oracle
from gpu_util import ensure_built, torch_cuda

pytestmark = pytest.mark.gpu
MARGIN = 1e-2
SPEC = dict(n_layers=3, hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1536, vocab=512, max_ctx=96)


@pytest.fixture(scope="module")
def nt():
    torch_cuda()
    ensure_built()
    from quantized_decode_dequant_gb300 import nt as _nt
    return _nt


def _greedy(nt, cfg, token, n, prefill):
    m = nt.nt_model_create(cfg)
    try:
        nt.nt_kv_prefill(m, *prefill)
        out, t = [], token
        for _ in range(n):
            t = nt.nt_decode_step(m, t)
            out.append(t)
        return out
    finally:
        nt.nt_model_destroy(m)


def _cycles(nt, m, token, n_draft, k, n_cycles):
    out, t = [], token
    for _ in range(n_cycles):
        emitted, j = nt.nt_speculative_step(m, t, n_draft, k)
        out.append((emitted, j))
        t = emitted[-1]
    return out


@pytest.mark.parametrize("n_draft,k,resident", [(3, 4, 3), (1, 4, 3), (1, 3, 1), (0, 2, 3), (2, 8, 2), (2, 3, 1)])
def test_speculative_stream_equals_greedy_and_the_oracle(nt, n_draft, k, resident):
    cfg = nt.make_config(**SPEC, seed=12)
    prefill = (20, 2)
    m = nt.nt_model_create(cfg)
    try:
        nt.nt_kv_prefill(m, *prefill)
        if resident < SPEC["n_layers"]:
            nt.nt_stream_layers(m, resident, 2)
        cycles = _cycles(nt, m, 9, n_draft, k, 6)
        stream = [t for e, _ in cycles for t in e]
        assert nt.nt_get_stats(m).pos == prefill[0] + len(stream)
        for e, j in cycles:
            assert 0 <= j <= k and len(e) == (j + 1 if j < k else k)
        if n_draft == SPEC["n_layers"]:
            assert all(j == k for _, j in cycles)
        # bit-exact property: the emitted stream is the device's own greedy stream
        assert stream == _greedy(nt, cfg, 9, len(stream), prefill)
        # the history holds the emitted tokens, and plain decoding continues from the cycle's end
        np.testing.assert_array_equal(nt.nt_get_tokens(m, prefill[0], len(stream)), stream)
        nxt = nt.nt_decode_step(m, stream[-1])
        assert nxt == _greedy(nt, cfg, 9, len(stream) + 1, prefill)[-1]
    finally:
        nt.nt_model_destroy(m)
    # the oracle's cycles.  Cycles are exact only while every greedy margin is above
    # the near-tie bar; seed 12 with this prefill and token keeps all of them above
    # 0.02 for 50 steps (checked with the oracle), so the comparison always runs.
    ospec = oracle.ModelSpec(**SPEC, seed=12)
    want = oracle.speculative_cycles(ospec, n_draft, k, 9, 6, prefill=prefill, nthreads=os.cpu_count() or 8)
    om = oracle.Model(ospec, nthreads=os.cpu_count() or 8)
    om.kv_prefill(*prefill)
    t, margins = 9, []
    for _ in range(len(stream)):
        _, t, mg = om.decode_step(t)
        margins.append(mg)
    om.close()
    assert min(margins) > MARGIN, margins
    assert cycles == [(list(e), j) for e, j in want]


# widths of whole 1024-column tiles: the verification's GEMVs run several tokens
# per launch; seed 54 keeps every greedy margin above 0.018 for 50 steps (checked
# with the oracle), so the comparison with the oracle's cycles always runs
WIDE = dict(n_layers=3, hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=2048, vocab=512, max_ctx=96)


@pytest.mark.parametrize("n_draft,k,resident", [(1, 4, 3), (0, 8, 3), (2, 3, 1)])
def test_multi_token_verification_equals_greedy_and_the_oracle(nt, n_draft, k, resident):
    cfg = nt.make_config(**WIDE, seed=54)
    prefill = (20, 2)
    m = nt.nt_model_create(cfg)
    try:
        nt.nt_kv_prefill(m, *prefill)
        if resident < WIDE["n_layers"]:
            nt.nt_stream_layers(m, resident, 2)
        cycles = []
        t = 9
        layer_bytes = sum(nt.nt_qtensor_info(nt.nt_model_tensor(m, 0, r))[3] for r in range(7))
        for _ in range(4):
            e, j = nt.nt_speculative_step(m, t, n_draft, k)
            cycles.append((e, j))
            t = e[-1]
            # the verified layers' weights are read fewer than k times per cycle
            vb = nt.nt_get_stats(m).verify_weight_bytes
            assert 0 < vb < k * layer_bytes * (WIDE["n_layers"] - n_draft)
        stream = [x for e, _ in cycles for x in e]
        assert stream == _greedy(nt, cfg, 9, len(stream), prefill)
    finally:
        nt.nt_model_destroy(m)
    ospec = oracle.ModelSpec(**WIDE, seed=54)
    want = oracle.speculative_cycles(ospec, n_draft, k, 9, 4, prefill=prefill, nthreads=os.cpu_count() or 8)
    assert cycles == [(list(e), j) for e, j in want]


def test_streamed_verification_copies_each_layer_once_per_cycle(nt):
    cfg = nt.make_config(**dict(SPEC, n_layers=4), seed=3)
    m = nt.nt_model_create(cfg)
    try:
        nt.nt_stream_layers(m, 1, 2)
        t = 5
        nt.nt_decode_step(m, t)
        per_step = nt.nt_get_stats(m).h2d_bytes          # three streamed layers
        nt.nt_kv_reset(m)
        for k in (1, 4, 8):
            e, _ = nt.nt_speculative_step(m, t, 1, k)
            assert nt.nt_get_stats(m).h2d_bytes == per_step   # draft layers are resident: copies only in the verification
            t = e[-1]
    finally:
        nt.nt_model_destroy(m)


def test_speculative_argument_checks(nt):
    m = nt.nt_model_create(nt.make_config(**dict(SPEC, max_ctx=8), seed=1))
    try:
        for args in [(0, 1, 0), (0, 1, 9), (0, 4, 2), (SPEC["vocab"], 1, 2), (0, -1, 2)]:
            with pytest.raises(nt.NtError) as ei:
                nt.nt_speculative_step(m, *args)
            assert ei.value.status == nt.NT_E_INVAL
        nt.nt_kv_prefill(m, 6, 2)
        with pytest.raises(nt.NtError):
            nt.nt_speculative_step(m, 0, 1, 3)      # 6 + 3 > max_ctx
        e, _ = nt.nt_speculative_step(m, 0, 1, 2)
        assert 1 <= len(e) <= 2
    finally:
        nt.nt_model_destroy(m)


def test_cycles_follow_draft_depth_k_and_skip_changes_on_one_model(nt):
    """One resident model through cycles of changing (n_draft, k) and a layer-skip
    change in between: each cycle's work must follow its own settings (the
    captured cycle is rebuilt or discarded), so the emitted stream equals a
    second model's plain greedy steps from the same state, bit for bit."""
    cfg = nt.make_config(**WIDE, seed=54)
    prefill = (20, 2)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        for m in (a, b):
            nt.nt_kv_prefill(m, *prefill)
        t_a = t_b = 9
        stream_a, stream_b = [], []
        schedule = [(1, 4), (1, 4), (2, 3), (1, 4), (0, 2), (2, 3)]
        for i, (n_draft, k) in enumerate(schedule):
            if i == 3:   # skip layer 1 from here on, in both models
                mask = np.zeros(WIDE["n_layers"], dtype=np.uint8)
                mask[1] = 1
                for m in (a, b):
                    nt.nt_set_layer_skip(m, mask)
            e, _ = nt.nt_speculative_step(a, t_a, n_draft, k)
            stream_a += list(e)
            t_a = e[-1]
            for _ in range(len(e)):
                t_b = nt.nt_decode_step(b, t_b)
                stream_b.append(t_b)
            assert stream_a == stream_b, (i, stream_a, stream_b)
        assert nt.nt_get_stats(a).pos == nt.nt_get_stats(b).pos
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)


# the Q4_K_M-style mix at whole-tile widths: Q/K in Q4_K and V in Q6_K go through the
# two-format Q/K/V launch, and in the verification through its two multi-token launches
Q4_K_M_WIDE = dict(WIDE, t_embd="q4_k", t_q="q4_k", t_k="q4_k", t_v="q6_k", t_o="q4_k", t_gate="q4_k",
                   t_up="q4_k", t_down="q6_k", t_out="q6_k")


@pytest.mark.parametrize("n_draft,k,resident", [(1, 4, 3), (0, 3, 3), (1, 4, 1)])
def test_verification_writes_the_kv_rows_of_plain_steps_bit_for_bit(nt, n_draft, k, resident):
    """Every K and V row a speculative cycle leaves in the cache (draft steps and
    multi-token verification, Q4_K_M mix, verified layers resident or read from
    the staging buffers) equals, bit for bit, the row plain greedy steps of a
    resident model write for the same tokens: the multi-token launches reproduce
    the single-token arithmetic row for row."""
    cfg = nt.make_config(**Q4_K_M_WIDE, seed=54)
    prefill = (20, 2)
    a, b = nt.nt_model_create(cfg), nt.nt_model_create(cfg)
    try:
        for m in (a, b):
            nt.nt_kv_prefill(m, *prefill)
        if resident < WIDE["n_layers"]:
            nt.nt_stream_layers(a, resident, 2)
        t_a = t_b = 9
        stream_a, stream_b = [], []
        for _ in range(4):
            e, _ = nt.nt_speculative_step(a, t_a, n_draft, k)
            stream_a += list(e)
            t_a = e[-1]
            for _ in range(len(e)):
                t_b = nt.nt_decode_step(b, t_b)
                stream_b.append(t_b)
        assert stream_a == stream_b
        pos = nt.nt_get_stats(a).pos
        assert pos == nt.nt_get_stats(b).pos == prefill[0] + len(stream_a)
        hd = WIDE["head_dim"]
        for layer in range(WIDE["n_layers"]):
            for kv in (0, 1):
                for g in range(WIDE["n_kv_heads"]):
                    ra = nt.nt_kv_export(a, layer, kv, g, 0, pos, hd)
                    rb = nt.nt_kv_export(b, layer, kv, g, 0, pos, hd)
                    np.testing.assert_array_equal(ra, rb, err_msg=f"layer {layer} kv {kv} head {g}")
    finally:
        nt.nt_model_destroy(a)
        nt.nt_model_destroy(b)
