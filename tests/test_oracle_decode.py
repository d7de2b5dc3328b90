"""Pins of the oracle's decode step through cases that reduce to its pinned parts."""
import numpy as np
import pytest

import oracle
from oracle import ModelSpec

TINY = dict(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1536, vocab=4096, max_ctx=64)


def _spec(**kw):
    d = dict(TINY)
    d.update(kw)
    return ModelSpec(**d)


def _w(spec, role, layer=0):
    rows, cols, fmt = {
        "q": (spec.n_heads * spec.head_dim, spec.hidden, spec.t_q),
        "k": (spec.n_kv_heads * spec.head_dim, spec.hidden, spec.t_k),
        "v": (spec.n_kv_heads * spec.head_dim, spec.hidden, spec.t_v),
        "o": (spec.hidden, spec.n_heads * spec.head_dim, spec.t_o),
        "gate": (spec.ffn_dim, spec.hidden, spec.t_gate),
        "up": (spec.ffn_dim, spec.hidden, spec.t_up),
        "down": (spec.hidden, spec.ffn_dim, spec.t_down),
    }[role]
    return fmt, rows, cols, oracle.qtensor_rows(fmt, rows, cols, spec.seed, oracle.uid_layer(layer, role),
                                                 spec.init_std)


def _embed(spec, tok):
    b = oracle.qtensor_rows(spec.t_embd, spec.vocab, spec.hidden, spec.seed, oracle.UID_EMBD, spec.init_std,
                            row0=tok, nrows=1)
    return oracle.dequant_row(spec.t_embd, b[0], spec.hidden).astype(np.float64)


def _logits(spec, x):
    b = oracle.qtensor_rows(spec.t_out, spec.vocab, spec.hidden, spec.seed, oracle.UID_OUTPUT, spec.init_std)
    return oracle.gemv(spec.t_out, b, spec.vocab, spec.hidden, oracle.rmsnorm(x, spec.rms_eps))


def test_zero_layer_model_is_norm_then_output_gemv():
    spec = _spec(n_layers=0, vocab=512)
    m = oracle.Model(spec)
    tok = 77
    lg, nx, mg = m.decode_step(tok)
    want = _logits(spec, _embed(spec, tok))
    np.testing.assert_array_equal(lg, want)
    i, marg = oracle.argmax(want)
    assert nx == i and mg == marg and m.pos == 1


def test_one_layer_at_position_zero_reduces_to_gemvs():
    # With one cached position softmax has a single weight 1, so every query head
    # j returns V of its group g = j // (n_heads / n_kv_heads), rounded to binary16.
    spec = _spec(n_layers=1, vocab=512, t_v="q6_k", t_down="q4_k", t_gate="q4_0")
    m = oracle.Model(spec)
    tok = 5
    lg, nx, _ = m.decode_step(tok)

    def gemv(role, x):
        fmt, rows, cols, b = _w(spec, role)
        return oracle.gemv(fmt, b, rows, cols, x)

    x = _embed(spec, tok)
    xn = oracle.rmsnorm(x, spec.rms_eps)
    v = gemv("v", xn)
    v16 = v.astype(np.float16).astype(np.float64)
    hd, group = spec.head_dim, spec.n_heads // spec.n_kv_heads
    o = np.concatenate([v16[(j // group) * hd:(j // group + 1) * hd] for j in range(spec.n_heads)])
    x = x + gemv("o", o)
    xn = oracle.rmsnorm(x, spec.rms_eps)
    g, u = gemv("gate", xn), gemv("up", xn)
    h = np.array([oracle.silu(a) for a in g]) * u
    x = x + gemv("down", h)
    want = _logits(spec, x)
    np.testing.assert_allclose(lg, want, rtol=1e-12, atol=1e-13)
    assert nx == oracle.argmax(want)[0]
    # the stored value at position 0 is the binary16 rounding of v
    for d in (0, 1, 63):
        assert m.kv_get(0, 1, 1, 0, d) == int(np.float16(v[hd + d]).view(np.uint16))


def test_all_zero_weights_give_zero_logits():
    m = oracle.Model(_spec(init_std=0.0))
    for tok in (0, 9):
        lg, nx, mg = m.decode_step(tok)
        assert not lg.any() and nx == 0 and mg == 0.0


def test_kv_prefill_is_rounded_unit_normal():
    spec = _spec()
    m = oracle.Model(spec)
    m.kv_prefill(10, seed=2)
    assert m.pos == 10
    for (l, kv, g, t, d) in [(0, 0, 0, 0, 0), (1, 1, 1, 9, 63), (0, 1, 1, 3, 17)]:
        i = (t * spec.n_kv_heads + g) * spec.head_dim + d
        z = oracle.normal(2, oracle.uid_kv(l, kv), i)
        assert m.kv_get(l, kv, g, t, d) == int(np.float16(z).view(np.uint16))


def test_decode_deterministic_lazy_equals_resident_and_position_limit():
    spec = _spec(max_ctx=4)
    a, b = oracle.Model(spec), oracle.Model(spec, lazy=True, nthreads=3)
    toks = oracle.tokens(0, 4, spec.vocab)
    for t in toks:
        la, na, _ = a.decode_step(t)
        lb, nb, _ = b.decode_step(t)
        np.testing.assert_array_equal(la, lb)
        assert na == nb
    with pytest.raises(RuntimeError):
        a.decode_step(0)
    a.kv_reset()
    assert a.pos == 0
    l0, _, _ = a.decode_step(toks[0])
    c = oracle.Model(spec)
    l1, _, _ = c.decode_step(toks[0])
    np.testing.assert_array_equal(l0, l1)


# ---- layer skip (cosine similarity between the residual entering and leaving a layer)

def test_cosine_closed_forms():
    a = np.array([3.0, 4.0])
    assert oracle.cosine(a, np.array([4.0, 3.0])) == pytest.approx(24 / 25, abs=1e-15)
    assert oracle.cosine(np.array([1.0, 0.0]), np.array([0.0, 2.0])) == 0.0
    assert oracle.cosine(a, 2.5 * a) == pytest.approx(1.0, abs=1e-15)
    assert oracle.cosine(a, -a) == pytest.approx(-1.0, abs=1e-15)
    assert oracle.cosine(a, np.zeros(2)) == 0.0
    # 45 degrees: (1, 0) against (1, 1)
    assert oracle.cosine(np.array([1.0, 0.0]), np.array([1.0, 1.0])) == pytest.approx(np.sqrt(0.5), abs=1e-15)


def test_skipping_the_last_layers_equals_a_shallower_model():
    deep, shallow = oracle.Model(_spec(n_layers=3)), oracle.Model(_spec(n_layers=1))
    deep.set_layer_skip([0, 1, 1])
    for t in oracle.tokens(4, 3, TINY["vocab"]):
        ld, nd, md = deep.decode_step(t)
        ls, ns, ms = shallow.decode_step(t)
        np.testing.assert_array_equal(ld, ls)
        assert (nd, md) == (ns, ms)
        np.testing.assert_array_equal(deep.hidden(), shallow.hidden())
    # skipped layers write no K/V row and report similarity 1
    assert all(deep.kv_get(l, kv, g, 2, d) == 0 for l in (1, 2) for kv in (0, 1) for g in (0, 1) for d in (0, 63))
    assert deep.kv_get(0, 0, 0, 2, 0) == shallow.kv_get(0, 0, 0, 2, 0)
    np.testing.assert_array_equal(deep.layer_cos()[1:], [1.0, 1.0])
    # skipping every layer is the zero-layer model
    every, none = oracle.Model(_spec(n_layers=2)), oracle.Model(_spec(n_layers=0))
    every.set_layer_skip([1, 1])
    np.testing.assert_array_equal(every.decode_step(9)[0], none.decode_step(9)[0])
    # clearing the mask restores the full model
    full, cleared = oracle.Model(_spec()), oracle.Model(_spec())
    cleared.set_layer_skip([1, 0])
    cleared.set_layer_skip(None)
    np.testing.assert_array_equal(full.decode_step(3)[0], cleared.decode_step(3)[0])


def test_layer_similarity_is_the_cosine_of_consecutive_residuals():
    # layer L-1's similarity compares the residuals after L-1 and after L layers,
    # which the (L-1)- and L-layer models give independently
    toks = oracle.tokens(6, 3, TINY["vocab"])
    models = [oracle.Model(_spec(n_layers=n)) for n in (1, 2, 3)]
    for t in toks:
        for m in models:
            m.decode_step(t)
    h = [_embed(_spec(), toks[-1])] + [m.hidden() for m in models]
    for n in (1, 2, 3):
        cos = models[n - 1].layer_cos()
        assert cos[n - 1] == pytest.approx(oracle.cosine(h[n - 1], h[n]), abs=1e-15)
    # the one-layer step at position 0 worked out from its parts above
    m = oracle.Model(_spec(n_layers=1))
    m.decode_step(toks[0])
    x0 = _embed(_spec(), toks[0])
    assert m.layer_cos()[0] == pytest.approx(oracle.cosine(x0, m.hidden()), abs=1e-15)
    assert -1.0 <= m.layer_cos()[0] <= 1.0


def test_skip_plan_threshold_and_cap():
    cos = [0.5, 0.99, 0.97, 0.98, 0.995, 0.99]
    np.testing.assert_array_equal(oracle.plan_layer_skip(cos, 0.98), [0, 1, 0, 1, 1, 1])
    np.testing.assert_array_equal(oracle.plan_layer_skip(cos, 0.98, max_skip=2), [0, 1, 0, 0, 1, 0])  # tie: lower layer
    np.testing.assert_array_equal(oracle.plan_layer_skip(cos, 0.999), [0] * 6)
    np.testing.assert_array_equal(oracle.plan_layer_skip(cos, -1.0, max_skip=1), [0, 0, 0, 0, 1, 0])


# ---- self-speculative decoding (resident layers as the draft)

def _greedy(spec, token, n, prefill=None):
    m = oracle.Model(spec)
    if prefill:
        m.kv_prefill(*prefill)
    out, t = [], token
    for _ in range(n):
        _, t, _ = m.decode_step(t)
        out.append(t)
    return out


@pytest.mark.parametrize("n_draft,k", [(3, 4), (1, 4), (0, 3), (2, 1)])
def test_speculative_stream_is_the_greedy_stream(n_draft, k):
    spec = _spec(n_layers=3, vocab=512, max_ctx=48)
    cycles = oracle.speculative_cycles(spec, n_draft, k, 7, 6, prefill=(5, 2))
    stream = [t for emitted, _ in cycles for t in emitted]
    assert stream == _greedy(spec, 7, len(stream), prefill=(5, 2))
    for emitted, j in cycles:
        assert 0 <= j <= k and len(emitted) == (j + 1 if j < k else k)
    if n_draft == spec.n_layers:           # the draft is the full model: everything is accepted
        assert all(j == k for _, j in cycles)
    if k == 1:
        assert all(len(e) == 1 for e, _ in cycles)


def test_speculative_zero_layer_draft_acceptance_is_agreement_with_the_head():
    # with n_draft = 0 the draft proposes argmax(head(norm(embedding(t)))): the
    # first proposal is accepted exactly when the full model's next token equals it
    spec = _spec(n_layers=2, vocab=256, max_ctx=32)
    cycles = oracle.speculative_cycles(spec, 0, 2, 11, 5)
    zero = oracle.Model(_spec(n_layers=0, vocab=256, max_ctx=32))
    greedy = _greedy(spec, 11, sum(len(e) for e, _ in cycles))
    pos, t = 0, 11
    for emitted, j in cycles:
        zero.set_pos(pos)
        _, d1, _ = zero.decode_step(t)
        assert (j >= 1) == (d1 == greedy[pos])
        pos += len(emitted)
        t = emitted[-1]
