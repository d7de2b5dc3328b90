"""Tier placement (nt_plan_residency): host arithmetic, no GPU needed.

The layer size is checked against the device stream layout written out here
independently (per-format stream sizes, each padded to 256 bytes); the placement
against its definition: the most layers that fit next to the fixed allocations
and, when any layer streams, two staging buffers of one layer.
"""
import pytest

from quantized_decode_dequant_gb300 import nt, workloads as W


def pad(n):
    return (n + 255) // 256 * 256


def stream_bytes(fmt, rows, cols):
    e = rows * cols
    if fmt == "q8_0":
        parts = [e, e // 32 * 2]
    elif fmt == "q4_0":
        parts = [e // 2, e // 32 * 2]
    elif fmt == "q4_k":
        parts = [e // 2, e // 256 * 16]
    elif fmt == "q5_k":   # low nibbles, fifth-bit words, 16 B per 256
        parts = [e // 2, e // 8, e // 256 * 16]
    else:  # q6_k: low nibbles, high-bit words, int8 scale per 16, f16 d per 256
        parts = [e // 2, e // 4, e // 16, e // 256 * 2]
    return sum(pad(p) for p in parts)


def layer_bytes(spec):
    h, f = spec["hidden"], spec["ffn_dim"]
    qd, kd = spec["n_heads"] * spec["head_dim"], spec["n_kv_heads"] * spec["head_dim"]
    t = {k: spec.get(k, "q8_0") for k in ("t_q", "t_k", "t_v", "t_o", "t_gate", "t_up", "t_down")}
    return (stream_bytes(t["t_q"], qd, h) + stream_bytes(t["t_k"], kd, h) + stream_bytes(t["t_v"], kd, h)
            + stream_bytes(t["t_o"], h, qd) + stream_bytes(t["t_gate"], f, h) + stream_bytes(t["t_up"], f, h)
            + stream_bytes(t["t_down"], h, f))


@pytest.fixture(scope="module")
def lib():
    try:
        nt.lib()
    except nt.NtLibraryMissing:
        import __graft_entry__
        __graft_entry__.build()
    return nt


@pytest.mark.parametrize("name", ["LLAMA_8B_Q8_0", "LLAMA_70B_Q4_K_M", "LLAMA_70B_Q6_K", "LLAMA_70B_Q5_K_M"])
def test_layer_bytes_match_the_stream_layout(lib, name):
    spec = getattr(W, name) if name != "LLAMA_70B_Q5_K_M" else dict(W.LLAMA_70B, max_ctx=4224, **W.Q5_K_M)
    n, dev, lay = lib.nt_plan_residency(lib.make_config(**spec), 1 << 50)
    assert lay == layer_bytes(spec)
    assert n == spec["n_layers"]
    assert dev > spec["n_layers"] * lay


def test_placement_is_the_most_layers_that_fit(lib):
    spec = W.LLAMA_70B_Q6_K
    cfg = lib.make_config(**spec)
    L = spec["n_layers"]
    _, all_dev, lay = lib.nt_plan_residency(cfg, 1 << 50)
    fixed = all_dev - L * lay
    assert fixed > 0
    for n_want in (0, 1, 26, L - 3):   # with L - 2 or more the budget holds every layer without staging
        budget = fixed + (n_want + 2) * lay         # exactly n_want layers plus two staging buffers
        n, dev, _ = lib.nt_plan_residency(cfg, budget)
        assert n == n_want and dev == budget
        if n_want > 0:
            n2, _, _ = lib.nt_plan_residency(cfg, budget - 1)
            assert n2 == n_want - 1
        else:   # one byte short of the staging buffers alone
            with pytest.raises(lib.NtError) as ei:
                lib.nt_plan_residency(cfg, budget - 1)
            assert ei.value.status == lib.NT_E_NOMEM
    # all layers resident needs no staging buffers
    n, dev, _ = lib.nt_plan_residency(cfg, fixed + L * lay)
    assert n == L and dev == fixed + L * lay
    # monotone in the budget
    prev = -1
    for b in range(fixed + 2 * lay, fixed + (L + 2) * lay, 7 * lay // 3):
        n, _, _ = lib.nt_plan_residency(cfg, b)
        assert n >= prev
        prev = n


def test_the_q4_k_m_mix_fits_more_layers_than_q6_k(lib):
    budget = 40 << 30
    n6, _, _ = lib.nt_plan_residency(lib.make_config(**W.LLAMA_70B_Q6_K), budget)
    n4, _, _ = lib.nt_plan_residency(lib.make_config(**dict(W.LLAMA_70B_Q6_K, **W.Q4_K_M)), budget)
    assert n4 > n6 > 0


def test_budget_errors(lib):
    cfg = lib.make_config(**W.LLAMA_70B_Q6_K)
    with pytest.raises(lib.NtError) as ei:
        lib.nt_plan_residency(cfg, 1 << 20)
    assert ei.value.status == lib.NT_E_NOMEM
    with pytest.raises(lib.NtError) as ei:
        lib.nt_plan_residency(cfg, -1)
    assert ei.value.status == lib.NT_E_INVAL
    with pytest.raises(lib.NtError) as ei:
        lib.nt_plan_residency(lib.make_config(**dict(W.TINY, n_kv_heads=3)), 1 << 40)
    assert ei.value.status == lib.NT_E_INVAL
