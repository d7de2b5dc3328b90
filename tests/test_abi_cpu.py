"""CPU: the CUDA library builds, loads and exports every function include/nt.h
declares; argument validation that happens before any device work."""
import ctypes

import pytest

from quantized_decode_dequant_gb300 import nt


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()
    return nt.lib()


def test_library_exports_every_header_function(built):
    names = nt.header_functions()
    assert len(names) >= 19
    lib = ctypes.CDLL(nt.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(nt._SIGS), "binding and header disagree"


def test_validation_before_device_work(built):
    assert isinstance(nt.nt_last_error(), str)
    with pytest.raises(nt.NtError) as ei:
        nt.nt_qtensor_create("q4_k", 4, 100, 0, 1, 0.02)      # cols not a multiple of 256
    assert ei.value.status == nt.NT_E_INVAL
    with pytest.raises(nt.NtError) as ei:
        nt.nt_qtensor_create("f16", 4, 256, 0, 1, 0.02)
    assert ei.value.status == nt.NT_E_UNSUPPORTED
    for bad in (dict(n_kv_heads=3), dict(head_dim=96), dict(hidden=500), dict(vocab=0)):
        base = dict(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1536, vocab=4096,
                    max_ctx=64)
        base.update(bad)
        with pytest.raises(nt.NtError) as ei:
            nt.nt_model_create(nt.make_config(**base))
        assert ei.value.status in (nt.NT_E_INVAL, nt.NT_E_UNSUPPORTED)
    with pytest.raises(nt.NtError):
        nt.nt_gemv_q(0, 0, 0)
    with pytest.raises(nt.NtError):
        nt.nt_decode_step(0, 0)


def test_attention_workspace_and_validation(built):
    # chunk C = max(32, 16 ceil(max_ctx / 128)) up to 2560 positions, min(320, 16 ceil(max_ctx / 256)) beyond,
    # and ceil(max_ctx / C) items per kv head:
    # tickets (n_kv x 4 B, to 16), the position (16 B), statistics (8 B), partial outputs (4 hd B) per item and head
    for (nh, nkv, hd, mc) in [(64, 8, 128, 4224), (8, 8, 64, 12000), (8, 2, 64, 64), (32, 8, 128, 768)]:
        c = max(32, 16 * -(-mc // 128)) if mc <= 2560 else min(320, 16 * -(-mc // 256))
        items = -(-mc // c)
        want = -(-nkv * 4 // 16) * 16 + 16 + -(-nh * items * 8 // 16) * 16 + nh * items * hd * 4
        assert nt.nt_attention_workspace_bytes(nh, nkv, hd, mc) == want
    for args, status in [((8, 3, 64, 64), nt.NT_E_INVAL), ((8, 2, 96, 64), nt.NT_E_UNSUPPORTED),
                         ((96, 3, 64, 64), nt.NT_E_UNSUPPORTED), ((8, 2, 64, 0), nt.NT_E_INVAL)]:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_attention_workspace_bytes(*args)
        assert ei.value.status == status
    with pytest.raises(nt.NtError) as ei:   # NULL pointers: refused before any launch
        nt.nt_attention(8, 2, 64, 64, 10, 0, 0, 0, 0, 0, 1 << 20)
    assert ei.value.status == nt.NT_E_INVAL
