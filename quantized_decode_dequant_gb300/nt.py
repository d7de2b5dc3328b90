"""ctypes binding of libnt.so (include/nt.h): argument marshalling only.

Every function here forwards to the C entry point of the same name; all work
runs in the CUDA library.  Device buffers are passed as integer addresses
(for example ``tensor.data_ptr()`` of a CUDA torch tensor) and streams as
``cudaStream_t`` integers (``torch.cuda.current_stream().cuda_stream``).
If the library is missing the first call raises ``NtLibraryMissing``: there
is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnt.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "nt.h")

NT_OK, NT_E_INVAL, NT_E_NOMEM, NT_E_CUDA, NT_E_TIMEOUT, NT_E_UNSUPPORTED, NT_E_STATE = range(7)
STATUS_NAMES = ["NT_OK", "NT_E_INVAL", "NT_E_NOMEM", "NT_E_CUDA", "NT_E_TIMEOUT", "NT_E_UNSUPPORTED", "NT_E_STATE"]
QTYPES = {"f32": 0, "f16": 1, "q8_0": 2, "q4_0": 3, "q4_k": 4, "q6_k": 5, "q5_k": 6}
ROLES = {"q": 0, "k": 1, "v": 2, "o": 3, "gate": 4, "up": 5, "down": 6, "embd": 16, "output": 17}
KC_GEMV, KC_ATTN, KC_OTHER = 0, 1, 2


class NtLibraryMissing(ImportError):
    pass


class NtError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{func}: {name}: {msg}")


class nt_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("vocab", C.c_int32), ("max_ctx", C.c_int32), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("init_std", C.c_float),
                ("t_embd", C.c_int), ("t_q", C.c_int), ("t_k", C.c_int), ("t_v", C.c_int), ("t_o", C.c_int),
                ("t_gate", C.c_int), ("t_up", C.c_int), ("t_down", C.c_int), ("t_out", C.c_int),
                ("seed", C.c_uint64)]


class nt_stats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("pos", C.c_int32), ("n_resident", C.c_int32),
                ("last_step_ms", C.c_double), ("h2d_bytes", C.c_double), ("h2d_ms", C.c_double),
                ("compute_ms", C.c_double), ("overlap", C.c_double), ("weight_bytes", C.c_int64),
                ("kv_bytes_per_pos", C.c_int64), ("verify_weight_bytes", C.c_double),
                ("h2d_layer_min_GBs", C.c_double), ("h2d_layer_max_GBs", C.c_double),
                ("h2d_layer_min_idx", C.c_int32)]


class nt_kernel_times(C.Structure):
    _fields_ = [("launches", C.c_int64 * 3), ("ms", C.c_double * 3), ("bytes", C.c_double * 3),
                ("step_ms", C.c_double), ("kernel_launches", C.c_int64)]


_lib = None
_vp, _i32, _i64, _u64, _f32p = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.POINTER(C.c_float)
_SIGS = {
    "nt_last_error": (C.c_char_p, []),
    "nt_model_create": (C.c_int, [C.POINTER(nt_config), C.POINTER(C.c_void_p)]),
    "nt_model_destroy": (None, [_vp]),
    "nt_kv_reset": (C.c_int, [_vp]),
    "nt_kv_prefill": (C.c_int, [_vp, _i32, _u64]),
    "nt_decode_step": (C.c_int, [_vp, _i32, C.POINTER(C.c_int32), _f32p, _f32p]),
    "nt_decode_run": (C.c_int, [_vp, _i32, _i32, _vp]),
    "nt_get_tokens": (C.c_int, [_vp, _i32, _i32, C.POINTER(C.c_int32)]),
    "nt_kv_export": (C.c_int, [_vp, _i32, _i32, _i32, _i32, _i32, C.POINTER(C.c_uint16)]),
    "nt_stream_layers": (C.c_int, [_vp, _i32, _i32]),
    "nt_get_stats": (C.c_int, [_vp, C.POINTER(nt_stats)]),
    "nt_profile_steps": (C.c_int, [_vp, _i32, _i32, C.POINTER(nt_kernel_times)]),
    "nt_profile_gemvs": (C.c_int, [_vp, _i32, C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(_i32)]),
    "nt_plan_residency": (C.c_int, [C.POINTER(nt_config), _i64, C.POINTER(_i32), C.POINTER(_i64), C.POINTER(_i64)]),
    "nt_auto_residency": (C.c_int, [_vp, _i64, C.POINTER(_i32)]),
    "nt_layer_similarity": (C.c_int, [_vp, _i32, C.POINTER(_i32), C.POINTER(C.c_double)]),
    "nt_set_layer_skip": (C.c_int, [_vp, C.POINTER(C.c_uint8)]),
    "nt_speculative_step": (C.c_int, [_vp, _i32, _i32, _i32, C.POINTER(_i32), C.POINTER(_i32), C.POINTER(_i32)]),
    "nt_plan_layer_skip": (C.c_int, [C.POINTER(C.c_double), _i32, C.c_double, _i32, C.POINTER(C.c_uint8),
                                     C.POINTER(_i32)]),
    "nt_model_tensor": (C.c_int, [_vp, _i32, _i32, C.POINTER(C.c_void_p)]),
    "nt_qtensor_create": (C.c_int, [C.c_int, _i64, _i64, _u64, C.c_uint32, C.c_float, C.POINTER(C.c_void_p)]),
    "nt_qtensor_destroy": (None, [_vp]),
    "nt_qtensor_info": (C.c_int, [_vp, C.POINTER(C.c_int), C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                  C.POINTER(C.c_size_t)]),
    "nt_qtensor_export": (C.c_int, [_vp, _i64, _i64, _vp, C.c_size_t]),
    "nt_dequant": (C.c_int, [_vp, _i64, _i64, _vp, _vp]),
    "nt_gemv_q": (C.c_int, [_vp, _vp, _vp, _vp]),
    "nt_gemv_q_batch": (C.c_int, [_vp, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), _i32, C.POINTER(_i32), _vp]),
    "nt_gemv_argmax_noalloc": (C.c_int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "nt_attention_workspace_bytes": (C.c_int, [_i32, _i32, _i32, _i32, C.POINTER(C.c_size_t)]),
    "nt_attention": (C.c_int, [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, C.c_size_t, _vp]),
}


def header_functions() -> list[str]:
    """Names of the functions include/nt.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(nt_[a-z0-9_]+)\s*\(", text,
                                 re.M)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise NtLibraryMissing(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                                   "(the CUDA library has no fallback)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def nt_last_error() -> str:
    return lib().nt_last_error().decode()


def _check(status: int, func: str):
    if status != NT_OK:
        raise NtError(status, func, nt_last_error())


def _stream(s) -> int | None:
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    return int(s)


# ----------------------------------------------------------------- configs --

def make_config(*, n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_ctx, rms_eps=1e-5,
                rope_theta=500000.0, init_std=0.02, seed=0, t_embd="q8_0", t_q="q8_0", t_k="q8_0", t_v="q8_0",
                t_o="q8_0", t_gate="q8_0", t_up="q8_0", t_down="q8_0", t_out="q8_0") -> nt_config:
    c = nt_config()
    for k, v in dict(n_layers=n_layers, hidden=hidden, n_heads=n_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                     ffn_dim=ffn_dim, vocab=vocab, max_ctx=max_ctx, rms_eps=rms_eps, rope_theta=rope_theta,
                     init_std=init_std, seed=seed).items():
        setattr(c, k, v)
    for k, v in dict(t_embd=t_embd, t_q=t_q, t_k=t_k, t_v=t_v, t_o=t_o, t_gate=t_gate, t_up=t_up, t_down=t_down,
                     t_out=t_out).items():
        setattr(c, k, QTYPES[v])
    return c


# ------------------------------------------------------------------- model --

_n_layers: dict[int, int] = {}   # layer count of each live model handle


def nt_model_create(cfg: nt_config) -> int:
    h = C.c_void_p()
    _check(lib().nt_model_create(C.byref(cfg), C.byref(h)), "nt_model_create")
    _n_layers[h.value] = cfg.n_layers
    return h.value


def nt_model_destroy(m: int) -> None:
    _n_layers.pop(m, None)
    lib().nt_model_destroy(m)


def stats_layers(m: int) -> int:
    """Layer count of a model created through this module."""
    return _n_layers[m]


def nt_kv_reset(m: int) -> None:
    _check(lib().nt_kv_reset(m), "nt_kv_reset")


def nt_kv_prefill(m: int, n_ctx: int, seed: int) -> None:
    _check(lib().nt_kv_prefill(m, n_ctx, seed), "nt_kv_prefill")


def nt_decode_step(m: int, token: int, logits: np.ndarray | None = None, want_margin: bool = False):
    """Returns next_token, or (next_token, margin) with want_margin; fills logits (float32[vocab]) if given."""
    nx = C.c_int32()
    mg = C.c_float()
    lp = None
    if logits is not None:
        assert logits.dtype == np.float32 and logits.flags.c_contiguous
        lp = logits.ctypes.data_as(_f32p)
    _check(lib().nt_decode_step(m, token, C.byref(nx), lp, C.byref(mg) if want_margin else None), "nt_decode_step")
    return (nx.value, mg.value) if want_margin else nx.value


def nt_decode_run(m: int, token: int, n_steps: int, stream=None) -> None:
    _check(lib().nt_decode_run(m, token, n_steps, _stream(stream)), "nt_decode_run")


def nt_get_tokens(m: int, t0: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _check(lib().nt_get_tokens(m, t0, n, out.ctypes.data_as(C.POINTER(C.c_int32))), "nt_get_tokens")
    return out


def nt_kv_export(m: int, layer: int, kv: int, kv_head: int, t0: int, n: int, head_dim: int) -> np.ndarray:
    out = np.empty((n, head_dim), np.uint16)
    _check(lib().nt_kv_export(m, layer, kv, kv_head, t0, n, out.ctypes.data_as(C.POINTER(C.c_uint16))),
           "nt_kv_export")
    return out


def nt_stream_layers(m: int, n_resident: int, n_staging: int = 2) -> None:
    _check(lib().nt_stream_layers(m, n_resident, n_staging), "nt_stream_layers")


def nt_get_stats(m: int) -> nt_stats:
    s = nt_stats()
    _check(lib().nt_get_stats(m, C.byref(s)), "nt_get_stats")
    return s


def nt_profile_steps(m: int, token: int, n_steps: int) -> nt_kernel_times:
    t = nt_kernel_times()
    _check(lib().nt_profile_steps(m, token, n_steps, C.byref(t)), "nt_profile_steps")
    return t


def nt_profile_gemvs(m: int, n_reps: int) -> tuple[float, float, int]:
    """(ms per GEMV launch, algorithmic bytes per launch, GEMV launches per step)."""
    ms, by, n = C.c_double(), C.c_double(), C.c_int32()
    _check(lib().nt_profile_gemvs(m, n_reps, C.byref(ms), C.byref(by), C.byref(n)), "nt_profile_gemvs")
    return ms.value, by.value, n.value


def nt_plan_residency(cfg, budget_bytes: int) -> tuple[int, int, int]:
    """(layers resident, device bytes of that placement, bytes of one layer) for a budget."""
    n, dev, lay = C.c_int32(), C.c_int64(), C.c_int64()
    _check(lib().nt_plan_residency(C.byref(cfg), budget_bytes, C.byref(n), C.byref(dev), C.byref(lay)),
           "nt_plan_residency")
    return n.value, dev.value, lay.value


def nt_auto_residency(m: int, margin_bytes: int = 1 << 30) -> int:
    n = C.c_int32()
    _check(lib().nt_auto_residency(m, margin_bytes, C.byref(n)), "nt_auto_residency")
    return n.value


def nt_layer_similarity(m: int, token: int) -> tuple[int, np.ndarray]:
    """One decode step that also returns the per-layer cosine between the residual entering and leaving it."""
    n = stats_layers(m)
    cos = np.empty(max(n, 1), np.float64)
    nx = C.c_int32()
    _check(lib().nt_layer_similarity(m, token, C.byref(nx), cos.ctypes.data_as(C.POINTER(C.c_double))),
           "nt_layer_similarity")
    return nx.value, cos[:n]


def nt_set_layer_skip(m: int, mask) -> None:
    """Skips the layers whose mask entry is nonzero (None: none)."""
    if mask is None:
        _check(lib().nt_set_layer_skip(m, None), "nt_set_layer_skip")
        return
    a = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
    assert a.size == stats_layers(m)
    _check(lib().nt_set_layer_skip(m, a.ctypes.data_as(C.POINTER(C.c_uint8))), "nt_set_layer_skip")


def nt_speculative_step(m: int, token: int, n_draft: int, k: int) -> tuple[list[int], int]:
    """One self-speculative cycle: (emitted tokens, accepted draft tokens)."""
    out = (_i32 * 8)()
    n, j = _i32(), _i32()
    _check(lib().nt_speculative_step(m, token, n_draft, k, out, C.byref(n), C.byref(j)), "nt_speculative_step")
    return [out[i] for i in range(n.value)], j.value


def nt_plan_layer_skip(cos, threshold: float, max_skip: int = 0) -> np.ndarray:
    """uint8 mask of the layers to skip for calibrated similarities (host arithmetic)."""
    c = np.ascontiguousarray(np.asarray(cos, np.float64))
    mask = np.zeros(max(c.size, 1), np.uint8)
    n = C.c_int32()
    _check(lib().nt_plan_layer_skip(c.ctypes.data_as(C.POINTER(C.c_double)), c.size, threshold, max_skip,
                                    mask.ctypes.data_as(C.POINTER(C.c_uint8)), C.byref(n)), "nt_plan_layer_skip")
    assert int(mask[:c.size].sum()) == n.value
    return mask[:c.size]


def nt_model_tensor(m: int, layer: int, role) -> int:
    out = C.c_void_p()
    r = ROLES[role] if isinstance(role, str) else int(role)
    _check(lib().nt_model_tensor(m, layer, r, C.byref(out)), "nt_model_tensor")
    return out.value


# -------------------------------------------------------- quantized tensors --

def nt_qtensor_create(qtype: str, rows: int, cols: int, seed: int, uid: int, std: float) -> int:
    h = C.c_void_p()
    _check(lib().nt_qtensor_create(QTYPES[qtype], rows, cols, seed, uid, std, C.byref(h)), "nt_qtensor_create")
    return h.value


def nt_qtensor_destroy(t: int) -> None:
    lib().nt_qtensor_destroy(t)


def nt_qtensor_info(t: int):
    ty, r, c, b = C.c_int(), C.c_int64(), C.c_int64(), C.c_size_t()
    _check(lib().nt_qtensor_info(t, C.byref(ty), C.byref(r), C.byref(c), C.byref(b)), "nt_qtensor_info")
    name = {v: k for k, v in QTYPES.items()}[ty.value]
    return name, r.value, c.value, b.value


def nt_qtensor_export(t: int, row0: int, nrows: int, block_elems: int, block_bytes: int, cols: int) -> np.ndarray:
    out = np.zeros((nrows, cols // block_elems * block_bytes), np.uint8)
    _check(lib().nt_qtensor_export(t, row0, nrows, out.ctypes.data, out.nbytes), "nt_qtensor_export")
    return out


def nt_dequant(t: int, row0: int, nrows: int, dev_out: int, stream=None) -> None:
    _check(lib().nt_dequant(t, row0, nrows, dev_out, _stream(stream)), "nt_dequant")


def nt_gemv_q(t: int, dev_x: int, dev_y: int, stream=None) -> None:
    _check(lib().nt_gemv_q(t, dev_x, dev_y, _stream(stream)), "nt_gemv_q")


def nt_gemv_q_batch(t: int, dev_xs, dev_ys, stream=None) -> int:
    """y_i = W x_i for the k device vectors dev_xs[i] -> dev_ys[i]; returns the launches used."""
    k = len(dev_xs)
    xs = (C.c_void_p * k)(*dev_xs)
    ys = (C.c_void_p * k)(*dev_ys)
    n = C.c_int32()
    _check(lib().nt_gemv_q_batch(t, xs, ys, k, C.byref(n), _stream(stream)), "nt_gemv_q_batch")
    return int(n.value)


def nt_attention_workspace_bytes(n_heads: int, n_kv_heads: int, head_dim: int, max_ctx: int) -> int:
    n = C.c_size_t()
    _check(lib().nt_attention_workspace_bytes(n_heads, n_kv_heads, head_dim, max_ctx, C.byref(n)),
           "nt_attention_workspace_bytes")
    return int(n.value)


def nt_attention(n_heads: int, n_kv_heads: int, head_dim: int, max_ctx: int, n_ctx: int, dev_q: int, dev_k: int,
                 dev_v: int, dev_out: int, dev_workspace: int, workspace_bytes: int, stream=None) -> None:
    """GQA attention of fp32 q over positions [0, n_ctx) of an f16 [n_kv][max_ctx][hd] K/V cache."""
    _check(lib().nt_attention(n_heads, n_kv_heads, head_dim, max_ctx, n_ctx, dev_q, dev_k, dev_v, dev_out,
                              dev_workspace, workspace_bytes, _stream(stream)), "nt_attention")


def nt_gemv_argmax_noalloc(t: int, dev_x: int, dev_y: int, dev_index: int, dev_margin: int, stream=None) -> None:
    """y = W x plus greedy index and top-2 margin on the device; allocates no device memory."""
    _check(lib().nt_gemv_argmax_noalloc(t, dev_x, dev_y, dev_index, dev_margin, _stream(stream)),
           "nt_gemv_argmax_noalloc")
