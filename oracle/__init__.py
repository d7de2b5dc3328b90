"""ctypes wrapper of the C oracle (oracle.c) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and it
never loads the CUDA library.  ``build()`` compiles ``liboracle.so`` with plain
gcc (``-ffp-contract=off`` so no multiply-add is fused behind the formulas'
back).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

QTYPES = {"f32": 0, "f16": 1, "q8_0": 2, "q4_0": 3, "q4_k": 4, "q6_k": 5, "q5_k": 6}
BLOCK_ELEMS = {"f32": 1, "f16": 1, "q8_0": 32, "q4_0": 32, "q4_k": 256, "q6_k": 256, "q5_k": 256}
BLOCK_BYTES = {"f32": 4, "f16": 2, "q8_0": 34, "q4_0": 18, "q4_k": 144, "q6_k": 210, "q5_k": 176}

UID_EMBD = 0x100000
UID_OUTPUT = 0x100001
UID_TOKENS = 0x300000
ROLES = ("q", "k", "v", "o", "gate", "up", "down")


def uid_layer(layer: int, role: str) -> int:
    return layer * 16 + ROLES.index(role)


def uid_kv(layer: int, kv: int) -> int:
    return 0x200000 + 2 * layer + kv


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src),
                                                   os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-o", tmp, src, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB_PATH)
        u8p, f32p, f64p, u16p = (C.POINTER(C.c_uint8), C.POINTER(C.c_float), C.POINTER(C.c_double),
                                 C.POINTER(C.c_uint16))
        L.orc_mix64.restype = C.c_uint64
        L.orc_mix64.argtypes = [C.c_uint64]
        L.orc_normal.restype = C.c_float
        L.orc_normal.argtypes = [C.c_uint64, C.c_uint32, C.c_uint64]
        L.orc_gen_normal.argtypes = [C.c_uint64, C.c_uint32, C.c_uint64, C.c_int64, C.c_float, f32p]
        L.orc_token.restype = C.c_int32
        L.orc_token.argtypes = [C.c_uint64, C.c_uint32, C.c_uint64, C.c_int32]
        L.orc_f16_from_double.restype = C.c_uint16
        L.orc_f16_from_double.argtypes = [C.c_double]
        L.orc_f16_to_double.restype = C.c_double
        L.orc_f16_to_double.argtypes = [C.c_uint16]
        L.orc_quantize_row.argtypes = [C.c_int, f32p, C.c_int64, u8p]
        L.orc_dequant_row.argtypes = [C.c_int, u8p, C.c_int64, f32p]
        L.orc_qtensor_rows.argtypes = [C.c_int, C.c_int64, C.c_int64, C.c_uint64, C.c_uint32, C.c_float,
                                       C.c_int64, C.c_int64, u8p, C.c_int]
        L.orc_gemv.argtypes = [C.c_int, u8p, C.c_int64, C.c_int64, f32p, f64p, C.c_int]
        L.orc_gemv_d.argtypes = [C.c_int, u8p, C.c_int64, C.c_int64, f64p, f64p, C.c_int]
        L.orc_rmsnorm.argtypes = [f64p, C.c_int64, C.c_double, f64p]
        L.orc_rope.argtypes = [f64p, C.c_int, C.c_int, C.c_int64, C.c_double]
        L.orc_softmax.argtypes = [f64p, C.c_int64, f64p]
        L.orc_silu.restype = C.c_double
        L.orc_silu.argtypes = [C.c_double]
        L.orc_attend.argtypes = [f64p, u16p, u16p, C.c_int64, C.c_int, f64p]
        L.orc_argmax.restype = C.c_int64
        L.orc_argmax.argtypes = [f64p, C.c_int64, f64p]
        L.orc_model_create.restype = C.c_void_p
        L.orc_model_create.argtypes = [C.POINTER(OrcConfig)]
        L.orc_model_destroy.argtypes = [C.c_void_p]
        L.orc_kv_reset.argtypes = [C.c_void_p]
        L.orc_kv_prefill.argtypes = [C.c_void_p, C.c_int32, C.c_uint64]
        L.orc_pos.restype = C.c_int32
        L.orc_pos.argtypes = [C.c_void_p]
        L.orc_set_threads.argtypes = [C.c_void_p, C.c_int32]
        L.orc_decode_step.argtypes = [C.c_void_p, C.c_int32, f64p, C.POINTER(C.c_int32), f64p]
        L.orc_kv_get.restype = C.c_uint16
        L.orc_kv_get.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.orc_set_layer_skip.argtypes = [C.c_void_p, u8p]
        L.orc_set_pos.argtypes = [C.c_void_p, C.c_int32]
        L.orc_layer_cos.argtypes = [C.c_void_p, f64p]
        L.orc_hidden.argtypes = [C.c_void_p, f64p]
        L.orc_cosine.restype = C.c_double
        L.orc_cosine.argtypes = [f64p, f64p, C.c_int64]
        _lib = L
    return _lib


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(C.POINTER(ct))


# ---------------------------------------------------------------- generator --

def mix64(z: int) -> int:
    return int(lib().orc_mix64(z & (2**64 - 1)))


def normal(seed: int, uid: int, i: int) -> float:
    return float(lib().orc_normal(seed, uid, i))


def gen_normal(seed: int, uid: int, i0: int, n: int, std: float) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().orc_gen_normal(seed, uid, i0, n, std, _p(out, C.c_float))
    return out


def token(seed: int, uid: int, i: int, vocab: int) -> int:
    return int(lib().orc_token(seed, uid, i, vocab))


def tokens(seed: int, n: int, vocab: int, uid: int = UID_TOKENS) -> list[int]:
    return [token(seed, uid, i, vocab) for i in range(n)]


# --------------------------------------------------------------------- f16 --

def f16_from_double(x: float) -> int:
    return int(lib().orc_f16_from_double(x))


def f16_to_double(h: int) -> float:
    return float(lib().orc_f16_to_double(h))


# ----------------------------------------------------------------- formats --

def row_bytes(qt: str, cols: int) -> int:
    return cols // BLOCK_ELEMS[qt] * BLOCK_BYTES[qt]


def quantize_row(qt: str, w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, np.float32)
    out = np.zeros(row_bytes(qt, w.size), np.uint8)
    rc = lib().orc_quantize_row(QTYPES[qt], _p(w, C.c_float), w.size, _p(out, C.c_uint8))
    if rc:
        raise ValueError("orc_quantize_row failed")
    return out


def dequant_row(qt: str, blocks: np.ndarray, n: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    out = np.empty(n, np.float32)
    rc = lib().orc_dequant_row(QTYPES[qt], _p(blocks, C.c_uint8), n, _p(out, C.c_float))
    if rc:
        raise ValueError("orc_dequant_row failed")
    return out


def qtensor_rows(qt: str, rows: int, cols: int, seed: int, uid: int, std: float, row0: int = 0,
                 nrows: int | None = None, nthreads: int = 1) -> np.ndarray:
    """Canonical block bytes of rows [row0, row0+nrows), shape (nrows, row_bytes)."""
    if nrows is None:
        nrows = rows - row0
    out = np.zeros((nrows, row_bytes(qt, cols)), np.uint8)
    rc = lib().orc_qtensor_rows(QTYPES[qt], rows, cols, seed, uid, std, row0, nrows,
                                _p(out, C.c_uint8), nthreads)
    if rc:
        raise ValueError("orc_qtensor_rows failed")
    return out


def dequant_rows(qt: str, blocks: np.ndarray, cols: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, np.uint8).reshape(-1, row_bytes(qt, cols))
    return np.stack([dequant_row(qt, blocks[r], cols) for r in range(blocks.shape[0])])


def gemv(qt: str, blocks: np.ndarray, rows: int, cols: int, x: np.ndarray, nthreads: int = 1) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    y = np.empty(rows, np.float64)
    if x.dtype == np.float64:
        x = np.ascontiguousarray(x)
        rc = lib().orc_gemv_d(QTYPES[qt], _p(blocks, C.c_uint8), rows, cols, _p(x, C.c_double),
                              _p(y, C.c_double), nthreads)
    else:
        x = np.ascontiguousarray(x, np.float32)
        rc = lib().orc_gemv(QTYPES[qt], _p(blocks, C.c_uint8), rows, cols, _p(x, C.c_float),
                            _p(y, C.c_double), nthreads)
    if rc:
        raise ValueError("orc_gemv failed")
    return y


# --------------------------------------------------------------- small ops --

def rmsnorm(x: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x, C.c_double), x.size, eps, _p(out, C.c_double))
    return out


def rope(v: np.ndarray, n_heads: int, head_dim: int, pos: int, theta: float = 500000.0) -> np.ndarray:
    v = np.array(v, np.float64, copy=True)
    lib().orc_rope(_p(v, C.c_double), n_heads, head_dim, pos, theta)
    return v


def softmax(s: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(s, np.float64)
    p = np.empty_like(s)
    lib().orc_softmax(_p(s, C.c_double), s.size, _p(p, C.c_double))
    return p


def silu(z: float) -> float:
    return float(lib().orc_silu(z))


def attend(q: np.ndarray, k_f16: np.ndarray, v_f16: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k_f16, np.uint16)
    v = np.ascontiguousarray(v_f16, np.uint16)
    n_ctx, hd = k.shape
    out = np.empty(hd, np.float64)
    lib().orc_attend(_p(q, C.c_double), _p(k, C.c_uint16), _p(v, C.c_uint16), n_ctx, hd, _p(out, C.c_double))
    return out


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    """Cosine similarity of two vectors in fp64 (0 when either is zero)."""
    a = np.ascontiguousarray(a, np.float64)
    b = np.ascontiguousarray(b, np.float64)
    return float(lib().orc_cosine(_p(a, C.c_double), _p(b, C.c_double), a.size))


def plan_layer_skip(cos, threshold: float, max_skip: int = 0) -> np.ndarray:
    """Which layers to skip from their calibrated similarities ([hotdry]
    "性能数据与瓶颈分析": layers whose similarity is at or above the threshold,
    0.98 there, are skipped).  Reading: every layer with cos >= threshold; when
    max_skip > 0 and more qualify, the max_skip most similar ones (ties: lower
    layer first).  Returns a uint8 mask."""
    cand = [(-float(c), l) for l, c in enumerate(cos) if float(c) >= threshold]
    cand.sort()
    if max_skip > 0:
        cand = cand[:max_skip]
    mask = np.zeros(len(cos), np.uint8)
    for _, l in cand:
        mask[l] = 1
    return mask


def argmax(x: np.ndarray) -> tuple[int, float]:
    x = np.ascontiguousarray(x, np.float64)
    m = C.c_double()
    i = lib().orc_argmax(_p(x, C.c_double), x.size, C.byref(m))
    return int(i), float(m.value)


# ------------------------------------------------------------------- model --

class OrcConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("vocab", C.c_int32), ("max_ctx", C.c_int32), ("rms_eps", C.c_double),
                ("rope_theta", C.c_double), ("init_std", C.c_float),
                ("t_embd", C.c_int32), ("t_q", C.c_int32), ("t_k", C.c_int32), ("t_v", C.c_int32),
                ("t_o", C.c_int32), ("t_gate", C.c_int32), ("t_up", C.c_int32), ("t_down", C.c_int32),
                ("t_out", C.c_int32), ("seed", C.c_uint64), ("lazy", C.c_int32), ("nthreads", C.c_int32)]


@dataclass
class ModelSpec:
    """Architecture + per-role formats; mirrors the workload definitions."""
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    max_ctx: int
    rms_eps: float = 1e-5
    rope_theta: float = 500000.0
    init_std: float = 0.02
    t_embd: str = "q8_0"
    t_q: str = "q8_0"
    t_k: str = "q8_0"
    t_v: str = "q8_0"
    t_o: str = "q8_0"
    t_gate: str = "q8_0"
    t_up: str = "q8_0"
    t_down: str = "q8_0"
    t_out: str = "q8_0"
    seed: int = 0


class Model:
    def __init__(self, spec: ModelSpec, lazy: bool = False, nthreads: int = 1):
        c = OrcConfig()
        for f in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab", "max_ctx",
                  "rms_eps", "rope_theta", "init_std", "seed"):
            setattr(c, f, getattr(spec, f))
        for f in ("t_embd", "t_q", "t_k", "t_v", "t_o", "t_gate", "t_up", "t_down", "t_out"):
            setattr(c, f, QTYPES[getattr(spec, f)])
        c.lazy = 1 if lazy else 0
        c.nthreads = nthreads
        self.spec = spec
        self._h = lib().orc_model_create(C.byref(c))
        if not self._h:
            raise MemoryError("orc_model_create failed")

    def close(self):
        if self._h:
            lib().orc_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def pos(self) -> int:
        return int(lib().orc_pos(self._h))

    def set_threads(self, n: int):
        lib().orc_set_threads(self._h, n)

    def kv_reset(self):
        lib().orc_kv_reset(self._h)

    def kv_prefill(self, n_ctx: int, seed: int):
        if lib().orc_kv_prefill(self._h, n_ctx, seed):
            raise ValueError("orc_kv_prefill failed")

    def kv_get(self, layer: int, kv: int, kv_head: int, t: int, d: int) -> int:
        return int(lib().orc_kv_get(self._h, layer, kv, kv_head, t, d))

    def decode_step(self, token: int):
        """Returns (logits float64[vocab], next_token, top2_margin)."""
        lg = np.empty(self.spec.vocab, np.float64)
        nx = C.c_int32()
        mg = C.c_double()
        rc = lib().orc_decode_step(self._h, token, _p(lg, C.c_double), C.byref(nx), C.byref(mg))
        if rc:
            raise RuntimeError(f"orc_decode_step failed ({rc})")
        return lg, int(nx.value), float(mg.value)

    def set_layer_skip(self, mask):
        """Skips the layers whose mask entry is nonzero (None: none)."""
        if mask is None:
            lib().orc_set_layer_skip(self._h, None)
            return
        m = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
        assert m.size == self.spec.n_layers
        if lib().orc_set_layer_skip(self._h, _p(m, C.c_uint8)):
            raise MemoryError("orc_set_layer_skip")

    def layer_cos(self) -> np.ndarray:
        """Per layer, last step: cosine between the residual stream entering and leaving it."""
        out = np.empty(self.spec.n_layers, np.float64)
        lib().orc_layer_cos(self._h, _p(out, C.c_double))
        return out

    def hidden(self) -> np.ndarray:
        """Last step: the residual stream after the last layer."""
        out = np.empty(self.spec.hidden, np.float64)
        lib().orc_hidden(self._h, _p(out, C.c_double))
        return out

    def set_pos(self, pos: int):
        """Moves the position back (or forward) without touching the cache."""
        if lib().orc_set_pos(self._h, pos):
            raise ValueError(pos)


def speculative_cycles(spec: ModelSpec, n_draft: int, k: int, token: int, n_cycles: int,
                       prefill: tuple[int, int] | None = None, nthreads: int = 1):
    """Self-speculative decoding ([hada] "Hauptfunktionen": the
    VRAM-resident layers serve as the draft model, no extra model), from its
    definition.  Per cycle at position p with input token t:
      draft    d_1..d_k = greedy continuation of the model restricted to layers
               [0, n_draft) and the output head, from t;
      verify   y_i = the full model's greedy token at position p + i after
               t, d_1..d_i (i < k);
      accept   j = the length of the longest prefix with y_i == d_{i+1};
               emitted: d_1..d_j, then y_j when j < k.
    Returns [(emitted tokens, j), ...].  The emitted stream is the full model's
    greedy stream; the draft only decides how many tokens a cycle yields."""
    full = Model(spec, nthreads=nthreads)
    draft = Model(spec, nthreads=nthreads)
    draft.set_layer_skip([1 if l >= n_draft else 0 for l in range(spec.n_layers)])
    try:
        if prefill:
            full.kv_prefill(*prefill)
            draft.kv_prefill(*prefill)
        out = []
        t = token
        for _ in range(n_cycles):
            p = full.pos
            d, tt = [], t
            for _ in range(k):              # the draft's own greedy continuation
                _, tt, _ = draft.decode_step(tt)
                d.append(tt)
            draft.set_pos(p)
            y, tt = [], t
            for i in range(k):              # the full model on t, d_1..d_{k-1}
                _, yi, _ = full.decode_step(tt)
                y.append(yi)
                if yi != d[i]:
                    break
                tt = d[i]
            j = len(y) if y[-1] == d[len(y) - 1] else len(y) - 1
            emitted = d[:j] + ([y[j]] if j < k else [])
            full.set_pos(p)
            for e in [t] + emitted[:-1]:    # both models advance over the emitted prefix
                full.decode_step(e)
                draft.decode_step(e)
            out.append((emitted, j))
            t = emitted[-1]
        return out
    finally:
        full.close()
        draft.close()
