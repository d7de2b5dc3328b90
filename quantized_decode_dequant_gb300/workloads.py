"""The workloads: architectures, per-role formats, contexts and seeds.

Llama shapes (hidden, heads, kv heads, head_dim, FFN, vocab) of the 8B and 70B
models the pages run; random-init weights stand in for the checkpoints.
Seeds: weights 0, activation vectors 1, KV prefill 2, prompt tokens 3.
"""
from __future__ import annotations

SEED_WEIGHTS, SEED_X, SEED_KV, SEED_PROMPT = 0, 1, 2, 3

TINY = dict(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1536, vocab=4096, max_ctx=64)
TINY_STEPS = 64

LLAMA_8B = dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=14336, vocab=128256)
LLAMA_8B_Q8_0 = dict(LLAMA_8B, max_ctx=512 + 256)
LLAMA_8B_CTX, LLAMA_8B_STEPS = 512, 256

LLAMA_70B = dict(n_layers=80, hidden=8192, n_heads=64, n_kv_heads=8, head_dim=128, ffn_dim=28672, vocab=128256)
# Q4_K_M-style mix: attn_v, ffn_down and output in Q6_K, everything else Q4_K
Q4_K_M = dict(t_embd="q4_k", t_q="q4_k", t_k="q4_k", t_v="q6_k", t_o="q4_k", t_gate="q4_k", t_up="q4_k",
              t_down="q6_k", t_out="q6_k")
LLAMA_70B_Q4_K_M = dict(LLAMA_70B, max_ctx=4096 + 128, **Q4_K_M)
LLAMA_70B_Q4_K_M_CTX, LLAMA_70B_Q4_K_M_STEPS = 4096, 128

ALL_Q6_K = {k: "q6_k" for k in Q4_K_M}
# Q5_K_M-style mix: attn_v, ffn_down and output in Q6_K, everything else Q5_K
Q5_K_M = dict(Q4_K_M, **{k: "q5_k" for k, v in Q4_K_M.items() if v == "q4_k"})
LLAMA_70B_Q6_K = dict(LLAMA_70B, max_ctx=1024 + 32, **ALL_Q6_K)
LLAMA_70B_Q6_K_CTX, LLAMA_70B_Q6_K_STEPS, LLAMA_70B_Q6_K_RESIDENT = 1024, 32, 26

# isolated dequant-GEMV sweep at 70B layer shapes (out x in)
GEMV_SHAPES = [(8192, 8192), (1024, 8192), (28672, 8192), (8192, 28672), (128256, 8192)]
GEMV_FORMATS = ["q4_0", "q8_0", "q4_k", "q6_k", "q5_k"]

BLOCK_ELEMS = {"q8_0": 32, "q4_0": 32, "q4_k": 256, "q6_k": 256, "q5_k": 256}
BLOCK_BYTES = {"q8_0": 34, "q4_0": 18, "q4_k": 144, "q6_k": 210, "q5_k": 176}


def weight_bytes(spec: dict) -> int:
    """Quantized weight bytes one decode step reads (layers + output; one embedding row is negligible)."""
    h, f, v = spec["hidden"], spec["ffn_dim"], spec["vocab"]
    qd, kd = spec["n_heads"] * spec["head_dim"], spec["n_kv_heads"] * spec["head_dim"]
    t = {k: spec.get(k, "q8_0") for k in ("t_q", "t_k", "t_v", "t_o", "t_gate", "t_up", "t_down", "t_out")}

    def b(fmt, rows, cols):
        return rows * cols // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]

    layer = (b(t["t_q"], qd, h) + b(t["t_k"], kd, h) + b(t["t_v"], kd, h) + b(t["t_o"], h, qd)
             + b(t["t_gate"], f, h) + b(t["t_up"], f, h) + b(t["t_down"], h, f))
    return spec["n_layers"] * layer + b(t["t_out"], v, h)


def kv_bytes(spec: dict, n_ctx: int) -> int:
    """f16 K and V bytes one decode step reads with n_ctx cached positions."""
    return spec["n_layers"] * 2 * spec["n_kv_heads"] * spec["head_dim"] * 2 * n_ctx
