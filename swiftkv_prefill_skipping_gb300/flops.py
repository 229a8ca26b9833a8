"""Work accounting for the bench: FLOPs of the SwiftKV prefill path, the
dense-equivalent FLOPs of the ordinary model on the same prompts, and the
algorithmic bytes/FLOPs of each kernel class (for roofline fractions).

Dense-equivalent follows the pages' "normalized to the baseline model's FLOPs"
convention ("SwiftKV" summary, section 5, combined-throughput figures): all L
layers for every prompt token (linear layers + exact causal attention) plus
the LM head of the last token of each prompt.
"""
from __future__ import annotations

from typing import Dict, Sequence


def _linear_per_token(d, n_q, n_kv, d_h, ffn):
    qkv = 2 * d * (n_q + 2 * n_kv) * d_h
    q = 2 * d * n_q * d_h
    kv = 2 * d * 2 * n_kv * d_h
    o = 2 * n_q * d_h * d
    mlp = 3 * 2 * d * ffn
    return qkv, q, kv, o, mlp


def _attn_pairs(lens: Sequence[int], ctx: Sequence[int] = None) -> int:
    """Sum over chunks of the causal (query, key) pairs: n(n+1)/2, plus n * ctx for a
    chunk that follows ctx cached tokens."""
    ctx = ctx if ctx is not None else [0] * len(lens)
    return sum(int(n) * (int(n) + 1) // 2 + int(n) * int(c) for n, c in zip(lens, ctx))


def prefill_flops(shape, lens: Sequence[int], l: int, g: int = 1, ctx: Sequence[int] = None) -> Dict[str, float]:
    """FLOPs of one SwiftKV prefill of prompts `lens` (executed) and of the ordinary
    model (dense-equivalent), by component. With ctx, chunk s follows ctx[s] cached
    tokens (serving forward)."""
    L, d, n_q, n_kv, d_h, F, V = shape.L, shape.d, shape.n_q, shape.n_kv, shape.d_h, shape.ffn, shape.vocab
    T, P = int(sum(lens)), len(lens)
    ctx = ctx if ctx is not None else [0] * P
    qkv, q, kv, o, mlp = _linear_per_token(d, n_q, n_kv, d_h, F)
    pairs = _attn_pairs(lens, ctx)
    attn_layer = 4 * n_q * d_h * pairs           # QK^T and PV over causal pairs
    G = (L - l) // g
    full_gemm = l * T * (qkv + o + mlp)
    wide_kv = T * G * kv
    # tail: last token of each prompt through layers l+1..L (Q, attention, O, MLP)
    tail_gemm = (L - l) * P * (q + o + mlp)
    tail_attn = (L - l) * 4 * n_q * d_h * sum(int(n) + int(c) for n, c in zip(lens, ctx))
    lm = P * 2 * d * V
    executed = full_gemm + wide_kv + l * attn_layer + tail_gemm + tail_attn + lm
    dense = L * T * (qkv + o + mlp) + L * attn_layer + lm
    return {
        "layers_gemm": float(full_gemm), "layers_attention": float(l * attn_layer),
        "wide_kv_gemm": float(wide_kv), "tail": float(tail_gemm + tail_attn), "lm_head": float(lm),
        "gemm": float(full_gemm + wide_kv + tail_gemm + lm),
        "executed": float(executed), "dense_equiv": float(dense),
    }


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def rmsnorm_bytes(rows: int, d: int) -> int:
    """fp32 row read + bf16 row write."""
    return rows * d * (4 + 2)
