"""Oracle: FLOP and KV-memory accounting written from the pages' own definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Per-token FLOPs by operation class follow [S] 3.4 "Concrete FLOPs breakdown
(Table 1)": each linear layer costs 2 * in * out per token; the K,V
projections still run for every skipped layer (once per AcrossKV group); Q,O,
MLP and attention of skipped layers are gone; the vocabulary column counts the
embedding and LM-head projections (2 * 2 * d * V). Attention per token per
layer is 4 * n_q * d_h * ctx (QK^T and PV), ctx the attended context.

KV memory follows [S] 3.4 AcrossKV "Memory reduction":
M_AcrossKV = (l + (L - l)/g) * 2 * d_k * h_kv * S.
"""
from __future__ import annotations

from typing import Dict


def per_token_gflops(L: int, d: int, n_q: int, n_kv: int, d_h: int, ffn: int, vocab: int,
                     l: int, g: int = 1, attn_ctx: float = 0.0) -> Dict[str, float]:
    """GFLOPs per prefill token by operation class, Table 1 style."""
    if l > L or g < 1 or (L - l) % g:
        raise ValueError("bad (l, g)")
    kv_sets = l + (L - l) // g
    kv = kv_sets * 2 * d * (2 * n_kv * d_h)
    qo = l * 2 * (2 * d * n_q * d_h)
    mlp = l * 3 * (2 * d * ffn)
    attn = l * 4 * n_q * d_h * attn_ctx
    voc = 2 * 2 * d * vocab
    out = {"vocab": voc, "kv": kv, "qo": qo, "mlp": mlp, "attention": attn}
    out = {k: v / 1e9 for k, v in out.items()}
    out["total"] = sum(out.values())
    return out


def kv_cache_layers(L: int, l: int, g: int) -> int:
    return l + (L - l) // g


def kv_bytes(L: int, l: int, g: int, n_kv: int, d_h: int, tokens: int, elem_bytes: int = 2) -> int:
    """Bytes of KV cache for `tokens` tokens: layers * 2 (K and V) * d_k * h_kv * S."""
    return kv_cache_layers(L, l, g) * 2 * d_h * n_kv * tokens * elem_bytes


def kv_reduction(L: int, l: int, g: int) -> float:
    """Fraction of the baseline (L layers) KV memory removed by AcrossKV."""
    return 1.0 - kv_cache_layers(L, l, g) / L
