"""Oracle for SwiftKV prefill skipping -- TEST INFRASTRUCTURE.

A plain, slow, float64 NumPy statement of what the method computes, written
from the pages' definitions (see ``oracle/model.py`` for the sources). Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. It shares no code with the CUDA library; the only
module both sides use is ``synth`` (seeded input generation).

Pins (tests/test_oracle_*.py) tie every function to something other than
itself: library routines (torch's RMSNorm / scaled-dot-product attention /
bfloat16 cast), closed forms and invariants of RoPE and attention, brute
force on tiny inputs, the pages' Table 1 FLOPs and AcrossKV memory figures,
and the method's own invariants (l = L is the ordinary model; skipping
equals the full SwiftKV model; AcrossKV g = 1 is plain SwiftKV; causality;
decode from the cache equals the full forward of the longer sequence).
"""
from __future__ import annotations

import numpy as np

from . import bookkeeping, flops, model
from .model import Config, Layer, Weights

__all__ = ["bookkeeping", "flops", "model", "Config", "Layer", "Weights", "config_of",
           "synth_weights"]


def config_of(shape) -> Config:
    return Config(L=shape.L, d=shape.d, n_q=shape.n_q, n_kv=shape.n_kv, d_h=shape.d_h,
                  ffn=shape.ffn, vocab=shape.vocab, rope_theta=shape.rope_theta,
                  rms_eps=shape.rms_eps, qkv_bias=shape.qkv_bias)


def synth_weights(shape, seed: int = 0, gain_std: float = 0.0, cache_layers: bool = True,
                  overrides=None) -> Weights:
    """Oracle weights built from the shared seeded generator (float32 storage of
    bfloat16 values; the oracle widens to float64 as it computes).

    ``overrides`` maps (layer, name) -> array to replace single tensors, for
    tests that perturb one weight."""
    import synth

    overrides = dict(overrides or {})
    f32 = synth.bf16_bits_to_f32
    cache = {}

    def layer_fn(j: int) -> Layer:
        if j in cache:
            return cache[j]
        raw = synth.layer_weights(shape, j, seed=seed, gain_std=gain_std)
        get = lambda n, conv=True: overrides.get((j, n), f32(raw[n]) if conv else raw.get(n))
        lw = Layer(gamma_attn=overrides.get((j, "gamma_attn"), raw["gamma_attn"]),
                   wq=get("wq"), wk=get("wk"), wv=get("wv"), wo=get("wo"),
                   gamma_mlp=overrides.get((j, "gamma_mlp"), raw["gamma_mlp"]),
                   wg=get("wg"), wu=get("wu"), wd=get("wd"),
                   bq=overrides.get((j, "bq"), raw.get("bq")),
                   bk=overrides.get((j, "bk"), raw.get("bk")),
                   bv=overrides.get((j, "bv"), raw.get("bv")))
        if cache_layers:
            cache[j] = lw
        return lw

    def embed_fn(tokens: np.ndarray) -> np.ndarray:
        return f32(synth.embed_rows(shape, tokens, seed=seed))

    g = synth.global_weights(shape, seed=seed, gain_std=gain_std, kinds=("gamma_final", "lm_head"))
    return Weights(layer_fn, embed_fn, g["gamma_final"], f32(g["lm_head"]))
