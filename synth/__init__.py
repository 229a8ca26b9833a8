"""Seeded synthetic inputs shared by the GPU path (tests, bench) and the oracle.

Holds no arithmetic of the model. Everything here is a deterministic function
of (seed, stream, index): weights ~ N(0, 0.02) rounded to bfloat16, RMSNorm
gains (1.0, or 1 + N(0, s) for tests that must see them), QKV biases,
uniform prompt lengths and token ids, and a page permutation for the block
table. The streams are splitmix64 + Box-Muller in ``gen.c``; this module
compiles that file with the host C compiler on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_SO = os.path.join(_HERE, "_synthgen.so")
_lock = threading.Lock()
_lib = None

# Seeds fixed for every workload: weights, inputs, page permutation.
SEED_WEIGHTS = 0
SEED_INPUTS = 1
SEED_PAGES = 2
INIT_STD = 0.02


def build(force: bool = False) -> str:
    """Compile gen.c into a shared object next to it (idempotent)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_splitmix64_at.restype = u64
            lib.synth_splitmix64_at.argtypes = [u64, u64]
            lib.synth_stream_state.restype = u64
            lib.synth_stream_state.argtypes = [u64, u64]
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, dbl, vp]
            lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, dbl, dbl, vp]
            lib.synth_uniform_int.argtypes = [u64, u64, u64, i64, i64, vp]
            lib.synth_permutation.argtypes = [u64, u64, i32, vp]
            lib.synth_bf16_to_f32.argtypes = [vp, u64, vp]
            _lib = lib
    return _lib


# ----------------------------------------------------------------------------- primitives

def splitmix64_at(state0: int, i: int) -> int:
    return int(_load().synth_splitmix64_at(state0, i))


def normal_bf16(seed: int, stream: int, shape, std: float = INIT_STD, mean: float = 0.0,
                offset: int = 0) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of mean + std * N(0,1), rounded from fp32."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(seed, stream, offset, out.size, mean, std, out.ctypes.data)
    return out


def normal_f32(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0,
               offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, stream, offset, out.size, mean, std, out.ctypes.data)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] inclusive, int32."""
    out = np.empty(n, dtype=np.int32)
    _load().synth_uniform_int(seed, stream, n, lo, hi, out.ctypes.data)
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_permutation(seed, stream, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().synth_bf16_to_f32(bits.ctypes.data, bits.size, out.ctypes.data)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 round-to-nearest-even, as bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- model shapes

@dataclass(frozen=True)
class ModelShape:
    name: str
    L: int          # decoder layers
    d: int          # model width
    n_q: int        # query heads
    n_kv: int       # key/value heads
    d_h: int        # head dim
    ffn: int        # SwiGLU intermediate width
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-5
    qkv_bias: bool = False


TINY = ModelShape("tiny", L=4, d=256, n_q=4, n_kv=2, d_h=64, ffn=688, vocab=1024, rope_theta=10000.0)
LLAMA8B = ModelShape("llama3.1-8b", L=32, d=4096, n_q=32, n_kv=8, d_h=128, ffn=14336,
                     vocab=128256, rope_theta=500000.0)
LLAMA70B = ModelShape("llama3.1-70b", L=80, d=8192, n_q=64, n_kv=8, d_h=128, ffn=28672,
                      vocab=128256, rope_theta=500000.0)
QWEN14B = ModelShape("qwen2.5-14b", L=48, d=5120, n_q=40, n_kv=8, d_h=128, ffn=13824,
                     vocab=152064, rope_theta=1000000.0, qkv_bias=True)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    l: int                  # full layers (1..l run in full)
    g: int                  # AcrossKV group size (1 = plain SwiftKV)
    num_prompts: int
    len_lo: int
    len_hi: int
    decode_steps: int = 0
    page_size: int = 16
    # serving-step mix (chunked prefill with decode tokens): mix_decode sequences with a
    # cached context U[mix_decode_ctx] contribute one decode token each; mix_chunks holds
    # (cached tokens, chunk tokens) of prompt chunks. Empty: a plain prompt batch.
    mix_decode: int = 0
    mix_decode_ctx: tuple = (0, 0)
    mix_chunks: tuple = ()
    kv_dtype: str = "bf16"  # "fp8": per-token float8 e4m3 KV cache

    @property
    def mixed(self) -> bool:
        return self.mix_decode > 0 or len(self.mix_chunks) > 0


# an 8192-token serving step: four 2016-token chunks of 8064-token prompts (at each of the
# four chunk offsets) and 128 decode tokens of requests with 2000-token prompts and up to
# 250 generated tokens
_MIX_8K = dict(mix_decode=128, mix_decode_ctx=(2000, 2250),
               mix_chunks=((0, 2016), (2016, 2016), (4032, 2016), (6048, 2016)))

WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_l2", TINY, l=2, g=1, num_prompts=1, len_lo=128, len_hi=128, decode_steps=8),
        Workload("llama8b_l16", LLAMA8B, l=16, g=1, num_prompts=16, len_lo=500, len_hi=1000),
        # the same prompts through the ordinary model (l = L): the baseline SwiftKV is measured against
        Workload("llama8b_full", LLAMA8B, l=32, g=1, num_prompts=16, len_lo=500, len_hi=1000),
        Workload("llama8b_l24", LLAMA8B, l=24, g=1, num_prompts=32, len_lo=500, len_hi=1000),
        Workload("llama8b_l24_g2", LLAMA8B, l=24, g=2, num_prompts=32, len_lo=500, len_hi=1000),
        Workload("llama8b_l16_g2", LLAMA8B, l=16, g=2, num_prompts=32, len_lo=500, len_hi=1000),
        Workload("llama70b_l40", LLAMA70B, l=40, g=1, num_prompts=8, len_lo=500, len_hi=1000),
        Workload("qwen14b_l24_g4", QWEN14B, l=24, g=4, num_prompts=24, len_lo=1000, len_hi=1000,
                 decode_steps=100),
        # 50 % SwiftKV + 4-way AcrossKV + per-token FP8 KV cache (the pages' Table B.1 / Table 3
        # configuration), bf16 and fp8 caches
        Workload("llama8b_l16_g4", LLAMA8B, l=16, g=4, num_prompts=16, len_lo=500, len_hi=1000),
        Workload("llama8b_l16_g4_fp8", LLAMA8B, l=16, g=4, num_prompts=16, len_lo=500, len_hi=1000,
                 kv_dtype="fp8"),
        Workload("qwen14b_l24_g4_fp8", QWEN14B, l=24, g=4, num_prompts=24, len_lo=1000, len_hi=1000,
                 decode_steps=100, kv_dtype="fp8"),
        Workload("llama8b_l16_mixed_fp8", LLAMA8B, l=16, g=1, num_prompts=0, len_lo=0, len_hi=0, kv_dtype="fp8",
                 **_MIX_8K),
        Workload("llama8b_l16_mixed", LLAMA8B, l=16, g=1, num_prompts=0, len_lo=0, len_hi=0, **_MIX_8K),
        # the same serving step through the ordinary model (l = L)
        Workload("llama8b_full_mixed", LLAMA8B, l=32, g=1, num_prompts=0, len_lo=0, len_hi=0, **_MIX_8K),
    ]
}

# ----------------------------------------------------------------------------- weights

# stream ids
_S_EMBED, _S_GFINAL, _S_LM = 1, 2, 3
(_K_GATTN, _K_WQ, _K_WK, _K_WV, _K_BQ, _K_BK, _K_BV, _K_WO, _K_GMLP, _K_WG, _K_WU,
 _K_WD) = range(12)


def _layer_stream(j: int, kind: int) -> int:
    return 256 * (j + 1) + kind


def _gain(seed: int, stream: int, n: int, gain_std: float) -> np.ndarray:
    if gain_std == 0.0:
        return np.ones(n, dtype=np.float32)
    bits = normal_bf16(seed, stream, (n,), std=gain_std, mean=1.0)
    return bf16_bits_to_f32(bits)


def layer_weights(shape: ModelShape, j: int, seed: int = SEED_WEIGHTS, gain_std: float = 0.0,
                  kinds=None) -> dict:
    """Weights of decoder layer j (0-based) in nn.Linear layout [out][in].

    Matrices are bfloat16 bit patterns (uint16); gains and biases float32
    holding bfloat16-representable values.
    """
    d, hq, hkv, dh, F = shape.d, shape.n_q * shape.d_h, shape.n_kv * shape.d_h, shape.d_h, shape.ffn
    del dh
    spec = {
        "wq": (_K_WQ, (hq, d)), "wk": (_K_WK, (hkv, d)), "wv": (_K_WV, (hkv, d)),
        "wo": (_K_WO, (d, hq)), "wg": (_K_WG, (F, d)), "wu": (_K_WU, (F, d)), "wd": (_K_WD, (d, F)),
    }
    out = {}
    want = set(kinds) if kinds is not None else None
    for name, (kind, shp) in spec.items():
        if want is None or name in want:
            out[name] = normal_bf16(seed, _layer_stream(j, kind), shp)
    for name, kind in (("gamma_attn", _K_GATTN), ("gamma_mlp", _K_GMLP)):
        if want is None or name in want:
            out[name] = _gain(seed, _layer_stream(j, kind), d, gain_std)
    if shape.qkv_bias:
        for name, kind, n in (("bq", _K_BQ, hq), ("bk", _K_BK, hkv), ("bv", _K_BV, hkv)):
            if want is None or name in want:
                out[name] = bf16_bits_to_f32(normal_bf16(seed, _layer_stream(j, kind), (n,)))
    return out


def global_weights(shape: ModelShape, seed: int = SEED_WEIGHTS, gain_std: float = 0.0,
                   kinds=None) -> dict:
    want = set(kinds) if kinds is not None else None
    out = {}
    if want is None or "embed" in want:
        out["embed"] = normal_bf16(seed, _S_EMBED, (shape.vocab, shape.d))
    if want is None or "gamma_final" in want:
        out["gamma_final"] = _gain(seed, _S_GFINAL, shape.d, gain_std)
    if want is None or "lm_head" in want:
        out["lm_head"] = normal_bf16(seed, _S_LM, (shape.vocab, shape.d))
    return out


def embed_rows(shape: ModelShape, tokens: np.ndarray, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """Rows of the embedding table for the given token ids (bf16 bits), without
    generating the whole table."""
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.empty((len(tokens), shape.d), dtype=np.uint16)
    for i, t in enumerate(tokens):
        out[i] = normal_bf16(seed, _S_EMBED, (shape.d,), offset=int(t) * shape.d)
    return out


# ----------------------------------------------------------------------------- prompts

@dataclass
class Batch:
    """A packed varlen prompt batch with its paged-KV block table."""
    lens: np.ndarray          # int32[P]
    cu_seqlens: np.ndarray    # int32[P+1]
    tokens: np.ndarray        # int32[T]
    block_table: np.ndarray   # int32[P][max_pages]; -1 past the end
    num_pages: int
    page_size: int = 16
    extra: dict = field(default_factory=dict)


def prompt_batch(vocab: int, num_prompts: int, len_lo: int, len_hi: int, page_size: int = 16,
                 reserve_tokens: int = 0, spare_pages: int = 0, seed: int = SEED_INPUTS,
                 page_seed: int = SEED_PAGES, lens=None) -> Batch:
    """Prompt lengths U[len_lo, len_hi], token ids U[0, vocab), and a block table
    drawn from a shuffled page pool. ``reserve_tokens`` leaves room in every
    sequence's block table for that many decode tokens."""
    if lens is None:
        lens = uniform_int(seed, 11, num_prompts, len_lo, len_hi)
    lens = np.asarray(lens, dtype=np.int32)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    tokens = uniform_int(seed, 12, T, 0, vocab - 1)
    pages_per = [(int(n) + reserve_tokens + page_size - 1) // page_size for n in lens]
    max_pages = max(pages_per) if pages_per else 1
    num_pages = sum(pages_per) + spare_pages
    perm = permutation(page_seed, 13, num_pages)
    bt = np.full((len(lens), max(max_pages, 1)), -1, dtype=np.int32)
    k = 0
    for s, m in enumerate(pages_per):
        bt[s, :m] = perm[k:k + m]
        k += m
    return Batch(lens=lens, cu_seqlens=cu, tokens=tokens, block_table=bt, num_pages=num_pages,
                 page_size=page_size)


def mixed_batch(vocab: int, chunks, num_decode: int, decode_ctx_lo: int, decode_ctx_hi: int,
                page_size: int = 16, seed: int = SEED_INPUTS, page_seed: int = SEED_PAGES) -> Batch:
    """A serving step: prompt chunks [(ctx, n)] followed by num_decode one-token chunks
    whose contexts are U[decode_ctx_lo, decode_ctx_hi]. lens / cu_seqlens / tokens describe
    the step's chunks; extra["ctx"] holds each sequence's cached length and
    extra["prefix_tokens"] / extra["prefix_cu"] the token ids of those cached prefixes
    (to fill the cache before the step). The block table covers ctx + n per sequence."""
    ctx = [int(c) for c, _ in chunks] + list(uniform_int(seed, 21, num_decode, decode_ctx_lo, decode_ctx_hi))
    lens = np.asarray([int(n) for _, n in chunks] + [1] * num_decode, dtype=np.int32)
    ctx = np.asarray(ctx, dtype=np.int32)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    tokens = uniform_int(seed, 22, int(cu[-1]), 0, vocab - 1)
    pcu = np.zeros(len(lens) + 1, dtype=np.int32)
    pcu[1:] = np.cumsum(ctx)
    prefix = uniform_int(seed, 23, int(pcu[-1]), 0, vocab - 1)
    pages_per = [(int(c) + int(n) + page_size - 1) // page_size for c, n in zip(ctx, lens)]
    num_pages = sum(pages_per)
    perm = permutation(page_seed, 24, num_pages)
    bt = np.full((len(lens), max(pages_per)), -1, dtype=np.int32)
    k = 0
    for s, m in enumerate(pages_per):
        bt[s, :m] = perm[k:k + m]
        k += m
    return Batch(lens=lens, cu_seqlens=cu, tokens=tokens, block_table=bt, num_pages=num_pages,
                 page_size=page_size, extra={"ctx": ctx, "prefix_tokens": prefix, "prefix_cu": pcu})


def workload_batch(w: Workload, reserve_tokens: int = 0) -> Batch:
    return prompt_batch(w.shape.vocab, w.num_prompts, w.len_lo, w.len_hi, w.page_size,
                        reserve_tokens=reserve_tokens)
