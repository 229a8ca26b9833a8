"""Oracle: the SwiftKV model and its prefill-skipping algorithm, in plain float64 NumPy.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module;
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` call it. It shares no code with the CUDA library.

Sources (page titles, sections):
  [S] "SwiftKV: Fast Prefill-Optimized Inference with Knowledge-Preserving
      Model Transformation" (paper summary page), section 3.
  [P] the SwiftKV paper text quoted on the "AISQL AI_PARSE_DOCUMENT" page,
      sections 3.4 "Efficient Distillation" and 3.5 "Optimized Implementation
      for Inference".

Precision. The pages run every model in BF16 ([S] section 5, hardware). The
oracle therefore keeps weights, the KV cache, the queries and every input of a
linear layer at bfloat16 values (``bf16``), and does all other arithmetic
(norms, accumulations, RoPE angles, softmax and its weights, residual stream)
in float64.

Layer indices are 0-based in code: layers 0..l-1 run in full (the pages'
layers 1..l), layers l..L-1 are skipped for prompt tokens, and "x_l" (the
pages' x_{l+1}) is the residual stream entering layer l.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------- numerics

def bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 value: 8 significant bits, ties to even.

    Works on float64 directly (no double rounding through float32)."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


# Precision mode. float64 everywhere is the definition. Tests evaluate the same model with
# everything except the model's own bfloat16 rounding points in float32 - accumulations (the
# linear layers' dot products, the attention scores, the softmax normaliser and weighted sum
# of V, the RMSNorm mean of squares) and every other operation (norm scaling, RoPE, SiLU and
# the SwiGLU product, softmax exponentials, bias and residual adds) - the GPU path's declared
# arithmetic (bfloat16 operands, float32 compute and accumulation), to measure the rounding
# floor any implementation of that precision faces against the definition. Nothing is rounded
# to a format narrower than float32 beyond the bfloat16 points the model itself has.
_LINEAR_ACC = [F64]


def _mode():
    """The precision mode's type (float64: the definition)."""
    return _LINEAR_ACC[-1]


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma."""
    x = np.asarray(x, dtype=F64)
    t = _mode()
    if t is F64:
        return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gamma, F64)
    xt = x.astype(t)
    ms = np.mean(xt * xt, axis=-1, keepdims=True, dtype=t)
    r = (t(1) / np.sqrt(ms + t(eps))).astype(t)
    return (xt * r * np.asarray(gamma).astype(t)).astype(F64)


class compute_in:
    """Context manager: evaluate every quantity that the model does not round to bfloat16
    itself (accumulations, norm scaling, RoPE, SiLU, softmax, bias and residual adds) in
    `dtype`; values that are bfloat16 stay exact."""

    def __init__(self, dtype):
        self.dtype = dtype

    def __enter__(self):
        _LINEAR_ACC.append(self.dtype)
        return self

    def __exit__(self, *exc):
        _LINEAR_ACC.pop()
        return False


def linear(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None,
           block: int = 8192) -> np.ndarray:
    """x @ w.T (+ b), w in nn.Linear layout [out][in]; w may be stored as float32
    (bfloat16 values) and is widened to float64 one block of output rows at a time."""
    acc = _mode()
    x = np.asarray(x, dtype=F64)
    xa = x.astype(acc)
    n_out = w.shape[0]
    out = np.empty(x.shape[:-1] + (n_out,), dtype=F64)
    for i in range(0, n_out, block):
        out[..., i:i + block] = xa @ np.asarray(w[i:i + block], dtype=acc).T
    if b is not None:
        if acc is F64:
            out += np.asarray(b, F64)
        else:
            out = (out.astype(acc) + np.asarray(b).astype(acc)).astype(F64)
    return out


def residual_add(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """The residual stream's update x + y (in the precision mode's type)."""
    t = _mode()
    if t is F64:
        return np.asarray(x, F64) + np.asarray(y, F64)
    return (np.asarray(x).astype(t) + np.asarray(y).astype(t)).astype(F64)


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half form, on x [n, heads, d_h].

    Dimension i < d_h/2 is paired with i + d_h/2 and rotated by the angle
    pos * theta^(-2i/d_h)."""
    x = np.asarray(x, dtype=F64)
    d_h = x.shape[-1]
    half = d_h // 2
    inv_freq = np.power(F64(theta), -2.0 * np.arange(half, dtype=F64) / d_h)
    ang = np.asarray(pos, dtype=F64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    t = _mode()
    if t is not F64:  # the rotation in the precision mode's type (angles in float64)
        c, s, x = c.astype(t), s.astype(t), x.astype(t)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1).astype(F64)


def silu(x: np.ndarray) -> np.ndarray:
    t = _mode()
    if t is not F64:
        xt = np.asarray(x).astype(t)
        return (xt / (t(1) + np.exp(-xt))).astype(F64)
    return x / (1.0 + np.exp(-x))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u (the product in the precision mode's type)."""
    t = _mode()
    if t is F64:
        return silu(g) * u
    return (silu(g).astype(t) * np.asarray(u).astype(t)).astype(F64)


def causal_gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
                         k_pos: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(d_h)) v with a causal mask (key position <= query
    position). q [n, n_q, d_h]; k, v [m, n_kv, d_h]; query head h reads key/value
    head h // (n_q / n_kv)."""
    n_q, d_h = q.shape[1], q.shape[2]
    grp = n_q // k.shape[1]
    allowed = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    out = np.empty(q.shape, dtype=F64)
    scale = 1.0 / np.sqrt(F64(d_h))
    t = _mode()
    for h in range(n_q):
        kv = h // grp
        if t is F64:
            s = (q[:, h, :] @ k[:, kv, :].T) * scale
            s = np.where(allowed, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[:, h, :] = p @ v[:, kv, :]
        else:  # everything in the mode's type; unnormalised weights applied to V, then divided
            s = (q[:, h, :].astype(t) @ k[:, kv, :].T.astype(t)) * t(scale)
            s = np.where(allowed, s, t(-np.inf))
            p = np.exp(s - s.max(axis=1, keepdims=True))
            denom = p.sum(axis=1, keepdims=True, dtype=t)
            out[:, h, :] = ((p @ v[:, kv, :].astype(t)) / denom).astype(F64)
    return out


# ----------------------------------------------------------------------------- model

@dataclass(frozen=True)
class Config:
    L: int
    d: int
    n_q: int
    n_kv: int
    d_h: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-5
    qkv_bias: bool = False


@dataclass
class Layer:
    """One decoder layer's weights, [out][in] matrices (bfloat16 values)."""
    gamma_attn: np.ndarray
    wq: np.ndarray
    wk: Optional[np.ndarray]
    wv: Optional[np.ndarray]
    wo: np.ndarray
    gamma_mlp: np.ndarray
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray
    bq: Optional[np.ndarray] = None
    bk: Optional[np.ndarray] = None
    bv: Optional[np.ndarray] = None


class Weights:
    """Weights of the whole model. ``layer(j)`` may load lazily."""

    def __init__(self, layer_fn: Callable[[int], Layer], embed_fn: Callable[[np.ndarray], np.ndarray],
                 gamma_final: np.ndarray, lm_head: np.ndarray):
        self._layer_fn = layer_fn
        self._embed_fn = embed_fn
        self.gamma_final = gamma_final
        self.lm_head = lm_head

    def layer(self, j: int) -> Layer:
        return self._layer_fn(j)

    def embed(self, tokens: np.ndarray) -> np.ndarray:
        return np.asarray(self._embed_fn(np.asarray(tokens)), dtype=F64)


# ----------------------------------------------------------------------------- FP8 KV cache
#
# Per-token FP8 KV-cache quantization ([S] 3.4 AcrossKV "Complementarity with KV
# quantization", Appendix B.1 / Table B.1; [S] Table 3): post-training, no retraining.
# Reading: each token's K (after RoPE) and V vector of one KV head -- the bfloat16 values a
# bf16 cache would hold -- gets one float32 scale, amax / 448, and float8 e4m3 codes of
# value / scale (448 is the largest finite e4m3 value); the attention uses code * scale.

E4M3_MAX = 448.0


def e4m3(x) -> np.ndarray:
    """Round to the nearest float8 e4m3 ("fn": no infinities, largest finite 448) value,
    ties to even: 4 significant bits for |x| >= 2^-6, steps of 2^-9 below (subnormals);
    magnitudes past 448 saturate to 448."""
    x = np.asarray(x, dtype=F64)
    a = np.abs(x)
    _, e = np.frexp(a)                  # a = m * 2^e, m in [0.5, 1): floor(log2 a) = e - 1
    quantum = np.exp2(np.maximum(e - 1.0, -6.0) - 3.0)
    r = np.rint(a / quantum) * quantum
    return np.sign(x) * np.minimum(r, E4M3_MAX)


def fp8_quantize(v: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Codes (as their e4m3 values) and float32 scales of bfloat16 vectors v[..., d_h]:
    scale = float32(amax) / 448 in float32, code = e4m3(float32(v) / scale) with a
    float32 division (a zero vector has scale 0 and codes 0)."""
    v32 = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v32), axis=-1, keepdims=True)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    q = (v32 / safe).astype(np.float32)
    codes = np.where(scale > 0, e4m3(q), 0.0)
    return codes, scale[..., 0]


def fp8_dequantize(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    return np.asarray(codes, F64) * np.asarray(scale, F64)[..., None]


_KV_FP8 = [False]


class kv_cache_fp8:
    """Context manager: the KV cache stores per-token FP8 (every cache write goes through
    fp8_quantize / fp8_dequantize), as with a float8 KV cache."""

    def __enter__(self):
        _KV_FP8.append(True)
        return self

    def __exit__(self, *exc):
        _KV_FP8.pop()
        return False


def _cache_values(t: np.ndarray) -> np.ndarray:
    """What the cache holds for the bfloat16 K or V rows t[tokens, n_kv, d_h]."""
    return fp8_dequantize(*fp8_quantize(t)) if _KV_FP8[-1] else t


KV = Tuple[np.ndarray, np.ndarray]   # (K, V), each [tokens, n_kv, d_h], values the cache holds


def _heads(x: np.ndarray, h: int, d_h: int) -> np.ndarray:
    return x.reshape(x.shape[0], h, d_h)


def qkv_proj(cfg: Config, lw: Layer, x: np.ndarray, pos: np.ndarray) -> Tuple[np.ndarray, KV]:
    """Ordinary attention input: RMSNorm, Q/K/V projections (+bias), RoPE on Q and K."""
    u = bf16(rms_norm(x, lw.gamma_attn, cfg.rms_eps))
    q = rope(_heads(linear(u, lw.wq, lw.bq), cfg.n_q, cfg.d_h), pos, cfg.rope_theta)
    k = rope(_heads(linear(u, lw.wk, lw.bk), cfg.n_kv, cfg.d_h), pos, cfg.rope_theta)
    v = _heads(linear(u, lw.wv, lw.bv), cfg.n_kv, cfg.d_h)
    return bf16(q), (_cache_values(bf16(k)), _cache_values(bf16(v)))


def q_proj(cfg: Config, lw: Layer, x: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Query of a skipped layer for a token that still runs it: RMSNorm, W_Q (+bias), RoPE."""
    u = bf16(rms_norm(x, lw.gamma_attn, cfg.rms_eps))
    return bf16(rope(_heads(linear(u, lw.wq, lw.bq), cfg.n_q, cfg.d_h), pos, cfg.rope_theta))


def swiftkv_kv(cfg: Config, rep: Layer, x_l: np.ndarray, pos: np.ndarray) -> KV:
    """SwiftKV rewiring ([S] 3.4 "The SwiftKV Rewiring Mechanism", Eq. 2; AcrossKV
    'KV_group = W_KV^rep x_{l+1}'): the KV of a skipped layer (or AcrossKV group)
    projected from the output of the last full layer with the representative
    layer's own input norm and K/V weights."""
    u = bf16(rms_norm(x_l, rep.gamma_attn, cfg.rms_eps))
    k = rope(_heads(linear(u, rep.wk, rep.bk), cfg.n_kv, cfg.d_h), pos, cfg.rope_theta)
    v = _heads(linear(u, rep.wv, rep.bv), cfg.n_kv, cfg.d_h)
    return _cache_values(bf16(k)), _cache_values(bf16(v))


def attn_out(cfg: Config, lw: Layer, x: np.ndarray, q: np.ndarray, kv: KV, q_pos: np.ndarray,
             k_pos: np.ndarray) -> np.ndarray:
    """Residual update of the attention block: x + W_O attention(q, K, V)."""
    a = causal_gqa_attention(q, kv[0], kv[1], q_pos, k_pos)
    a = bf16(a.reshape(a.shape[0], cfg.n_q * cfg.d_h))
    return residual_add(x, linear(a, lw.wo))


def mlp(cfg: Config, lw: Layer, x: np.ndarray) -> np.ndarray:
    """Residual update of the SwiGLU MLP: x + W_down (silu(W_gate u) * (W_up u))."""
    u = bf16(rms_norm(x, lw.gamma_mlp, cfg.rms_eps))
    h = bf16(swiglu(linear(u, lw.wg), linear(u, lw.wu)))
    return residual_add(x, linear(h, lw.wd))


def lm_head(cfg: Config, w: Weights, x: np.ndarray) -> np.ndarray:
    """Final RMSNorm and vocabulary projection."""
    return linear(bf16(rms_norm(x, w.gamma_final, cfg.rms_eps)), w.lm_head)


# ----------------------------------------------------------------------------- cache map

def num_caches(L: int, l: int, g: int) -> int:
    """KV caches kept: l full layers plus (L - l)/g AcrossKV groups
    ([S] 3.4 AcrossKV, "Memory reduction", M_AcrossKV)."""
    check_lg(L, l, g)
    return l + (L - l) // g


def cache_of_layer(j: int, l: int, g: int) -> int:
    """Cache read by layer j (0-based): its own for j < l, else its group's.
    Groups are consecutive runs of g skipped layers ([S] 3.4 AcrossKV "Mechanism")."""
    return j if j < l else l + (j - l) // g


def representative(c: int, l: int, g: int) -> int:
    """Layer whose W_KV (and input norm) fills cache c. For an AcrossKV group this
    is its first layer (the pages say only that one layer is designated)."""
    return c if c < l else l + (c - l) * g


def check_lg(L: int, l: int, g: int) -> None:
    if not (1 <= l <= L):
        raise ValueError(f"l={l} outside [1, {L}]")
    if g < 1 or (L - l) % g != 0:
        raise ValueError(f"AcrossKV group {g} does not divide L-l={L - l}")


# ----------------------------------------------------------------------------- forwards

def ordinary_forward(cfg: Config, w: Weights, tokens: Sequence[int]) -> Tuple[List[KV], np.ndarray]:
    """The unmodified model on one sequence: per-layer KV cache and logits of every token."""
    tokens = np.asarray(tokens)
    pos = np.arange(len(tokens))
    x = w.embed(tokens)
    caches: List[KV] = []
    for j in range(cfg.L):
        lw = w.layer(j)
        q, kv = qkv_proj(cfg, lw, x, pos)
        caches.append(kv)
        x = attn_out(cfg, lw, x, q, kv, pos, pos)
        x = mlp(cfg, lw, x)
    return caches, lm_head(cfg, w, x)


def swiftkv_full_forward(cfg: Config, w: Weights, tokens: Sequence[int], l: int,
                         g: int = 1) -> Tuple[List[KV], np.ndarray]:
    """The SwiftKV model M_swift(l, g) with every token run through every layer.

    Layers j < l are ordinary. At layer l the caches of all AcrossKV groups are
    projected from x_l ([S] Eq. 2). Every layer j >= l computes its own query
    from its own input x_j and attends to its group's cache; its O and MLP are
    ordinary. Returns the caches (l + (L-l)/g of them) and all tokens' logits."""
    check_lg(cfg.L, l, g)
    tokens = np.asarray(tokens)
    pos = np.arange(len(tokens))
    x = w.embed(tokens)
    caches: List[KV] = [None] * num_caches(cfg.L, l, g)  # type: ignore[list-item]
    for j in range(cfg.L):
        lw = w.layer(j)
        if j < l:
            q, kv = qkv_proj(cfg, lw, x, pos)
            caches[j] = kv
        else:
            if j == l:
                for c in range(l, len(caches)):
                    caches[c] = swiftkv_kv(cfg, w.layer(representative(c, l, g)), x, pos)
            q = q_proj(cfg, lw, x, pos)
            kv = caches[cache_of_layer(j, l, g)]
        x = attn_out(cfg, lw, x, q, kv, pos, pos)
        x = mlp(cfg, lw, x)
    return caches, lm_head(cfg, w, x)


def swiftkv_prefill_one(cfg: Config, w: Weights, tokens: Sequence[int], l: int,
                        g: int = 1) -> Tuple[List[KV], np.ndarray]:
    """Prefill skipping on one prompt ([S] 3.2, 3.4 "What operations are skipped",
    "What the first generated token does differently"; [P] 3.5):

    1. every prompt token runs layers 0..l-1 in full, filling caches 0..l-1;
    2. the caches of all skipped layers / AcrossKV groups are projected from x_l;
    3. no prompt token runs Q/attention/O/MLP of layers >= l, except the last,
       which continues through every layer (attending to the projected caches)
       so that its final hidden state gives the first output token's logits.
    Returns all caches and the last token's logits [V]."""
    check_lg(cfg.L, l, g)
    tokens = np.asarray(tokens)
    n = len(tokens)
    if n == 0:
        raise ValueError("empty prompt")
    pos = np.arange(n)
    x = w.embed(tokens)
    caches: List[KV] = [None] * num_caches(cfg.L, l, g)  # type: ignore[list-item]
    for j in range(l):
        lw = w.layer(j)
        q, kv = qkv_proj(cfg, lw, x, pos)
        caches[j] = kv
        x = attn_out(cfg, lw, x, q, kv, pos, pos)
        x = mlp(cfg, lw, x)
    for c in range(l, len(caches)):
        caches[c] = swiftkv_kv(cfg, w.layer(representative(c, l, g)), x, pos)
    xt, pt = x[n - 1:], pos[n - 1:]
    for j in range(l, cfg.L):
        lw = w.layer(j)
        q = q_proj(cfg, lw, xt, pt)
        xt = attn_out(cfg, lw, xt, q, caches[cache_of_layer(j, l, g)], pt, pos)
        xt = mlp(cfg, lw, xt)
    return caches, lm_head(cfg, w, xt)[0]


def swiftkv_prefill(cfg: Config, w: Weights, prompts: Sequence[Sequence[int]], l: int,
                    g: int = 1) -> Tuple[List[List[KV]], np.ndarray]:
    """Prefill skipping on a batch of independent prompts: per-prompt caches and
    the [P, V] last-token logits."""
    caches, logits = [], []
    for toks in prompts:
        c, lg = swiftkv_prefill_one(cfg, w, toks, l, g)
        caches.append(c)
        logits.append(lg)
    return caches, np.stack(logits) if logits else np.zeros((0, cfg.vocab))


def swiftkv_decode_step(cfg: Config, w: Weights, caches: List[KV], token: int, l: int,
                        g: int = 1) -> Tuple[List[KV], np.ndarray]:
    """One decode token of a sequence whose caches hold its n earlier tokens.

    The token runs every layer ([S] 3.2: decode tokens continue through all
    layers). In layers < l it appends its own K/V to that layer's cache. At
    layer l it appends its KV for every skipped cache, projected from its own
    x_l through the representative's W_KV exactly like a prompt token: after
    distillation the original KV projections of layers > l are discarded at
    inference ([P] 3.4). Layers >= l compute their own queries and attend to
    their group's cache. Returns the extended caches and the logits [V]."""
    check_lg(cfg.L, l, g)
    n = caches[0][0].shape[0]
    pos = np.array([n])
    kpos = np.arange(n + 1)
    x = w.embed(np.array([token]))
    out: List[KV] = list(caches)

    def append(c: int, kv: KV) -> None:
        out[c] = (np.concatenate([out[c][0], kv[0]]), np.concatenate([out[c][1], kv[1]]))

    for j in range(cfg.L):
        lw = w.layer(j)
        if j < l:
            q, kv = qkv_proj(cfg, lw, x, pos)
            append(j, kv)
        else:
            if j == l:
                for c in range(l, len(out)):
                    append(c, swiftkv_kv(cfg, w.layer(representative(c, l, g)), x, pos))
            q = q_proj(cfg, lw, x, pos)
        x = attn_out(cfg, lw, x, q, out[cache_of_layer(j, l, g)], pos, kpos)
        x = mlp(cfg, lw, x)
    return out, lm_head(cfg, w, x)[0]


def swiftkv_forward_one(cfg: Config, w: Weights, caches: Optional[List[KV]], tokens: Sequence[int], l: int,
                        g: int = 1) -> Tuple[List[KV], np.ndarray]:
    """One chunk of a sequence whose caches already hold its first ctx tokens (caches None
    or empty for ctx = 0): the serving forward of [S] 3.4 "Inference Implementation in
    Production Serving Frameworks" / [P] 3.5, where every token of the chunk runs layers
    0..l-1 (attending to the cached prefix and to the chunk causally), the caches of every
    skipped layer / AcrossKV group are computed for the chunk's tokens from x_l, and only
    the chunk's last token continues through layers l..L-1. A decode token is a chunk of
    one token; a prompt may be fed in several chunks. Returns the extended caches and the
    last token's logits [V]."""
    check_lg(cfg.L, l, g)
    tokens = np.asarray(tokens)
    n = len(tokens)
    if n == 0:
        raise ValueError("empty chunk")
    C = num_caches(cfg.L, l, g)
    if caches:
        ctx = caches[0][0].shape[0]
        out: List[KV] = list(caches)
    else:
        ctx = 0
        empty = np.zeros((0, cfg.n_kv, cfg.d_h))
        out = [(empty, empty)] * C
    pos = np.arange(ctx, ctx + n)
    kpos = np.arange(ctx + n)

    def append(c: int, kv: KV) -> None:
        out[c] = (np.concatenate([out[c][0], kv[0]]), np.concatenate([out[c][1], kv[1]]))

    x = w.embed(tokens)
    for j in range(l):
        lw = w.layer(j)
        q, kv = qkv_proj(cfg, lw, x, pos)
        append(j, kv)
        x = attn_out(cfg, lw, x, q, out[j], pos, kpos)
        x = mlp(cfg, lw, x)
    for c in range(l, C):
        append(c, swiftkv_kv(cfg, w.layer(representative(c, l, g)), x, pos))
    xt, pt = x[n - 1:], pos[n - 1:]
    for j in range(l, cfg.L):
        lw = w.layer(j)
        q = q_proj(cfg, lw, xt, pt)
        xt = attn_out(cfg, lw, xt, q, out[cache_of_layer(j, l, g)], pt, kpos)
        xt = mlp(cfg, lw, xt)
    return out, lm_head(cfg, w, xt)[0]


def greedy(logits: np.ndarray) -> int:
    """Greedy next token: the lowest index among the maxima."""
    return int(np.argmax(logits))
