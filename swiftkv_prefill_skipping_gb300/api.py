"""Torch-facing layer over the C ABI: weights in, paged caches, prefill, decode.

PyTorch provides device memory and streams only; all computation happens in
libswiftkv.so. Every call checks the library's return code and raises
``SwiftKVError`` on failure.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import binding as B


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    assert a.is_contiguous()
    return a.data_ptr()


@dataclass
class Shape:
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

    @classmethod
    def of(cls, s):
        return cls(L=s.L, d=s.d, n_q=s.n_q, n_kv=s.n_kv, d_h=s.d_h, ffn=s.ffn, vocab=s.vocab,
                   rope_theta=s.rope_theta, rms_eps=s.rms_eps, qkv_bias=s.qkv_bias)

    def config(self) -> B.ModelConfig:
        return B.ModelConfig(self.L, self.d, self.n_q, self.n_kv, self.d_h, self.ffn, self.vocab,
                             int(self.qkv_bias), self.rope_theta, self.rms_eps)


class Model:
    """A SwiftKV model on the current CUDA device, packed for (l, g)."""

    def __init__(self, shape, l: int, g: int = 1):
        self.shape = Shape.of(shape)
        self.l, self.g = l, g
        self.num_caches = B.cache_count(self.shape.L, l, g)
        self._cfg = self.shape.config()
        h = C.c_void_p()
        B.check(B.lib().swiftkv_model_create(C.byref(self._cfg), l, g, C.byref(h)))
        self.handle = h

    def load_layer(self, j: int, w: dict, stream=None) -> None:
        lw = B.LayerWeights(*[_ptr(w.get(k)) for k in (
            "gamma_attn", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "gamma_mlp", "wg", "wu", "wd")])
        B.check(B.lib().swiftkv_load_layer(self.handle, j, C.byref(lw), _stream(stream)))

    def load_globals(self, w: dict, stream=None) -> None:
        B.check(B.lib().swiftkv_load_globals(self.handle, _ptr(w["embed"]), _ptr(w["gamma_final"]),
                                             _ptr(w["lm_head"]), _stream(stream)))

    def free(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            B.lib().swiftkv_free(self.handle)
            self.handle = C.c_void_p()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def status(self, clear: bool = True) -> int:
        return B.check(B.lib().swiftkv_status(self.handle, int(clear)))

    def memory(self):
        wb, sb = C.c_size_t(), C.c_size_t()
        B.check(B.lib().swiftkv_memory(self.handle, C.byref(wb), C.byref(sb)))
        return wb.value, sb.value


def load_synthetic(shape, l: int, g: int = 1, seed: int = 0, gain_std: float = 0.0) -> Model:
    """Model with the seeded synthetic weights of the shared generator (inputs only)."""
    import synth
    m = Model(shape, l, g)
    for j in range(shape.L):
        rep = j < l or (j - l) % g == 0
        kinds = None if rep else ("wq", "wo", "wg", "wu", "wd", "gamma_attn", "gamma_mlp", "bq")
        m.load_layer(j, synth.layer_weights(shape, j, seed=seed, gain_std=gain_std, kinds=kinds))
    m.load_globals(synth.global_weights(shape, seed=seed, gain_std=gain_std))
    return m


class KVCache:
    """Caller-owned paged KV cache: num_caches x (K, V) pools of [num_pages][n_kv][16][d_h]
    elements plus a device block table. dtype "bf16": bfloat16 elements; dtype "fp8":
    uint8 float8-e4m3 codes with float32 scales [num_pages][n_kv][16] per pool (per-token
    FP8)."""

    def __init__(self, model: Model, num_pages: int, block_table: np.ndarray, device=None, dtype: str = "bf16"):
        if dtype not in ("bf16", "fp8"):
            raise ValueError(f"KV cache dtype {dtype!r}")
        s = model.shape
        dev = device or torch.device("cuda", torch.cuda.current_device())
        self.num_pages, self.dtype = num_pages, dtype
        shape = (model.num_caches, num_pages, s.n_kv, 16, s.d_h)
        elem = torch.bfloat16 if dtype == "bf16" else torch.uint8
        self.k = torch.zeros(shape, dtype=elem, device=dev)
        self.v = torch.zeros(shape, dtype=elem, device=dev)
        self.k_scale = self.v_scale = None
        if dtype == "fp8":
            self.k_scale = torch.zeros(shape[:-1], dtype=torch.float32, device=dev)
            self.v_scale = torch.zeros(shape[:-1], dtype=torch.float32, device=dev)
        self.block_table = torch.as_tensor(np.ascontiguousarray(block_table, dtype=np.int32), device=dev)
        n = model.num_caches
        self._kp = (C.c_void_p * n)(*[self.k[c].data_ptr() for c in range(n)])
        self._vp = (C.c_void_p * n)(*[self.v[c].data_ptr() for c in range(n)])
        self._ks = self._vs = None
        if dtype == "fp8":
            self._ks = (C.c_void_p * n)(*[self.k_scale[c].data_ptr() for c in range(n)])
            self._vs = (C.c_void_p * n)(*[self.v_scale[c].data_ptr() for c in range(n)])
        self.num_caches = n
        self.pages = self._pages(self.block_table)

    def _pages(self, block_table: torch.Tensor) -> B.KVPages:
        ptr = lambda a: C.cast(a, C.POINTER(C.c_void_p)) if a is not None else None  # noqa: E731
        return B.KVPages(ptr(self._kp), ptr(self._vp), self.num_caches, self.num_pages, 16, block_table.data_ptr(),
                         block_table.shape[1], 1 if self.dtype == "fp8" else 0, ptr(self._ks), ptr(self._vs))

    def view(self, rows: Sequence[int]) -> "KVCache":
        """The same pools with block table rows `rows` (in that order): a batch that holds
        only some of the sequences, or holds them in another order."""
        out = object.__new__(KVCache)
        out.__dict__.update(self.__dict__)
        out.block_table = self.block_table[torch.as_tensor(list(rows), dtype=torch.long,
                                                           device=self.block_table.device)].contiguous()
        out.pages = out._pages(out.block_table)
        return out

    def _rows(self, pool: torch.Tensor, s: int, n: int) -> torch.Tensor:
        bt = self.block_table[s]
        pos = torch.arange(n, device=pool.device)
        return pool[bt[pos // 16].long(), :, pos % 16]

    def gather(self, c: int, s: int, n: int, which: str = "k") -> torch.Tensor:
        """Cache c's first n rows of sequence s, [n, n_kv, d_h] (test/inspection helper);
        for an fp8 cache the values code * scale in float32."""
        pool = self.k[c] if which == "k" else self.v[c]
        if self.dtype == "bf16":
            return self._rows(pool, s, n)
        return self.codes(c, s, n, which) * self.scales(c, s, n, which)[..., None]

    def codes(self, c: int, s: int, n: int, which: str = "k") -> torch.Tensor:
        """fp8 cache: the e4m3 codes of cache c's first n rows of sequence s, as float32."""
        pool = self.k[c] if which == "k" else self.v[c]
        return self._rows(pool, s, n).view(torch.float8_e4m3fn).float()

    def scales(self, c: int, s: int, n: int, which: str = "k") -> torch.Tensor:
        """fp8 cache: the float32 scales [n, n_kv] of cache c's first n rows of sequence s."""
        pool = self.k_scale[c] if which == "k" else self.v_scale[c]
        return self._rows(pool, s, n)


def prefill(model: Model, tokens: torch.Tensor, cu_seqlens: Sequence[int], kv: KVCache,
            logits: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """SwiftKV prefill: fills every cache of kv, returns [P, V] last-token logits."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    P = len(cu) - 1
    if logits is None:
        logits = torch.empty((P, model.shape.vocab), dtype=torch.float32, device=kv.k.device)
    tokens = tokens.to(torch.int32).contiguous()
    B.check(B.lib().swiftkv_prefill(model.handle, tokens.data_ptr(), cu.ctypes.data, P, model.l, model.g,
                                    C.byref(kv.pages), logits.data_ptr(), _stream(stream)))
    return logits


def prefill_host(model: Model, tokens: np.ndarray, cu_seqlens: Sequence[int], kv: KVCache,
                 logits: Optional[np.ndarray] = None, stream=None) -> np.ndarray:
    """prefill with host token ids and host logits (copies inside the call; synchronous)."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    P = len(cu) - 1
    if logits is None:
        logits = np.empty((P, model.shape.vocab), dtype=np.float32)
    B.check(B.lib().swiftkv_prefill_host(model.handle, _ptr(tokens), cu.ctypes.data, P, model.l, model.g,
                                         C.byref(kv.pages), _ptr(logits), _stream(stream)))
    return logits


def forward(model: Model, tokens: torch.Tensor, cu_seqlens: Sequence[int], ctx_lens: Optional[Sequence[int]],
            kv: KVCache, logits: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Serving forward over prompt chunks and decode tokens: chunk s follows ctx_lens[s]
    tokens already in kv (None: none); returns [P, V] logits of each chunk's last token."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    P = len(cu) - 1
    ctx = None if ctx_lens is None else np.ascontiguousarray(ctx_lens, dtype=np.int32)
    if ctx is not None and len(ctx) != P:
        raise ValueError(f"ctx_lens has {len(ctx)} entries for {P} chunks")
    if logits is None:
        logits = torch.empty((P, model.shape.vocab), dtype=torch.float32, device=kv.k.device)
    tokens = tokens.to(torch.int32).contiguous()
    B.check(B.lib().swiftkv_forward(model.handle, tokens.data_ptr(), cu.ctypes.data,
                                    None if ctx is None else ctx.ctypes.data, P, model.l, model.g,
                                    C.byref(kv.pages), logits.data_ptr(), _stream(stream)))
    return logits


def decode_step(model: Model, tokens: torch.Tensor, seq_lens: Sequence[int], kv: KVCache, stream=None):
    """One decode token per sequence; returns (logits [B, V], next token ids [B])."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    Bsz = len(sl)
    dev = kv.k.device
    logits = torch.empty((Bsz, model.shape.vocab), dtype=torch.float32, device=dev)
    nxt = torch.empty((Bsz,), dtype=torch.int32, device=dev)
    tokens = tokens.to(torch.int32).contiguous()
    B.check(B.lib().swiftkv_decode_step(model.handle, tokens.data_ptr(), sl.ctypes.data, Bsz, C.byref(kv.pages),
                                        logits.data_ptr(), nxt.data_ptr(), _stream(stream)))
    return logits, nxt
