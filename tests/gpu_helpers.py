"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare them at the stated tolerances."""
from __future__ import annotations

import numpy as np

import oracle
import synth
from oracle import model as OM

KV_REL_TOL = 1e-2      # per cache and K/V tensor: ||gpu - ref||_2 / ||ref||_2
LOGIT_ABS_TOL = 5e-2   # last-token logits, max |gpu - ref|
# Element-wise, per cache and K/V tensor: max |gpu - ref| / max |ref| (one wrong element or
# row shows here even when it hides under the L2 norm).
KV_MAXREL_TOL = 1e-2
# The fused-RMSNorm mode (swiftkv_set_norm_fusion 1) rounds each GEMM input to bf16 at
# gamma * x instead of gamma * x / rms, so about a quarter of the cache entries sit one bf16
# ulp from the oracle's rounding already at the first layer. One ulp of a value just above a
# power of two is 2^-7 of it, and after a few layers the largest entries may sit two ulps
# apart: that mode's element-wise bound is two bf16 ulps of the largest value.
FUSED_MAXREL_TOL = 2.0 ** -6

# d_head = 128 shape with several 128-row GEMM tiles and attention tiles (tcgen05 attention)
SMALL128 = synth.ModelShape("small-d128", L=6, d=512, n_q=4, n_kv=2, d_h=128, ffn=1000, vocab=2048,
                            rope_theta=500000.0)
# wide enough that the Q/K/V (6144), gate/up (9728), skipped-layer KV at l = 1 (6144) and LM
# head (5120) GEMMs of the tail and of decode take the TMA-fed skinny kernel (>= 76 tiles)
MEDIUM = synth.ModelShape("medium-wide", L=4, d=1024, n_q=32, n_kv=8, d_h=128, ffn=4864, vocab=5120,
                          rope_theta=500000.0)
# GQA group of 8 query heads per KV head (the Llama-3.1-70B ratio): the largest group the
# single-row attention kernels take as rows of one MMA operand
GQA8 = synth.ModelShape("small-gqa8", L=4, d=512, n_q=16, n_kv=2, d_h=128, ffn=768, vocab=1024,
                        rope_theta=500000.0)
# Q/K/V bias (Qwen-style), single KV head
SMALL_BIAS = synth.ModelShape("small-bias", L=4, d=640, n_q=5, n_kv=1, d_h=128, ffn=704, vocab=1024,
                              rope_theta=1000000.0, qkv_bias=True)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def max_rel(a, b) -> float:
    """Element-wise error of a whole tensor: max |a - b| / max |b| (one bad element or row
    shows here even when it hides under the L2 norm)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def run_gpu_prefill(shape, l, g, batch, gain_std=0.0, seed=0, model=None):
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    m = model or api.load_synthetic(shape, l, g, seed=seed, gain_std=gain_std)
    kv = api.KVCache(m, batch.num_pages, batch.block_table)
    tok = torch.as_tensor(batch.tokens, device="cuda")
    logits = api.prefill(m, tok, batch.cu_seqlens, kv)
    torch.cuda.synchronize()
    return m, kv, logits


def oracle_prefill(shape, l, g, batch, prompts=None, gain_std=0.0, seed=0, cache_layers=True):
    w = oracle.synth_weights(shape, seed=seed, gain_std=gain_std, cache_layers=cache_layers)
    cfg = oracle.config_of(shape)
    idx = range(len(batch.lens)) if prompts is None else prompts
    toks = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in idx]
    caches, logits = OM.swiftkv_prefill(cfg, w, toks, l, g)
    return list(idx), caches, logits, w


def compare_prefill(kv, logits_gpu, batch, idx, caches, logits_ref, num_caches):
    """Worst errors over the prompts in idx: (KV relative L2, KV element-wise max|d|/max|ref|,
    logits max-abs), each cache's K and V tensors compared separately."""
    worst_kv, worst_el, worst_lg = 0.0, 0.0, 0.0
    lg = logits_gpu.float().cpu().numpy()
    for i, s in enumerate(idx):
        n = int(batch.lens[s])
        for c in range(num_caches):
            for which, t in (("k", 0), ("v", 1)):
                got = kv.gather(c, s, n, which).float().cpu().numpy()
                worst_kv = max(worst_kv, rel_l2(got, caches[i][c][t]))
                worst_el = max(worst_el, max_rel(got, caches[i][c][t]))
        worst_lg = max(worst_lg, float(np.abs(lg[s] - logits_ref[i]).max()))
    return worst_kv, worst_el, worst_lg


def untouched_rows_are_zero(kv, batch) -> bool:
    """Bookkeeping: nothing was written outside the sequences' own (page, row) slots."""
    import torch
    used = torch.zeros(kv.k.shape[1] * 16, dtype=torch.bool)
    for s, n in enumerate(batch.lens):
        for p in range(int(n)):
            used[int(batch.block_table[s][p // 16]) * 16 + p % 16] = True
    k = kv.k.float().abs().sum(dim=(2, 4)).permute(1, 2, 0).reshape(-1, kv.k.shape[0]).cpu()
    v = kv.v.float().abs().sum(dim=(2, 4)).permute(1, 2, 0).reshape(-1, kv.v.shape[0]).cpu()
    return bool((k[~used] == 0).all() and (v[~used] == 0).all() and (k[used] > 0).all())
