"""Per-token FP8 KV cache on the GPU against the oracle's kv_cache_fp8 mode: codes and
scales of every cache, logits of prefill, decode and chunked serving forward.

Codes are an integer decision taken in float32 on both sides from the bfloat16 K/V rows,
so where the GPU's bf16 row equals the oracle's the codes and scale are identical. Cache 0
(the first layer: inputs are embedding rows, the same on both sides) isolates the
quantizer: >= 99 % identical codes, any other code within two e4m3 steps, scales within a
bf16 ulp of the row's largest value. Deeper caches inherit the ~1e-2 relative K/V
differences of float32 vs float64 accumulation, and one e4m3 step is 6-12 % of a value, so
about one code in ten moves by a step there; those are bounded on the dequantized values
(relative L2 <= 5e-2 per cache). Logits: the usual 5e-2."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import GQA8, LOGIT_ABS_TOL, SMALL128, SMALL_BIAS
from oracle import model as OM

pytestmark = pytest.mark.gpu


def _setup(shape, l, g, lens, reserve=0, gain_std=0.0, spare_pages=2):
    # unit gains: the GPU folds a skipped group's input gain into its W_KV rows (one more
    # bf16 rounding of the weights), which with random gains flips many more bf16 K/V values
    # of the skipped caches than the accumulation order alone and so blurs the code check
    from swiftkv_prefill_skipping_gb300 import api
    batch = synth.prompt_batch(shape.vocab, len(lens), 0, 0, lens=lens, reserve_tokens=reserve,
                               spare_pages=spare_pages)
    m = api.load_synthetic(shape, l, g, seed=0, gain_std=gain_std)
    kv = api.KVCache(m, batch.num_pages, batch.block_table, dtype="fp8")
    w = oracle.synth_weights(shape, seed=0, gain_std=gain_std, cache_layers=True)
    return m, kv, batch, w, oracle.config_of(shape)


def _check_cache(m, kv, s, n, caches):
    """GPU codes/scales of sequence s (n rows) against the oracle's fp8 cache values."""
    for c in range(m.num_caches):
        for which, t in (("k", 0), ("v", 1)):
            ref_codes, ref_scale = OM.fp8_quantize(caches[c][t])
            got_codes = kv.codes(c, s, n, which).cpu().numpy().astype(np.float64)
            got_scale = kv.scales(c, s, n, which).cpu().numpy()
            got = got_codes * got_scale[..., None]
            ref = OM.fp8_dequantize(ref_codes, ref_scale)
            rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
            assert rel <= 5e-2, (c, which, rel)
            if c == 0:
                eq = got_codes == ref_codes
                assert eq.mean() >= 0.99, (which, eq.mean())
                step = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref_codes), 2.0 ** -6))) - 3)
                assert np.all(np.abs(got_codes - ref_codes)[~eq] <= 2 * step[~eq] + 1e-12), which
                amax = np.abs(ref).max(axis=-1)
                assert np.all(np.abs(got_scale - ref_scale) <= amax / 448.0 * 2.0 ** -7 + 1e-30), which


@pytest.mark.parametrize("case", ["tiny_d64", "small_d128", "bias_gqa5", "gqa8"])
def test_fp8_prefill_codes_scales_and_logits(case):
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    shape, l, g, lens = {"tiny_d64": (synth.TINY, 2, 2, [1, 17, 130, 64]),
                         "small_d128": (SMALL128, 2, 2, [300, 77, 5]),
                         "bias_gqa5": (SMALL_BIAS, 2, 1, [129, 40]),
                         "gqa8": (GQA8, 2, 2, [700, 33, 1])}[case]
    m, kv, batch, w, cfg = _setup(shape, l, g, lens)
    lg = api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv).cpu().numpy()
    assert m.status() == 0
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(len(lens))]
    with OM.kv_cache_fp8():
        caches, refs = OM.swiftkv_prefill(cfg, w, seq, l, g)
    for s in range(len(lens)):
        assert float(np.abs(lg[s] - refs[s]).max()) <= LOGIT_ABS_TOL, s
        _check_cache(m, kv, s, lens[s], caches[s])


def test_fp8_untouched_rows_stay_zero():
    """Bookkeeping: codes and scales are written at the prompt tokens' slots only."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    lens = [33, 70]
    m, kv, batch, _, _ = _setup(SMALL128, 3, 1, lens, spare_pages=3)
    api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv)
    torch.cuda.synchronize()
    used = torch.zeros(kv.num_pages * 16, dtype=torch.bool)
    for s, n in enumerate(lens):
        for p in range(n):
            used[int(batch.block_table[s][p // 16]) * 16 + p % 16] = True
    for sc in (kv.k_scale, kv.v_scale):
        rows = sc.abs().sum(dim=2).permute(1, 2, 0).reshape(-1, sc.shape[0]).cpu()   # [page*16+row][cache]
        assert (rows[~used] == 0).all() and (rows[used] > 0).all()
    for pool in (kv.k, kv.v):
        rows = pool.float().abs().sum(dim=(2, 4)).permute(1, 2, 0).reshape(-1, pool.shape[0]).cpu()
        assert (rows[~used] == 0).all()


def test_fp8_decode_steps():
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    lens = [64, 200, 9]
    l, g = 2, 2
    m, kv, batch, w, cfg = _setup(SMALL128, l, g, lens, reserve=4)
    lg = api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(3)]
    with OM.kv_cache_fp8():
        caches, refs = OM.swiftkv_prefill(cfg, w, seq, l, g)
    cur = list(lens)
    for step in range(3):
        toks = [OM.greedy(r) for r in refs]
        lg, _ = api.decode_step(m, torch.tensor(toks, dtype=torch.int32, device="cuda"), cur, kv)
        lg = lg.cpu().numpy()
        with OM.kv_cache_fp8():
            out = [OM.swiftkv_decode_step(cfg, w, caches[s], toks[s], l, g) for s in range(3)]
        caches, refs = [o[0] for o in out], [o[1] for o in out]
        cur = [x + 1 for x in cur]
        for s in range(3):
            assert float(np.abs(lg[s] - refs[s]).max()) <= LOGIT_ABS_TOL, (step, s)
    for s in range(3):
        _check_cache(m, kv, s, cur[s], caches[s])
    assert m.status() == 0


def test_fp8_chunked_forward_and_mixed_batch():
    """Prompt chunks after cached prefixes (the bf16 expansion of cached pages for the
    prompt tiles) mixed with a decode token, against the oracle's serving forward."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    l, g = 2, 2
    lens = [300, 150, 40]
    m, kv, batch, w, cfg = _setup(SMALL128, l, g, lens, reserve=2)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(3)]
    plan = [[(0, 0, 100), (1, 0, 150), (2, 0, 40)],
            [(0, 100, 230), (2, 40, None)],
            [(0, 230, 300)]]
    ref = [None, None, None]
    nxt = None
    with OM.kv_cache_fp8():
        for call in plan:
            chunks, toks = [], []
            for s, a, b in call:
                t = seq[s][a:b] if b is not None else np.array([nxt], np.int32)
                chunks.append((s, a, t))
            tt = np.concatenate([np.asarray(t, np.int32) for _, _, t in chunks])
            cu = np.concatenate([[0], np.cumsum([len(t) for _, _, t in chunks])]).astype(np.int32)
            lg = api.forward(m, torch.as_tensor(tt, device="cuda"), cu, [a for _, a, _ in chunks],
                             kv.view([s for s, _, _ in chunks])).cpu().numpy()
            for i, (s, a, t) in enumerate(chunks):
                ref[s], lr = OM.swiftkv_forward_one(cfg, w, ref[s], t, l, g)
                assert float(np.abs(lg[i] - lr).max()) <= LOGIT_ABS_TOL, (s, a)
                if s == 2 and nxt is None:
                    nxt = OM.greedy(lr)
    assert m.status() == 0
    for s, n in ((0, 300), (1, 150), (2, 41)):
        _check_cache(m, kv, s, n, ref[s])


def test_fp8_cache_is_half_the_bytes():
    from swiftkv_prefill_skipping_gb300 import api
    m = api.load_synthetic(synth.TINY, 2, 1)
    bt = np.arange(8, dtype=np.int32)[None]
    a = api.KVCache(m, 8, bt)
    b = api.KVCache(m, 8, bt, dtype="fp8")
    assert b.k.numel() * b.k.element_size() * 2 == a.k.numel() * a.k.element_size()
    assert b.k_scale.shape == (m.num_caches, 8, synth.TINY.n_kv, 16)
