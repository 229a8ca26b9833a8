"""Serving forward (prompt chunks after a cached prefix, decode tokens, both in one
batch) on the GPU against the oracle's swiftkv_forward_one. Tolerances as in the other
parity tests: KV 1e-2 relative (per cache and K/V tensor, L2), logits 5e-2 max-abs."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import GQA8, KV_REL_TOL, LOGIT_ABS_TOL, MEDIUM, SMALL128, rel_l2
from oracle import model as OM

pytestmark = pytest.mark.gpu


def _setup(shape, l, g, lens, attn_impl=0, reserve=0, gain_std=0.1):
    from swiftkv_prefill_skipping_gb300 import api, binding
    batch = synth.prompt_batch(shape.vocab, len(lens), 0, 0, lens=lens, reserve_tokens=reserve, spare_pages=2)
    m = api.load_synthetic(shape, l, g, seed=0, gain_std=gain_std)
    binding.check(binding.lib().swiftkv_set_attention_impl(m.handle, attn_impl))
    kv = api.KVCache(m, batch.num_pages, batch.block_table)
    w = oracle.synth_weights(shape, seed=0, gain_std=gain_std, cache_layers=True)
    return m, kv, batch, w, oracle.config_of(shape)


def _call(m, kv, chunks):
    """One swiftkv_forward over chunks [(seq, ctx, token ids)]; returns [P, V] logits."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    toks = np.concatenate([np.asarray(t, np.int32) for _, _, t in chunks])
    cu = np.concatenate([[0], np.cumsum([len(t) for _, _, t in chunks])]).astype(np.int32)
    lg = api.forward(m, torch.as_tensor(toks, device="cuda"), cu, [c for _, c, _ in chunks],
                     kv.view([s for s, _, _ in chunks]))
    torch.cuda.synchronize()
    return lg.cpu().numpy()


def _check_kv(m, kv, s, n, caches):
    for c in range(m.num_caches):
        for which, t in (("k", 0), ("v", 1)):
            got = kv.gather(c, s, n, which).float().cpu().numpy()
            err = rel_l2(got, caches[c][t])
            assert err <= KV_REL_TOL, (s, c, which, err)


@pytest.mark.parametrize("case", ["d128_tc", "d128_mma", "d64"])
def test_chunked_prefill_matches_oracle_chunks_and_whole_prompt(case):
    """Prompts fed in chunks of ragged sizes (one token, below and above one attention
    tile, crossing page and tile boundaries), several sequences per call."""
    shape, impl = {"d128_tc": (SMALL128, 0), "d128_mma": (SMALL128, 1), "d64": (synth.TINY, 1)}[case]
    l, g = 2, 2 if shape.L % 2 == 0 else 1
    lens = [300, 77, 5]
    m, kv, batch, w, cfg = _setup(shape, l, g, lens, attn_impl=impl)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(3)]
    plan = [[(0, 0, 130), (1, 0, 1), (2, 0, 5)],
            [(1, 1, 76), (0, 130, 131)],
            [(0, 131, 300), (1, 76, 77)]]
    ref = [None, None, None]
    for call in plan:
        lg = _call(m, kv, [(s, a, seq[s][a:b]) for s, a, b in call])
        for i, (s, a, b) in enumerate(call):
            ref[s], lg_ref = OM.swiftkv_forward_one(cfg, w, ref[s], seq[s][a:b], l, g)
            err = float(np.abs(lg[i] - lg_ref).max())
            assert err <= LOGIT_ABS_TOL, (call, s, err)
    assert m.status() == 0
    whole, whole_lg = OM.swiftkv_prefill(cfg, w, seq, l, g)
    for s in range(3):
        _check_kv(m, kv, s, lens[s], ref[s])
        _check_kv(m, kv, s, lens[s], whole[s])


def test_mixed_batch_prefill_chunk_and_decode():
    """One call holding a decode token, a fresh prompt and a chunk after a cached prefix,
    with the sequences in a different order from the block table's."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    l, g = 3, 1
    lens = [100, 150, 154]
    m, kv, batch, w, cfg = _setup(SMALL128, l, g, lens, reserve=4)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(3)]
    # sequence 0 fully prefilled, sequence 2's first 64 tokens prefilled
    pre = np.concatenate([seq[0], seq[2][:64]])
    api.prefill(m, torch.as_tensor(pre, device="cuda"), [0, 100, 164], kv.view([0, 2]))
    c0, lg0 = OM.swiftkv_prefill_one(cfg, w, seq[0], l, g)
    c2, _ = OM.swiftkv_prefill_one(cfg, w, seq[2][:64], l, g)
    nxt = OM.greedy(lg0)
    lg = _call(m, kv, [(2, 64, seq[2][64:]), (0, 100, [nxt]), (1, 0, seq[1])])
    assert m.status() == 0
    r2, ref2 = OM.swiftkv_forward_one(cfg, w, c2, seq[2][64:], l, g)
    r0, ref0 = OM.swiftkv_decode_step(cfg, w, c0, nxt, l, g)
    r1, ref1 = OM.swiftkv_prefill_one(cfg, w, seq[1], l, g)
    for got, want in ((lg[0], ref2), (lg[1], ref0), (lg[2], ref1)):
        assert float(np.abs(got - want).max()) <= LOGIT_ABS_TOL
    _check_kv(m, kv, 0, 101, r0)
    _check_kv(m, kv, 1, 150, r1)
    _check_kv(m, kv, 2, 154, r2)


def test_forward_without_prefix_is_prefill_bit_exact():
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    lens = [129, 40, 256]
    m, kv, batch, _, _ = _setup(SMALL128, 2, 2, lens)
    tok = torch.as_tensor(batch.tokens, device="cuda")
    a = api.prefill(m, tok, batch.cu_seqlens, kv).cpu()
    ka, va = kv.k.clone(), kv.v.clone()
    kv.k.zero_()
    kv.v.zero_()
    b = api.forward(m, tok, batch.cu_seqlens, None, kv).cpu()
    assert torch.equal(a, b) and torch.equal(ka, kv.k) and torch.equal(va, kv.v)
    kv.k.zero_()
    kv.v.zero_()
    c = api.forward(m, tok, batch.cu_seqlens, [0, 0, 0], kv).cpu()
    assert torch.equal(a, c) and torch.equal(ka, kv.k) and torch.equal(va, kv.v)


def test_decode_tokens_through_forward_match_decode_step():
    """A batch of one-token chunks is a decode step: the same logits and new K/V rows
    within the tolerances (the two entries use different attention kernels)."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    lens = [33, 200, 64, 1]
    m, kv, batch, w, cfg = _setup(SMALL128, 2, 1, lens, reserve=2)
    tok = torch.as_tensor(batch.tokens, device="cuda")
    lg = api.prefill(m, tok, batch.cu_seqlens, kv)
    nxt = torch.argmax(lg, dim=1).to(torch.int32)
    k0, v0 = kv.k.clone(), kv.v.clone()
    a, _ = api.decode_step(m, nxt, lens, kv)
    a = a.cpu().numpy()
    kd, vd = kv.k.clone(), kv.v.clone()
    kv.k.copy_(k0)
    kv.v.copy_(v0)
    b = api.forward(m, nxt, list(range(len(lens) + 1)), lens, kv).cpu().numpy()
    assert float(np.abs(a - b).max()) <= LOGIT_ABS_TOL
    for s, n in enumerate(lens):   # the one row each call wrote: position n of sequence s
        page, row = int(batch.block_table[s][n // 16]), n % 16
        for pool, ref in ((kv.k, kd), (kv.v, vd)):
            for c in range(m.num_caches):
                got = pool[c, page, :, row, :].float().cpu().numpy()
                assert rel_l2(got, ref[c, page, :, row, :].float().cpu().numpy()) <= KV_REL_TOL, (s, c)


def test_forward_host_errors():
    import torch
    from swiftkv_prefill_skipping_gb300 import api, binding
    m, kv, batch, _, _ = _setup(synth.TINY, 2, 1, [20, 30])
    tok = torch.as_tensor(batch.tokens, device="cuda")
    with pytest.raises(binding.SwiftKVError) as e:
        api.forward(m, tok, batch.cu_seqlens, [0, -1], kv)
    assert e.value.code == -4
    cap = batch.block_table.shape[1] * 16
    with pytest.raises(binding.SwiftKVError) as e:
        api.forward(m, tok, batch.cu_seqlens, [cap - 19, 0], kv)   # 20 tokens after cap - 19: one past the table
    assert e.value.code == -5
    with pytest.raises(ValueError):
        api.forward(m, tok, batch.cu_seqlens, [0], kv)
    assert m.status() == 0


def test_wide_skinny_gemms_prefill_tail_and_decode():
    """Tail and decode GEMMs wide enough for the TMA-fed skinny kernel, with every epilogue
    (Q/K/V + RoPE + cache write, skipped-layer KV, SwiGLU, residual, LM head)."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    l, g = 1, 1
    lens = [40, 57, 9]
    m, kv, batch, w, cfg = _setup(MEDIUM, l, g, lens, reserve=2)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(3)]
    lg = api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv).cpu().numpy()
    caches, refs = OM.swiftkv_prefill(cfg, w, seq, l, g)
    for s in range(3):
        assert float(np.abs(lg[s] - refs[s]).max()) <= LOGIT_ABS_TOL
        _check_kv(m, kv, s, lens[s], caches[s])
    toks = [OM.greedy(r) for r in refs]
    lg2, _ = api.decode_step(m, torch.tensor(toks, dtype=torch.int32, device="cuda"), lens, kv)
    lg2 = lg2.cpu().numpy()
    for s in range(3):
        c2, ref2 = OM.swiftkv_decode_step(cfg, w, caches[s], toks[s], l, g)
        assert float(np.abs(lg2[s] - ref2).max()) <= LOGIT_ABS_TOL
        _check_kv(m, kv, s, lens[s] + 1, c2)
    assert m.status() == 0


def test_gqa8_prefill_decode_and_long_tail():
    """Eight query heads per KV head (the 70B ratio): prompt tiles, a tail row with more than
    one 256-key split, one-token chunks and decode steps against the oracle."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    l, g = 2, 2
    lens = [700, 33, 1]
    m, kv, batch, w, cfg = _setup(GQA8, l, g, lens, reserve=2)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(3)]
    lg = api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv).cpu().numpy()
    caches, refs = OM.swiftkv_prefill(cfg, w, seq, l, g)
    for s in range(3):
        assert float(np.abs(lg[s] - refs[s]).max()) <= LOGIT_ABS_TOL, s
        _check_kv(m, kv, s, lens[s], caches[s])
    toks = [OM.greedy(r) for r in refs]
    lg2, _ = api.decode_step(m, torch.tensor(toks, dtype=torch.int32, device="cuda"), lens, kv)
    lg2 = lg2.cpu().numpy()
    for s in range(3):
        _, ref2 = OM.swiftkv_decode_step(cfg, w, caches[s], toks[s], l, g)
        assert float(np.abs(lg2[s] - ref2).max()) <= LOGIT_ABS_TOL, s
    assert m.status() == 0


@pytest.mark.parametrize("shape", [SMALL128, MEDIUM])
def test_rows_impl_chained_and_per_launch_agree(shape):
    """The last-token tail and decode rows after each attention: one chained cooperative
    launch per layer (default) and one launch per GEMM / RMSNorm. Both against the oracle
    (prefill logits and three greedy decode steps), and against each other."""
    import torch
    from oracle import model as OM
    from swiftkv_prefill_skipping_gb300 import api, binding
    lens = [130, 7, 260]
    l, g = 2, 1
    batch = synth.prompt_batch(shape.vocab, len(lens), 0, 0, lens=lens, reserve_tokens=4)
    w = oracle.synth_weights(shape, gain_std=0.1, cache_layers=True)
    cfg = oracle.config_of(shape)
    seq = [batch.tokens[batch.cu_seqlens[s]:batch.cu_seqlens[s + 1]] for s in range(len(lens))]
    caches, refs = OM.swiftkv_prefill(cfg, w, seq, l, g)
    out = {}
    for impl in (0, 1):
        m = api.load_synthetic(shape, l, g, gain_std=0.1)
        binding.check(binding.lib().swiftkv_set_rows_impl(m.handle, impl))
        kv = api.KVCache(m, batch.num_pages, batch.block_table)
        lg = api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv).cpu().numpy()
        steps = [lg]
        cur, cc, rr = list(lens), list(caches), list(refs)
        for s in range(len(lens)):
            assert float(np.abs(lg[s] - refs[s]).max()) <= LOGIT_ABS_TOL, (impl, "prefill", s)
        for step in range(3):
            toks = [OM.greedy(r) for r in rr]
            dl, nxt = api.decode_step(m, torch.tensor(toks, dtype=torch.int32, device="cuda"), cur, kv)
            dl = dl.cpu().numpy()
            res = [OM.swiftkv_decode_step(cfg, w, cc[s], toks[s], l, g) for s in range(len(lens))]
            cc, rr = [r[0] for r in res], [r[1] for r in res]
            cur = [x + 1 for x in cur]
            for s in range(len(lens)):
                assert float(np.abs(dl[s] - rr[s]).max()) <= LOGIT_ABS_TOL, (impl, step, s)
            steps.append(dl)
        assert m.status() == 0
        out[impl] = steps
        m.free()
    for a, b in zip(out[0], out[1]):
        assert float(np.abs(a - b).max()) <= LOGIT_ABS_TOL
    assert binding.lib().swiftkv_set_rows_impl(None, 0) == -1
