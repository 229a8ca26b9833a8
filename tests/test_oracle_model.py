"""Pins for the oracle's model and its SwiftKV algorithm.

The ordinary layer is pinned to an independent composition of torch library
routines; the SwiftKV parts are pinned by the invariants the pages fix:
l = L is the ordinary model, prefill skipping returns exactly the SwiftKV
model's caches and last-token logits, a skipped layer's K/V depend only on
x_l and the representative's W_KV, AcrossKV g = 1 is plain SwiftKV,
causality, and decode from the cache equals the full forward.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import model as M

TINY = synth.TINY
CFG = oracle.config_of(TINY)
TOL = dict(rtol=1e-11, atol=1e-12)   # different BLAS row groupings only


@pytest.fixture(scope="module")
def w_gain():
    """Tiny model with non-unit RMSNorm gains so a dropped gain shows."""
    return oracle.synth_weights(TINY, gain_std=0.1)


@pytest.fixture(scope="module")
def tokens():
    return synth.uniform_int(synth.SEED_INPUTS, 12, 48, 0, TINY.vocab - 1)


def _eq_kv(a, b):
    return np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------------ ordinary model vs torch

def test_ordinary_forward_matches_torch_composition(monkeypatch, w_gain, tokens):
    """With bf16 rounding switched off, the oracle's ordinary forward equals a
    composition of torch.nn.functional routines (rms_norm, linear,
    scaled_dot_product_attention with GQA, silu) and a complex-number RoPE."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    monkeypatch.setattr(M, "bf16", lambda x: np.asarray(x, dtype=np.float64))
    cfg = M.Config(**{**CFG.__dict__, "qkv_bias": False})
    caches, logits = M.ordinary_forward(cfg, w_gain, tokens)

    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    n, dh = len(tokens), cfg.d_h
    pos = torch.arange(n, dtype=torch.float64)
    freq = cfg.rope_theta ** (-torch.arange(dh // 2, dtype=torch.float64) * 2 / dh)
    rot = torch.polar(torch.ones(n, dh // 2, dtype=torch.float64), pos[:, None] * freq[None])

    def rope_c(x):  # x [n, h, dh]
        z = torch.complex(x[..., : dh // 2], x[..., dh // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    x = T(w_gain.embed(tokens))
    for j in range(cfg.L):
        lw = w_gain.layer(j)
        u = F.rms_norm(x, (cfg.d,), T(lw.gamma_attn), eps=cfg.rms_eps)
        q = rope_c(F.linear(u, T(lw.wq)).view(n, cfg.n_q, dh))
        k = rope_c(F.linear(u, T(lw.wk)).view(n, cfg.n_kv, dh))
        v = F.linear(u, T(lw.wv)).view(n, cfg.n_kv, dh)
        np.testing.assert_allclose(caches[j][0], k.numpy(), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(caches[j][1], v.numpy(), rtol=1e-10, atol=1e-11)
        a = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                           v.transpose(0, 1)[None], is_causal=True, enable_gqa=True)
        x = x + F.linear(a[0].transpose(0, 1).reshape(n, -1), T(lw.wo))
        u = F.rms_norm(x, (cfg.d,), T(lw.gamma_mlp), eps=cfg.rms_eps)
        x = x + F.linear(F.silu(F.linear(u, T(lw.wg))) * F.linear(u, T(lw.wu)), T(lw.wd))
    ref = F.linear(F.rms_norm(x, (cfg.d,), T(w_gain.gamma_final), eps=cfg.rms_eps), T(w_gain.lm_head))
    np.testing.assert_allclose(logits, ref.numpy(), rtol=1e-9, atol=1e-10)


def test_ordinary_forward_is_causal(w_gain, tokens):
    c_full, lg_full = M.ordinary_forward(CFG, w_gain, tokens)
    c_pre, lg_pre = M.ordinary_forward(CFG, w_gain, tokens[:20])
    np.testing.assert_allclose(lg_pre, lg_full[:20], **TOL)
    for j in range(CFG.L):
        np.testing.assert_allclose(c_pre[j][0], c_full[j][0][:20], **TOL)


# ------------------------------------------------------------------ SwiftKV invariants

def test_l_equals_L_is_the_ordinary_model_bit_for_bit(w_gain, tokens):
    c0, lg0 = M.ordinary_forward(CFG, w_gain, tokens)
    c1, lg1 = M.swiftkv_full_forward(CFG, w_gain, tokens, l=CFG.L)
    assert np.array_equal(lg0, lg1)
    assert all(_eq_kv(a, b) for a, b in zip(c0, c1))
    c2, lg2 = M.swiftkv_prefill_one(CFG, w_gain, tokens, l=CFG.L)
    assert all(_eq_kv(a, b) for a, b in zip(c0, c2))
    np.testing.assert_allclose(lg2, lg0[-1], **TOL)


@pytest.mark.parametrize("l", [1, 2, 3])
def test_layers_below_l_match_ordinary_kv_bit_exact(w_gain, tokens, l):
    c0, _ = M.ordinary_forward(CFG, w_gain, tokens)
    c1, _ = M.swiftkv_prefill_one(CFG, w_gain, tokens, l=l)
    for j in range(l):
        assert _eq_kv(c0[j], c1[j])
    # the first skipped layer's input is x_l itself, so its KV is the ordinary one too
    assert _eq_kv(c0[l], c1[l])
    # deeper skipped layers differ (they project x_l, not their own x_j)
    for j in range(l + 1, CFG.L):
        assert not np.allclose(c0[j][0], c1[j][0])


@pytest.mark.parametrize("l,g", [(2, 1), (1, 3), (2, 2), (1, 1)])
def test_skipping_equals_full_swiftkv_model(w_gain, tokens, l, g):
    cf, lgf = M.swiftkv_full_forward(CFG, w_gain, tokens, l=l, g=g)
    cp, lgp = M.swiftkv_prefill_one(CFG, w_gain, tokens, l=l, g=g)
    assert len(cf) == len(cp) == l + (CFG.L - l) // g
    for a, b in zip(cf, cp):
        assert _eq_kv(a, b)
    np.testing.assert_allclose(lgp, lgf[-1], **TOL)


def test_skipped_caches_depend_only_on_x_l_and_rep_kv_weights(tokens):
    l = 2
    base = oracle.synth_weights(TINY, gain_std=0.1)
    c0, lg0 = M.swiftkv_prefill_one(CFG, base, tokens, l=l)
    # perturb Q/O/MLP of a skipped layer: caches identical, last logits move
    lw = base.layer(3)
    pert = {(3, "wq"): lw.wq * 1.5, (3, "wo"): -lw.wo, (3, "wd"): lw.wd * 0.5}
    c1, lg1 = M.swiftkv_prefill_one(CFG, oracle.synth_weights(TINY, gain_std=0.1, overrides=pert),
                                    tokens, l=l)
    assert all(_eq_kv(a, b) for a, b in zip(c0, c1))
    assert np.abs(lg1 - lg0).max() > 1e-3
    # perturb W_K of skipped layer 3 (g = 1): only cache 3 changes
    c2, _ = M.swiftkv_prefill_one(
        CFG, oracle.synth_weights(TINY, gain_std=0.1, overrides={(3, "wk"): lw.wk[::-1].copy()}),
        tokens, l=l)
    assert [_eq_kv(a, b) for a, b in zip(c0, c2)] == [True, True, True, False]
    # the skipped layer's own input gain acts on x_l
    c3, _ = M.swiftkv_prefill_one(
        CFG, oracle.synth_weights(TINY, gain_std=0.1, overrides={(2, "gamma_attn"): lw.gamma_attn * 2}),
        tokens, l=l)
    assert [_eq_kv(a, b) for a, b in zip(c0, c3)] == [True, True, False, True]


def test_acrosskv_groups_share_the_representatives_cache(tokens):
    l, g = 2, 2     # skipped layers 2, 3 form one group whose representative is layer 2
    base = oracle.synth_weights(TINY, gain_std=0.1)
    c0, lg0 = M.swiftkv_prefill_one(CFG, base, tokens, l=l, g=g)
    assert len(c0) == 3
    # g = 1 caches: the group cache equals the representative's own SwiftKV cache
    c1, _ = M.swiftkv_prefill_one(CFG, base, tokens, l=l, g=1)
    assert _eq_kv(c0[2], c1[2])
    # the non-representative's K/V weights are unused
    lw3 = base.layer(3)
    c2, lg2 = M.swiftkv_prefill_one(
        CFG, oracle.synth_weights(TINY, gain_std=0.1, overrides={(3, "wk"): -lw3.wk, (3, "wv"): -lw3.wv}),
        tokens, l=l, g=g)
    assert all(_eq_kv(a, b) for a, b in zip(c0, c2))
    assert np.array_equal(lg0, lg2)
    # layer 3 attends to the group cache: equals the full model where layer 3 reads cache 2
    cf, lgf = M.swiftkv_full_forward(CFG, base, tokens, l=l, g=g)
    np.testing.assert_allclose(lgf[-1], lg0, **TOL)


def test_acrosskv_group_size_one_is_plain_swiftkv(w_gain, tokens):
    for l in (1, 2, 3):
        ca, la = M.swiftkv_prefill_one(CFG, w_gain, tokens, l=l, g=1)
        assert len(ca) == CFG.L
        assert [M.cache_of_layer(j, l, 1) for j in range(CFG.L)] == list(range(CFG.L))
        assert [M.representative(c, l, 1) for c in range(CFG.L)] == list(range(CFG.L))


def test_swiftkv_prefill_is_causal_and_packing_independent(w_gain, tokens):
    l = 2
    c_full, _ = M.swiftkv_prefill_one(CFG, w_gain, tokens, l=l)
    c_pre, lg_pre = M.swiftkv_prefill_one(CFG, w_gain, tokens[:17], l=l)
    for a, b in zip(c_pre, c_full):
        np.testing.assert_allclose(a[0], b[0][:17], **TOL)
        np.testing.assert_allclose(a[1], b[1][:17], **TOL)
    # a batch is its prompts, one by one
    cb, lgb = M.swiftkv_prefill(CFG, w_gain, [tokens[:17], tokens], l=l)
    np.testing.assert_array_equal(lgb[0], lg_pre)
    assert all(_eq_kv(a, b) for a, b in zip(cb[1], c_full))


def test_decode_from_cache_equals_full_swiftkv_forward(w_gain, tokens):
    l, g = 2, 2
    n0 = 30
    seq = list(tokens[:n0])
    caches, lg = M.swiftkv_prefill_one(CFG, w_gain, seq, l=l, g=g)
    for _ in range(5):
        nxt = M.greedy(lg)
        seq.append(nxt)
        caches, lg = M.swiftkv_decode_step(CFG, w_gain, caches, nxt, l=l, g=g)
        cf, lgf = M.swiftkv_full_forward(CFG, w_gain, seq, l=l, g=g)
        np.testing.assert_allclose(lg, lgf[-1], **TOL)
        for a, b in zip(caches, cf):
            np.testing.assert_allclose(a[0], b[0], **TOL)
            np.testing.assert_allclose(a[1], b[1], **TOL)
    # greedy continuation agrees with greedy on the full model's logits
    assert [M.greedy(r) for r in lgf[n0 - 1:-1]] == seq[n0:]


def test_invalid_l_and_g_are_rejected(w_gain, tokens):
    with pytest.raises(ValueError):
        M.swiftkv_prefill_one(CFG, w_gain, tokens, l=0)
    with pytest.raises(ValueError):
        M.swiftkv_prefill_one(CFG, w_gain, tokens, l=5)
    with pytest.raises(ValueError):
        M.swiftkv_prefill_one(CFG, w_gain, tokens, l=1, g=2)   # 3 skipped layers, groups of 2
    with pytest.raises(ValueError):
        M.swiftkv_prefill_one(CFG, w_gain, [], l=2)


def test_qkv_bias_is_added_before_rope():
    shape = synth.ModelShape("tiny-bias", L=2, d=64, n_q=2, n_kv=1, d_h=32, ffn=96, vocab=128,
                             rope_theta=10000.0, qkv_bias=True)
    cfg = oracle.config_of(shape)
    w = oracle.synth_weights(shape)
    toks = np.array([5, 9, 100, 3])
    caches, _ = M.swiftkv_prefill_one(cfg, w, toks, l=1)
    lw = w.layer(0)
    # K at position 0 is unrotated: it must equal bf16(W_k u + b_k)
    u = M.bf16(M.rms_norm(w.embed(toks), lw.gamma_attn, cfg.rms_eps))
    kb = (u @ lw.wk.astype(np.float64).T + lw.bk).reshape(len(toks), 1, 32)
    np.testing.assert_array_equal(caches[0][0][0], M.bf16(kb[0]))
    # at later positions the bias is rotated with the projection, not added after RoPE
    pos = np.arange(len(toks))
    np.testing.assert_array_equal(caches[0][0], M.bf16(M.rope(kb, pos, cfg.rope_theta)))
    kb_after = M.rope(kb - lw.bk.reshape(1, 1, 32), pos, cfg.rope_theta) + lw.bk.reshape(1, 1, 32)
    assert not np.allclose(caches[0][0][1:], M.bf16(kb_after[1:]))


def test_forward_chunks_equal_whole_prompt_and_decode(w_gain, tokens):
    """The serving forward: a prompt fed as chunks gives the caches and last logits of the
    whole prompt; a one-token chunk is a decode step; a chunk with no prefix is prefill."""
    l, g = 2, 2
    c_all, lg_all = M.swiftkv_prefill_one(CFG, w_gain, tokens, l, g)
    c0, lg0 = M.swiftkv_forward_one(CFG, w_gain, None, tokens, l, g)
    for a, b in zip(c0, c_all):
        np.testing.assert_allclose(a[0], b[0], **TOL)
    np.testing.assert_allclose(lg0, lg_all, **TOL)
    cc, lgc = None, None
    for a, b in [(0, 5), (5, 6), (6, 31), (31, len(tokens))]:
        cc, lgc = M.swiftkv_forward_one(CFG, w_gain, cc, tokens[a:b], l, g)
    for a, b in zip(cc, c_all):
        np.testing.assert_allclose(a[0], b[0], **TOL)
        np.testing.assert_allclose(a[1], b[1], **TOL)
    np.testing.assert_allclose(lgc, lg_all, **TOL)
    nxt = M.greedy(lg_all)
    c_dec, lg_dec = M.swiftkv_decode_step(CFG, w_gain, c_all, nxt, l, g)
    c_fw, lg_fw = M.swiftkv_forward_one(CFG, w_gain, c_all, [nxt], l, g)
    np.testing.assert_allclose(lg_fw, lg_dec, **TOL)
    for a, b in zip(c_fw, c_dec):
        np.testing.assert_allclose(a[0], b[0], **TOL)
    with pytest.raises(ValueError):
        M.swiftkv_forward_one(CFG, w_gain, c_all, [], l, g)


def test_fp8_cache_mode_quantizes_every_cache_write(w_gain, tokens):
    """Under kv_cache_fp8 every cache (full layers and skipped groups) holds per-token
    code * scale values of its bf16 rows; the logits move by a small nonzero amount."""
    l, g = 2, 2
    c_bf, lg_bf = M.swiftkv_prefill_one(CFG, w_gain, tokens, l, g)
    with M.kv_cache_fp8():
        c_f8, lg_f8 = M.swiftkv_prefill_one(CFG, w_gain, tokens, l, g)
        c_dec, _ = M.swiftkv_decode_step(CFG, w_gain, c_f8, 7, l, g)
    for c in range(len(c_f8)):
        for t in range(2):
            got = c_f8[c][t]
            codes, scale = M.fp8_quantize(got)
            np.testing.assert_array_equal(M.fp8_dequantize(codes, scale), got)   # already on the grid
            assert np.abs(got - c_bf[c][t]).max() > 0
            rel = np.linalg.norm(got - c_bf[c][t]) / np.linalg.norm(c_bf[c][t])
            assert rel < 0.05, (c, t, rel)
        assert c_dec[c][0].shape[0] == len(tokens) + 1
    d = np.abs(lg_f8 - lg_bf).max()
    assert 0 < d < 0.5, d
