"""The pins have teeth: plant plausible mistakes in the oracle (on the CPU,
by monkeypatching) and check that the pins covering that part fail."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from oracle import model as M  # noqa: E402
import test_oracle_model as TM
import test_oracle_numerics as TN


def _fails(fn, *args, **kw):
    try:
        fn(*args, **kw)
    except AssertionError:
        return True
    return False


def test_rope_sign_error_is_caught(monkeypatch):
    good = M.rope

    def bad(x, pos, theta):
        return good(x, -np.asarray(pos), theta)
    monkeypatch.setattr(M, "rope", bad)
    assert _fails(TN.test_rope_closed_form_small)


def test_rope_wrong_pairing_is_caught(monkeypatch):
    def interleaved(x, pos, theta):   # pairs (2i, 2i+1) instead of (i, i + d/2)
        d = x.shape[-1]
        perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
        inv = np.argsort(perm)
        return M.__dict__["_rope_good"](x[..., perm], pos, theta)[..., inv]
    monkeypatch.setitem(M.__dict__, "_rope_good", M.rope)
    monkeypatch.setattr(M, "rope", interleaved)
    assert _fails(TN.test_rope_complex_form_and_invariants)


def test_gqa_head_map_error_is_caught(monkeypatch):
    good = M.causal_gqa_attention

    def bad(q, k, v, qp, kp):   # head h reads kv head h % n_kv instead of h // group
        n_q, n_kv = q.shape[1], k.shape[1]
        perm = np.array([(h % n_kv) * (n_q // n_kv) + h // n_kv for h in range(n_q)])
        return good(q[:, perm], k, v, qp, kp)[:, np.argsort(perm)]
    monkeypatch.setattr(M, "causal_gqa_attention", bad)
    assert _fails(TN.test_attention_matches_torch_sdpa_gqa)


def test_kv_from_own_input_instead_of_x_l_is_caught(monkeypatch, w_gain, tokens):
    """A 'SwiftKV' that keeps computing every layer's KV from its own input is
    just the ordinary model; the skipped-cache pins must notice."""
    def bad_prefill(cfg, w, toks, l, g=1):
        caches, logits = M.ordinary_forward(cfg, w, toks)
        return caches[: M.num_caches(cfg.L, l, g)], logits[-1]
    monkeypatch.setattr(M, "swiftkv_prefill_one", bad_prefill)
    assert _fails(TM.test_layers_below_l_match_ordinary_kv_bit_exact, w_gain, tokens, 1)


def test_wrong_representative_is_caught(monkeypatch, tokens):
    monkeypatch.setattr(M, "representative", lambda c, l, g: c if c < l else l + (c - l) * g + g - 1)
    assert _fails(TM.test_acrosskv_groups_share_the_representatives_cache, tokens)


def test_dropped_gain_is_caught(monkeypatch, w_gain, tokens):
    good = M.rms_norm
    monkeypatch.setattr(M, "rms_norm", lambda x, gamma, eps: good(x, np.ones_like(gamma), eps))
    with pytest.MonkeyPatch.context() as mp:
        assert _fails(TM.test_ordinary_forward_matches_torch_composition, mp, w_gain, tokens)


@pytest.fixture(scope="module")
def w_gain():
    import oracle
    import synth
    return oracle.synth_weights(synth.TINY, gain_std=0.1)


@pytest.fixture(scope="module")
def tokens():
    import synth
    return synth.uniform_int(synth.SEED_INPUTS, 12, 48, 0, synth.TINY.vocab - 1)


def test_fp8_scale_off_by_range_is_caught(monkeypatch):
    """Scales computed for the wrong e4m3 range (amax / 240) leave the codes off +-448."""
    good = M.fp8_quantize

    def bad(v):
        codes, scale = good(v)
        return M.e4m3(codes * 240.0 / 448.0), (scale * np.float32(448.0 / 240.0)).astype(np.float32)
    monkeypatch.setattr(M, "fp8_quantize", bad)
    assert _fails(TN.test_fp8_quantize_per_token_and_head)


def test_fp8_e4m3_with_bf16_precision_is_caught(monkeypatch):
    """Rounding codes to 8 significant bits (a bf16 'fp8') is not e4m3."""
    monkeypatch.setattr(M, "e4m3", lambda x: np.minimum(np.abs(M.bf16(x)), 448.0) * np.sign(x))
    assert _fails(TN.test_e4m3_matches_torch_float8_cast)


def test_fp8_mode_skipping_v_is_caught(monkeypatch, w_gain, tokens):
    """A cache mode that quantizes K but stores V unquantized is caught by the model pin."""
    good = M._cache_values
    calls = {"n": 0}

    def k_only(t):
        calls["n"] += 1
        return good(t) if calls["n"] % 2 == 1 else t   # K then V at every write
    monkeypatch.setattr(M, "_cache_values", k_only)
    assert _fails(TM.test_fp8_cache_mode_quantizes_every_cache_write, w_gain, tokens)
