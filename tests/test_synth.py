"""The shared seeded input generator: published test vectors and distribution checks."""
import json
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_reference_outputs():
    ref = json.load(open(os.path.join(GOLDEN, "splitmix64_seed0.json")))["outputs_hex"]
    got = ["%016x" % synth.splitmix64_at(0, i) for i in range(len(ref))]
    assert got == ref


def test_normal_moments_and_offsets():
    w = synth.bf16_bits_to_f32(synth.normal_bf16(0, 77, (512, 512)))
    assert abs(float(w.mean())) < 2e-4
    assert abs(float(w.std()) - 0.02) < 2e-4
    # standard normal: ~4.55% of draws beyond 2 sigma
    assert abs(float(np.mean(np.abs(w) > 0.04)) - 0.0455) < 0.003
    flat = w.ravel()
    for off, n in [(0, 5), (1, 4), (7, 3), (1000, 33)]:
        part = synth.bf16_bits_to_f32(synth.normal_bf16(0, 77, (n,), offset=off))
        assert np.array_equal(part, flat[off:off + n])


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = synth.normal_f32(3, 1, (4096,), std=3.0)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -7 * (1 + 2 ** -8)], np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), ref)
    back = synth.bf16_bits_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_uniform_int_and_permutation():
    a = synth.uniform_int(1, 11, 20000, 500, 1000)
    assert a.min() == 500 and a.max() == 1000
    assert abs(a.mean() - 750) < 3
    p = synth.permutation(2, 13, 1000)
    assert np.array_equal(np.sort(p), np.arange(1000))
    assert not np.array_equal(p, np.arange(1000))


def test_prompt_batch_block_table():
    b = synth.prompt_batch(1024, 5, 10, 40, page_size=16, reserve_tokens=3)
    assert b.cu_seqlens[-1] == len(b.tokens) == b.lens.sum()
    used = b.block_table[b.block_table >= 0]
    assert len(np.unique(used)) == len(used) == b.num_pages
    for s, n in enumerate(b.lens):
        assert (b.block_table[s] >= 0).sum() == (n + 3 + 15) // 16
    assert b.tokens.min() >= 0 and b.tokens.max() < 1024


def test_mixed_batch_layout():
    """Serving-step batch: chunks then decode tokens, prefixes and block table sized to
    ctx + n, every page used once."""
    b = synth.mixed_batch(1000, ((0, 40), (33, 17)), 5, 10, 30)
    ctx = b.extra["ctx"]
    assert list(b.lens) == [40, 17, 1, 1, 1, 1, 1]
    assert list(ctx[:2]) == [0, 33] and all(10 <= c <= 30 for c in ctx[2:])
    assert b.cu_seqlens[-1] == len(b.tokens) == 62
    assert b.extra["prefix_cu"][-1] == len(b.extra["prefix_tokens"]) == ctx.sum()
    used = []
    for s in range(7):
        need = (int(ctx[s]) + int(b.lens[s]) + 15) // 16
        row = b.block_table[s]
        assert (row[:need] >= 0).all() and (row[need:] == -1).all()
        used += list(row[:need])
    assert sorted(used) == list(range(b.num_pages))
    assert (b.tokens >= 0).all() and (b.tokens < 1000).all()


def test_serving_flops_count_cached_pairs():
    """Causal pairs of a chunk after a cached prefix: brute-force count of (query, key)
    with key <= query position; a prefix-free batch keeps the prefill count."""
    from swiftkv_prefill_skipping_gb300 import flops as FL
    lens, ctx = [5, 1, 7], [0, 9, 3]
    brute = sum(1 for n, c in zip(lens, ctx) for i in range(n) for k in range(c + n) if k <= c + i)
    assert FL._attn_pairs(lens, ctx) == brute
    assert FL._attn_pairs(lens) == sum(n * (n + 1) // 2 for n in lens)
    a = FL.prefill_flops(synth.TINY, lens, 2, 1, ctx=ctx)
    b = FL.prefill_flops(synth.TINY, lens, 2, 1)
    assert a["executed"] > b["executed"] and a["wide_kv_gemm"] == b["wide_kv_gemm"]
