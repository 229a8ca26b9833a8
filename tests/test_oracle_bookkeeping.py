"""Pins for the oracle's bookkeeping and FLOP/memory accounting: brute force,
invariants, and the pages' printed Table 1 and AcrossKV memory figures."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import bookkeeping as B
from oracle import flops as FL
from oracle import model as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_plan_positions_slots_last():
    b = synth.prompt_batch(1000, 6, 1, 70, page_size=16, spare_pages=5)
    pos, slot, last = B.plan(b.cu_seqlens, b.block_table, 16)
    # positions restart at zero in every prompt
    expect_pos = np.concatenate([np.arange(n) for n in b.lens])
    assert np.array_equal(pos, expect_pos)
    # slots are distinct and land inside each sequence's own pages
    assert len(np.unique(slot)) == len(slot)
    for s in range(len(b.lens)):
        own = set(int(p) for p in b.block_table[s] if p >= 0)
        for t in range(b.cu_seqlens[s], b.cu_seqlens[s + 1]):
            assert slot[t] // 16 in own
            assert slot[t] % 16 == pos[t] % 16
    assert np.array_equal(last, b.cu_seqlens[1:] - 1)


def test_page_scatter_gather_roundtrip():
    b = synth.prompt_batch(100, 3, 5, 40, page_size=16)
    pool = np.zeros((b.num_pages, 2, 16, 8))
    rng = np.random.default_rng(0)
    seqs = [rng.standard_normal((n, 2, 8)) for n in b.lens]
    for s, kv in enumerate(seqs):
        B.scatter_to_pages(kv, b.block_table[s], pool)
    for s, kv in enumerate(seqs):
        assert np.array_equal(B.gather_from_pages(pool, b.block_table[s], len(kv)), kv)


def test_cache_map_brute_force():
    for L, l, g in [(32, 16, 1), (32, 16, 2), (32, 24, 2), (48, 24, 4), (4, 2, 1), (32, 32, 1)]:
        C = M.num_caches(L, l, g)
        groups = [list(range(l + i * g, l + (i + 1) * g)) for i in range((L - l) // g)]
        for j in range(L):
            c = M.cache_of_layer(j, l, g)
            if j < l:
                assert c == j
            else:
                gi = [i for i, grp in enumerate(groups) if j in grp][0]
                assert c == l + gi and M.representative(c, l, g) == groups[gi][0]
        assert C == l + len(groups)


def test_table1_flops_reproduced():
    ref = json.load(open(os.path.join(GOLDEN, "table1_llama70b_gflops.json")))
    m = ref["model"]
    base_attn = None
    for row in ref["rows"]:
        got = FL.per_token_gflops(m["L"], m["d"], m["n_q"], m["n_kv"], m["d_h"], m["ffn"],
                                  m["vocab"], row["l"], row["g"])
        # printed to two significant digits
        for k in ("kv", "qo", "mlp", "vocab"):
            assert abs(got[k] - row[k]) <= max(0.1, 0.03 * row[k]), (row["name"], k, got[k])
        if base_attn is None:
            base_attn = row["attention"]
        # attention scales with the number of full layers (its context is not stated)
        assert abs(base_attn * row["l"] / m["L"] - row["attention"]) <= 0.5
        total = sum(got[k] for k in ("kv", "qo", "mlp", "vocab")) + row["attention"]
        assert abs(total - row["total"]) <= 1.0, (row["name"], total)


def test_acrosskv_memory_reduction_exact():
    ref = json.load(open(os.path.join(GOLDEN, "acrosskv_memory_llama8b.json")))
    for row in ref["rows"]:
        assert FL.kv_cache_layers(ref["L"], ref["l"], row["g"]) == row["cache_layers"]
        assert FL.kv_reduction(ref["L"], ref["l"], row["g"]) * 100 == row["reduction_pct"]
        assert M.num_caches(ref["L"], ref["l"], row["g"]) == row["cache_layers"]
    # bytes: 8B, 1000 tokens, no AcrossKV: 32 * 2 * 128 * 8 * 1000 * 2
    assert FL.kv_bytes(32, 32, 1, 8, 128, 1000) == 32 * 2 * 128 * 8 * 1000 * 2
