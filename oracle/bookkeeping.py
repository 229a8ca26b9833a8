"""Oracle: token/page bookkeeping of a packed, paged prefill batch (integer, exact).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Prompts are packed back to back ("varlen") and described by cu_seqlens; the
KV cache lives in fixed-size pages named by a per-sequence block table, the
PagedAttention arrangement the pages' serving integration writes into
([S] 3.4 "Inference Implementation in Production Serving Frameworks").
Positions restart at 0 in every prompt.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np


def plan(cu_seqlens: np.ndarray, block_table: np.ndarray, page_size: int = 16
         ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """positions[t], slot[t] and last[s] for packed tokens t and prompts s.

    slot = block_table[s][pos // page_size] * page_size + pos % page_size is the
    row of the token in a cache pool viewed as [num_pages * page_size] token rows;
    last[s] = cu_seqlens[s+1] - 1 is the token whose logits prefill returns."""
    cu = [int(c) for c in cu_seqlens]
    T = cu[-1]
    positions = np.zeros(T, dtype=np.int32)
    slots = np.zeros(T, dtype=np.int32)
    last = np.zeros(len(cu) - 1, dtype=np.int32)
    for s in range(len(cu) - 1):
        for t in range(cu[s], cu[s + 1]):
            p = t - cu[s]
            positions[t] = p
            slots[t] = int(block_table[s][p // page_size]) * page_size + p % page_size
        last[s] = cu[s + 1] - 1
    return positions, slots, last


def scatter_to_pages(kv_seq: np.ndarray, block_row: np.ndarray, pool: np.ndarray,
                     page_size: int = 16) -> None:
    """Write one sequence's cache [n, n_kv, d_h] into a pool [num_pages, n_kv, page_size, d_h]."""
    for p in range(kv_seq.shape[0]):
        pool[int(block_row[p // page_size]), :, p % page_size, :] = kv_seq[p]


def gather_from_pages(pool: np.ndarray, block_row: np.ndarray, n: int,
                      page_size: int = 16) -> np.ndarray:
    """Read one sequence's first n cache rows back out of a pool."""
    out = np.empty((n, pool.shape[1], pool.shape[3]), dtype=pool.dtype)
    for p in range(n):
        out[p] = pool[int(block_row[p // page_size]), :, p % page_size, :]
    return out


def pages_needed(lens: List[int], page_size: int = 16) -> List[int]:
    return [(int(n) + page_size - 1) // page_size for n in lens]
