"""Small hand-built decode cases shared by the CPU pin tests and the GPU parity tests.

Only layout of inputs happens here (which physical blocks a sequence owns, random values from
the shared generator); nothing here computes slots, cache writes or attention.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from paged_kv_cache_block_gb300 import workloads as W


@dataclass
class Case:
    lengths: np.ndarray        # int32 [B]
    block_table: np.ndarray    # int32 [B, width]
    first_block: np.ndarray    # int64 [B]: contiguous layout only, first physical block
    num_blocks: int
    block_size: int
    q_len: int
    q: np.ndarray              # uint16 [B*q_len, Hq, D]
    k_cache: np.ndarray        # uint16 [NB, bs, Hkv, D] (16-bit caches)
    v_cache: np.ndarray
    dtype: str


def contiguous_case(lengths: Sequence[int], num_q_heads: int, num_kv_heads: int, head_dim: int,
                    block_size: int, q_len: int = 1, dtype: str = "f16", seed: int = 7,
                    spare_blocks: int = 2, table_pad: int = 1) -> Case:
    """Sequences own consecutive physical blocks in batch order (an identity-like table), so
    sequence b's keys are rows first_block[b]*bs .. +L of the flat [NB*bs, Hkv, D] view."""
    L = np.asarray(lengths, np.int64)
    need = -(-L // block_size)
    first = np.concatenate([[spare_blocks], spare_blocks + np.cumsum(need)[:-1]]).astype(np.int64)
    NB = int(spare_blocks + need.sum() + spare_blocks)
    width = int(need.max()) + table_pad
    table = np.full((len(L), width), -1, np.int32)
    for b in range(len(L)):
        table[b, :need[b]] = np.arange(first[b], first[b] + need[b])
    shape = (NB, block_size, num_kv_heads, head_dim)
    kc = W.normal_bits(seed, 1, shape, dtype)
    vc = W.normal_bits(seed, 2, shape, dtype)
    q = W.normal_bits(seed, 3, (len(L) * q_len, num_q_heads, head_dim), dtype)
    return Case(L.astype(np.int32), table, first, NB, block_size, q_len, q, kc, vc, dtype)


def relabel_blocks(case: Case, perm: np.ndarray) -> Case:
    """Move physical block p to perm[p] and rewrite the table to match."""
    kc = np.empty_like(case.k_cache)
    vc = np.empty_like(case.v_cache)
    kc[perm] = case.k_cache
    vc[perm] = case.v_cache
    table = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1).astype(np.int32)
    return Case(case.lengths, table, case.first_block, case.num_blocks, case.block_size,
                case.q_len, case.q, kc, vc, case.dtype)
