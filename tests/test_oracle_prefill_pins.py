"""Pins of the oracle's chunked-prefill attention (a different number of query rows per
sequence, given by query_start_loc): against PyTorch's scaled_dot_product_attention in float64
with an explicit mask on contiguous caches, and against facts any correct implementation obeys
(splitting a chunk in two, block relabelling, one query row per sequence = the decode call)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_block_gb300 import workloads as W
from tests.cases import contiguous_case, relabel_blocks


def varlen_case(lengths, counts, Hq, Hkv, D, bs, dtype, seed):
    """contiguous_case with sum(counts) query rows; sequence b's rows are its last counts[b]
    positions."""
    case = contiguous_case(lengths, Hq, Hkv, D, bs, 1, dtype, seed=seed)
    qsl = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    case.q = W.normal_bits(seed, 9, (int(qsl[-1]), Hq, D), dtype)
    return case, qsl


def sdpa_prefill(case, qsl, scale, window):
    NB, bs, H, D = case.k_cache.shape
    kf = W.bits_to_float(case.k_cache, case.dtype).astype(np.float64).reshape(NB * bs, H, D)
    vf = W.bits_to_float(case.v_cache, case.dtype).astype(np.float64).reshape(NB * bs, H, D)
    qf = W.bits_to_float(case.q, case.dtype).astype(np.float64)
    Hq = qf.shape[1]
    outs, lses = [], []
    for b, L in enumerate(case.lengths):
        n = int(qsl[b + 1] - qsl[b])
        if n == 0:
            continue
        s0 = int(case.first_block[b]) * bs
        K = torch.from_numpy(kf[s0:s0 + L]).permute(1, 0, 2)[None]
        V = torch.from_numpy(vf[s0:s0 + L]).permute(1, 0, 2)[None]
        Q = torch.from_numpy(qf[qsl[b]:qsl[b + 1]]).permute(1, 0, 2)[None]
        p = (L - n + np.arange(n))[:, None]
        j = np.arange(L)[None, :]
        allowed = j <= p
        if window > 0:
            allowed &= j > p - window
        mask = torch.from_numpy(allowed)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale, enable_gqa=(Hq != H))
        outs.append(o[0].permute(1, 0, 2).numpy())
        Kr = K.repeat_interleave(Hq // H, dim=1)
        sc = ((Q @ Kr.transpose(-1, -2)) * scale).masked_fill(~mask, float("-inf"))
        lses.append(torch.logsumexp(sc, dim=-1)[0].permute(1, 0).numpy())
    return np.concatenate(outs), np.concatenate(lses)


def run(case, qsl, scale, window=0):
    return oracle.paged_attention_varlen(case.q, case.dtype, case.k_cache, case.v_cache, case.dtype,
                                         case.block_table, case.lengths, qsl, scale, window, threads=3)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs,window", [
    ("f16", 4, 1, 16, 4, 0),
    ("bf16", 8, 2, 32, 16, 0),
    ("f16", 4, 4, 16, 8, 7),
    ("bf16", 6, 2, 16, 4, 20),
])
def test_prefill_matches_sdpa(dtype, Hq, Hkv, D, bs, window):
    # whole prompts (no context), chunks after some context, a single token, an empty chunk
    lengths, counts = [37, 50, 9, 12, 30], [37, 13, 1, 0, 30]
    case, qsl = varlen_case(lengths, counts, Hq, Hkv, D, bs, dtype, seed=Hq * 7 + bs)
    scale = 1.0 / math.sqrt(D)
    out, lse = run(case, qsl, scale, window)
    ref_out, ref_lse = sdpa_prefill(case, qsl, scale, window)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_prefill_chunk_split_in_two_gives_the_same_rows():
    """Chunked prefill: computing 40 new tokens at once or as 25 then 15 (the first call with
    the sequence 15 tokens shorter) gives every row the same result bit for bit."""
    case, qsl = varlen_case([70, 41], [40, 41], 4, 2, 16, 4, "bf16", seed=31)
    whole = run(case, qsl, 0.3, window=9)
    first = varlen_case([70 - 15, 41], [25, 41], 4, 2, 16, 4, "bf16", seed=31)[0]
    first.k_cache, first.v_cache, first.block_table = case.k_cache, case.v_cache, case.block_table
    first.q = np.concatenate([case.q[:25], case.q[40:]])
    a = run(first, np.array([0, 25, 66], np.int32), 0.3, window=9)
    second = varlen_case([70, 41], [15, 41], 4, 2, 16, 4, "bf16", seed=31)[0]
    second.k_cache, second.v_cache, second.block_table = case.k_cache, case.v_cache, case.block_table
    second.q = np.concatenate([case.q[25:40], case.q[40:]])
    b = run(second, np.array([0, 15, 56], np.int32), 0.3, window=9)
    assert np.array_equal(whole[0][:25], a[0][:25]) and np.array_equal(whole[1][:25], a[1][:25])
    assert np.array_equal(whole[0][25:40], b[0][:15]) and np.array_equal(whole[1][25:40], b[1][:15])
    assert np.array_equal(whole[0][40:], a[0][25:])


def test_prefill_one_row_per_sequence_equals_decode():
    case, qsl = varlen_case([5, 33, 18], [1, 1, 1], 8, 2, 16, 8, "f16", seed=32)
    v = run(case, qsl, 0.25, window=6)
    d = oracle.paged_attention(case.q, "f16", case.k_cache, case.v_cache, "f16", case.block_table,
                               case.lengths, 1, 0.25, 6)
    assert np.array_equal(v[0], d[0]) and np.array_equal(v[1], d[1])


def test_prefill_block_relabelling_invariance():
    case, qsl = varlen_case([29, 64], [29, 20], 4, 2, 16, 4, "f16", seed=33)
    perm = np.random.default_rng(5).permutation(case.num_blocks)
    moved = relabel_blocks(case, perm)
    a, b = run(case, qsl, 0.4), run(moved, qsl, 0.4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
