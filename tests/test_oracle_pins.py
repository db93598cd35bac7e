"""Pins for the CPU oracle: checks against facts that do not come from the oracle itself.

* slot mapping: the worked examples the pages print (tests/golden/slot_examples.json) and a
  brute-force enumeration of each table (physical*bs + offset for every logical block);
* E4M3 codec: the format's fixed points, PyTorch's float8_e4m3fn on all 256 codes, round-trip
  and ties-to-even at every midpoint, saturation;
* cache write: read-back through a flat [slots, Hkv, D] view, untouched slots unchanged,
  PyTorch's e4m3 conversion for the quantised path;
* attention: torch scaled_dot_product_attention in float64 with explicit masks on contiguous
  caches (GQA through its own head grouping), block-id permutation invariance, GQA == MHA with
  repeated kv heads, closed forms (one key, equal keys, zero scale), window >= length equals
  full, NaN poison outside the window, speculative queries == one-token calls at shorter
  lengths, and the fp8 path against SDPA on PyTorch-dequantised caches.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_block_gb300 import workloads as W
from tests.cases import contiguous_case, relabel_blocks


# ---------------------------------------------------------------- slot mapping

def _load_slot_examples(golden_dir):
    with open(os.path.join(golden_dir, "slot_examples.json")) as f:
        return {c["id"]: c for c in json.load(f)["cases"]}


def test_slot_token7_block37(golden_dir):
    c = _load_slot_examples(golden_dir)["token7_block37"]
    slots, err = oracle.slot_mapping(c["block_table"], [0, 1], c["positions"], c["block_size"], 64)
    assert err == 0
    assert slots.tolist() == c["slots"]
    assert [s // c["block_size"] for s in slots] == [37]
    assert [s % c["block_size"] for s in slots] == c["offsets"]


def test_slot_48_tokens_three_blocks(golden_dir):
    c = _load_slot_examples(golden_dir)["48_tokens_3_blocks"]
    pos = np.arange(48)
    slots, err = oracle.slot_mapping(c["block_table"], [0, 48], pos, c["block_size"], 100)
    assert err == 0
    used = sorted({int(s) // c["block_size"] for s in slots})
    assert len(used) == c["num_logical_blocks"]
    expect = np.concatenate([np.arange(lo, hi) for lo, hi in c["slot_ranges"]])
    assert np.array_equal(slots, expect)


def test_slot_worker_rows(golden_dir):
    c = _load_slot_examples(golden_dir)["worker_rows"]
    slots, err = oracle.slot_mapping(c["block_table"], c["query_start_loc"], c["positions"],
                                     c["block_size"], 100)
    assert err == 0
    assert slots.tolist() == c["slots"]


def test_slot_block_of_4_spill(golden_dir):
    c = _load_slot_examples(golden_dir)["block_of_4_spill"]
    slots, err = oracle.slot_mapping(c["block_table"], [0, 5], c["positions"], c["block_size"], 8)
    assert err == 0
    assert slots.tolist() == c["slots"]
    # the fifth token lands in a block that is not adjacent to the first one
    assert abs(slots[4] // 4 - slots[0] // 4) > 1


@pytest.mark.parametrize("bs", [4, 8, 16, 32])
def test_slot_bruteforce_enumeration(bs):
    rng = np.random.default_rng(bs)
    B, width, NB = 5, 7, 64
    table = rng.permutation(NB)[:B * width].reshape(B, width).astype(np.int32)
    # dense map built the other way round: every (logical block, offset) of every row
    dense = {}
    for r in range(B):
        for lb in range(width):
            for off in range(bs):
                dense[(r, lb * bs + off)] = int(table[r, lb]) * bs + off
    counts = rng.integers(0, 6, size=B)
    qsl = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(qsl[-1]) + 3                        # three trailing tokens belong to no request
    pos = rng.integers(-2, width * bs, size=T).astype(np.int32)
    slots, err = oracle.slot_mapping(table, qsl, pos, bs, NB)
    assert err == 0
    for t in range(T):
        rows = [r for r in range(B) if qsl[r] <= t < qsl[r + 1]]
        if not rows or pos[t] < 0:
            assert slots[t] == -1
        else:
            assert slots[t] == dense[(rows[0], int(pos[t]))]


def test_slot_error_bits():
    table = np.array([[3, -1, 99]], np.int32)
    slots, err = oracle.slot_mapping(table, [0, 4], [0, 5, 9, 12], 4, 10)
    # pos 5 -> logical 1 -> id -1 (bad); pos 9 -> id 99 >= NB (bad); pos 12 -> past the table
    assert slots.tolist() == [12, -1, -1, -1]
    assert err == (1 | 4)


# ---------------------------------------------------------------- E4M3 codec

def _torch_e4m3_decode(codes):
    return torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_fixed_points(golden_dir):
    with open(os.path.join(golden_dir, "e4m3_points.json")) as f:
        pts = json.load(f)["codes"]
    for p in pts:
        v = oracle.e4m3_to_double(p["code"])
        if p["value"] == "nan":
            assert math.isnan(v)
        else:
            assert v == p["value"] and math.copysign(1, v) == math.copysign(1, p["value"])


def test_e4m3_decode_all_codes_vs_torch():
    ours = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    ref = _torch_e4m3_decode(list(range(256)))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_encode_roundtrip_and_ties():
    finite = [c for c in range(256) if (c & 0x7f) != 0x7f]
    for c in finite:
        assert oracle.e4m3_from_float(oracle.e4m3_to_double(c)) == c
    pos = sorted({c for c in finite if c < 0x80}, key=oracle.e4m3_to_double)
    for a, b in zip(pos, pos[1:]):
        lo, hi = oracle.e4m3_to_double(a), oracle.e4m3_to_double(b)
        mid = (lo + hi) / 2                     # exact in float32
        got = oracle.e4m3_from_float(mid)
        even = a if a % 2 == 0 else b
        assert got == even, (a, b, mid, got)
        assert oracle.e4m3_from_float(np.nextafter(np.float32(mid), np.float32(0))) == a
        assert oracle.e4m3_from_float(np.nextafter(np.float32(mid), np.float32(1e9))) == b
        assert oracle.e4m3_from_float(-mid) == even | 0x80


def test_e4m3_encode_vs_torch_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = np.clip(x, -448, 448).astype(np.float32)
    ours = np.array([oracle.e4m3_from_float(v) for v in x], np.uint8)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturation():
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_from_float(v) == 0x7E
        assert oracle.e4m3_from_float(-v) == 0xFE
    assert (oracle.e4m3_from_float(float("nan")) & 0x7F) == 0x7F


# ---------------------------------------------------------------- cache write

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_cache_write_roundtrip_16bit(dtype):
    NB, bs, H, D, T = 12, 4, 3, 16, 9
    rng = np.random.default_rng(3)
    kc = W.normal_bits(11, 1, (NB, bs, H, D), dtype)
    vc = W.normal_bits(11, 2, (NB, bs, H, D), dtype)
    before_k, before_v = kc.copy(), vc.copy()
    key = W.normal_bits(11, 3, (T, H, D), dtype)
    val = W.normal_bits(11, 4, (T, H, D), dtype)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[2] = -1                               # padding token: skipped
    err = oracle.reshape_and_cache(key, val, dtype, slots, kc, vc, dtype, bs)
    assert err == 0
    flat_k, flat_v = kc.reshape(NB * bs, H, D), vc.reshape(NB * bs, H, D)
    written = slots >= 0
    assert np.array_equal(flat_k[slots[written]], key[written])
    assert np.array_equal(flat_v[slots[written]], val[written])
    untouched = np.setdiff1d(np.arange(NB * bs), slots[written])
    assert np.array_equal(flat_k[untouched], before_k.reshape(NB * bs, H, D)[untouched])
    assert np.array_equal(flat_v[untouched], before_v.reshape(NB * bs, H, D)[untouched])


def test_cache_write_bad_slot_sets_error():
    kc = np.zeros((2, 4, 1, 8), np.uint16)
    vc = np.zeros_like(kc)
    key = np.ones((1, 1, 8), np.uint16)
    err = oracle.reshape_and_cache(key, key, "f16", np.array([8], np.int64), kc, vc, "f16", 4)
    assert err == 2 and not kc.any()


def test_cache_write_fp8_matches_torch_conversion():
    NB, bs, H, D, T = 6, 16, 2, 32, 40
    key, ak = W.normal_bits(12, 1, (T, H, D), "bf16", want_amax=True)
    val, av = W.normal_bits(12, 2, (T, H, D), "bf16", want_amax=True)
    ks, vs = np.float32(ak) / np.float32(448), np.float32(av) / np.float32(448)
    kc = np.zeros((NB, bs, H, D), np.uint8)
    vc = np.zeros_like(kc)
    slots = np.random.default_rng(0).choice(NB * bs, size=T, replace=False).astype(np.int64)
    assert oracle.reshape_and_cache(key, val, "bf16", slots, kc, vc, "e4m3", bs, ks, vs) == 0
    for src, cache, s in ((key, kc, ks), (val, vc, vs)):
        x = torch.from_numpy(W.bits_to_float(src, "bf16")) / torch.tensor(s, dtype=torch.float32)
        ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(cache.reshape(NB * bs, H, D)[slots], ref)


# ---------------------------------------------------------------- attention

def _sdpa_reference(case, scale, window=0, k_scale=1.0, v_scale=1.0, cache_dtype=None):
    """float64 SDPA per sequence on the contiguous rows of a contiguous_case cache."""
    cd = cache_dtype or case.dtype
    NB, bs, H, D = case.k_cache.shape
    if cd == "e4m3":
        kf = _torch_e4m3_decode(case.k_cache.reshape(-1)).reshape(NB * bs, H, D) * k_scale
        vf = _torch_e4m3_decode(case.v_cache.reshape(-1)).reshape(NB * bs, H, D) * v_scale
    else:
        kf = W.bits_to_float(case.k_cache, cd).astype(np.float64).reshape(NB * bs, H, D)
        vf = W.bits_to_float(case.v_cache, cd).astype(np.float64).reshape(NB * bs, H, D)
    qf = W.bits_to_float(case.q, case.dtype).astype(np.float64)
    Hq = qf.shape[1]
    ql = case.q_len
    outs, lses = [], []
    for b, L in enumerate(case.lengths):
        s0 = int(case.first_block[b]) * bs
        K = torch.from_numpy(kf[s0:s0 + L]).permute(1, 0, 2)[None]      # [1, H, L, D]
        V = torch.from_numpy(vf[s0:s0 + L]).permute(1, 0, 2)[None]
        Q = torch.from_numpy(qf[b * ql:(b + 1) * ql]).permute(1, 0, 2)[None]   # [1, Hq, ql, D]
        p = (L - ql + np.arange(ql))[:, None]
        j = np.arange(L)[None, :]
        allowed = j <= p
        if window > 0:
            allowed &= j > p - window
        mask = torch.from_numpy(allowed)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale,
                                           enable_gqa=(Hq != H))
        outs.append(o[0].permute(1, 0, 2).numpy())
        # lse from the library's own softmax pieces: logsumexp of the masked scores
        Kr = K.repeat_interleave(Hq // H, dim=1)
        sc = (Q @ Kr.transpose(-1, -2)) * scale
        sc = sc.masked_fill(~mask, float("-inf"))
        lses.append(torch.logsumexp(sc, dim=-1)[0].permute(1, 0).numpy())
    return np.concatenate(outs), np.concatenate(lses)


def _oracle(case, scale, window=0, cache_dtype=None, k_scale=1.0, v_scale=1.0, seqs=None):
    return oracle.paged_attention(case.q, case.dtype, case.k_cache, case.v_cache,
                                  cache_dtype or case.dtype, case.block_table, case.lengths,
                                  case.q_len, scale, window, k_scale, v_scale, seqs=seqs, threads=3)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs,ql,window", [
    ("f16", 4, 2, 16, 4, 1, 0),
    ("bf16", 8, 2, 32, 8, 3, 0),
    ("f16", 6, 6, 8, 16, 1, 0),
    ("bf16", 8, 1, 16, 4, 4, 5),
    ("f16", 4, 4, 16, 8, 2, 9),
])
def test_attention_matches_sdpa(dtype, Hq, Hkv, D, bs, ql, window):
    case = contiguous_case([1 + ql, 7, 13, 33, 4 + ql], Hq, Hkv, D, bs, ql, dtype, seed=Hq * D + bs)
    scale = 1.0 / math.sqrt(D)
    out, lse = _oracle(case, scale, window)
    ref_out, ref_lse = _sdpa_reference(case, scale, window)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attention_block_permutation_invariance():
    case = contiguous_case([5, 17, 30, 2], 4, 2, 16, 4, 2, "f16", seed=9)
    perm = np.random.default_rng(4).permutation(case.num_blocks)
    moved = relabel_blocks(case, perm)
    assert not np.array_equal(moved.block_table, case.block_table)
    a = _oracle(case, 0.3)
    b = _oracle(moved, 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_attention_gqa_equals_mha_with_repeated_heads():
    case = contiguous_case([9, 21], 8, 2, 16, 4, 1, "bf16", seed=10)
    g = 4
    mha = contiguous_case([9, 21], 8, 8, 16, 4, 1, "bf16", seed=10)
    mha.k_cache = np.repeat(case.k_cache, g, axis=2)
    mha.v_cache = np.repeat(case.v_cache, g, axis=2)
    mha.q = case.q
    a = _oracle(case, 0.25)
    b = _oracle(mha, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_attention_closed_forms():
    D = 16
    # one key: out = V_0, lse = scale * q.k_0
    case = contiguous_case([1, 1], 2, 1, D, 4, 1, "f16", seed=11)
    out, lse = _oracle(case, 0.5)
    for b in range(2):
        s0 = int(case.first_block[b]) * 4
        v0 = W.bits_to_float(case.v_cache.reshape(-1, 1, D)[s0, 0], "f16").astype(np.float64)
        k0 = W.bits_to_float(case.k_cache.reshape(-1, 1, D)[s0, 0], "f16").astype(np.float64)
        for h in range(2):
            qv = W.bits_to_float(case.q[b, h], "f16").astype(np.float64)
            assert np.array_equal(out[b, h], v0)
            assert lse[b, h] == pytest.approx(0.5 * float(qv @ k0), abs=1e-12)
    # scale 0: uniform weights, out = mean of the visible V rows, lse = ln(count)
    case = contiguous_case([6, 11], 4, 2, D, 4, 3, "bf16", seed=12)
    out, lse = _oracle(case, 0.0, window=4)
    vf = W.bits_to_float(case.v_cache, "bf16").astype(np.float64).reshape(-1, 2, D)
    for b, L in enumerate(case.lengths):
        s0 = int(case.first_block[b]) * 4
        for i in range(3):
            p = L - 3 + i
            keys = [j for j in range(L) if j <= p and j > p - 4]
            for hq in range(4):
                mean = vf[s0 + np.array(keys), hq // 2].mean(axis=0)
                np.testing.assert_allclose(out[b * 3 + i, hq], mean, atol=1e-12)
                assert lse[b * 3 + i, hq] == pytest.approx(math.log(len(keys)), abs=1e-12)
    # equal keys: weights are uniform whatever the scale
    case = contiguous_case([7], 2, 1, D, 4, 1, "f16", seed=13)
    flat = case.k_cache.reshape(-1, 1, D)
    s0 = int(case.first_block[0]) * 4
    flat[s0:s0 + 7] = flat[s0]
    out, _ = _oracle(case, 0.9)
    vf = W.bits_to_float(case.v_cache, "f16").astype(np.float64).reshape(-1, 1, D)
    np.testing.assert_allclose(out[0, 0], vf[s0:s0 + 7, 0].mean(axis=0), atol=1e-12)


def test_attention_window_covering_everything_equals_full():
    case = contiguous_case([5, 19, 40], 4, 2, 16, 8, 2, "f16", seed=14)
    full = _oracle(case, 0.2, window=0)
    wide = _oracle(case, 0.2, window=40)
    assert np.array_equal(full[0], wide[0]) and np.array_equal(full[1], wide[1])
    narrow = _oracle(case, 0.2, window=6)
    assert not np.allclose(full[0], narrow[0])


def test_attention_window_ignores_poisoned_old_blocks():
    bs, W_ = 4, 6
    case = contiguous_case([30, 23], 4, 2, 16, bs, 2, "bf16", seed=15)
    clean = _oracle(case, 0.3, window=W_)
    nan_bits = np.uint16(0x7FC0)
    touched = 0
    for b, L in enumerate(case.lengths):
        lo = max(0, L - 2 - W_ + 1)                 # first key any of the 2 queries may see
        for lb in range(lo // bs):                  # blocks wholly before the window
            case.k_cache[case.block_table[b, lb]] = nan_bits
            case.v_cache[case.block_table[b, lb]] = nan_bits
            touched += 1
        # the page's bound: a window needs at most about W / block_size blocks
        nblocks = (L - 1) // bs - lo // bs + 1
        assert nblocks <= math.ceil((W_ + 2 - 1) / bs) + 1
    assert touched > 0
    poisoned = _oracle(case, 0.3, window=W_)
    assert np.isfinite(poisoned[0]).all()
    assert np.array_equal(clean[0], poisoned[0]) and np.array_equal(clean[1], poisoned[1])


def test_attention_window_released_entries_are_not_read():
    """Blocks wholly before every query's window may have gone back to the pool ("vLLM Worker侧
    GPU KV Cache初始化流程深度解析", section "混合注意力机制"): with -1 in their table entries the
    result is the same and no error is raised."""
    bs, W_ = 4, 6
    case = contiguous_case([30, 23, 9], 4, 2, 16, bs, 2, "f16", seed=25)
    clean = _oracle(case, 0.3, window=W_)
    released = 0
    for b, L in enumerate(case.lengths):
        lo = max(0, L - 2 - W_ + 1)
        for lb in range(lo // bs):
            case.block_table[b, lb] = -1
            released += 1
    assert released > 0
    again = _oracle(case, 0.3, window=W_)
    assert np.array_equal(clean[0], again[0]) and np.array_equal(clean[1], again[1])
    with pytest.raises(ValueError):  # without a window every entry is read
        _oracle(case, 0.3, window=0)


def test_attention_speculative_queries_equal_shorter_single_queries():
    ql = 4
    case = contiguous_case([9, 26], 4, 2, 16, 4, ql, "f16", seed=16)
    out, lse = _oracle(case, 0.4, window=7)
    for i in range(ql):
        one = contiguous_case([9, 26], 4, 2, 16, 4, 1, "f16", seed=16)
        one.k_cache, one.v_cache, one.block_table = case.k_cache, case.v_cache, case.block_table
        one.lengths = (case.lengths - ql + 1 + i).astype(np.int32)
        one.q = case.q.reshape(2, ql, 4, 16)[:, i].copy()
        o1, l1 = _oracle(one, 0.4, window=7)
        assert np.array_equal(o1, out.reshape(2, ql, 4, 16)[:, i])
        assert np.array_equal(l1, lse.reshape(2, ql, 4)[:, i])


def test_attention_fp8_cache_matches_sdpa_on_dequantised_cache():
    case = contiguous_case([3, 17, 32], 8, 2, 32, 16, 1, "bf16", seed=17)
    NB, bs, H, D = case.k_cache.shape
    kc8 = np.zeros((NB, bs, H, D), np.uint8)
    vc8 = np.zeros_like(kc8)
    ident = np.arange(NB * bs, dtype=np.int64)
    src_k = case.k_cache.reshape(NB * bs, H, D)
    src_v = case.v_cache.reshape(NB * bs, H, D)
    ks, vs = 0.02, 0.015
    assert oracle.reshape_and_cache(src_k, src_v, "bf16", ident, kc8, vc8, "e4m3", bs, ks, vs) == 0
    case.k_cache, case.v_cache = kc8, vc8
    out, lse = _oracle(case, 0.125, cache_dtype="e4m3", k_scale=ks, v_scale=vs)
    ref_out, ref_lse = _sdpa_reference(case, 0.125, cache_dtype="e4m3", k_scale=ks, v_scale=vs)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_attention_subset_of_sequences():
    case = contiguous_case([5, 8, 12], 2, 1, 8, 4, 1, "f16", seed=18)
    full = _oracle(case, 0.3)
    part = _oracle(case, 0.3, seqs=[2])
    assert np.isnan(part[0][0]).all() and np.isnan(part[0][1]).all()
    assert np.array_equal(part[0][2], full[0][2])


def test_tiny_workload_by_hand():
    """The tiny decode batch: lengths {5,4,9,13} at block size 4 put the new tokens at
    positions 4, 3, 8, 12; three of the four open a fresh block (the block-of-4 spill)."""
    wl = W.make_workload(W.TINY)
    assert wl.positions.tolist() == [4, 3, 8, 12]
    assert [int(p) % 4 for p in wl.positions].count(0) == 3
    slots, err = oracle.slot_mapping(wl.block_table, wl.query_start_loc, wl.positions, 4,
                                     wl.num_blocks)
    assert err == 0
    for b, p in enumerate(wl.positions):
        assert slots[b] == wl.block_table[b, p // 4] * 4 + p % 4
    used = wl.block_table[wl.block_table >= 0]
    assert len(used) == 10 and len(set(used.tolist())) == 10
