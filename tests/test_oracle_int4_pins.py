"""Pins of the oracle's INT4 cache (the half-byte KV format of "KV Cache技术背景", with given group
scales): the 16 codes
against numpy's two's-complement sign extension, encoding against numpy's round-half-to-even and
clip, the cache write against a numpy quantisation of the same inputs (float32 division, nibble
order, group index), and attention over INT4 caches against float64 SDPA on numpy-dequantised
caches."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_block_gb300 import workloads as W
from tests.cases import contiguous_case


def np_sign_extend(nibbles: np.ndarray) -> np.ndarray:
    return (np.asarray(nibbles, np.uint8) << 4).view(np.int8) >> 4


def np_quantise(x32: np.ndarray, s32: np.ndarray) -> np.ndarray:
    """Expected codes: float32 division, round half to even, clip to [-8, 7]."""
    return np.clip(np.rint(np.float32(x32) / np.float32(s32)), -8, 7).astype(np.int8)


def np_dequantise(cache: np.ndarray, scales: np.ndarray, group: int) -> np.ndarray:
    """uint8 [NB, bs, H, D/2] + float32 [H, D/G] -> float64 [NB, bs, H, D]."""
    lo = np_sign_extend(cache & 0xF)
    hi = np_sign_extend(cache >> 4)
    q = np.stack([lo, hi], axis=-1).reshape(*cache.shape[:-1], cache.shape[-1] * 2).astype(np.float64)
    D = q.shape[-1]
    sc = np.repeat(np.asarray(scales, np.float64), group, axis=1)  # [H, D]
    return q * sc[None, None, :, :D]


def test_int4_decodes_all_16_codes():
    codes = np.arange(16)
    assert [oracle.int4_to_double(c) for c in codes] == np_sign_extend(codes).astype(float).tolist()


def test_int4_encode_rounds_half_to_even_and_saturates():
    rng = np.random.default_rng(41)
    xs = np.concatenate([np.arange(-12, 12.25, 0.25), rng.normal(0, 5, 500)]).astype(np.float32)
    want = np_quantise(xs, np.float32(1.0)).astype(np.int64) & 0xF
    got = np.array([oracle.int4_from_float(x) for x in xs])
    assert np.array_equal(got, want)
    for q in range(-8, 8):
        assert oracle.int4_to_double(oracle.int4_from_float(q)) == q


def test_int4_encode_non_finite():
    assert oracle.int4_to_double(oracle.int4_from_float(np.float32(np.inf))) == 7
    assert oracle.int4_to_double(oracle.int4_from_float(np.float32(-np.inf))) == -8
    assert oracle.int4_from_float(np.float32(np.nan)) == 0
    assert oracle.int4_to_double(oracle.int4_from_float(np.float32(3e38))) == 7


@pytest.mark.parametrize("group", [32, 64, 128])
def test_int4_cache_write_matches_numpy_quantisation(group):
    T, H, D, NB, bs = 5, 3, 128, 6, 4
    rng = np.random.default_rng(group)
    k = W.normal_bits(7, 1, (T, H, D), "bf16")
    v = W.normal_bits(7, 2, (T, H, D), "bf16")
    ks = rng.uniform(0.05, 0.6, (H, D // group)).astype(np.float32)
    vs = rng.uniform(0.05, 0.6, (H, D // group)).astype(np.float32)
    slots = np.array([3, -1, 17, 0, NB * bs - 1], np.int64)
    kc = oracle.cache_zeros(NB, bs, H, D, "int4")
    vc = oracle.cache_zeros(NB, bs, H, D, "int4")
    kc[:] = 0xAB
    vc[:] = 0xAB
    assert oracle.reshape_and_cache_int4(k, v, "bf16", slots, kc, vc, bs, ks, vs, group) == 0
    for src, scales, cache in ((k, ks, kc), (v, vs, vc)):
        xf = W.bits_to_float(src, "bf16")
        s_full = np.repeat(scales, group, axis=1)  # [H, D]
        flat = cache.reshape(NB * bs, H, D // 2)
        for t, slot in enumerate(slots):
            if slot < 0:
                continue
            q = np_quantise(xf[t], s_full)                          # [H, D]
            want = (q[:, 0::2].astype(np.uint8) & 0xF) | ((q[:, 1::2].astype(np.uint8) & 0xF) << 4)
            assert np.array_equal(flat[slot], want)
        untouched = np.ones(NB * bs, bool)
        untouched[slots[slots >= 0]] = False
        assert (flat[untouched] == 0xAB).all()


@pytest.mark.parametrize("Hq,Hkv,q_len,window,group", [(8, 2, 1, 0, 32), (8, 8, 3, 0, 64), (16, 2, 2, 9, 128)])
def test_int4_attention_matches_sdpa_on_dequantised_cache(Hq, Hkv, q_len, window, group):
    D, bs = 128, 8
    case = contiguous_case([1 + q_len, 13, 40, 7 + q_len], Hq, Hkv, D, bs, q_len, "bf16", seed=Hq + group)
    NB = case.num_blocks
    rng = np.random.default_rng(group + Hq)
    kc = rng.integers(0, 256, (NB, bs, Hkv, D // 2), dtype=np.uint8)
    vc = rng.integers(0, 256, (NB, bs, Hkv, D // 2), dtype=np.uint8)
    ks = rng.uniform(0.1, 0.5, (Hkv, D // group)).astype(np.float32)
    vs = rng.uniform(0.1, 0.5, (Hkv, D // group)).astype(np.float32)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.paged_attention_int4(case.q, "bf16", kc, vc, case.block_table, case.lengths, q_len,
                                           scale, window, ks, vs, group, threads=3)
    kf = np_dequantise(kc, ks, group).reshape(NB * bs, Hkv, D)
    vf = np_dequantise(vc, vs, group).reshape(NB * bs, Hkv, D)
    qf = W.bits_to_float(case.q, "bf16").astype(np.float64)
    for b, L in enumerate(case.lengths):
        s0 = int(case.first_block[b]) * bs
        K = torch.from_numpy(kf[s0:s0 + L]).permute(1, 0, 2)[None]
        V = torch.from_numpy(vf[s0:s0 + L]).permute(1, 0, 2)[None]
        Q = torch.from_numpy(qf[b * q_len:(b + 1) * q_len]).permute(1, 0, 2)[None]
        p = (L - q_len + np.arange(q_len))[:, None]
        j = np.arange(L)[None, :]
        allowed = j <= p
        if window > 0:
            allowed &= j > p - window
        mask = torch.from_numpy(allowed)
        ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale, enable_gqa=(Hq != Hkv))
        np.testing.assert_allclose(out[b * q_len:(b + 1) * q_len], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        Kr = K.repeat_interleave(Hq // Hkv, dim=1)
        sc = ((Q @ Kr.transpose(-1, -2)) * scale).masked_fill(~mask, float("-inf"))
        np.testing.assert_allclose(lse[b * q_len:(b + 1) * q_len], torch.logsumexp(sc, -1)[0].permute(1, 0).numpy(),
                                   rtol=0, atol=1e-12)
