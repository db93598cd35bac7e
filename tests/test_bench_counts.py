"""The byte and FLOP counts behind bench.py's GB/s and TFLOP/s, against brute force on small
workloads (no GPU needed): attention reads each distinct physical cache slot any query attends
once (a prefix shared through the block table counts once), plus q, out and the table entries of
the attended blocks; prefill counts 4·D·Hq FLOP per visible (query, key) pair."""
import dataclasses

import numpy as np

import bench
from paged_kv_cache_block_gb300 import workloads as W


def brute_attention_bytes(wl, window):
    s = wl.spec
    bs = s.block_size
    row = int(2 * s.num_kv_heads * s.head_dim * W.elem_bytes(s.cache_dtype))
    slots, nblocks = set(), 0
    for b in range(len(wl.seq_lens)):
        L = int(wl.seq_lens[b])
        first = max(0, L - s.q_len - window + 1) if window > 0 else 0
        blocks = set()
        for key in range(first, L):  # every key some query of the sequence attends
            slots.add((int(wl.block_table[b, key // bs]), key % bs))
            blocks.add(key // bs)
        nblocks += len(blocks)
    q_out = 2 * wl.num_tokens * s.num_q_heads * s.head_dim * 2
    scales = 2 * s.num_kv_heads * (s.head_dim // s.group_size) * 4 if s.cache_dtype == "int4" else 0
    return len(slots) * row + q_out + 4 * nblocks + scales


def test_attention_bytes_without_sharing():
    spec = W.TINY.replace(lengths=("fixed", (5, 4, 9, 13)))
    wl = W.make_workload(spec)
    got = bench.algorithmic_bytes(wl)["layers"][0]["attention"]
    assert got == brute_attention_bytes(wl, 0)
    # no slot is shared: the distinct slots are all the attended keys
    row = 2 * spec.num_kv_heads * spec.head_dim * 2
    keys = int(wl.seq_lens.sum())
    assert got - 4 * sum(-(-int(L) // 4) for L in wl.seq_lens) - 2 * wl.num_tokens * 4 * 64 * 2 == keys * row


def test_attention_bytes_with_a_shared_prefix_and_windows():
    spec = W.MISTRAL_HYBRID.replace(num_seqs=12, lengths=("fixed", (1100, 1500, 2100, 1050, 1300, 3000,
                                                                    1200, 1090, 1700, 2500, 1088, 4000)),
                                    windows=(0, 700), seed=77)
    wl = W.make_workload(spec)
    assert wl.shared.sum() >= 2, "the case needs sequences that share the prefix"
    counts = bench.algorithmic_bytes(wl)
    assert len(counts["layers"]) == 2
    for layer, lay in zip(wl.layers, counts["layers"]):
        assert lay["attention"] == brute_attention_bytes(wl, layer.window)
    # the shared prefix is read once: the full-attention layer moves fewer K/V bytes than the
    # keys its queries attend
    full = counts["layers"][0]
    q_out = 2 * wl.num_tokens * spec.num_q_heads * spec.head_dim * 2
    table = 4 * sum(-(-int(L) // spec.block_size) for L in wl.seq_lens)
    assert full["attention"] - q_out - table < full["logical_kv"]


def test_int4_bytes_are_half_a_byte_per_element_plus_scales():
    wl = W.make_workload(W.LLAMA3_8B_INT4.replace(num_seqs=3, lengths=("fixed", (40, 17, 300))))
    assert bench.algorithmic_bytes(wl)["layers"][0]["attention"] == brute_attention_bytes(wl, 0)


def test_prefill_flops_count_visible_pairs():
    spec = dataclasses.replace(W.PREFILL_LLAMA3_8B, num_seqs=3, chunk=("fixed", 40), context=("fixed", 25))
    pw = W.make_prefill(spec)
    pairs = 0
    for L, n in zip(pw.seq_lens, pw.chunks):
        for i in range(int(n)):
            p = int(L) - int(n) + i
            pairs += sum(1 for j in range(int(L)) if j <= p)
    assert bench.prefill_flops(pw) == 4 * spec.head_dim * spec.num_q_heads * pairs
    wspec = dataclasses.replace(spec, window=9)
    pw = W.make_prefill(wspec)
    pairs = 0
    for L, n in zip(pw.seq_lens, pw.chunks):
        for i in range(int(n)):
            p = int(L) - int(n) + i
            pairs += sum(1 for j in range(int(L)) if p - 9 < j <= p)
    assert bench.prefill_flops(pw) == 4 * spec.head_dim * spec.num_q_heads * pairs


def test_window_summary_and_headline_summary():
    w = bench.window_summary([10.0, 12.0, 11.0, 30.0, 10.5], 20)
    assert w["count"] == 5 and w["steps_each"] == 20
    assert w["ms_per_step_median"] == 11.0 / 20 and w["ms_per_step_min"] == 10.0 / 20
    full = {"metric": "m", "value": 1.0, "unit": "GB/s", "ms_per_step": 0.5, "roofline": {"frac": 0.9},
            "e2e": {"value": 0.8}, "cpu_baseline": {"value": 0.01}, "step_bytes": 123, "n_gpus": 1}
    s = bench.summary(full)
    assert s["roofline"]["frac"] == 0.9 and s["e2e"]["value"] == 0.8 and "step_bytes" not in s


def test_both_arms_print_the_same_decode_config():
    import argparse
    wl = W.make_workload(W.TINY)
    args = argparse.Namespace(workers=0, mode=None)
    attn = sum(l["attention"] for l in bench.algorithmic_bytes(wl)["layers"])
    a = bench.decode_config(wl, args, 1, attn, bench.decode_mode(args, "tiny"))
    b = bench.decode_config(W.make_workload(W.TINY), args, 1, attn, bench.decode_mode(args, "tiny"))
    assert a == b and a["mode"] == "fused"
    assert bench.decode_mode(args, "llama3_8b_int4") == "calls"
