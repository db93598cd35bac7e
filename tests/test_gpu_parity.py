"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same seeded inputs.

Slot mapping and cache writes are compared bit for bit; attention element by element at the
specification's tolerances (max abs 1e-3 fp16, 8e-3 bf16; fp8 caches 2e-2 of max|oracle|).
Small cases span several pipeline stages, partitions and a ragged tail; the full-size workloads
run in the launch configuration the benchmark times and are compared on every row and every
cache slot.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_block_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


def _small(spec: W.WorkloadSpec, **kw) -> W.WorkloadSpec:
    return spec.replace(**kw)


SMALL = {
    "tiny": W.TINY,
    "opt125m_small": _small(W.OPT125M, num_seqs=6, lengths=("uniform", 17, 700), num_blocks=400),
    "llama3_8b_small": _small(W.LLAMA3_8B, num_seqs=5, lengths=("uniform", 100, 1500)),
    "llama70b_fp8_small": _small(W.LLAMA70B_FP8, num_seqs=3, lengths=("fixed", (600, 129, 1024)),
                                 num_blocks=200),
    "mistral_hybrid_small": _small(W.MISTRAL_HYBRID, num_seqs=8,
                                   lengths=("lognormal", 300, 1.0, 64, 3000),
                                   shared_prefix_tokens=128, windows=(0, 200)),
}


def _run_both(wl, layer, num_workers=0, seqs=None):
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = H.gpu_step(wl, layer, kc, vc, num_workers=num_workers)
    o = H.oracle_step(wl, layer, seqs=seqs)
    return g, o


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("num_workers", [0, 7])
def test_small_configs_match_oracle(kv, name, num_workers):
    wl = W.make_workload(SMALL[name])
    for layer in wl.layers:
        g, o = _run_both(wl, layer, num_workers)
        assert g.err == 0
        assert np.array_equal(g.slots.cpu().numpy(), o.slots)
        assert np.array_equal(H.cache_bits(g.k_cache), o.k_cache.reshape(H.cache_bits(g.k_cache).shape))
        assert np.array_equal(H.cache_bits(g.v_cache), o.v_cache.reshape(H.cache_bits(g.v_cache).shape))
        H.check_attention(wl, g, o)


def test_tiny_config_by_value(kv):
    """The tiny batch end to end, with the slots the oracle derives from the table."""
    wl = W.make_workload(W.TINY)
    g, o = _run_both(wl, wl.layers[0])
    assert g.slots.cpu().tolist() == o.slots.tolist()
    assert all(s >= 0 for s in o.slots)
    H.check_attention(wl, g, o)


FULL = ["opt125m", "llama3_8b", "llama70b_fp8", "mistral_hybrid"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(kv, name):
    """Full workload in the launch configuration the benchmark times (one worker per SM): every
    output and lse row of every layer against the oracle, the slot mapping, and the whole cache
    (every slot of every block, written or not) bit for bit."""
    wl = W.make_workload(W.BY_NAME[name])
    for layer in wl.layers:
        kc, vc = H.gpu_fill_cache(wl, layer)
        g = H.gpu_step(wl, layer, kc, vc)
        assert g.err == 0
        o = H.oracle_step(wl, layer)
        assert np.array_equal(g.slots.cpu().numpy(), o.slots)
        H.check_whole_cache(g, o)
        H.check_attention(wl, g, o)
        del kc, vc, g, o
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- shapes and options

def _spec(**kw):
    base = dict(name="custom", num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                dtype="bf16", cache_dtype="bf16", lengths=("fixed", (1, 17, 300, 95)), seed=77)
    base.update(kw)
    return W.WorkloadSpec(**base)


@pytest.mark.parametrize("bs", [4, 8, 16, 32])
@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (64, "bf16"), (128, "f16")])
def test_block_sizes_and_head_dims(kv, bs, D, dtype):
    wl = W.make_workload(_spec(block_size=bs, head_dim=D, dtype=dtype, cache_dtype=dtype,
                               lengths=("fixed", (1, 2 * bs + 1, 9 * bs - 3, 40 * bs))))
    g, o = _run_both(wl, wl.layers[0], num_workers=13)
    H.check_attention(wl, g, o)


@pytest.mark.parametrize("Hq,Hkv,ql", [(8, 8, 1), (8, 1, 1), (32, 4, 8), (16, 2, 5), (12, 4, 3), (64, 8, 1)])
def test_gqa_groups_and_speculative_lengths(kv, Hq, Hkv, ql):
    wl = W.make_workload(_spec(num_q_heads=Hq, num_kv_heads=Hkv, q_len=ql,
                               lengths=("fixed", (ql, ql + 16, 333, 1000))))
    g, o = _run_both(wl, wl.layers[0])
    H.check_attention(wl, g, o)


@pytest.mark.parametrize("window", [1, 7, 16, 100, 4096])
def test_sliding_windows(kv, window):
    wl = W.make_workload(_spec(q_len=4, lengths=("fixed", (4, 50, 333, 2000)), windows=(window,)))
    g, o = _run_both(wl, wl.layers[0], num_workers=5)
    H.check_attention(wl, g, o)


def test_fp8_cache_f16_queries(kv):
    wl = W.make_workload(_spec(dtype="f16", cache_dtype="e4m3", num_q_heads=16, num_kv_heads=2,
                               lengths=("fixed", (5, 100, 700, 1600))))
    g, o = _run_both(wl, wl.layers[0])
    assert np.array_equal(H.cache_bits(g.k_cache), o.k_cache)
    H.check_attention(wl, g, o)


@pytest.mark.parametrize("bs", [4, 8, 16, 32])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fp8_cache_block_sizes(kv, bs, dtype):
    """E4M3 caches at every block size: 16-token blocks run the kernel built for that block size,
    the others the general one; two speculative tokens, several stages, a ragged tail."""
    wl = W.make_workload(_spec(block_size=bs, dtype=dtype, cache_dtype="e4m3", num_q_heads=16, num_kv_heads=2,
                               q_len=2, lengths=("fixed", (2, 2 * bs + 1, 9 * bs - 3, 40 * bs))))
    g, o = _run_both(wl, wl.layers[0], num_workers=13)
    assert np.array_equal(H.cache_bits(g.k_cache), o.k_cache)
    H.check_attention(wl, g, o)


def test_worker_count_invariance(kv):
    """Shares of 1 to 1000 workers cut the sequences at different keys; every split gives the
    same result within tolerance (and the oracle's)."""
    wl = W.make_workload(_spec(lengths=("fixed", (2000, 1500, 999, 3))))
    layer = wl.layers[0]
    outs = []
    for workers in (1, 2, 7, 64, 1000, 0):
        kc, vc = H.gpu_fill_cache(wl, layer)
        g = H.gpu_step(wl, layer, kc, vc, num_workers=workers)
        assert g.err == 0
        outs.append(g.out.float())
    o = H.oracle_step(wl, layer)
    for x in outs:
        assert (x - outs[0]).abs().max().item() <= 8e-3
    H.check_attention(wl, g, o)


def test_block_permutation_invariance_bit_exact(kv):
    wl = W.make_workload(_spec(lengths=("fixed", (40, 300, 1000, 77)), num_blocks=200))
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    a = H.gpu_step(wl, layer, kc, vc, num_workers=9).out
    perm = np.random.default_rng(3).permutation(wl.num_blocks)
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[torch.from_numpy(perm).cuda()] = kc
    vc2[torch.from_numpy(perm).cuda()] = vc
    table = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    b = H.gpu_step(wl, layer, kc2, vc2, num_workers=9, block_table=table).out
    assert torch.equal(a, b)


def test_nan_poison_outside_what_is_read(kv):
    """Unused pool blocks, blocks wholly before the window and the unused tail slots of each
    sequence's last block hold NaN; the output stays finite and equal to the oracle's."""
    spec = _spec(q_len=2, lengths=("fixed", (37, 301, 999, 64)), windows=(90,), num_blocks=120)
    wl = W.make_workload(spec)
    layer = wl.layers[0]
    bs = spec.block_size
    nan = np.uint16(0x7FC0)
    used = set()
    for b, L in enumerate(wl.seq_lens):
        lo = max(0, L - 2 - 90 + 1)
        for lb in range(-(-L // bs)):
            blk = wl.block_table[b, lb]
            if lb < lo // bs:
                layer.pool_k[blk * bs:(blk + 1) * bs] = nan
                layer.pool_v[blk * bs:(blk + 1) * bs] = nan
            else:
                used.add(int(blk))
        last = wl.block_table[b, (L - 1) // bs]
        for off in range(L % bs or bs, bs):           # slots past the sequence's end
            layer.pool_k[last * bs + off] = nan
            layer.pool_v[last * bs + off] = nan
    for blk in range(wl.num_blocks):
        if blk not in used and blk not in wl.block_table:
            layer.pool_k[blk * bs:(blk + 1) * bs] = nan
            layer.pool_v[blk * bs:(blk + 1) * bs] = nan
    g, o = _run_both(wl, layer, num_workers=11)
    assert torch.isfinite(g.out).all()
    H.check_attention(wl, g, o)


# ---------------------------------------------------------------- data errors and edge cases

def test_slot_mapping_edges(kv):
    bt = torch.tensor([[3, -1, 99, 5]], dtype=torch.int32, device="cuda")
    qsl = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    pos = torch.tensor([0, 5, 9, 16, -1, 2], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = kv.compute_slot_mapping(bt, qsl, pos, 4, 10, d_err=err)
    ref, ref_err = oracle.slot_mapping(bt.cpu().numpy(), qsl.cpu().numpy(), pos.cpu().numpy(), 4, 10)
    assert s.cpu().tolist() == ref.tolist() == [12, -1, -1, -1, -1, -1]
    assert err.item() == ref_err == (1 | 4)
    empty = kv.compute_slot_mapping(bt, qsl, pos[:0], 4, 10)
    assert empty.numel() == 0


def test_cache_write_bad_slot_and_guard_blocks(kv):
    NB, bs, Hh, D = 6, 16, 2, 64
    guard = 2
    big = torch.full(((NB + 2 * guard) * bs * Hh * D,), 0x5A5A, dtype=torch.int16, device="cuda")
    kc = big.view(NB + 2 * guard, bs, Hh, D)[guard:guard + NB].view(torch.float16)
    big_v = big.clone()
    vc = big_v.view(NB + 2 * guard, bs, Hh, D)[guard:guard + NB].view(torch.float16)
    key = torch.randn(4, Hh, D, device="cuda", dtype=torch.float16)
    slots = torch.tensor([0, NB * bs - 1, NB * bs, -1], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.reshape_and_cache(key, key, slots, kc, vc, d_err=err)
    torch.cuda.synchronize()
    assert err.item() == 2
    flat = kc.reshape(NB * bs, Hh, D)
    assert torch.equal(flat[0], key[0]) and torch.equal(flat[NB * bs - 1], key[1])
    g = guard * bs * Hh * D
    assert (big[:g] == 0x5A5A).all() and (big[-g:] == 0x5A5A).all()
    assert (big_v[:g] == 0x5A5A).all() and (big_v[-g:] == 0x5A5A).all()


def test_bad_lengths_and_block_ids_set_error_bits(kv):
    wl = W.make_workload(_spec(q_len=2, lengths=("fixed", (10, 300, 40, 64))))
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    bt = torch.from_numpy(wl.block_table).cuda()
    bt[1, 3] = -7                                   # a used entry of sequence 1
    L = torch.from_numpy(wl.seq_lens).cuda()
    L[2] = 1                                        # shorter than q_len
    q = H.to_dev(layer.q, "bf16")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_attention_decode(q, kc, vc, bt, L, wl.max_seq_len, 2, 0.1, d_err=err)
    torch.cuda.synchronize()
    assert err.item() & kv.KV_DERR_BAD_BLOCK and err.item() & kv.KV_DERR_BAD_LEN
    assert torch.isfinite(out).all()
    assert (out[4:6] == 0).all()                    # the bad-length sequence's rows
    err.zero_()
    L2 = torch.from_numpy(wl.seq_lens).cuda()
    kv.paged_attention_decode(q, kc, vc, torch.from_numpy(wl.block_table).cuda(), L2, 100, 2, 0.1,
                              d_err=err)            # max_seq_len below a real length
    torch.cuda.synchronize()
    assert err.item() == kv.KV_DERR_BAD_LEN


def test_host_errors(kv):
    wl = W.make_workload(_spec())
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    q = H.to_dev(layer.q, "bf16")
    bt = torch.from_numpy(wl.block_table).cuda()
    L = torch.from_numpy(wl.seq_lens).cuda()
    with pytest.raises(kv.KVError) as e:
        kv.paged_attention_decode(q.half(), kc, vc, bt, L, wl.max_seq_len, 1, 0.1)
    assert e.value.status == 2                      # fp16 q over a bf16 cache
    with pytest.raises(kv.KVError) as e:
        kv.paged_attention_workspace_size(4, 1, 8, 2, 96, 16, 1, 300)
    need = kv.paged_attention_workspace_size(4, 1, 8, 2, 128, 16, 1, 300, 0, 16)
    assert need > 0
    small = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    rc = kv.lib.kv_paged_attention_decode(
        q.data_ptr(), 1, 4, 1, 8, kc.data_ptr(), vc.data_ptr(), 1, 2, 128, 16, wl.num_blocks,
        bt.data_ptr(), bt.stride(0), bt.shape[1], L.data_ptr(), 300, 0.1, 0, 1.0, 1.0, 16,
        small.data_ptr(), small.numel(), q.data_ptr(), None, None, None)
    assert rc == 4                                  # KV_ERR_WORKSPACE, nothing launched


def test_empty_batch(kv):
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(0, 4, dtype=torch.int32, device="cuda")
    L = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = kv.paged_attention_decode(q, kc, kc, bt, L, 64, 1, 0.1)
    assert out.numel() == 0


def test_many_short_sequences(kv):
    """4,000 sequences of 1..40 tokens: a large per-CTA stage table, most shares splitting
    sequences, many one-block items; every row against the oracle."""
    wl = W.make_workload(_spec(num_seqs=4000, lengths=("uniform", 1, 40), seed=91))
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = H.gpu_step(wl, layer, kc, vc)
    assert g.err == 0
    o = H.oracle_step(wl, layer)
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    H.check_attention(wl, g, o)


@pytest.mark.parametrize("fused", [False, True])
def test_eight_thousand_sequences_keep_the_ring(kv, fused):
    """8,000 sequences at the Llama-3-8B layer shape: the schedule's shared-memory table does not
    squeeze the pipeline below three 64 KB stages, and every row matches the oracle."""
    spec = W.LLAMA3_8B.replace(num_seqs=8000, lengths=("uniform", 16, 300), seed=93)
    info = kv.paged_attention_plan_info(8000, 1, 32, 8, 128, 16, kv.KV_BF16, 300)
    assert info["stages"] >= 3 and info["stage_bytes"] == 64 * 1024
    wl = W.make_workload(spec)
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = (H.gpu_step_fused if fused else H.gpu_step)(wl, layer, kc, vc)
    assert g.err == 0
    o = H.oracle_step(wl, layer)
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    H.check_whole_cache(g, o)
    H.check_attention(wl, g, o)


def test_batch_too_large_for_the_stage_table(kv):
    """A batch whose per-CTA schedule cannot fit in shared memory is refused on the host."""
    with pytest.raises(kv.KVError) as e:
        kv.paged_attention_workspace_size(200000, 1, 8, 2, 128, 16, kv.KV_BF16, 64)
    assert e.value.status == kv.KV_ERR_UNSUPPORTED
