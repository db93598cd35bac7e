"""Parity of the INT4 cache path (include/pagedkv_int4.h) with the CPU oracle.

The INT4 format of "KV Cache技术背景" (half a byte per element, with given group scales): cache
writes are compared bit for bit, attention element by element at 1e-2 of max|oracle| (the
kernel rounds q * k_scale and the softmax weights to fp16) and the log-sum-exp at 2e-3.
Small cases span several stages, CTAs and a ragged tail; the full-size batch runs in the launch
configuration the benchmark times and is compared on every row and every cache slot.
"""
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


def _spec(**kw):
    base = dict(name="custom_int4", num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                block_size=16, dtype="bf16", cache_dtype="int4", group_size=32,
                lengths=("fixed", (1, 17, 300, 95)), seed=78)
    base.update(kw)
    return W.WorkloadSpec(**base)


def _run_both(wl, layer, num_workers=0, seqs=None):
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = H.gpu_step(wl, layer, kc, vc, num_workers=num_workers)
    o = H.oracle_step(wl, layer, seqs=seqs)
    return g, o


def _check_all(wl, g, o):
    assert g.err == 0
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    assert np.array_equal(g.k_cache.cpu().numpy(), o.k_cache)
    assert np.array_equal(g.v_cache.cpu().numpy(), o.v_cache)
    return H.check_attention(wl, g, o)


# ---------------------------------------------------------------- cache write

@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("group", [8, 32, 128])
def test_cache_write_bit_exact_with_specials(kv, dtype, group):
    """Random rows plus values at and around every rounding boundary, +-inf, NaN, huge values and
    signed zeros; slots -1 skip, one slot past the pool sets KV_DERR_BAD_SLOT."""
    T, Hh, D, NB, bs = 40, 3, 128, 7, 8
    rng = np.random.default_rng(group)
    k = W.normal_bits(9, group, (T, Hh, D), dtype)
    v = W.normal_bits(9, group + 1, (T, Hh, D), dtype)
    ks = rng.uniform(0.05, 0.9, (Hh, D // group)).astype(np.float32)
    vs = rng.uniform(0.05, 0.9, (Hh, D // group)).astype(np.float32)
    ks[0, 0] = vs[0, 0] = 1.0                       # so the specials below land exactly
    specials = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 6.5, 7.5, -7.5, -8.5, 7.49, -8.49,
                         np.inf, -np.inf, np.nan, 1e30, -1e30, 0.0, -0.0, 3.0, -3.0], np.float32)
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    sp_bits = torch.from_numpy(specials).to(tdt).view(torch.int16).numpy().view(np.uint16)
    n = min(len(sp_bits), group)
    k[0, 0, :n] = sp_bits[:n]
    v[0, 0, :n] = sp_bits[:n]
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = -1
    slots[5] = NB * bs                              # past the pool
    okc = oracle.cache_zeros(NB, bs, Hh, D, "int4")
    ovc = oracle.cache_zeros(NB, bs, Hh, D, "int4")
    oslots = np.where(slots >= NB * bs, -1, slots)
    assert oracle.reshape_and_cache_int4(k, v, dtype, oslots, okc, ovc, bs, ks, vs, group) == 0
    kc = torch.zeros((NB, bs, Hh, D // 2), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.reshape_and_cache_int4(H.to_dev(k, dtype), H.to_dev(v, dtype), torch.from_numpy(slots).cuda(),
                              kc, vc, torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(), d_err=err)
    torch.cuda.synchronize()
    assert err.item() == kv.KV_DERR_BAD_SLOT
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


# ---------------------------------------------------------------- attention

SMALL = {
    "llama3_8b_int4_small": W.LLAMA3_8B_INT4.replace(num_seqs=5, lengths=("uniform", 100, 1500)),
    "int4_spec_window": _spec(num_q_heads=32, num_kv_heads=8, q_len=4, windows=(0, 200),
                              lengths=("lognormal", 300, 1.0, 64, 3000), num_seqs=8),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("num_workers", [0, 7])
def test_small_configs_match_oracle(kv, name, num_workers):
    wl = W.make_workload(SMALL[name])
    for layer in wl.layers:
        g, o = _run_both(wl, layer, num_workers)
        _check_all(wl, g, o)


@pytest.mark.parametrize("bs", [4, 8, 16, 32])
@pytest.mark.parametrize("group", [8, 16, 32, 64, 128])
def test_block_sizes_and_groups(kv, bs, group):
    wl = W.make_workload(_spec(block_size=bs, group_size=group,
                               lengths=("fixed", (1, 2 * bs + 1, 9 * bs - 3, 40 * bs))))
    g, o = _run_both(wl, wl.layers[0], num_workers=13)
    _check_all(wl, g, o)


@pytest.mark.parametrize("Hq,Hkv,ql,dtype", [(8, 8, 1, "bf16"), (8, 1, 1, "f16"), (32, 4, 8, "bf16"),
                                             (16, 2, 5, "f16"), (12, 4, 3, "bf16"), (64, 8, 1, "bf16")])
def test_gqa_groups_and_speculative_lengths(kv, Hq, Hkv, ql, dtype):
    wl = W.make_workload(_spec(num_q_heads=Hq, num_kv_heads=Hkv, q_len=ql, dtype=dtype,
                               lengths=("fixed", (ql, ql + 16, 333, 1000))))
    g, o = _run_both(wl, wl.layers[0])
    _check_all(wl, g, o)


@pytest.mark.parametrize("window", [1, 16, 100])
def test_sliding_windows(kv, window):
    wl = W.make_workload(_spec(q_len=4, lengths=("fixed", (4, 50, 333, 2000)), windows=(window,)))
    g, o = _run_both(wl, wl.layers[0], num_workers=5)
    _check_all(wl, g, o)


def test_worker_count_invariance(kv):
    wl = W.make_workload(_spec(lengths=("fixed", (2000, 1500, 999, 3))))
    layer = wl.layers[0]
    outs = []
    for workers in (1, 2, 64, 1000, 0):
        kc, vc = H.gpu_fill_cache(wl, layer)
        g = H.gpu_step(wl, layer, kc, vc, num_workers=workers)
        assert g.err == 0
        outs.append(g.out.float())
    o = H.oracle_step(wl, layer)
    for x in outs:
        assert (x - outs[0]).abs().max().item() <= 1e-2 * outs[0].abs().max().item()
    H.check_attention(wl, g, o)


def test_full_size_every_row(kv):
    """The benchmarked INT4 batch (256 sequences of U{512..8192}) in the benchmark's launch
    configuration: every output and lse row against the oracle, the slot mapping, and the whole
    cache bit for bit."""
    wl = W.make_workload(W.LLAMA3_8B_INT4)
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = H.gpu_step(wl, layer, kc, vc)
    assert g.err == 0
    o = H.oracle_step(wl, layer)
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    H.check_whole_cache(g, o)
    H.check_attention(wl, g, o)


# ---------------------------------------------------------------- the one-launch step

FUSED = {
    "llama3_8b_int4_small": W.LLAMA3_8B_INT4.replace(num_seqs=5, lengths=("uniform", 100, 1500)),
    "spec_window": _spec(num_q_heads=32, num_kv_heads=8, q_len=4, windows=(0, 200),
                         lengths=("lognormal", 300, 1.0, 64, 3000), num_seqs=8),
    "bs8_g16": _spec(block_size=8, group_size=16, lengths=("fixed", (3, 17, 71, 400))),
    "mqa_bs32": _spec(num_q_heads=8, num_kv_heads=1, block_size=32, dtype="f16",
                      lengths=("fixed", (1, 33, 65, 129))),
}


@pytest.mark.parametrize("name", list(FUSED))
@pytest.mark.parametrize("num_workers", [0, 7, 1000])
def test_fused_step_equals_the_calls(kv, name, num_workers):
    """kv_decode_step_int4 gives the three calls' slots, caches, outputs and lse bit for bit."""
    wl = W.make_workload(FUSED[name])
    for layer in wl.layers:
        kc, vc = H.gpu_fill_cache(wl, layer)
        sep = H.gpu_step(wl, layer, kc, vc, num_workers=num_workers)
        kc2, vc2 = H.gpu_fill_cache(wl, layer)
        fus = H.gpu_step_fused(wl, layer, kc2, vc2, num_workers=num_workers)
        assert fus.err == sep.err == 0
        assert torch.equal(fus.slots, sep.slots)
        assert torch.equal(kc2, kc) and torch.equal(vc2, vc)
        assert torch.equal(fus.out, sep.out) and torch.equal(fus.lse, sep.lse)


def test_fused_step_matches_oracle_full_size(kv):
    wl = W.make_workload(W.LLAMA3_8B_INT4)
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = H.gpu_step_fused(wl, layer, kc, vc)
    assert g.err == 0
    o = H.oracle_step(wl, layer)
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    H.check_whole_cache(g, o)
    H.check_attention(wl, g, o)


def test_bad_lengths_give_zero_rows(kv):
    wl = W.make_workload(_spec(q_len=2, lengths=("fixed", (10, 300, 40, 64))))
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    ks, vs = H.int4_scales(layer)
    bt = torch.from_numpy(wl.block_table).cuda()
    bt[1, 3] = -7
    L = torch.from_numpy(wl.seq_lens).cuda()
    L[2] = 1
    q = H.to_dev(layer.q, "bf16")
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_attention_decode_int4(q, kc, vc, bt, L, wl.max_seq_len, 2, 0.1, ks, vs,
                                         lse_out=lse, d_err=err)
    torch.cuda.synchronize()
    assert err.item() & kv.KV_DERR_BAD_BLOCK and err.item() & kv.KV_DERR_BAD_LEN
    assert torch.isfinite(out).all()
    assert (out[4:6] == 0).all() and torch.isneginf(lse[4:6]).all()


def test_host_errors(kv):
    wl = W.make_workload(_spec())
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    ks, vs = H.int4_scales(layer)
    q = H.to_dev(layer.q, "bf16")
    bt = torch.from_numpy(wl.block_table).cuda()
    L = torch.from_numpy(wl.seq_lens).cuda()
    bad = torch.ones(2, 10, dtype=torch.float32, device="cuda")     # group size 12.8 -> 12
    with pytest.raises(kv.KVError) as e:
        kv.paged_attention_decode_int4(q, kc, vc, bt, L, wl.max_seq_len, 1, 0.1, bad, bad)
    assert e.value.status == kv.KV_ERR_UNSUPPORTED
    rc = kv.lib.kv_reshape_and_cache(q.data_ptr(), q.data_ptr(), 1, 1024, 1024, 1, 2, 128, bt.data_ptr(),
                                     kc.data_ptr(), vc.data_ptr(), kv.KV_INT4, wl.num_blocks, 16,
                                     1.0, 1.0, None, None)
    assert rc == kv.KV_ERR_UNSUPPORTED               # INT4 has its own cache-write call
    rc = kv.lib.kv_paged_attention_decode(
        q.data_ptr(), 1, 4, 1, 8, kc.data_ptr(), vc.data_ptr(), kv.KV_INT4, 2, 128, 16, wl.num_blocks,
        bt.data_ptr(), bt.stride(0), bt.shape[1], L.data_ptr(), 300, 0.1, 0, 1.0, 1.0, 0,
        None, 0, q.data_ptr(), None, None, None)
    assert rc == kv.KV_ERR_UNSUPPORTED


@pytest.mark.parametrize("cache", ["int4", "bf16"])
@pytest.mark.parametrize("lengths", [(37,), (1, 40, 300), (5, 17, 33, 64, 100, 129, 250, 700)])
def test_small_batches_default_workers(kv, cache, lengths):
    """1, 3 and 8 sequences with the default worker count (eight INT4 workers a CTA, one
    16-bit worker a CTA, on every SM): far more workers than stages, so only as many shares as
    stages are cut and every sequence is split into at most as many pieces as it has stages.
    Every row against the oracle, and the attention call's plan agrees."""
    kw = dict(lengths=("fixed", lengths), num_seqs=len(lengths))
    if cache == "bf16":
        kw.update(cache_dtype="bf16", group_size=0)
    wl = W.make_workload(_spec(**kw))
    layer = wl.layers[0]
    g, o = _run_both(wl, layer)
    assert g.err == 0
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    H.check_whole_cache(g, o)
    H.check_attention(wl, g, o)
    info = kv.paged_attention_plan_info(len(lengths), 1, 8, 2, 128, 16, kv.KV_INT4 if cache == "int4" else kv.KV_BF16,
                                        wl.max_seq_len)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert info["ctas"] == sms
