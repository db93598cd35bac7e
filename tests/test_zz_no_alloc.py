"""kv_paged_attention_decode_noalloc, the decode entry point that allocates nothing, against
kv_paged_attention_decode with a caller-provided workspace, through the C ABI.

Some callers cannot allocate device memory: a plugin inside a framework that owns every device
allocation, a real-time decode loop where cudaMalloc could synchronise the device or fail, a C
caller with no allocator.  The no-alloc entry point takes inputs and outputs only and uses a
static scratch array inside the library.  Calls in a row (different batches, so each finds the
previous one's scratch contents) must each equal the workspace entry point bit for bit.  This
file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_block_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


def _batch(kv, spec):
    """A decode batch on the GPU: pool written into the cache, then this step's slot mapping and
    cache write of the new K/V rows (as the oracle does)."""
    wl = W.make_workload(spec)
    layer = wl.layers[0]
    s = wl.spec
    kc, vc = H.gpu_fill_cache(wl, layer)
    bt = torch.from_numpy(wl.block_table).cuda()
    slots = kv.compute_slot_mapping(bt, torch.from_numpy(wl.query_start_loc).cuda(),
                                    torch.from_numpy(wl.positions).cuda(), s.block_size, wl.num_blocks)
    kv.reshape_and_cache(H.to_dev(layer.new_k, s.dtype), H.to_dev(layer.new_v, s.dtype), slots, kc, vc,
                         layer.k_scale, layer.v_scale)
    dev = dict(q=H.to_dev(layer.q, s.dtype), kc=kc, vc=vc, bt=bt, L=torch.from_numpy(wl.seq_lens).cuda())
    return wl, layer, dev


# more stream-K workers than the batches below have (kv-head group, sequence) items: with every
# share non-empty, some item must then span two shares, so its rows go through the scratch array
# (partial results and log-sum-exp values) and the merge kernel
WORKERS = 40


def _both(kv, wl, layer, d):
    s = wl.spec
    args = (d["q"], d["kc"], d["vc"], d["bt"], d["L"], wl.max_seq_len, s.q_len, s.softmax_scale,
            layer.window, layer.k_scale, layer.v_scale)
    T, Hq = d["q"].shape[0], d["q"].shape[1]
    ref_lse = torch.empty(T, Hq, dtype=torch.float32, device="cuda")
    ref = kv.paged_attention_decode(*args, num_workers=WORKERS, lse_out=ref_lse)
    out = torch.empty_like(d["q"])
    lse = torch.empty(T, Hq, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = kv.lib.kv_paged_attention_decode_noalloc(
        d["q"].data_ptr(), kv.dtype_code(d["q"].dtype), s.num_seqs, s.q_len, Hq,
        d["kc"].data_ptr(), d["vc"].data_ptr(), kv.dtype_code(d["kc"].dtype), s.num_kv_heads,
        s.head_dim, s.block_size, wl.num_blocks, d["bt"].data_ptr(), d["bt"].stride(0),
        d["bt"].shape[1], d["L"].data_ptr(), wl.max_seq_len, s.softmax_scale, layer.window,
        layer.k_scale, layer.v_scale, WORKERS, out.data_ptr(), lse.data_ptr(), err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0, kv.lib.kv_last_error().decode()
    assert err.item() == 0
    return ref, ref_lse, out, lse


def _check(kv, wl, layer, d):
    ref, ref_lse, out, lse = _both(kv, wl, layer, d)
    # the same kernels with the same launch plan: the outputs are equal bit for bit
    assert torch.equal(out, ref)
    assert torch.equal(lse, ref_lse)
    # and both agree with the oracle on a few sequences
    seqs = [0, wl.spec.num_seqs - 1]
    o = H.oracle_step(wl, layer, seqs=seqs)
    g = H.GpuStep(None, None, None, out, lse, 0)
    H.check_attention(wl, g, o, rows=H.rows_of(wl, seqs))


def test_noalloc_matches_workspace_entry_point_on_two_calls(kv):
    # a 12-sequence batch, then a smaller one (10 sequences, fewer items and stages, so the scratch
    # still holds the first call's partial results past what the second writes), then the first
    # batch again after the second
    big = _batch(kv, W.LLAMA3_8B.replace(num_seqs=12, lengths=("uniform", 200, 3000)))
    small = _batch(kv, W.MISTRAL_HYBRID.replace(num_seqs=10, lengths=("lognormal", 400, 1.0, 64, 4000),
                                                shared_prefix_tokens=256, windows=(300,)))
    for wl, layer, d in (big, small, big):
        _check(kv, wl, layer, d)


def test_noalloc_rejects_sizes_beyond_its_scratch(kv):
    # 3000 sequences of a 32/8-head layer need more than the 32 MiB of static scratch
    B, Hq, Hkv, D, bs = 3000, 32, 8, 128, 16
    need = kv.paged_attention_workspace_size(B, 1, Hq, Hkv, D, bs, kv.KV_BF16, 64)
    assert need > 32 << 20
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(8, bs, Hkv, D, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(B, 4, dtype=torch.int32, device="cuda")
    L = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    with pytest.raises(kv.KVError) as e:
        kv.paged_attention_decode_noalloc(q, kc, kc, bt, L, 64, 1, 0.1, out=out)
    assert e.value.status == 4 and "static scratch" in str(e.value)
    torch.cuda.synchronize()
    assert (out == 7.0).all()          # nothing was launched
