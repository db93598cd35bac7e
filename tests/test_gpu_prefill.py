"""Chunked-prefill attention (kv_paged_attention_prefill, tcgen05) against the oracle's varlen
attention, element by element at the stated tolerance: whole prompts, chunks after a cached
context, single tokens and empty chunks in one batch; several query and key tiles with ragged
tails; GQA groups of 1, 2, 4, 8, 16 and 32; block sizes 8, 16, 32; windows (with the entries of
blocks that left every query's window set to -1, which must never be read)."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_block_gb300 import workloads as W

from .harness import LSE_TOL, TOL, out_ulp, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kc():
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


def make_case(seed, contexts, chunks, Hq, Hkv, bs, dtype, window=0, D=128):
    rng = np.random.default_rng(seed)
    L = np.array([c + n for c, n in zip(contexts, chunks)], np.int32)
    nblk = -(-L // bs)
    NB = int(nblk.sum()) + 7
    width = int(nblk.max()) + 2
    perm = rng.permutation(NB).astype(np.int32)
    table = np.full((len(L), width), -1, np.int32)
    o = 0
    for b in range(len(L)):
        table[b, :nblk[b]] = perm[o:o + nblk[b]]
        o += nblk[b]
        if window > 0:  # blocks no query of the chunk can see may have gone back to the pool
            first_key = max(0, int(L[b]) - chunks[b] - window + 1)
            table[b, :first_key // bs] = -1
    qsl = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(qsl[-1])
    q = W.normal_bits(seed, 1, (T, Hq, D), dtype)
    kcache = W.normal_bits(seed, 2, (NB, bs, Hkv, D), dtype)
    vcache = W.normal_bits(seed, 3, (NB, bs, Hkv, D), dtype)
    return dict(L=L, table=table, qsl=qsl, q=q, k=kcache, v=vcache, NB=NB, bs=bs, dtype=dtype,
                window=window, chunks=chunks, D=D)


def run_gpu(kc, c, scale):
    dev = "cuda"
    q = to_dev(c["q"], c["dtype"], dev)
    k = to_dev(c["k"], c["dtype"], dev)
    v = to_dev(c["v"], c["dtype"], dev)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kc.paged_attention_prefill(q, k, v, torch.from_numpy(c["table"]).to(dev), torch.from_numpy(c["L"]).to(dev),
                               torch.from_numpy(c["qsl"]).to(dev), int(c["L"].max()), max(c["chunks"]),
                               scale, c["window"], out=out, lse_out=lse, d_err=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), int(err.item())


def check(c, out, lse, ref_out, ref_lse):
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=LSE_TOL)
    diff = np.abs(out - ref_out)
    allowed = TOL[c["dtype"]] + 0.5 * out_ulp(ref_out, c["dtype"])
    worst = np.unravel_index(np.argmax(diff - allowed), diff.shape)
    assert (diff <= allowed).all(), (f"error {diff[worst]:.3e} at {worst} (oracle {ref_out[worst]:.5f}), "
                                     f"max abs error {diff.max():.3e}")
    return float(diff.max())


CASES = [
    # (contexts, chunks, Hq, Hkv, bs, dtype, window)
    ([0, 500, 1000, 7, 130], [300, 77, 1, 0, 128], 8, 2, 16, "bf16", 0),
    ([0, 260], [257, 33], 4, 4, 8, "f16", 0),
    ([64, 0, 1900], [200, 129, 64], 32, 4, 32, "bf16", 0),
    ([0, 2000, 333], [300, 64, 40], 16, 2, 16, "bf16", 100),
    ([5, 700], [250, 130], 8, 8, 16, "f16", 257),
    ([0], [1024], 64, 8, 16, "bf16", 0),
    ([0, 300], [200, 57], 32, 2, 16, "bf16", 0),      # g 16: 8 tokens a Q tile
    ([100, 0], [129, 300], 8, 4, 8, "f16", 0),        # g 2: 64 tokens a Q tile
    ([50, 900], [77, 40], 32, 1, 16, "bf16", 150),    # g 32: 4 tokens a Q tile, with a window
]


@pytest.mark.parametrize("case", CASES, ids=lambda x: f"{x[5]}_g{x[2]//x[3]}_bs{x[4]}_w{x[6]}")
def test_prefill_matches_oracle(kc, case):
    contexts, chunks, Hq, Hkv, bs, dtype, window = case
    c = make_case(sum(contexts) + 7 * sum(chunks) + Hq + bs, contexts, chunks, Hq, Hkv, bs,
                  dtype, window)
    scale = 1.0 / math.sqrt(128)
    out, lse, err = run_gpu(kc, c, scale)
    assert err == 0
    ref_out, ref_lse = oracle.paged_attention_varlen(c["q"], dtype, c["k"], c["v"], dtype, c["table"], c["L"],
                                                     c["qsl"], scale, window)
    check(c, out, lse, ref_out, ref_lse)


def test_prefill_rejected_length_rows_are_zero(kc):
    c = make_case(5, [10, 40], [20, 30], 8, 2, 16, "bf16")
    c["L"] = c["L"].copy()
    c["L"][0] = 5  # fewer tokens than query rows: rejected
    out, lse, err = run_gpu(kc, c, 0.1)
    assert err & 16
    assert (out[:20] == 0).all() and np.isneginf(lse[:20]).all()
    ref_out, ref_lse = oracle.paged_attention_varlen(c["q"], "bf16", c["k"], c["v"], "bf16", c["table"],
                                                     c["L"], c["qsl"], 0.1, 0, seqs=[1])
    check(c, out[20:], lse[20:], ref_out[20:], ref_lse[20:])


@pytest.mark.parametrize("name", ["prefill_llama3_8b", "prefill_prompt_llama3_8b"])
def test_prefill_full_size_every_row(kc, name):
    """The benchmark's chunked-prefill batches (16 sequences, 1024-token chunks after up to 7168
    cached tokens; 8 whole 2048-token prompts; Llama-3-8B attention shape): every output and lse
    row against the oracle."""
    from paged_kv_cache_block_gb300 import workloads as W
    pw = W.make_prefill(W.PREFILL_BY_NAME[name])
    s = pw.spec
    shape = (pw.num_blocks, s.block_size, s.num_kv_heads, s.head_dim)
    q = to_dev(pw.q, s.dtype)
    kcache = to_dev(pw.pool_k, s.dtype).view(shape)
    vcache = to_dev(pw.pool_v, s.dtype).view(shape)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kc.paged_attention_prefill(q, kcache, vcache, torch.from_numpy(pw.block_table).cuda(),
                                     torch.from_numpy(pw.seq_lens).cuda(),
                                     torch.from_numpy(pw.query_start_loc).cuda(), int(pw.seq_lens.max()),
                                     int(pw.chunks.max()), s.softmax_scale, s.window, lse_out=lse, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    NB, bs = pw.num_blocks, s.block_size
    ref_out, ref_lse = oracle.paged_attention_varlen(
        pw.q, s.dtype, pw.pool_k.reshape(NB, bs, s.num_kv_heads, s.head_dim),
        pw.pool_v.reshape(NB, bs, s.num_kv_heads, s.head_dim), s.dtype, pw.block_table, pw.seq_lens,
        pw.query_start_loc, s.softmax_scale, s.window)
    c = dict(dtype=s.dtype)
    check(c, o, l, ref_out, ref_lse)
