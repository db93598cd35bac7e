"""The block manager's device side and a whole serving loop against the oracle.

kv_apply_block_updates (block-table writes + zero fill of new blocks) is compared with the
oracle's apply_updates bit for bit; a multi-step serving loop - requests admitted with their
prompt K/V, prefixes shared, one (or several speculative) tokens decoded per step, requests
ending and their rows reused, a sliding window releasing blocks - runs the library's C++ block
manager + kv_apply_block_updates + kv_decode_step on the GPU and the oracle's block manager +
cache write + attention on the CPU, comparing block tables and whole caches bit for bit and
attention at the stated tolerance after every step.
"""
import random
import zlib
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
from oracle import block_manager as bmo
from paged_kv_cache_block_gb300 import workloads as W

from .harness import TORCH_DT, cache_bits, check_attention, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kc():
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


def random_cache_bits(rng: np.random.Generator, shape, cache_dtype):
    if cache_dtype == "e4m3":
        return rng.integers(0, 256, size=shape, dtype=np.uint8)
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


def dev_cache(bits: np.ndarray, cache_dtype: str) -> torch.Tensor:
    if cache_dtype == "e4m3":
        return torch.from_numpy(bits.copy()).cuda()
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(TORCH_DT[cache_dtype])


# ------------------------------------------------------------------------- apply_block_updates

GEOMETRIES = [  # (block_size, kv heads, head dim, cache dtype, caches): block bytes 1 KB .. 64 KB
    (4, 2, 64, "f16", 2),
    (16, 12, 64, "f16", 3),     # 24 KB: a 16 KB and an 8 KB chunk
    (16, 8, 128, "e4m3", 4),    # exactly one 16 KB chunk
    (16, 8, 128, "bf16", 6),    # 32 KB
    (32, 8, 128, "bf16", 2),    # 64 KB
]


@pytest.mark.parametrize("geom", GEOMETRIES, ids=lambda g: f"bs{g[0]}_h{g[1]}_d{g[2]}_{g[3]}_x{g[4]}")
def test_apply_updates_matches_oracle(kc, geom):
    bs, H, D, cdt, ncache = geom
    NB, rows, stride, maxb = 97, 7, 40, 33
    rng = np.random.default_rng(zlib.crc32(repr(geom).encode()))
    caches_np = [random_cache_bits(rng, (NB, bs, H, D), cdt) for _ in range(ncache)]
    table_np = rng.integers(-1, NB, size=(rows, stride), dtype=np.int32)
    # staged writes from a block manager trace, plus entries the kernel must refuse
    bm = bmo.BlockManager(NB, bs, rows, maxb, window=5)
    prng = random.Random(11)
    for _ in range(60):
        r = prng.randrange(rows)
        u = prng.random()
        if u < 0.6:
            bm.allocate(r, prng.choice([1, 3, 8, 20]) * max(1, bs // 4))
        elif u < 0.8:
            bm.free(r)
        else:
            bm.share(r, prng.randrange(rows), prng.randint(1, 3))
    ups, zero = bm.flush()
    assert len(ups) > 10 and len(zero) > 5
    bad = np.array([[rows, 0, 1], [0, maxb, 1], [1, 2, NB], [2, 1, -2], [-1, 0, 0]], np.int32)
    ups = np.concatenate([ups, bad])
    zero = np.concatenate([zero, np.array([NB, -1], np.int32)])

    exp_table = table_np.copy()
    exp_caches = [c.copy() for c in caches_np]
    exp_err = bmo.apply_updates(exp_table[:, :maxb], exp_caches, ups, zero, NB)
    assert exp_err == 32

    table = torch.from_numpy(table_np).cuda()
    caches = [dev_cache(c, cdt) for c in caches_np]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc.apply_block_updates(torch.from_numpy(ups).cuda(), table, torch.from_numpy(zero).cuda(),
                           caches, NB, d_err=err, max_blocks_per_row=maxb)
    torch.cuda.synchronize()
    assert int(err.item()) == exp_err
    assert np.array_equal(table.cpu().numpy(), exp_table)
    for c, e in zip(caches, exp_caches):
        assert np.array_equal(cache_bits(c), e)


def test_apply_updates_nothing_to_do_and_host_checks(kc):
    table = torch.full((2, 4), 7, dtype=torch.int32, device="cuda")
    cache = torch.ones((8, 16, 2, 64), dtype=torch.float16, device="cuda")
    empty = torch.zeros((0, 3), dtype=torch.int32, device="cuda")
    kc.apply_block_updates(empty, table, torch.zeros(0, dtype=torch.int32, device="cuda"), [cache], 8)
    torch.cuda.synchronize()
    assert (table == 7).all() and (cache == 1).all()
    bad = torch.empty(8 * 16 * 2 * 64 + 1, dtype=torch.float16, device="cuda")[1:].view(8, 16, 2, 64)
    with pytest.raises(kc.KVError) as e:  # a cache that is not 16-byte aligned
        kc.apply_block_updates(empty, table, torch.tensor([1], dtype=torch.int32, device="cuda"),
                               [bad], 8)
    assert e.value.status == kc.KV_ERR_INVALID_ARG


def test_apply_updates_full_size_admission(kc):
    """At the size the benchmark times (Llama-3-8B blocks: 16 tokens x 8 heads x 128 dims bf16,
    32 KB per cache; 2048 new blocks of a 8192-block pool, K and V): every listed block is zero,
    every other byte unchanged (checked on the device: too large for the oracle loop)."""
    NB, bs, H, D = 8192, 16, 8, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    k = torch.randint(1, 1 << 14, (NB, bs, H, D), dtype=torch.int16, device="cuda", generator=g)
    v = torch.randint(1, 1 << 14, (NB, bs, H, D), dtype=torch.int16, device="cuda", generator=g)
    k0, v0 = k.clone(), v.clone()
    ids = torch.randperm(NB, device="cuda", generator=g)[:2048].sort().values.to(torch.int32)
    table = torch.full((256, 1024), -1, dtype=torch.int32, device="cuda")
    ups = torch.stack([torch.arange(2048, device="cuda") // 8, torch.arange(2048, device="cuda") % 8,
                       ids.long()], 1).to(torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc.apply_block_updates(ups, table, ids, [k.view(torch.bfloat16), v.view(torch.bfloat16)], NB, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    mask = torch.zeros(NB, dtype=torch.bool, device="cuda")
    mask[ids.long()] = True
    assert (k[mask] == 0).all() and (v[mask] == 0).all()
    assert torch.equal(k[~mask], k0[~mask]) and torch.equal(v[~mask], v0[~mask])
    assert torch.equal(table[:256, :8].reshape(-1), ids)
    assert (table[:, 8:] == -1).all()


# ------------------------------------------------------------------------- serving loop


class Serving:
    """One attention layer served for several steps by both sides."""

    def __init__(self, kc, seed, dtype, cache_dtype, q_len, window, rows=10, NB=420, bs=16,
                 Hq=8, Hkv=2, D=128, maxb=64):
        self.kc, self.dtype, self.cdt, self.q_len, self.window = kc, dtype, cache_dtype, q_len, window
        self.rows, self.NB, self.bs, self.Hq, self.Hkv, self.D, self.maxb = rows, NB, bs, Hq, Hkv, D, maxb
        self.seed, self.stream = seed, 0
        self.rng = random.Random(seed)
        self.k_scale = self.v_scale = 0.05 if cache_dtype == "e4m3" else 1.0
        self.scale = 1.0 / np.sqrt(D)
        self.lib_bm = kc.BlockManager(NB, bs, rows, maxb, window=window)
        self.ora_bm = bmo.BlockManager(NB, bs, rows, maxb, window=window)
        init = random_cache_bits(np.random.default_rng(seed), (2, NB, bs, Hkv, D), cache_dtype)
        self.kc_np, self.vc_np = init[0].copy(), init[1].copy()
        self.k_dev, self.v_dev = dev_cache(self.kc_np, cache_dtype), dev_cache(self.vc_np, cache_dtype)
        self.table_np = np.full((rows, maxb), -1, np.int32)
        self.table_dev = torch.from_numpy(self.table_np).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def bits(self, shape):
        self.stream += 1
        return W.normal_bits(self.seed, self.stream, shape, self.dtype)

    def sync_tables(self):
        ups, zero = self.lib_bm.flush()
        oups, ozero = self.ora_bm.flush()
        assert np.array_equal(ups, oups) and np.array_equal(zero, ozero)
        assert bmo.apply_updates(self.table_np, [self.kc_np, self.vc_np], oups, ozero, self.NB) == 0
        self.kc.apply_block_updates(torch.from_numpy(np.ascontiguousarray(ups)).cuda(), self.table_dev,
                                    torch.from_numpy(np.ascontiguousarray(zero)).cuda(),
                                    [self.k_dev, self.v_dev], self.NB, d_err=self.err)

    def write_tokens(self, row, first, n):
        """K/V of positions first..first+n-1 of a row (a prompt), written by both sides."""
        k = self.bits((n, self.Hkv, self.D))
        v = self.bits((n, self.Hkv, self.D))
        qsl = np.array([0, n], np.int32)
        pos = np.arange(first, first + n, dtype=np.int32)
        slots, e = oracle.slot_mapping(self.table_np[row:row + 1], qsl, pos, self.bs, self.NB)
        assert e == 0
        assert oracle.reshape_and_cache(k, v, self.dtype, slots, self.kc_np, self.vc_np, self.cdt,
                                        self.bs, self.k_scale, self.v_scale) == 0
        kv = self.kc
        dslots = kv.compute_slot_mapping(self.table_dev[row:row + 1], torch.from_numpy(qsl).cuda(),
                                         torch.from_numpy(pos).cuda(), self.bs, self.NB, d_err=self.err)
        kv.reshape_and_cache(to_dev(k, self.dtype), to_dev(v, self.dtype), dslots, self.k_dev,
                             self.v_dev, self.k_scale, self.v_scale, d_err=self.err)

    def admit(self, row, share_from=None):
        """A new request in an empty row: optionally the first full blocks of another row's
        prompt, then its own prompt tokens."""
        first = 0
        if share_from is not None:
            t, _ = self.lib_bm.row(share_from)
            k = min(t // self.bs, self.rng.randint(1, 4))
            st = self.lib_bm.share_prefix(row, share_from, k)
            assert st == self.ora_bm.share(row, share_from, k)
            if st == 0:
                first = k * self.bs
        n = self.rng.randint(self.q_len, 300)
        st = self.lib_bm.allocate(row, n)
        assert st == self.ora_bm.allocate(row, n) == 0
        self.sync_tables()
        self.write_tokens(row, first, n)

    def decode(self):
        B, ql = self.rows, self.q_len
        st = self.lib_bm.allocate_batch(list(range(B)), [ql] * B)
        assert st.tolist() == [self.ora_bm.allocate(r, ql) for r in range(B)] == [0] * B
        self.sync_tables()
        L = np.array([self.ora_bm.tokens[r] for r in range(B)], np.int32)
        assert L.tolist() == [self.lib_bm.row(r)[0] for r in range(B)]
        pos = (L[:, None] - ql + np.arange(ql)[None, :]).reshape(-1).astype(np.int32)
        qsl = (np.arange(B + 1) * ql).astype(np.int32)
        k = self.bits((B * ql, self.Hkv, self.D))
        v = self.bits((B * ql, self.Hkv, self.D))
        q = self.bits((B * ql, self.Hq, self.D))
        # oracle
        slots, e = oracle.slot_mapping(self.table_np, qsl, pos, self.bs, self.NB)
        assert e == 0
        assert oracle.reshape_and_cache(k, v, self.dtype, slots, self.kc_np, self.vc_np, self.cdt,
                                        self.bs, self.k_scale, self.v_scale) == 0
        ref_out, ref_lse = oracle.paged_attention(q, self.dtype, self.kc_np, self.vc_np, self.cdt,
                                                  self.table_np, L, ql, self.scale, self.window,
                                                  self.k_scale, self.v_scale)
        # library
        kv = self.kc
        lse = torch.empty(B * ql, self.Hq, dtype=torch.float32, device="cuda")
        out = kv.decode_step(self.table_dev, torch.from_numpy(qsl).cuda(), torch.from_numpy(pos).cuda(),
                             to_dev(k, self.dtype), to_dev(v, self.dtype), to_dev(q, self.dtype),
                             self.k_dev, self.v_dev, torch.from_numpy(L).cuda(), int(L.max()), ql,
                             self.scale, self.window, self.k_scale, self.v_scale, lse_out=lse,
                             d_err=self.err)
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0
        assert np.array_equal(self.table_dev.cpu().numpy(), self.table_np)
        assert np.array_equal(cache_bits(self.k_dev), self.kc_np)
        assert np.array_equal(cache_bits(self.v_dev), self.vc_np)
        spec = SimpleNamespace(spec=SimpleNamespace(dtype=self.dtype, cache_dtype=self.cdt))
        check_attention(spec, SimpleNamespace(out=out, lse=lse), SimpleNamespace(out=ref_out, lse=ref_lse))


@pytest.mark.parametrize("dtype,cdt,q_len,window", [
    ("bf16", "bf16", 1, 0),
    ("bf16", "bf16", 1, 40),
    ("f16", "f16", 3, 37),
    ("bf16", "e4m3", 1, 0),
    ("f16", "f16", 2, 0),
])
def test_serving_loop_matches_oracle(kc, dtype, cdt, q_len, window):
    sv = Serving(kc, seed=300 + q_len * 7 + window, dtype=dtype, cache_dtype=cdt, q_len=q_len,
                 window=window)
    for r in range(sv.rows):
        sv.admit(r, share_from=(r - 1) if r % 3 == 2 else None)
    for step in range(14):
        sv.decode()
        if step % 3 == 2:  # a request ends; a new one takes its row, sometimes sharing a prefix
            r = sv.rng.randrange(sv.rows)
            assert sv.lib_bm.free(r) == sv.ora_bm.free(r) == 0
            src = (r + 1) % sv.rows
            sv.admit(r, share_from=src if step % 2 == 0 else None)
    assert sv.lib_bm.num_free_blocks() == sv.ora_bm.num_free()
    if window:
        # the window returned blocks: every row holds at most ceil((W + q_len - 1) / bs) + 1
        for r in range(sv.rows):
            live = [b for b in sv.lib_bm.row(r)[1] if b >= 0]
            assert len(live) <= -(-(window + q_len - 1) // sv.bs) + 1
