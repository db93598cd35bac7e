"""The library's C++ block manager (kv_bm_*) against the block manager oracle, on the CPU: the
same seeded traces of allocations, frees, prefix shares and flushes must give the same statuses,
rows, reference counts, free-pool sizes and flushed writes, bit for bit."""
import random

import numpy as np
import pytest

from oracle import block_manager as bmo


@pytest.fixture(scope="module")
def kc():
    from paged_kv_cache_block_gb300 import build
    build.build()
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


def same_state(kc, lib_bm, ora):
    assert lib_bm.num_free_blocks() == ora.num_free()
    for r in range(ora.num_rows):
        t, blocks = lib_bm.row(r)
        assert t == ora.tokens[r], f"row {r}"
        assert blocks == ora.rows[r], f"row {r}"
    refs = [lib_bm.ref_count(b) for b in range(ora.num_blocks)]
    assert refs == ora.ref
    assert lib_bm.ref_count(-1) == -1 and lib_bm.ref_count(ora.num_blocks) == -1


def run_trace(kc, seed, steps, window, zero_fill):
    rng = random.Random(seed)
    bs = rng.choice([1, 4, 8, 16])
    nb = rng.randint(16, 96)
    rows = rng.randint(2, 9)
    mb = rng.choice([8, 24, 64])
    lib_bm = kc.BlockManager(nb, bs, rows, mb, window=window, zero_fill=zero_fill)
    ora = bmo.BlockManager(nb, bs, rows, mb, window=window, zero_fill=zero_fill)
    for _ in range(steps):
        u = rng.random()
        r = rng.randrange(-1, rows + 1)  # rows -1 and `rows` are invalid on purpose
        if u < 0.45:
            n = rng.choice([0, 1, 1, 1, 2, 3, 5, 17, 40, 130, -1])
            assert lib_bm.allocate(r, n) == ora.allocate(r, n)
        elif u < 0.55:
            k = rng.randint(1, 6)
            rs = [rng.randrange(rows) for _ in range(k)]
            ns = [rng.choice([1, 1, 2, 9]) for _ in range(k)]
            st = lib_bm.allocate_batch(rs, ns)
            assert st.tolist() == [ora.allocate(a, b) for a, b in zip(rs, ns)]
        elif u < 0.67:
            assert lib_bm.free(r) == ora.free(r)
        elif u < 0.85:
            src = rng.randrange(-1, rows + 1)
            k = rng.choice([0, 1, 2, 3, 6, 20])
            assert lib_bm.share_prefix(r, src, k) == ora.share(r, src, k)
        else:
            nu, nz = lib_bm.pending()
            up, zero = lib_bm.flush()
            oup, ozero = ora.flush()
            assert (nu, nz) == (len(oup), len(ozero))
            assert np.array_equal(up, oup)
            assert np.array_equal(zero, ozero)
        same_state(kc, lib_bm, ora)


@pytest.mark.parametrize("window", [0, 5, 16, 33])
@pytest.mark.parametrize("zero_fill", [True, False])
def test_random_traces_match_oracle(kc, window, zero_fill):
    for seed in range(12):
        run_trace(kc, 1000 * window + seed + (7 if zero_fill else 0), 250, window, zero_fill)


def test_flush_capacity_and_bad_arguments(kc):
    bm = kc.BlockManager(8, 4, 2, 4)
    assert bm.allocate(0, 9) == kc.KV_OK
    up = np.empty((2, 3), np.int32)
    with pytest.raises(kc.KVError) as e:
        bm.flush(updates=up)
    assert e.value.status == kc.KV_ERR_WORKSPACE
    assert bm.pending() == (3, 3)  # nothing was handed out
    u, z = bm.flush()
    assert u.tolist() == [[0, 0, 0], [0, 1, 1], [0, 2, 2]] and z.tolist() == [0, 1, 2]
    assert bm.pending() == (0, 0)
    with pytest.raises(kc.KVError):
        kc.BlockManager(0, 4, 2, 4)
    assert bm.allocate(0, 8) == kc.KV_ERR_INVALID_ARG  # 17 tokens > 4 blocks of 4
    assert b"would need" in kc.lib.kv_last_error()
    small = kc.BlockManager(4, 4, 2, 4)
    assert small.allocate(0, 12) == kc.KV_OK
    assert small.allocate(1, 5) == kc.KV_ERR_OUT_OF_BLOCKS  # 2 blocks needed, 1 free
    assert b"1 free" in kc.lib.kv_last_error()
    assert small.row(1) == (0, []) and small.num_free_blocks() == 1


def test_serving_shape_trace_matches_oracle(kc):
    """A decode-shaped trace at scale: 256 rows with prompts, one token a step, requests ending
    and new ones sharing a 64-block prompt prefix, window 4096 on a second manager."""
    rng = random.Random(7)
    for window in (0, 4096):
        nb, bs, rows, mb = 70000, 16, 256, 1024
        lib_bm = kc.BlockManager(nb, bs, rows, mb, window=window)
        ora = bmo.BlockManager(nb, bs, rows, mb, window=window)
        assert lib_bm.allocate(0, 1024 + 5) == ora.allocate(0, 1024 + 5) == 0
        for r in range(1, rows):
            if r % 4 == 0:
                assert lib_bm.share_prefix(r, 0, 64) == ora.share(r, 0, 64) == 0
            n = rng.randint(16, 3000)
            assert lib_bm.allocate(r, n) == ora.allocate(r, n)
        for step in range(60):
            rs = list(range(rows))
            st = lib_bm.allocate_batch(rs, [1] * rows)
            assert st.tolist() == [ora.allocate(r, 1) for r in rs]
            if step % 10 == 9:
                r = rng.randrange(1, rows)
                assert lib_bm.free(r) == ora.free(r)
                assert lib_bm.share_prefix(r, 0, 64) == ora.share(r, 0, 64)
            up, zero = lib_bm.flush()
            oup, ozero = ora.flush()
            assert np.array_equal(up, oup) and np.array_equal(zero, ozero)
        same_state(kc, lib_bm, ora)
