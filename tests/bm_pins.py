"""Pins of the block manager oracle, written as functions of the oracle module so that the same
checks run against the oracle and against copies of it with planted mistakes.

Each pin rests on something other than the oracle: a worked example printed on the pages, a
brute-force enumeration, or a conservation law any correct allocator obeys.
"""
from __future__ import annotations

import random

import numpy as np

# ---------------------------------------------------------------------------------------------
# brute-force checks of a manager's state


def check_conservation(bm) -> None:
    """Every block's count equals the number of table entries that name it; the free pool holds
    exactly the blocks nobody names, each once."""
    named = {}
    for row in bm.rows:
        for b in row:
            if b >= 0:
                named[b] = named.get(b, 0) + 1
    for b in range(bm.num_blocks):
        assert bm.ref[b] == named.get(b, 0), f"block {b}: count {bm.ref[b]}, named {named.get(b, 0)}"
    pool = list(bm.free_pool)
    assert len(pool) == len(set(pool)), "a block sits in the free pool twice"
    assert set(pool) == {b for b in range(bm.num_blocks) if b not in named}


def check_row_shape(bm) -> None:
    """A row holding T tokens has exactly ceil(T / block_size) logical blocks, and with a window
    its live ones are exactly the blocks of positions max(0, T_last - W + 1) .. T - 1 at most."""
    for r, row in enumerate(bm.rows):
        T = bm.tokens[r]
        assert len(row) == -(-T // bm.block_size)
        if bm.window <= 0:
            assert all(b >= 0 for b in row)


def window_live_blocks(first_query: int, num_tokens: int, window: int, block_size: int) -> set:
    """Brute force: the logical blocks that some query at positions first_query..num_tokens-1
    can read under a window (keys p - W < j <= p)."""
    live = set()
    for p in range(first_query, num_tokens):
        for j in range(max(0, p - window + 1), p + 1):
            live.add(j // block_size)
    return live


# ---------------------------------------------------------------------------------------------
# pins


def pin_48_tokens_three_blocks(mod) -> None:
    """"vLLM Worker侧...", section "调度视角": 48 computed tokens at block size 16 occupy 3
    logical blocks; the pool loses exactly 3."""
    assert mod.blocks_for_tokens(48, 16) == 3
    bm = mod.BlockManager(num_blocks=10, block_size=16, num_rows=2, max_blocks_per_row=8)
    assert bm.allocate(0, 48) == mod.OK
    assert len(bm.rows[0]) == 3 and bm.num_free() == 7
    assert bm.allocate(0, 0) == mod.OK and len(bm.rows[0]) == 3
    assert bm.allocate(0, 1) == mod.OK and len(bm.rows[0]) == 4  # token 48 opens a fourth
    check_conservation(bm)


def pin_block_of_four_lazy(mod) -> None:
    """"Understanding PageAttention Memory Optimization": with 4-token blocks a new block is
    taken only when the current one is full - "fathers brought a car" fills one block, the
    next token opens a second one, wherever the pool finds it."""
    bm = mod.BlockManager(num_blocks=6, block_size=4, num_rows=3, max_blocks_per_row=4)
    assert bm.allocate(1, 1) == mod.OK  # another request takes a block first
    for t in range(4):
        assert bm.allocate(0, 1) == mod.OK
        assert len(bm.rows[0]) == 1
    assert bm.allocate(0, 1) == mod.OK
    assert len(bm.rows[0]) == 2 and bm.rows[0][0] != bm.rows[0][1]
    assert bm.rows[0][1] != bm.rows[1][0]
    check_conservation(bm)


def pin_shared_system_prompt(mod) -> None:
    """"vLLM Worker侧...", section "PagedAttention与Block管理": 100 requests that start with the
    same 2000-token system prompt keep one copy of it (125 blocks of 16 instead of 12,500),
    every table's first 125 entries name the same blocks, each block counted 100 times, and a
    block goes back to the pool only when its count reaches zero."""
    bs, prompt = 16, 2000
    nblk = prompt // bs
    assert nblk == 125
    bm = mod.BlockManager(num_blocks=400, block_size=bs, num_rows=100, max_blocks_per_row=200)
    assert bm.allocate(0, prompt) == mod.OK
    for r in range(1, 100):
        assert bm.share(r, 0, nblk) == mod.OK
        assert bm.tokens[r] == prompt
    assert bm.num_free() == 400 - 125
    for r in range(100):
        assert bm.rows[r] == bm.rows[0]
    assert all(bm.ref[b] == 100 for b in bm.rows[0])
    # each request's own continuation is private
    for r in range(100):
        assert bm.allocate(r, 1) == mod.OK
    assert bm.num_free() == 400 - 125 - 100
    tails = {bm.rows[r][-1] for r in range(100)}
    assert len(tails) == 100 and not tails & set(bm.rows[0][:125])
    check_conservation(bm)
    for r in range(99):
        assert bm.free(r) == mod.OK
    assert bm.num_free() == 400 - 125 - 1  # the prompt is still held by the last request
    assert all(bm.ref[b] == 1 for b in bm.rows[99][:125])
    assert bm.free(99) == mod.OK
    assert bm.num_free() == 400
    check_conservation(bm)


def pin_window_release(mod) -> None:
    """"vLLM Worker侧...", section "混合注意力机制": a sliding-window layer (W = 4096, block size
    16) returns blocks that left the window, so decoding 12,000 tokens holds a bounded number of
    blocks: exactly the blocks some query of the step can still read (brute force), never more
    than W / block_size + 1 (W / block_size when the window start is block-aligned)."""
    W, bs = 4096, 16
    bm = mod.BlockManager(num_blocks=300, block_size=bs, num_rows=1, max_blocks_per_row=1000,
                          window=W)
    assert bm.allocate(0, 5) == mod.OK
    sizes = set()
    for _ in range(12000):
        T = bm.tokens[0]
        assert bm.allocate(0, 1) == mod.OK
        live = {j for j, b in enumerate(bm.rows[0]) if b >= 0}
        assert live == window_live_blocks(T, T + 1, W, bs), f"T={T}"
        sizes.add(len(live))
        if (T - W + 1) % bs == 0 and T >= W:
            assert len(live) == W // bs
    assert max(sizes) == W // bs + 1
    check_conservation(bm)


def pin_window_speculative(mod) -> None:
    """Several new tokens in one step (speculative queries): the earliest query still sees its
    whole window, so only the blocks no query of the step can read are released."""
    W, bs = 10, 4
    rng = random.Random(3)
    bm = mod.BlockManager(num_blocks=40, block_size=bs, num_rows=1, max_blocks_per_row=200,
                          window=W)
    for _ in range(150):
        T = bm.tokens[0]
        n = rng.randint(1, 5)
        assert bm.allocate(0, n) == mod.OK
        live = {j for j, b in enumerate(bm.rows[0]) if b >= 0}
        assert live == window_live_blocks(T, T + n, W, bs)
        check_conservation(bm)


def pin_all_or_nothing(mod) -> None:
    """"vLLM의 KV cache 연결 흐름", section "EngineCore가 하는 일": a request whose blocks cannot
    be secured does not run; the failed allocation changes nothing.  Tokens that fit in the
    row's last, partly filled block need no new block."""
    bm = mod.BlockManager(num_blocks=5, block_size=4, num_rows=2, max_blocks_per_row=10)

    def snapshot():
        return ([list(r) for r in bm.rows], list(bm.tokens), list(bm.free_pool), list(bm.ref),
                dict(bm.staged))

    assert bm.allocate(0, 10) == mod.OK  # 3 blocks, 2 slots left in the third
    before = snapshot()
    assert bm.allocate(1, 9) == mod.OUT_OF_BLOCKS  # needs 3, 2 free
    assert snapshot() == before
    assert bm.allocate(1, 8) == mod.OK
    assert bm.num_free() == 0
    assert bm.allocate(0, 2) == mod.OK and len(bm.rows[0]) == 3 and bm.tokens[0] == 12
    before = snapshot()
    assert bm.allocate(0, 1) == mod.OUT_OF_BLOCKS
    assert snapshot() == before
    check_conservation(bm)


def pin_capacity_and_args(mod) -> None:
    """A row cannot outgrow its table row; sharing needs an empty destination and full, live
    source blocks."""
    bm = mod.BlockManager(num_blocks=20, block_size=4, num_rows=3, max_blocks_per_row=3)
    assert bm.allocate(0, 13) == mod.INVALID_ARG  # 4 blocks > 3
    assert bm.allocate(0, 12) == mod.OK
    assert bm.allocate(0, 1) == mod.INVALID_ARG
    assert bm.share(1, 0, 4) == mod.INVALID_ARG
    assert bm.share(1, 0, 3) == mod.OK
    assert bm.share(1, 0, 1) == mod.INVALID_ARG  # destination not empty
    assert bm.allocate(2, 6) == mod.OK
    assert bm.share(1, 2, 2) == mod.INVALID_ARG
    assert bm.free(1) == mod.OK
    assert bm.share(1, 2, 2) == mod.INVALID_ARG  # second block of row 2 holds 2 of 4 tokens
    assert bm.share(1, 2, 1) == mod.OK
    assert bm.share(0, 0, 1) == mod.INVALID_ARG
    check_conservation(bm)


def random_trace(mod, seed: int, steps: int, window: int = 0, zero_fill: bool = True,
                 check=None):
    """Drive a manager through a seeded mix of allocations (1..40 tokens), frees and prefix
    shares; `check(bm, op, result)` runs after each operation."""
    rng = random.Random(seed)
    bs = rng.choice([4, 8, 16])
    nb = rng.randint(24, 80)
    rows = rng.randint(3, 8)
    bm = mod.BlockManager(num_blocks=nb, block_size=bs, num_rows=rows, max_blocks_per_row=64,
                          window=window, zero_fill=zero_fill)
    ops = []
    for _ in range(steps):
        u = rng.random()
        r = rng.randrange(rows)
        if u < 0.6:
            op = ("allocate", r, rng.choice([1, 1, 1, 2, 3, 5, 17, 40]))
        elif u < 0.75:
            op = ("free", r)
        elif u < 0.9:
            op = ("share", r, rng.randrange(rows), rng.randint(0, 6))
        else:
            op = ("flush",)
        ops.append(op)
        if op[0] == "allocate":
            res = bm.allocate(op[1], op[2])
        elif op[0] == "free":
            res = bm.free(op[1])
        elif op[0] == "share":
            res = bm.share(op[1], op[2], op[3])
        else:
            res = bm.flush()
        if check is not None:
            check(bm, op, res)
    return bm, ops


def pin_random_conservation(mod) -> None:
    """Brute force over random traces: counts, pool and row shapes stay consistent; with a
    window, each row's live blocks are exactly those its latest step could read."""
    for seed in range(30):
        for window in (0, 7, 33):
            last = {}

            def check(bm, op, res, window=window, last=last):
                check_conservation(bm)
                check_row_shape(bm)
                if window > 0 and op[0] == "allocate" and res == mod.OK:
                    r, n = op[1], op[2]
                    T = bm.tokens[r] - n
                    live = {j for j, b in enumerate(bm.rows[r]) if b >= 0}
                    assert live == window_live_blocks(T, T + n, window, bm.block_size)

            random_trace(mod, seed, 200, window=window, check=check)


def pin_flush_rebuilds_tables(mod) -> None:
    """Applying every flush to a table that starts as all -1 reproduces each row's block list
    (brute force); a zero-fill list names every block held now that nobody held at the last
    flush, only blocks held now, and never a block whose place in a row has been held without a
    break since the last flush (its contents are live)."""
    for seed in range(30):
        for window in (0, 9):
            state = {}

            def check(bm, op, res, state=state):
                if "table" not in state:
                    state["table"] = np.full((bm.num_rows, bm.max_blocks_per_row), -1, np.int32)
                    state["held"] = set()
                    state["unbroken"] = set()
                held_now = {(r, j, b) for r, row in enumerate(bm.rows) for j, b in enumerate(row)
                            if b >= 0}
                if op[0] != "flush":
                    state["unbroken"] &= held_now
                    return
                ups, zero = res
                table = state["table"]
                for r, c, v in ups:
                    table[r, c] = v
                for r, row in enumerate(bm.rows):
                    assert list(table[r, :len(row)]) == row
                live_now = {b for (_, _, b) in held_now}
                live_before = {b for (_, _, b) in state["held"]}
                unbroken = {b for (_, _, b) in state["unbroken"]}
                z = set(zero.tolist())
                assert list(zero) == sorted(z)
                assert z <= live_now
                assert (live_now - live_before) <= z
                assert not (z & unbroken)
                state["held"] = held_now
                state["unbroken"] = set(held_now)

            random_trace(mod, 100 + seed, 300, window=window, check=check)


def pin_apply_updates(mod) -> None:
    """The worker's side: staged (row, column, id) writes land in the table, listed blocks are
    zeroed in every cache, everything else is untouched, bad entries are skipped with bit 32."""
    table = np.full((3, 4), 2, np.int32)
    k = np.arange(6 * 8, dtype=np.float32).reshape(6, 8) + 1
    v = -k
    k0, v0 = k.copy(), v.copy()
    ups = np.array([[0, 0, 5], [1, 2, 3], [2, 3, -1], [3, 0, 1], [0, 4, 1], [1, 1, 6]], np.int32)
    err = mod.apply_updates(table, [k, v], ups, np.array([5, 3, 9], np.int32), 6)
    assert err == 32
    expect = np.full((3, 4), 2, np.int32)
    expect[0, 0], expect[1, 2], expect[2, 3] = 5, 3, -1
    assert (table == expect).all()
    for b in range(6):
        if b in (3, 5):
            assert not k[b].any() and not v[b].any()
        else:
            assert (k[b] == k0[b]).all() and (v[b] == v0[b]).all()
    assert mod.apply_updates(table, [k], np.zeros((0, 3), np.int32), np.zeros(0, np.int32), 6) == 0


ALL_PINS = [pin_48_tokens_three_blocks, pin_block_of_four_lazy, pin_shared_system_prompt,
            pin_window_release, pin_window_speculative, pin_all_or_nothing, pin_capacity_and_args,
            pin_random_conservation, pin_flush_rebuilds_tables, pin_apply_updates]
