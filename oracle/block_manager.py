"""Block manager oracle: the free block pool, reference counts, per-request block tables,
sliding-window release, and the worker-side table writes + zero fill (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this module.
It is plain Python (lists, a deque, a dict) written from the pages; it shares no code with the
library's C++ block manager or its CUDA kernel, and neither imports it.

What the pages fix:
  * "vLLM의 KV cache 연결 흐름", section "KVCacheManager가 하는 일": the manager tracks the blocks
    each request already holds, works out whether new tokens need a new block, hands blocks out
    of the free pool, takes them back when the request ends, and produces the block ids the
    worker receives.  Section "EngineCore가 하는 일": a request whose blocks cannot be secured
    does not run this step (here: the allocation is all-or-nothing and changes nothing when it
    fails).  Section "SchedulerOutput이 건네는 것": the worker is told the newly assigned block
    ids and which new blocks must be initialised.  Section "GPU worker가 하는 일": the worker
    appends the new ids to its per-request block table rows and zero-fills new blocks.
  * "Understanding PageAttention Memory Optimization" (page title section): blocks are handed
    out lazily - a new block only when the previous one is full (block of 4 tokens: the fifth
    token opens the second block).
  * "vLLM Worker侧GPU KV Cache初始化流程深度解析", section "PagedAttention与Block管理": sequences
    with a common prompt prefix point the first entries of their block tables at the same
    physical blocks; a reference count per physical block tells how many logical blocks use
    it, and the block returns to the pool only when the count reaches zero.  Section "调度视角":
    48 computed tokens at block size 16 occupy 3 logical blocks.  Section "混合注意力机制": in
    a sliding-window layer, blocks whose tokens have all left the window go back to the pool,
    so such a layer holds a bounded number of blocks (about W / block_size).

Readings where the pages are silent (each one stated once here):
  * Free-pool order: first in, first out.  The pool starts as 0, 1, ..., num_blocks-1; an
    allocation takes from the front; a block whose count reaches zero joins the back, blocks
    released together joining in logical order.
  * allocate(row, n) makes room for n more tokens at positions T .. T+n-1 (T = tokens the row
    holds) and then counts them as held.  With a window W > 0 it first releases every live block
    whose last position is <= T - W, the blocks no query at position >= T can see (keys
    p - W < j <= p); the release happens even when the allocation then fails.
  * share(dst, src, k): an empty row dst takes src's first k blocks (all full and live) with
    each count raised by one, and holds k * block_size tokens.
  * free(row) returns the row's live blocks and empties it; it stages no table writes (entries
    past a row's blocks are never read).
  * Table writes are staged per (row, column), the last value winning; flush() hands them out
    sorted by (row, column), with the ids handed out since the previous flush that are still
    held (sorted, each once) as the blocks to zero-fill (none when zero fill is off).
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List, Sequence, Tuple

import numpy as np

OK, INVALID_ARG, OUT_OF_BLOCKS = 0, 1, 5


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    """Logical blocks that hold num_tokens tokens: a block opens only when the last one is full."""
    return (num_tokens + block_size - 1) // block_size


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, num_rows: int, max_blocks_per_row: int,
                 window: int = 0, zero_fill: bool = True):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.num_rows = num_rows
        self.max_blocks_per_row = max_blocks_per_row
        self.window = window
        self.zero_fill = zero_fill
        self.free_pool = deque(range(num_blocks))
        self.ref = [0] * num_blocks
        self.rows: List[List[int]] = [[] for _ in range(num_rows)]  # physical id, -1 = released
        self.tokens = [0] * num_rows
        self.staged: Dict[Tuple[int, int], int] = {}
        self.fresh: set = set()

    # -- pool -------------------------------------------------------------------------------
    def _take(self) -> int:
        b = self.free_pool.popleft()
        assert self.ref[b] == 0
        self.ref[b] = 1
        self.fresh.add(b)
        return b

    def _drop(self, b: int) -> None:
        assert self.ref[b] > 0
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free_pool.append(b)

    def num_free(self) -> int:
        return len(self.free_pool)

    # -- operations -------------------------------------------------------------------------
    def _release_outside_window(self, row: int) -> None:
        """Blocks whose last position is <= T - W are invisible to every query at >= T."""
        if self.window <= 0:
            return
        first_query = self.tokens[row]
        blocks = self.rows[row]
        for j, b in enumerate(blocks):
            last_pos = (j + 1) * self.block_size - 1
            if last_pos > first_query - self.window:
                break
            if b >= 0:
                self._drop(b)
                blocks[j] = -1
                self.staged[(row, j)] = -1

    def allocate(self, row: int, num_new_tokens: int) -> int:
        if not (0 <= row < self.num_rows) or num_new_tokens < 0:
            return INVALID_ARG
        total = self.tokens[row] + num_new_tokens
        need_blocks = blocks_for_tokens(total, self.block_size)
        if need_blocks > self.max_blocks_per_row:
            return INVALID_ARG
        self._release_outside_window(row)
        missing = need_blocks - len(self.rows[row])
        if missing > len(self.free_pool):
            return OUT_OF_BLOCKS
        for _ in range(missing):
            b = self._take()
            self.rows[row].append(b)
            self.staged[(row, len(self.rows[row]) - 1)] = b
        self.tokens[row] = total
        return OK

    def free(self, row: int) -> int:
        if not (0 <= row < self.num_rows):
            return INVALID_ARG
        for b in self.rows[row]:
            if b >= 0:
                self._drop(b)
        self.rows[row] = []
        self.tokens[row] = 0
        return OK

    def share(self, dst: int, src: int, num_blocks: int) -> int:
        if not (0 <= dst < self.num_rows and 0 <= src < self.num_rows) or dst == src:
            return INVALID_ARG
        if self.rows[dst] or self.tokens[dst] or num_blocks < 0:
            return INVALID_ARG
        if num_blocks > len(self.rows[src]) or self.tokens[src] < num_blocks * self.block_size:
            return INVALID_ARG
        prefix = self.rows[src][:num_blocks]
        if any(b < 0 for b in prefix):
            return INVALID_ARG
        for j, b in enumerate(prefix):
            self.ref[b] += 1
            self.rows[dst].append(b)
            self.staged[(dst, j)] = b
        self.tokens[dst] = num_blocks * self.block_size
        return OK

    def flush(self) -> Tuple[np.ndarray, np.ndarray]:
        """(updates int32 [n, 3] of (row, column, block id), zero-fill ids int32 [m])."""
        ups = np.array([(r, c, v) for (r, c), v in sorted(self.staged.items())],
                       dtype=np.int32).reshape(-1, 3)
        zero = sorted(b for b in self.fresh if self.ref[b] > 0) if self.zero_fill else []
        self.staged = {}
        self.fresh = set()
        return ups, np.array(zero, dtype=np.int32)


def apply_updates(block_table: np.ndarray, caches: Sequence[np.ndarray], updates: np.ndarray,
                  zero_ids: np.ndarray, num_blocks: int) -> int:
    """The worker's side ("GPU worker가 하는 일"): write each staged (row, column, id) into the
    block table and zero every cache's rows of each listed block.  block_table is int32
    [rows, columns]; each cache is indexed by block id along its first axis.  Updates outside the
    table or with an id outside [-1, num_blocks), and zero-fill ids outside [0, num_blocks), are
    skipped; the return value is the error word the device sets for them (32 = bad update)."""
    err = 0
    rows, cols = block_table.shape
    for r, c, v in np.asarray(updates, dtype=np.int64).reshape(-1, 3):
        if not (0 <= r < rows and 0 <= c < cols) or not (-1 <= v < num_blocks):
            err |= 32
            continue
        block_table[r, c] = v
    for b in np.asarray(zero_ids, dtype=np.int64):
        if not (0 <= b < num_blocks):
            err |= 32
            continue
        for cache in caches:
            cache[b] = 0
    return err
