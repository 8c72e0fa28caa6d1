"""Plain-Python oracle of the host-side block manager (test infrastructure:
only tests/, __graft_entry__.smoke() and bench.py's CPU baseline use it).

Each rule follows a page:

- tiny-llm paged_kv.py, BlockAllocator: fixed-size blocks on a free stack
  that hands out the lowest ids first and reuses the last freed block first;
  freeing a block that is not in use is an error; the peak of blocks in use is
  kept.
- AstrAI cache.py, PagedCache.alloc / alloc_n / free: a reference count per
  block, 1 on allocation, dropped by free; a block is free again when its count
  reaches 0; a multi-block allocation is all or nothing.
- libmir-metal paged/mod.rs, PagedStore::snapshot / release: sharing a
  sequence's pages raises each page's reference count by one; releasing lowers
  it.
- tiny-llm paged_kv.py, PagedKVCache: can_admit needs ceil((n + 1) / bs) free
  blocks per prompt; admit takes ceil(n / bs) blocks; reserve_step preempts the
  newest admissions until the next step's new blocks fit; begin_step gives a
  sequence whose blocks are full one more block; end_step counts the token.

Readings where the pages are silent (the same in the library): a failing call
changes nothing (admit is all or nothing, free checks every block first);
copy-on-write -- the block a sequence is about to write into, if shared, is
replaced by a fresh private block and the (source, destination) pair is
reported for a device copy; reserve_step counts such copies as needed blocks;
releasing an inactive slot does nothing; a forked sequence is the newest
admission.  Parity with the library is exact (same ids, same order).
"""
from __future__ import annotations


class BlockError(RuntimeError):
    pass


class OutOfBlocks(BlockError):
    pass


class StateError(BlockError):
    pass


class RangeError(BlockError):
    pass


class InvalidArg(BlockError):
    pass


def blocks_for(tokens: int, block_size: int) -> int:
    return -(-tokens // block_size)


class BlockManagerOracle:
    def __init__(self, n_blocks: int, block_size: int, n_slots: int, max_blocks: int):
        if min(n_blocks, block_size, n_slots, max_blocks) <= 0:
            raise InvalidArg("sizes must be positive")
        self.n_blocks, self.block_size = n_blocks, block_size
        self.n_slots, self.max_blocks = n_slots, max_blocks
        # stack: the last element is handed out next, so block 0 goes first
        self.free_stack = [n_blocks - 1 - i for i in range(n_blocks)]
        self.refs = [0] * n_blocks
        self.peak_used = 0
        self.tables = [[] for _ in range(n_slots)]
        self.lens = [0] * n_slots
        self.active = [False] * n_slots
        self.admit_no = [0] * n_slots
        self.admits = 0

    # -- blocks ---------------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self.free_stack)

    def _take(self) -> int:
        b = self.free_stack.pop()
        self.refs[b] = 1
        self.peak_used = max(self.peak_used, self.n_blocks - len(self.free_stack))
        return b

    def _drop(self, b: int) -> None:
        self.refs[b] -= 1
        if self.refs[b] == 0:
            self.free_stack.append(b)

    def alloc(self) -> int:
        if not self.free_stack:
            raise OutOfBlocks(f"all {self.n_blocks} blocks in use")
        return self._take()

    def free(self, blocks) -> None:
        blocks = list(blocks)
        for b in blocks:
            if not 0 <= b < self.n_blocks:
                raise InvalidArg(f"block id {b}")
        for b in set(blocks):
            if blocks.count(b) > self.refs[b]:
                raise StateError(f"block {b} freed more often than it is held")
        for b in blocks:
            self._drop(b)

    def refcount(self, b: int) -> int:
        return self.refs[b] if 0 <= b < self.n_blocks else -1

    # -- slots ----------------------------------------------------------------
    def _slot(self, s: int) -> None:
        if not 0 <= s < self.n_slots:
            raise InvalidArg(f"slot {s}")

    def can_admit(self, lengths) -> bool:
        if any(n < 0 for n in lengths):
            raise InvalidArg("negative length")
        return sum(blocks_for(n + 1, self.block_size) for n in lengths) <= self.num_free

    def admit(self, s: int, n_tokens: int) -> None:
        self._slot(s)
        if n_tokens < 0:
            raise InvalidArg("negative length")
        if self.active[s]:
            raise StateError(f"slot {s} is active")
        if n_tokens >= self.max_blocks * self.block_size:
            raise RangeError(f"{n_tokens} tokens do not leave room in {self.max_blocks} blocks")
        need = blocks_for(n_tokens, self.block_size)
        if need > self.num_free:
            raise OutOfBlocks(f"{need} blocks wanted, {self.num_free} free")
        self.tables[s] = [self._take() for _ in range(need)]
        self.lens[s] = n_tokens
        self.active[s] = True
        self.admits += 1
        self.admit_no[s] = self.admits

    def release(self, s: int) -> None:
        self._slot(s)
        for b in self.tables[s]:
            self._drop(b)
        self.tables[s] = []
        self.lens[s] = 0
        self.active[s] = False

    def fork(self, src: int, dst: int) -> None:
        self._slot(src)
        self._slot(dst)
        if src == dst:
            raise InvalidArg("fork onto itself")
        if not self.active[src] or self.active[dst]:
            raise StateError("fork needs an active source and an inactive destination")
        self.tables[dst] = list(self.tables[src])
        for b in self.tables[dst]:
            self.refs[b] += 1
        self.lens[dst] = self.lens[src]
        self.active[dst] = True
        self.admits += 1
        self.admit_no[dst] = self.admits

    def _needs_block(self, s: int) -> bool:
        """The coming step's token (position lens[s]) needs a new block: the
        table is full, or the block holding that position is shared."""
        t, n = self.tables[s], self.lens[s]
        if len(t) * self.block_size <= n:
            return True
        return self.refs[t[n // self.block_size]] > 1

    def _total_need(self) -> int:
        return sum(1 for s in range(self.n_slots) if self.active[s] and self._needs_block(s))

    def reserve_step(self) -> list[int]:
        victims = []
        while any(self.active) and self._total_need() > self.num_free:
            newest = max((s for s in range(self.n_slots) if self.active[s]), key=lambda s: self.admit_no[s])
            self.release(newest)
            victims.append(newest)
        return victims

    def begin_step(self) -> list[tuple[int, int]]:
        for s in range(self.n_slots):
            if self.active[s] and self.lens[s] >= self.max_blocks * self.block_size:
                raise RangeError(f"slot {s} is full")
        if self._total_need() > self.num_free:
            raise OutOfBlocks("not enough free blocks for this step")
        copies = []
        for s in range(self.n_slots):
            if not self.active[s]:
                continue
            t, n = self.tables[s], self.lens[s]
            if len(t) * self.block_size <= n:
                t.append(self._take())
                continue
            j = n // self.block_size
            old = t[j]
            if self.refs[old] > 1:
                fresh = self._take()
                self.refs[old] -= 1
                t[j] = fresh
                copies.append((old, fresh))
        return copies

    def end_step(self) -> None:
        for s in range(self.n_slots):
            if self.active[s]:
                self.lens[s] += 1

    def export(self):
        """(tables as lists padded with the scratch id n_blocks, lens, active)."""
        tables = [t + [self.n_blocks] * (self.max_blocks - len(t)) for t in self.tables]
        lens = [self.lens[s] if self.active[s] else 0 for s in range(self.n_slots)]
        return tables, lens, [int(a) for a in self.active]


def copy_blocks(pool, pairs):
    """Device-copy oracle: every destination block becomes its source block
    (numpy / torch arrays indexed by block id on the first axis)."""
    for src, dst in pairs:
        pool[dst] = pool[src]
    return pool
