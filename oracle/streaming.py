"""Plain-Python oracle of the tile plan for decode streamed from a host tier
(test infrastructure: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline use it).

It follows metrale high_speed_swap impl_more.rs, attend_layer_on_stream_with_q_pos:
a sequence's blocks are attended one tile of at most resident_blocks blocks at a
time; for each tile a block already in the scratch pool keeps its slot, a missing
block is given a slot (its previous block forgotten) and read from the tier, and
the tile's table and counts go to the device; offload_block's invariant -- a
rewritten block loses its scratch-pool copy -- is `invalidate`.

Readings where the page is silent (the same in the library): the page's
predictor-driven eviction ranking is replaced by least recently used (a slot
used by the current tile is never taken); empty slots are used first, in id
order; a tile takes the blocks of the whole batch in order, sequence after
sequence, so one tile may hold the end of one sequence and the start of the
next; a sequence's tokens in a tile are its tokens of the blocks taken (the
last block of a sequence may be partial).  A tile may be capped below the
pool size (the library caps it at half the pool when the batch does not fit,
so that staging the next tile never overwrites a slot the current one reads).

The attention itself is checked against oracle.decode over the whole context:
tiling, like split-KV, does not change the result beyond rounding.
"""
from __future__ import annotations


class ScratchPoolOracle:
    def __init__(self, n_slots: int):
        self.n_slots = n_slots
        self.slot_of = {}                     # host block -> slot
        self.block_of = [None] * n_slots      # slot -> host block
        self.order = list(range(n_slots))     # least recently used first

    def _touch(self, slot: int) -> None:
        self.order.remove(slot)
        self.order.append(slot)

    def lookup(self, host_block: int) -> int:
        return self.slot_of.get(host_block, -1)

    def invalidate(self, host_block: int) -> None:
        slot = self.slot_of.pop(host_block, None)
        if slot is None:
            return
        self.block_of[slot] = None
        self.order.remove(slot)
        self.order.insert(0, slot)            # reused first

    def plan_tile(self, host_tables, ctx_lens, block_size: int, cursor, tile_blocks: int = 0, max_blocks=None):
        """Next tile of at most tile_blocks blocks (0 or more than n_slots: all
        slots) from cursor = [sequence, block]; returns (tile_tables as lists
        padded with n_slots to min(tile size, max_blocks) entries, tile_lens,
        pairs [(host block, slot)], done) and advances cursor.  max_blocks
        defaults to the longest table row (at least 1)."""
        cap = self.n_slots if tile_blocks <= 0 or tile_blocks > self.n_slots else tile_blocks
        if max_blocks is None:
            max_blocks = max([1] + [len(r) for r in host_tables])
        width = min(cap, max_blocks)
        n = len(ctx_lens)
        nb = [-(-int(L) // block_size) for L in ctx_lens]
        tables = [[] for _ in range(n)]
        lens = [0] * n
        pairs = []
        used = set()
        s, j = cursor
        taken = 0
        while s < n and taken < cap:
            if j >= nb[s]:
                s, j = s + 1, 0
                continue
            hb = int(host_tables[s][j])
            slot = self.slot_of.get(hb)
            if slot is None:
                slot = next(x for x in self.order if x not in used)
                old = self.block_of[slot]
                if old is not None:
                    del self.slot_of[old]
                self.block_of[slot] = hb
                self.slot_of[hb] = slot
                pairs.append((hb, slot))
            used.add(slot)
            self._touch(slot)
            tables[s].append(slot)
            lens[s] += min(block_size, int(ctx_lens[s]) - j * block_size)
            j += 1
            taken += 1
        while s < n and j >= nb[s]:
            s, j = s + 1, 0
        cursor[0], cursor[1] = s, j
        padded = [t + [self.n_slots] * (width - len(t)) for t in tables]
        return padded, lens, pairs, s >= n
