"""Pins of the block-manager oracle (oracle/block_manager.py) against the
pages' allocation rules, on hand-worked cases and invariants (CPU only)."""
import random

import pytest

from oracle.block_manager import (BlockManagerOracle, InvalidArg, OutOfBlocks, RangeError, StateError,
                                  copy_blocks)


def test_fresh_pool_hands_out_lowest_ids_first():
    # tiny-llm BlockAllocator: "Lowest ids are handed out first"
    m = BlockManagerOracle(5, 4, 2, 4)
    assert [m.alloc() for _ in range(5)] == [0, 1, 2, 3, 4]
    with pytest.raises(OutOfBlocks):
        m.alloc()


def test_freed_blocks_come_back_last_freed_first():
    # the free list is a stack: a freed block is the next one handed out
    m = BlockManagerOracle(6, 4, 2, 4)
    for _ in range(4):
        m.alloc()                      # 0 1 2 3 in use, 4 5 free
    m.free([1])
    assert m.alloc() == 1
    m.free([0, 2])                     # pushed in list order: 2 on top
    assert [m.alloc(), m.alloc(), m.alloc()] == [2, 0, 4]


def test_double_free_and_bad_ids_change_nothing():
    m = BlockManagerOracle(4, 4, 1, 4)
    a, b = m.alloc(), m.alloc()
    with pytest.raises(StateError):
        m.free([a, a])                 # held once, dropped twice
    with pytest.raises(StateError):
        m.free([a, 3])                 # 3 was never allocated
    with pytest.raises(InvalidArg):
        m.free([a, 9])
    assert m.refs[:2] == [1, 1] and m.num_free == 2
    m.free([b, a])
    assert m.num_free == 4 and m.alloc() == a


def test_reference_counts_of_shared_blocks():
    # AstrAI: free drops one reference; libmir-metal snapshot adds one per page
    m = BlockManagerOracle(8, 4, 3, 4)
    m.admit(0, 6)                      # blocks 0, 1
    m.fork(0, 1)
    assert m.tables[1] == [0, 1] and m.refs[:2] == [2, 2]
    m.release(0)
    assert m.refs[:2] == [1, 1] and m.num_free == 6
    m.release(1)
    assert m.refs[:2] == [0, 0] and m.num_free == 8
    assert m.peak_used == 2


def test_can_admit_counts_room_for_the_first_decode_token():
    # tiny-llm can_admit: sum ceil((n + 1) / bs) <= free blocks
    m = BlockManagerOracle(3, 16, 4, 8)
    assert m.can_admit([15, 16])       # 1 + 2 = 3
    assert not m.can_admit([16, 16])   # 2 + 2 = 4
    assert m.can_admit([])
    assert m.can_admit([0, 0, 0])      # 1 + 1 + 1


def test_admit_takes_ceil_blocks_all_or_nothing():
    m = BlockManagerOracle(4, 16, 3, 8)
    m.admit(0, 17)                     # ceil(17/16) = 2 blocks
    assert m.tables[0] == [0, 1] and m.lens[0] == 17
    with pytest.raises(OutOfBlocks):
        m.admit(1, 40)                 # 3 blocks wanted, 2 free: nothing taken
    assert m.num_free == 2 and not m.active[1]
    with pytest.raises(StateError):
        m.admit(0, 1)
    with pytest.raises(RangeError):
        m.admit(2, 8 * 16)             # no room left for a decode token
    m.admit(2, 0)
    assert m.tables[2] == [] and m.active[2]


def test_begin_step_grows_only_full_tables():
    m = BlockManagerOracle(8, 16, 2, 4)
    m.admit(0, 16)                     # block 0 full: the token at position 16 needs a block
    m.admit(1, 15)                     # block 1 has room for position 15
    assert m.begin_step() == []
    assert m.tables == [[0, 2], [1]]
    m.end_step()
    assert m.lens == [17, 16]
    m.begin_step()
    assert m.tables == [[0, 2], [1, 3]]


def test_reserve_step_preempts_newest_first():
    # three sequences at a block boundary need 3 blocks; one is free.  Releasing
    # slot 2 (the newest) frees its block: 2 free, 2 needed -> done
    m = BlockManagerOracle(4, 4, 3, 4)
    m.admit(0, 4)
    m.admit(1, 4)
    m.admit(2, 4)
    assert m.num_free == 1 and m._total_need() == 3
    assert m.reserve_step() == [2]
    assert m.num_free == 2 and m._total_need() == 2


def test_reserve_step_victims_by_hand():
    m = BlockManagerOracle(5, 4, 4, 4)
    m.admit(0, 4)                      # each at a block boundary: needs one block
    m.admit(1, 4)
    m.admit(2, 4)
    m.admit(3, 3)                      # room in its block: needs none
    # free 1, need 3 -> release slot 3 (newest; frees 1, need stays 3) -> free 2
    # -> release slot 2 (frees 1, need 2) -> free 3 >= 2: stop
    assert m.reserve_step() == [3, 2]
    assert m.num_free == 3 and m._total_need() == 2
    assert m.reserve_step() == []


def test_fork_then_copy_on_write():
    m = BlockManagerOracle(8, 16, 3, 4)
    m.admit(0, 20)                     # blocks 0 (full), 1 (4 tokens)
    m.fork(0, 1)                       # shares 0 and 1
    copies = m.begin_step()            # both write position 20 in block 1 (shared)
    # slot 0 comes first: it gets a private copy (block 2); slot 1 then holds
    # block 1 alone and writes in place
    assert copies == [(1, 2)]
    assert m.tables[0] == [0, 2] and m.tables[1] == [0, 1]
    assert m.refs[:3] == [2, 1, 1]
    m.end_step()
    assert m.begin_step() == []        # nothing shared at position 21 any more


def test_reserve_step_counts_copy_on_write():
    m = BlockManagerOracle(2, 16, 2, 4)
    m.admit(0, 20)                     # both blocks used
    m.fork(0, 1)
    assert m.num_free == 0 and m._total_need() == 2
    assert m.reserve_step() == [1]     # the fork is newest; then block 1 is private
    assert m._total_need() == 0


def test_begin_step_refuses_a_full_sequence_and_missing_blocks():
    m = BlockManagerOracle(2, 4, 1, 2)
    m.admit(0, 7)
    m.begin_step()
    m.end_step()                       # 8 tokens = max_blocks * bs
    with pytest.raises(RangeError):
        m.begin_step()
    m2 = BlockManagerOracle(1, 4, 1, 4)
    m2.admit(0, 4)
    with pytest.raises(OutOfBlocks):
        m2.begin_step()
    assert m2.tables[0] == [0]


def test_export_pads_with_the_scratch_id():
    m = BlockManagerOracle(6, 4, 3, 3)
    m.admit(1, 5)
    tables, lens, active = m.export()
    assert tables == [[6, 6, 6], [0, 1, 6], [6, 6, 6]]
    assert lens == [0, 5, 0] and active == [0, 1, 0]


def _check_invariants(m):
    held = [0] * m.n_blocks
    for s in range(m.n_slots):
        if not m.active[s]:
            assert m.tables[s] == [] and m.lens[s] == 0
            continue
        for b in m.tables[s]:
            held[b] += 1
        # a table covers the stored tokens, plus at most the block of the next token
        assert len(m.tables[s]) in (-(-m.lens[s] // m.block_size), -(-(m.lens[s] + 1) // m.block_size))
    loose = [m.refs[b] - held[b] for b in range(m.n_blocks)]
    assert all(x >= 0 for x in loose)
    assert sorted(m.free_stack) == [b for b in range(m.n_blocks) if m.refs[b] == 0]
    assert len(set(m.free_stack)) == len(m.free_stack)
    return loose


def test_invariants_under_a_random_serving_loop():
    rng = random.Random(7)
    m = BlockManagerOracle(40, 4, 8, 12)
    for _ in range(400):
        op = rng.random()
        s = rng.randrange(8)
        try:
            if op < 0.25:
                m.admit(s, rng.randrange(0, 30))
            elif op < 0.35:
                m.release(s)
            elif op < 0.45:
                m.fork(s, rng.randrange(8))
            else:
                m.reserve_step()
                m.begin_step()
                m.end_step()
        except (OutOfBlocks, StateError, RangeError, InvalidArg):
            pass
        loose = _check_invariants(m)
        assert all(x == 0 for x in loose)   # every reference is a table entry


def test_copy_blocks_oracle():
    import numpy as np
    pool = np.arange(5 * 3).reshape(5, 3)
    copy_blocks(pool, [(0, 4), (2, 3)])
    assert pool[4].tolist() == [0, 1, 2] and pool[3].tolist() == [6, 7, 8]
