"""Pins of the streamed-decode tile-plan oracle (oracle/streaming.py): tiles of
at most n_slots blocks in batch order, resident blocks reused, missing blocks
staged into the least recently used slot, invalidation (CPU only)."""
import random

from oracle.streaming import ScratchPoolOracle


def run_all(sp, tables, lens, bs):
    cursor, tiles = [0, 0], []
    while True:
        t = sp.plan_tile(tables, lens, bs, cursor)
        tiles.append(t)
        if t[3]:
            return tiles


def test_one_sequence_in_tiles_of_two_slots():
    sp = ScratchPoolOracle(2)
    tiles = run_all(sp, [[10, 11, 12, 13, 14]], [70], 16)   # blocks of 16, 16, 16, 16, 6 tokens
    assert [t[0][0][:2] for t in tiles] == [[0, 1], [0, 1], [0, 2]]
    assert [t[1] for t in tiles] == [[32], [32], [6]]
    # tile 2 reuses slots 0 then 1 (least recently used first); tile 3's block goes to slot 0
    assert [t[2] for t in tiles] == [[(10, 0), (11, 1)], [(12, 0), (13, 1)], [(14, 0)]]
    assert [t[3] for t in tiles] == [False, False, True]


def test_resident_blocks_are_not_staged_again():
    sp = ScratchPoolOracle(8)
    first = run_all(sp, [[3, 4], [5]], [20, 9], 16)
    assert first[0][2] == [(3, 0), (4, 1), (5, 2)]
    again = run_all(sp, [[3, 4], [5]], [20, 9], 16)
    assert again[0][2] == [] and again[0][0][0][:2] == [0, 1] and again[0][1] == [20, 9]


def test_a_block_shared_by_two_sequences_is_staged_once():
    sp = ScratchPoolOracle(4)
    (tables, lens, pairs, done), = run_all(sp, [[7, 8], [7, 9]], [32, 20], 16)
    assert pairs == [(7, 0), (8, 1), (9, 2)]
    assert tables[0][:2] == [0, 1] and tables[1][:2] == [0, 2] and lens == [32, 20] and done


def test_tiles_cross_sequence_boundaries():
    sp = ScratchPoolOracle(4)
    tiles = run_all(sp, [[0, 1, 2], [3, 4]], [48, 17], 16)
    assert tiles[0][0] == [[0, 1, 2], [3, 4, 4]] and tiles[0][1] == [48, 16]   # rows: min(4 slots, 3 blocks)
    assert tiles[1][1] == [0, 1] and tiles[1][0][1][0] == 0    # block 4 takes the oldest slot


def test_empty_sequences_and_empty_batch():
    sp = ScratchPoolOracle(3)
    tiles = run_all(sp, [[5], [], [6]], [0, 0, 3], 16)
    assert len(tiles) == 1 and tiles[0][1] == [0, 0, 3] and tiles[0][2] == [(6, 0)]
    assert run_all(ScratchPoolOracle(2), [[1], [2]], [0, 0], 16)[0][1:] == ([0, 0], [], True)


def test_invalidate_frees_the_slot_for_reuse_first():
    sp = ScratchPoolOracle(3)
    run_all(sp, [[1, 2, 3]], [48], 16)
    sp.invalidate(2)
    assert sp.lookup(2) == -1 and sp.lookup(1) == 0
    (tables, _, pairs, _), = run_all(sp, [[1, 2, 3]], [48], 16)
    assert pairs == [(2, 1)] and tables[0] == [0, 1, 2]


def test_tiles_cover_every_block_once_in_order():
    rng = random.Random(3)
    for _ in range(50):
        n = rng.randrange(1, 6)
        bs = 16
        lens = [rng.randrange(0, 200) for _ in range(n)]
        tables = [[rng.randrange(0, 30) for _ in range(-(-L // bs))] for L in lens]
        sp = ScratchPoolOracle(rng.randrange(1, 9))
        seen = [[] for _ in range(n)]
        tok = [0] * n
        for tt, tl, pairs, _ in run_all(sp, tables, lens, bs):
            staged = dict((s, h) for h, s in pairs)
            assert len(staged) == len(pairs)                 # distinct destination slots
            for s in range(n):
                k = -(-tl[s] // bs)
                seen[s] += tt[s][:k]
                tok[s] += tl[s]
                assert all(x == sp.n_slots for x in tt[s][k:])
        assert tok == lens
        assert [len(x) for x in seen] == [len(t) for t in tables]


def test_capped_tiles_take_at_most_tile_blocks():
    sp = ScratchPoolOracle(6)
    cursor, sizes = [0, 0], []
    while True:
        tt, tl, pairs, done = sp.plan_tile([[0, 1, 2, 3, 4, 5, 6]], [112], 16, cursor, tile_blocks=3)
        sizes.append(sum(1 for x in tt[0] if x != 6))
        if done:
            break
    assert sizes == [3, 3, 1]


def test_half_pool_tiles_never_stage_into_the_previous_tiles_slots():
    # least recently used: with tiles of at most n_slots // 2 blocks the slots a
    # tile stages into are never the slots the tile before it reads, whatever
    # the residency left by earlier calls and invalidations
    rng = random.Random(11)
    for _ in range(200):
        n_slots = rng.randrange(2, 12)
        sp = ScratchPoolOracle(n_slots)
        for call in range(3):
            n = rng.randrange(1, 5)
            bs = 16
            lens = [rng.randrange(0, 300) for _ in range(n)]
            tables = [[rng.randrange(0, 40) for _ in range(-(-L // bs))] for L in lens]
            cursor, prev = [0, 0], set()
            while True:
                tt, tl, pairs, done = sp.plan_tile(tables, lens, bs, cursor, tile_blocks=n_slots // 2)
                used = {x for row in tt for x in row if x != n_slots}
                assert not ({slot for _, slot in pairs} & prev)
                prev = used
                if done:
                    break
            if rng.random() < 0.5:
                sp.invalidate(rng.randrange(0, 40))
