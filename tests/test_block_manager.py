"""The library's host-side block manager (include/pagedkv_blocks.h) against the
oracle (oracle/block_manager.py): every operation of random serving loops
gives the same result -- block ids, victims, copy-on-write pairs, errors --
and the same exported state afterwards.  CPU only (no CUDA call)."""
import random

import pytest
import torch

from oracle.block_manager import BlockManagerOracle, InvalidArg, OutOfBlocks, RangeError, StateError

STATUS = {OutOfBlocks: 6, StateError: 7, RangeError: 3, InvalidArg: 1}


@pytest.fixture(scope="module")
def P():
    from paged_kv_cache_212_gb300 import build as B
    try:
        B.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    B.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


def both(P, ref, lib, name, *args):
    """Run one operation on both; return (ref result, lib result) or the
    matching error status."""
    try:
        r = getattr(ref, name)(*args)
        r_st = 0
    except tuple(STATUS) as e:
        r, r_st = None, STATUS[type(e)]
    try:
        l = getattr(lib, name)(*args)
        l_st = 0
    except P.PagedKVError as e:
        l, l_st = None, e.status
    assert r_st == l_st, (name, args, r_st, l_st)
    assert r == l, (name, args, r, l)


def same_state(ref, lib):
    t, n, a = lib.export()
    rt, rn, ra = ref.export()
    assert t.tolist() == rt and n.tolist() == rn and a.tolist() == ra
    assert lib.num_free == ref.num_free and lib.peak_used == ref.peak_used
    assert [lib.refcount(b) for b in range(ref.n_blocks)] == ref.refs
    assert lib.refcount(-1) == -1 and lib.refcount(ref.n_blocks) == -1


@pytest.mark.parametrize("seed,n_blocks,bs,n_slots,max_blocks",
                         [(1, 40, 4, 8, 12), (2, 12, 16, 6, 4), (3, 200, 16, 32, 32), (4, 5, 4, 4, 3)])
def test_random_serving_loops_match_the_oracle(P, seed, n_blocks, bs, n_slots, max_blocks):
    rng = random.Random(seed)
    ref = BlockManagerOracle(n_blocks, bs, n_slots, max_blocks)
    lib = P.BlockManager(n_blocks, bs, n_slots, max_blocks)
    for _ in range(1500):
        op = rng.random()
        s = rng.randrange(-1, n_slots + 1)      # includes out-of-range slots
        if op < 0.22:
            both(P, ref, lib, "admit", s, rng.randrange(-1, max_blocks * bs + 2))
        elif op < 0.30:
            both(P, ref, lib, "release", s)
        elif op < 0.40:
            both(P, ref, lib, "fork", s, rng.randrange(-1, n_slots + 1))
        elif op < 0.45:
            lens = [rng.randrange(0, 3 * bs) for _ in range(rng.randrange(0, 4))]
            both(P, ref, lib, "can_admit", lens)
        elif op < 0.50:
            both(P, ref, lib, "alloc")
        elif op < 0.55:
            held = [b for b in range(n_blocks) if ref.refs[b] > 0]
            pick = [rng.choice(held) for _ in range(rng.randrange(1, 3))] if held and rng.random() < 0.8 \
                else [rng.randrange(-1, n_blocks + 1)]
            both(P, ref, lib, "free", pick)
        elif op < 0.75:
            both(P, ref, lib, "reserve_step")
        elif op < 0.92:
            both(P, ref, lib, "begin_step")
        else:
            both(P, ref, lib, "end_step")
        same_state(ref, lib)


def test_invalid_construction(P):
    with pytest.raises(P.PagedKVError):
        P.BlockManager(0, 16, 4, 4)
    with pytest.raises(P.PagedKVError):
        P.BlockManager(8, 16, 4, -1)


def test_export_is_what_the_kernels_take(P):
    """Tables exported for the kernels: int32 [n_slots, max_blocks], unused
    entries = the scratch id n_blocks."""
    lib = P.BlockManager(10, 16, 3, 5)
    lib.admit(2, 40)
    tables, lens, active = lib.export()
    assert tables.dtype == torch.int32 and tables.shape == (3, 5)
    assert tables[2].tolist() == [0, 1, 2, 10, 10] and tables[0].tolist() == [10] * 5
    assert lens.tolist() == [0, 0, 40] and active.tolist() == [0, 0, 1]
