"""The library's tile planner for decode streamed from a host tier
(pkv_sp_plan_tile) against the oracle (oracle/streaming.py): same tiles, same
staged pairs, same residency, over random batches, repeated calls and
invalidations.  CPU only (no CUDA call)."""
import random

import pytest
import torch

from oracle.streaming import ScratchPoolOracle


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


@pytest.mark.parametrize("seed", range(10))
def test_planner_matches_the_oracle(P, seed):
    rng = random.Random(seed)
    bs = rng.choice([16, 32])
    n_slots = rng.randrange(1, 24)
    max_seqs = 8
    lib = P.ScratchPool(n_slots, max_seqs)
    ref = ScratchPoolOracle(n_slots)
    n_host = rng.randrange(4, 60)
    for call in range(12):
        n = rng.randrange(1, max_seqs + 1)
        lens = [rng.randrange(0, 12 * bs) for _ in range(n)]
        max_blocks = max(1, max(-(-L // bs) for L in lens))
        tables = [[rng.randrange(0, n_host) for _ in range(max_blocks)] for _ in range(n)]
        t_tab, t_len = torch.tensor(tables, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32)
        cl, cr = [0, 0], [0, 0]
        cap = rng.choice([0, 0, n_slots // 2, rng.randrange(1, n_slots + 2)])
        while True:
            tt, tl, pairs, done = lib.plan_tile(t_tab, t_len, bs, cl, tile_blocks=cap)
            rtt, rtl, rpairs, rdone = ref.plan_tile(tables, lens, bs, cr, tile_blocks=cap, max_blocks=max_blocks)
            assert tt.tolist() == rtt and tl.tolist() == rtl and pairs == rpairs and done == rdone
            assert cl == cr
            if done:
                break
        for b in range(n_host):
            assert lib.lookup(b) == ref.lookup(b)
        for _ in range(rng.randrange(0, 3)):
            b = rng.randrange(0, n_host)
            lib.invalidate(b)
            ref.invalidate(b)


def test_planner_rejects_lengths_past_the_table(P):
    lib = P.ScratchPool(4, 2)
    with pytest.raises(P.PagedKVError):
        lib.plan_tile(torch.zeros((1, 2), dtype=torch.int32), torch.tensor([33], dtype=torch.int32), 16, [0, 0])


def test_planner_rejects_a_negative_host_id_without_changing_state(P):
    lib = P.ScratchPool(4, 2)
    tab = torch.tensor([[3, -1]], dtype=torch.int32)
    with pytest.raises(P.PagedKVError):
        lib.plan_tile(tab, torch.tensor([20], dtype=torch.int32), 16, [0, 0])
    assert lib.lookup(3) == -1
    tt, tl, pairs, done = lib.plan_tile(tab, torch.tensor([16], dtype=torch.int32), 16, [0, 0])
    assert pairs == [(3, 0)] and tt.tolist() == [[0, 4]] and done


def test_streamed_decode_host_checks(P):
    """paged_decode_streamed returns its host-checkable errors before any CUDA
    call (device pointers here are placeholders that are never dereferenced)."""
    import ctypes
    lib = P.load_library()
    sp = P.ScratchPool(4, 2)
    fake = ctypes.c_void_p(0x1000)
    d = P.Dims(4, 16, 2, 64)                     # the scratch pool: n_blocks = n_slots = 4
    tables = (ctypes.c_int32 * 4)(0, 1, 2, 3)    # [2 sequences][2 blocks]
    lens = (ctypes.c_int32 * 2)(20, 32)
    need = P.streamed_workspace_bytes(2, 8, 64, 4, 16)

    def call(**kw):
        return lib.paged_decode_streamed(
            kw.get("q", fake), 8, fake, fake, kw.get("n_host", 10), fake, fake, kw.get("dims", d),
            kw.get("sp", sp._h), kw.get("tables", tables), 2, kw.get("lens", lens), kw.get("n", 2),
            kw.get("scale", 0.125), fake, None, kw.get("ws", fake), kw.get("wsb", need), None, None)

    assert call(n=0) == 0
    assert call(sp=None) == 1
    assert call(dims=P.Dims(5, 16, 2, 64)) == 1            # pool size is not the scratch pool's
    assert call(n=3) == 1                                    # more sequences than the pool plans for
    assert call(q=None) == 1
    for sc in (0.0, -1.0, float("nan"), float("inf")):
        assert call(scale=sc) == 1
    assert call(dims=P.Dims(4, 16, 2, 96)) == 2              # head_dim
    assert call(lens=(ctypes.c_int32 * 2)(20, 33)) == 3      # past the table (2 blocks of 16)
    assert call(n_host=3) == 3                               # host id 3 outside a 3-block tier
    assert call(wsb=need - 1) == 4
    assert call(ws=ctypes.c_void_p(0x1010)) == 4               # not 256-byte aligned
    assert need > 0


def test_stage_blocks_host_checks(P):
    import ctypes
    lib = P.load_library()
    fake, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1004)
    d = P.Dims(4, 16, 2, 64)

    def call(**kw):
        return lib.paged_kv_stage_blocks(kw.get("pairs", fake), kw.get("n", 3), kw.get("hk", fake), fake, 10,
                                         fake, fake, kw.get("dims", d), None, None)

    assert call(n=0) == 0
    assert call(n=-1) == 1
    assert call(pairs=None) == 1
    assert call(pairs=odd) == 1                          # pairs are read as 8-byte int2
    assert call(hk=ctypes.c_void_p(0x1008)) == 1         # 16-byte vectors
    assert call(dims=P.Dims(4, 16, 2, 96)) == 2
