"""Pins for the oracle's page write and gather (CPU only).

What fixes the expected values:
  * identity tables: with table[j] = j the pool, read in storage order, IS the
    sequence (libmir-metal paged/mod.rs, context: the identity table skips the
    take and reshapes the arena directly);
  * permutation: a permuted table only relocates whole pages (tiny-llm
    paged_kv.py docstring: block table = page table);
  * AstrAI cache.py PagedCache.write's own page loop and tiny-llm's gather
    (pool[table].transpose(1, 2).reshape), both written with torch indexing;
  * the waste bound of the tiny-llm docstring (at most block_size - 1 unused
    slots per sequence).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_pools import BF16_NAN, bits, dims_of, empty_pools, logical_rows, \
    oracle_pools_after_step, write_prefix
from paged_kv_cache_212_gb300 import workloads as W


def _rows(gen, n, hkv, d):
    return torch.randn((n, hkv, d), generator=gen).to(torch.bfloat16)


@pytest.mark.parametrize("bs,hkv,d", [(4, 2, 8), (16, 2, 64), (16, 8, 128), (32, 3, 16)])
def test_write_identity_table_is_storage_order(bs, hkv, d):
    gen = torch.Generator().manual_seed(1)
    L = 5 * bs + 3  # ragged last block
    nb = L // bs + 2
    dims = oracle.Dims(nb, bs, hkv, d)
    table = np.full((1, nb + 1), nb, np.int32)
    table[0, :nb] = np.arange(nb)
    k, v = _rows(gen, L, hkv, d), _rows(gen, L, hkv, d)
    kp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
    vp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
    # three writes that start and end inside blocks
    for a, b in ((0, 3), (3, bs + 1), (bs + 1, L)):
        st = oracle.write_bf16(k[None, a:b], v[None, a:b], kp, vp, dims, table,
                               np.array([a], np.int32))
        assert st == oracle.OK
    flat_k = kp.reshape(-1, hkv, d)
    flat_v = vp.reshape(-1, hkv, d)
    assert np.array_equal(flat_k[:L], bits(k))
    assert np.array_equal(flat_v[:L], bits(v))
    assert (flat_k[L:] == BF16_NAN).all() and (flat_v[L:] == BF16_NAN).all()


def test_write_permuted_table_relocates_whole_pages():
    gen = torch.Generator().manual_seed(2)
    bs, hkv, d, L = 8, 2, 16, 45
    nb = 8
    dims = oracle.Dims(nb, bs, hkv, d)
    k, v = _rows(gen, L, hkv, d), _rows(gen, L, hkv, d)
    ident = np.arange(nb, dtype=np.int32)[None]
    perm = np.random.default_rng(3).permutation(nb).astype(np.int32)[None]
    pools = {}
    for name, table in (("id", ident), ("perm", perm)):
        kp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
        vp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
        assert oracle.write_bf16(k[None], v[None], kp, vp, dims, table,
                                 np.zeros(1, np.int32)) == oracle.OK
        pools[name] = (kp, vp)
    for j in range(nb):
        assert np.array_equal(pools["perm"][0][perm[0, j]], pools["id"][0][j])
        assert np.array_equal(pools["perm"][1][perm[0, j]], pools["id"][1][j])
    # the scratch row is never touched
    assert (pools["perm"][0][nb] == BF16_NAN).all()


def _astrai_page_write(k_cache, v_cache, page_table, start_pos, k, v, page_size):
    """AstrAI cache.py PagedCache.write: loop over the pages a chunk touches,
    one indexed assignment per page, all sequences sharing start_pos."""
    seq_len = k.size(1)
    written = 0
    first_page, last_page = start_pos // page_size, (start_pos + seq_len - 1) // page_size
    for pi in range(first_page, last_page + 1):
        phys = page_table[:, pi].long()
        page_start = pi * page_size
        ws = max(page_start, start_pos)
        we = min(page_start + page_size, start_pos + seq_len)
        off, n = ws - page_start, we - ws
        k_cache[phys, off:off + n] = k[:, written:written + n]
        v_cache[phys, off:off + n] = v[:, written:written + n]
        written += n


@pytest.mark.parametrize("start,n", [(0, 1), (5, 11), (13, 40), (31, 2)])
def test_write_matches_page_loop_formulation(start, n):
    gen = torch.Generator().manual_seed(4)
    S, bs, hkv, d, nb = 3, 8, 2, 16, 40
    dims = oracle.Dims(nb, bs, hkv, d)
    mb = (start + n + bs - 1) // bs
    table = torch.randperm(nb, generator=gen)[:S * mb].view(S, mb).to(torch.int32)
    k = torch.randn((S, n, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((S, n, hkv, d), generator=gen).to(torch.bfloat16)
    kc = torch.full(dims.pool_shape, float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    _astrai_page_write(kc, vc, table, start, k, v, bs)
    kp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
    vp = kp.copy()
    assert oracle.write_bf16(k, v, kp, vp, dims, table, np.full(S, start, np.int32)) == oracle.OK
    assert np.array_equal(kp, bits(kc)) and np.array_equal(vp, bits(vc))


def test_write_bad_slots_are_skipped_and_reported():
    bs, hkv, d, nb = 4, 1, 8, 6
    dims = oracle.Dims(nb, bs, hkv, d)
    table = np.array([[0, 1], [nb + 1, 2], [-1, 3], [4, 5]], np.int32)
    k = torch.arange(4 * 2 * d, dtype=torch.float32).view(4, 2, 1, d).to(torch.bfloat16)
    kp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
    vp = kp.copy()
    # seq 1 and 2 name invalid ids, seq 3 writes past its table (position 8 -> block 2)
    start = np.array([0, 0, 0, 7], np.int32)
    st = oracle.write_bf16(k, k, kp, vp, dims, table, start)
    assert st == oracle.BAD_INDEX
    assert np.array_equal(kp[0, 0:2, 0], bits(k[0, :, 0]))        # seq 0 fine
    assert np.array_equal(kp[5, 3, 0], bits(k[3, 0, 0]))          # seq 3 position 7 fine
    untouched = np.ones(nb + 1, bool)
    untouched[[0, 5]] = False
    assert (kp[untouched] == BF16_NAN).all()


def test_all_scratch_row_writes_into_scratch_block():
    """tiny-llm paged_kv.py: the extra block is never allocated and free slots
    write there."""
    bs, hkv, d, nb = 4, 2, 8, 3
    dims = oracle.Dims(nb, bs, hkv, d)
    table = np.full((1, 2), nb, np.int32)
    k = torch.ones((1, 1, hkv, d), dtype=torch.bfloat16)
    kp = np.full(dims.pool_shape, BF16_NAN, np.uint16)
    vp = kp.copy()
    assert oracle.write_bf16(k, k, kp, vp, dims, table, np.array([2], np.int32)) == oracle.OK
    assert (kp[nb, 2] == bits(k[0, 0])).all()
    assert (kp[:nb] == BF16_NAN).all()


def _tiny_llm_gather(pool: torch.Tensor, table: torch.Tensor) -> torch.Tensor:
    """tiny-llm paged_kv.py gather, for a token-major pool [n, bs, H, D]:
    pool[table] is (S, nb, bs, H, D) -> (S, H, nb*bs, D)."""
    S, nb = table.shape
    g = pool[table.long()]                      # (S, nb, bs, H, D)
    g = g.permute(0, 3, 1, 2, 4)                # (S, H, nb, bs, D)
    return g.reshape(S, g.shape[1], nb * pool.shape[1], pool.shape[3])


@pytest.mark.parametrize("cfg", ["tiny", "ragged"])
def test_gather_matches_tiny_llm_view_and_zero_tail(cfg):
    if cfg == "tiny":
        w = W.tiny_decode()
    else:
        w = W.gather_workload("g", 7, [1, 15, 16, 17, 70, 0], 3, 32, 16, out_tokens=80)
    kp, vp, _, _ = oracle_pools_after_step(w, poison=True)
    lens = w.ctx_lens
    out_tokens = int(lens.max()) + 5
    st, ko, vo = oracle.gather(kp, vp, dims_of(w), w.tables, lens, out_tokens)
    assert st == oracle.OK
    from oracle_pools import from_bits
    for pool, out in ((kp, ko), (vp, vo)):
        ref = _tiny_llm_gather(from_bits(pool), w.tables)
        for s in range(w.n_seqs):
            L = int(lens[s])
            assert np.array_equal(out[s, :, :L], bits(ref[s, :, :L]))
            assert (out[s, :, L:] == 0).all()


def test_gather_round_trips_logical_rows():
    w = W.tiny_decode()
    kp, vp, _, _ = oracle_pools_after_step(w)
    lens = w.ctx_lens
    st, ko, vo = oracle.gather(kp, vp, dims_of(w), w.tables, lens, int(lens.max()))
    assert st == oracle.OK
    for s in range(w.n_seqs):
        k, v = logical_rows(w, s)
        L = k.shape[0]
        assert np.array_equal(ko[s, :, :L], bits(k.transpose(0, 1)))
        assert np.array_equal(vo[s, :, :L], bits(v.transpose(0, 1)))


def test_gather_length_beyond_view_is_reported():
    w = W.tiny_decode()
    kp, vp, _, _ = oracle_pools_after_step(w)
    st, _, _ = oracle.gather(kp, vp, dims_of(w), w.tables, w.ctx_lens, 10)
    assert st == oracle.BAD_INDEX


@pytest.mark.parametrize("make", [W.tiny_decode, lambda: W.skewed_prefix_decode(n_seqs=32, median=600,
                                                                 max_len=2000)])
def test_tables_waste_at_most_block_size_minus_one(make):
    """tiny-llm paged_kv.py docstring: at most block_size - 1 wasted slots per
    sequence (its last, partly filled block); tables hold distinct ids except
    for ref-counted shared prefix blocks."""
    w = make()
    ctx = w.ctx_lens
    for s in range(w.n_seqs):
        used = int((w.tables[s] < w.n_blocks).sum())
        assert 0 <= used * w.block_size - int(ctx[s]) <= w.block_size - 1
    ids = w.tables[w.tables < w.n_blocks]
    counts = torch.bincount(ids.long(), minlength=w.n_blocks)
    assert int(counts.max()) <= max(w.group_size, 1)
    if w.shared_blocks:
        assert int((counts == w.group_size).sum()) == w.shared_blocks * (w.n_seqs // w.group_size)


def test_shared_prefix_blocks_hold_one_copy():
    w = W.skewed_prefix_decode(n_seqs=32, median=600, max_len=2000)
    kp, vp, _, _ = oracle_pools_after_step(w)
    lens = w.ctx_lens
    st, ko, _ = oracle.gather(kp, vp, dims_of(w), w.tables, lens, int(lens.max()))
    assert st == oracle.OK
    for s in range(16):  # one group: members see the same first 512 tokens
        assert np.array_equal(ko[s, :, :512], ko[0, :, :512])
        k, _ = logical_rows(w, s)
        assert np.array_equal(ko[s, :, :k.shape[0]], bits(k.transpose(0, 1)))
