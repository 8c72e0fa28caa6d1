"""GPU tests of decode streamed from a host tier (include/pagedkv_stream.h):
staging is bit-exact; the streamed decode equals the oracle's decode over each
whole context, whatever the tiling; residency carries over between calls;
invalidation after a host-tier rewrite; host memory that is not pinned is
refused before any device work."""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import attention_errors, host, i32

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL = 1e-2, 1e-3, 2e-3


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_212_gb300 import build as B
    B.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


def tier(gen, n_host, bs, hkv, d):
    k = torch.randn((n_host, bs, hkv, d), generator=gen).to(torch.bfloat16).pin_memory()
    v = torch.randn((n_host, bs, hkv, d), generator=gen).to(torch.bfloat16).pin_memory()
    return k, v


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_stage_blocks_bit_exact(P):
    gen = torch.Generator().manual_seed(41)
    hk, hv = tier(gen, 30, 16, 4, 128)
    pool_k = torch.zeros((13, 16, 4, 128), dtype=torch.bfloat16, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    pairs = [(0, 3), (29, 0), (7, 12), (7, 5), (15, 1)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.paged_kv_stage_blocks(i32(pairs), hk, hv, pool_k, pool_v, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for src, dst in ((hk, pool_k), (hv, pool_v)):
        ref = np.zeros((13, 16, 4, 128), np.uint16)
        for h, s in pairs:
            ref[s] = bits(src)[h]
        assert np.array_equal(host(dst), ref)


def test_unpinned_host_tier_is_refused(P):
    k = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16)        # pageable
    pool = torch.zeros((3, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.PagedKVError) as e:
        P.paged_kv_stage_blocks(i32([(0, 0)]), k, k, pool, pool)
    assert e.value.status == 1


def scratch(hk, n_slots):
    pool_k = torch.zeros((n_slots + 1,) + tuple(hk.shape[1:]), dtype=torch.bfloat16, device="cuda")
    return pool_k, torch.zeros_like(pool_k)


def run_streamed(P, sp, q, hk, hv, pools, tables, lens, scale):
    pool_k, pool_v = pools
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.paged_decode_streamed(q, hk, hv, pool_k, pool_v, sp, torch.as_tensor(tables, dtype=torch.int32),
                                  torch.as_tensor(lens, dtype=torch.int32), scale, lse_out=lse, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, lse, (pool_k, pool_v)


def oracle_ref(q, hk, hv, tables, lens, scale):
    d = oracle.Dims(hk.shape[0] - 1, hk.shape[1], hk.shape[2], hk.shape[3])   # ids 0 .. n_host - 1
    code, ref, ref_lse = oracle.decode(bits(q.cpu()), bits(hk), bits(hv), d, np.array(tables, np.int32),
                                       np.array(lens, np.int32), scale)
    assert code == 0
    return ref, ref_lse


# 24 and 7 slots: the batch (100 blocks) does not fit, tiles of half the pool
# stage on the copy stream while the tile before is attended; 2 slots: tiles of
# one block; 400 slots: one tile
@pytest.mark.parametrize("n_slots,head_dim,g", [(24, 128, 4), (7, 64, 8), (2, 128, 4), (400, 128, 2)])
def test_streamed_decode_matches_the_oracle(P, n_slots, head_dim, g):
    gen = torch.Generator().manual_seed(9 + n_slots)
    bs, hkv, n_host, n = 16, 4, 90, 6
    hk, hv = tier(gen, n_host, bs, hkv, head_dim)
    lens = [700, 0, 1, 333, 16, 520]
    max_blocks = 44
    perm = torch.randperm(n_host, generator=gen).tolist()
    tables = [[perm[(7 * s + j) % n_host] for j in range(max_blocks)] for s in range(n)]
    tables[3][:5] = tables[0][:5]                          # a shared prefix
    q = torch.randn((n, hkv * g, head_dim), generator=gen).to(torch.bfloat16).cuda()
    scale = 1.0 / head_dim ** 0.5
    sp = P.ScratchPool(n_slots, n)
    pools = scratch(hk, n_slots)
    out, lse, _ = run_streamed(P, sp, q, hk, hv, pools, tables, lens, scale)
    ref, ref_lse = oracle_ref(q, hk, hv, tables, lens, scale)
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    live = np.array(lens) > 0
    assert np.abs(lse.cpu().numpy()[live] - ref_lse[live]).max() <= LSE_TOL
    assert np.all(out.float().cpu().numpy()[~live] == 0) and np.all(np.isneginf(lse.cpu().numpy()[~live]))
    # a second call on the same scratch pool (residency left by the first) gives the same bits
    again, lse2, _ = run_streamed(P, sp, q, hk, hv, pools, tables, lens, scale)
    assert torch.equal(again, out) and torch.equal(lse2, lse)


def test_residency_carries_over_and_invalidation_restages(P):
    gen = torch.Generator().manual_seed(17)
    bs, hkv, d, n_host, n_slots = 16, 4, 128, 40, 64   # the batch fits: a second call stages nothing
    hk, hv = tier(gen, n_host, bs, hkv, d)
    lens = [300, 200]
    tables = [list(range(0, 19)) + [0] * 5, list(range(19, 32)) + [0] * 11]
    t_tab, t_len = torch.tensor(tables, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32)
    q = torch.randn((2, hkv * 4, d), generator=gen).to(torch.bfloat16).cuda()
    scale = 1.0 / d ** 0.5
    # one scratch pool (device memory and its residency) across the calls
    pool_k = torch.zeros((n_slots + 1, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    sp = P.ScratchPool(n_slots, 2)
    out1 = P.paged_decode_streamed(q, hk, hv, pool_k, pool_v, sp, t_tab, t_len, scale).clone()
    torch.cuda.synchronize()          # the staging has read the tier before it is rewritten below
    slots = [sp.lookup(b) for b in range(32)]
    assert all(x >= 0 for x in slots)
    cursor = [0, 0]
    assert sp.plan_tile(t_tab, t_len, bs, cursor)[2] == []       # nothing left to stage
    # rewrite blocks 5 (K) and 7 (V) in the tier and drop their resident copies:
    # the next call restages exactly those two
    hk[5].copy_(torch.randn(hk[5].shape, generator=gen).to(torch.bfloat16))
    hv[7].copy_(torch.randn(hv[7].shape, generator=gen).to(torch.bfloat16))
    sp.invalidate(5)
    sp.invalidate(7)
    assert sp.lookup(5) == -1 and sp.lookup(7) == -1
    out2 = P.paged_decode_streamed(q, hk, hv, pool_k, pool_v, sp, t_tab, t_len, scale)
    torch.cuda.synchronize()
    assert sp.lookup(5) >= 0 and sp.lookup(7) >= 0
    ref, _ = oracle_ref(q, hk, hv, tables, lens, scale)
    mx, mean = attention_errors(out2, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert not torch.equal(out1, out2)


def test_config1_batch_streamed_in_the_benchmarked_shape(P):
    """The Llama-3-8B-shaped batch (8,296 blocks) from a host tier holding the oracle's
    pools, through the 2048-slot scratch pool bench.py --stream 2048 times:
    every output against the oracle's decode over the whole context."""
    from oracle_pools import dims_of, oracle_pools_after_step
    from gpu_support import NTHREADS
    from paged_kv_cache_212_gb300 import workloads as W
    w = W.llama8b_decode()
    kp, vp, _, _ = oracle_pools_after_step(w, poison=True)
    code, ref, ref_lse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale,
                                       n_threads=NTHREADS)
    assert code == 0
    hk = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16).pin_memory()
    sp = P.ScratchPool(2048, w.n_seqs)
    pools = scratch(hk, 2048)
    q = w.q.cuda()
    out, lse, _ = run_streamed(P, sp, q, hk, hv, pools, w.tables, w.ctx_lens, w.softmax_scale)
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_TOL
