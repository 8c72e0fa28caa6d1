"""Pins for the oracle's paged decode and chunked prefill attention (CPU only).

Independent references:
  * textbook softmax attention in numpy float64 on a contiguous copy built by
    torch indexing (tiny-llm paged_kv.py: gather the blocks, then attention);
  * torch.nn.functional.scaled_dot_product_attention in float64 on the
    tiny-llm-style gathered view with the decode mask k_pos < ctx (tiny-llm
    paged_kv.py, begin_step attn_mask) and GQA by repeat-interleave;
  * closed forms: one token gives o = v_0; identical keys give mean(V); a
    dominating key gives its value row;
  * invariants: identity and permuted tables give bit-identical results;
    poisoned (NaN) unused memory changes nothing; split-KV with the LSE merge
    equals the unsplit result.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle_pools import bits, dims_of, f64, from_bits, logical_rows, oracle_pools_after_step
from paged_kv_cache_212_gb300 import workloads as W


def _numpy_attention(q, k, v, scale):
    """q [Hq, D], k/v [L, Hkv, D] float64 -> (o [Hq, D], lse [Hq])."""
    Hq, Hkv = q.shape[0], k.shape[1]
    G = Hq // Hkv
    o = np.zeros_like(q)
    lse = np.zeros(Hq)
    for h in range(Hq):
        kh, vh = k[:, h // G], v[:, h // G]
        s = scale * (kh @ q[h])
        m = s.max()
        w = np.exp(s - m)
        o[h] = (w[:, None] * vh).sum(0) / w.sum()
        lse[h] = m + math.log(w.sum())
    return o, lse


def _small_decode(seed=11, lens=(1, 16, 17, 40, 63), hq=8, hkv=2, d=32, bs=16, fmt="bf16"):
    return W.decode_workload("t", seed, list(lens), hq, hkv, d, bs, n_new=1, kv_format=fmt)


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
def test_decode_equals_textbook_softmax_on_contiguous_copy(fmt):
    w = _small_decode(fmt=fmt)
    kp, vp, ks, vs = oracle_pools_after_step(w)
    st, out, lse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale,
                                 ks, vs)
    assert st == oracle.OK
    q = f64(w.q)
    for s in range(w.n_seqs):
        L = int(w.ctx_lens[s])
        tab = w.tables[s].long()
        # contiguous copy by torch indexing of whole pages, cut at L
        if fmt == "bf16":
            k = f64(from_bits(kp)[tab].reshape(-1, w.n_kv_heads, w.head_dim)[:L])
            v = f64(from_bits(vp)[tab].reshape(-1, w.n_kv_heads, w.head_dim)[:L])
        else:
            kc = torch.from_numpy(kp)[tab].reshape(-1, w.n_kv_heads, w.head_dim)[:L].double()
            vc = torch.from_numpy(vp)[tab].reshape(-1, w.n_kv_heads, w.head_dim)[:L].double()
            ksc = torch.from_numpy(ks)[tab].reshape(-1, w.n_kv_heads)[:L].double()
            vsc = torch.from_numpy(vs)[tab].reshape(-1, w.n_kv_heads)[:L].double()
            k = (kc * ksc[..., None]).numpy()
            v = (vc * vsc[..., None]).numpy()
        o_ref, lse_ref = _numpy_attention(q[s], k, v, w.softmax_scale)
        np.testing.assert_allclose(out[s], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[s], lse_ref, rtol=0, atol=1e-12)


def _sdpa_decode(w, kp, vp):
    """tiny-llm semantics: gather (S, H, nb*bs, D), mask k_pos < ctx, SDPA."""
    tab = w.tables.long()
    S, nb = tab.shape
    def gather(pool):
        g = from_bits(pool).double()[tab]                  # (S, nb, bs, H, D)
        return g.permute(0, 3, 1, 2, 4).reshape(S, w.n_kv_heads, nb * w.block_size, w.head_dim)
    K, V = gather(kp), gather(vp)
    K = torch.nan_to_num(K)  # slots past ctx are masked; SDPA would still multiply NaN by 0
    V = torch.nan_to_num(V)
    G = w.n_q_heads // w.n_kv_heads
    K = K.repeat_interleave(G, dim=1)
    V = V.repeat_interleave(G, dim=1)
    q = w.q.double()[:, :, None, :]                         # (S, Hq, 1, D)
    k_pos = torch.arange(nb * w.block_size)
    mask = (k_pos[None, :] < w.ctx_lens[:, None])[:, None, None, :]
    o = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=w.softmax_scale)
    return o[:, :, 0].numpy()


@pytest.mark.parametrize("make", [W.tiny_decode, lambda: _small_decode(hq=16, hkv=4, d=64, bs=32)])
def test_decode_equals_sdpa_on_gathered_view(make):
    w = make()
    kp, vp, _, _ = oracle_pools_after_step(w)
    st, out, _ = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale)
    assert st == oracle.OK
    np.testing.assert_allclose(out, _sdpa_decode(w, kp, vp), rtol=0, atol=1e-12)


def test_gqa_maps_query_head_to_contiguous_group():
    """kv head = h // G: the head-interleaved alternative (h % Hkv) differs."""
    w = _small_decode(hq=8, hkv=4, d=16)
    kp, vp, _, _ = oracle_pools_after_step(w)
    _, out, _ = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale)
    q = f64(w.q)
    s = 3
    k, v = (f64(x) for x in logical_rows(w, s))
    o_ref, _ = _numpy_attention(q[s], k, v, w.softmax_scale)
    np.testing.assert_allclose(out[s], o_ref, atol=1e-12)
    perm = [h % 4 * 2 + h // 4 for h in range(8)]  # query order that pairs h with h % Hkv
    o_alt, _ = _numpy_attention(q[s][perm], k, v, w.softmax_scale)
    assert np.abs(out[s][perm] - o_alt).max() > 1e-3


def test_closed_forms():
    gen = torch.Generator().manual_seed(3)
    bs, hkv, d, nb = 16, 1, 16, 8
    dims = oracle.Dims(nb, bs, hkv, d)
    table = torch.randperm(nb, generator=gen)[:4].to(torch.int32)[None]
    q = torch.randn((1, 2, d), generator=gen).to(torch.bfloat16)
    # one token: o = v_0 exactly, lse = scale * q.k_0
    k = torch.randn((1, 40, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((1, 40, hkv, d), generator=gen).to(torch.bfloat16)
    kp = np.full(dims.pool_shape, 0x7FC0, np.uint16)
    vp = kp.copy()
    oracle.write_bf16(k, v, kp, vp, dims, table, np.zeros(1, np.int32))
    st, out, lse = oracle.decode(q, kp, vp, dims, table, np.array([1], np.int32), 0.25)
    assert st == 0
    assert np.array_equal(out[0], np.repeat(f64(v[0, 0]), 2, axis=0))
    np.testing.assert_allclose(lse[0], 0.25 * f64(q[0]) @ f64(k[0, 0, 0]), atol=1e-14)
    # identical keys: uniform weights -> mean of V, lse = s + ln L
    kk = k.clone()
    kk[:] = k[0, 0]
    oracle.write_bf16(kk, v, kp, vp, dims, table, np.zeros(1, np.int32))
    st, out, lse = oracle.decode(q, kp, vp, dims, table, np.array([40], np.int32), 0.25)
    np.testing.assert_allclose(out[0], np.repeat(f64(v[0]).mean(0), 2, axis=0), atol=1e-14)
    np.testing.assert_allclose(lse[0], 0.25 * f64(q[0]) @ f64(k[0, 0, 0]) + math.log(40),
                               atol=1e-13)
    # one key aligned with q and large scale: o -> v of that key
    kd = torch.zeros_like(k)
    kd[0, 23, 0] = q[0, 0]
    oracle.write_bf16(kd, v, kp, vp, dims, table, np.zeros(1, np.int32))
    st, out, _ = oracle.decode(q, kp, vp, dims, table, np.array([40], np.int32), 1000.0)
    np.testing.assert_allclose(out[0, 0], f64(v[0, 23, 0]), atol=1e-12)


def test_empty_context_gives_zero_output_and_minus_inf_lse():
    w = _small_decode(lens=(0, 5))
    kp, vp, _, _ = oracle_pools_after_step(w)
    ctx = torch.tensor([0, 6], dtype=torch.int32)
    st, out, lse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, ctx, w.softmax_scale)
    assert st == 0 and (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(out[1]).all()


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
def test_identity_and_permuted_tables_agree_bit_exactly(fmt):
    w = _small_decode(fmt=fmt, lens=(3, 33, 80))
    kp, vp, ks, vs = oracle_pools_after_step(w)
    res = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale, ks, vs)
    # relocate every page to a fresh permutation and rewrite the table
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.n_blocks)
    move = np.append(perm, w.n_blocks)           # scratch stays scratch
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[move], vp2[move] = kp, vp
    ks2 = vs2 = None
    if fmt == "int8":
        ks2, vs2 = np.empty_like(ks), np.empty_like(vs)
        ks2[move], vs2[move] = ks, vs
    t2 = torch.from_numpy(move[w.tables.numpy()]).to(torch.int32)
    res2 = oracle.decode(w.q, kp2, vp2, dims_of(w), t2, w.ctx_lens, w.softmax_scale, ks2, vs2)
    assert res[0] == res2[0] == 0
    assert np.array_equal(res[1], res2[1]) and np.array_equal(res[2], res2[2])


def test_poisoned_unused_memory_is_never_read():
    w = _small_decode(lens=(5, 20, 47))
    kp, vp, _, _ = oracle_pools_after_step(w, poison=True)
    st, out, lse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale)
    assert st == 0 and np.isfinite(out).all() and np.isfinite(lse).all()
    kz, vz, _, _ = oracle_pools_after_step(w, poison=False)
    t2 = w.tables.clone()
    for s in range(w.n_seqs):  # garbage ids past the context are never followed
        nb = -(-int(w.ctx_lens[s]) // w.block_size)
        t2[s, nb:] = 10**6
    st2, out2, _ = oracle.decode(w.q, kz, vz, dims_of(w), t2, w.ctx_lens, w.softmax_scale)
    assert st2 == 0 and np.array_equal(out, out2)


@pytest.mark.parametrize("split", [1, 7, 16, 50, 512])
def test_split_merge_equals_unsplit(split):
    w = _small_decode(lens=(1, 16, 17, 99, 200))
    kp, vp, _, _ = oracle_pools_after_step(w)
    _, out, lse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale)
    st, out_s, lse_s = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens,
                                     w.softmax_scale, split_tokens=split)
    assert st == 0
    np.testing.assert_allclose(out_s, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_s, lse, rtol=0, atol=1e-12)


def test_threads_do_not_change_results():
    w = _small_decode(lens=(100, 3, 250, 64))
    kp, vp, _, _ = oracle_pools_after_step(w)
    a = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale)
    b = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale,
                      n_threads=3)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_decode_reports_context_beyond_table():
    w = _small_decode(lens=(5, 20))
    kp, vp, _, _ = oracle_pools_after_step(w)
    ctx = torch.tensor([6, w.max_blocks * w.block_size + 1], dtype=torch.int32)
    st, out, _ = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, ctx, w.softmax_scale)
    assert st == oracle.BAD_INDEX and (out[1] == 0).all()


# ---------------------------------------------------------------------------
# chunked prefill
# ---------------------------------------------------------------------------

def _sdpa_prefill(w, kp, vp):
    tab = w.tables.long()
    S, nb = tab.shape
    def gather(pool):
        g = from_bits(pool).double()[tab]
        g = g.permute(0, 3, 1, 2, 4).reshape(S, w.n_kv_heads, nb * w.block_size, w.head_dim)
        return torch.nan_to_num(g).repeat_interleave(w.n_q_heads // w.n_kv_heads, dim=1)
    K, V = gather(kp), gather(vp)
    q = w.q.double().permute(0, 2, 1, 3)                          # (S, Hq, C, D)
    pos = w.stored_lens[:, None] + torch.arange(w.n_new)[None]    # absolute query positions
    k_pos = torch.arange(nb * w.block_size)
    mask = (k_pos[None, None, :] <= pos[:, :, None])[:, None]     # (S, 1, C, keys)
    o = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=w.softmax_scale)
    return o.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("prefix", [(0, 5, 16, 37), (0, 0), (100, 1)])
def test_prefill_equals_masked_sdpa(prefix):
    w = W.prefill_workload("p", 5, list(prefix), 24, 8, 2, 32, 16)
    kp, vp, _, _ = oracle_pools_after_step(w)
    st, out, lse = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens,
                                  w.softmax_scale, n_threads=2)
    assert st == 0
    np.testing.assert_allclose(out, _sdpa_prefill(w, kp, vp), rtol=0, atol=1e-12)


def test_prefill_without_prefix_is_causal_sdpa():
    w = W.prefill_workload("p", 6, [0, 0], 40, 4, 4, 16, 16)
    kp, vp, _, _ = oracle_pools_after_step(w)
    _, out, _ = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens, w.softmax_scale)
    q = w.q.double().permute(0, 2, 1, 3)
    k = w.k_new.double().permute(0, 2, 1, 3)
    v = w.v_new.double().permute(0, 2, 1, 3)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=w.softmax_scale)
    np.testing.assert_allclose(out, o.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_prefill_row_equals_decode_at_that_position():
    w = W.prefill_workload("p", 7, [30, 3], 20, 8, 2, 32, 16)
    kp, vp, _, _ = oracle_pools_after_step(w)
    sel = np.zeros((2, 20), bool)
    sel[0, 7] = sel[1, 19] = True
    _, out, lse = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens,
                                 w.softmax_scale, row_select=sel)
    for s, i in ((0, 7), (1, 19)):
        ctx = torch.tensor([int(w.stored_lens[s]) + i + 1], dtype=torch.int32)
        _, od, ld = oracle.decode(w.q[s, i][None], kp, vp, dims_of(w), w.tables[s:s + 1], ctx,
                                  w.softmax_scale)
        assert np.array_equal(out[s, i], od[0]) and np.array_equal(lse[s, i], ld[0])
    assert np.isnan(out[0, 0]).all()
