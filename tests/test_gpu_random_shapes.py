"""Parity over seeded random shapes: every decode and prefill configuration the
library accepts, drawn at random (head_dim 64 / 128, group sizes, kv heads,
block sizes, length mixes with empty, one-token and long contexts, several
new rows, fixed and automatic splits, bf16 and int8 pages, every decode
kernel), against the float64 oracle.

Decode runs as the fused step (paged_decode_step): the pools must equal the
oracle's write bit for bit and the output must match the oracle's decode of
them (bf16 pages: max-abs 1e-2, mean-abs 1e-3; int8 pages: max-abs 2e-2; lse
within 2e-3, and -inf exactly where the context is empty).  Prefill runs on
pools holding the oracle's chunk write, every row checked.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import NTHREADS, attention_errors, dev, host, i32
from oracle_pools import dims_of, empty_pools, oracle_pools_after_step, write_prefix
from paged_kv_cache_212_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, INT8_MAX, LSE_TOL = 1e-2, 1e-3, 2e-2, 2e-3
DECODE_SEEDS = list(range(20))      # 16..19: short contexts, the one-launch small-batch path
PREFILL_SEEDS = list(range(8))


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_212_gb300 import build
    build.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


def _lengths(rng, n, cap):
    """A mix of empty, one-token, short, medium and long contexts."""
    kinds = rng.choice(5, size=n, p=[0.05, 0.1, 0.3, 0.35, 0.2])
    hi = np.minimum(np.array([0, 1, 40, 600, cap])[kinds], cap)
    lo = np.minimum(np.array([0, 1, 2, 40, 600])[kinds], hi)
    return [int(rng.integers(a, b + 1)) for a, b in zip(lo, hi)]


def draw_decode_case(seed):
    rng = np.random.default_rng(7000 + seed)
    if seed >= 16:
        # bf16 pages, automatic splitting, at most 240 stored tokens: a batch the
        # one-launch path takes whole
        D = int(rng.choice([64, 128]))
        Hkv, G, bs = int(rng.choice([1, 2, 4, 8])), int(rng.choice([1, 2, 4, 8])), int(rng.choice([16, 32, 64]))
        n_seqs = int(rng.integers(1, 152 // Hkv + 1))
        lens = _lengths(rng, n_seqs, 240)
        w = W.decode_workload(f"random small decode {seed}", 9000 + seed, lens, Hkv * G, Hkv, D, bs,
                              n_new=int(rng.integers(1, 5)))
        return w, "auto"
    int8 = bool(rng.random() < 0.4)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([4, 8])) if int8 else int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32, 64, 128]))
    n_seqs = int(rng.integers(1, 41))
    lens = _lengths(rng, n_seqs, 3000)
    n_new = int(rng.integers(1, 5))
    split = int(rng.choice([0, 0, 16, 64, 512]))
    impls = ["auto", "split"]
    if int8 and D == 128 and G <= 8:
        impls.append("tc")
    impl = str(rng.choice(impls))
    w = W.decode_workload(f"random decode {seed}", 9000 + seed, lens, Hkv * G, Hkv, D, bs, n_new=n_new,
                          kv_format="int8" if int8 else "bf16", split_tokens=split)
    return w, impl


def draw_prefill_case(seed):
    rng = np.random.default_rng(8000 + seed)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    while Hkv * G > 32:
        G //= 2
    bs = int(rng.choice([16, 32, 64]))
    n_seqs = int(rng.integers(1, 5))
    prefixes = [int(x) for x in rng.integers(0, 1001, n_seqs)]
    prefixes[int(rng.integers(0, n_seqs))] = int(rng.choice([0, 1, 127, 128]))
    chunk = int(rng.integers(1, 201))
    return W.prefill_workload(f"random prefill {seed}", 9500 + seed, prefixes, chunk, Hkv * G, Hkv, D, bs)


@pytest.mark.parametrize("seed", DECODE_SEEDS)
def test_random_decode_step(P, seed, monkeypatch):
    w, impl = draw_decode_case(seed)
    if impl == "auto":
        monkeypatch.delenv("PKV_DECODE_IMPL", raising=False)
    else:
        monkeypatch.setenv("PKV_DECODE_IMPL", impl)
    int8 = w.kv_format == "int8"
    kp, vp, ks, vs = empty_pools(w, poison=True)
    write_prefix(w, kp, vp, ks, vs)
    gk, gv = dev(kp), dev(vp)
    gks, gvs = (dev(ks), dev(vs)) if int8 else (None, None)
    q = w.q.cuda()
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.paged_decode_step(w.k_new.cuda(), w.v_new.cuda(), i32(w.start_pos), q, gk, gv, i32(w.tables),
                              i32(w.ctx_lens), w.softmax_scale, k_scales=gks, v_scales=gvs,
                              split_tokens=w.split_tokens, lse_out=lse, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, rks, rvs = oracle_pools_after_step(w, poison=True)
    assert np.array_equal(host(gk), rk) and np.array_equal(host(gv), rv)
    if int8:
        assert np.array_equal(host(gks).view(np.uint32), rks.view(np.uint32))
        assert np.array_equal(host(gvs).view(np.uint32), rvs.view(np.uint32))
    code, ref, ref_lse = oracle.decode(w.q, rk, rv, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale, rks, rvs,
                                       n_threads=NTHREADS)
    assert code == oracle.OK
    mx, mean = attention_errors(out, ref)
    if int8:
        assert mx <= INT8_MAX, (impl, mx)
    else:
        assert mx <= BF16_MAX and mean <= BF16_MEAN, (impl, mx, mean)
    g = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(g), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    if fin.any():
        assert np.abs(g[fin] - ref_lse[fin]).max() <= LSE_TOL


@pytest.mark.parametrize("seed", PREFILL_SEEDS)
def test_random_prefill(P, seed):
    w = draw_prefill_case(seed)
    kp, vp, _, _ = oracle_pools_after_step(w, poison=True)
    q = w.q.cuda()
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.paged_prefill_attention(q, dev(kp), dev(vp), i32(w.tables), i32(w.stored_lens), w.softmax_scale,
                                    lse_out=lse, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    code, ref, ref_lse = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens, w.softmax_scale,
                                        n_threads=NTHREADS)
    assert code == 0
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_TOL
