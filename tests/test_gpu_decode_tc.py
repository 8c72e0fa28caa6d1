"""Parity of the tensor-core decode (tcgen05, int8 pages, head_dim 128) with the
CPU oracle, through the C ABI.

The kernel is selected with PKV_DECODE_IMPL=tc.  It shares the work list,
the producer and the partial merge with the mma.sync kernel but contracts
128-token tiles on the 5th-generation tensor cores with the query heads
padded to 16, so the cases cover group sizes 1, 4 and 8, lengths around
the 16-token stages and the 128-token tiles, fixed and automatic splits, the
fused write + decode step, table permutations and the error paths.  Bar: the
int8 tolerance of the mma.sync kernel (max-abs 2e-2 against the oracle
computed from the same codes and scales; lse within 2e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import NTHREADS, attention_errors, dev, host, i32
from oracle_pools import dims_of, oracle_pools_after_step
from paged_kv_cache_212_gb300 import workloads as W

pytestmark = pytest.mark.gpu

INT8_MAX, LSE_TOL = 2e-2, 2e-3


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_212_gb300 import build
    build.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


@pytest.fixture(autouse=True)
def tensor_core_path(monkeypatch):
    monkeypatch.setenv("PKV_DECODE_IMPL", "tc")


_CASES = {
    # lengths around the 16-token stages and the 128-token tiles; G = 4
    "g4": lambda: W.decode_workload("tc4", 31, [0, 1, 14, 15, 16, 17, 111, 112, 127, 128, 129, 300, 1000], 32, 8,
                                    128, 16, n_new=3, kv_format="int8"),
    # G = 8 and block size 32
    "g8": lambda: W.decode_workload("tc8", 32, [5, 127, 129, 640, 2000], 64, 8, 128, 32, n_new=1, kv_format="int8"),
    # G = 8 with four kv heads (one scale box per CTA pair of heads)
    "g8h4": lambda: W.decode_workload("tc8h4", 33, [40, 250, 513], 32, 4, 128, 16, n_new=2, kv_format="int8"),
    # G = 1
    "g1": lambda: W.decode_workload("tc1", 34, [3, 130, 777], 8, 8, 128, 16, n_new=1, kv_format="int8"),
}
_CACHE = {}


def case(name):
    if name not in _CACHE:
        w = W.llama8b_decode_int8() if name == "llama8b_int8" else _CASES[name]()
        _CACHE[name] = (w, oracle_pools_after_step(w, poison=True))
    return _CACHE[name]


def run(P, w, pools, split=None, tables=None, ctx=None):
    kp, vp, ks, vs = pools
    tables = w.tables if tables is None else tables
    ctx = w.ctx_lens if ctx is None else ctx
    q = w.q.cuda()
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.paged_decode_attention(q, dev(kp), dev(vp), i32(tables), i32(ctx), w.softmax_scale,
                                   k_scales=dev(ks), v_scales=dev(vs),
                                   split_tokens=w.split_tokens if split is None else split, lse_out=lse,
                                   max_total_ctx_tokens=int(torch.as_tensor(ctx).sum()), dev_status=st)
    torch.cuda.synchronize()
    return out, lse, int(st.item())


def reference(w, pools, tables=None, ctx=None):
    kp, vp, ks, vs = pools
    code, out, lse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables if tables is None else tables,
                                   w.ctx_lens if ctx is None else ctx, w.softmax_scale, ks, vs, n_threads=NTHREADS)
    assert code == oracle.OK
    return out, lse


def check(out, lse, ref, ref_lse):
    mx, _ = attention_errors(out, ref)
    assert mx <= INT8_MAX, mx
    g = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(g), np.isneginf(ref_lse))
    if fin.any():
        assert np.abs(g[fin] - ref_lse[fin]).max() <= LSE_TOL


@pytest.mark.parametrize("name", ["llama8b_int8", "g4", "g8", "g8h4", "g1"])
def test_tc_decode_int8_parity(P, name):
    w, pools = case(name)
    out, lse, st = run(P, w, pools)
    assert st == 0
    check(out, lse, *reference(w, pools))


@pytest.mark.parametrize("split", [16, 128, 144, 512, 4096])
def test_tc_decode_fixed_splits(P, split):
    w, pools = case("g4")
    out, lse, st = run(P, w, pools, split=split)
    assert st == 0
    check(out, lse, *reference(w, pools))


def test_tc_decode_identity_vs_permuted_tables_bit_exact(P):
    # the same logical pages under another physical placement give the same bits
    w, pools = case("g8")
    kp, vp, ks, vs = pools
    nb = kp.shape[0] - 1
    perm = np.random.default_rng(5).permutation(nb)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(nb)
    kp2, vp2 = kp.copy(), vp.copy()
    ks2, vs2 = ks.copy(), vs.copy()
    kp2[:nb], vp2[:nb] = kp[inv], vp[inv]
    ks2[:nb], vs2[:nb] = ks[inv], vs[inv]
    t = np.asarray(w.tables).copy()
    used = t < nb
    t[used] = perm[t[used]]
    a, la, sa = run(P, w, pools)
    b, lb, sb = run(P, w, (kp2, vp2, ks2, vs2), tables=torch.as_tensor(t))
    assert sa == 0 and sb == 0
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_tc_decode_step_fused_write(P):
    # paged_decode_step: the int8 write of the step's rows, then the decode, in one call
    w = _CASES["g4"]()
    from oracle_pools import empty_pools, write_prefix
    kp, vp, ks, vs = empty_pools(w, poison=True)
    write_prefix(w, kp, vp, ks, vs)
    gk, gv, gks, gvs = dev(kp), dev(vp), dev(ks), dev(vs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = w.q.cuda()
    out = P.paged_decode_step(w.k_new.cuda(), w.v_new.cuda(), i32(w.start_pos), q, gk, gv, i32(w.tables),
                              i32(w.ctx_lens), w.softmax_scale, k_scales=gks, v_scales=gvs, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    after = oracle_pools_after_step(w, poison=True)
    assert np.array_equal(host(gk), after[0]) and np.array_equal(host(gv), after[1])
    ref, _ = reference(w, after)
    mx, _ = attention_errors(out, ref)
    assert mx <= INT8_MAX, mx


def test_tc_decode_bad_table_entry_is_flagged(P):
    # a table entry outside [0, n_blocks]: the status bit, no fault
    w, pools = case("g4")
    t = np.asarray(w.tables).copy()
    t[5, 0] = 10 ** 6
    _, _, st = run(P, w, pools, tables=torch.as_tensor(t))
    assert st & 1   # PKV_DEV_BAD_BLOCK_ID
