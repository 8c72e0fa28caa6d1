"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Inputs are the seeded synthetic workloads; every pool the GPU reads is built
by the ORACLE's own write from the drawn rows (unused memory poisoned with
NaN / code 127 + NaN scales) and copied to the device, so no oracle input comes
from the CUDA path.  Bars:
  * write, int8 write (codes and scales) and gather: bit-exact, whole pools;
  * attention, bf16 pages: max-abs <= 1e-2 and mean-abs <= 1e-3 against the
    float64 oracle; int8 pages: max-abs <= 2e-2 against the oracle computed
    from the same codes and scales; lse within 2e-3 (fp32 accumulation).
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


@pytest.fixture(scope="session")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_212_gb300 import build
    build.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


_CACHE = {}


def workload(name):
    """Full-size named workloads are drawn once per session."""
    if name not in _CACHE:
        makers = {
            "tiny": W.tiny_decode, "llama8b": W.llama8b_decode, "llama8b_int8": W.llama8b_decode_int8,
            "chunked_prefill": W.chunked_prefill, "skewed_prefix": W.skewed_prefix_decode,
            "gather_16x2048": W.gather_16x2048,
            "ragged_d64": lambda: W.decode_workload("ragged", 5, [1, 15, 16, 17, 31, 33, 200, 511], 16, 4, 64, 16),
            "ragged_g8_bs32": lambda: W.decode_workload("g8", 6, [1, 31, 32, 33, 100, 700, 1500], 64, 8, 128, 32),
            "ragged_g1": lambda: W.decode_workload("g1", 7, [3, 40, 129], 4, 4, 128, 16),
            # at the one-launch path's limits (the context in shared memory): 512 tokens at
            # head_dim 64 (block size 32), 256 at head_dim 128; G = 8
            "small_limits": lambda: W.decode_workload("sl", 15, [0, 1, 511, 300, 511], 64, 8, 64, 32),
            "small_limits_d128": lambda: W.decode_workload("sl128", 16, [255, 0, 100, 17, 255], 64, 8, 128, 16),
            "int8_small": lambda: W.decode_workload("i8", 8, [0, 1, 15, 16, 100, 333], 16, 4, 128, 16, n_new=3,
                                                    kv_format="int8"),
            "int8_d64": lambda: W.decode_workload("i8d64", 9, [5, 77, 300], 8, 4, 64, 32, n_new=2,
                                                  kv_format="int8"),
            "prefill_small": lambda: W.prefill_workload("p", 10, [0, 5, 16, 100, 250], 40, 8, 2, 64, 16),
            "prefill_g8": lambda: W.prefill_workload("p8", 11, [0, 33, 300], 37, 64, 8, 128, 16),
            "prefill_g1": lambda: W.prefill_workload("p1", 12, [7, 64], 70, 4, 4, 128, 32),
            # more sequences than the kernel orders by prefix length (natural order)
            "prefill_many": lambda: W.prefill_workload("pm", 13, [(37 * i) % 301 for i in range(40)], 9, 8, 2,
                                                       64, 16),
            # equal prefix lengths: the longest-first order breaks ties by index
            "prefill_ties": lambda: W.prefill_workload("pt", 14, [100, 100, 0, 100, 37], 20, 16, 4, 128, 16),
        }
        _CACHE[name] = makers[name]()
    return _CACHE[name]


_POOLS = {}


def pools(name, after_step=True):
    key = (name, after_step)
    if key not in _POOLS:
        w = workload(name)
        if after_step:
            _POOLS[key] = oracle_pools_after_step(w, poison=True)
        else:
            kp, vp, ks, vs = empty_pools(w, poison=True)
            write_prefix(w, kp, vp, ks, vs)
            _POOLS[key] = (kp, vp, ks, vs)
    return _POOLS[key]


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------------------
# writes and gather: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "llama8b", "chunked_prefill", "skewed_prefix", "ragged_d64"])
def test_write_bf16_bit_exact(P, name):
    w = workload(name)
    kp, vp, _, _ = pools(name, after_step=False)
    gk, gv = dev(kp), dev(vp)
    st = status_tensor()
    P.paged_kv_write(w.k_new.cuda(), w.v_new.cuda(), gk, gv, i32(w.tables), i32(w.start_pos), dev_status=st)
    torch.cuda.synchronize()
    rk, rv, _, _ = pools(name, after_step=True)
    assert int(st.item()) == 0
    assert np.array_equal(host(gk), rk)
    assert np.array_equal(host(gv), rv)


@pytest.mark.parametrize("name", ["llama8b_int8", "int8_small", "int8_d64"])
def test_write_int8_bit_exact(P, name):
    w = workload(name)
    kp, vp, ks, vs = pools(name, after_step=False)
    gk, gv, gks, gvs = dev(kp), dev(vp), dev(ks), dev(vs)
    st = status_tensor()
    P.paged_kv_write_int8(w.k_new.cuda(), w.v_new.cuda(), gk, gv, gks, gvs, i32(w.tables), i32(w.start_pos),
                          dev_status=st)
    torch.cuda.synchronize()
    rk, rv, rks, rvs = pools(name, after_step=True)
    assert int(st.item()) == 0
    assert np.array_equal(host(gk), rk) and np.array_equal(host(gv), rv)
    # scales compared as bit patterns (NaN poison included)
    assert np.array_equal(host(gks).view(np.uint32), rks.view(np.uint32))
    assert np.array_equal(host(gvs).view(np.uint32), rvs.view(np.uint32))


def test_write_to_bad_slots_is_flagged_and_skipped(P):
    w = workload("tiny")
    kp, vp, _, _ = pools("tiny", after_step=False)
    gk, gv = dev(kp), dev(vp)
    tables = w.tables.clone()
    tables[1, int(w.start_pos[1]) // w.block_size] = w.n_blocks + 5      # id out of range
    start = w.start_pos.clone()
    start[2] = w.max_blocks * w.block_size                                # past the table
    st = status_tensor()
    P.paged_kv_write(w.k_new.cuda(), w.v_new.cuda(), gk, gv, i32(tables), i32(start), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == (P.DEV_BAD_BLOCK_ID | P.DEV_BAD_POSITION)
    rk = kp.copy()
    rv = vp.copy()
    code = oracle.write_bf16(w.k_new, w.v_new, rk, rv, dims_of(w), tables, start)
    assert code == oracle.BAD_INDEX
    assert np.array_equal(host(gk), rk) and np.array_equal(host(gv), rv)


@pytest.mark.parametrize("name,extra", [("gather_16x2048", 0), ("tiny", 13), ("ragged_d64", 1), ("ragged_g8_bs32", 7)])
def test_gather_bit_exact(P, name, extra):
    w = workload(name)
    kp, vp, _, _ = pools(name, after_step=w.kind != "gather")
    lens = w.ctx_lens if w.kind != "gather" else w.stored_lens
    out_tokens = int(lens.max()) + extra
    st = status_tensor()
    ko, vo = P.paged_kv_gather(dev(kp), dev(vp), i32(w.tables), i32(lens), out_tokens, dev_status=st)
    torch.cuda.synchronize()
    code, rk, rv = oracle.gather(kp, vp, dims_of(w), w.tables, lens, out_tokens)
    assert code == oracle.OK and int(st.item()) == 0
    assert np.array_equal(host(ko), rk) and np.array_equal(host(vo), rv)


def test_gather_zero_length_and_bad_length(P):
    w = workload("tiny")
    kp, vp, _, _ = pools("tiny")
    lens = torch.tensor([0, 5, 10**6, 65], dtype=torch.int32)
    st = status_tensor()
    ko, vo = P.paged_kv_gather(dev(kp), dev(vp), i32(w.tables), i32(lens), 70, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.DEV_BAD_LENGTH
    ok_lens = lens.clone()
    ok_lens[2] = 0  # the bad sequence's view is zero-filled, like an empty one
    _, rk, rv = oracle.gather(kp, vp, dims_of(w), w.tables, ok_lens, 70)
    assert np.array_equal(host(ko), rk) and np.array_equal(host(vo), rv)


# ---------------------------------------------------------------------------
# decode attention
# ---------------------------------------------------------------------------

def run_decode(P, w, kp, vp, ks=None, vs=None, split=None, tables=None, ctx=None, lse=True):
    tables = w.tables if tables is None else tables
    ctx = w.ctx_lens if ctx is None else ctx
    q = w.q.cuda()
    lse_t = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda") if lse else None
    st = status_tensor()
    out = P.paged_decode_attention(q, dev(kp), dev(vp), i32(tables), i32(ctx), w.softmax_scale,
                                   k_scales=None if ks is None else dev(ks),
                                   v_scales=None if vs is None else dev(vs),
                                   split_tokens=w.split_tokens if split is None else split,
                                   lse_out=lse_t, max_total_ctx_tokens=int(torch.as_tensor(ctx).sum()),
                                   dev_status=st)
    torch.cuda.synchronize()
    return out, lse_t, int(st.item())


def oracle_decode(w, kp, vp, ks=None, vs=None, tables=None, ctx=None):
    tables = w.tables if tables is None else tables
    ctx = w.ctx_lens if ctx is None else ctx
    code, out, lse = oracle.decode(w.q, kp, vp, dims_of(w), tables, ctx, w.softmax_scale, ks, vs,
                                   n_threads=NTHREADS)
    assert code == oracle.OK
    return out, lse


def check_lse(lse_gpu, lse_ref):
    g = lse_gpu.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(g), np.isneginf(lse_ref))
    if fin.any():
        assert np.abs(g[fin] - lse_ref[fin]).max() <= LSE_TOL


@pytest.mark.parametrize("name", ["tiny", "llama8b", "skewed_prefix", "ragged_d64", "ragged_g8_bs32", "ragged_g1", "small_limits",
                                  "small_limits_d128"])
def test_decode_bf16_parity(P, name, decode_impl):
    w = workload(name)
    kp, vp, _, _ = pools(name)
    out, lse, st = run_decode(P, w, kp, vp)
    ref, ref_lse = oracle_decode(w, kp, vp)
    assert st == 0
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    check_lse(lse, ref_lse)


@pytest.mark.parametrize("name", ["llama8b_int8", "int8_small", "int8_d64"])
def test_decode_int8_parity(P, name):
    w = workload(name)
    kp, vp, ks, vs = pools(name)
    out, lse, st = run_decode(P, w, kp, vp, ks, vs)
    ref, ref_lse = oracle_decode(w, kp, vp, ks, vs)
    assert st == 0
    mx, _ = attention_errors(out, ref)
    assert mx <= INT8_MAX, mx
    check_lse(lse, ref_lse)


@pytest.mark.parametrize("split", [16, 48, 128, 512, 4096])
def test_decode_split_sizes(P, split):
    w = workload("ragged_g8_bs32")
    kp, vp, _, _ = pools("ragged_g8_bs32")
    out, lse, st = run_decode(P, w, kp, vp, split=split)
    ref, ref_lse = oracle_decode(w, kp, vp)
    assert st == 0
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (split, mx, mean)
    check_lse(lse, ref_lse)


@pytest.mark.parametrize("name", ["llama8b", "int8_small", "ragged_d64"])
def test_decode_identity_vs_permuted_tables_bit_exact(P, name, decode_impl):
    """Results do not depend on which physical pages the table names."""
    w = workload(name)
    kp, vp, ks, vs = pools(name)
    out, lse, _ = run_decode(P, w, kp, vp, ks, vs)
    perm = np.random.default_rng(1).permutation(w.n_blocks)
    move = np.append(perm, w.n_blocks)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[move], vp2[move] = kp, vp
    ks2 = vs2 = None
    if ks is not None:
        ks2, vs2 = np.empty_like(ks), np.empty_like(vs)
        ks2[move], vs2[move] = ks, vs
    t2 = torch.from_numpy(move[w.tables.numpy()]).to(torch.int32)
    out2, lse2, _ = run_decode(P, w, kp2, vp2, ks2, vs2, tables=t2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)


def test_decode_edge_lengths(P, decode_impl):
    w = workload("ragged_d64")
    kp, vp, _, _ = pools("ragged_d64")
    ctx = w.ctx_lens.clone()
    ctx[0] = 0            # empty context: o = 0, lse = -inf
    ctx[1] = 1            # a single token: o = v_0
    ctx[3] = 16           # exactly one block
    out, lse, st = run_decode(P, w, kp, vp, ctx=ctx)
    ref, ref_lse = oracle_decode(w, kp, vp, ctx=ctx)
    assert st == 0
    assert (out[0] == 0).all() and torch.isneginf(lse[0]).all()
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN
    check_lse(lse, ref_lse)


def test_decode_bad_table_and_length_are_flagged(P, decode_impl):
    w = workload("ragged_d64")
    kp, vp, _, _ = pools("ragged_d64")
    tables = w.tables.clone()
    tables[6, 3] = -7
    ctx = w.ctx_lens.clone()
    ctx[2] = w.max_blocks * w.block_size + 1
    out, lse, st = run_decode(P, w, kp, vp, tables=tables, ctx=ctx)
    assert st & P.DEV_BAD_BLOCK_ID and st & P.DEV_BAD_LENGTH
    assert (out[2] == 0).all()
    ref, _ = oracle_decode(w, kp, vp)
    good = [0, 1, 3, 4, 5, 7]
    mx, _ = attention_errors(out[good], ref[good])
    assert mx <= BF16_MAX


def test_decode_workspace_overflow_is_flagged(P):
    w = workload("ragged_d64")
    kp, vp, _, _ = pools("ragged_d64")
    q = w.q.cuda()
    small = P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, 16, 16)
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    st = status_tensor()
    out = P.paged_decode_attention(q, dev(kp), dev(vp), i32(w.tables), i32(w.ctx_lens), w.softmax_scale,
                                   split_tokens=16, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.DEV_WORKSPACE_OVERFLOW
    assert (out == 0).all()


def test_decode_balanced_overflow_is_flagged(P, monkeypatch):
    # automatic splitting with a workspace of exactly n_seqs partial slots (the
    # size pkv_decode_workspace_bytes gives for 16-token splits of no tokens):
    # no room for the balanced items, so the plan flags the overflow, writes no
    # item and leaves o = 0
    monkeypatch.setenv("PKV_DECODE_IMPL", "split")
    w = workload("ragged_d64")
    kp, vp, _, _ = pools("ragged_d64")
    q = w.q.cuda()
    ws = torch.empty(P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, 0, 16), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()
    out = P.paged_decode_attention(q, dev(kp), dev(vp), i32(w.tables), i32(w.ctx_lens), w.softmax_scale,
                                   workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.DEV_WORKSPACE_OVERFLOW
    assert (out == 0).all()


# ---------------------------------------------------------------------------
# the decode step as the benchmark runs it: GPU write, then GPU decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["llama8b", "llama8b_int8"])
def test_step_write_then_decode_full_size(P, name):
    w = workload(name)
    kp, vp, ks, vs = pools(name, after_step=False)
    gk, gv = dev(kp), dev(vp)
    tables, start, ctx = i32(w.tables), i32(w.start_pos), i32(w.ctx_lens)
    st = status_tensor()
    if w.kv_format == "int8":
        gks, gvs = dev(ks), dev(vs)
        P.paged_kv_write_int8(w.k_new.cuda(), w.v_new.cuda(), gk, gv, gks, gvs, tables, start, dev_status=st)
    else:
        gks = gvs = None
        P.paged_kv_write(w.k_new.cuda(), w.v_new.cuda(), gk, gv, tables, start, dev_status=st)
    out = P.paged_decode_attention(w.q.cuda(), gk, gv, tables, ctx, w.softmax_scale, k_scales=gks,
                                   v_scales=gvs, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, rks, rvs = pools(name, after_step=True)
    ref, _ = oracle_decode(w, rk, rv, rks, rvs)
    mx, mean = attention_errors(out, ref)
    if w.kv_format == "int8":
        assert mx <= INT8_MAX, mx
    else:
        assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)


# ---------------------------------------------------------------------------
# chunked prefill
# ---------------------------------------------------------------------------

def run_prefill(P, w, kp, vp, tables=None):
    tables = w.tables if tables is None else tables
    q = w.q.cuda()
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    st = status_tensor()
    out = P.paged_prefill_attention(q, dev(kp), dev(vp), i32(tables), i32(w.stored_lens), w.softmax_scale,
                                    lse_out=lse, dev_status=st)
    torch.cuda.synchronize()
    return out, lse, int(st.item())


@pytest.mark.parametrize("name", ["prefill_small", "prefill_g8", "prefill_g1", "prefill_many", "prefill_ties"])
def test_prefill_parity_all_rows(P, name):
    w = workload(name)
    kp, vp, _, _ = pools(name)
    out, lse, st = run_prefill(P, w, kp, vp)
    code, ref, ref_lse = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens, w.softmax_scale,
                                        n_threads=NTHREADS)
    assert code == 0 and st == 0
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_TOL


def test_prefill_full_size_all_rows(P):
    """The chunked prefill (8 sequences x 512-token chunks, prefixes up to
    5549 tokens) at full size, every row of every sequence and query head
    against the float64 oracle (about a minute of CPU time on 16 cores)."""
    w = workload("chunked_prefill")
    kp, vp, _, _ = pools("chunked_prefill")
    out, lse, st = run_prefill(P, w, kp, vp)
    assert st == 0
    code, ref, ref_lse = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens, w.softmax_scale,
                                        n_threads=NTHREADS)
    assert code == 0
    mx, mean = attention_errors(out, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_TOL
    assert torch.isfinite(out).all()


def test_prefill_identity_vs_permuted_tables_bit_exact(P):
    w = workload("prefill_small")
    kp, vp, _, _ = pools("prefill_small")
    out, lse, _ = run_prefill(P, w, kp, vp)
    perm = np.random.default_rng(2).permutation(w.n_blocks)
    move = np.append(perm, w.n_blocks)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[move], vp2[move] = kp, vp
    t2 = torch.from_numpy(move[w.tables.numpy()]).to(torch.int32)
    out2, lse2, _ = run_prefill(P, w, kp2, vp2, tables=t2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)


def test_write_prefill_gather_back_to_back_on_one_stream(P):
    """Library kernels launched back to back on one stream with no host
    synchronisation, each a programmatic dependent of the one before: the
    chunk write, the prefill that attends the rows just written, a gather of
    the same pages, a second write of the same rows and a second prefill.
    Pools and gather are the oracle's bit for bit, both prefills within the
    parity tolerances (and identical to each other)."""
    w = workload("prefill_small")
    kp, vp, _, _ = empty_pools(w, poison=True)
    write_prefix(w, kp, vp, None, None)
    gk, gv = dev(kp), dev(vp)
    tables, prefix = i32(w.tables), i32(w.stored_lens)
    k_new, v_new, q = w.k_new.cuda(), w.v_new.cuda(), w.q.cuda()
    total = w.stored_lens + w.n_new
    lens = i32(total)
    T = int(total.max())
    st = status_tensor()
    P.paged_kv_write(k_new, v_new, gk, gv, tables, i32(w.start_pos), dev_status=st)
    out1 = P.paged_prefill_attention(q, gk, gv, tables, prefix, w.softmax_scale, dev_status=st)
    ko, vo = P.paged_kv_gather(gk, gv, tables, lens, T, dev_status=st)
    P.paged_kv_write(k_new, v_new, gk, gv, tables, i32(w.start_pos), dev_status=st)
    out2 = P.paged_prefill_attention(q, gk, gv, tables, prefix, w.softmax_scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, _, _ = oracle_pools_after_step(w, poison=True)
    assert np.array_equal(host(gk), rk) and np.array_equal(host(gv), rv)
    code, gk_ref, gv_ref = oracle.gather(rk, rv, dims_of(w), w.tables, total, T)
    assert code == oracle.OK
    assert np.array_equal(host(ko), gk_ref) and np.array_equal(host(vo), gv_ref)
    code, ref, _ = oracle.prefill(w.q, rk, rv, dims_of(w), w.tables, w.stored_lens, w.softmax_scale,
                                  n_threads=NTHREADS)
    assert code == 0
    mx, mean = attention_errors(out1, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


# ---------------------------------------------------------------------------
# the fused decode step: write + decode in one call
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "llama8b", "llama8b_int8", "ragged_d64", "int8_small"])
def test_fused_decode_step(P, name, decode_impl):
    """paged_decode_step = paged_kv_write(_int8) then paged_decode_attention:
    the pool bit-exact with the oracle's write, the output identical bit for
    bit to the two-call path and within tolerance of the oracle."""
    w = workload(name)
    kp, vp, ks, vs = pools(name, after_step=False)
    tables, start, ctx = i32(w.tables), i32(w.start_pos), i32(w.ctx_lens)
    q, kn, vn = w.q.cuda(), w.k_new.cuda(), w.v_new.cuda()
    int8 = w.kv_format == "int8"
    # fused
    gk, gv = dev(kp), dev(vp)
    gks, gvs = (dev(ks), dev(vs)) if int8 else (None, None)
    st = status_tensor()
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    out = P.paged_decode_step(kn, vn, start, q, gk, gv, tables, ctx, w.softmax_scale, k_scales=gks, v_scales=gvs,
                              lse_out=lse, dev_status=st)
    # two calls
    gk2, gv2 = dev(kp), dev(vp)
    if int8:
        gks2, gvs2 = dev(ks), dev(vs)
        P.paged_kv_write_int8(kn, vn, gk2, gv2, gks2, gvs2, tables, start)
    else:
        gks2 = gvs2 = None
        P.paged_kv_write(kn, vn, gk2, gv2, tables, start)
    lse2 = torch.empty_like(lse)
    out2 = P.paged_decode_attention(q, gk2, gv2, tables, ctx, w.softmax_scale, k_scales=gks2, v_scales=gvs2,
                                    lse_out=lse2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, rks, rvs = pools(name, after_step=True)
    assert np.array_equal(host(gk), rk) and np.array_equal(host(gv), rv)
    if int8:
        assert np.array_equal(host(gks).view(np.uint32), rks.view(np.uint32))
        assert np.array_equal(host(gvs).view(np.uint32), rvs.view(np.uint32))
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)
    ref, _ = oracle_decode(w, rk, rv, rks, rvs)
    mx, mean = attention_errors(out, ref)
    if int8:
        assert mx <= INT8_MAX, mx
    else:
        assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)


@pytest.mark.parametrize("name", ["tiny", "int8_small", "ragged_d64"])
def test_decode_plan_matches_calls(P, name, decode_impl):
    """DecodePlan.run (the fixed arguments checked once): the step (write +
    decode) bit for bit the result of paged_decode_step, the decode alone over
    the written pools the same bits again, and both within tolerance of the
    oracle."""
    w = workload(name)
    kp, vp, ks, vs = pools(name, after_step=False)
    tables, start, ctx = i32(w.tables), i32(w.start_pos), i32(w.ctx_lens)
    q, kn, vn = w.q.cuda(), w.k_new.cuda(), w.v_new.cuda()
    int8 = w.kv_format == "int8"
    gk, gv = dev(kp), dev(vp)
    gks, gvs = (dev(ks), dev(vs)) if int8 else (None, None)
    st = status_tensor()
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    plan = P.DecodePlan(gk, gv, tables, ctx, w.softmax_scale, q.shape[1], k_scales=gks, v_scales=gvs, lse_out=lse,
                        dev_status=st)
    out_step = plan.run(q, kn, vn, start).clone()
    lse_step = lse.clone()
    out_decode = plan.run(q).clone()
    gk2, gv2 = dev(kp), dev(vp)
    gks2, gvs2 = (dev(ks), dev(vs)) if int8 else (None, None)
    lse2 = torch.empty_like(lse)
    out2 = P.paged_decode_step(kn, vn, start, q, gk2, gv2, tables, ctx, w.softmax_scale, k_scales=gks2,
                               v_scales=gvs2, lse_out=lse2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, rks, rvs = pools(name, after_step=True)
    assert np.array_equal(host(gk), rk) and np.array_equal(host(gv), rv)
    assert torch.equal(out_step.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse_step, lse2)
    assert torch.equal(out_decode.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)
    ref, _ = oracle_decode(w, rk, rv, rks, rvs)
    mx, mean = attention_errors(out_step, ref)
    if int8:
        assert mx <= INT8_MAX, mx
    else:
        assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)


def test_calls_run_on_the_current_stream(P):
    """Without an explicit stream the calls enqueue on the caller's current
    stream: under torch.cuda.stream(side), a decode step whose inputs are
    produced on that stream gives the default-stream result, and the default
    stream sees it only after waiting for the side stream."""
    w = workload("tiny")
    kp, vp, _, _ = pools("tiny", after_step=False)
    tables, start, ctx = i32(w.tables), i32(w.start_pos), i32(w.ctx_lens)
    gk, gv = dev(kp), dev(vp)
    ref = P.paged_decode_step(w.k_new.cuda(), w.v_new.cuda(), start, w.q.cuda(), gk, gv, tables, ctx,
                              w.softmax_scale)
    torch.cuda.synchronize()
    gk2, gv2 = dev(kp), dev(vp)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(2_000_000)                        # the side stream is busy for a while
        q = w.q.cuda()                                      # produced on the side stream
        plan = P.DecodePlan(gk2, gv2, tables, ctx, w.softmax_scale, q.shape[1])
        out = plan.run(q, w.k_new.cuda(), w.v_new.cuda(), start)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_decode_plan_refuses_mismatched_calls(P):
    w = workload("tiny")
    kp, vp, _, _ = pools("tiny", after_step=False)
    tables, ctx = i32(w.tables), i32(w.ctx_lens)
    plan = P.DecodePlan(dev(kp), dev(vp), tables, ctx, w.softmax_scale, w.q.shape[1])
    q = w.q.cuda()
    with pytest.raises(ValueError):
        plan.run(q[:-1].contiguous())                       # fewer sequences than planned
    with pytest.raises(ValueError):
        plan.run(q, v_new=w.v_new.cuda())                   # v_new without k_new
    with pytest.raises(ValueError):
        plan.run(q, w.k_new.cuda()[:, :, :1].contiguous(), w.v_new.cuda(), i32(w.start_pos))   # wrong kv heads
    with pytest.raises(ValueError):
        plan.run(q.float())                                 # wrong dtype


def test_decode_refuses_an_unaligned_workspace(P):
    """A workspace that does not start on a 256-byte boundary is refused on the
    host (PKV_ERR_WORKSPACE, nothing enqueued); the same bytes one slice
    later, aligned, give the workspace-allocating call's result."""
    w = workload("int8_small")
    kp, vp, ks, vs = pools("int8_small")
    args = (w.q.cuda(), dev(kp), dev(vp), i32(w.tables), i32(w.ctx_lens), w.softmax_scale)
    kw = dict(k_scales=dev(ks), v_scales=dev(vs), split_tokens=64)
    need = P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, int(w.ctx_lens.sum()), 64)
    buf = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    assert buf.data_ptr() % 256 == 0
    with pytest.raises(P.PagedKVError) as e:
        P.paged_decode_attention(*args, workspace=buf[16:16 + need], **kw)
    assert e.value.status == 4
    got = P.paged_decode_attention(*args, workspace=buf[256:256 + need], **kw)
    ref = P.paged_decode_attention(*args, **kw)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def test_int8_write_near_ties_bit_exact(P):
    """Rows whose codes sit at or next to a half-integer quotient -- where a
    reciprocal multiply and the IEEE division by the stored scale can round
    differently -- are quantised exactly as the oracle's division says."""
    u = np.arange(0x3e00, 0x4100, dtype=np.uint32)
    vals = (u << 16).view(np.float32)
    rows = []
    for amax in vals:
        scale = np.float32(amax) / np.float32(127)
        rcp = np.float32(1) / scale
        xs = vals[vals <= amax]
        q = xs * rcp
        near = np.abs(q - np.floor(q) - np.float32(0.5)) <= np.float32(1e-4)
        picked = xs[near][:63]
        if len(picked):
            row = np.zeros(128, np.float32)
            row[0] = amax
            row[1:1 + len(picked)] = picked
            row[64:64 + len(picked)] = -picked
            rows.append(row)
    assert len(rows) >= 64
    Hkv, D, bs = 4, 128, 16
    n_tok = -(-len(rows) // Hkv)
    data = np.zeros((n_tok * Hkv, D), np.float32)
    data[:len(rows)] = np.stack(rows)
    new = torch.from_numpy(data.reshape(1, n_tok, Hkv, D)).to(torch.bfloat16)
    kn = new.view(torch.int16).numpy().view(np.uint16)
    vn = (-new).view(torch.int16).numpy().view(np.uint16)
    nb = -(-n_tok // bs)
    d = oracle.Dims(nb, bs, Hkv, D)
    tables = np.arange(nb, dtype=np.int32)[None]
    start = np.zeros(1, np.int32)
    okp, ovp = np.zeros(d.pool_shape, np.int8), np.zeros(d.pool_shape, np.int8)
    oks, ovs = np.zeros(d.scale_shape, np.float32), np.zeros(d.scale_shape, np.float32)
    assert oracle.write_int8(kn, vn, okp, ovp, oks, ovs, d, tables, start) == oracle.OK
    gk, gv = dev(okp * 0), dev(ovp * 0)
    gks, gvs = dev(oks * 0), dev(ovs * 0)
    st = status_tensor()
    P.paged_kv_write_int8(dev(kn), dev(vn), gk, gv, gks, gvs, i32(tables), i32(start), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(host(gk), okp) and np.array_equal(host(gv), ovp)
    assert np.array_equal(host(gks).view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(host(gvs).view(np.uint32), ovs.view(np.uint32))
