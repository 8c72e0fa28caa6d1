"""paged_decode_attention_noalloc: the decode entry point for callers that may
not allocate device memory (a plugin whose host owns all device memory, a
runtime with a fixed memory budget).  Its split-KV scratch is the library's
static device array instead of a caller workspace.

Checked against the float64 CPU oracle and against paged_decode_attention
(caller workspace) on the GPU, on two calls in a row -- the second call finds
the first call's leftovers in the shared array -- within the parity tolerances
of the other decode tests.  This file is collected last so that a run stopping
at the first failure has already run every other test; it also passes alone in
a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import NTHREADS, attention_errors
from oracle_pools import dims_of, oracle_pools_after_step
from paged_kv_cache_212_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, INT8_MAX = 1e-2, 1e-3, 2e-2


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_212_gb300 import build
    build.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


def _dev(a):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    return t.cuda()


def _errors(a, b):
    d = (a.double() - b.double()).abs()
    return float(d.max()), float(d.mean())


def _ragged():
    return W.decode_workload("ragged", 31, [1, 15, 16, 17, 300, 777, 2000], 32, 8, 128, 16)


def _int8():
    return W.decode_workload("int8", 32, [5, 90, 1200], 16, 4, 128, 32, n_new=2, kv_format="int8")


def _tiny():
    # one wave of (sequence, kv head) units with contexts of at most 256 tokens:
    # automatic splitting takes the one-launch path, which uses no scratch
    return W.decode_workload("tiny", 34, [10, 100, 255], 16, 4, 128, 16)


# split 64: several fixed splits per sequence, so the shared scratch carries
# partials; split 0: the automatic balanced split over the whole array
@pytest.mark.parametrize("make,split,tol_max,tol_mean", [
    (_ragged, 64, BF16_MAX, BF16_MEAN),
    (_int8, 64, INT8_MAX, None),
    (_ragged, 0, BF16_MAX, BF16_MEAN),
    (_int8, 0, INT8_MAX, None),
    (_tiny, 0, BF16_MAX, BF16_MEAN),
])
def test_noalloc_matches_workspace_entry_point_on_two_calls(P, make, split, tol_max, tol_mean):
    w = make()
    kp, vp, ks, vs = oracle_pools_after_step(w)
    gk, gv = _dev(kp), _dev(vp)
    gks = gvs = None
    if ks is not None:
        gks, gvs = _dev(ks), _dev(vs)
    q = w.q.cuda()
    tables, ctx = w.tables.cuda(), w.ctx_lens.cuda()
    total = int(w.ctx_lens.sum())
    ref_lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ref = P.paged_decode_attention(q, gk, gv, tables, ctx, w.softmax_scale, k_scales=gks, v_scales=gvs,
                                   split_tokens=split, lse_out=ref_lse)
    code, oref, olse = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale, ks, vs,
                                     n_threads=NTHREADS)
    assert code == oracle.OK
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        P.paged_decode_attention_noalloc(q, gk, gv, tables, ctx, w.softmax_scale, total, out, k_scales=gks,
                                         v_scales=gvs, split_tokens=split, lse_out=lse, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        for against in (ref, oref):
            mx, mean = _errors(out, against) if isinstance(against, torch.Tensor) else attention_errors(out, against)
            assert mx <= tol_max, (call, mx)
            if tol_mean is not None:
                assert mean <= tol_mean, (call, mean)
        assert float((lse - ref_lse).abs().max()) <= 2e-3, call
        g = lse.cpu().numpy().astype(np.float64)
        fin = np.isfinite(olse)
        assert np.array_equal(np.isneginf(g), np.isneginf(olse)), call
        assert not fin.any() or np.abs(g[fin] - olse[fin]).max() <= 2e-3, call


def test_noalloc_rejects_requests_larger_than_its_scratch(P):
    w = W.decode_workload("small", 33, [10, 20], 8, 2, 64, 16)
    q = w.q.cuda()
    gk = torch.zeros(w.pool_shape, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    huge = P.NOALLOC_DECODE_SCRATCH_BYTES  # tokens: far more splits than 16 MiB of partials can hold
    with pytest.raises(P.PagedKVError) as e:
        P.paged_decode_attention_noalloc(q, gk, gk, w.tables.cuda(), w.ctx_lens.cuda(), w.softmax_scale, huge,
                                         out, split_tokens=16)
    assert e.value.status == 4  # PKV_ERR_WORKSPACE, nothing enqueued
