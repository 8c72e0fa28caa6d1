"""Failure detection without a GPU fault: a bounded pipeline wait that runs out.

Every pipeline wait of the split-KV decode (mma.sync and tensor-core kernels)
and of the tcgen05 prefill gives up after a limit the host sets
(pkv_set_pipeline_wait_ns, 4 s by default).  With a 1 ns limit the waits that
are not already satisfied run out at once: the kernel reports PKV_DEV_TIMEOUT
in dev_status, its CTAs wind down (the copies and tensor-core operations
already issued finish before shared memory or TMEM is released) and the call
returns.  The next call on the same stream, with the default limit back,
matches the float64 oracle.  (libmir-metal paged/mod.rs: the store's calls
return errors instead of aborting.)
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import NTHREADS, attention_errors, dev, i32
from oracle_pools import dims_of, oracle_pools_after_step
from paged_kv_cache_212_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PKV_DEV_TIMEOUT = 16
TRIES = 5          # calls with the short limit; at least one of them must run out


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_212_gb300 import build
    build.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


class short_waits:
    """Pipeline waits limited to `ns` inside the block; the default after."""

    def __init__(self, P, ns):
        self.lib, self.ns = P.load_library(), ns

    def __enter__(self):
        self.lib.pkv_set_pipeline_wait_ns(self.ns)

    def __exit__(self, *exc):
        self.lib.pkv_set_pipeline_wait_ns(0)


# split: the mma.sync split-KV kernels; tc: the tensor-core kernel (int8 pages),
# whose warpgroups leave their loop as one after any wait that gives up
@pytest.mark.parametrize("kv_format,impl", [("bf16", "split"), ("int8", "split"), ("int8", "tc")])
def test_decode_wait_runs_out_then_recovers(P, kv_format, impl, monkeypatch):
    monkeypatch.setenv("PKV_DECODE_IMPL", impl)             # the pipelined kernels
    w = W.decode_workload("timeout", 31, [300, 700, 1500, 64, 2000, 5], 32, 8, 128, 16, n_new=1,
                          kv_format=kv_format)
    kp, vp, ks, vs = oracle_pools_after_step(w, poison=True)
    gk, gv = dev(kp), dev(vp)
    gks, gvs = (dev(ks), dev(vs)) if kv_format == "int8" else (None, None)
    q, tables, ctx = w.q.cuda(), i32(w.tables), i32(w.ctx_lens)
    ws = torch.empty(P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, int(w.ctx_lens.sum())),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)

    def call(st):
        P.paged_decode_attention(q, gk, gv, tables, ctx, w.softmax_scale, k_scales=gks, v_scales=gvs, out=out,
                                 workspace=ws, dev_status=st)

    seen = 0
    with short_waits(P, 1):
        for _ in range(TRIES):
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            call(st)                                # the call itself returns PKV_OK
            torch.cuda.synchronize()                # and the kernels end
            seen |= int(st.item())
    assert seen & PKV_DEV_TIMEOUT, f"no wait ran out in {TRIES} calls (status {seen})"
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    call(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    code, ref, _ = oracle.decode(w.q, kp, vp, dims_of(w), w.tables, w.ctx_lens, w.softmax_scale,
                                 k_scales=ks, v_scales=vs, n_threads=NTHREADS)
    assert code == 0
    mx, mean = attention_errors(out, ref)
    if kv_format == "int8":
        assert mx <= 2e-2, mx
    else:
        assert mx <= 1e-2 and mean <= 1e-3, (mx, mean)


def test_prefill_wait_runs_out_then_recovers(P):
    # at most two 128-key tiles per CTA: every K and V copy fits the rings, so
    # both K producers issue every tile and their wind-down waits complete
    w = W.prefill_workload("timeout prefill", 32, [0, 100, 37], 64, 16, 4, 128, 16)
    kp, vp, _, _ = oracle_pools_after_step(w, poison=True)
    gk, gv = dev(kp), dev(vp)
    q, tables, prefix = w.q.cuda(), i32(w.tables), i32(w.stored_lens)
    out = torch.empty_like(q)

    def call(st):
        P.paged_prefill_attention(q, gk, gv, tables, prefix, w.softmax_scale, out=out, dev_status=st)

    seen = 0
    with short_waits(P, 1):
        for _ in range(TRIES):
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            call(st)
            torch.cuda.synchronize()
            seen |= int(st.item())
    assert seen & PKV_DEV_TIMEOUT, f"no wait ran out in {TRIES} calls (status {seen})"
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    call(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    code, ref, _ = oracle.prefill(w.q, kp, vp, dims_of(w), w.tables, w.stored_lens, w.softmax_scale,
                                  n_threads=NTHREADS)
    assert code == 0
    mx, mean = attention_errors(out, ref)
    assert mx <= 1e-2 and mean <= 1e-3, (mx, mean)
