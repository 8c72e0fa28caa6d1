"""The Python binding refuses tensors whose shapes disagree (host side, no GPU):
a smaller out, lse_out, ctx_lens or scale tensor would otherwise become an
out-of-bounds device access."""
import pytest
import torch

import paged_kv_cache_212_gb300 as P


def _decode_tensors(n_seqs=3, hq=8, hkv=2, d=64, nb=10, bs=16, max_blocks=4, int8=False):
    dt = torch.int8 if int8 else torch.bfloat16
    q = torch.zeros((n_seqs, hq, d), dtype=torch.bfloat16)
    kp = torch.zeros((nb + 1, bs, hkv, d), dtype=dt)
    vp = torch.zeros_like(kp)
    ks = torch.zeros((nb + 1, bs, hkv), dtype=torch.float32) if int8 else None
    vs = torch.zeros_like(ks) if int8 else None
    tables = torch.zeros((n_seqs, max_blocks), dtype=torch.int32)
    ctx = torch.zeros(n_seqs, dtype=torch.int32)
    out = torch.zeros_like(q)
    lse = torch.zeros((n_seqs, hq), dtype=torch.float32)
    return dict(q=q, k_pool=kp, v_pool=vp, k_scales=ks, v_scales=vs, block_tables=tables, ctx_lens=ctx, out=out,
                lse_out=lse, dev_status=None)


def test_matching_decode_shapes_pass():
    P._check_decode(**_decode_tensors())
    P._check_decode(**_decode_tensors(int8=True))


@pytest.mark.parametrize("name,bad", [
    ("out", lambda t: t["out"][:-1]),
    ("lse_out", lambda t: t["lse_out"][:, :-1]),
    ("ctx_lens", lambda t: t["ctx_lens"][:-1]),
    ("block_tables", lambda t: t["block_tables"][:-1]),
    ("v_pool", lambda t: t["v_pool"][:-1]),
])
def test_decode_shape_mismatch_raises(name, bad):
    t = _decode_tensors()
    t[name] = bad(t)
    with pytest.raises(ValueError):
        P._check_decode(**t)


@pytest.mark.parametrize("name", ["k_scales", "v_scales"])
def test_int8_scale_shape_mismatch_raises(name):
    t = _decode_tensors(int8=True)
    t[name] = t[name][:, :-1]
    with pytest.raises(ValueError):
        P._check_decode(**t)


def test_decode_plan_refuses_host_tensors():
    t = _decode_tensors()
    with pytest.raises(ValueError):
        P.DecodePlan(t["k_pool"], t["v_pool"], t["block_tables"], t["ctx_lens"], 0.125, 8)


def test_head_dim_mismatch_raises():
    t = _decode_tensors()
    t["q"] = torch.zeros((3, 8, 128), dtype=torch.bfloat16)
    t["out"] = torch.zeros_like(t["q"])
    with pytest.raises(ValueError):
        P._check_decode(**t)


@pytest.mark.gpu
def test_wrappers_refuse_mismatched_cuda_tensors():
    """The same checks in the calls themselves, before anything is enqueued."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_212_gb300 import build
    build.build()
    P.load_library()
    t = {k: (v.cuda() if v is not None else None) for k, v in _decode_tensors().items()}
    short_out = t["out"][:-1].contiguous()
    with pytest.raises(ValueError):
        P.paged_decode_attention_noalloc(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["ctx_lens"], 0.125,
                                         64, short_out)
    with pytest.raises(ValueError):
        P.paged_decode_attention(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["ctx_lens"][:-1].contiguous(),
                                 0.125)
    with pytest.raises(ValueError):
        P.paged_decode_attention(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["ctx_lens"], 0.125,
                                 lse_out=t["lse_out"][:, :-1].contiguous())
    q4 = torch.zeros((3, 8, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        P.paged_prefill_attention(q4, t["k_pool"], t["v_pool"], t["block_tables"], t["ctx_lens"], 0.125,
                                  out=q4[:, :-1].contiguous())
