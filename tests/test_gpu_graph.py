"""GPU test of a multi-layer decode step captured as one CUDA graph: every
layer's write + decode (paged_decode_step, or DecodePlan.run with one plan per
layer; three launches chained by programmatic dependent launch) replays from
the graph with the same bits as the eager calls, and layer outputs match the
oracle's write + decode."""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import attention_errors, host

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, INT8_MAX = 1e-2, 1e-3, 2e-2


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_212_gb300 import build as B
    B.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()
    return P


@pytest.mark.parametrize("use_plan", [False, True])
@pytest.mark.parametrize("int8", [False, True])
def test_layer_step_graph_replays_the_eager_bits(P, int8, use_plan, decode_impl):
    n_layers, n, Hkv, G, D, bs, n_blocks, max_blocks = 4, 5, 4, 4, 128, 16, 60, 10   # int8 decode: Hkv % 4 == 0
    Hq = Hkv * G
    gen = torch.Generator().manual_seed(303 + int8)
    lens = [17, 100, 0, 130, 64]                                  # stored tokens; the step writes one more
    perm = torch.randperm(n_blocks, generator=gen).tolist()
    tables = np.full((n, max_blocks), n_blocks, np.int32)
    k = 0
    for s, L in enumerate(lens):
        nb = -(-(L + 1) // bs)
        tables[s, :nb] = perm[k:k + nb]
        k += nb
    start = np.array(lens, np.int32)
    ctx = start + 1
    d = oracle.Dims(n_blocks, bs, Hkv, D)
    dev = "cuda"
    t_tab, t_start, t_ctx = (torch.from_numpy(x).to(dev) for x in (tables, start, ctx))
    layers = []
    for _ in range(n_layers):
        x = {"q": torch.randn((n, Hq, D), generator=gen).to(torch.bfloat16),
             "k_new": torch.randn((n, 1, Hkv, D), generator=gen).to(torch.bfloat16),
             "v_new": torch.randn((n, 1, Hkv, D), generator=gen).to(torch.bfloat16)}
        if int8:
            x["kp"] = torch.randint(-127, 128, d.pool_shape, generator=gen, dtype=torch.int8)
            x["vp"] = torch.randint(-127, 128, d.pool_shape, generator=gen, dtype=torch.int8)
            x["ks"] = torch.rand(d.scale_shape, generator=gen) * 0.02
            x["vs"] = torch.rand(d.scale_shape, generator=gen) * 0.02
        else:
            x["kp"] = torch.randn(d.pool_shape, generator=gen).to(torch.bfloat16)
            x["vp"] = torch.randn(d.pool_shape, generator=gen).to(torch.bfloat16)
            x["ks"] = x["vs"] = None
        x["cpu"] = {key: (None if v is None else v.clone()) for key, v in x.items()}
        for key in ("q", "k_new", "v_new", "kp", "vp", "ks", "vs"):
            if x[key] is not None:
                x[key] = x[key].to(dev)
        x["out"] = torch.empty((n, Hq, D), dtype=torch.bfloat16, device=dev)
        layers.append(x)
    ws = torch.empty(P.decode_workspace_bytes(n, Hq, D, int(ctx.sum())), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / D ** 0.5

    plans = [P.DecodePlan(x["kp"], x["vp"], t_tab, t_ctx, scale, Hq, k_scales=x["ks"], v_scales=x["vs"],
                          out=x["out"], workspace=ws, dev_status=st) for x in layers] if use_plan else None

    def step():
        if use_plan:
            for x, plan in zip(layers, plans):
                plan.run(x["q"], x["k_new"], x["v_new"], t_start)
            return
        for x in layers:
            P.paged_decode_step(x["k_new"], x["v_new"], t_start, x["q"], x["kp"], x["vp"], t_tab, t_ctx, scale,
                                k_scales=x["ks"], v_scales=x["vs"], out=x["out"], workspace=ws, dev_status=st)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                            # eager (the write is idempotent: same rows, same places)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [x["out"].clone() for x in layers]
    pools = [(x["kp"].clone(), x["vp"].clone()) for x in layers]
    for x in layers:
        x["out"].zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, e, (kp, vp) in zip(layers, eager, pools):
        assert torch.equal(x["out"], e)
        assert torch.equal(x["kp"], kp) and torch.equal(x["vp"], vp)
    # the step each layer computed is the oracle's write + decode on that layer's pools
    for x in layers:
        c = x["cpu"]
        kn, vn = host(c["k_new"]), host(c["v_new"])
        if int8:
            kp, vp, ks, vs = c["kp"].numpy().copy(), c["vp"].numpy().copy(), c["ks"].numpy().copy(), \
                c["vs"].numpy().copy()
            oracle.write_int8(kn, vn, kp, vp, ks, vs, d, tables, start)
        else:
            kp, vp, ks, vs = host(c["kp"]).copy(), host(c["vp"]).copy(), None, None
            oracle.write_bf16(kn, vn, kp, vp, d, tables, start)
        code, ref, _ = oracle.decode(host(c["q"]), kp, vp, d, tables, ctx, scale, k_scales=ks, v_scales=vs)
        assert code == 0
        live = ctx > 0
        mx, mean = attention_errors(x["out"][torch.from_numpy(live)], ref[live])
        assert mx <= (INT8_MAX if int8 else BF16_MAX), mx
        if not int8:
            assert mean <= BF16_MEAN, mean
