"""GPU tests of copy-on-write and of the block manager driving the kernels:
paged_kv_copy_blocks is bit-exact with the oracle's block copy, and a serving
loop whose tables, copy-on-write pairs and lengths come from the library's
block manager (admissions, forks, preemption) gives the oracle's decode output
at every step, with the oracle running the same loop on its own pools."""
import numpy as np
import pytest
import torch

import oracle
from gpu_support import attention_errors, dev, host, i32
from oracle.block_manager import copy_blocks

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


def _bf16_bits(gen, shape):
    x = torch.randn(shape, generator=gen).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("head_dim,int8", [(128, False), (64, False), (128, True)])
def test_copy_blocks_bit_exact(P, head_dim, int8):
    gen = torch.Generator().manual_seed(31 + head_dim + int8)
    d = oracle.Dims(40, 16, 4, head_dim)
    if int8:
        kp = torch.randint(-127, 128, d.pool_shape, generator=gen, dtype=torch.int8).numpy()
        vp = torch.randint(-127, 128, d.pool_shape, generator=gen, dtype=torch.int8).numpy()
        ks = torch.rand(d.scale_shape, generator=gen).numpy()
        vs = torch.rand(d.scale_shape, generator=gen).numpy()
    else:
        kp, vp = _bf16_bits(gen, d.pool_shape), _bf16_bits(gen, d.pool_shape)
        ks = vs = None
    # distinct destinations, none of them a source; the scratch block may be copied from
    pairs = [(0, 30), (5, 31), (40, 32), (7, 33), (5, 34), (12, 35), (39, 36)]
    gk, gv = dev(kp), dev(vp)
    gks, gvs = (dev(ks), dev(vs)) if int8 else (None, None)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.paged_kv_copy_blocks(i32(pairs), gk, gv, gks, gvs, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for pool, g in ((kp, gk), (vp, gv)) + (((ks, gks), (vs, gvs)) if int8 else ()):
        ref = copy_blocks(pool.copy(), pairs)
        assert np.array_equal(host(g), ref)


def test_copy_blocks_bad_ids_are_flagged_and_skipped(P):
    gen = torch.Generator().manual_seed(5)
    d = oracle.Dims(8, 16, 2, 64)
    kp, vp = _bf16_bits(gen, d.pool_shape), _bf16_bits(gen, d.pool_shape)
    gk, gv = dev(kp), dev(vp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.paged_kv_copy_blocks(i32([(1, 2), (3, 9), (-1, 4)]), gk, gv, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.DEV_BAD_BLOCK_ID
    ref = copy_blocks(kp.copy(), [(1, 2)])
    assert np.array_equal(host(gk), ref)


@pytest.mark.parametrize("int8", [False, True])
def test_serving_loop_driven_by_the_block_manager(P, int8, decode_impl):
    gen = torch.Generator().manual_seed(77 + int8)
    n_blocks, bs, n_slots, max_blocks = 22, 16, 8, 8
    Hkv, G, D = 4, 4, 128
    Hq = Hkv * G
    d = oracle.Dims(n_blocks, bs, Hkv, D)
    bm = P.BlockManager(n_blocks, bs, n_slots, max_blocks)
    # both sides start from the same (zero) pools
    if int8:
        okp, ovp = np.zeros(d.pool_shape, np.int8), np.zeros(d.pool_shape, np.int8)
        oks, ovs = np.zeros(d.scale_shape, np.float32), np.zeros(d.scale_shape, np.float32)
    else:
        okp, ovp = np.zeros(d.pool_shape, np.uint16), np.zeros(d.pool_shape, np.uint16)
        oks = ovs = None
    gk, gv = dev(okp), dev(ovp)
    gks, gvs = (dev(oks), dev(ovs)) if int8 else (None, None)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / D ** 0.5

    def write_both(k, v, tables, start):
        """k, v: uint16 bf16 bits [n, n_new, Hkv, D]; the same rows to both sides."""
        if int8:
            oracle.write_int8(k, v, okp, ovp, oks, ovs, d, tables, start)
            P.paged_kv_write_int8(dev(k), dev(v), gk, gv, gks, gvs, i32(tables), i32(start), dev_status=st)
        else:
            oracle.write_bf16(k, v, okp, ovp, d, tables, start)
            P.paged_kv_write(dev(k), dev(v), gk, gv, i32(tables), i32(start), dev_status=st)

    def admit(slot, n):
        bm.admit(slot, n)
        tables, _, _ = bm.export()
        t = tables[slot:slot + 1].numpy()
        write_both(_bf16_bits(gen, (1, n, Hkv, D)), _bf16_bits(gen, (1, n, Hkv, D)), t, np.array([0], np.int32))

    for slot, n in ((0, 20), (1, 33), (2, 16), (3, 5)):
        admit(slot, n)
    bm.fork(0, 4)
    bm.fork(1, 5)
    n_copies = n_victims = 0
    ws = torch.empty(P.decode_workspace_bytes(n_slots, Hq, D, n_slots * max_blocks * bs), dtype=torch.uint8,
                     device="cuda")
    for step in range(36):
        victims = bm.reserve_step()
        n_victims += len(victims)
        copies = bm.begin_step()
        if copies:
            n_copies += len(copies)
            for pool in (okp, ovp) + ((oks, ovs) if int8 else ()):
                copy_blocks(pool, copies)
            P.paged_kv_copy_blocks(i32(copies), gk, gv, gks, gvs, dev_status=st)
        tables, lens, active = bm.export()
        act = active.numpy().astype(bool)
        start = lens.numpy().astype(np.int32)                 # this step's token position
        ctx = np.where(act, start + 1, 0).astype(np.int32)
        k_new, v_new = _bf16_bits(gen, (n_slots, 1, Hkv, D)), _bf16_bits(gen, (n_slots, 1, Hkv, D))
        q = _bf16_bits(gen, (n_slots, Hq, D))
        out = torch.empty((n_slots, Hq, D), dtype=torch.bfloat16, device="cuda")
        P.paged_decode_step(dev(k_new), dev(v_new), i32(start), dev(q), gk, gv, i32(tables), i32(ctx), scale,
                            k_scales=gks, v_scales=gvs, out=out, workspace=ws, dev_status=st)
        # oracle: the same write, then the decode
        if int8:
            oracle.write_int8(k_new, v_new, okp, ovp, oks, ovs, d, tables.numpy(), start)
        else:
            oracle.write_bf16(k_new, v_new, okp, ovp, d, tables.numpy(), start)
        code, ref, _ = oracle.decode(q, okp, ovp, d, tables.numpy(), ctx, scale, k_scales=oks, v_scales=ovs)
        torch.cuda.synchronize()
        assert code == 0 and int(st.item()) == 0
        mx, mean = attention_errors(out[torch.from_numpy(act)], ref[act])
        assert mx <= (INT8_MAX if int8 else BF16_MAX), (step, mx)
        if not int8:
            assert mean <= BF16_MEAN, (step, mean)
        bm.end_step()
        if step == 12:
            bm.release(2)
            if bm.can_admit([40]):
                admit(2, 40)
        if step == 20:
            _, _, active = bm.export()
            live = [s for s in range(n_slots) if active[s]]
            idle = [s for s in range(n_slots) if not active[s]]
            if live and idle:
                bm.fork(live[0], idle[0])
    # the loop exercised copy-on-write and preemption
    assert n_copies >= 2 and n_victims >= 1, (n_copies, n_victims)
