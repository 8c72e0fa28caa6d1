"""Test-side helpers: materialise a workload's resident prefix in oracle pools
(numpy arrays) with the oracle's own write, and small bf16 conversions.

Unused pool memory is poisoned: bf16 pools with the NaN pattern 0x7FC0, int8
pools with code 127 and NaN scales, so that any read of a slot outside a
sequence's context shows up as a NaN in the result.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_NAN = 0x7FC0


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def f64(a) -> np.ndarray:
    """bf16 bit patterns (numpy uint16) or a bf16 tensor, widened exactly to float64."""
    if isinstance(a, torch.Tensor):
        return a.detach().cpu().to(torch.float64).numpy()
    u = np.asarray(a, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def dims_of(w) -> oracle.Dims:
    return oracle.Dims(w.n_blocks, w.block_size, w.n_kv_heads, w.head_dim)


def empty_pools(w, poison=True):
    if w.kv_format == "int8":
        kp = np.full(w.pool_shape, 127 if poison else 0, np.int8)
        vp = np.full(w.pool_shape, 127 if poison else 0, np.int8)
        ks = np.full(w.scale_shape, np.nan if poison else 0, np.float32)
        vs = np.full(w.scale_shape, np.nan if poison else 0, np.float32)
        return kp, vp, ks, vs
    kp = np.full(w.pool_shape, BF16_NAN if poison else 0, np.uint16)
    vp = np.full(w.pool_shape, BF16_NAN if poison else 0, np.uint16)
    return kp, vp, None, None


def write_prefix(w, kp, vp, ks=None, vs=None):
    """Place every prefix segment with the oracle's write (bf16 or int8)."""
    d = dims_of(w)
    for seg in w.prefix:
        tb = w.tables[seg.seq:seg.seq + 1]
        sp = np.array([seg.start], np.int32)
        if w.kv_format == "int8":
            st = oracle.write_int8(seg.k[None], seg.v[None], kp, vp, ks, vs, d, tb, sp)
        else:
            st = oracle.write_bf16(seg.k[None], seg.v[None], kp, vp, d, tb, sp)
        assert st == oracle.OK


def oracle_pools_after_step(w, poison=True):
    """Pools holding the prefix and this step's new rows (written by the oracle)."""
    kp, vp, ks, vs = empty_pools(w, poison)
    write_prefix(w, kp, vp, ks, vs)
    d = dims_of(w)
    if w.n_new:
        if w.kv_format == "int8":
            st = oracle.write_int8(w.k_new, w.v_new, kp, vp, ks, vs, d, w.tables, w.start_pos)
        else:
            st = oracle.write_bf16(w.k_new, w.v_new, kp, vp, d, w.tables, w.start_pos)
        assert st == oracle.OK
    return kp, vp, ks, vs


def logical_rows(w, s):
    """The logical K/V rows [ctx, Hkv, D] of sequence s after the step (prefix
    segments then the new rows), assembled from the workload's draws."""
    L = int(w.stored_lens[s])
    k = torch.empty((L + w.n_new, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16)
    v = torch.empty_like(k)
    # shared segments are written through the group leader's row
    g0 = (s // w.group_size) * w.group_size if w.group_size > 1 else s
    for seg in w.prefix:
        if seg.seq == s or (w.group_size > 1 and seg.seq == g0 and seg.start == 0):
            n = seg.k.shape[0]
            k[seg.start:seg.start + n] = seg.k.cpu()
            v[seg.start:seg.start + n] = seg.v.cpu()
    if w.n_new:
        k[L:] = w.k_new[s].cpu()
        v[L:] = w.v_new[s].cpu()
    return k, v
