"""Plain CPU oracle for the paged KV-cache hot path (binary64 attention, bit-exact
write / gather / int8 quantisation).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the CPU-baseline
leg of the benchmark are the only callers.  The product package never imports
this module, and this module imports nothing from the product package; the two
share only the seeded input generators' outputs (plain arrays).

The arithmetic lives in ``pkv_oracle.c`` (built here with gcc on first use, or
by ``build()``); this file only marshals numpy arrays to it.  bf16 tensors are
passed as their raw 16-bit patterns (numpy ``uint16``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lib = None

OK, BAD_ARG, BAD_INDEX = 0, -1, -2


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into libpkv_oracle.so (IEEE semantics, no FMA
    contraction) and return the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
             "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        _lib.pkvo_write_bf16.argtypes = [P, P, P, P, i32, i32, i32, i32, P, i32, P, i32, i32]
        _lib.pkvo_write_int8.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P, i32, P, i32, i32]
        _lib.pkvo_gather.argtypes = [P, P, i32, i32, i32, i32, P, i32, P, i32, i32, P, P]
        _lib.pkvo_decode.argtypes = [P, i32, P, P, P, P, i32, i32, i32, i32, i32, P, i32, P, i32,
                                     ctypes.c_float, i32, P, P, i32]
        _lib.pkvo_prefill.argtypes = [P, i32, P, P, i32, i32, i32, i32, P, i32, P, i32, i32,
                                      ctypes.c_float, P, P, P, i32]
        for fn in ("pkvo_write_bf16", "pkvo_write_int8", "pkvo_gather", "pkvo_decode",
                   "pkvo_prefill"):
            getattr(_lib, fn).restype = ctypes.c_int
    return _lib


def _arr(x, dtype):
    """Contiguous numpy array of the given dtype; torch bf16 tensors become their
    uint16 bit patterns."""
    if hasattr(x, "detach"):  # a torch tensor
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != np.dtype(dtype):
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and \
                np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class Dims:
    """Pool geometry: n_blocks physical blocks (the pool has n_blocks + 1 rows,
    the last being the scratch block), block_size, n_kv_heads, head_dim."""

    def __init__(self, n_blocks, block_size, n_kv_heads, head_dim):
        self.n_blocks, self.block_size = int(n_blocks), int(block_size)
        self.n_kv_heads, self.head_dim = int(n_kv_heads), int(head_dim)

    @property
    def pool_shape(self):
        return (self.n_blocks + 1, self.block_size, self.n_kv_heads, self.head_dim)

    @property
    def scale_shape(self):
        return (self.n_blocks + 1, self.block_size, self.n_kv_heads)


def write_bf16(k_new, v_new, k_pool, v_pool, dims: Dims, tables, start_pos):
    """In-place page write into numpy uint16 pools k_pool / v_pool.  Returns the
    oracle status (0, or BAD_INDEX when a row had no valid slot)."""
    kn, vn = _arr(k_new, np.uint16), _arr(v_new, np.uint16)
    tb, sp = _arr(tables, np.int32), _arr(start_pos, np.int32)
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    n_seqs, n_new = kn.shape[0], kn.shape[1]
    return _load().pkvo_write_bf16(_p(kn), _p(vn), _p(k_pool), _p(v_pool), dims.n_blocks,
                                   dims.block_size, dims.n_kv_heads, dims.head_dim, _p(tb),
                                   tb.shape[1], _p(sp), n_seqs, n_new)


def write_int8(k_new, v_new, k_pool, v_pool, k_scales, v_scales, dims: Dims, tables, start_pos):
    """In-place quantised page write into numpy int8 pools and float32 scales."""
    kn, vn = _arr(k_new, np.uint16), _arr(v_new, np.uint16)
    tb, sp = _arr(tables, np.int32), _arr(start_pos, np.int32)
    for a, dt in ((k_pool, np.int8), (v_pool, np.int8), (k_scales, np.float32),
                  (v_scales, np.float32)):
        assert a.dtype == dt and a.flags.c_contiguous
    n_seqs, n_new = kn.shape[0], kn.shape[1]
    return _load().pkvo_write_int8(_p(kn), _p(vn), _p(k_pool), _p(v_pool), _p(k_scales),
                                   _p(v_scales), dims.n_blocks, dims.block_size, dims.n_kv_heads,
                                   dims.head_dim, _p(tb), tb.shape[1], _p(sp), n_seqs, n_new)


def gather(k_pool, v_pool, dims: Dims, tables, lens, out_tokens):
    """Returns (status, k_out, v_out) with k_out/v_out uint16
    [n_seqs, n_kv_heads, out_tokens, head_dim]."""
    kp, vp = _arr(k_pool, np.uint16), _arr(v_pool, np.uint16)
    tb, ln = _arr(tables, np.int32), _arr(lens, np.int32)
    n_seqs = tb.shape[0]
    shape = (n_seqs, dims.n_kv_heads, int(out_tokens), dims.head_dim)
    ko, vo = np.empty(shape, np.uint16), np.empty(shape, np.uint16)
    st = _load().pkvo_gather(_p(kp), _p(vp), dims.n_blocks, dims.block_size, dims.n_kv_heads,
                             dims.head_dim, _p(tb), tb.shape[1], _p(ln), n_seqs, int(out_tokens),
                             _p(ko), _p(vo))
    return st, ko, vo


def decode(q, k_pool, v_pool, dims: Dims, tables, ctx_lens, softmax_scale, k_scales=None,
           v_scales=None, split_tokens=0, n_threads=1):
    """Paged decode attention in binary64.  q: bf16 [n_seqs, Hq, D].  Pools are
    uint16 (bf16 bits) or int8 (then k_scales/v_scales float32 are required).
    Returns (status, out float64 [n_seqs, Hq, D], lse float64 [n_seqs, Hq])."""
    qa = _arr(q, np.uint16)
    n_seqs, n_q_heads, D = qa.shape
    int8 = np.asarray(k_pool).dtype == np.int8 if not hasattr(k_pool, "detach") else \
        str(k_pool.dtype) == "torch.int8"
    if int8:
        kp, vp = _arr(k_pool, np.int8), _arr(v_pool, np.int8)
        ks, vs = _arr(k_scales, np.float32), _arr(v_scales, np.float32)
    else:
        kp, vp = _arr(k_pool, np.uint16), _arr(v_pool, np.uint16)
        ks = vs = None
    tb, cl = _arr(tables, np.int32), _arr(ctx_lens, np.int32)
    out = np.zeros((n_seqs, n_q_heads, D), np.float64)
    lse = np.zeros((n_seqs, n_q_heads), np.float64)
    st = _load().pkvo_decode(_p(qa), n_q_heads, _p(kp), _p(vp), _p(ks), _p(vs), 1 if int8 else 0,
                             dims.n_blocks, dims.block_size, dims.n_kv_heads, dims.head_dim,
                             _p(tb), tb.shape[1], _p(cl), n_seqs, float(softmax_scale),
                             int(split_tokens), _p(out), _p(lse), int(n_threads))
    return st, out, lse


def prefill(q, k_pool, v_pool, dims: Dims, tables, prefix_lens, softmax_scale, row_select=None,
            n_threads=1):
    """Chunked paged prefill in binary64.  q: bf16 [n_seqs, chunk, Hq, D].
    row_select (optional bool [n_seqs, chunk]) limits the rows computed; the
    others stay NaN.  Returns (status, out float64 [n_seqs, chunk, Hq, D],
    lse float64 [n_seqs, chunk, Hq])."""
    qa = _arr(q, np.uint16)
    n_seqs, chunk, n_q_heads, D = qa.shape
    kp, vp = _arr(k_pool, np.uint16), _arr(v_pool, np.uint16)
    tb, pl = _arr(tables, np.int32), _arr(prefix_lens, np.int32)
    rs = None if row_select is None else _arr(np.asarray(row_select, dtype=bool), np.uint8)
    out = np.full((n_seqs, chunk, n_q_heads, D), np.nan, np.float64)
    lse = np.full((n_seqs, chunk, n_q_heads), np.nan, np.float64)
    st = _load().pkvo_prefill(_p(qa), n_q_heads, _p(kp), _p(vp), dims.n_blocks, dims.block_size,
                              dims.n_kv_heads, dims.head_dim, _p(tb), tb.shape[1], _p(pl), n_seqs,
                              chunk, float(softmax_scale), _p(rs), _p(out), _p(lse),
                              int(n_threads))
    return st, out, lse
