"""GB300-native paged KV cache: page write (bf16 / int8), gather, in-place paged
decode attention with split-KV, and chunked paged prefill, as hand-written
sm_103a CUDA kernels behind the C ABI of ``libpagedkv.so`` (``include/pagedkv.h``).

This module is argument marshalling only: it checks tensor shapes, dtypes and
devices, passes raw device pointers and the current CUDA stream to the
library, and turns a non-zero status into an exception.  Every step of the
computation runs in the library's kernels; there is no CPU or PyTorch
fallback, and using any call without the built library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")

PKV_KV_BF16, PKV_KV_INT8 = 0, 1
DEV_BAD_BLOCK_ID, DEV_BAD_POSITION, DEV_BAD_LENGTH = 1, 2, 4
DEV_WORKSPACE_OVERFLOW, DEV_TIMEOUT = 8, 16

EXPORTS = ("pkv_status_string", "pkv_last_cuda_error", "pkv_set_pipeline_wait_ns", "paged_kv_write",
           "paged_kv_write_int8",
           "paged_kv_gather", "pkv_decode_workspace_bytes", "paged_decode_attention",
           "paged_prefill_attention", "paged_decode_attention_noalloc", "paged_decode_step",
           "paged_kv_copy_blocks",
           # host-side block manager (include/pagedkv_blocks.h)
           "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_alloc", "pkv_bm_free", "pkv_bm_num_free",
           "pkv_bm_peak_used", "pkv_bm_refcount", "pkv_bm_can_admit", "pkv_bm_admit", "pkv_bm_release",
           "pkv_bm_fork", "pkv_bm_reserve_step", "pkv_bm_begin_step", "pkv_bm_end_step", "pkv_bm_export",
           # decode streamed from a host tier (include/pagedkv_stream.h)
           "pkv_sp_create", "pkv_sp_destroy", "pkv_sp_lookup", "pkv_sp_invalidate", "pkv_sp_plan_tile",
           "paged_kv_stage_blocks", "pkv_streamed_workspace_bytes", "paged_decode_streamed")
NOALLOC_DECODE_SCRATCH_BYTES = 16 * 1024 * 1024


class PagedKVError(RuntimeError):
    """A library call returned a non-zero PKV_* status (``status``; for
    PKV_ERR_CUDA the CUDA error code is in the message)."""

    def __init__(self, fn, status, name, cuda_error=0):
        msg = f"{fn} returned {name} ({status})"
        if cuda_error:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)
        self.status = status


class Dims(ctypes.Structure):
    """pkv_dims: pool geometry (n_blocks physical blocks, the pool tensors have
    n_blocks + 1 with the scratch block last)."""
    _fields_ = [("n_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_212_gb300.build.build() "
                           "(nvcc, sm_103a); there is no fallback path")
    lib = ctypes.CDLL(path)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_last_cuda_error.argtypes = []
    lib.pkv_last_cuda_error.restype = ctypes.c_int
    lib.pkv_set_pipeline_wait_ns.argtypes = [ctypes.c_uint64]
    lib.pkv_set_pipeline_wait_ns.restype = ctypes.c_uint64
    lib.paged_kv_write.argtypes = [P, P, P, P, Dims, P, i32, P, i32, i32, P, P]
    lib.paged_kv_write_int8.argtypes = [P, P, P, P, P, P, Dims, P, i32, P, i32, i32, P, P]
    lib.paged_kv_gather.argtypes = [P, P, Dims, P, i32, P, i32, i32, P, P, P, P]
    lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32, i64, i32]
    lib.pkv_decode_workspace_bytes.restype = sz
    lib.paged_decode_attention.argtypes = [P, i32, P, P, P, P, i32, Dims, P, i32, P, i32, ctypes.c_float,
                                           i32, P, P, P, sz, P, P]
    lib.paged_prefill_attention.argtypes = [P, i32, P, P, Dims, P, i32, P, i32, i32, ctypes.c_float, P, P,
                                            P, P]
    lib.paged_decode_attention_noalloc.argtypes = [P, i32, P, P, P, P, i32, Dims, P, i32, P, i32,
                                                   ctypes.c_float, i32, i64, P, P, P, P]
    lib.paged_decode_step.argtypes = [P, P, P, i32, P, i32, P, P, P, P, i32, Dims, P, i32, P, i32,
                                      ctypes.c_float, i32, P, P, P, sz, P, P]
    lib.paged_kv_copy_blocks.argtypes = [P, i32, P, P, P, P, i32, Dims, P, P]
    for fn in ("paged_kv_write", "paged_kv_write_int8", "paged_kv_gather", "paged_decode_attention",
               "paged_prefill_attention", "paged_decode_attention_noalloc", "paged_decode_step",
               "paged_kv_copy_blocks"):
        getattr(lib, fn).restype = ctypes.c_int
    PP = ctypes.POINTER(ctypes.c_void_p)
    lib.pkv_bm_create.argtypes = [i32, i32, i32, i32, PP]
    lib.pkv_bm_destroy.argtypes = [P]
    lib.pkv_bm_destroy.restype = None
    lib.pkv_bm_alloc.argtypes = [P, P]
    lib.pkv_bm_free.argtypes = [P, P, i32]
    lib.pkv_bm_num_free.argtypes = [P]
    lib.pkv_bm_peak_used.argtypes = [P]
    lib.pkv_bm_refcount.argtypes = [P, i32]
    lib.pkv_bm_can_admit.argtypes = [P, P, i32, P]
    lib.pkv_bm_admit.argtypes = [P, i32, i32]
    lib.pkv_bm_release.argtypes = [P, i32]
    lib.pkv_bm_fork.argtypes = [P, i32, i32]
    lib.pkv_bm_reserve_step.argtypes = [P, P, P]
    lib.pkv_bm_begin_step.argtypes = [P, P, P]
    lib.pkv_bm_end_step.argtypes = [P]
    lib.pkv_bm_export.argtypes = [P, P, P, P]
    for fn in EXPORTS:
        if fn.startswith("pkv_bm_") and fn != "pkv_bm_destroy":
            getattr(lib, fn).restype = ctypes.c_int
    lib.pkv_sp_create.argtypes = [i32, i32, PP]
    lib.pkv_sp_destroy.argtypes = [P]
    lib.pkv_sp_destroy.restype = None
    lib.pkv_sp_lookup.argtypes = [P, i32]
    lib.pkv_sp_invalidate.argtypes = [P, i32]
    lib.pkv_sp_plan_tile.argtypes = [P, P, i32, P, i32, i32, i32, P, P, P, P, P, P]
    lib.paged_kv_stage_blocks.argtypes = [P, i32, P, P, i32, P, P, Dims, P, P]
    lib.pkv_streamed_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.pkv_streamed_workspace_bytes.restype = sz
    lib.paged_decode_streamed.argtypes = [P, i32, P, P, i32, P, P, Dims, P, P, i32, P, i32, ctypes.c_float, P, P,
                                          P, sz, P, P]
    for fn in ("pkv_sp_create", "pkv_sp_lookup", "pkv_sp_invalidate", "pkv_sp_plan_tile", "paged_kv_stage_blocks",
               "paged_decode_streamed"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn, status):
    if status != 0:
        lib = load_library()
        raise PagedKVError(fn, status, lib.pkv_status_string(status).decode(),
                           lib.pkv_last_cuda_error())


def _ptr(t):
    # ctypes turns an int into the void * argument
    return None if t is None else t.data_ptr()


try:
    from torch._C import _cuda_getCurrentRawStream as _raw_stream, _cuda_getDevice as _current_device
except ImportError:      # pragma: no cover - older PyTorch builds
    _raw_stream = _current_device = None


def _stream(stream):
    """The cudaStream_t of `stream`, or of the current stream of the current
    device (as an int)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(_current_device())
    return torch.cuda.current_stream().cuda_stream


def _device_of(t, name):
    """CUDA device index of the tensor the other arguments must share."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    d = t.get_device()
    if d < 0:
        raise ValueError(f"{name} must be a CUDA tensor")
    return d


def _need(t, name, dtype=None, ndim=None, device=None):
    """A contiguous CUDA tensor of the given dtype, rank and device index; the
    common case is one test, the messages come from _refuse."""
    if (isinstance(t, torch.Tensor) and (dtype is None or t.dtype is dtype) and (ndim is None or t.dim() == ndim)
            and t.is_contiguous() and (t.get_device() == device if device is not None else t.is_cuda)):
        return
    _refuse(t, name, dtype, ndim, device)


def _refuse(t, name, dtype, ndim, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.get_device() != device:
        raise ValueError(f"{name} is on {t.device}, expected cuda:{device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    raise ValueError(f"{name} was refused")


def _shape(t, name, shape):
    """A tensor of the wrong shape would become an out-of-bounds device access:
    refuse it here."""
    if t is not None and t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check_status(dev_status, device):
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, device)
        if dev_status.numel() < 1:
            raise ValueError("dev_status needs at least one int32")


def _check_pools(k_pool, v_pool, k_scales=None, v_scales=None):
    _shape(v_pool, "v_pool", k_pool.shape)
    _shape(k_scales, "k_scales", k_pool.shape[:3])
    _shape(v_scales, "v_scales", k_pool.shape[:3])


def _check_batch(n_seqs, block_tables, lens, lens_name):
    if block_tables.shape[0] != n_seqs:
        raise ValueError(f"block_tables has {block_tables.shape[0]} rows for {n_seqs} sequences")
    _shape(lens, lens_name, (n_seqs,))


def pool_dims(k_pool: torch.Tensor) -> Dims:
    """Geometry of a [n_blocks + 1, block_size, n_kv_heads, head_dim] pool (the
    last row is the scratch block)."""
    nb1, bs, hkv, d = k_pool.shape
    return Dims(nb1 - 1, bs, hkv, d)


_dims_cache = {}


def _dims(k_pool):
    """pool_dims, one shared (never modified) structure per pool shape."""
    d = _dims_cache.get(k_pool.shape)
    if d is None:
        if len(_dims_cache) > 64:
            _dims_cache.clear()
        d = _dims_cache[k_pool.shape] = pool_dims(k_pool)
    return d


def paged_kv_write(k_new, v_new, k_pool, v_pool, block_tables, start_pos, dev_status=None, stream=None):
    """Native bf16 page write: k_new/v_new [n_seqs, n_new, Hkv, D] to positions
    start_pos[s] .. of each sequence."""
    lib = load_library()
    dev = _device_of(k_pool, "k_pool")
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, n, torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(start_pos, "start_pos", torch.int32, 1, dev)
    _check_status(dev_status, dev)
    _check_pools(k_pool, v_pool)
    _shape(k_new, "k_new", (k_new.shape[0], k_new.shape[1]) + tuple(k_pool.shape[2:]))
    _shape(v_new, "v_new", k_new.shape)
    _check_batch(k_new.shape[0], block_tables, start_pos, "start_pos")
    st = lib.paged_kv_write(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _dims(k_pool),
                            _ptr(block_tables), block_tables.shape[1], _ptr(start_pos), k_new.shape[0],
                            k_new.shape[1], _ptr(dev_status), _stream(stream))
    _check("paged_kv_write", st)


def paged_kv_write_int8(k_new, v_new, k_pool, v_pool, k_scales, v_scales, block_tables, start_pos,
                        dev_status=None, stream=None):
    """Quantised page write: int8 pools [NB+1, bs, Hkv, D], fp32 scales [NB+1, bs, Hkv]."""
    lib = load_library()
    dev = _device_of(k_pool, "k_pool")
    _need(k_new, "k_new", torch.bfloat16, 4, dev)
    _need(v_new, "v_new", torch.bfloat16, 4, dev)
    _need(k_pool, "k_pool", torch.int8, 4, dev)
    _need(v_pool, "v_pool", torch.int8, 4, dev)
    _need(k_scales, "k_scales", torch.float32, 3, dev)
    _need(v_scales, "v_scales", torch.float32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(start_pos, "start_pos", torch.int32, 1, dev)
    _check_status(dev_status, dev)
    _check_pools(k_pool, v_pool, k_scales, v_scales)
    _shape(k_new, "k_new", (k_new.shape[0], k_new.shape[1]) + tuple(k_pool.shape[2:]))
    _shape(v_new, "v_new", k_new.shape)
    _check_batch(k_new.shape[0], block_tables, start_pos, "start_pos")
    st = lib.paged_kv_write_int8(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales),
                                 _ptr(v_scales), _dims(k_pool), _ptr(block_tables), block_tables.shape[1],
                                 _ptr(start_pos), k_new.shape[0], k_new.shape[1], _ptr(dev_status),
                                 _stream(stream))
    _check("paged_kv_write_int8", st)


def paged_kv_gather(k_pool, v_pool, block_tables, lens, out_tokens, k_out=None, v_out=None, dev_status=None,
                    stream=None):
    """Contiguous copy [n_seqs, Hkv, out_tokens, D] of every sequence's pages
    (zeros past its length).  Returns (k_out, v_out)."""
    lib = load_library()
    dev = _device_of(k_pool, "k_pool")
    _need(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _need(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(lens, "lens", torch.int32, 1, dev)
    n_seqs = block_tables.shape[0]
    shape = (n_seqs, k_pool.shape[2], int(out_tokens), k_pool.shape[3])
    if k_out is None:
        k_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    if v_out is None:
        v_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    _need(k_out, "k_out", torch.bfloat16, 4, dev)
    _need(v_out, "v_out", torch.bfloat16, 4, dev)
    _check_status(dev_status, dev)
    _check_pools(k_pool, v_pool)
    _check_batch(n_seqs, block_tables, lens, "lens")
    _shape(k_out, "k_out", shape)
    _shape(v_out, "v_out", shape)
    st = lib.paged_kv_gather(_ptr(k_pool), _ptr(v_pool), _dims(k_pool), _ptr(block_tables),
                             block_tables.shape[1], _ptr(lens), n_seqs, int(out_tokens), _ptr(k_out), _ptr(v_out),
                             _ptr(dev_status), _stream(stream))
    _check("paged_kv_gather", st)
    return k_out, v_out


def paged_kv_copy_blocks(pairs, k_pool, v_pool, k_scales=None, v_scales=None, dev_status=None, stream=None):
    """Copy whole pool blocks: pairs int32 [n, 2] of (source, destination) ids
    on the device (the device half of copy-on-write)."""
    lib = load_library()
    dev = _device_of(k_pool, "k_pool")
    _need(pairs, "pairs", torch.int32, 2, dev)
    int8 = k_pool.dtype == torch.int8
    if int8:
        _need(k_scales, "k_scales", torch.float32, 3, dev)
        _need(v_scales, "v_scales", torch.float32, 3, dev)
    else:
        _need(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _need(v_pool, "v_pool", k_pool.dtype, 4, dev)
    _check_status(dev_status, dev)
    _check_pools(k_pool, v_pool, k_scales if int8 else None, v_scales if int8 else None)
    if pairs.shape[1] != 2:
        raise ValueError(f"pairs must be [n, 2], got {tuple(pairs.shape)}")
    st = lib.paged_kv_copy_blocks(_ptr(pairs), pairs.shape[0], _ptr(k_pool), _ptr(v_pool), _ptr(k_scales),
                                  _ptr(v_scales), PKV_KV_INT8 if int8 else PKV_KV_BF16, _dims(k_pool),
                                  _ptr(dev_status), _stream(stream))
    _check("paged_kv_copy_blocks", st)


def decode_workspace_bytes(n_seqs, n_q_heads, head_dim, max_total_ctx_tokens, split_tokens=0) -> int:
    """Device workspace a decode call needs for batches of n_seqs sequences whose
    contexts sum to at most max_total_ctx_tokens (pkv_decode_workspace_bytes)."""
    n = load_library().pkv_decode_workspace_bytes(int(n_seqs), int(n_q_heads), int(head_dim),
                                                  int(max_total_ctx_tokens), int(split_tokens))
    if n == 0:
        raise ValueError("invalid arguments to pkv_decode_workspace_bytes")
    return int(n)


def _check_decode(q, k_pool, v_pool, k_scales, v_scales, block_tables, ctx_lens, out, lse_out, dev_status):
    """Shapes of a decode call's tensors against q [n_seqs, Hq, D] and the pool."""
    n_seqs, n_q_heads, D = q.shape
    _check_status(dev_status, q.get_device())
    _check_pools(k_pool, v_pool, k_scales, v_scales)
    if k_pool.shape[3] != D:
        raise ValueError(f"q has head_dim {D}, the pool {k_pool.shape[3]}")
    _check_batch(n_seqs, block_tables, ctx_lens, "ctx_lens")
    _shape(out, "out", q.shape)
    _shape(lse_out, "lse_out", (n_seqs, n_q_heads))


def paged_decode_attention(q, k_pool, v_pool, block_tables, ctx_lens, softmax_scale, k_scales=None,
                           v_scales=None, split_tokens=0, out=None, lse_out=None, workspace=None,
                           max_total_ctx_tokens=None, dev_status=None, stream=None):
    """In-place paged GQA decode attention.  q [n_seqs, Hq, D] bf16; bf16 pools,
    or int8 pools with k_scales/v_scales.  Returns out [n_seqs, Hq, D] bf16.
    ``workspace`` (uint8 CUDA tensor) is allocated when not given, sized from
    max_total_ctx_tokens (default: every table entry full)."""
    lib = load_library()
    dev = _device_of(q, "q")
    _need(q, "q", torch.bfloat16, 3, dev)
    int8 = k_pool.dtype == torch.int8
    _need(k_pool, "k_pool", torch.int8 if int8 else torch.bfloat16, 4, dev)
    _need(v_pool, "v_pool", torch.int8 if int8 else torch.bfloat16, 4, dev)
    if int8:
        _need(k_scales, "k_scales", torch.float32, 3, dev)
        _need(v_scales, "v_scales", torch.float32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, 1, dev)
    n_seqs, n_q_heads, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3, dev)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, 2, dev)
    _check_decode(q, k_pool, v_pool, k_scales, v_scales, block_tables, ctx_lens, out, lse_out, dev_status)
    if workspace is None:
        if max_total_ctx_tokens is None:
            max_total_ctx_tokens = n_seqs * block_tables.shape[1] * k_pool.shape[1]
        nbytes = decode_workspace_bytes(n_seqs, n_q_heads, D, max_total_ctx_tokens, split_tokens)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, 1, dev)
    st = lib.paged_decode_attention(_ptr(q), n_q_heads, _ptr(k_pool), _ptr(v_pool), _ptr(k_scales),
                                    _ptr(v_scales), PKV_KV_INT8 if int8 else PKV_KV_BF16, _dims(k_pool),
                                    _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), n_seqs,
                                    float(softmax_scale), int(split_tokens), _ptr(out), _ptr(lse_out),
                                    _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream))
    _check("paged_decode_attention", st)
    return out


def paged_decode_step(k_new, v_new, start_pos, q, k_pool, v_pool, block_tables, ctx_lens, softmax_scale,
                      k_scales=None, v_scales=None, split_tokens=0, out=None, lse_out=None, workspace=None,
                      max_total_ctx_tokens=None, dev_status=None, stream=None):
    """One decode step of one layer: the page write of k_new/v_new
    [n_seqs, n_new, Hkv, D] at start_pos (int8 pools: quantised) and paged
    decode attention over ctx_lens tokens (which count the new rows), in one
    call.  Returns out [n_seqs, Hq, D] bf16."""
    lib = load_library()
    dev = _device_of(q, "q")
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(k_new, "k_new", torch.bfloat16, 4, dev)
    _need(v_new, "v_new", torch.bfloat16, 4, dev)
    _need(start_pos, "start_pos", torch.int32, 1, dev)
    int8 = k_pool.dtype == torch.int8
    _need(k_pool, "k_pool", torch.int8 if int8 else torch.bfloat16, 4, dev)
    _need(v_pool, "v_pool", torch.int8 if int8 else torch.bfloat16, 4, dev)
    if int8:
        _need(k_scales, "k_scales", torch.float32, 3, dev)
        _need(v_scales, "v_scales", torch.float32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, 1, dev)
    n_seqs, n_q_heads, D = q.shape
    if k_new.shape[0] != n_seqs:
        raise ValueError("k_new and q disagree on n_seqs")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3, dev)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, 2, dev)
    _check_decode(q, k_pool, v_pool, k_scales, v_scales, block_tables, ctx_lens, out, lse_out, dev_status)
    _shape(k_new, "k_new", (n_seqs, k_new.shape[1]) + tuple(k_pool.shape[2:]))
    _shape(v_new, "v_new", k_new.shape)
    _shape(start_pos, "start_pos", (n_seqs,))
    if workspace is None:
        if max_total_ctx_tokens is None:
            max_total_ctx_tokens = n_seqs * block_tables.shape[1] * k_pool.shape[1]
        nbytes = decode_workspace_bytes(n_seqs, n_q_heads, D, max_total_ctx_tokens, split_tokens)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, 1, dev)
    st = lib.paged_decode_step(_ptr(k_new), _ptr(v_new), _ptr(start_pos), k_new.shape[1], _ptr(q), n_q_heads,
                               _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
                               PKV_KV_INT8 if int8 else PKV_KV_BF16, _dims(k_pool), _ptr(block_tables),
                               block_tables.shape[1], _ptr(ctx_lens), n_seqs, float(softmax_scale),
                               int(split_tokens), _ptr(out), _ptr(lse_out), _ptr(workspace), workspace.numel(),
                               _ptr(dev_status), _stream(stream))
    _check("paged_decode_step", st)
    return out


class DecodePlan:
    """paged_decode_attention / paged_decode_step with the arguments that stay
    the same from call to call checked once: the pools (and int8 scales), the
    block tables and lengths, the workspace, out, lse_out and dev_status.
    ``run(q)`` then checks only q (and, for a step, k_new / v_new / start_pos)
    before the library call, which keeps the host's cost per call low where
    the GPU work is short (small batches, one call per layer).

    The plan keeps references to its tensors and reads their contents at every
    call (so block tables and lengths may be rewritten in place between calls);
    they must keep their shapes and storage: resizing one after planning is not
    allowed.  ``max_total_ctx_tokens`` bounds sum(ctx_lens) over every call.
    Returns ``out`` from ``run``."""

    def __init__(self, k_pool, v_pool, block_tables, ctx_lens, softmax_scale, n_q_heads, k_scales=None,
                 v_scales=None, split_tokens=0, out=None, lse_out=None, workspace=None, max_total_ctx_tokens=None,
                 dev_status=None):
        dev = _device_of(k_pool, "k_pool")
        self._lib = load_library()
        n_seqs, D = block_tables.shape[0], k_pool.shape[3]
        q_like = torch.empty((n_seqs, int(n_q_heads), D), dtype=torch.bfloat16, device=dev)
        if out is None:
            out = torch.empty_like(q_like)
        # the one-call checks against a query of the planned shape
        self.int8 = k_pool.dtype is torch.int8
        _need(k_pool, "k_pool", torch.int8 if self.int8 else torch.bfloat16, 4, dev)
        _need(v_pool, "v_pool", torch.int8 if self.int8 else torch.bfloat16, 4, dev)
        if self.int8:
            _need(k_scales, "k_scales", torch.float32, 3, dev)
            _need(v_scales, "v_scales", torch.float32, 3, dev)
        _need(block_tables, "block_tables", torch.int32, 2, dev)
        _need(ctx_lens, "ctx_lens", torch.int32, 1, dev)
        _need(out, "out", torch.bfloat16, 3, dev)
        if lse_out is not None:
            _need(lse_out, "lse_out", torch.float32, 2, dev)
        _check_decode(q_like, k_pool, v_pool, k_scales, v_scales, block_tables, ctx_lens, out, lse_out, dev_status)
        if workspace is None:
            if max_total_ctx_tokens is None:
                max_total_ctx_tokens = n_seqs * block_tables.shape[1] * k_pool.shape[1]
            workspace = torch.empty(decode_workspace_bytes(n_seqs, n_q_heads, D, max_total_ctx_tokens,
                                                           split_tokens), dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, 1, dev)
        self.device, self.q_shape, self.out = dev, q_like.shape, out
        self.new_shape_tail = tuple(k_pool.shape[2:])
        # held so that the pointers below stay valid
        self._tensors = (k_pool, v_pool, k_scales, v_scales, block_tables, ctx_lens, out, lse_out, workspace,
                         dev_status)
        self._pools = (_ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
                       PKV_KV_INT8 if self.int8 else PKV_KV_BF16, pool_dims(k_pool), _ptr(block_tables),
                       block_tables.shape[1], _ptr(ctx_lens), n_seqs, float(softmax_scale), int(split_tokens),
                       _ptr(out), _ptr(lse_out), _ptr(workspace), workspace.numel(), _ptr(dev_status))
        self.n_q_heads, self.n_seqs = int(n_q_heads), n_seqs

    def run(self, q, k_new=None, v_new=None, start_pos=None, stream=None):
        """Decode attention of q [n_seqs, Hq, D] (bf16) over the planned pools;
        with k_new / v_new [n_seqs, n_new, Hkv, D] and start_pos [n_seqs] the
        step's page write runs first, in the same call (paged_decode_step)."""
        dev = self.device
        _need(q, "q", torch.bfloat16, 3, dev)
        _shape(q, "q", self.q_shape)
        if k_new is None:
            if v_new is not None or start_pos is not None:
                raise ValueError("v_new and start_pos come with k_new")
            st = self._lib.paged_decode_attention(q.data_ptr(), self.n_q_heads, *self._pools, _stream(stream))
            _check("paged_decode_attention", st)
            return self.out
        _need(k_new, "k_new", torch.bfloat16, 4, dev)
        _need(v_new, "v_new", torch.bfloat16, 4, dev)
        _need(start_pos, "start_pos", torch.int32, 1, dev)
        n_new = k_new.shape[1]
        _shape(k_new, "k_new", (self.n_seqs, n_new) + self.new_shape_tail)
        _shape(v_new, "v_new", k_new.shape)
        _shape(start_pos, "start_pos", (self.n_seqs,))
        st = self._lib.paged_decode_step(k_new.data_ptr(), v_new.data_ptr(), start_pos.data_ptr(), n_new,
                                         q.data_ptr(), self.n_q_heads, *self._pools, _stream(stream))
        _check("paged_decode_step", st)
        return self.out


def paged_decode_attention_noalloc(q, k_pool, v_pool, block_tables, ctx_lens, softmax_scale,
                                   max_total_ctx_tokens, out, k_scales=None, v_scales=None, split_tokens=0,
                                   lse_out=None, dev_status=None, stream=None):
    """paged_decode_attention for callers that cannot allocate device memory:
    the split-KV scratch is the library's own static 16 MiB device array, so
    no workspace is passed and the call allocates nothing (``out`` must be
    given).  max_total_ctx_tokens bounds sum(ctx_lens); a request whose
    scratch would not fit raises (PKV_ERR_WORKSPACE).  Calls share the one
    array: do not let two of them overlap on the GPU."""
    lib = load_library()
    dev = _device_of(q, "q")
    _need(q, "q", torch.bfloat16, 3, dev)
    int8 = k_pool.dtype == torch.int8
    _need(k_pool, "k_pool", torch.int8 if int8 else torch.bfloat16, 4, dev)
    _need(v_pool, "v_pool", torch.int8 if int8 else torch.bfloat16, 4, dev)
    if int8:
        _need(k_scales, "k_scales", torch.float32, 3, dev)
        _need(v_scales, "v_scales", torch.float32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, 1, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, 2, dev)
    _check_decode(q, k_pool, v_pool, k_scales, v_scales, block_tables, ctx_lens, out, lse_out, dev_status)
    n_seqs, n_q_heads, _ = q.shape
    st = lib.paged_decode_attention_noalloc(_ptr(q), n_q_heads, _ptr(k_pool), _ptr(v_pool), _ptr(k_scales),
                                            _ptr(v_scales), PKV_KV_INT8 if int8 else PKV_KV_BF16,
                                            _dims(k_pool), _ptr(block_tables), block_tables.shape[1],
                                            _ptr(ctx_lens), n_seqs, float(softmax_scale), int(split_tokens),
                                            int(max_total_ctx_tokens), _ptr(out), _ptr(lse_out),
                                            _ptr(dev_status), _stream(stream))
    _check("paged_decode_attention_noalloc", st)
    return out


def paged_prefill_attention(q, k_pool, v_pool, block_tables, prefix_lens, softmax_scale, out=None,
                            lse_out=None, dev_status=None, stream=None):
    """Chunked paged prefill: q [n_seqs, chunk, Hq, D] bf16 (the chunk's K/V
    already written at prefix_lens[s] ..).  Returns out, same shape as q."""
    lib = load_library()
    dev = _device_of(q, "q")
    _need(q, "q", torch.bfloat16, 4, dev)
    _need(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _need(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(prefix_lens, "prefix_lens", torch.int32, 1, dev)
    n_seqs, chunk, n_q_heads, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4, dev)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, 3, dev)
    _check_status(dev_status, dev)
    _check_pools(k_pool, v_pool)
    if k_pool.shape[3] != q.shape[3]:
        raise ValueError(f"q has head_dim {q.shape[3]}, the pool {k_pool.shape[3]}")
    _check_batch(n_seqs, block_tables, prefix_lens, "prefix_lens")
    _shape(out, "out", q.shape)
    _shape(lse_out, "lse_out", q.shape[:3])
    st = lib.paged_prefill_attention(_ptr(q), n_q_heads, _ptr(k_pool), _ptr(v_pool), _dims(k_pool),
                                     _ptr(block_tables), block_tables.shape[1], _ptr(prefix_lens), n_seqs,
                                     chunk, float(softmax_scale), _ptr(out), _ptr(lse_out), _ptr(dev_status),
                                     _stream(stream))
    _check("paged_prefill_attention", st)
    return out


class BlockManager:
    """The library's host-side block manager (include/pagedkv_blocks.h): free
    stack and reference counts of n_blocks blocks, n_slots sequence slots with
    tables of max_blocks entries.  Methods mirror the C calls; failures raise
    PagedKVError (nothing changed)."""

    def __init__(self, n_blocks, block_size, n_slots, max_blocks):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check("pkv_bm_create", self._lib.pkv_bm_create(int(n_blocks), int(block_size), int(n_slots),
                                                          int(max_blocks), ctypes.byref(h)))
        self._h = h
        self.n_blocks, self.block_size, self.n_slots, self.max_blocks = n_blocks, block_size, n_slots, max_blocks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pkv_bm_destroy(h)
            self._h = None

    def _call(self, fn, *args):
        _check(fn, getattr(self._lib, fn)(self._h, *args))

    @staticmethod
    def _ints(values):
        arr = (ctypes.c_int32 * max(1, len(values)))(*values)
        return arr

    def alloc(self) -> int:
        b = ctypes.c_int32()
        self._call("pkv_bm_alloc", ctypes.byref(b))
        return b.value

    def free(self, blocks):
        self._call("pkv_bm_free", self._ints(list(blocks)), len(blocks))

    @property
    def num_free(self) -> int:
        return self._lib.pkv_bm_num_free(self._h)

    @property
    def peak_used(self) -> int:
        return self._lib.pkv_bm_peak_used(self._h)

    def refcount(self, block) -> int:
        return self._lib.pkv_bm_refcount(self._h, int(block))

    def can_admit(self, lengths) -> bool:
        ok = ctypes.c_int32()
        self._call("pkv_bm_can_admit", self._ints(list(lengths)), len(lengths), ctypes.byref(ok))
        return bool(ok.value)

    def admit(self, slot, n_tokens):
        self._call("pkv_bm_admit", int(slot), int(n_tokens))

    def release(self, slot):
        self._call("pkv_bm_release", int(slot))

    def fork(self, src_slot, dst_slot):
        self._call("pkv_bm_fork", int(src_slot), int(dst_slot))

    def reserve_step(self):
        victims = (ctypes.c_int32 * self.n_slots)()
        n = ctypes.c_int32()
        self._call("pkv_bm_reserve_step", victims, ctypes.byref(n))
        return list(victims[:n.value])

    def begin_step(self):
        copies = (ctypes.c_int32 * (2 * self.n_slots))()
        n = ctypes.c_int32()
        self._call("pkv_bm_begin_step", copies, ctypes.byref(n))
        return [(copies[2 * i], copies[2 * i + 1]) for i in range(n.value)]

    def end_step(self):
        self._call("pkv_bm_end_step")

    def export(self):
        """(tables [n_slots][max_blocks], lens [n_slots], active [n_slots]) as int32 CPU tensors."""
        tables = torch.empty((self.n_slots, self.max_blocks), dtype=torch.int32)
        lens = torch.empty(self.n_slots, dtype=torch.int32)
        active = torch.empty(self.n_slots, dtype=torch.int32)
        self._call("pkv_bm_export", ctypes.c_void_p(tables.data_ptr()), ctypes.c_void_p(lens.data_ptr()),
                   ctypes.c_void_p(active.data_ptr()))
        return tables, lens, active


class ScratchPool:
    """Residency of a device scratch pool of n_slots blocks for decode streamed
    from a host tier (include/pagedkv_stream.h)."""

    def __init__(self, n_slots, max_seqs):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check("pkv_sp_create", self._lib.pkv_sp_create(int(n_slots), int(max_seqs), ctypes.byref(h)))
        self._h = h
        self.n_slots, self.max_seqs = int(n_slots), int(max_seqs)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pkv_sp_destroy(h)
            self._h = None

    def lookup(self, host_block) -> int:
        return self._lib.pkv_sp_lookup(self._h, int(host_block))

    def invalidate(self, host_block):
        _check("pkv_sp_invalidate", self._lib.pkv_sp_invalidate(self._h, int(host_block)))

    def plan_tile(self, host_tables, ctx_lens, block_size, cursor, tile_blocks=0):
        """Plan the next tile of at most tile_blocks blocks (0: n_slots) from host
        int32 tensors; returns (tile_tables, tile_lens, pairs list, done) and
        advances cursor (a 2-element list)."""
        host_tables = host_tables.to(torch.int32).contiguous()
        ctx_lens = ctx_lens.to(torch.int32).contiguous()
        n_seqs = ctx_lens.shape[0]
        cap = self.n_slots if tile_blocks <= 0 or tile_blocks > self.n_slots else int(tile_blocks)
        tt = torch.empty((n_seqs, min(cap, host_tables.shape[1])), dtype=torch.int32)
        tl = torch.empty(n_seqs, dtype=torch.int32)
        pr = torch.empty((self.n_slots, 2), dtype=torch.int32)
        cur = (ctypes.c_int32 * 2)(*cursor)
        n, done = ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_sp_plan_tile", self._lib.pkv_sp_plan_tile(
            self._h, ctypes.c_void_p(host_tables.data_ptr()), host_tables.shape[1],
            ctypes.c_void_p(ctx_lens.data_ptr()), n_seqs, int(block_size), int(tile_blocks), cur,
            ctypes.c_void_p(tt.data_ptr()),
            ctypes.c_void_p(tl.data_ptr()), ctypes.c_void_p(pr.data_ptr()), ctypes.byref(n), ctypes.byref(done)))
        cursor[0], cursor[1] = cur[0], cur[1]
        return tt, tl, [tuple(x) for x in pr[:n.value].tolist()], bool(done.value)


def paged_kv_stage_blocks(pairs, host_k, host_v, pool_k, pool_v, dev_status=None, stream=None):
    """Copy host-tier blocks (pinned CPU tensors [n_host_blocks, bs, Hkv, D]
    bf16) into scratch-pool slots (device [n_slots + 1, bs, Hkv, D]):
    pairs int32 [n, 2] (host block, slot) on the device."""
    lib = load_library()
    dev = _device_of(pool_k, "pool_k")
    _need(pairs, "pairs", torch.int32, 2, dev)
    for t, n in ((host_k, "host_k"), (host_v, "host_v")):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 CPU tensor [n_host_blocks, bs, Hkv, D]")
    _need(pool_k, "pool_k", torch.bfloat16, 4, dev)
    _need(pool_v, "pool_v", torch.bfloat16, 4, dev)
    _check_status(dev_status, dev)
    _check_pools(pool_k, pool_v)
    if pairs.shape[1] != 2:
        raise ValueError(f"pairs must be [n, 2], got {tuple(pairs.shape)}")
    if tuple(host_k.shape[1:]) != tuple(pool_k.shape[1:]) or host_v.shape != host_k.shape:
        raise ValueError("host_k / host_v blocks must match the scratch pool's [bs, Hkv, D]")
    st = lib.paged_kv_stage_blocks(_ptr(pairs), pairs.shape[0], ctypes.c_void_p(host_k.data_ptr()),
                                   ctypes.c_void_p(host_v.data_ptr()), host_k.shape[0], _ptr(pool_k), _ptr(pool_v),
                                   _dims(pool_k), _ptr(dev_status), _stream(stream))
    _check("paged_kv_stage_blocks", st)


def streamed_workspace_bytes(n_seqs, n_q_heads, head_dim, n_slots, block_size) -> int:
    """Device workspace paged_decode_streamed needs (pkv_streamed_workspace_bytes)."""
    n = load_library().pkv_streamed_workspace_bytes(int(n_seqs), int(n_q_heads), int(head_dim), int(n_slots),
                                                    int(block_size))
    if n == 0:
        raise ValueError("invalid arguments to pkv_streamed_workspace_bytes")
    return int(n)


def paged_decode_streamed(q, host_k, host_v, pool_k, pool_v, scratch_pool, host_tables, ctx_lens, softmax_scale,
                          out=None, lse_out=None, workspace=None, dev_status=None, stream=None):
    """Decode attention over blocks in a host tier (pinned CPU tensors), streamed
    through the device scratch pool (pool_k/pool_v [n_slots + 1, bs, Hkv, D]) one
    tile of at most n_slots blocks at a time.  host_tables / ctx_lens: int32 CPU
    tensors.  Returns out (bf16 [n_seqs, Hq, D])."""
    lib = load_library()
    dev = _device_of(q, "q")
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(pool_k, "pool_k", torch.bfloat16, 4, dev)
    _need(pool_v, "pool_v", torch.bfloat16, 4, dev)
    for t, n in ((host_k, "host_k"), (host_v, "host_v")):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 CPU tensor [n_host_blocks, bs, Hkv, D]")
    host_tables = host_tables.to(torch.int32).contiguous()
    ctx_lens = ctx_lens.to(torch.int32).contiguous()
    if host_tables.device.type != "cpu" or ctx_lens.device.type != "cpu":
        raise ValueError("host_tables and ctx_lens are host (CPU) tensors")
    n_seqs, n_q_heads, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3, dev)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, 2, dev)
    _check_status(dev_status, dev)
    _check_pools(pool_k, pool_v)
    if tuple(host_k.shape[1:]) != tuple(pool_k.shape[1:]) or host_v.shape != host_k.shape:
        raise ValueError("host_k / host_v blocks must match the scratch pool's [bs, Hkv, D]")
    if pool_k.shape[3] != D:
        raise ValueError(f"q has head_dim {D}, the pool {pool_k.shape[3]}")
    _check_batch(n_seqs, host_tables, ctx_lens, "ctx_lens")
    _shape(out, "out", q.shape)
    _shape(lse_out, "lse_out", (n_seqs, n_q_heads))
    if workspace is None:
        workspace = torch.empty(streamed_workspace_bytes(n_seqs, n_q_heads, D, pool_k.shape[0] - 1,
                                                         pool_k.shape[1]), dtype=torch.uint8, device=dev)
    st = lib.paged_decode_streamed(
        _ptr(q), n_q_heads, ctypes.c_void_p(host_k.data_ptr()), ctypes.c_void_p(host_v.data_ptr()),
        host_k.shape[0], _ptr(pool_k), _ptr(pool_v), _dims(pool_k), scratch_pool._h,
        ctypes.c_void_p(host_tables.data_ptr()), host_tables.shape[1], ctypes.c_void_p(ctx_lens.data_ptr()), n_seqs,
        float(softmax_scale), _ptr(out), _ptr(lse_out), _ptr(workspace), workspace.numel(), _ptr(dev_status),
        _stream(stream))
    _check("paged_decode_streamed", st)
    return out
