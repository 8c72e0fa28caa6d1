"""Helpers for the GPU parity tests: move oracle-built numpy pools to the
device and back.  Nothing here computes any part of the hot path."""
import os

import numpy as np
import torch

NTHREADS = max(1, os.cpu_count() or 1)


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays become bf16 (same bits)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy; bf16 becomes its uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def i32(t) -> torch.Tensor:
    return torch.as_tensor(np.asarray(t), dtype=torch.int32).cuda()


def attention_errors(gpu_out: torch.Tensor, ref: np.ndarray):
    """(max-abs, mean-abs) of the bf16 GPU output against the float64 oracle."""
    g = gpu_out.detach().cpu().to(torch.float64).numpy()
    err = np.abs(g - ref)
    return float(err.max()), float(err.mean())
