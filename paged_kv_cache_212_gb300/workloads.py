"""Seeded synthetic inputs shaped like the paged-KV serving scenarios.

This module only draws inputs: sequence lengths, block tables (a seeded random
permutation of the physical block ids dealt out to the sequences), and bf16
~N(0,1) values for queries, new K/V rows and the resident prefix.  It holds
none of the hot path's arithmetic (no token -> slot map, no quantisation, no
attention): both the oracle and the CUDA library receive these plain tensors
and place the resident prefix into their own pools with their own write.

Every draw comes from one ``torch.Generator`` seeded per workload, in a fixed
order, so a workload is a pure function of its parameters.  Values are drawn
as float32 N(0,1) and rounded to bf16 (round-to-nearest-even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

SEED_BASE = 20260


def _randn_bf16(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


@dataclass
class Segment:
    """Rows k/v ([n, n_kv_heads, head_dim] bf16) that belong at positions
    start .. start+n-1 of sequence ``seq`` (written through that sequence's
    table row)."""
    seq: int
    start: int
    k: torch.Tensor
    v: torch.Tensor


@dataclass
class Workload:
    name: str
    seed: int
    n_seqs: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    n_blocks: int                 # physical blocks; the pool has n_blocks + 1 rows
    max_blocks: int               # table width
    tables: torch.Tensor          # int32 [n_seqs, max_blocks]; unused entries = n_blocks
    stored_lens: torch.Tensor     # int32 [n_seqs]: tokens resident before the step
    n_new: int                    # tokens written this step per sequence
    k_new: torch.Tensor           # bf16 [n_seqs, n_new, Hkv, D]
    v_new: torch.Tensor
    q: torch.Tensor               # decode: [n_seqs, Hq, D]; prefill: [n_seqs, n_new, Hq, D]
    prefix: List[Segment]         # the resident prefix, to be placed by each side's own write
    kv_format: str = "bf16"       # "bf16" or "int8" pages
    kind: str = "decode"          # "decode" or "prefill"
    split_tokens: int = 0         # decode split size; 0 = the library chooses
    shared_blocks: int = 0        # blocks shared per group (prefix sharing), 0 if none
    group_size: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def start_pos(self) -> torch.Tensor:
        return self.stored_lens.clone()

    @property
    def ctx_lens(self) -> torch.Tensor:
        """Tokens attended by the decode query: the resident ones plus this
        step's new ones (the mask k_pos <= len of the pages' decode step)."""
        return (self.stored_lens + self.n_new).to(torch.int32)

    @property
    def softmax_scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.head_dim), dtype=torch.float32))

    @property
    def pool_shape(self) -> Tuple[int, int, int, int]:
        return (self.n_blocks + 1, self.block_size, self.n_kv_heads, self.head_dim)

    @property
    def scale_shape(self) -> Tuple[int, int, int]:
        return (self.n_blocks + 1, self.block_size, self.n_kv_heads)

    def blocks_used(self) -> int:
        return int((self.tables < self.n_blocks).sum())


def _deal_tables(gen, n_seqs, max_blocks, blocks_per_seq, n_blocks, shared=None):
    """A seeded random permutation of the n_blocks physical ids, dealt out in
    consecutive slices to the sequences in order.  With ``shared`` =
    (group_size, shared_blocks), each group of sequences first receives one
    common slice of shared_blocks ids, then each member its own slice."""
    perm = torch.randperm(n_blocks, generator=gen)
    tables = torch.full((n_seqs, max_blocks), n_blocks, dtype=torch.int32)
    cursor = 0
    if shared is None:
        for s in range(n_seqs):
            nb = blocks_per_seq[s]
            tables[s, :nb] = perm[cursor:cursor + nb].to(torch.int32)
            cursor += nb
        return tables
    group_size, n_shared = shared
    for g0 in range(0, n_seqs, group_size):
        common = perm[cursor:cursor + n_shared].to(torch.int32)
        cursor += n_shared
        for s in range(g0, min(g0 + group_size, n_seqs)):
            nb = blocks_per_seq[s]
            tables[s, :n_shared] = common
            tables[s, n_shared:nb] = perm[cursor:cursor + nb - n_shared].to(torch.int32)
            cursor += nb - n_shared
    return tables


def decode_workload(name, seed, stored_lens, n_q_heads, n_kv_heads, head_dim, block_size,
                    n_new=1, n_blocks=None, pool_factor=1.25, max_blocks=None, kv_format="bf16",
                    split_tokens=0, group_size=1, shared_tokens=0, device="cpu") -> Workload:
    """A decode step: every sequence holds stored_lens[s] tokens, writes n_new
    more at positions stored_lens[s] .., then one query per sequence attends
    all stored_lens[s] + n_new tokens.  The pool holds n_blocks physical blocks
    (default: pool_factor x the blocks needed after the write)."""
    gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in stored_lens]
    n_seqs = len(lens)
    bpt = [-(-(L + n_new) // block_size) for L in lens]
    n_shared = shared_tokens // block_size if group_size > 1 else 0
    if n_shared:
        unique = sum(b - n_shared for b in bpt) + n_shared * (-(-n_seqs // group_size))
    else:
        unique = sum(bpt)
    if n_blocks is None:
        n_blocks = max(int(math.ceil(pool_factor * unique)), 1)
    if max_blocks is None:
        max_blocks = max(bpt) if bpt else 1
    tables = _deal_tables(gen, n_seqs, max_blocks, bpt, n_blocks,
                          (group_size, n_shared) if n_shared else None)
    q = _randn_bf16(gen, (n_seqs, n_q_heads, head_dim), "cpu")
    k_new = _randn_bf16(gen, (n_seqs, n_new, n_kv_heads, head_dim), "cpu")
    v_new = _randn_bf16(gen, (n_seqs, n_new, n_kv_heads, head_dim), "cpu")
    prefix = _draw_prefix(gen, lens, n_kv_heads, head_dim, group_size, n_shared * block_size,
                          device)
    return Workload(name=name, seed=seed, n_seqs=n_seqs, n_q_heads=n_q_heads,
                    n_kv_heads=n_kv_heads, head_dim=head_dim, block_size=block_size,
                    n_blocks=n_blocks, max_blocks=max_blocks, tables=tables,
                    stored_lens=torch.tensor(lens, dtype=torch.int32), n_new=n_new,
                    k_new=k_new.to(device), v_new=v_new.to(device), q=q.to(device),
                    prefix=prefix, kv_format=kv_format, kind="decode",
                    split_tokens=split_tokens, shared_blocks=n_shared, group_size=group_size)


def _draw_prefix(gen, lens, n_kv_heads, head_dim, group_size, shared_tokens, device):
    """Resident prefix rows.  Without sharing, one segment per sequence.  With
    sharing, each group's first shared_tokens rows are drawn once (written
    through the group leader's table) and every member draws its own rest.
    Large prefixes are drawn on ``device`` from a device generator seeded from
    the CPU stream, so CPU and GPU copies of a workload only agree when
    device == "cpu"."""
    segs: List[Segment] = []
    dev_gen = gen
    if str(device) != "cpu":
        dev_gen = torch.Generator(device=device).manual_seed(
            int(torch.randint(0, 2**62, (1,), generator=gen)))
    n_seqs = len(lens)
    if shared_tokens:
        for g0 in range(0, n_seqs, group_size):
            members = range(g0, min(g0 + group_size, n_seqs))
            k = _randn_bf16(dev_gen, (shared_tokens, n_kv_heads, head_dim), device)
            v = _randn_bf16(dev_gen, (shared_tokens, n_kv_heads, head_dim), device)
            segs.append(Segment(g0, 0, k, v))
            for s in members:
                n = lens[s] - shared_tokens
                if n > 0:
                    k = _randn_bf16(dev_gen, (n, n_kv_heads, head_dim), device)
                    v = _randn_bf16(dev_gen, (n, n_kv_heads, head_dim), device)
                    segs.append(Segment(s, shared_tokens, k, v))
        return segs
    for s, L in enumerate(lens):
        if L > 0:
            k = _randn_bf16(dev_gen, (L, n_kv_heads, head_dim), device)
            v = _randn_bf16(dev_gen, (L, n_kv_heads, head_dim), device)
            segs.append(Segment(s, 0, k, v))
    return segs


def prefill_workload(name, seed, prefix_lens, chunk, n_q_heads, n_kv_heads, head_dim, block_size,
                     pool_factor=1.25, max_blocks=None, device="cpu") -> Workload:
    """A chunked-prefill step: sequence s holds prefix_lens[s] resident tokens,
    writes a chunk of ``chunk`` new rows at positions prefix_lens[s] .., and
    its ``chunk`` queries attend causally (query i sees positions <= P + i)."""
    gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in prefix_lens]
    n_seqs = len(lens)
    bpt = [-(-(L + chunk) // block_size) for L in lens]
    n_blocks = max(int(math.ceil(pool_factor * sum(bpt))), 1)
    if max_blocks is None:
        max_blocks = max(bpt) if bpt else 1
    tables = _deal_tables(gen, n_seqs, max_blocks, bpt, n_blocks)
    q = _randn_bf16(gen, (n_seqs, chunk, n_q_heads, head_dim), "cpu")
    k_new = _randn_bf16(gen, (n_seqs, chunk, n_kv_heads, head_dim), "cpu")
    v_new = _randn_bf16(gen, (n_seqs, chunk, n_kv_heads, head_dim), "cpu")
    prefix = _draw_prefix(gen, lens, n_kv_heads, head_dim, 1, 0, device)
    return Workload(name=name, seed=seed, n_seqs=n_seqs, n_q_heads=n_q_heads,
                    n_kv_heads=n_kv_heads, head_dim=head_dim, block_size=block_size,
                    n_blocks=n_blocks, max_blocks=max_blocks, tables=tables,
                    stored_lens=torch.tensor(lens, dtype=torch.int32), n_new=chunk,
                    k_new=k_new.to(device), v_new=v_new.to(device), q=q.to(device),
                    prefix=prefix, kind="prefill")


def gather_workload(name, seed, lens, n_kv_heads, head_dim, block_size, out_tokens=None,
                    pool_factor=1.25, device="cpu") -> Workload:
    """Resident bf16 sequences of the given lengths to be gathered into a
    contiguous [n_seqs, n_kv_heads, out_tokens, head_dim] view."""
    gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in lens]
    n_seqs = len(lens)
    bpt = [-(-L // block_size) for L in lens]
    n_blocks = max(int(math.ceil(pool_factor * sum(bpt))), 1)
    max_blocks = max(max(bpt) if bpt else 1, 1)
    tables = _deal_tables(gen, n_seqs, max_blocks, bpt, n_blocks)
    prefix = _draw_prefix(gen, lens, n_kv_heads, head_dim, 1, 0, device)
    empty = torch.empty((n_seqs, 0, n_kv_heads, head_dim), dtype=torch.bfloat16)
    w = Workload(name=name, seed=seed, n_seqs=n_seqs, n_q_heads=n_kv_heads,
                 n_kv_heads=n_kv_heads, head_dim=head_dim, block_size=block_size,
                 n_blocks=n_blocks, max_blocks=max_blocks, tables=tables,
                 stored_lens=torch.tensor(lens, dtype=torch.int32), n_new=0, k_new=empty,
                 v_new=empty, q=empty, prefix=prefix, kind="gather")
    w.extra["out_tokens"] = int(out_tokens if out_tokens is not None else max(lens + [0]))
    return w


# ---------------------------------------------------------------------------
# The five named scenarios.  ``scale`` < 1 keeps every shape but draws fewer
# sequences / shorter lengths, for oracle-sized test cases.
# ---------------------------------------------------------------------------

def tiny_decode(device="cpu") -> Workload:
    """Tiny decode step: stored lengths {17, 64, 100, 255}, Hq 8, Hkv 2, D 64,
    bs 16, 64 physical blocks + scratch, one new token, attend len + 1."""
    return decode_workload("tiny decode (4 seqs, Hq8/Hkv2/D64/bs16)", SEED_BASE + 0,
                           [17, 64, 100, 255], 8, 2, 64, 16, n_new=1, n_blocks=64, max_blocks=16,
                           device=device)


def _uniform_lens(gen, n, lo, hi):
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def llama8b_decode(device="cpu", n_seqs=64, lo=512, hi=4096) -> Workload:
    """Llama-3-8B-shaped decode: batch 64, stored lengths U[512, 4096], Hq 32,
    Hkv 8 (GQA 4), D 128, bs 16, pool 1.25x the blocks needed, one new token."""
    seed = SEED_BASE + 1
    lens = _uniform_lens(torch.Generator().manual_seed(seed ^ 0x5EED), n_seqs, lo, hi)
    return decode_workload(f"llama3-8b decode (batch {n_seqs}, ctx U[{lo + 1},{hi + 1}], "
                           "Hq32/Hkv8/D128/bs16)", seed, lens, 32, 8, 128, 16, n_new=1,
                           max_blocks=-(-(hi + 1) // 16), device=device)


def llama8b_decode_int8(device="cpu", n_seqs=64, lo=512, hi=4096) -> Workload:
    """The Llama-3-8B-shaped decode with int8 pages (fp32 absmax/127 scale per
    token and kv head); 16 new tokens per sequence are quantised, then one
    decode query at the last position attends stored + 16 tokens."""
    seed = SEED_BASE + 2
    lens = _uniform_lens(torch.Generator().manual_seed(seed ^ 0x5EED), n_seqs, lo, hi)
    return decode_workload(f"int8 decode (batch {n_seqs}, ctx U[{lo + 16},{hi + 16}], "
                           "Hq32/Hkv8/D128/bs16)", seed, lens, 32, 8, 128, 16, n_new=16,
                           max_blocks=-(-(hi + 16) // 16), kv_format="int8", device=device)


def gather_16x2048(device="cpu", n_seqs=16, length=2048) -> Workload:
    """The bf16 gather timed beside the int8 decode: 16 sequences of 2048 tokens,
    Hkv 8, D 128, bs 16, into a [16, 8, 2048, 128] contiguous view."""
    return gather_workload(f"gather ({n_seqs} x {length}, Hkv8/D128/bs16)", SEED_BASE + 2 + 100,
                           [length] * n_seqs, 8, 128, 16, out_tokens=length, device=device)


def chunked_prefill(device="cpu", n_seqs=8, chunk=512, prefix_hi=8192) -> Workload:
    """Chunked prefill: 8 sequences with resident prefix U{0 .. 8191}, each
    appends a 512-token chunk (paged write) attended causally within the chunk
    and fully over the prefix; Hq 32, Hkv 8, D 128, bs 16."""
    seed = SEED_BASE + 3
    g = torch.Generator().manual_seed(seed ^ 0x5EED)
    lens = [int(x) for x in torch.randint(0, prefix_hi, (n_seqs,), generator=g)]
    return prefill_workload(f"chunked prefill ({n_seqs} x {chunk} chunk, prefix U[0,{prefix_hi}), "
                            "Hq32/Hkv8/D128/bs16)", seed, lens, chunk, 32, 8, 128, 16,
                            max_blocks=-(-(prefix_hi - 1 + chunk) // 16), device=device)


def skewed_prefix_decode(device="cpu", n_seqs=256, median=1024, max_len=32768, group=16,
            shared_tokens=512) -> Workload:
    """Long skewed decode with shared prefixes: batch 256, stored lengths
    lognormal (median 1024, sigma 1 in log space) clipped to [16, 32768] and
    raised to at least the 512 shared tokens, Hq 64, Hkv 8, D 128, bs 32;
    groups of 16 share their first 512 tokens' blocks; 512-token splits."""
    seed = SEED_BASE + 4
    g = torch.Generator().manual_seed(seed ^ 0x5EED)
    z = torch.randn((n_seqs,), generator=g, dtype=torch.float64)
    lens = torch.round(torch.exp(math.log(median) + z)).clamp(16, max_len)
    lens = [max(int(x), shared_tokens) for x in lens]
    return decode_workload(f"skewed shared-prefix decode (batch {n_seqs}, lognormal median "
                           f"{median}, Hq64/Hkv8/D128/bs32, split 512)", seed, lens, 64, 8, 128, 32,
                           n_new=1, max_blocks=-(-(max_len + 1) // 32), split_tokens=512,
                           group_size=group, shared_tokens=shared_tokens, device=device)


WORKLOADS = {0: tiny_decode, 1: llama8b_decode, 2: llama8b_decode_int8, 3: chunked_prefill,
             4: skewed_prefix_decode}
