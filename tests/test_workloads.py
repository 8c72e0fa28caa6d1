"""Seeded input generators and the boundary between product and oracle (CPU)."""
import os
import re

import torch

from paged_kv_cache_212_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_draws_are_a_pure_function_of_the_parameters():
    a, b = W.tiny_decode(), W.tiny_decode()
    assert torch.equal(a.tables, b.tables) and torch.equal(a.q, b.q)
    assert all(torch.equal(x.k, y.k) for x, y in zip(a.prefix, b.prefix))
    c = W.decode_workload("x", 1, [5, 6], 8, 2, 64, 16)
    d = W.decode_workload("x", 2, [5, 6], 8, 2, 64, 16)
    assert not torch.equal(c.q, d.q)


def test_named_scenarios_have_the_stated_shapes():
    w0 = W.tiny_decode()
    assert w0.stored_lens.tolist() == [17, 64, 100, 255] and w0.n_blocks == 64 and w0.max_blocks == 16
    assert (w0.n_q_heads, w0.n_kv_heads, w0.head_dim, w0.block_size) == (8, 2, 64, 16)
    assert w0.ctx_lens.tolist() == [18, 65, 101, 256]
    w1 = W.llama8b_decode(n_seqs=16)
    assert w1.stored_lens.min() >= 512 and w1.stored_lens.max() <= 4096
    needed = sum(-(-int(c) // 16) for c in w1.ctx_lens)
    assert w1.n_blocks == -(-5 * needed // 4)                 # pool 1.25x the blocks needed
    w2 = W.llama8b_decode_int8(n_seqs=4)
    assert w2.kv_format == "int8" and w2.n_new == 16
    w3 = W.chunked_prefill(n_seqs=2)
    assert w3.kind == "prefill" and w3.n_new == 512 and w3.stored_lens.max() < 8192
    w4 = W.skewed_prefix_decode(n_seqs=32, median=600, max_len=2000)
    assert w4.stored_lens.min() >= 512 and w4.split_tokens == 512 and w4.block_size == 32
    g = W.gather_16x2048(n_seqs=2, length=64)
    assert g.extra["out_tokens"] == 64 and g.stored_lens.tolist() == [64, 64]


def test_tables_name_distinct_blocks_and_scratch_elsewhere():
    w = W.llama8b_decode(n_seqs=8)
    for s in range(w.n_seqs):
        used = w.tables[s][w.tables[s] < w.n_blocks]
        assert len(used) == -(-int(w.ctx_lens[s]) // w.block_size)
        assert (w.tables[s][len(used):] == w.n_blocks).all()      # unused entries hold the scratch id
    ids = w.tables[w.tables < w.n_blocks]
    assert len(ids.unique()) == len(ids)


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_212_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "pkv_oracle" not in text, f


def test_bench_counts_algorithmic_bytes():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    w = W.tiny_decode()
    decode_b, write_b = bench.algorithmic_bytes(w)
    tokens = int(w.ctx_lens.sum())
    kv = tokens * 2 * 2 * 64 * 2
    qo = 2 * 4 * 8 * 64 * 2
    tab = sum(-(-int(c) // 16) for c in w.ctx_lens) * 4 + 4 * 4
    assert decode_b == kv + qo + tab
    assert write_b == 2 * 2 * (4 * 1 * 2) * 64 * 2 + 4 * 8
