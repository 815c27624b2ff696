"""The synthetic inputs are the recipe the measurements are quoted on: each
workload's shape, policy and algorithmic K/V bytes (seed 0), and the
structure of its placement (every sequence's blocks distinct and inside a pool
of ceil(1.25 x needed) blocks).  CPU only; the large batch is checked through
its length generator, without drawing its 3 GB of values."""

import numpy as np
import pytest

from oracle import policy as P
from paged_kv_decode_splitk_gb300 import workloads as W


def _placement_ok(w):
    need = -(-w.context_lens.astype(np.int64) // w.block_size)
    used = np.concatenate([w.block_table[s, :n] for s, n in enumerate(need)] or [np.zeros(0, np.int32)])
    assert len(np.unique(used)) == len(used), "a block serves two places"
    assert used.min(initial=0) >= 0 and used.max(initial=0) < w.num_blocks


def test_tiny():
    w = W.tiny()
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks) == (4, 1, 64, 16, 16)
    assert w.context_lens.tolist() == [37, 100] and w.inv_sqrt_d == 0.125
    assert w.kv_bytes == 35_072
    _placement_ok(w)


def test_gqa_packed():
    w = W.gqa_packed()
    assert (w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size) == (32, 16, 2, 256, 16)
    assert w.context_lens.min() >= 512 and w.context_lens.max() <= 4096
    assert w.gqa_pack and P.gqa_pack_shape_ok(16, 2, 256)
    assert w.kv_bytes == 150_677_504
    need = int((-(-w.context_lens.astype(np.int64) // 16)).sum())
    assert w.num_blocks == int(np.ceil(1.25 * need))
    _placement_ok(w)


def test_long_context():
    w = W.long_context()
    assert (w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim) == (1, 24, 8, 128)
    assert w.kv_bytes == 32768 * 8 * 128 * 2 * 2 == 134_217_728
    assert P.num_splits(P.POLICY_AUTO, 0, w.sm_count, w.num_q_heads, 1, 0) == 13


def test_large_batch_lengths():
    lens = W.large_batch_lens()
    assert lens.size == 256 and lens.min() >= 16 and lens.max() <= 16384
    assert abs(float(np.median(lens)) - 2048) < 400
    assert int(lens.sum()) * 8 * 128 * 2 * 2 == 3_174_469_632
    assert P.num_splits(P.POLICY_AUTO, 0, 148, 32, 256, 0) == 10


def test_tiled():
    tw = W.tiled()
    assert (tw.num_seqs, tw.num_q_heads, tw.num_kv_heads, tw.head_dim, tw.block_size) == (64, 16, 4, 256, 16)
    assert tw.tile_capacity == 64 and tw.num_calls == 4 and tw.layout == "scratch"
    assert tw.kv_bytes == 510_287_872
    assert int((tw.blocks_per_seq == 0).sum()) >= 2
    # right-aligned calls: full blocks before the last call, 5 valid slots in it
    assert list(tw.last_block_valid_slots[:-1]) == [16] * 3 and tw.last_block_valid_slots[-1] == 5


def test_fp8_variant_halves_the_bytes():
    w = W.fp8_variant(W.custom([100, 700], 8, 2, 128, seed=3), k_scale=0.5, v_scale=0.25, seed=4)
    assert w.kv_dtype == "e4m3" and w.k_cache.dtype == np.uint8 and w.kv_elem_bytes == 1
    bf = W.custom([100, 700], 8, 2, 128, seed=3)
    assert 2 * w.kv_bytes == bf.kv_bytes
    # no NaN code (0x7f / 0xff) in the cache
    assert not np.any((w.k_cache & 0x7F) == 0x7F) and not np.any((w.v_cache & 0x7F) == 0x7F)


def test_gqa_packed_long_pair():
    """Few long sequences at the packed shape: the non-split and the split
    variant draw the same sequences, cache and block table."""
    a, b = W.gqa_packed_long(), W.gqa_packed_long_splitk()
    for w in (a, b):
        assert (w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size) == (2, 16, 2, 256, 16)
        assert w.context_lens.tolist() == [32768, 32768]
        assert w.kv_bytes == 2 * 32768 * 2 * 256 * 2 * 2 == 134_217_728
        _placement_ok(w)
    assert a.gqa_pack == 1 and a.policy == "pinned" and a.pin == 1
    assert b.gqa_pack == 2 and P.num_splits(P.POLICY_AUTO, 0, b.sm_count, b.num_q_heads, 2, 0) == 16
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.q, b.q)


def test_first_seqs_keeps_values_and_compacts_the_cache():
    """A sub-batch for profiler captures: the first n sequences, the same K/V rows
    through a cache that holds only their blocks."""
    w = W.custom([37, 300, 1000, 5, 2049], 8, 2, 64, seed=12)
    sub = W.first_seqs(w, 3)
    assert sub.num_seqs == 3 and sub.context_lens.tolist() == [37, 300, 1000]
    assert np.array_equal(sub.q, w.q[:3])
    need = [-(-int(L) // 16) for L in sub.context_lens]
    assert sub.num_blocks == sum(need)
    for s, k in enumerate(need):
        for j in range(k):
            assert np.array_equal(sub.k_cache[sub.block_table[s, j]], w.k_cache[w.block_table[s, j]])
            assert np.array_equal(sub.v_cache[sub.block_table[s, j]], w.v_cache[w.block_table[s, j]])
    _placement_ok(sub)
