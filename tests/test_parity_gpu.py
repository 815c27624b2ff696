"""GPU parity: libpd (through the C ABI) against the FP64 oracle, element by
element, within |gpu - ref| <= ulp_bf16(ref) + 1e-3.

Covers the five workloads at full size (whole outputs; the large-batch
reference is computed on every host core), every split count on the tiny
workload, ragged and edge-case shapes (empty sequences, 1-token sequences,
partial last tiles, head dims that are not multiples of 64, group widths from
1 to 32, block sizes 16/32/64/256, 4096 short sequences, 32 single-head groups
at head dim 256) and both tiled layouts."""

import numpy as np
import pytest

import oracle
from oracle import policy as P
from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

from helpers import assert_within_tolerance, oracle_all_rows

pytestmark = pytest.mark.gpu


def _run(w, device, num_splits=None, gqa_pack=None):
    inp = api.PagedInputs(w, device)
    out = api.run_paged(inp, num_splits=num_splits, gqa_pack=gqa_pack)
    assert out is not None
    assert pd.pd_device_status() == 0
    return api.bf16_to_f64(out)


@pytest.mark.parametrize("pin", [1, 3])
def test_tiny_pinned_1_and_3(cuda_device, pin):
    w = W.tiny(pin=pin)
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    assert_within_tolerance(_run(w, cuda_device, num_splits=pin), ref, f"tiny N={pin}")


def test_tiny_every_split_count(cuda_device):
    w = W.tiny()
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    for n in list(range(1, 17)) + [40, 148]:
        assert_within_tolerance(_run(w, cuda_device, num_splits=n), ref, f"tiny N={n}")


EDGE_SHAPES = [
    # lens, Hq, Hkv, D, bs, N
    ([0, 1, 15, 16, 17, 31, 33, 255, 256, 257, 1000], 8, 2, 128, 16, 1),
    ([0, 1, 15, 16, 17, 31, 33, 255, 256, 257, 1000], 8, 2, 128, 16, 5),
    ([1, 7, 300, 2000], 4, 4, 64, 16, 3),        # MHA (group 1)
    ([5, 600, 1200], 12, 4, 128, 16, 2),         # group 3
    ([17, 513, 3000], 24, 8, 128, 16, 13),
    ([40, 700], 16, 1, 256, 16, 4),              # group 16 (two 8-row halves)
    ([40, 700], 32, 1, 64, 16, 2),               # group 32 (two CTAs per KV head)
    ([90, 333], 12, 1, 96, 16, 3),               # head dim padded 96 -> 128
    ([90, 333], 4, 2, 8, 16, 2),                 # head dim 8
    ([90, 333], 8, 2, 160, 16, 1),               # head dim padded 160 -> 256
    ([77, 500, 1025], 8, 1, 128, 32, 3),         # block size 32
    ([77, 500, 1025], 8, 2, 128, 64, 4),         # block size 64
    ([0, 0, 0], 8, 2, 128, 16, 3),               # nothing at all
    ([3000, 5, 256], 8, 2, 256, 256, 2),         # block size 256 at head dim 256, group 4
    ([70000], 8, 1, 64, 16, 16),                 # one very long sequence at 16 splits
    ([300, 9, 2600], 32, 2, 128, 16, 3),         # group 16 at head dim 128
]


@pytest.mark.parametrize("N", [1, 4])
def test_many_short_sequences(cuda_device, N):
    # 4096 sequences of 1..64 tokens: a grid of many waves of one-CTA units and,
    # at N = 4, a merge over 32768 rows (most sequences use one split)
    lens = np.random.default_rng(77).integers(1, 65, size=4096).tolist()
    w = W.custom(lens, 8, 2, 128, seed=78)
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    assert_within_tolerance(_run(w, cuda_device, num_splits=N, gqa_pack=False), ref, f"4096 short N={N}")


def test_wide_multi_head_at_head_dim_256(cuda_device):
    # group 1 at the largest head dim: 32 KV heads, one query head each
    w = W.custom([1, 300, 2500], 32, 32, 256, seed=79)
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    for n in (1, 3):
        assert_within_tolerance(_run(w, cuda_device, num_splits=n, gqa_pack=False), ref, f"MHA D256 N={n}")


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,N", EDGE_SHAPES)
def test_edge_shapes(cuda_device, lens, Hq, Hkv, D, bs, N):
    w = W.custom(lens, Hq, Hkv, D, block_size=bs, seed=31)
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    got = _run(w, cuda_device, num_splits=N, gqa_pack=False)
    assert_within_tolerance(got, ref, f"{lens} Hq{Hq} Hkv{Hkv} D{D} bs{bs} N{N}")
    for s, L in enumerate(lens):
        if L == 0:
            assert np.all(got[s] == 0.0)


def test_gqa_packed_full_size(cuda_device):
    w = W.gqa_packed()
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    assert_within_tolerance(_run(w, cuda_device, num_splits=1, gqa_pack=True), ref, "gqa_packed")


def test_gqa_packed_ragged_and_empty(cuda_device):
    w = W.custom([0, 1, 16, 17, 250, 4097], 16, 2, 256, seed=32)
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    got = _run(w, cuda_device, num_splits=1, gqa_pack=True)
    assert_within_tolerance(got, ref, "packed ragged")
    assert np.all(got[0] == 0.0)


def test_gqa_pack_not_applicable_launches_nothing(cuda_device):
    import torch
    w = W.custom([50], 8, 2, 256, seed=33)  # group 4: not the packed shape
    inp = api.PagedInputs(w, cuda_device)
    out = torch.full((1, 8, 256), 7.0, dtype=torch.bfloat16, device=cuda_device)
    rc = pd.pd_decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, out, w.inv_sqrt_d,
                           1, None, True)
    assert rc == pd.PD_NOT_APPLICABLE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def test_long_context_full_size(cuda_device):
    w = W.long_context()
    n = pd.pd_num_splits("auto", 0, 148, w.num_q_heads, 1, 0)
    assert n == 13
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    assert_within_tolerance(_run(w, cuda_device, num_splits=n), ref, "long_context")


def test_large_batch_full_size_whole_output(cuda_device):
    """All 256 x 32 x 128 outputs of the large-batch step (10 splits, several
    waves, longest-first order off) against the oracle, element by element."""
    w = W.large_batch()
    n = pd.pd_num_splits("auto", 0, 148, w.num_q_heads, w.num_seqs, 0)
    assert n == 10
    got = _run(w, cuda_device, num_splits=n)
    assert_within_tolerance(got, oracle_all_rows(w), "large_batch whole output")


def _tiled_check(tw, device, what):
    inp = api.TiledInputs(tw, device)
    got = api.bf16_to_f64(api.run_tiled(inp))
    assert pd.pd_device_status() == 0
    if tw.layout == "scratch":
        kf, vf = W.scratch_pool_views(tw.pool)
        strides = oracle.scratch_pool_strides(tw.num_kv_heads, tw.head_dim, tw.block_size)
    else:
        kf, vf = tw.pool, tw.v_pool
        strides = oracle.paged_strides(tw.num_kv_heads, tw.head_dim, tw.block_size)
    ref = oracle.tiled_attn(tw.q, kf, vf, tw.tile_blocks, tw.tile_block_counts,
                            tw.last_block_valid_slots, tw.num_kv_heads, tw.block_size, strides)
    assert_within_tolerance(got, ref, what)
    zero = np.where(tw.tile_block_counts.sum(axis=0) == 0)[0]
    assert len(zero) >= 1
    assert np.all(got[zero] == 0.0)


def test_tiled_scratch_pool_full_size(cuda_device):
    _tiled_check(W.tiled(), cuda_device, "tiled scratch")


def test_tiled_paged_layout(cuda_device):
    _tiled_check(W.tiled(num_seqs=16, layout="paged", max_blocks=150), cuda_device, "tiled paged")


@pytest.mark.parametrize("G,D", [(1, 64), (3, 128), (8, 128), (16, 64)])
def test_tiled_other_groups(cuda_device, G, D):
    tw = W.tiled(num_seqs=9, num_q_heads=2 * G, num_kv_heads=2, head_dim=D, tile_capacity=8,
                 num_calls=3, max_blocks=24, last_valid=11, seed=5)
    _tiled_check(tw, cuda_device, f"tiled G{G} D{D}")


def test_split_geometry_matches_oracle_policy():
    for L in (0, 1, 255, 256, 257, 32768):
        for n in (1, 3, 13):
            assert pd.pd_split_chunk_tokens(L, n, 16) == P.split_chunk_tokens(L, n, 16)


def _mixed_ref(mw):
    kflat, vflat = W.scratch_pool_views(mw.scratch)
    Hkv, D, bs = mw.num_kv_heads, mw.head_dim, mw.block_size
    calls = []
    for kind, tb, tc, lb in mw.calls:
        if kind == "paged":
            calls.append(dict(k_pool=mw.paged_k, v_pool=mw.paged_v, tile_blocks=tb, tile_block_counts=tc,
                              last_block_valid_slots=lb, strides=oracle.paged_strides(Hkv, D, bs)))
        else:
            calls.append(dict(k_pool=kflat, v_pool=vflat, tile_blocks=tb, tile_block_counts=tc,
                              last_block_valid_slots=lb, strides=oracle.scratch_pool_strides(Hkv, D, bs)))
    return oracle.tiled_attn_multi(mw.q, calls, Hkv, bs)


def test_tiled_mixed_sources_full_size(cuda_device):
    """pd_tiled_run over the paged cache then the scratch pool (tiled_attention.rs
    page: step_tile takes its pools and strides per call), 64 sequences."""
    mw = W.tiled_mixed()
    got = api.bf16_to_f64(api.run_tiled_mixed(api.MixedTiledInputs(mw, cuda_device)))
    assert pd.pd_device_status() == 0
    ref = _mixed_ref(mw)
    assert_within_tolerance(got, ref, "tiled mixed sources")
    zero = np.where(mw.blocks_per_seq == 0)[0]
    assert len(zero) >= 2 and np.all(got[zero] == 0.0)


@pytest.mark.parametrize("G,D,tcap", [(1, 64, 3), (3, 128, 8), (8, 256, 5)])
def test_tiled_mixed_sources_shapes(cuda_device, G, D, tcap):
    mw = W.tiled_mixed(num_seqs=9, num_q_heads=2 * G, num_kv_heads=2, head_dim=D, tile_capacity=tcap,
                       max_blocks=30, last_valid=7, seed=6)
    got = api.bf16_to_f64(api.run_tiled_mixed(api.MixedTiledInputs(mw, cuda_device)))
    assert_within_tolerance(got, _mixed_ref(mw), f"tiled mixed G{G} D{D}")


def test_gqa_packed_splitk_full_size(cuda_device):
    """The packed pass with splits (gqa_pack mode 2): the packed workload's
    sequences at Auto's 16 splits, partials through the workspace and the merge."""
    w = W.gqa_packed_splitk()
    inp = api.PagedInputs(w, cuda_device)
    n = inp.splits()
    assert n == 16
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    assert_within_tolerance(_run(w, cuda_device, num_splits=n, gqa_pack=2), ref, "gqa_packed splitk")


@pytest.mark.parametrize("N", [1, 2, 3, 16])
def test_gqa_packed_splitk_ragged(cuda_device, N):
    w = W.custom([0, 1, 16, 17, 255, 256, 257, 700, 2500, 4097], 16, 2, 256, seed=34)
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    got = _run(w, cuda_device, num_splits=N, gqa_pack=2)
    assert_within_tolerance(got, ref, f"packed splitk N={N}")
    assert np.all(got[0] == 0.0)


def test_gqa_packed_splitk_shape_gate(cuda_device):
    import torch
    w = W.custom([300], 8, 2, 256, seed=35)  # group 4: not the packed shape
    inp = api.PagedInputs(w, cuda_device)
    out = torch.full((1, 8, 256), 7.0, dtype=torch.bfloat16, device=cuda_device)
    ws = api.workspace(1, 8, 256, 4, cuda_device)
    rc = pd.pd_decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, out, w.inv_sqrt_d,
                           4, ws, pd.PD_GQA_PACK_SPLITK)
    assert rc == pd.PD_NOT_APPLICABLE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    with pytest.raises(pd.PdError) as e:
        pd.pd_decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, out, w.inv_sqrt_d,
                          1, None, 3)
    assert e.value.code == pd.PD_ERR_INVALID


@pytest.mark.parametrize("name", ["gqa_packed_long", "gqa_packed_long_splitk"])
def test_gqa_packed_long_full_size(cuda_device, name):
    """Few long sequences at the packed shape (2 x 32768 tokens, Hq 16, Hkv 2,
    D 256), through the non-split packed pass and through the packed pass with
    Auto's 16 splits, on the same inputs."""
    w = W.WORKLOADS[name]()
    inp = api.PagedInputs(w, cuda_device)
    n = inp.splits()
    assert n == (16 if w.gqa_pack == 2 else 1)
    ref = oracle_all_rows(w)
    assert_within_tolerance(_run(w, cuda_device, num_splits=n, gqa_pack=w.gqa_pack), ref, name)
