"""Error paths on the GPU, all made on the host or caught by the kernels' own
bounds checks (no trap, no fault): out-of-range block ids read zeros and raise
a device status flag, oversized context lengths and tile counts are clamped
and flagged, capacity and allocation failures come back as error codes."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

from helpers import assert_within_tolerance

pytestmark = pytest.mark.gpu


def test_status_starts_clear(cuda_device):
    pd.pd_device_status()
    assert pd.pd_device_status() == 0


def test_out_of_range_block_id_is_flagged_not_fatal(cuda_device):
    w = W.custom([40, 40], 8, 2, 128, seed=51)
    w.block_table[1, 1] = w.num_blocks + 1000   # outside the cache: reads zeros
    inp = api.PagedInputs(w, cuda_device)
    out = api.run_paged(inp, num_splits=1, gqa_pack=False)
    assert pd.pd_device_status() & pd.PD_DEV_BAD_BLOCK_ID
    got = api.bf16_to_f64(out)
    assert np.all(np.isfinite(got))
    # sequence 0 is untouched by the bad id
    good = W.custom([40, 40], 8, 2, 128, seed=51)
    ref = oracle.decode_attn(good.q[:1], good.k_cache, good.v_cache, good.block_table[:1],
                             good.context_lens[:1], good.inv_sqrt_d)
    assert_within_tolerance(got[:1], ref, "clean sequence")
    # the library keeps working afterwards
    out2 = api.run_paged(api.PagedInputs(good, cuda_device), num_splits=2, gqa_pack=False)
    assert pd.pd_device_status() == 0
    assert_within_tolerance(api.bf16_to_f64(out2)[:1], ref, "after the fault")


def test_negative_block_id_is_flagged(cuda_device):
    w = W.custom([20], 4, 1, 64, seed=52)
    w.block_table[0, 0] = -5
    api.run_paged(api.PagedInputs(w, cuda_device), num_splits=1, gqa_pack=False)
    assert pd.pd_device_status() & pd.PD_DEV_BAD_BLOCK_ID


def test_context_len_beyond_block_table_is_clamped(cuda_device):
    w = W.custom([32, 32], 4, 1, 64, seed=53)
    bad = w.context_lens.copy()
    bad[1] = 10_000                             # the table holds 2 blocks (32 tokens)
    inp = api.PagedInputs(w, cuda_device)
    inp.context_lens = api.i32_tensor(bad, cuda_device)
    out = api.run_paged(inp, num_splits=3, gqa_pack=False)
    assert pd.pd_device_status() & pd.PD_DEV_BAD_CONTEXT_LEN
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    assert_within_tolerance(api.bf16_to_f64(out), ref, "clamped to the table")


def test_tile_count_above_capacity_is_clamped(cuda_device):
    tw = W.tiled(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=64, tile_capacity=4,
                 num_calls=2, max_blocks=8, seed=54)
    inp = api.TiledInputs(tw, cuda_device)
    counts = tw.tile_block_counts[0].copy()
    counts[0] = 99
    inp.tile_counts[0] = api.i32_tensor(counts, cuda_device)
    api.run_tiled(inp)
    assert pd.pd_device_status() & pd.PD_DEV_BAD_TILE_COUNT


def test_tiled_capacity_errors(cuda_device):
    t = pd.Tiled(4, 8, 2, 64, 16, 8)
    try:
        with pytest.raises(pd.PdError) as e:
            t.begin(5)
        assert e.value.code == pd.PD_ERR_CAPACITY
        out = torch.empty((5, 8, 64), dtype=torch.bfloat16, device=cuda_device)
        with pytest.raises(pd.PdError) as e:
            t.finalize(out, 5)
        assert e.value.code == pd.PD_ERR_CAPACITY
        q = torch.zeros((4, 8, 64), dtype=torch.bfloat16, device=cuda_device)
        blocks = torch.zeros((4, 8), dtype=torch.int32, device=cuda_device)
        with pytest.raises(pd.PdError) as e:
            t.step(q, q, q, blocks, blocks[:, 0], 5, t.paged_strides(), 16)
        assert e.value.code == pd.PD_ERR_CAPACITY
        with pytest.raises(pd.PdError) as e:
            t.step(q, q, q, blocks, blocks[:, 0], 4, (12, 64, 64), 16)  # stride not a multiple of 8
        assert e.value.code == pd.PD_ERR_INVALID
    finally:
        t.close()


def test_tiled_create_allocation_failure_is_reported(cuda_device):
    pd.pd_debug_fail_next_allocs(1)
    with pytest.raises(pd.PdError) as e:
        pd.Tiled(4, 8, 2, 64, 16, 8)
    assert e.value.code == pd.PD_ERR_ALLOC
    pd.pd_debug_fail_next_allocs(0)
    t = pd.Tiled(4, 8, 2, 64, 16, 8)   # and the next create works
    t.close()


def test_workspace_too_small(cuda_device):
    w = W.custom([300], 8, 2, 128, seed=55)
    inp = api.PagedInputs(w, cuda_device)
    out = torch.empty((1, 8, 128), dtype=torch.bfloat16, device=cuda_device)
    ws = torch.empty(100, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(pd.PdError) as e:
        pd.pd_decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, out, w.inv_sqrt_d,
                          4, ws, False)
    assert e.value.code == pd.PD_ERR_WORKSPACE


def test_begin_resets_state(cuda_device):
    tw = W.tiled(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=64, tile_capacity=8,
                 num_calls=2, max_blocks=16, seed=56)
    inp = api.TiledInputs(tw, cuda_device)
    t = pd.Tiled(4, 8, 2, 64, 16, 8)
    try:
        a = api.bf16_bits(api.run_tiled(inp, t))
        b = api.bf16_bits(api.run_tiled(inp, t))   # same handle, second decode step
        assert np.array_equal(a, b)
        # begin then finalize with no step in between: l = 0 everywhere -> output 0
        out = torch.full((4, 8, 64), 3.0, dtype=torch.bfloat16, device=cuda_device)
        t.begin(4)
        t.finalize(out, 4)
        torch.cuda.synchronize()
        assert bool((out == 0).all())
    finally:
        t.close()


def test_tiled_run_checks_every_source_before_launching(cuda_device):
    """A bad source anywhere in the list is reported before anything launches:
    the running state and the output keep their contents."""
    mw = W.tiled_mixed(num_seqs=5, num_q_heads=8, num_kv_heads=2, head_dim=64, tile_capacity=4,
                       max_blocks=16, seed=57)
    inp = api.MixedTiledInputs(mw, cuda_device)
    t = pd.Tiled(5, 8, 2, 64, 16, 4)
    try:
        good = inp.sources(t)
        out = torch.full((5, 8, 64), 3.0, dtype=torch.bfloat16, device=cuda_device)
        bad = list(good)
        k, v, tb, tc, st, lb = bad[-1]
        bad[-1] = (k, v, tb, tc, (st[0], 12, st[2]), lb)     # tok stride not a multiple of 8
        with pytest.raises(pd.PdError) as e:
            t.run(inp.q, bad, out, 5)
        assert e.value.code == pd.PD_ERR_INVALID
        assert "source %d" % (len(bad) - 1) in pd.last_error()
        torch.cuda.synchronize()
        assert bool(torch.all(out == 3.0))
        with pytest.raises(pd.PdError) as e:
            t.run(inp.q, good, out, 6)                        # above max_seqs
        assert e.value.code == pd.PD_ERR_CAPACITY
        # no source: begin then finalize, every output 0
        t.run(inp.q, [], out, 5)
        torch.cuda.synchronize()
        assert bool(torch.all(out == 0))
    finally:
        t.close()


def test_fused_tiled_run_on_a_fresh_handle_is_capturable(cuda_device):
    """pd_tiled_create allocates the fused run's partials with the state, so the
    first pd_tiled_run on a handle allocates nothing and can be the first call
    inside a CUDA graph capture; the replay equals the calls made one by one
    on another handle."""
    mw = W.tiled_mixed(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=64, tile_capacity=8,
                       max_blocks=16, seed=58)
    inp = api.MixedTiledInputs(mw, cuda_device)
    ref_t = pd.Tiled(3, 8, 2, 64, 16, 8)
    t = None
    try:
        # the calls one by one on one handle (this also loads the kernels)
        ref = torch.empty((3, 8, 64), dtype=torch.bfloat16, device=cuda_device)
        ref_t.begin(3)
        for k, v, tb, tc, st, lb in inp.sources(ref_t):
            ref_t.step(inp.q, k, v, tb, tc, 3, st, lb)
        ref_t.finalize(ref, 3)
        torch.cuda.synchronize()
        # a fresh handle whose first call is the captured run
        t = pd.Tiled(3, 8, 2, 64, 16, 8)
        out = torch.full((3, 8, 64), 7.0, dtype=torch.bfloat16, device=cuda_device)
        srcs = inp.sources(t)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            t.run(inp.q, srcs, out, 3)
        g.replay()
        torch.cuda.synchronize()
        assert pd.pd_device_status() == 0
        assert np.array_equal(api.bf16_bits(out), api.bf16_bits(ref))
    finally:
        ref_t.close()
        if t is not None:
            t.close()
