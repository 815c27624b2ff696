"""GPU stress cases: scores far from N(0,1) and calls running on several
streams at once.

Peaked softmax: q is scaled up so the scores of a sequence spread over
hundreds of units (the largest weight dwarfs the rest and most weights
underflow to 0 in FP32).  The running max, the rescale factors that
underflow, the fold of parts whose maxima differ widely and the merge of
splits are all exercised; the oracle's FP64 definition is the reference.
Flat softmax: q = 0 makes every score 0, so every output row is the
arithmetic mean of the sequence's V rows.

Concurrency: a packed pass, a split-K pass with its merge and a fused tiled
run launched on three streams without ordering between them give the bits
each gives alone (the library's shared state - tensor-map cache, status
word - is not disturbed by calls in flight on other streams)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

from helpers import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _scaled_q(w, factor):
    w.q = W.bf16_bits(W.bf16_to_f32(w.q) * np.float32(factor))
    return w


def _check(w, device, num_splits, gqa_pack, what):
    ref = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.inv_sqrt_d)
    inp = api.PagedInputs(w, device)
    out = api.run_paged(inp, num_splits=num_splits, gqa_pack=gqa_pack)
    assert out is not None
    assert pd.pd_device_status() == 0
    got = api.bf16_to_f64(out)
    assert_within_tolerance(got, ref, what)
    return got, ref


PEAKED = [
    # lens, Hq, Hkv, D, N, pack (0 off, 1 packed non-split, 2 packed split-K)
    ([1, 40, 700, 3000], 8, 2, 128, 1, 0),
    ([1, 40, 700, 3000], 8, 2, 128, 7, 0),
    ([5, 513, 2600], 4, 4, 64, 3, 0),
    ([33, 1500, 4000], 16, 2, 256, 1, 1),
    ([33, 1500, 4000], 16, 2, 256, 5, 2),
]


@pytest.mark.parametrize("factor", [8.0, 24.0])
@pytest.mark.parametrize("lens,Hq,Hkv,D,N,pack", PEAKED)
def test_peaked_softmax(cuda_device, lens, Hq, Hkv, D, N, pack, factor):
    w = _scaled_q(W.custom(lens, Hq, Hkv, D, seed=41), factor)
    got, ref = _check(w, cuda_device, N, pack, f"peaked x{factor} N={N} pack={pack}")
    # the scores really are spread out: the top weight of a long sequence's
    # rows carries most of the mass, so the output sits near one V row
    assert np.abs(ref).max() > 1.0


@pytest.mark.parametrize("N,pack", [(1, 0), (6, 0), (1, 1), (6, 2)])
def test_flat_softmax_is_the_mean_of_v(cuda_device, N, pack):
    lens = [1, 17, 300, 2049]
    w = W.custom(lens, 16, 2, 256, seed=43)
    w.q = np.zeros_like(w.q)
    got, _ = _check(w, cuda_device, N, pack, f"flat N={N} pack={pack}")
    G, bs = 8, w.block_size
    kv = W.bf16_to_f32(w.v_cache).astype(np.float64)
    for s, L in enumerate(lens):
        rows = np.stack([kv[w.block_table[s, t // bs], t % bs] for t in range(L)])  # [L, Hkv, D]
        mean = rows.mean(axis=0)
        for h in range(16):
            assert_within_tolerance(got[s, h][None], mean[h // G][None], f"flat mean s={s} h={h}")


def test_three_streams_at_once_match_solo_runs(cuda_device):
    wp = W.custom([700, 2500, 4096, 90, 1800], 16, 2, 256, seed=51)        # packed pass
    wl = W.custom([30000], 24, 8, 128, seed=52)                            # 13 splits + merge
    tw = W.tiled(num_seqs=12, num_q_heads=8, num_kv_heads=2, head_dim=128, tile_capacity=16,
                 max_blocks=60, seed=53)                                   # fused tiled run
    ip, il, it = api.PagedInputs(wp, cuda_device), api.PagedInputs(wl, cuda_device), api.TiledInputs(tw, cuda_device)
    n_long = 13
    t = pd.Tiled(tw.num_seqs, tw.num_q_heads, tw.num_kv_heads, tw.head_dim, tw.block_size, tw.tile_capacity)
    st = t.scratch_pool_strides() if tw.layout == "scratch" else t.paged_strides()
    srcs = [(it.k_pool, it.v_pool, it.tile_blocks[c], it.tile_counts[c], st, int(tw.last_block_valid_slots[c]))
            for c in range(tw.num_calls)]
    outs = {k: torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=cuda_device)
            for k, w in (("p", wp), ("l", wl), ("t", tw))}
    ws_l = api.workspace(wl.num_seqs, wl.num_q_heads, wl.head_dim, n_long, cuda_device)
    try:
        def launch(which, stream):
            if which == "p":
                assert api.run_paged(ip, num_splits=1, gqa_pack=1, out=outs["p"], stream=stream) is not None
            elif which == "l":
                assert api.run_paged(il, num_splits=n_long, gqa_pack=0, out=outs["l"], ws=ws_l,
                                     stream=stream) is not None
            else:
                assert t.run(it.q, srcs, outs["t"], tw.num_seqs, stream) == pd.PD_OK

        solo = {}
        for k in ("p", "l", "t"):
            launch(k, None)
            torch.cuda.synchronize()
            solo[k] = outs[k].clone()
            outs[k].zero_()
        torch.cuda.synchronize()
        streams = [torch.cuda.Stream(device=cuda_device) for _ in range(3)]
        for rep in range(5):
            for k in outs:
                outs[k].zero_()
            torch.cuda.synchronize()
            for k, s in zip(("l", "p", "t"), streams):
                launch(k, s)
            torch.cuda.synchronize()
            assert pd.pd_device_status() == 0
            for k in outs:
                assert torch.equal(outs[k].view(torch.int16), solo[k].view(torch.int16)), (rep, k)
    finally:
        torch.cuda.synchronize()
        t.close()


def test_split_launches_with_their_own_workspaces_on_two_streams(cuda_device):
    """Two split launches (partial pass + merge pass each) at once, each with its
    own workspace, on two streams, five times: every output equals the launch
    made alone."""
    wa = W.custom([9000, 300, 2600], 24, 8, 128, seed=54)
    wb = W.custom([5000, 17, 4000, 1200], 16, 4, 128, seed=55)
    ia, ib = api.PagedInputs(wa, cuda_device), api.PagedInputs(wb, cuda_device)
    ws_a = api.workspace(wa.num_seqs, 24, 128, 13, cuda_device)
    ws_b = api.workspace(wb.num_seqs, 16, 128, 7, cuda_device)
    oa = torch.empty((wa.num_seqs, 24, 128), dtype=torch.bfloat16, device=cuda_device)
    ob = torch.empty((wb.num_seqs, 16, 128), dtype=torch.bfloat16, device=cuda_device)

    def launch(stream):
        sa, sb = stream if stream else (None, None)
        assert api.run_paged(ia, num_splits=13, gqa_pack=0, out=oa, ws=ws_a, stream=sa) is not None
        assert api.run_paged(ib, num_splits=7, gqa_pack=0, out=ob, ws=ws_b, stream=sb) is not None

    launch(None)
    torch.cuda.synchronize()
    solo_a, solo_b = oa.clone(), ob.clone()
    streams = (torch.cuda.Stream(device=cuda_device), torch.cuda.Stream(device=cuda_device))
    for rep in range(5):
        oa.zero_()
        ob.zero_()
        torch.cuda.synchronize()
        launch(streams)
        torch.cuda.synchronize()
        assert pd.pd_device_status() == 0
        assert torch.equal(oa.view(torch.int16), solo_a.view(torch.int16)), rep
        assert torch.equal(ob.view(torch.int16), solo_b.view(torch.int16)), rep


def _rising(lens, D, per_tile_log2, qa, seed):
    """Scores that rise with the token index by about per_tile_log2 (base 2)
    per 16-token tile: q is qa on column 0 only, K's column 0 grows with t."""
    w = W.custom(lens, 8, 2, D, seed=seed)
    q = np.zeros((len(lens), 8, D), np.float32)
    q[:, :, 0] = qa
    w.q = W.bf16_bits(q)
    k = W.bf16_to_f32(w.k_cache).copy()
    step = per_tile_log2 / 16 / np.log2(np.e) / w.inv_sqrt_d / qa  # K rise per token
    bs = w.block_size
    for s, L in enumerate(lens):
        for t in range(L):
            k[w.block_table[s, t // bs], t % bs, :, 0] = t * step
    w.k_cache = W.bf16_bits(k)
    return w


@pytest.mark.parametrize("per_tile", [7.9, 8.1, 12.0, 30.0])
@pytest.mark.parametrize("N", [1, 5])
def test_rising_scores(cuda_device, per_tile, N):
    # every tile's maximum passes the previous ones: the kernels' reference
    # max moves at every tile (rise above 8 base-2 units per tile) or every
    # other tile (just below 8), with weights up to 2^8 in between
    w = _rising([40, 700, 3000], 128, per_tile, 1.0, seed=47)
    _check(w, cuda_device, N, 0, f"rising {per_tile}/tile N={N}")


@pytest.mark.parametrize("per_tile", [7.9, 12.0])
def test_rising_scores_fp8(cuda_device, per_tile):
    w = _rising([40, 700, 3000], 128, per_tile, 16.0, seed=48)
    k_scale, v_scale = np.float32(0.5), np.float32(0.25)
    k = W.bf16_to_f32(w.k_cache) / k_scale
    v = W.bf16_to_f32(w.v_cache) / v_scale
    w.k_cache = W.e4m3_codes(np.clip(k, -448, 448))
    w.v_cache = W.e4m3_codes(np.clip(v, -448, 448))
    w.kv_dtype, w.k_scale, w.v_scale = "e4m3", float(k_scale), float(v_scale)
    ref = oracle.decode_attn_fp8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale, w.block_table,
                                 w.context_lens, w.inv_sqrt_d)
    inp = api.PagedInputs(w, cuda_device)
    out = api.run_paged(inp, num_splits=5, gqa_pack=0)
    assert pd.pd_device_status() == 0
    assert_within_tolerance(api.bf16_to_f64(out), ref, f"rising fp8 {per_tile}/tile")
