"""Pins of the FP64 oracle against things other than itself (CPU only).

* a library routine: torch's scaled_dot_product_attention in float64, on the
  special case where the paged cache is a plain reshape of contiguous K/V;
* high-precision brute force (mpmath, 50 digits) on tiny inputs;
* closed forms: one token, q = 0, constant V, a dominant key, huge scores;
* invariants: relocating physical blocks, identical q rows, split count;
* the l = 0 -> 0 rule;
* mutation checks: mistakes planted in a copy of the oracle's C source (a
  wrong GQA map, a sign error, swapped K/V, a dropped max shift, a wrong
  stride) must each fail one of these pins.
"""

import math
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import policy
from paged_kv_decode_splitk_gb300 import workloads as W

torch = pytest.importorskip("torch")


def _contiguous_workload(lens, Hq, Hkv, D, bs, seed):
    """Paged cache whose block table is the identity over consecutive blocks, so each
    sequence's K/V are contiguous rows of k_cache.reshape(-1, Hkv, D)."""
    lens = list(lens)
    need = [-(-L // bs) for L in lens]
    nb = max(1, sum(need))
    q = W.normal_bf16((len(lens), Hq, D), seed)
    k = W.normal_bf16((nb, bs, Hkv, D), seed + 1)
    v = W.normal_bf16((nb, bs, Hkv, D), seed + 2)
    bt = np.zeros((len(lens), max(1, max(need))), dtype=np.int32)
    starts, off = [], 0
    for s, n in enumerate(need):
        bt[s, :n] = np.arange(off, off + n)
        starts.append(off * bs)
        off += n
    return q, k, v, bt, np.array(lens, dtype=np.int32), starts


def _sdpa_reference(q, k, v, lens, starts, Hq, Hkv, D, bs, scale):
    """torch SDPA (float64) over contiguous K/V rows; GQA by repeat_interleave."""
    G = Hq // Hkv
    kf = torch.from_numpy(W.bf16_to_f32(k).astype(np.float64)).reshape(-1, Hkv, D)
    vf = torch.from_numpy(W.bf16_to_f32(v).astype(np.float64)).reshape(-1, Hkv, D)
    qf = torch.from_numpy(W.bf16_to_f32(q).astype(np.float64))
    out = np.zeros((len(lens), Hq, D))
    for s, L in enumerate(lens):
        if L == 0:
            continue
        ks = kf[starts[s]:starts[s] + L].permute(1, 0, 2).repeat_interleave(G, dim=0)
        vs = vf[starts[s]:starts[s] + L].permute(1, 0, 2).repeat_interleave(G, dim=0)
        qs = qf[s].unsqueeze(1)  # [Hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(
            qs.unsqueeze(0), ks.unsqueeze(0), vs.unsqueeze(0), scale=scale)
        out[s] = o[0, :, 0, :].numpy()
    return out


SDPA_CASES = [
    # lens, Hq, Hkv, D, bs
    ([37, 100], 4, 1, 64, 16),
    ([1, 2, 15, 16, 17, 70], 8, 2, 32, 16),
    ([5, 33, 64], 6, 3, 16, 4),
    ([40, 9], 3, 3, 8, 8),
    ([130], 16, 2, 24, 32),
]


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs", SDPA_CASES)
def test_matches_torch_sdpa_float64(lens, Hq, Hkv, D, bs):
    q, k, v, bt, cl, starts = _contiguous_workload(lens, Hq, Hkv, D, bs, seed=7)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    got = oracle.decode_attn(q, k, v, bt, cl, scale)
    want = _sdpa_reference(q, k, v, lens, starts, Hq, Hkv, D, bs, scale)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def _mp_attention(qrow, krows, vrows, scale):
    import mpmath
    mpmath.mp.dps = 50
    qf = [mpmath.mpf(float(x)) for x in W.bf16_to_f32(qrow)]
    xs = []
    for kr in krows:
        kf = W.bf16_to_f32(kr)
        xs.append(mpmath.mpf(scale) * mpmath.fsum(qf[d] * mpmath.mpf(float(kf[d]))
                                                  for d in range(len(qf))))
    ws = [mpmath.e ** x for x in xs]
    den = mpmath.fsum(ws)
    out = []
    for d in range(len(qf)):
        out.append(mpmath.fsum(ws[t] * mpmath.mpf(float(W.bf16_to_f32(vrows[t])[d]))
                               for t in range(len(ws))) / den)
    return [float(x) for x in out]


def test_brute_force_mpmath_tiny():
    w = W.custom([13, 40], 4, 2, 8, block_size=4, seed=3, pool_factor=1.5)
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.5)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        for h in range(w.num_q_heads):
            kvh = h // G
            krows, vrows = [], []
            for t in range(L):
                blk = int(w.block_table[s, t // w.block_size])
                krows.append(w.k_cache[blk, t % w.block_size, kvh])
                vrows.append(w.v_cache[blk, t % w.block_size, kvh])
            want = _mp_attention(w.q[s, h], krows, vrows, 0.5)
            np.testing.assert_allclose(got[s, h], want, rtol=0, atol=1e-12)


def test_single_token_returns_its_value_row():
    w = W.custom([1, 1, 1], 4, 2, 32, seed=11)
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.17)
    for s in range(3):
        blk = int(w.block_table[s, 0])
        for h in range(4):
            want = W.bf16_to_f32(w.v_cache[blk, 0, h // 2]).astype(np.float64)
            assert np.array_equal(got[s, h], want)


def test_zero_query_gives_mean_of_values():
    w = W.custom([37, 100], 4, 1, 64, seed=12)
    w.q[:] = 0
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.125)
    for s, L in enumerate(w.context_lens):
        rows = [W.bf16_to_f32(w.v_cache[w.block_table[s, t // 16], t % 16, 0]) for t in range(L)]
        mean = np.array([math.fsum(float(r[d]) for r in rows) / L for d in range(64)])
        for h in range(4):
            np.testing.assert_allclose(got[s, h], mean, rtol=0, atol=1e-14)


def test_constant_value_rows_give_that_constant():
    w = W.custom([50, 3], 8, 2, 16, seed=13)
    c = W.bf16_bits(np.float32(-1.375))
    w.v_cache[:] = c
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.25)
    np.testing.assert_allclose(got, -1.375, rtol=0, atol=1e-15)


@pytest.mark.parametrize("margin", [60.0, 4000.0])
def test_dominant_key_selects_its_value(margin):
    """One key scores `margin` above every other: the output is that key's V (exp(-60) is
    below 1e-26); at a 4000 margin a softmax without the max shift overflows."""
    w = W.custom([48], 2, 1, 16, seed=14)
    w.q[:] = 0
    w.k_cache[:] = 0
    one = W.bf16_bits(np.float32(1.0))
    w.q[0, :, 0] = one
    blk, row = int(w.block_table[0, 1]), 5  # token 21
    w.k_cache[blk, row, 0, 0] = W.bf16_bits(np.float32(margin))
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 1.0)
    want = W.bf16_to_f32(w.v_cache[blk, row, 0]).astype(np.float64)
    for h in range(2):
        assert np.all(np.isfinite(got[0, h]))
        np.testing.assert_allclose(got[0, h], want, rtol=0, atol=1e-20 + 1e-15 * (margin < 100))


def test_empty_sequence_is_exactly_zero():
    w = W.custom([0, 20, 0], 4, 1, 32, seed=15)
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.2)
    assert np.all(got[0] == 0.0) and np.all(got[2] == 0.0)
    assert np.any(got[1] != 0.0)


def test_block_relocation_is_invisible():
    """Moving physical blocks and rewriting the table leaves every output bit unchanged."""
    w = W.custom([37, 100, 64], 8, 2, 32, seed=16, pool_factor=2.0)
    base = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.3)
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt2 = perm[w.block_table].astype(np.int32)
    moved = oracle.decode_attn(w.q, k2, v2, bt2, w.context_lens, 0.3)
    assert np.array_equal(base, moved)


def test_identical_query_rows_in_a_group_agree():
    w = W.custom([77], 8, 2, 32, seed=17)
    w.q[0, 1:4] = w.q[0, 0]
    got = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.3)
    for h in (1, 2, 3):
        assert np.array_equal(got[0, h], got[0, 0])
    assert not np.array_equal(got[0, 4], got[0, 0])


@pytest.mark.parametrize("min_kv", [16, 256])
def test_split_replay_matches_direct_for_every_split_count(min_kv):
    w = W.custom([1, 15, 16, 17, 300, 1000, 4100], 6, 2, 32, seed=18)
    direct = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.2)
    for n in range(1, policy.MAX_DECODE_SPLITS + 1):
        chunks = [policy.split_chunk_tokens(int(L), n, 16, min_kv) for L in w.context_lens]
        rep = oracle.split_replay(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.2,
                                  chunks)
        np.testing.assert_allclose(rep, direct, rtol=0, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 7, 16, 5000])
def test_split_replay_odd_chunks(chunk):
    w = W.custom([0, 33, 257], 4, 4, 16, seed=19)
    direct = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.4)
    rep = oracle.split_replay(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 0.4, chunk)
    np.testing.assert_allclose(rep, direct, rtol=0, atol=1e-12)
    assert np.all(rep[0] == 0)


def _tiles_cover_whole_sequences(w, tcap, calls):
    """A tile plan that walks every sequence of a paged workload front to back."""
    S = w.num_seqs
    bs = w.block_size
    tb = np.zeros((calls, S, tcap), dtype=np.int32)
    tc = np.zeros((calls, S), dtype=np.int32)
    for s in range(S):
        n = -(-int(w.context_lens[s]) // bs)
        for c in range(calls):
            ids = w.block_table[s, c * tcap:min(n, (c + 1) * tcap)]
            tc[c, s] = len(ids)
            tb[c, s, :len(ids)] = ids
        assert n <= calls * tcap
    return tb, tc


def test_tiled_full_blocks_equals_paged():
    """Whole blocks through the tiled interface == the paged definition (D=256 -> scale 1/16)."""
    lens = [32, 160, 0, 48]
    w = W.custom(lens, 8, 2, 256, seed=20)
    tb, tc = _tiles_cover_whole_sequences(w, tcap=4, calls=3)
    lb = np.full(3, 16, dtype=np.int32)
    got = oracle.tiled_attn(w.q, w.k_cache, w.v_cache, tb, tc, lb, 2, 16,
                            oracle.paged_strides(2, 256, 16))
    want = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, 1 / 16)
    assert np.array_equal(got, want)


def test_tiled_last_block_valid_slots_truncates():
    """The last block of each tile in a call holds last_block_valid_slots tokens."""
    w = W.custom([64, 64], 4, 1, 64, seed=21)
    tb = w.block_table[None, :, :4].copy()
    tc = np.array([[4, 2]], dtype=np.int32)
    got = oracle.tiled_attn(w.q, w.k_cache, w.v_cache, tb, tc, np.array([5], np.int32), 1, 16,
                            oracle.paged_strides(1, 64, 16))
    scale = float(np.float32(1 / 8))
    want = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table,
                              np.array([3 * 16 + 5, 16 + 5], np.int32), scale)
    assert np.array_equal(got, want)
    # full-block codes: 0, 16 and -1 all mean a full block
    for code in (0, 16, -1):
        full = oracle.tiled_attn(w.q, w.k_cache, w.v_cache, tb, tc, np.array([code], np.int32),
                                 1, 16, oracle.paged_strides(1, 64, 16))
        want_full = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table,
                                       np.array([64, 32], np.int32), scale)
        assert np.array_equal(full, want_full)


def test_scratch_pool_and_paged_layouts_agree():
    """The same blocks stored in the paged layout and in the scratch-pool layout give
    bit-identical results through their own strides."""
    tw = W.tiled(num_seqs=6, num_q_heads=8, num_kv_heads=2, head_dim=32, tile_capacity=8,
                 num_calls=3, max_blocks=20, seed=22)
    kflat, vflat = W.scratch_pool_views(tw.pool)
    got_scratch = oracle.tiled_attn(tw.q, kflat, vflat, tw.tile_blocks, tw.tile_block_counts,
                                    tw.last_block_valid_slots, 2, 16,
                                    oracle.scratch_pool_strides(2, 32, 16))
    # rebuild a paged cache [slots, bs, Hkv, D] holding the same rows
    kp = np.ascontiguousarray(tw.pool[:, 0].transpose(0, 2, 1, 3))
    vp = np.ascontiguousarray(tw.pool[:, 1].transpose(0, 2, 1, 3))
    got_paged = oracle.tiled_attn(tw.q, kp, vp, tw.tile_blocks, tw.tile_block_counts,
                                  tw.last_block_valid_slots, 2, 16,
                                  oracle.paged_strides(2, 32, 16))
    assert np.array_equal(got_scratch, got_paged)
    zero_seqs = np.where(tw.blocks_per_seq == 0)[0]
    assert len(zero_seqs) >= 2
    assert np.all(got_scratch[zero_seqs] == 0)


def _mixed_small(seed=23):
    return W.tiled_mixed(num_seqs=7, num_q_heads=8, num_kv_heads=2, head_dim=32, tile_capacity=4,
                         max_blocks=18, seed=seed)


def _mixed_calls(mw):
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
    return calls


def test_tiled_multi_source_matches_torch_sdpa_float64():
    """One step mixing the paged cache and the scratch pool: the token rows are
    gathered here by plain array indexing of each layout (no strides), and torch's
    float64 SDPA over them must agree with the oracle."""
    mw = _mixed_small()
    S, Hq, D = mw.q.shape
    Hkv, bs = mw.num_kv_heads, mw.block_size
    G = Hq // Hkv
    want = np.zeros((S, Hq, D))
    scale = float(np.float32(1 / math.sqrt(D)))
    for s in range(S):
        for kvh in range(Hkv):
            ks, vs = [], []
            for kind, tb, tc, lb in mw.calls:
                cnt = int(tc[s])
                for i in range(cnt):
                    blk = int(tb[s, i])
                    ntok = lb if (i == cnt - 1 and 1 <= lb < bs) else bs
                    for t in range(ntok):
                        if kind == "paged":
                            ks.append(mw.paged_k[blk, t, kvh]); vs.append(mw.paged_v[blk, t, kvh])
                        else:
                            ks.append(mw.scratch[blk, 0, kvh, t]); vs.append(mw.scratch[blk, 1, kvh, t])
            if not ks:
                continue
            kt = torch.from_numpy(W.bf16_to_f32(np.stack(ks)).astype(np.float64))
            vt = torch.from_numpy(W.bf16_to_f32(np.stack(vs)).astype(np.float64))
            qt = torch.from_numpy(W.bf16_to_f32(mw.q[s, kvh * G:(kvh + 1) * G]).astype(np.float64))
            o = torch.nn.functional.scaled_dot_product_attention(
                qt[None, :, None, :], kt[None, None].expand(1, G, -1, -1),
                vt[None, None].expand(1, G, -1, -1), scale=scale)
            want[s, kvh * G:(kvh + 1) * G] = o[0, :, 0, :].numpy()
    got = oracle.tiled_attn_multi(mw.q, _mixed_calls(mw), Hkv, bs)
    assert np.max(np.abs(got - want)) < 1e-12
    zero = np.where(mw.blocks_per_seq == 0)[0]
    assert len(zero) >= 1 and np.all(got[zero] == 0)
    assert sum(1 for c in mw.calls if c[0] == "paged") >= 1
    assert sum(1 for c in mw.calls if c[0] == "scratch") >= 1


def test_tiled_multi_with_one_source_equals_tiled():
    """Every call naming the same pool and strides is the single-source step."""
    tw = W.tiled(num_seqs=6, num_q_heads=8, num_kv_heads=2, head_dim=32, tile_capacity=8,
                 num_calls=3, max_blocks=20, seed=24)
    kflat, vflat = W.scratch_pool_views(tw.pool)
    st = oracle.scratch_pool_strides(2, 32, 16)
    calls = [dict(k_pool=kflat, v_pool=vflat, tile_blocks=tw.tile_blocks[c],
                  tile_block_counts=tw.tile_block_counts[c],
                  last_block_valid_slots=int(tw.last_block_valid_slots[c]), strides=st)
             for c in range(tw.num_calls)]
    got = oracle.tiled_attn_multi(tw.q, calls, 2, 16)
    want = oracle.tiled_attn(tw.q, kflat, vflat, tw.tile_blocks, tw.tile_block_counts,
                             tw.last_block_valid_slots, 2, 16, st)
    assert np.array_equal(got, want)


def test_e4m3_decoding_matches_torch_float8():
    """Every FP8 E4M3 code against torch's float8_e4m3fn (a library routine)."""
    got = oracle.e4m3_values()
    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert int(np.isnan(got).sum()) == 2 and np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9


def _fp8_contiguous(lens, Hq, Hkv, D, seed, ks, vs):
    q, k, v, bt, cl, starts = _contiguous_workload(lens, Hq, Hkv, D, 16, seed)
    rng = np.random.default_rng(seed)
    k8 = W.e4m3_codes(rng.standard_normal(k.shape).astype(np.float32) / np.float32(ks))
    v8 = W.e4m3_codes(rng.standard_normal(v.shape).astype(np.float32) / np.float32(vs))
    return q, k8, v8, bt, cl, starts


@pytest.mark.parametrize("ks,vs", [(0.5, 0.25), (0.37, 1.7)])
def test_fp8_attention_matches_torch_sdpa_float64(ks, vs):
    """FP8 cache: torch float8 decode times the scale, then torch SDPA in float64."""
    lens, Hq, Hkv, D = [1, 15, 16, 17, 70], 8, 2, 32
    q, k8, v8, bt, cl, starts = _fp8_contiguous(lens, Hq, Hkv, D, 61, ks, vs)
    f8 = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)
    kf = (f8(k8) * float(np.float32(ks))).reshape(-1, Hkv, D)
    vf = (f8(v8) * float(np.float32(vs))).reshape(-1, Hkv, D)
    qf = torch.from_numpy(W.bf16_to_f32(q).astype(np.float64))
    scale = float(np.float32(1 / math.sqrt(D)))
    G = Hq // Hkv
    want = np.zeros((len(lens), Hq, D))
    for s, L in enumerate(lens):
        kk = kf[starts[s]:starts[s] + L].permute(1, 0, 2).repeat_interleave(G, dim=0)
        vv = vf[starts[s]:starts[s] + L].permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qf[s].unsqueeze(1)[None], kk[None], vv[None],
                                                             scale=scale)
        want[s] = o[0, :, 0, :].numpy()
    got = oracle.decode_attn_fp8(q, k8, v8, ks, vs, bt, cl, scale)
    assert np.max(np.abs(got - want)) < 1e-12


def test_fp8_equals_bf16_definition_on_exact_values():
    """With power-of-two scales every dequantised value is a BF16 value: the FP8
    oracle must equal the BF16 oracle on those values, bit for bit."""
    w = W.custom([0, 5, 33, 160], 8, 2, 64, seed=62)
    w8 = W.fp8_variant(w, k_scale=0.5, v_scale=4.0, seed=3)
    val = oracle.e4m3_values()
    kb = W.bf16_bits((val[w8.k_cache] * 0.5).astype(np.float32))
    vb = W.bf16_bits((val[w8.v_cache] * 4.0).astype(np.float32))
    assert np.array_equal(W.bf16_to_f32(kb).astype(np.float64), val[w8.k_cache] * 0.5)
    got = oracle.decode_attn_fp8(w8.q, w8.k_cache, w8.v_cache, 0.5, 4.0, w8.block_table, w8.context_lens,
                                 w8.inv_sqrt_d)
    want = oracle.decode_attn(w8.q, kb, vb, w8.block_table, w8.context_lens, w8.inv_sqrt_d)
    assert np.array_equal(got, want)
    assert np.all(got[0] == 0.0)


def test_fp8_scales_fold_into_the_softmax_scale_and_the_output():
    """K scale a with softmax scale b == K scale 1 with scale a*b; V scale c scales
    the output by c (closed forms of the definition)."""
    w8 = W.fp8_variant(W.custom([40, 77], 8, 2, 64, seed=63), seed=4)
    base = oracle.decode_attn_fp8(w8.q, w8.k_cache, w8.v_cache, 1.0, 1.0, w8.block_table, w8.context_lens,
                                  0.125)
    a = oracle.decode_attn_fp8(w8.q, w8.k_cache, w8.v_cache, 2.0, 1.0, w8.block_table, w8.context_lens,
                               0.0625)
    assert np.array_equal(a, base)
    c = oracle.decode_attn_fp8(w8.q, w8.k_cache, w8.v_cache, 1.0, 3.0, w8.block_table, w8.context_lens,
                               0.125)
    assert np.max(np.abs(c - 3.0 * base)) < 1e-13


def test_tolerance_helper():
    assert oracle.bf16_ulp(1.0) == 2.0 ** -7
    assert oracle.bf16_ulp(1.99) == 2.0 ** -7
    assert oracle.bf16_ulp(-0.75) == 2.0 ** -8
    assert oracle.bf16_ulp(0.0) == 0.0
    assert oracle.tolerance(0.0) == 1e-3


def test_bf16_rounding_is_nearest_even():
    xs = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3], dtype=np.float32)
    bits = W.bf16_bits(xs)
    back = W.bf16_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                 # tie -> even
    assert back[2] == 1.0 + 2 ** -6       # tie -> even (up)
    assert back[3] == -2.5
    assert abs(back[4] - 1e-3) <= 2 ** -17


# ---------------------------------------------------------------------------
# Mutation checks: each planted mistake must be caught by a pin above.
# ---------------------------------------------------------------------------

MUTATIONS = {
    "gqa_map_modulo": ("int kvh = h / G;", "int kvh = h % num_kv_heads;"),
    "exp_sign": ("double w = exp(x[t] - xmax);", "double w = exp(xmax - x[t]);"),
    "swap_k_v": ("krows[t] = k_cache + row;\n        vrows[t] = v_cache + row;",
                 "krows[t] = v_cache + row;\n        vrows[t] = k_cache + row;"),
    "no_max_shift": ("double w = exp(x[t] - xmax);", "double w = exp(x[t]);"),
    "token_stride": ("int64_t row = ((blk * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;",
                     "int64_t row = ((blk * block_size + t % block_size) + kvh) * head_dim;"),
    "split_merge_weight": ("double w = exp(m - M);", "double w = exp(M - m);"),
    "multi_source_tok_stride": ("(int64_t)t * strides[3 * c + 1] +", "(int64_t)t * strides[3 * c + 2] +"),
    "e4m3_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "fp8_v_scale": ("vr[t * head_dim + d] = orc_e4m3_value(v_cache[row + d]) * vs;",
                    "vr[t * head_dim + d] = orc_e4m3_value(v_cache[row + d]) * ks;"),
}


def _mutant_lib(name, tmpdir):
    import ctypes
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pd_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, name
    path = os.path.join(tmpdir, f"{name}.c")
    open(path, "w").write(src.replace(old, new))
    so = os.path.join(tmpdir, f"{name}.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True)
    return ctypes.CDLL(so)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    # scratch beside the oracle's own build (an ignored build folder of the repository)
    scratch = os.path.join(os.path.dirname(oracle.__file__), "_build")
    os.makedirs(scratch, exist_ok=True)
    tmp = tempfile.mkdtemp(dir=scratch)
    try:
        lib = _mutant_lib(name, tmp)
        real = oracle._load()
        for f in ("orc_decode_attn", "orc_split_replay", "orc_tiled_attn", "orc_tiled_attn_multi",
                  "orc_decode_attn_fp8", "orc_e4m3_value"):
            getattr(lib, f).argtypes = getattr(real, f).argtypes
            getattr(lib, f).restype = getattr(real, f).restype
        monkeypatch.setattr(oracle, "_lib", lib)
        pins = [
            lambda: test_matches_torch_sdpa_float64(*SDPA_CASES[1]),
            lambda: test_dominant_key_selects_its_value(4000.0),
            lambda: test_split_replay_matches_direct_for_every_split_count(16),
            lambda: test_tiled_multi_source_matches_torch_sdpa_float64(),
            lambda: test_e4m3_decoding_matches_torch_float8(),
            lambda: test_fp8_attention_matches_torch_sdpa_float64(0.37, 1.7),
        ]
        failed = 0
        for pin in pins:
            try:
                with np.errstate(all="ignore"):
                    pin()
            except (AssertionError, ValueError):
                failed += 1
        assert failed >= 1, f"mutation {name} survived every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_mutation_list_targets_real_source_lines():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pd_oracle.c")).read()
    for name, (old, _) in MUTATIONS.items():
        assert src.count(old) >= 1, name
    assert re.search(r"kvh = h / G", src)
