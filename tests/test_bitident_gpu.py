"""Batch invariance on the GPU: a sequence's output bytes do not depend on the
sequences it is batched with, nor on where its blocks live in the cache, under
the Auto and Pinned policies (Module attn_splitk page: the split count moves
only with (sm_count, num_q_heads) and the pin, because the split merge is not
associative).  The bitwise A/B comparison follows the microtest idea of the
prefill_attn_fa128.rs page (0 differing values)."""

import numpy as np
import pytest
import torch

from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _sub_batch(w, order, relocate_seed=None):
    """A new paged workload holding the sequences `order` of w (in that order), with
    their blocks copied into a fresh cache, optionally at shuffled physical positions."""
    bs = w.block_size
    need = [-(-int(w.context_lens[s]) // bs) for s in order]
    total = max(1, sum(need))
    nb = total + 3
    pos = np.arange(nb)
    if relocate_seed is not None:
        pos = np.random.default_rng(relocate_seed).permutation(nb)
    k = np.zeros((nb,) + w.k_cache.shape[1:], dtype=np.uint16)
    v = np.zeros_like(k)
    bt = np.zeros((len(order), max(1, max(need))), dtype=np.int32)
    off = 0
    for i, s in enumerate(order):
        for j in range(need[i]):
            src = int(w.block_table[s, j])
            dst = int(pos[off])
            k[dst] = w.k_cache[src]
            v[dst] = w.v_cache[src]
            bt[i, j] = dst
            off += 1
    return W.PagedWorkload(name="sub", num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                           head_dim=w.head_dim, block_size=bs, q=w.q[list(order)], k_cache=k,
                           v_cache=v, block_table=bt, context_lens=w.context_lens[list(order)],
                           inv_sqrt_d=w.inv_sqrt_d, policy=w.policy, pin=w.pin,
                           sm_count=w.sm_count, gqa_pack=w.gqa_pack)


def _bits(w, device, n, pack=False):
    inp = api.PagedInputs(w, device)
    out = api.run_paged(inp, num_splits=n, gqa_pack=pack)
    torch.cuda.synchronize()
    return api.bf16_bits(out)


@pytest.fixture(scope="module")
def large():
    return W.large_batch()


def _probes(w):
    lens = w.context_lens
    return [int(np.argmax(lens)), int(np.argmin(lens)), int(np.argsort(lens)[len(lens) // 2])]


@pytest.mark.parametrize("policy,pin", [("auto", 0), ("pinned", 3), ("pinned", 1)])
def test_large_batch_probe_sequences_are_batch_invariant(cuda_device, large, policy, pin):
    w = large
    probes = _probes(w)
    # the split count of every batch below is the same under Auto / Pinned
    counts = {pd.pd_num_splits(policy, pin, 148, w.num_q_heads, b, 0) for b in (1, 17, 256)}
    assert len(counts) == 1
    n = counts.pop()
    full = _bits(w, cuda_device, n)
    rng = np.random.default_rng(11)
    others = [s for s in range(w.num_seqs) if s not in probes]
    for p_i, s in enumerate(probes):
        alone = _bits(_sub_batch(w, [s], relocate_seed=3 + p_i), cuda_device, n)
        assert np.array_equal(alone[0], full[s]), f"probe {s} alone vs full batch"
        mates = list(rng.choice(others, 16, replace=False))
        order = mates[:p_i * 5] + [s] + mates[p_i * 5:]
        mid = _bits(_sub_batch(w, order, relocate_seed=17 + p_i), cuda_device, n)
        assert np.array_equal(mid[order.index(s)], full[s]), f"probe {s} in a batch of 17"


def test_legacy_split_count_moves_with_the_batch(large):
    """Negative control: Legacy reads the batch, so its split count (and with it a
    sequence's rounding) changes between batch sizes."""
    counts = [pd.pd_num_splits("legacy", 0, 148, 32, b, 0) for b in (1, 2, 4)]
    assert len(set(counts)) > 1


def test_packed_pass_is_batch_invariant(cuda_device):
    w = W.gqa_packed()
    full = _bits(w, cuda_device, 1, pack=True)
    for s in (0, 7, 31):
        alone = _bits(_sub_batch(w, [s], relocate_seed=s), cuda_device, 1, pack=True)
        assert np.array_equal(alone[0], full[s])


def test_long_context_alone_vs_with_others(cuda_device):
    w = W.long_context()
    n = pd.pd_num_splits("auto", 0, 148, w.num_q_heads, 1, 0)
    alone = _bits(w, cuda_device, n)
    extra = W.custom([100, 5000, 32768], 24, 8, 128, seed=41)
    both = W.PagedWorkload(
        name="mix", num_q_heads=24, num_kv_heads=8, head_dim=128, block_size=16,
        q=np.concatenate([extra.q[:2], w.q]), k_cache=np.concatenate([extra.k_cache, w.k_cache]),
        v_cache=np.concatenate([extra.v_cache, w.v_cache]),
        block_table=np.concatenate([
            np.pad(extra.block_table[:2], ((0, 0), (0, w.block_table.shape[1] - extra.block_table.shape[1]))),
            w.block_table + extra.num_blocks]).astype(np.int32),
        context_lens=np.concatenate([extra.context_lens[:2], w.context_lens]).astype(np.int32),
        inv_sqrt_d=w.inv_sqrt_d)
    mixed = _bits(both, cuda_device, n)
    assert np.array_equal(mixed[2], alone[0])


def test_repeat_launches_are_bitwise_stable(cuda_device):
    w = W.custom([3000, 20, 700], 32, 8, 128, seed=42)
    a = _bits(w, cuda_device, 10)
    b = _bits(w, cuda_device, 10)
    assert np.array_equal(a, b)


def test_tiled_sequence_is_batch_invariant(cuda_device):
    tw = W.tiled(num_seqs=12, max_blocks=200, seed=9)
    full = api.bf16_bits(api.run_tiled(api.TiledInputs(tw, cuda_device)))
    s = int(np.argmax(tw.blocks_per_seq))
    one = W.TiledWorkload(name="one", num_q_heads=tw.num_q_heads, num_kv_heads=tw.num_kv_heads,
                          head_dim=tw.head_dim, block_size=tw.block_size,
                          tile_capacity=tw.tile_capacity, q=tw.q[[s]], pool=tw.pool,
                          layout=tw.layout, tile_blocks=tw.tile_blocks[:, [s]],
                          tile_block_counts=tw.tile_block_counts[:, [s]],
                          last_block_valid_slots=tw.last_block_valid_slots,
                          blocks_per_seq=tw.blocks_per_seq[[s]])
    alone = api.bf16_bits(api.run_tiled(api.TiledInputs(one, cuda_device)))
    assert np.array_equal(alone[0], full[s])


@pytest.mark.parametrize("kind", ["splitk", "packed", "tiled"])
def test_part_layout_does_not_change_bits(cuda_device, kind):
    """A unit's range is cut into parts by its own length and the parts fold in a
    fixed order; whether they run in one CTA or one per CTA of a cluster (the
    launch picks from occupancy, so from the batch) must not change a bit."""
    outs = []
    try:
        for layout in (1, 2):
            pd.pd_debug_set_tuning(0, layout, -1)
            if kind == "tiled":
                tw = W.tiled(num_seqs=8, max_blocks=256, seed=3)
                outs.append(api.bf16_bits(api.run_tiled(api.TiledInputs(tw, cuda_device))))
            elif kind == "packed":
                w = W.custom([4096, 700, 33, 2500], 16, 2, 256, seed=72)
                outs.append(_bits(w, cuda_device, 1, pack=True))
            else:
                w = W.custom([5000, 3000, 17, 2600], 24, 8, 128, seed=71)
                outs.append(_bits(w, cuda_device, 3))
    finally:
        pd.pd_debug_set_tuning(0, 0, -1)
    assert np.array_equal(outs[0], outs[1])


def test_ring_depth_does_not_change_bits(cuda_device):
    """The ring depth per warp is a launch choice (a launch of several waves of
    one-CTA units takes a deeper ring than a single-wave one): the per-warp
    tile order and every fold are the same, so no bit may change."""
    lens = [int(x) for x in np.random.default_rng(5).integers(200, 2000, size=160)]
    w = W.custom(lens, 32, 8, 128, seed=75)   # 160 x 8 x 10 units: several waves
    outs = []
    try:
        for tun in ((0, 0, -1), (1, 1, -1), (2, 1, -1), (3, 1, -1)):
            pd.pd_debug_set_tuning(*tun)
            outs.append(_bits(w, cuda_device, 10))
    finally:
        pd.pd_debug_set_tuning(0, 0, -1)
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_tiled_run_equals_separate_calls(cuda_device):
    """pd_tiled_run is begin, the steps in order and finalize: same bits as the
    calls made one by one."""
    mw = W.tiled_mixed(num_seqs=10, max_blocks=120, seed=8)
    inp = api.MixedTiledInputs(mw, cuda_device)
    t = pd.Tiled(mw.num_seqs, mw.num_q_heads, mw.num_kv_heads, mw.head_dim, mw.block_size,
                 mw.tile_capacity)
    try:
        a = api.bf16_bits(api.run_tiled_mixed(inp, t))
        out = torch.empty((mw.num_seqs, mw.num_q_heads, mw.head_dim), dtype=torch.bfloat16,
                          device=cuda_device)
        t.begin(mw.num_seqs)
        for k, v, tb, tc, st, lb in inp.sources(t):
            t.step(inp.q, k, v, tb, tc, mw.num_seqs, st, lb)
        t.finalize(out, mw.num_seqs)
        torch.cuda.synchronize()
        assert np.array_equal(a, api.bf16_bits(out))
    finally:
        t.close()


def test_packed_with_splits_is_batch_invariant(cuda_device):
    """gqa_pack mode 2 at 16 splits: a sequence's bits alone == in the batch; and
    mode 2 at one split is the packed pass itself (same bits as mode 1)."""
    w = W.gqa_packed_splitk()
    full = _bits(w, cuda_device, 16, pack=2)
    for s in (0, 9, 31):
        alone = _bits(_sub_batch(w, [s], relocate_seed=s + 1), cuda_device, 16, pack=2)
        assert np.array_equal(alone[0], full[s])
    assert np.array_equal(_bits(w, cuda_device, 1, pack=2), _bits(w, cuda_device, 1, pack=1))


def test_packed_long_sequence_with_splits_alone_vs_pair(cuda_device):
    """gqa_pack mode 2 at Auto's 16 splits: each 32768-token sequence of the
    long packed workload gives the same bits alone as next to the other one."""
    w = W.gqa_packed_long_splitk()
    n = api.PagedInputs(w, cuda_device).splits()
    both = _bits(w, cuda_device, n, pack=2)
    for s in range(w.num_seqs):
        alone = _bits(_sub_batch(w, [s], relocate_seed=40 + s), cuda_device, n, pack=2)
        assert np.array_equal(alone[0], both[s])
