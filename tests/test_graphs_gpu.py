"""CUDA-graph capture of whole decode steps (the launches carry programmatic
dependent launch edges): a replayed graph gives the same bits as the eager
calls, reads its inputs live (new q written in place shows up in the next
replay), and several steps in one graph chain correctly.  The Module
attn_splitk page resolves the pack switch once so that a captured graph stays
consistent with later launches; these tests exercise capture itself."""

import numpy as np
import pytest
import torch

from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _graph(fn):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()  # warm-up on the capture stream (tensor maps, attributes, buffers)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return g


@pytest.mark.parametrize("kind", ["splitk", "packed", "fp8", "tiled_run"])
def test_graph_replay_matches_eager_and_reads_live_inputs(cuda_device, kind):
    if kind == "tiled_run":
        mw = W.tiled_mixed(num_seqs=6, num_q_heads=8, num_kv_heads=2, head_dim=128, tile_capacity=8,
                           max_blocks=40, seed=41)
        inp = api.MixedTiledInputs(mw, cuda_device)
        t = pd.Tiled(mw.num_seqs, mw.num_q_heads, mw.num_kv_heads, mw.head_dim, mw.block_size, mw.tile_capacity)
        out = torch.empty((mw.num_seqs, mw.num_q_heads, mw.head_dim), dtype=torch.bfloat16, device=cuda_device)
        srcs = inp.sources(t)
        fn = lambda: t.run(inp.q, srcs, out, mw.num_seqs)
        q_host = mw.q
    else:
        base = {"splitk": W.custom([0, 33, 700, 2600], 16, 4, 128, seed=42),
                "packed": W.custom([5, 260, 1500], 16, 2, 256, seed=43),
                "fp8": W.fp8_variant(W.custom([40, 900], 8, 2, 128, seed=44), seed=9)}[kind]
        w = base
        inp = api.PagedInputs(w, cuda_device)
        n, pack = {"splitk": (3, 0), "packed": (1, 1), "fp8": (2, 0)}[kind]
        out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=cuda_device)
        ws = api.workspace(w.num_seqs, w.num_q_heads, w.head_dim, n, cuda_device)
        fn = lambda: api.decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, w.inv_sqrt_d, n,
                                     pack, out, ws, None, w.k_scale, w.v_scale)
        q_host = w.q
    fn()
    torch.cuda.synchronize()
    eager = api.bf16_bits(out)
    g = _graph(fn)
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(api.bf16_bits(out), eager)
    # new q written in place: the replay reads it
    q2 = W.normal_bf16(q_host.shape, 12345)
    inp.q.copy_(api.bf16_tensor(q2, cuda_device))
    fn()
    torch.cuda.synchronize()
    eager2 = api.bf16_bits(out)
    assert not np.array_equal(eager2, eager)
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(api.bf16_bits(out), eager2)
    assert pd.pd_device_status() == 0
    if kind == "tiled_run":
        t.close()


def test_multi_step_graph_chains_steps(cuda_device):
    """Three split-K steps (partial + merge each) in one graph over three
    different caches: each step's output equals its eager result."""
    outs, fns, eager = [], [], []
    for i in range(3):
        w = W.custom([100 + 50 * i, 2049, 17], 24, 8, 128, seed=45 + i)
        inp = api.PagedInputs(w, cuda_device)
        out = torch.empty((w.num_seqs, 24, 128), dtype=torch.bfloat16, device=cuda_device)
        ws = api.workspace(w.num_seqs, 24, 128, 13, cuda_device)
        fn = (lambda inp=inp, w=w, out=out, ws=ws:
              api.decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, w.inv_sqrt_d, 13, 0, out, ws))
        fn()
        torch.cuda.synchronize()
        eager.append(api.bf16_bits(out))
        outs.append(out)
        fns.append(fn)
    g = _graph(lambda: [f() for f in fns])
    for o in outs:
        o.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    for o, e in zip(outs, eager):
        assert np.array_equal(api.bf16_bits(o), e)
