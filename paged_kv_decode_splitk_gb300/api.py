"""Torch-level helpers over the C ABI: device placement of host inputs and
one-call wrappers that allocate outputs and the split-K workspace.

Plumbing only: every computation is a libpd kernel launched through `pd`.
"""

from __future__ import annotations

import numpy as np
import torch

from . import pd


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """A torch BF16 tensor holding the given BF16 bit patterns (uint16)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def i32_tensor(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """BF16 bit patterns (uint16) of a torch BF16 tensor, on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class PagedInputs:
    """Device copies of a workloads.PagedWorkload."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.device = torch.device(device)
        self.q = bf16_tensor(w.q, self.device)
        if getattr(w, "kv_dtype", "bf16") == "e4m3":   # FP8 E4M3 codes, one byte each
            self.k = torch.from_numpy(np.ascontiguousarray(w.k_cache, dtype=np.uint8)).to(self.device)
            self.v = torch.from_numpy(np.ascontiguousarray(w.v_cache, dtype=np.uint8)).to(self.device)
        else:
            self.k = bf16_tensor(w.k_cache, self.device)
            self.v = bf16_tensor(w.v_cache, self.device)
        self.block_table = i32_tensor(w.block_table, self.device)
        self.context_lens = i32_tensor(w.context_lens, self.device)

    def splits(self, policy: str | None = None, pin: int | None = None, sm_count: int | None = None,
               max_decode_seqs: int | None = None) -> int:
        w = self.w
        return pd.pd_num_splits(policy or w.policy, w.pin if pin is None else pin,
                                w.sm_count if sm_count is None else sm_count, w.num_q_heads,
                                w.num_seqs, w.max_decode_seqs if max_decode_seqs is None
                                else max_decode_seqs)


def workspace(num_seqs: int, num_q_heads: int, head_dim: int, num_splits: int, device) -> torch.Tensor | None:
    n = pd.pd_workspace_bytes(num_seqs, num_q_heads, head_dim, num_splits)
    if num_splits <= 1 or n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode_attn(q, k_cache, v_cache, block_table, context_lens, inv_sqrt_d: float, num_splits: int,
                gqa_pack: int = 0, out=None, ws=None, stream=None, k_scale: float = 1.0,
                v_scale: float = 1.0):
    """Paged-decode attention; returns out [S, Hq, D] BF16 (or None when the packed
    pass does not apply to the shape, mirroring PD_NOT_APPLICABLE).  uint8 caches
    are FP8 E4M3 codes with per-tensor scales k_scale / v_scale."""
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=q.device)
    if ws is None and num_splits > 1:
        ws = workspace(S, Hq, D, num_splits, q.device)
    if k_cache.dtype == torch.uint8:
        rc = pd.pd_decode_attn_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, out,
                                   inv_sqrt_d, num_splits, ws, gqa_pack, stream)
    else:
        rc = pd.pd_decode_attn(q, k_cache, v_cache, block_table, context_lens, out, inv_sqrt_d,
                               num_splits, ws, gqa_pack, stream)
    if rc == pd.PD_NOT_APPLICABLE:
        return None
    return out


def run_paged(inp: PagedInputs, num_splits: int | None = None, gqa_pack: bool | None = None, out=None,
              ws=None, stream=None):
    w = inp.w
    n = inp.splits() if num_splits is None else num_splits
    pack = w.gqa_pack if gqa_pack is None else gqa_pack
    return decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, w.inv_sqrt_d, n,
                       pack, out, ws, stream, getattr(w, "k_scale", 1.0), getattr(w, "v_scale", 1.0))


class TiledInputs:
    """Device copies of a workloads.TiledWorkload."""

    def __init__(self, tw, device="cuda"):
        self.w = tw
        self.device = torch.device(device)
        self.q = bf16_tensor(tw.q, self.device)
        self.pool = bf16_tensor(tw.pool, self.device)
        if tw.layout == "scratch":
            flat = self.pool.view(-1)
            stripe = tw.num_kv_heads * tw.block_size * tw.head_dim
            self.k_pool = flat
            self.v_pool = flat[stripe:]
        else:
            self.k_pool = self.pool
            self.v_pool = bf16_tensor(tw.v_pool, self.device)
        self.tile_blocks = [i32_tensor(tw.tile_blocks[c], self.device) for c in range(tw.num_calls)]
        self.tile_counts = [i32_tensor(tw.tile_block_counts[c], self.device) for c in range(tw.num_calls)]


def run_tiled(inp: TiledInputs, tiled: pd.Tiled | None = None, out=None, stream=None):
    """begin_step, one step_tile per call, finalize; returns out [S, Hq, D] BF16."""
    tw = inp.w
    own = tiled is None
    if own:
        tiled = pd.Tiled(tw.num_seqs, tw.num_q_heads, tw.num_kv_heads, tw.head_dim, tw.block_size,
                         tw.tile_capacity)
    try:
        strides = tiled.scratch_pool_strides() if tw.layout == "scratch" else tiled.paged_strides()
        if out is None:
            out = torch.empty((tw.num_seqs, tw.num_q_heads, tw.head_dim), dtype=torch.bfloat16,
                              device=inp.device)
        tiled.begin(tw.num_seqs, stream)
        for c in range(tw.num_calls):
            tiled.step(inp.q, inp.k_pool, inp.v_pool, inp.tile_blocks[c], inp.tile_counts[c],
                       tw.num_seqs, strides, int(tw.last_block_valid_slots[c]), stream)
        tiled.finalize(out, tw.num_seqs, stream)
    finally:
        if own:
            torch.cuda.current_stream().synchronize()
            tiled.close()
    return out


class MixedTiledInputs:
    """Device copies of a workloads.MixedTiledWorkload."""

    def __init__(self, mw, device="cuda"):
        self.w = mw
        self.device = torch.device(device)
        self.q = bf16_tensor(mw.q, self.device)
        self.paged_k = bf16_tensor(mw.paged_k, self.device)
        self.paged_v = bf16_tensor(mw.paged_v, self.device)
        self.scratch = bf16_tensor(mw.scratch, self.device)
        flat = self.scratch.view(-1)
        stripe = mw.num_kv_heads * mw.block_size * mw.head_dim
        self.scratch_k = flat
        self.scratch_v = flat[stripe:]
        self.tile_blocks = [i32_tensor(c[1], self.device) for c in mw.calls]
        self.tile_counts = [i32_tensor(c[2], self.device) for c in mw.calls]

    def sources(self, tiled: pd.Tiled):
        out = []
        for i, (kind, _, _, lbvs) in enumerate(self.w.calls):
            if kind == "paged":
                k, v, st = self.paged_k, self.paged_v, tiled.paged_strides()
            else:
                k, v, st = self.scratch_k, self.scratch_v, tiled.scratch_pool_strides()
            out.append((k, v, self.tile_blocks[i], self.tile_counts[i], st, int(lbvs)))
        return out


def run_tiled_mixed(inp: MixedTiledInputs, tiled: pd.Tiled | None = None, out=None, stream=None):
    """One pd_tiled_run: begin, one step per source (paged, then scratch pool), finalize."""
    mw = inp.w
    own = tiled is None
    if own:
        tiled = pd.Tiled(mw.num_seqs, mw.num_q_heads, mw.num_kv_heads, mw.head_dim, mw.block_size,
                         mw.tile_capacity)
    try:
        if out is None:
            out = torch.empty((mw.num_seqs, mw.num_q_heads, mw.head_dim), dtype=torch.bfloat16,
                              device=inp.device)
        tiled.run(inp.q, inp.sources(tiled), out, mw.num_seqs, stream)
    finally:
        if own:
            torch.cuda.current_stream().synchronize()
            tiled.close()
    return out
