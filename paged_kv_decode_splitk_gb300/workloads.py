"""Seeded synthetic inputs for paged-decode attention.

This module only draws inputs: random BF16 values, context lengths, block
tables and tile plans.  It holds none of the attention arithmetic, imports
neither the CUDA binding nor the oracle, and is the one module both sides of
every parity check take their inputs from.

Recipe (stated once, used everywhere):
  * values: numpy ``default_rng(seed)`` standard normal in FP32, rounded to
    BF16 with round-to-nearest-even; q, K and V from independent streams;
  * placement: a second ``default_rng(seed + 1)`` draws context lengths, then a
    random permutation of the pool's physical blocks; sequence s takes the next
    ceil(L_s / block_size) entries of that permutation;
  * pool: ceil(1.25 x the blocks the sequences need), every block filled with
    values, so a kernel that reads a wrong block reads plausible data.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_VALUES = 0


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP32 to BF16 (nearest, ties to even); returns the uint16 bit patterns."""
    shape = np.shape(x)
    u = np.ascontiguousarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16).reshape(shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to FP32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, 1) BF16 bit patterns of the given shape, drawn in bounded chunks."""
    n = int(np.prod(shape))
    rng = np.random.default_rng(seed)
    out = np.empty(n, dtype=np.uint16)
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        out[a:b] = bf16_bits(rng.standard_normal(b - a, dtype=np.float32))
    return out.reshape(shape)


@dataclass
class PagedWorkload:
    """Inputs of one paged-decode launch, host side (numpy)."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q: np.ndarray               # [S, Hq, D] uint16 (BF16 bits)
    k_cache: np.ndarray         # [num_blocks, block_size, Hkv, D] uint16
    v_cache: np.ndarray         # same
    block_table: np.ndarray     # [S, max_blocks_per_seq] int32
    context_lens: np.ndarray    # [S] int32
    inv_sqrt_d: float
    policy: str = "auto"        # "legacy" | "auto" | "pinned"
    pin: int = 0
    sm_count: int = 148
    max_decode_seqs: int = 0
    gqa_pack: int = 0            # 0 split-K path, 1 packed (non-split), 2 packed with splits
    seeds: dict = field(default_factory=dict)
    kv_dtype: str = "bf16"       # "bf16": k/v_cache hold BF16 bits; "e4m3": FP8 E4M3 codes (uint8)
    k_scale: float = 1.0         # e4m3 only: K = code value * k_scale, V = code value * v_scale
    v_scale: float = 1.0

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "e4m3" else 2

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes of one launch: live tokens only."""
        return (int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim
                * self.kv_elem_bytes * 2)


def _paged(name, lens, num_q_heads, num_kv_heads, head_dim, block_size, seed, pool_factor=1.25,
           pool_blocks=None, **kw) -> PagedWorkload:
    lens = np.asarray(lens, dtype=np.int64)
    S = lens.size
    need = [(-(-int(L) // block_size)) for L in lens]
    total = int(sum(need))
    nb = pool_blocks if pool_blocks is not None else max(1, int(np.ceil(pool_factor * total)))
    assert nb >= total
    place = np.random.default_rng(seed + 1)
    perm = place.permutation(nb).astype(np.int32)
    max_b = max(1, max(need) if need else 1)
    bt = np.zeros((S, max_b), dtype=np.int32)
    off = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[off:off + n]
        off += n
    q = normal_bf16((S, num_q_heads, head_dim), 10_000 + seed * 3 + 0)
    k = normal_bf16((nb, block_size, num_kv_heads, head_dim), 10_000 + seed * 3 + 1)
    v = normal_bf16((nb, block_size, num_kv_heads, head_dim), 10_000 + seed * 3 + 2)
    inv = float(np.float32(1.0 / np.sqrt(head_dim)))
    kw.setdefault("inv_sqrt_d", inv)
    return PagedWorkload(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                         head_dim=head_dim, block_size=block_size, q=q, k_cache=k, v_cache=v,
                         block_table=bt, context_lens=lens.astype(np.int32),
                         seeds={"values": seed, "placement": seed + 1}, **kw)


def tiny(pin: int = 1, seed: int = SEED_VALUES) -> PagedWorkload:
    """2 sequences of 37 and 100 tokens; Hq 4, Hkv 1, D 64, block 16; a 16-block pool
    whose block table is the first 3 + next 7 entries of a random permutation; scale 1/8."""
    w = _paged("tiny_2x{37,100}_h4kv1_d64", [37, 100], 4, 1, 64, 16, seed, pool_blocks=16,
               inv_sqrt_d=0.125, policy="pinned", pin=pin)
    return w


def gqa_packed(seed: int = SEED_VALUES) -> PagedWorkload:
    """32 sequences, lengths uniform in [512, 4096]; Hq 16, Hkv 2 (pack width 8), D 256,
    block 16; non-split launch through the GQA-packed pass."""
    lens = np.random.default_rng(seed + 1).integers(512, 4096, size=32, endpoint=True)
    return _paged("gqa_packed_32seq_h16kv2_d256", lens, 16, 2, 256, 16, seed + 100,
                  policy="pinned", pin=1, gqa_pack=True)


def gqa_packed_splitk(seed: int = SEED_VALUES) -> PagedWorkload:
    """The GQA-packed workload's sequences through the packed pass with splits
    (gqa_pack mode 2): Auto at 148 SMs and 16 q heads gives ceil(296 / 16) = 19,
    clamped to 16 splits."""
    lens = np.random.default_rng(seed + 1).integers(512, 4096, size=32, endpoint=True)
    return _paged("gqa_packed_splitk_32seq_h16kv2_d256", lens, 16, 2, 256, 16, seed + 100,
                  policy="auto", sm_count=148, gqa_pack=2)


def _packed_long_lens() -> list:
    return [32768, 32768]


def gqa_packed_long(seed: int = SEED_VALUES) -> PagedWorkload:
    """Few long sequences at the packed shape: 2 sequences of 32768 tokens; Hq 16,
    Hkv 2 (pack width 8), D 256, block 16; non-split launch through the packed
    pass (only 2 x 2 = 4 units)."""
    return _paged("gqa_packed_long_2x32768_h16kv2_d256", _packed_long_lens(), 16, 2, 256, 16, seed + 400,
                  policy="pinned", pin=1, gqa_pack=True)


def gqa_packed_long_splitk(seed: int = SEED_VALUES) -> PagedWorkload:
    """The same sequences, cache and block table through the packed pass with
    splits (gqa_pack mode 2) at Auto: ceil(296 / 16) = 19, clamped to 16 splits
    of 2048 tokens each."""
    return _paged("gqa_packed_long_splitk_2x32768_h16kv2_d256", _packed_long_lens(), 16, 2, 256, 16,
                  seed + 400, policy="auto", sm_count=148, gqa_pack=2)


def long_context(seed: int = SEED_VALUES) -> PagedWorkload:
    """1 sequence of 32768 tokens; Hq 24, Hkv 8, D 128, block 16; Auto at 148 SMs (13 splits)."""
    return _paged("long_context_1x32768_h24kv8_d128", [32768], 24, 8, 128, 16, seed + 200,
                  policy="auto", sm_count=148)


def large_batch_lens(num_seqs: int = 256, seed: int = SEED_VALUES, sigma: float = 1.0) -> np.ndarray:
    """Lognormal lengths with median 2048 (sigma 1.0), rounded, clipped to [16, 16384]."""
    rng = np.random.default_rng(seed + 301)
    raw = rng.lognormal(mean=np.log(2048.0), sigma=sigma, size=num_seqs)
    return np.clip(np.round(raw), 16, 16384).astype(np.int64)


def large_batch(seed: int = SEED_VALUES, num_seqs: int = 256) -> PagedWorkload:
    """256 sequences, lognormal lengths (median 2048, clipped [16, 16384]); Hq 32, Hkv 8,
    D 128, block 16; Auto at 148 SMs (10 splits)."""
    lens = large_batch_lens(num_seqs, seed)
    return _paged(f"large_batch_{num_seqs}seq_h32kv8_d128", lens, 32, 8, 128, 16, seed + 300,
                  policy="auto", sm_count=148)


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round FP32 values to FP8 E4M3 (nearest, ties to even, as torch's float8_e4m3fn
    cast does); returns the uint8 codes.  Inputs must lie within +-448."""
    import torch
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert np.all(np.abs(x) <= 448.0), "outside the E4M3 range"
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def fp8_variant(w: PagedWorkload, k_scale: float = 0.5, v_scale: float = 0.25,
                seed: int = SEED_VALUES) -> PagedWorkload:
    """The same shape, sequences and block table with an FP8 E4M3 KV cache: fresh
    N(0, 1) draws divided by the per-tensor scale and rounded to E4M3 (so the
    dequantised cache is again about N(0, 1); about 1% of the codes are subnormal)."""
    shape = w.k_cache.shape
    n = int(np.prod(shape))
    out = []
    for i, sc in enumerate((k_scale, v_scale)):
        rng = np.random.default_rng(20_000 + seed * 3 + i)
        vals = np.empty(n, dtype=np.uint8)
        chunk = 1 << 24
        for a in range(0, n, chunk):
            b = min(n, a + chunk)
            vals[a:b] = e4m3_codes(np.clip(rng.standard_normal(b - a, dtype=np.float32) / np.float32(sc),
                                           -448.0, 448.0))
        out.append(vals.reshape(shape))
    kw = dict(w.__dict__)
    kw.update(name=w.name + "_e4m3", k_cache=out[0], v_cache=out[1], kv_dtype="e4m3",
              k_scale=float(np.float32(k_scale)), v_scale=float(np.float32(v_scale)))
    kw["seeds"] = dict(w.seeds, fp8=seed)
    return PagedWorkload(**kw)


def long_context_fp8(seed: int = SEED_VALUES) -> PagedWorkload:
    """The long-context workload (1 x 32768 tokens, Hq 24, Hkv 8, D 128, 13 splits)
    over an FP8 E4M3 cache with k_scale 0.5, v_scale 0.25."""
    return fp8_variant(long_context(seed), seed=seed)


def large_batch_fp8(seed: int = SEED_VALUES) -> PagedWorkload:
    """The large-batch workload (256 lognormal sequences, Hq 32, Hkv 8, D 128, 10
    splits) over an FP8 E4M3 cache with k_scale 0.5, v_scale 0.25."""
    return fp8_variant(large_batch(seed), seed=seed)


def gqa_packed_fp8(seed: int = SEED_VALUES) -> PagedWorkload:
    """The GQA-packed workload (32 sequences, Hq 16, Hkv 2, D 256, packed, non-split)
    over an FP8 E4M3 cache with k_scale 0.5, v_scale 0.25."""
    return fp8_variant(gqa_packed(seed), seed=seed)


def first_seqs(w: PagedWorkload, n: int) -> PagedWorkload:
    """The first n sequences of a paged workload, with a cache holding only their
    blocks (same values; a block keeps its place relative to the others), so a
    profiler capture of the same recipe fits in a few GB."""
    n = max(1, min(int(n), w.num_seqs))
    bs = w.block_size
    need = [-(-int(L) // bs) for L in w.context_lens[:n]]
    used = np.unique(np.concatenate([w.block_table[s, :k] for s, k in enumerate(need)] or
                                    [np.zeros(0, np.int32)])).astype(np.int64)
    remap = np.full(w.num_blocks, -1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    bt = np.zeros((n, max(1, max(need) if need else 1)), dtype=np.int32)
    for s, k in enumerate(need):
        bt[s, :k] = remap[w.block_table[s, :k]]
    kw = dict(w.__dict__)
    kw.update(name=f"{w.name}_first{n}", q=w.q[:n], k_cache=w.k_cache[used] if used.size else w.k_cache[:1],
              v_cache=w.v_cache[used] if used.size else w.v_cache[:1], block_table=bt,
              context_lens=w.context_lens[:n].copy())
    return PagedWorkload(**kw)


def custom(lens, num_q_heads, num_kv_heads, head_dim, block_size=16, seed=SEED_VALUES,
           **kw) -> PagedWorkload:
    """Any shape, same recipe (used for edge cases and ragged tails)."""
    return _paged(f"custom_{len(lens)}seq_h{num_q_heads}kv{num_kv_heads}_d{head_dim}", lens,
                  num_q_heads, num_kv_heads, head_dim, block_size, seed, **kw)


@dataclass
class TiledWorkload:
    """Inputs of one tiled decode step: begin, num_calls step_tile calls, finalize."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    tile_capacity: int
    q: np.ndarray                 # [S, Hq, D] uint16
    pool: np.ndarray              # scratch pool [slots, 2, Hkv, bs, D] or paged [nb, bs, Hkv, D] x2
    layout: str                   # "scratch" | "paged"
    tile_blocks: np.ndarray       # [T, S, tcap] int32
    tile_block_counts: np.ndarray  # [T, S] int32
    last_block_valid_slots: np.ndarray  # [T] int32
    blocks_per_seq: np.ndarray    # [S] total blocks of each sequence
    v_pool: np.ndarray | None = None    # paged layout only: V cache
    seeds: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_calls(self) -> int:
        return int(self.tile_blocks.shape[0])

    @property
    def kv_tokens(self) -> int:
        bs = self.block_size
        n = 0
        for c in range(self.num_calls):
            lb = int(self.last_block_valid_slots[c])
            for s in range(self.num_seqs):
                cnt = int(self.tile_block_counts[c, s])
                if cnt:
                    n += (cnt - 1) * bs + (lb if 1 <= lb < bs else bs)
        return n

    @property
    def kv_bytes(self) -> int:
        return self.kv_tokens * self.num_kv_heads * self.head_dim * 2 * 2


def tiled(seed: int = SEED_VALUES, num_seqs: int = 64, num_q_heads: int = 16, num_kv_heads: int = 4,
          head_dim: int = 256, block_size: int = 16, tile_capacity: int = 64, num_calls: int = 4,
          max_blocks: int = 256, last_valid: int = 5, layout: str = "scratch",
          min_zero: int = 2) -> TiledWorkload:
    """64 sequences with block counts uniform in [0, 256] (at least two with none) in the
    scratch-pool layout [slot, K|V, Hkv, block, D]; Hq 16, Hkv 4, D 256; tiles of 64 blocks
    over 4 right-aligned step_tile calls, so every sequence's final block falls in the last
    call, which passes last_block_valid_slots = 5 (earlier calls pass a full block)."""
    place = np.random.default_rng(seed + 401)
    n = place.integers(0, max_blocks, size=num_seqs, endpoint=True).astype(np.int64)
    zeros = int((n == 0).sum())
    for s in range(num_seqs):
        if zeros >= min_zero:
            break
        if n[s] != 0:
            n[s] = 0
            zeros += 1
    total = int(n.sum())
    slots = max(1, int(np.ceil(1.25 * total)))
    perm = place.permutation(slots).astype(np.int32)
    T, tcap = num_calls, tile_capacity
    tb = np.zeros((T, num_seqs, tcap), dtype=np.int32)
    tc = np.zeros((T, num_seqs), dtype=np.int32)
    off = 0
    for s in range(num_seqs):
        ids = perm[off:off + n[s]]
        off += n[s]
        for c in range(T):
            lo = max(0, int(n[s]) - (T - c) * tcap)
            hi = max(0, int(n[s]) - (T - 1 - c) * tcap)
            cnt = hi - lo
            assert cnt <= tcap
            tc[c, s] = cnt
            tb[c, s, :cnt] = ids[lo:hi]
    assert off == total
    lbvs = np.full(T, block_size, dtype=np.int32)
    lbvs[-1] = last_valid
    q = normal_bf16((num_seqs, num_q_heads, head_dim), seed * 3 + 400)
    if layout == "scratch":
        pool = normal_bf16((slots, 2, num_kv_heads, block_size, head_dim), seed * 3 + 401)
        vp = None
    elif layout == "paged":
        pool = normal_bf16((slots, block_size, num_kv_heads, head_dim), seed * 3 + 401)
        vp = normal_bf16((slots, block_size, num_kv_heads, head_dim), seed * 3 + 402)
    else:
        raise ValueError(layout)
    return TiledWorkload(name=f"tiled_{num_seqs}seq_h{num_q_heads}kv{num_kv_heads}_d{head_dim}_"
                              f"tcap{tile_capacity}_{layout}",
                         num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                         block_size=block_size, tile_capacity=tcap, q=q, pool=pool, layout=layout,
                         tile_blocks=tb, tile_block_counts=tc, last_block_valid_slots=lbvs,
                         blocks_per_seq=n, v_pool=vp, seeds={"values": seed, "placement": seed + 401})


@dataclass
class MixedTiledWorkload:
    """Inputs of one tiled decode step whose step_tile calls read different
    sources: each sequence's older blocks sit in a paged cache [nb, bs, Hkv, D]
    (K and V separate), its newer blocks in a scratch pool [slot, K|V, Hkv, bs, D].
    calls[c] = (source "paged" | "scratch", tile_blocks [S, tcap],
    tile_block_counts [S], last_block_valid_slots)."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    tile_capacity: int
    q: np.ndarray                 # [S, Hq, D] uint16
    paged_k: np.ndarray           # [nb, bs, Hkv, D] uint16
    paged_v: np.ndarray
    scratch: np.ndarray           # [slots, 2, Hkv, bs, D] uint16
    calls: list
    blocks_per_seq: np.ndarray    # [S]
    seeds: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def kv_tokens(self) -> int:
        bs = self.block_size
        n = 0
        for _, _, tc, lb in self.calls:
            for cnt in tc:
                if cnt:
                    n += (int(cnt) - 1) * bs + (lb if 1 <= lb < bs else bs)
        return n

    @property
    def kv_bytes(self) -> int:
        return self.kv_tokens * self.num_kv_heads * self.head_dim * 2 * 2


def _right_aligned_calls(ids_per_seq, ncalls: int, tcap: int):
    """Split each sequence's block list over ncalls tiles of tcap, last tile last."""
    S = len(ids_per_seq)
    out = []
    for c in range(ncalls):
        tb = np.zeros((S, tcap), dtype=np.int32)
        tc = np.zeros(S, dtype=np.int32)
        for s, ids in enumerate(ids_per_seq):
            n = len(ids)
            lo = max(0, n - (ncalls - c) * tcap)
            hi = max(0, n - (ncalls - 1 - c) * tcap)
            tc[s] = hi - lo
            tb[s, :hi - lo] = ids[lo:hi]
        out.append((tb, tc))
    return out


def tiled_mixed(seed: int = SEED_VALUES, num_seqs: int = 64, num_q_heads: int = 16,
                num_kv_heads: int = 4, head_dim: int = 256, block_size: int = 16,
                tile_capacity: int = 64, max_blocks: int = 256, last_valid: int = 5,
                min_zero: int = 2) -> MixedTiledWorkload:
    """The tiled workload's shape (block counts uniform in [0, 256], at least two
    sequences with none, Hq 16, Hkv 4, D 256, tiles of 64 blocks) with each
    sequence's first half of blocks (rounded down) in the paged cache and the rest
    in the scratch pool.  The step reads the paged source in right-aligned tiles,
    then the scratch source likewise; only the last call passes
    last_block_valid_slots = 5, so every non-empty sequence's final block holds 5
    tokens."""
    place = np.random.default_rng(seed + 501)
    n = place.integers(0, max_blocks, size=num_seqs, endpoint=True).astype(np.int64)
    zeros = int((n == 0).sum())
    for s in range(num_seqs):
        if zeros >= min_zero:
            break
        if n[s] != 0:
            n[s] = 0
            zeros += 1
    npg = n // 2
    nsc = n - npg
    nb = max(1, int(np.ceil(1.25 * int(npg.sum()))))
    slots = max(1, int(np.ceil(1.25 * int(nsc.sum()))))
    perm_p = place.permutation(nb).astype(np.int32)
    perm_s = place.permutation(slots).astype(np.int32)
    ids_p, ids_s = [], []
    op = os_ = 0
    for s in range(num_seqs):
        ids_p.append(perm_p[op:op + npg[s]])
        op += npg[s]
        ids_s.append(perm_s[os_:os_ + nsc[s]])
        os_ += nsc[s]
    cp = max(1, -(-int(npg.max()) // tile_capacity)) if len(npg) else 1
    cs = max(1, -(-int(nsc.max()) // tile_capacity)) if len(nsc) else 1
    calls = [("paged", tb, tc, block_size) for tb, tc in _right_aligned_calls(ids_p, cp, tile_capacity)]
    sc = _right_aligned_calls(ids_s, cs, tile_capacity)
    for c, (tb, tc) in enumerate(sc):
        calls.append(("scratch", tb, tc, last_valid if c == len(sc) - 1 else block_size))
    q = normal_bf16((num_seqs, num_q_heads, head_dim), seed * 3 + 500)
    pk = normal_bf16((nb, block_size, num_kv_heads, head_dim), seed * 3 + 501)
    pv = normal_bf16((nb, block_size, num_kv_heads, head_dim), seed * 3 + 502)
    sp = normal_bf16((slots, 2, num_kv_heads, block_size, head_dim), seed * 3 + 503)
    return MixedTiledWorkload(name=f"tiled_mixed_{num_seqs}seq_h{num_q_heads}kv{num_kv_heads}_d{head_dim}_"
                                   f"tcap{tile_capacity}",
                              num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                              block_size=block_size, tile_capacity=tile_capacity, q=q, paged_k=pk,
                              paged_v=pv, scratch=sp, calls=calls, blocks_per_seq=n,
                              seeds={"values": seed, "placement": seed + 501})


def scratch_pool_views(pool: np.ndarray):
    """Flat K and V views of a scratch pool [slot, 2, Hkv, bs, D]: K starts at element 0,
    V one K|V stripe (Hkv*bs*D elements) later."""
    slots, two, hkv, bs, d = pool.shape
    flat = pool.reshape(-1)
    stripe = hkv * bs * d
    return flat, flat[stripe:]


WORKLOADS = {
    "tiny": tiny,
    "gqa_packed": gqa_packed,
    "gqa_packed_splitk": gqa_packed_splitk,
    "gqa_packed_long": gqa_packed_long,
    "gqa_packed_long_splitk": gqa_packed_long_splitk,
    "gqa_packed_fp8": gqa_packed_fp8,
    "long_context_fp8": long_context_fp8,
    "large_batch_fp8": large_batch_fp8,
    "long_context": long_context,
    "large_batch": large_batch,
    "tiled": tiled,
    "tiled_mixed": tiled_mixed,
}
