// pd_unit.cuh -- the unit kernel: one (sequence, KV head, split) of paged-decode
// attention, serving a whole group of query heads from one read of K and V.
// The same kernel, by template mode, is the tiled step (one (sequence, KV
// head) of a step_tile call) and the fused tiled run (one (sequence, KV head,
// call) of every call at once).
//
// What a unit computes (Module attn_splitk page: split-K partials kept as
// [o, m, l]; tiled_attention.rs page: the running (m, l, o) fold):
//   for the query rows g of the group and the tokens t of the unit's range,
//     x[g,t] = (q[g] . K[t]) * inv_sqrt_d
//     m[g]   = max_t x[g,t],  l[g] = sum_t e^(x[g,t]-m[g]),  o[g] = sum_t e^(x[g,t]-m[g]) V[t]
//   (kept internally in base-2 units: m is max_t x[g,t]*log2(e), or in paged
//   mode a reference at most 8 below it, with l and o taken against it).
//
// GB300 mapping:
//   * The unit's range of 16-token tiles is cut into V length-defined parts
//     (V = clamp(ceil(tiles / PT), 1, max_parts), PT = 32, or 24 in the packed
//     pass).  A CTA of kWarps
//     warps takes a part; warp w folds its tiles w, w+kWarps, ... with its own
//     online-softmax state and the warps merge in warp order.  The parts fold
//     left to right with pinned rounding, either in one CTA walking them in
//     turn or across a thread-block cluster (one part per rank, combined
//     through distributed shared memory).  V, the warp interleave and every
//     fold order depend only on the unit's own length and build constants,
//     so a sequence's bits depend neither on the batch nor on the layout.
//   * Cluster ranks beyond V leave at once; the others hand their parts over
//     through mbarriers (bounded waits), or through the hardware cluster
//     barrier when every rank holds a part.
//   * K and V tiles move global -> shared with 4-D TMA tensor loads gathered
//     through the block table (BF16: one 128-byte-swizzled box per 64
//     columns; FP8 E4M3 from head dim 128 up: K and V in 128-byte-swizzled
//     boxes of 128 codes whose codes each thread converts straight into its
//     mma operands, V's pairs of tokens gathered by byte permutes; at head dim
//     64 both go through f16 tiles converted by the warp).
//     Each warp runs a private ring
//     of `stages` buffers with separate K and V mbarriers, refilled as soon
//     as their data has been read, so the next tiles' loads overlap the
//     current tile's math (over an FP8 cache at head dim 128, with two stages
//     per warp, a tile's K and V share one barrier and are refilled together).
//   * In paged mode a column's reference max moves only when a tile's max
//     passes it by more than 8 (base 2); every fold uses the reference each
//     partial carries.  A paged unit of one part skips the part fold and the
//     cluster hand-off (outside the packed pass it is written straight from
//     the warp partials).
//   * Both products run on the tensor cores (mma.sync m16n8k16, BF16 or f16
//     operands, FP32 accumulate) with the tokens as the M dimension:
//     S^T[t,g] = K[t,:] q[g,:]^T (the group fills N = 8), then
//     O^T[d,g] += V^T[d,t] P^T[t,g].  P^T comes from the S^T accumulators
//     through an in-register 8x8 transpose (movmatrix).  P is split into a
//     high part and a residual, which keeps ~16 significant bits of every
//     weight; for groups of at most 4 the residual rides in the otherwise
//     idle columns 4..7 of the same mma.
//   * Column max and column sums of S^T use warp shuffles over the 8 lanes
//     that hold a column.
//   * Before waiting for the previous kernel (programmatic dependent launch),
//     a single-wave paged launch prefetches each CTA's first tiles into L2
//     from speculative, L2-only reads of the lengths and block ids; nothing
//     read before the wait feeds a result.
#pragma once

#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "pd_device.cuh"
#include "pd_internal.h"

// The packed pass is compiled for one group width and one head dim (Module
// attn_splitk page: constants DECODE_GQA_PACK_WIDTH, the kernels' PD_GQA, and
// DECODE_GQA_PACK_HEAD_DIM, the kernels' PD_HDIM).  pd_build_info() reports
// these, so the header's copies can be checked against them.
#define PD_GQA 8
#define PD_HDIM 256

namespace pd {

namespace cg = cooperative_groups;

constexpr unsigned int kDevBadBlockId = 1;
constexpr unsigned int kDevBadContextLen = 2;
constexpr unsigned int kDevBadTileCount = 4;
constexpr unsigned int kDevWaitTimeout = 8;

// Shared-memory plan of a unit CTA (host and device agree on it).  Offsets are
// from the 1024-byte-aligned base.  The warp-merge area and the CTA result
// reuse the stage ring once every tile has been consumed.
struct UnitSmem {
    int stages;  // stage ring (offset 0, 1024-aligned)
    int cvt;     // FP8 caches: the f16 tiles each warp converts the landed FP8 tiles into
    int merge;   // per-warp o [kWarps][rows][dpad+4]: overlaps the ring
    int result;  // CTA result o [rows][dpad+4], read by the cluster peers: overlaps the ring
    int qs;      // the CTA's query rows, BF16, padded rows
    int stats;   // per-warp m, l, weights; part m, l; row factors; fold factors; running m, l
    int bars;    // two mbarriers (K, V) per stage, then the cluster's ready and done barriers
    int lpt;     // longest-first order: context lengths + the pick
    int total;   // bytes to request, including the alignment slack
};

__host__ __device__ constexpr int unit_stat_floats(int rows) {
    return rows * (3 * kWarps + 2 + 4 + 2 * kMaxParts + 2);
}

__host__ __device__ inline UnitSmem unit_smem_plan(int dpad, int rows, int stages_per_warp,
                                                   bool kv8 = false) {
    UnitSmem s;
    const int elem = kv8 ? 1 : 2;
    const int stage_bytes = 2 * kTileTokens * dpad * elem;
    const int ring = kWarps * stages_per_warp * stage_bytes;
    const int ostride = dpad + 4;
    const int merge = kWarps * rows * ostride * 4;
    const int result = rows * ostride * 4;
    s.stages = 0;
    s.cvt = (ring + 1023) / 1024 * 1024;
    // f16 tiles per warp: K and V apart at head dims up to 64; from 128 up none
    // (both operands are built in registers from the landed codes)
    const int cvt_tiles = dpad <= 64 ? 2 : 0;
    const int loop_end = kv8 ? s.cvt + kWarps * cvt_tiles * kTileTokens * dpad * 2 : ring;
    s.merge = 0;
    s.result = merge;
    int end = s.result + result;
    if (loop_end > end) end = loop_end;
    s.qs = (end + 15) / 16 * 16;
    s.stats = s.qs + rows * (dpad * 2 + 16);
    s.bars = s.stats + (unit_stat_floats(rows) * 4 + 15) / 16 * 16;
    s.lpt = s.bars + (kWarps * stages_per_warp * 2 + 2) * 8;
    s.total = 1024 /* alignment slack */ + s.lpt + (kLptMaxSeqs + 4) * 4;
    return s;
}

// FP8 E4M3 tile (16 rows x DPAD bytes, row-major, as the TMA landed it) ->
// f16 tile in the 128-byte-swizzled box layout the BF16 path loads, so the same
// ldmatrix addressing serves both.  One hardware conversion per code pair;
// every E4M3 value (subnormals included) is an f16 value, so it is exact.  The
// products of an FP8 cache then run on the f16 tensor-core path.
template <int DPAD>
__device__ __forceinline__ void e4m3_tile_to_f16(const uint8_t *src, uint8_t *dst, int lane) {
    constexpr int CPR = DPAD / 16;  // 16-byte chunks per FP8 row
    // every chunk in flight at head dims up to 128; two at a time at 256, where
    // a full unroll would hold every chunk's registers on top of the o accumulators
#pragma unroll(DPAD <= 128 ? DPAD / 32 : 2)
    for (int i = 0; i < DPAD / 32; ++i) {
        // Iteration i covers rows 8*(i / (CPR/4)) .. +7; a quarter-warp takes 2
        // rows x 4 chunks of one box (the second row the neighbouring box when
        // there are two or more), so its eight 16-byte stores land in distinct
        // swizzled positions and its loads in distinct banks (no conflict).
        const int kb = i % (CPR / 4), rb = i / (CPR / 4);
        const int q = lane >> 3, j = lane & 7;
        const int kbx = CPR >= 8 ? (kb ^ (j >> 2)) : kb;
        const int t = 8 * rb + 2 * q + (j >> 2), k = 4 * kbx + (j & 3);
        const int c = t * CPR + k;
        const uint4 v = *reinterpret_cast<const uint4 *>(src + c * 16);
        uint4 lo, hi;
        dev::e4m3x4_to_f16x4(v.x, lo.x, lo.y);
        dev::e4m3x4_to_f16x4(v.y, lo.z, lo.w);
        dev::e4m3x4_to_f16x4(v.z, hi.x, hi.y);
        dev::e4m3x4_to_f16x4(v.w, hi.z, hi.w);
        const int col = 16 * k;
        uint8_t *box = dst + (col / kBoxCols) * (kTileTokens * 128);
        const int c8 = (col % kBoxCols) / 8;
        *reinterpret_cast<uint4 *>(box + t * 128 + ((c8 ^ (t & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(box + t * 128 + (((c8 + 1) ^ (t & 7)) << 4)) = hi;
    }
}

// The tensor-core product of the path: BF16 operands, or f16 over an FP8 cache.
template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    if constexpr (F16)
        dev::mma_f16_16816(d, a0, a1, a2, a3, b0, b1);
    else
        dev::mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
}

// CAP4: the same kernel held to 128 registers (4 CTAs per SM; no spill over an
// FP8 cache at head dim 128 with groups of up to 4 rows), for launches of
// many waves of short CTAs, where more resident CTAs hide more of each CTA's
// start and end.  Otherwise the compiler chooses (a bound of 0 blocks).
template <int DPAD, int GN, bool HL, int MODE, bool PACKED, bool KV8, bool CAP4 = false>
__global__ void __launch_bounds__(kThreads, CAP4 ? 4 : 0)
    unit_kernel(const __grid_constant__ KvMaps<MODE == kModeTiledRun ? kMaxRunSources : 1> maps,
                const __grid_constant__ UnitParams p) {
    constexpr int KS = DPAD / 16;      // mma k-steps of K.q^T == m-tiles of V^T.P^T
    // Tiles a part aims for: the packed pass cuts its (sequence, KV head) units
    // finer (more of its one wave's CTAs busy; measured 24 against 16 and 32).
    constexpr int PT = PACKED ? kPartTilesPacked : kPartTiles;
    constexpr int NBOX = DPAD / kBoxCols;                 // BF16 boxes per tile (64 columns each)
    // FP8 cache from head dim 128 up: K's and V's codes go from the (128-byte
    // swizzled) FP8 tiles straight into the mma operands.
    constexpr bool KDIRECT = KV8 && DPAD >= 128;
    constexpr bool VDIRECT = KDIRECT;
    // K and V of a tile on one barrier, issued together (FP8 at head dim 128;
    // at 256, where a tile's math takes twice as long, the packed pass
    // measured slower with it)
    constexpr bool KV1BAR = KV8 && DPAD == 128;
    constexpr int TILE_BYTES = kTileTokens * DPAD * (KV8 ? 1 : 2);  // one landed K or V tile
    constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static_assert(!KV8 || MODE == kModePaged, "FP8 caches are a paged-mode source");
    constexpr bool RUN = MODE == kModeTiledRun;
    constexpr int RT = 8 * GN;         // query rows per CTA
    constexpr int OSTRIDE = DPAD + 4;  // padded row stride of o in shared memory
    constexpr int QST = DPAD * 2 + 16; // padded row stride of q in shared memory (bytes)
    constexpr int QPT = RT * (DPAD / 2) / kThreads;  // q words per thread
    static_assert(QPT * kThreads == RT * (DPAD / 2), "q staging must divide evenly");
    const float kNegInf = -__int_as_float(0x7f800000);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const UnitSmem plan = unit_smem_plan(DPAD, RT, S, KV8);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + plan.bars);  // [kWarps*S][K, V]
    // Cluster hand-off (one phase each): `ready` of a row owner completes when
    // every active rank has published its part; `done` of an active rank when
    // every owner has finished reading it.  Both expect kMaxParts arrivals; a
    // CTA arrives for the ranks that will not.
    uint64_t *bar_ready = bars + 2 * kWarps * p.stages;
    uint64_t *bar_done = bar_ready + 1;
    uint8_t *ring = smem + plan.stages;
    uint8_t *qsm = smem + plan.qs;
    float *stats = reinterpret_cast<float *>(smem + plan.stats);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // Shared-memory set-up needs no global memory: do it before waiting for
    // the previous kernel in the stream.
    if (tid == 0) {
        for (int i = 0; i < 2 * kWarps * S; ++i) dev::mbar_init(dev::smem_addr(&bars[i]), 1);
        dev::mbar_init(dev::smem_addr(bar_ready), kMaxParts);
        dev::mbar_init(dev::smem_addr(bar_done), kMaxParts);
        dev::fence_mbar_init();
    }
    // Every rank of a cluster arrives here, so a rank may leave early (an idle
    // rank, an empty unit) without holding the others; ranks that signal peers
    // wait on this barrier first, which makes the initialisations visible.
    if (p.cluster > 1) dev::cluster_arrive_relaxed();

    // ---- which unit (launch geometry only) ------------------------------------
    const int C = p.cluster;
    int part = 0;
    int u = blockIdx.x;
    if (C > 1) {
        part = u % C;
        u /= C;
    }
    int split = 0;  // paged: the split; fused tiled run: the source (step_tile call)
    if constexpr (MODE == kModePaged) {
        const int un = fast_div(u, p.fd_split);
        split = u - un * p.num_splits;
        u = un;
    } else if constexpr (RUN) {
        split = u % p.num_sources;
        u /= p.num_sources;
    }
    const CUtensorMap *tmk = &maps.k[RUN ? split : 0];
    const CUtensorMap *tmv = &maps.v[RUN ? split : 0];
    const int tok_dim = RUN ? p.src_tok_dim[split] : p.tok_dim;
    if (tid == 0) {
        dev::prefetch_tensormap(tmk);
        dev::prefetch_tensormap(tmv);
    }
    int qt = 0;
    if (p.qtiles > 1) {
        qt = u % p.qtiles;
        u /= p.qtiles;
    }
    int s = fast_div(u, p.fd_kvh);
    const int kvh = u - s * p.num_kv_heads;
    const int bs = p.block_size;
    const int Lmax = p.max_blocks_per_seq * bs;
    const int tiles_per_block = bs / kTileTokens;

    // The s-th longest sequence (ties by index), so that the longest units
    // start first.  Only which CTA serves a sequence changes; its arithmetic
    // does not.  `spec`: lengths read through L2 only, before the wait.
    auto longest_first = [&](bool spec) -> int {
        int *lens_s = reinterpret_cast<int *>(smem + plan.lpt);
        int &pick_s = lens_s[kLptMaxSeqs];
        const int ns = p.num_seqs;
        for (int c = tid; c < ns; c += kThreads) {
            const int Lc = spec ? __ldcg(p.context_lens + c) : p.context_lens[c];
            lens_s[c] = Lc < 0 ? 0 : (Lc > Lmax ? Lmax : Lc);
        }
        __syncthreads();
        for (int c = tid; c < ns; c += kThreads) {
            const int Lc = lens_s[c];
            int rank = 0;
            for (int j = 0; j < ns; ++j) rank += (lens_s[j] > Lc) || (lens_s[j] == Lc && j < c);
            if (rank == s) pick_s = c;
        }
        __syncthreads();
        const int picked = pick_s;
        __syncthreads();  // lens_s may be rewritten by the next call
        return picked;
    };

    // ---- speculative L2 prefetch, before the wait ------------------------------
    // The previous kernel in the stream may still be writing the lengths, the
    // block table or the caches, so nothing read here is used for results:
    // lengths and block ids are read through L2 only (no stale L1 line is left
    // behind), and they only choose which of this CTA's first tiles to prefetch
    // into L2 (a prefetch reads no value; L2 is where writes land, so a line
    // prefetched early is never stale).  Everything is read again after the
    // wait.  This fills the DRAM idle time at the previous kernel's tail.  The
    // tiled step's tile counts and tile lists are treated the same way.
    if (!RUN && p.prefetch_tiles > 0) {
        int t0 = 0, t1 = 0, ss = s;
        const int32_t *ids;
        if constexpr (MODE == kModePaged) {
            ss = p.lpt ? longest_first(true) : s;
            int L = __ldcg(p.context_lens + ss);
            L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
            const int chunk = split_chunk_tokens_fd(L, p.fd_split, p.fd_bs, p.min_kv_per_split);
            const long long a = static_cast<long long>(split) * chunk;
            t0 = static_cast<int>(a < L ? a : L);
            t1 = static_cast<int>(a + chunk < L ? a + chunk : L);
            ids = p.block_table + static_cast<long long>(ss) * p.max_blocks_per_seq;
        } else {
            int cnt = __ldcg(p.tile_counts + s);
            cnt = cnt < 0 ? 0 : (cnt > p.tile_capacity ? p.tile_capacity : cnt);
            const int lv = (p.last_valid >= 1 && p.last_valid < bs) ? p.last_valid : bs;
            t1 = cnt > 0 ? (cnt - 1) * bs + lv : 0;
            ids = p.tile_blocks + static_cast<long long>(s) * p.tile_capacity;
        }
        if (t0 < t1) {
            const int tile0 = t0 / kTileTokens;
            const int ntiles = (t1 + kTileTokens - 1) / kTileTokens - tile0;
            const int V = max(1, min(p.max_parts, (ntiles + PT - 1) / PT));
            const int j = C == 1 ? 0 : part;
            if (j < V) {
                const int my0 = tile0 + (j * ntiles) / V;
                const int n = min(tile0 + ((j + 1) * ntiles) / V - my0, p.prefetch_tiles);
                for (int t = tid; t < n; t += kThreads) {
                    const int gt = my0 + t;
                    const int blk = tiles_per_block > 1 ? gt / tiles_per_block : gt;
                    const int id = __ldcg(ids + blk);
                    if (id >= 0 && id < p.num_blocks) {
                        const int sub = (gt - blk * tiles_per_block) * kTileTokens;
                        const int c1 = tok_dim == 1 ? sub : kvh;
                        const int c2 = tok_dim == 1 ? kvh : sub;
                        if constexpr (KDIRECT) {
#pragma unroll
                            for (int b = 0; b < DPAD / 128; ++b) {
                                dev::tma_prefetch_4d(tmk, b * 128, c1, c2, id);
                                dev::tma_prefetch_4d(tmv, b * 128, c1, c2, id);
                            }
                        } else {
#pragma unroll
                            for (int b = 0; b < (KV8 ? 1 : NBOX); ++b) {
                                dev::tma_prefetch_4d(tmv, b * kBoxCols, c1, c2, id);
                                dev::tma_prefetch_4d(tmk, b * kBoxCols, c1, c2, id);
                            }
                        }
                    }
                }
            }
        }
    }

    dev::griddep_wait();  // the previous kernel's writes (q, caches, tables, out) are visible
    if constexpr (MODE == kModePaged) {
        if (p.lpt) s = longest_first(false);
    }
    const int G = PACKED ? PD_GQA : p.group;
    const int D = PACKED ? PD_HDIM : p.head_dim;
    const int Hq = PACKED ? p.num_kv_heads * PD_GQA : p.num_q_heads;
    const int g0 = qt * RT;                       // first group row of this CTA
    const int Gt = min(RT, G - g0);               // valid rows
    const int h0 = kvh * G + g0;                  // first query head

    // ---- query rows: issue the loads now, they do not depend on the range ----
    uint32_t qv[QPT];
    {
        const __nv_bfloat16 *qb = p.q + (static_cast<long long>(s) * Hq + h0) * D;
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            const int e = tid + i * kThreads;
            const int g = e / (DPAD / 2);
            const int d = (e - g * (DPAD / 2)) * 2;
            qv[i] = (g < Gt && d < D)
                        ? __ldg(reinterpret_cast<const unsigned int *>(qb + static_cast<long long>(g) * D + d))
                        : 0u;
        }
    }

    // ---- token range of the unit --------------------------------------------
    int tok0 = 0, tok1 = 0;
    bool direct = true;  // paged: write normalised output instead of a partial
    const int32_t *ids_base;
    if constexpr (MODE == kModePaged) {
        int L = p.context_lens[s];
        if (L < 0 || L > Lmax) {
            if (tid == 0 && part == 0 && split == 0 && qt == 0 && kvh == 0)
                dev::flag_status(p.status, kDevBadContextLen);
            L = L < 0 ? 0 : Lmax;
        }
        const int chunk = split_chunk_tokens_fd(L, p.fd_split, p.fd_bs, p.min_kv_per_split);
        const long long a = static_cast<long long>(split) * chunk;
        tok0 = static_cast<int>(a < L ? a : L);
        tok1 = static_cast<int>(a + chunk < L ? a + chunk : L);
        direct = L <= chunk;  // at most one non-empty split
        ids_base = p.block_table + static_cast<long long>(s) * p.max_blocks_per_seq;
        if (tok0 >= tok1) {
            // Empty split.  Split 0 of an empty sequence owns the zero output.
            if (L == 0 && split == 0 && part == 0) {
                for (int e = tid; e < Gt * (D / 2); e += kThreads) {
                    const int g = e / (D / 2), d = (e - g * (D / 2)) * 2;
                    *reinterpret_cast<uint32_t *>(p.out + (static_cast<long long>(s) * Hq + h0 + g) * D + d) = 0u;
                }
            }
            return;  // uniform across the cluster: every rank sees the same range
        }
    } else {
        // tiled step, or one call of a fused run: the call's tile list
        const int32_t *counts = RUN ? p.src_counts[split] : p.tile_counts;
        int cnt = counts[s];
        if (cnt < 0 || cnt > p.tile_capacity) {
            if (tid == 0 && part == 0 && qt == 0 && kvh == 0)
                dev::flag_status(p.status, kDevBadTileCount);
            cnt = cnt < 0 ? 0 : p.tile_capacity;
        }
        if (cnt == 0) return;  // nothing to fold: the state is unchanged
        const int lvc = RUN ? p.src_last_valid[split] : p.last_valid;
        const int lv = (lvc >= 1 && lvc < bs) ? lvc : bs;
        tok0 = 0;
        tok1 = (cnt - 1) * bs + lv;
        ids_base = (RUN ? p.src_blocks[split] : p.tile_blocks) + static_cast<long long>(s) * p.tile_capacity;
    }

    // 16-token tiles of the range, cut into V parts of about PT tiles
    // (at most p.max_parts).  V depends only on the range's own length; the
    // launch decides only where the parts run: all in this CTA one after
    // another (cluster == 1), or one per CTA of a cluster (cluster == max_parts).
    const int tile0 = tok0 / kTileTokens;
    const int ntiles = (tok1 + kTileTokens - 1) / kTileTokens - tile0;
    const int V = max(1, min(p.max_parts, (ntiles + PT - 1) / PT));
    // A rank of a cluster beyond the unit's parts has nothing to do: no peer
    // reads or signals it, so it leaves now and frees its slot.
    if (C > 1 && part >= V) return;
    // A paged unit of one part: its result is that part's, in either layout
    // (no fold into a running result, no hand-off between ranks).
    const bool solo = MODE == kModePaged && V == 1;

    // ---- q to shared memory (the barriers were initialised at the start) ----------
    // Over an FP8 cache the products run in f16: q is staged as f16 scaled by a
    // power of two 2^-kq that brings the CTA's largest |q| below 2^15 (kq = 0
    // for ordinary q, where the conversion is exact), and 2^kq goes back into
    // the softmax scale.  The rows are one (sequence, KV head)'s, so kq depends
    // on the sequence's own q only.
    float scale_log2 = p.scale_log2;
    if constexpr (KV8) {
        float qmax = 0.f;
#pragma unroll
        for (int i = 0; i < QPT; ++i)
            qmax = fmaxf(qmax, fmaxf(fabsf(dev::bf16_lo_f32(qv[i])), fabsf(dev::bf16_hi_f32(qv[i]))));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
        if (lane == 0) stats[warp] = qmax;
        __syncthreads();
        qmax = fmaxf(fmaxf(stats[0], stats[1]), fmaxf(stats[2], stats[3]));
        // qmax < 2^(E - 126) for a normal float with biased exponent E
        const int ex = ((__float_as_int(qmax) >> 23) & 0xff) - 126;
        const int kq = ex > 15 ? (ex - 15 < 126 ? ex - 15 : 126) : 0;
        const float down = __int_as_float((127 - kq) << 23);
        scale_log2 = p.scale_log2 * __int_as_float((127 + kq) << 23);
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            const int e = tid + i * kThreads;
            const int g = e / (DPAD / 2);
            int d = (e - g * (DPAD / 2)) * 2;
            if constexpr (KDIRECT) {
                // column pair P sits where the direct K operand uses it: in a
                // 128-column box, chunk c (8 pairs) is read by the lanes of quad
                // position qd = half (c even, block c/2) or 2 + half (c odd,
                // block ((c ^ 4) - 1) / 2); its pair j goes to k-step 2*block +
                // (j >> 1), pair qd + 4*(j & 1) of that k-step
                const int P = d >> 1, Pb = P & 63, c = Pb >> 3, half = (Pb >> 2) & 1, j = Pb & 3;
                const int kb = (P >> 6) * 4 + ((c & 1) ? (((c ^ 4) - 1) >> 1) : (c >> 1));
                const int qd = (c & 1) ? 2 + half : half;
                d = ((2 * kb + (j >> 1)) * 8 + qd + 4 * (j & 1)) * 2;
            }
            *reinterpret_cast<uint32_t *>(qsm + g * QST + d * 2) =
                dev::pack_f16x2(dev::bf16_lo_f32(qv[i]) * down, dev::bf16_hi_f32(qv[i]) * down);
        }
    } else {
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            const int e = tid + i * kThreads;
            const int g = e / (DPAD / 2);
            const int d = (e - g * (DPAD / 2)) * 2;
            *reinterpret_cast<uint32_t *>(qsm + g * QST + d * 2) = qv[i];
        }
    }
    // Running result of the parts folded so far (cluster == 1), starting empty:
    // m and l per row in shared memory, o in registers (element e = tid + i *
    // kThreads of the [RT][DPAD] rows, the same elements for every part).
    constexpr int RACC = RT * DPAD / kThreads;
    float racc[RACC];
#pragma unroll
    for (int i = 0; i < RACC; ++i) racc[i] = 0.f;
    float *rM = stats + unit_stat_floats(RT) - 2 * RT;  // [RT]
    float *rL = rM + RT;                                 // [RT]
    if (tid < RT) {
        rM[tid] = kNegInf;
        rL[tid] = 0.f;
    }
    __syncthreads();

    const uint64_t policy = dev::l2_evict_first_policy();

    // B operand of S^T = K q^T (q^T: d x g), one x2 ldmatrix per k-step and
    // n-tile: lanes 0-7 address rows g of columns k0..k0+7, lanes 8-15 k0+8..15.
    const uint32_t q_lm = dev::smem_addr(qsm) + (lane & 7) * QST + ((lane >> 3) & 1) * 16;

    // ---- per-lane ldmatrix offsets (128B swizzle: chunk c of row t at c ^ (t & 7)) ----
    // K as the A operand (t x d): matrices {t 0-7 | 8-15} x {d 0-7 | 8-15}, t fastest.
    // V^T as the A operand (d x t, via .trans): {t 0-7 | 8-15} slowest, d halves fastest.
    const int lm_j = lane >> 3;
    uint32_t lmk_off[4], lmv_off[4];
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2) {
        const int tk = ((lm_j & 1) << 3) | (lane & 7);
        lmk_off[c2] = tk * 128 + ((((2 * c2) + (lm_j >> 1)) ^ (lane & 7)) << 4);
        const int tv = ((lm_j >> 1) << 3) | (lane & 7);
        lmv_off[c2] = tv * 128 + ((((2 * c2) + (lm_j & 1)) ^ (lane & 7)) << 4);
    }

    const int tq = lane >> 2;         // token row of the S^T fragment
    const int gq = (lane & 3) * 2;    // first column (group row) of this thread
    float *wo = reinterpret_cast<float *>(smem + plan.merge);  // [kWarps][RT][OSTRIDE]
    float *wm = stats;                                         // [kWarps][RT]
    float *wl = wm + kWarps * RT;                              // [kWarps][RT]
    float *ww = wl + kWarps * RT;                              // [kWarps][RT] weights
    float *cm = ww + kWarps * RT;                              // [RT] part max
    float *cl = cm + RT;                                       // [RT] part sum
    float *fx = cl + RT;                                       // [RT][4] row factors of the final combine
    float *fr = fx + 4 * RT;                                   // [RT][2*kMaxParts] fold factors
    float *co = reinterpret_cast<float *>(smem + plan.result);  // [RT][OSTRIDE] part result
    constexpr int GCOLS = HL ? 4 : 8;  // meaningful columns per n-tile

    int rr = 0;  // tiles this warp has taken through its ring so far (stage phases)
    int k_next = 0;         // ring position of the warp's next tile: stage,
    uint32_t par_next = 0;  // and phase parity
    const int jfirst = C == 1 ? 0 : part;
    const int jstep = C == 1 ? 1 : C;
    for (int j = jfirst; j < V; j += jstep) {
        const int my0 = V == 1 ? tile0 : tile0 + (j * ntiles) / V;
        const int my1 = V == 1 ? tile0 + ntiles : tile0 + ((j + 1) * ntiles) / V;
        const int nloc = my1 - my0 > warp ? (my1 - my0 - warp + kWarps - 1) / kWarps : 0;

        // Block id of this warp's local tile r of the part (lane-parallel window loads).
        auto load_id = [&](int r) -> int {
            if (r >= nloc) return -1;
            const int gt = my0 + warp + kWarps * r;
            int id = __ldg(ids_base + (tiles_per_block > 1 ? gt / tiles_per_block : gt));
            // TMA reads zeros outside the tensor map's block extent (num_blocks).
            if (id < 0 || id >= p.num_blocks) dev::flag_status(p.status, kDevBadBlockId);
            return id;
        };
        // TMA of the K (half 0) or V (half 1) tile of local tile r into stage k.
        auto issue = [&](const CUtensorMap *map, int half, int r, int k, int id) {
            const int gt = my0 + warp + kWarps * r;
            int sub = 0;  // first token of the tile within its cache block
            if (tiles_per_block > 1) sub = (gt % tiles_per_block) * kTileTokens;
            const uint32_t bar = dev::smem_addr(&bars[(warp * S + k) * 2 + half]);
            const uint32_t dst = dev::smem_addr(ring + (warp * S + k) * STAGE_BYTES + half * TILE_BYTES);
            const int c1 = tok_dim == 1 ? sub : kvh;
            const int c2 = tok_dim == 1 ? kvh : sub;
            dev::mbar_arrive_expect_tx(bar, TILE_BYTES);
            // BF16: NBOX swizzled boxes of 64 columns.  FP8 from head dim 128
            // up: 128-byte swizzled boxes of 128 codes; at head dim 64 one
            // unswizzled box of the whole row.
            if (KDIRECT) {
#pragma unroll
                for (int b = 0; b < DPAD / 128; ++b)
                    dev::tma_load_4d(dst + b * (kTileTokens * 128), map, bar, b * 128, c1, c2, id, policy);
            } else {
#pragma unroll
                for (int b = 0; b < (KV8 ? 1 : NBOX); ++b)
                    dev::tma_load_4d(dst + b * (kTileTokens * 128), map, bar, b * kBoxCols, c1, c2, id, policy);
            }
        };
        // KV1BAR: K and V of a tile land on one barrier (half 0), issued
        // together after the tile's P.V, which saves a wait and an issue per
        // tile; the two stages per warp keep the next tile in flight meanwhile.
        auto issue_kv = [&](int r, int k, int id) {
            const int gt = my0 + warp + kWarps * r;
            int sub = 0;
            if (tiles_per_block > 1) sub = (gt % tiles_per_block) * kTileTokens;
            const uint32_t bar = dev::smem_addr(&bars[(warp * S + k) * 2]);
            const uint32_t dst = dev::smem_addr(ring + (warp * S + k) * STAGE_BYTES);
            const int c1 = tok_dim == 1 ? sub : kvh;
            const int c2 = tok_dim == 1 ? kvh : sub;
            dev::mbar_arrive_expect_tx(bar, STAGE_BYTES);
#pragma unroll
            for (int b = 0; b < DPAD / 128; ++b)
                dev::tma_load_4d(dst + b * (kTileTokens * 128), tmk, bar, b * 128, c1, c2, id, policy);
#pragma unroll
            for (int b = 0; b < DPAD / 128; ++b)
                dev::tma_load_4d(dst + TILE_BYTES + b * (kTileTokens * 128), tmv, bar, b * 128, c1, c2, id, policy);
        };

        // Block ids of local tiles [32*win, 32*win + 64): lane l of id_cur holds
        // tile 32*win + l, lane l of id_nxt tile 32*win + 32 + l.
        int win = 0;
        int id_cur = load_id(lane);
        int id_nxt = load_id(32 + lane);
        auto id_at = [&](int r) -> int {
            const int a = __shfl_sync(0xffffffffu, id_cur, r & 31);
            const int b = __shfl_sync(0xffffffffu, id_nxt, r & 31);
            return (r >> 5) == win ? a : b;
        };
        // Ring position of local tile 0: stage k with phase parity par; the
        // tiles take the stages in turn, the parity flipping at each wrap.
        int k = k_next;
        uint32_t par = par_next;
        const int npro = nloc < S ? nloc : S;
        for (int r = 0; r < npro; ++r) {
            const int id = __shfl_sync(0xffffffffu, id_cur, r);
            const int kr = k + r < S ? k + r : k + r - S;
            if (lane == 0) {
                if constexpr (KV1BAR) {
                    issue_kv(r, kr, id);
                } else {
                    issue(tmk, 0, r, kr, id);
                    issue(tmv, 1, r, kr, id);
                }
            }
        }

        // ---- online-softmax state ---------------------------------------------------
        // Accumulator layouts (m16n8 fragments): S^T[t][g] with t = lane/4 (+8),
        // g = nt*8 + (lane%4)*2 (+1); O^T[d][g] with d = mt*16 + lane/4 (+8) and the
        // same g.  Each thread keeps (m, l) of its two columns g.  With HL (groups of
        // at most 4) columns 4..7 of the single n-tile carry the BF16 residual of P
        // for columns 0..3, so one mma per m-tile serves both halves of P.
        float o[KS][GN][4];
#pragma unroll
        for (int a_ = 0; a_ < KS; ++a_)
#pragma unroll
            for (int b_ = 0; b_ < GN; ++b_)
#pragma unroll
                for (int c = 0; c < 4; ++c) o[a_][b_][c] = 0.f;
        float m_run[GN][2], l_run[GN][2];
#pragma unroll
        for (int nt = 0; nt < GN; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                m_run[nt][c] = kNegInf;
                l_run[nt][c] = 0.f;
            }
        int fail_r = -1;

        for (int r = 0; r < nloc; ++r) {
            const int rn = r + S;
            int id_next = -1;
            if (rn < nloc) {
                if ((rn >> 5) != win) {
                    id_cur = id_nxt;
                    win = rn >> 5;
                    id_nxt = load_id((win + 1) * 32 + lane);
                }
                id_next = id_at(rn);
            }
            if (!dev::mbar_wait_bounded(dev::smem_addr(&bars[(warp * S + k) * 2 + 0]), par)) {
                fail_r = r;
                break;
            }
            const int gt = my0 + warp + kWarps * r;
            const int nvalid = min(kTileTokens, tok1 - gt * kTileTokens);
            uint8_t *stage = ring + (warp * S + k) * STAGE_BYTES;
            uint32_t kbase = dev::smem_addr(stage);
            uint32_t vbase = kbase + TILE_BYTES;
            constexpr bool KV8_APART = KV8 && !KDIRECT;  // K and V in f16 tiles of their own
            if constexpr (KV8_APART) {
                uint8_t *cvt = smem + plan.cvt + warp * 2 * (kTileTokens * DPAD * 2);
                // both halves landed -> both f16 tiles, converted back to back; the
                // stage is then free for tile r + S
                if (!dev::mbar_wait_bounded(dev::smem_addr(&bars[(warp * S + k) * 2 + 1]), par)) {
                    fail_r = r;
                    break;
                }
                __syncwarp();  // the previous tile's reads of the f16 tiles are done
                e4m3_tile_to_f16<DPAD>(stage, cvt, lane);
                e4m3_tile_to_f16<DPAD>(stage + TILE_BYTES, cvt + kTileTokens * DPAD * 2, lane);
                __syncwarp();
                if (rn < nloc && lane == 0) {
                    issue(tmk, 0, rn, k, id_next);
                    issue(tmv, 1, rn, k, id_next);
                }
                kbase = dev::smem_addr(cvt);
                vbase = kbase + kTileTokens * DPAD * 2;
            }

            // S^T = K . q^T, two accumulator chains (even / odd k-steps)
            float sc[GN][2][4];
#pragma unroll
            for (int nt = 0; nt < GN; ++nt)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sc[nt][h2][c] = 0.f;
            if constexpr (KDIRECT) {
                // FP8 K codes straight into the A operand: per block kb of 32
                // codes a thread reads 8 codes of row tq and 8 of row tq + 8
                // (half (qd & 1) of one 16-byte chunk), one conversion per code
                // pair, and uses them as columns 2qd, 2qd+1 | 2qd+8, 2qd+9 of
                // k-steps 2kb and 2kb+1.  Quad positions 0-1 read chunk 2kb',
                // 2-3 chunk (2kb'+1) ^ 4 of the box (kb' = kb mod 4): under the
                // 128-byte swizzle the 16 lanes of each half-warp then cover the
                // 32 banks once.  q was staged in the matching column order, so
                // the sum is the same dot product over another order of d.
#pragma unroll(GN == 1 ? DPAD / 32 : 2)
                for (int kb = 0; kb < DPAD / 32; ++kb) {
                    const int qd = lane & 3;
                    const int kbp = kb & 3;
                    const int ch = (qd < 2 ? 2 * kbp : ((2 * kbp + 1) ^ 4)) ^ (tq & 7);  // swizzled 16-byte chunk
                    const uint32_t a_lo = kbase + (kb >> 2) * (kTileTokens * 128) + tq * 128 + ch * 16 + (qd & 1) * 8;
                    uint32_t w0x, w0y, w1x, w1y;
                    dev::lds_v2(a_lo, w0x, w0y);
                    dev::lds_v2(a_lo + 8 * 128, w1x, w1y);
                    uint32_t h0[4], h1[4];
                    dev::e4m3x4_to_f16x4(w0x, h0[0], h0[1]);
                    dev::e4m3x4_to_f16x4(w0y, h0[2], h0[3]);
                    dev::e4m3x4_to_f16x4(w1x, h1[0], h1[1]);
                    dev::e4m3x4_to_f16x4(w1y, h1[2], h1[3]);
#pragma unroll
                    for (int nt = 0; nt < GN; ++nt) {
                        uint32_t b0, b1, b2, b3;
                        dev::ldsm_x2(q_lm + nt * 8 * QST + (2 * kb) * 32, b0, b1);
                        dev::ldsm_x2(q_lm + nt * 8 * QST + (2 * kb + 1) * 32, b2, b3);
                        mma_16816<true>(sc[nt][0], h0[0], h1[0], h0[1], h1[1], b0, b1);
                        mma_16816<true>(sc[nt][1], h0[2], h1[2], h0[3], h1[3], b2, b3);
                    }
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    dev::ldsm_x4(kbase + (ks >> 2) * (kTileTokens * 128) + lmk_off[ks & 3], a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < GN; ++nt) {
                        uint32_t b0, b1;
                        dev::ldsm_x2(q_lm + nt * 8 * QST + ks * 32, b0, b1);
                        mma_16816<KV8>(sc[nt][ks & 1], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
            // The K half is read (every lane's ldmatrix result has been consumed by
            // an mma): refill it with tile r + S.  A read-then-overwrite by the TMA
            // needs no proxy fence once the read values are in registers.
            // (KV1BAR: refilled with the V half below.)
            if constexpr (!KV8 || (KDIRECT && !KV1BAR)) {
                if (rn < nloc) {
                    __syncwarp();
                    if (lane == 0) issue(tmk, 0, rn, k, id_next);
                }
            }

            // column softmax over the tile's tokens, base 2, tokens past the range masked
            float alpha[GN][2];
            float pv[GN][4];
#pragma unroll
            for (int nt = 0; nt < GN; ++nt) {
                float x[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int t = tq + (c >> 1) * 8;
                    const float v = (sc[nt][0][c] + sc[nt][1][c]) * scale_log2;
                    x[c] = t < nvalid ? v : kNegInf;
                }
                float cmx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    cmx[0] = fmaxf(cmx[0], __shfl_xor_sync(0xffffffffu, cmx[0], off));
                    cmx[1] = fmaxf(cmx[1], __shfl_xor_sync(0xffffffffu, cmx[1], off));
                }
                // Paged mode: the reference max of a column moves only when a
                // tile's max passes it by more than 8 (base-2 units), so most
                // tiles rescale nothing and the weights stay below 2^8 (any
                // reference gives the same m, l, o relation; the part, split and
                // merge folds use the one kept).  The tiled modes keep the true
                // running max, which their state exposes.
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float m_old = m_run[nt][c];
                    const float m_new = MODE == kModePaged ? (cmx[c] > m_old + 8.f ? cmx[c] : m_old)
                                                           : fmaxf(m_old, cmx[c]);
                    alpha[nt][c] = dev::exp2_approx(m_old - m_new);
                    const float e0 = dev::exp2_approx(x[c] - m_new);
                    const float e1 = dev::exp2_approx(x[c + 2] - m_new);
                    pv[nt][c] = e0;
                    pv[nt][c + 2] = e1;
                    l_run[nt][c] = l_run[nt][c] * alpha[nt][c] + (e0 + e1);
                    m_run[nt][c] = m_new;
                }
            }

            // P^T as the B operand of O^T += V^T P^T: pack to BF16 (high part and
            // residual) and transpose each 8x8 block in registers.
            uint32_t bh[GN][2], bl[GN][2];
#pragma unroll
            for (int nt = 0; nt < GN; ++nt)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const float e0 = pv[nt][2 * h2], e1 = pv[nt][2 * h2 + 1];
                    uint32_t hi, lo;
                    if constexpr (KV8) {
                        hi = dev::pack_f16x2(e0, e1);
                        lo = dev::pack_f16x2(e0 - dev::f16_lo_f32(hi), e1 - dev::f16_hi_f32(hi));
                    } else {
                        hi = dev::pack_bf16x2(e0, e1);
                        lo = dev::pack_bf16x2(e0 - dev::bf16_lo_f32(hi), e1 - dev::bf16_hi_f32(hi));
                    }
                    bh[nt][h2] = dev::movmatrix_trans(hi);
                    bl[nt][h2] = dev::movmatrix_trans(lo);
                }
            if constexpr (HL) {
                // lanes 16..31 hold rows g = 4..7 of the transposed blocks: give them
                // the residual of rows 0..3 instead
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const uint32_t lo_src = __shfl_sync(0xffffffffu, bl[0][h2], lane & 15);
                    bh[0][h2] = lane < 16 ? bh[0][h2] : lo_src;
                }
            }

            // rescale O^T columns whose max moved (HL: columns 4..7 follow 0..3)
            bool any = false;
#pragma unroll
            for (int nt = 0; nt < GN; ++nt) any |= (alpha[nt][0] != 1.f) | (alpha[nt][1] != 1.f);
            if (__any_sync(0xffffffffu, any)) {
#pragma unroll
                for (int nt = 0; nt < GN; ++nt) {
                    float a0 = alpha[nt][0], a1 = alpha[nt][1];
                    if constexpr (HL) {
                        const float p0 = __shfl_xor_sync(0xffffffffu, a0, 2);
                        const float p1 = __shfl_xor_sync(0xffffffffu, a1, 2);
                        if (lane & 2) {
                            a0 = p0;
                            a1 = p1;
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        o[mt][nt][0] *= a0;
                        o[mt][nt][1] *= a1;
                        o[mt][nt][2] *= a0;
                        o[mt][nt][3] *= a1;
                    }
                }
            }

            if constexpr (!KV8_APART && !KV1BAR) {
                if (!dev::mbar_wait_bounded(dev::smem_addr(&bars[(warp * S + k) * 2 + 1]), par)) {
                    fail_r = r;
                    break;
                }
            }
            // O^T += V^T . P^T  (V rows past the range may hold anything: mask them)
            auto pv_tile = [&](uint32_t mask01, uint32_t mask89) {
                if constexpr (VDIRECT) {
                    // FP8 V codes straight into the A operand V^T (d x t).  The
                    // m-tiles' rows are a permutation of d: row r of m-tile mt
                    // is d = 128*(mt/8) + 16*(r%8) + 2*(mt%8) + r/8, so that the
                    // rows tq, tq+8 this thread holds are two neighbouring codes
                    // and all its rows of a 128-code box are one 16-byte chunk
                    // of each token row.  The thread reads that chunk of its
                    // four token rows 2qd, 2qd+1, 2qd+8, 2qd+9 (chunk tq sits at
                    // tq ^ (t & 7) under the swizzle: every quarter-warp covers
                    // the 32 banks once) and pairs the tokens of each code by
                    // byte permutes: {t, t+1} of codes d, d+1 -> two f16x2.
                    const int qd = lane & 3;
#pragma unroll
                    for (int bx = 0; bx < DPAD / 128; ++bx) {
                        uint32_t R[4][4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int t = 2 * qd + (j & 1) + (j >> 1) * 8;
                            dev::lds_v4(vbase + bx * (kTileTokens * 128) + t * 128 + ((tq ^ (t & 7)) << 4),
                                        R[j][0], R[j][1], R[j][2], R[j][3]);
                        }
#pragma unroll
                        for (int m8 = 0; m8 < 8; ++m8) {
                            const int mt = bx * 8 + m8;
                            const uint32_t sel = (m8 & 1) ? 0x7362u : 0x5140u;
                            uint32_t a0, a1, a2, a3;
                            dev::e4m3x4_to_f16x4(dev::prmt(R[0][m8 >> 1], R[1][m8 >> 1], sel), a0, a1);
                            dev::e4m3x4_to_f16x4(dev::prmt(R[2][m8 >> 1], R[3][m8 >> 1], sel), a2, a3);
                            a0 &= mask01;
                            a1 &= mask01;
                            a2 &= mask89;
                            a3 &= mask89;
#pragma unroll
                            for (int nt = 0; nt < GN; ++nt) {
                                mma_16816<true>(o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
                                if constexpr (!HL) mma_16816<true>(o[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
                            }
                        }
                    }
                    return;
                }
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    dev::ldsm_x4_trans(vbase + (mt >> 2) * (kTileTokens * 128) + lmv_off[mt & 3], a0, a1, a2, a3);
                    a0 &= mask01;
                    a1 &= mask01;
                    a2 &= mask89;
                    a3 &= mask89;
#pragma unroll
                    for (int nt = 0; nt < GN; ++nt) {
                        mma_16816<KV8>(o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
                        if constexpr (!HL) mma_16816<KV8>(o[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
                    }
                }
            };
            if (nvalid == kTileTokens) {
                pv_tile(0xffffffffu, 0xffffffffu);
            } else {
                const int tv0 = (lane & 3) * 2;
                pv_tile((tv0 < nvalid ? 0x0000ffffu : 0u) | (tv0 + 1 < nvalid ? 0xffff0000u : 0u),
                        (tv0 + 8 < nvalid ? 0x0000ffffu : 0u) | (tv0 + 9 < nvalid ? 0xffff0000u : 0u));
            }
            // the V half is read: refill it with tile r + S (KV1BAR: both halves)
            if constexpr (!KV8 || VDIRECT) {
                if (rn < nloc) {
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (KV1BAR)
                            issue_kv(rn, k, id_next);
                        else
                            issue(tmv, 1, rn, k, id_next);
                    }
                }
            }
            if (++k == S) {
                k = 0;
                par ^= 1u;
            }
        }
        if (fail_r >= 0) {
            // A bounded wait ran out.  Record it and drain (bounded) whatever this
            // warp may still have in flight before the ring is reused.
            if (lane == 0) dev::flag_status(p.status, kDevWaitTimeout);
            const int last = fail_r + S + 1 < nloc ? fail_r + S + 1 : nloc;
            for (int r = fail_r; r < last; ++r)
                for (int h = 0; h < (KV1BAR ? 1 : 2); ++h)
                    dev::mbar_wait_bounded(dev::smem_addr(&bars[(warp * S + (rr + r) % S) * 2 + h]),
                                           ((rr + r) / S) & 1, 100000000ull);
            k = (rr + nloc) % S;  // as if every tile had gone through
            par = ((rr + nloc) / S) & 1;
        }
        rr += nloc;
        k_next = k;
        par_next = par;

        // ---- warp merge of the part (fixed warp order) -----------------------------
        // column sums over the tokens of all lanes of a column
#pragma unroll
        for (int nt = 0; nt < GN; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
                    l_run[nt][c] += __shfl_xor_sync(0xffffffffu, l_run[nt][c], off);
        if constexpr (HL) {
            // columns 0..3 = high part + residual held in columns 4..7
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) o[mt][0][c] += __shfl_xor_sync(0xffffffffu, o[mt][0][c], 2);
        }
        __syncthreads();  // every warp is done with the ring; reuse it for the merge
        if (tq == 0) {
#pragma unroll
            for (int nt = 0; nt < GN; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int g = nt * 8 + gq + c;
                    if (g - nt * 8 < GCOLS) {
                        wm[warp * RT + g] = m_run[nt][c];
                        wl[warp * RT + g] = l_run[nt][c];
                    }
                }
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int nt = 0; nt < GN; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // row slot mt*16 + r of the accumulators (r = tq, tq + 8): d itself, or
                    // with FP8 V read directly a permutation of d that the sum below undoes
                    // (stored by slot, a warp's stores hit distinct banks)
                    const int g = nt * 8 + gq + (c & 1);
                    const int slot = mt * 16 + tq + (c >> 1) * 8;
                    if (g - nt * 8 < GCOLS) wo[(warp * RT + g) * OSTRIDE + slot] = o[mt][nt][c];
                }
        __syncthreads();

        if constexpr (MODE == kModePaged && !PACKED) {
            if (solo) {
                // A unit of one part: each output pair straight from the warp
                // partials, with the operations, in the order, of the general
                // path below (part max, warp weights, sums in warp order; then
                // the epilogue's scale and division), and no fold or hand-off.
                // (Not compiled into the packed pass, whose units are rarely
                // that short: measured slower there.)
                dev::griddep_launch_dependents();
                const int halfD = D / 2;
                for (int e = tid; e < Gt * halfD; e += kThreads) {
                    const int g = e / halfD;
                    const int d = (e - g * halfD) * 2;
                    // accumulator slots of d and d + 1 (the inverse of the FP8
                    // direct-V permutation of d, where d + 1 sits 8 slots on)
                    int sl0 = d, sl1 = d + 1;
                    if constexpr (VDIRECT) {
                        const int r = d & 127;
                        sl0 = (d - r) + (r >> 4) + 16 * ((r >> 1) & 7);
                        sl1 = sl0 + 8;
                    }
                    float M = kNegInf;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * RT + g]);
                    float Lsum = 0.f, acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        const float mw = wm[w * RT + g];
                        const float wt = mw == kNegInf ? 0.f : dev::exp2_approx(mw - M);
                        Lsum += wt * wl[w * RT + g];
                        acc0 += wt * wo[(w * RT + g) * OSTRIDE + sl0];
                        acc1 += wt * wo[(w * RT + g) * OSTRIDE + sl1];
                    }
                    const long long row = static_cast<long long>(s) * Hq + h0 + g;
                    if constexpr (KV8) {  // V = code value * v_scale
                        acc0 *= p.v_scale;
                        acc1 *= p.v_scale;
                    }
                    if (direct) {
                        const bool pos = Lsum > 0.f;
                        const __nv_bfloat162 v = __floats2bfloat162_rn(pos ? __fdiv_rn(acc0, Lsum) : 0.f,
                                                                       pos ? __fdiv_rn(acc1, Lsum) : 0.f);
                        *reinterpret_cast<__nv_bfloat162 *>(p.out + row * D + d) = v;
                    } else {
                        const long long slot_row = row * p.num_splits + split;
                        *reinterpret_cast<float2 *>(p.ws_o + slot_row * D + d) = make_float2(acc0, acc1);
                        if (d == 0) {
                            p.ws_ml[slot_row * 2 + 0] = M;
                            p.ws_ml[slot_row * 2 + 1] = Lsum;
                        }
                    }
                }
                return;
            }
        }

        // part statistics of each valid row: max, warp weights, sum
        if (tid < Gt) {
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * RT + tid]);
            float Lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = wm[w * RT + tid];
                const float wt = mw == kNegInf ? 0.f : dev::exp2_approx(mw - M);
                ww[w * RT + tid] = wt;
                Lsum += wt * wl[w * RT + tid];
            }
            cm[tid] = M;
            cl[tid] = Lsum;
        }
        __syncthreads();
        // the part's o: warp partials weighted and summed in warp order (walked by
        // slot; slot mt*16 + r holds d = 128*(mt/8) + 16*(r%8) + 2*(mt%8) + r/8
        // when FP8 V was read directly, else d = slot)
        for (int e = tid; e < Gt * DPAD; e += kThreads) {
            const int g = e / DPAD, sl = e - g * DPAD;
            const int d = VDIRECT ? (sl >> 7) * 128 + 16 * (sl & 7) + 2 * ((sl >> 4) & 7) + ((sl >> 3) & 1) : sl;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += ww[w * RT + g] * wo[(w * RT + g) * OSTRIDE + sl];
            co[g * OSTRIDE + d] = acc;
        }
        if (C == 1 && !solo) {
            // fold the part into the running result, in part order
            __syncthreads();
            if (tid < Gt) {
                float Mn, fa, fb;
                dev::fold_factors(rM[tid], cm[tid], Mn, fa, fb);
                rL[tid] = dev::fold_value(rL[tid], fa, cl[tid], fb);
                rM[tid] = Mn;
                fx[tid * 4 + 2] = fa;
                fx[tid * 4 + 3] = fb;
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < RACC; ++i) {
                const int e = tid + i * kThreads;
                const int g = e / DPAD, d = e - g * DPAD;
                if (g < Gt) racc[i] = dev::fold_value(racc[i], fx[g * 4 + 2], co[g * OSTRIDE + d], fx[g * 4 + 3]);
            }
            __syncthreads();  // the ring (and co over it) is free for the next part
        }
    }

    // Programmatic dependent launch: the next kernel in the stream may start
    // launching once every CTA of this grid has streamed its tiles (it waits,
    // with griddepcontrol.wait, for this grid to finish before it uses any
    // memory).  Triggering here rather than at the start lets its CTAs take
    // the SMs this grid is leaving, in launch order, instead of whatever slots
    // happen to be free early.
    dev::griddep_launch_dependents();

    // ---- the unit's result: rows dealt to the active ranks round-robin --------
    // Row g is owned by rank g % V and is the left fold, in part order, of the
    // parts' results (cluster == 1: already folded into the running result).
    // The epilogue then writes the output, the split's partial, or folds into
    // the tiled state.
    // When every rank of the cluster holds a part, the hand-offs are the
    // hardware cluster barrier; otherwise the idle ranks have left and the
    // active ones hand off through the ready / done mbarriers.
    cg::cluster_group cluster = cg::this_cluster();
    const bool multi = C > 1 && !solo;             // parts on several ranks
    const int RK = multi ? V : 1;                  // ranks rows are dealt to
    const int nown = multi ? min(V, Gt) : 1;       // ranks that own a row
    const bool full = multi && V == C;
    if (full) {
        dev::cluster_wait();  // (the arrive at the start)
        cluster.sync();       // every part is published
    } else if (multi) {
        dev::cluster_wait();  // the peers' barriers are initialised
        __syncthreads();      // this part's co, cm and cl are complete
        if (tid == 0) {
            // release at cluster scope: the CTA's writes above (ordered before
            // this thread by the barrier) are visible to an owner that acquires
            for (int r = 0; r < nown; ++r)
                dev::mbar_arrive_cluster(dev::map_to_rank(dev::smem_addr(bar_ready), r));
            if (part < nown && V < kMaxParts) dev::mbar_arrive_count(dev::smem_addr(bar_ready), kMaxParts - V);
            if (nown < kMaxParts) dev::mbar_arrive_count(dev::smem_addr(bar_done), kMaxParts - nown);
        }
        if (part < nown) {
            if (!dev::mbar_wait_cluster_bounded(dev::smem_addr(bar_ready), 0) && tid == 0)
                dev::flag_status(p.status, kDevWaitTimeout);
        }
    } else {
        // the folded o goes to shared memory for the epilogue (the ring is
        // free); a single part's is there already
        if (!solo) {
#pragma unroll
            for (int i = 0; i < RACC; ++i) {
                const int e = tid + i * kThreads;
                const int g = e / DPAD, d = e - g * DPAD;
                if (g < Gt) co[g * OSTRIDE + d] = racc[i];
            }
        }
        __syncthreads();
    }
    const int nmine = Gt > part ? (Gt - part + RK - 1) / RK : 0;  // rows g = part + i*RK
    // per-row factors: fx[i] = {M, L, a, b} of the epilogue; fr[i] = fold factors
    if (tid < nmine) {
        const int g = part + tid * RK;
        float M = kNegInf, Lsum = 0.f;
        if (multi) {
            for (int jj = 0; jj < V; ++jj) {
                const float mj = cluster.map_shared_rank(cm, jj)[g];
                const float lj = cluster.map_shared_rank(cl, jj)[g];
                float Mn, fa, fb;
                dev::fold_factors(M, mj, Mn, fa, fb);
                Lsum = dev::fold_value(Lsum, fa, lj, fb);
                M = Mn;
                fr[tid * 2 * kMaxParts + 2 * jj + 0] = fa;
                fr[tid * 2 * kMaxParts + 2 * jj + 1] = fb;
            }
        } else if (!solo) {
            M = rM[g];
            Lsum = rL[g];
        } else {
            M = cm[g];
            Lsum = cl[g];
        }
        const long long row = static_cast<long long>(s) * Hq + h0 + g;
        float fa = 0.f, fb = 0.f;
        if constexpr (MODE == kModePaged || RUN) {
            // a split's, or a fused run's call's, partial [o, m, l]
            if (RUN || !direct) {
                p.ws_ml[(row * p.num_splits + split) * 2 + 0] = M;
                p.ws_ml[(row * p.num_splits + split) * 2 + 1] = Lsum;
            } else {
                fb = Lsum > 0.f ? 1.f : 0.f;
            }
        } else {
            // TiledAttention::step_tile: fold into the running state (the fused
            // run's merge replays exactly this, in call order)
            const float m_old = p.st_m[row];
            const float m_new = fmaxf(m_old, M);
            fa = m_old == kNegInf ? 0.f : dev::exp2_approx(m_old - m_new);
            fb = M == kNegInf ? 0.f : dev::exp2_approx(M - m_new);
            p.st_l[row] = dev::fold_value(p.st_l[row], fa, Lsum, fb);
            p.st_m[row] = m_new;
        }
        fx[tid * 4 + 0] = M;
        fx[tid * 4 + 1] = Lsum;
        fx[tid * 4 + 2] = fa;
        fx[tid * 4 + 3] = fb;
    }
    __syncthreads();
    // elements (row i of this rank, column pair d)
    const int halfD = D / 2;
    for (int e = tid; e < nmine * halfD; e += kThreads) {
        const int i = e / halfD;
        const int d = (e - i * halfD) * 2;
        const int g = part + i * RK;
        float acc0 = 0.f, acc1 = 0.f;
        if (multi) {
            float v0[kMaxParts], v1[kMaxParts];
#pragma unroll
            for (int jj = 0; jj < kMaxParts; ++jj) {
                if (jj < V) {
                    const float2 v = *reinterpret_cast<const float2 *>(
                        cluster.map_shared_rank(co, jj) + g * OSTRIDE + d);
                    v0[jj] = v.x;
                    v1[jj] = v.y;
                }
            }
#pragma unroll
            for (int jj = 0; jj < kMaxParts; ++jj) {
                if (jj < V) {
                    const float fa = fr[i * 2 * kMaxParts + 2 * jj + 0];
                    const float fb = fr[i * 2 * kMaxParts + 2 * jj + 1];
                    acc0 = dev::fold_value(acc0, fa, v0[jj], fb);
                    acc1 = dev::fold_value(acc1, fa, v1[jj], fb);
                }
            }
        } else {
            acc0 = co[g * OSTRIDE + d];
            acc1 = co[g * OSTRIDE + d + 1];
        }
        const long long row = static_cast<long long>(s) * Hq + h0 + g;
        if constexpr (KV8) {  // V = code value * v_scale
            acc0 *= p.v_scale;
            acc1 *= p.v_scale;
        }
        if constexpr (MODE == kModePaged || RUN) {
            if (!RUN && direct) {
                const float Lsum = fx[i * 4 + 1];
                const bool pos = fx[i * 4 + 3] > 0.f;
                const __nv_bfloat162 v = __floats2bfloat162_rn(pos ? __fdiv_rn(acc0, Lsum) : 0.f,
                                                               pos ? __fdiv_rn(acc1, Lsum) : 0.f);
                *reinterpret_cast<__nv_bfloat162 *>(p.out + row * D + d) = v;
            } else {
                *reinterpret_cast<float2 *>(p.ws_o + (row * p.num_splits + split) * D + d) =
                    make_float2(acc0, acc1);
            }
        } else {
            const float fa = fx[i * 4 + 2], fb = fx[i * 4 + 3];
            float2 *so = reinterpret_cast<float2 *>(p.st_o + row * D + d);
            float2 cur = *so;
            cur.x = dev::fold_value(cur.x, fa, acc0, fb);
            cur.y = dev::fold_value(cur.y, fa, acc1, fb);
            *so = cur;
        }
    }
    if (full) {
        cluster.sync();  // peers keep their shared memory until every rank has read it
    } else if (multi) {
        // Tell every active rank that this owner has read it (relaxed: the
        // reads have returned, and the output stores need not drain first);
        // keep this CTA's shared memory alive until its own readers are done.
        __syncthreads();
        if (tid == 0) {
            if (part < nown)
                for (int r = 0; r < V; ++r)
                    dev::mbar_arrive_cluster_relaxed(dev::map_to_rank(dev::smem_addr(bar_done), r));
            if (!dev::mbar_wait_cluster_bounded(dev::smem_addr(bar_done), 0))
                dev::flag_status(p.status, kDevWaitTimeout);
        }
    }
}

}  // namespace pd
