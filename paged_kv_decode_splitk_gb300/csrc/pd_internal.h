// pd_internal.h -- declarations shared by the host side (pd_api.cu) and the
// kernel translation units of libpd.  Not installed; the public ABI is pd.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pd {

// Warps of a unit CTA.  Each warp folds every kWarps-th 16-token tile of the
// CTA's range; the warps' states are then merged in warp order.  It is part of
// the arithmetic (it fixes the summation order), so it is a build constant.
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileTokens = 16;   // tokens per mma tile (the K/V stage)
constexpr int kBoxCols = 64;      // BF16 columns per TMA box (128 bytes, 128B swizzle)
constexpr int kMaxStagesPerWarp = 8;
constexpr int kMaxParts = 8;   // parts of a unit (and CTAs of a unit cluster) at most
constexpr int kLptMaxSeqs = 64;

// Tokens per split (module description of attn_splitk: the split size is
// floored at PD_MIN_KV_PER_SPLIT from the sequence's own length), rounded up
// to whole cache blocks.  Shared by the host ABI and every kernel so that the
// split geometry is one function of (context_len, num_splits, block_size).
__host__ __device__ inline int split_chunk_tokens(int context_len, int num_splits, int block_size,
                                                  int min_kv_per_split) {
    int per = context_len > 0 ? (context_len + num_splits - 1) / num_splits : 0;
    int c = per > min_kv_per_split ? per : min_kv_per_split;
    return (c + block_size - 1) / block_size * block_size;
}

__host__ __device__ inline int splits_used(int context_len, int chunk) {
    return context_len > 0 ? (context_len + chunk - 1) / chunk : 0;
}

// Tiles (16 tokens each) a part of a unit's range aims for: the range is cut
// into ceil(tiles / kPartTiles) parts, at most max_parts (the packed pass:
// kPartTilesPacked).
constexpr int kPartTiles = 32;
constexpr int kPartTilesPacked = 24;

// Division by a divisor fixed for a launch, as a multiply-high, an add and a
// shift (T. Granlund and P. L. Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994, section 4): for a divisor d >= 1 let
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, which is below 2^32
// because d > 2^(l-1).  Then floor(n / d) = (mulhi(n, m) + n) >> l for every
// 0 <= n < 2^32, and for n < 2^31 the sum cannot overflow 32 bits.  The
// kernels use it for the split geometry and the unit decode, whose quotients
// must equal the plain integer division's.
struct FastDiv {
    uint32_t d;  // the divisor
    uint32_t m;  // multiplier
    uint32_t l;  // shift
};

inline FastDiv make_fastdiv(int d) {
    FastDiv f;
    f.d = static_cast<uint32_t>(d < 1 ? 1 : d);
    f.l = 0;
    while ((uint64_t{1} << f.l) < f.d) ++f.l;
    f.m = static_cast<uint32_t>((((uint64_t{1} << f.l) - f.d) << 32) / f.d + 1);
    return f;
}

// floor(n / f.d) for 0 <= n < 2^31.
__host__ __device__ inline int fast_div(int n, const FastDiv &f) {
    const uint32_t u = static_cast<uint32_t>(n);
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi(u, f.m);
#else
    const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(u) * f.m) >> 32);
#endif
    return static_cast<int>((t + u) >> f.l);
}

// split_chunk_tokens with the split count and the block size as FastDiv
// (same value for every argument the kernels pass: 0 <= context_len and
// context_len + num_splits, chunk + block_size below 2^31).
__host__ __device__ inline int split_chunk_tokens_fd(int context_len, const FastDiv &num_splits,
                                                     const FastDiv &block_size, int min_kv_per_split) {
    const int n = static_cast<int>(num_splits.d), bs = static_cast<int>(block_size.d);
    int per = context_len > 0 ? fast_div(context_len + n - 1, num_splits) : 0;
    int c = per > min_kv_per_split ? per : min_kv_per_split;
    return fast_div(c + bs - 1, block_size) * bs;
}

enum UnitMode : int {
    kModePaged = 0,     // pd_decode_attn: block_table gather, split ranges, out / workspace
    kModeTiled = 1,     // pd_tiled_step: tile list, fold into the running state
    kModeTiledRun = 2,  // pd_tiled_run: every call's tile list at once, one partial per call
};

// Sources (step_tile calls) one fused pd_tiled_run launch serves at most.
constexpr int kMaxRunSources = 8;

// The K and V tensor maps a launch reads: one pair, or one per source of a
// fused tiled run.  Passed by value as a kernel parameter.
template <int N>
struct KvMaps {
    CUtensorMap k[N];
    CUtensorMap v[N];
};

// Everything a unit kernel reads besides the two tensor maps.
struct UnitParams {
    const __nv_bfloat16 *q;  // [S, Hq, D]
    // paged mode
    const int32_t *block_table;  // [S, max_blocks_per_seq]
    const int32_t *context_lens; // [S]
    int max_blocks_per_seq;
    int num_blocks;
    int num_splits;
    int min_kv_per_split;
    // tiled mode
    const int32_t *tile_blocks;  // [S, tile_capacity]
    const int32_t *tile_counts;  // [S]
    int tile_capacity;
    int last_valid;
    // fused tiled run: per source (step_tile call) c < num_sources
    int num_sources;
    const int32_t *src_blocks[kMaxRunSources];  // [S, tile_capacity]
    const int32_t *src_counts[kMaxRunSources];  // [S]
    int src_last_valid[kMaxRunSources];
    int src_tok_dim[kMaxRunSources];
    // outputs
    __nv_bfloat16 *out;  // [S, Hq, D]
    float *ws_o;         // [S, Hq, N, D]   unnormalised o of each split
    float *ws_ml;        // [S, Hq, N, 2]   (m, l) of each split, m in log2 units
    float *st_m;         // tiled running state [max_seqs, Hq] (log2 units)
    float *st_l;
    float *st_o;         // [max_seqs, Hq, D]
    // shape
    int num_seqs, num_q_heads, num_kv_heads, group, head_dim, block_size;
    int qtiles;       // CTAs per (s, kvh): ceil(group / rows per CTA)
    FastDiv fd_split;    // num_splits (paged mode; 1 otherwise): split geometry and unit decode
    FastDiv fd_bs;       // block_size
    FastDiv fd_kvh;      // num_kv_heads
    int cluster;      // CTAs per unit: 1 (parts in sequence) or max_parts (one part per CTA)
    int max_parts;    // parts a unit's range is cut into at most
    int stages;       // pipeline stages per warp
    int lpt;          // paged mode: serve sequences longest first (needs num_seqs <= kLptMaxSeqs)
    int prefetch_tiles;  // first tiles of the CTA's part prefetched into L2 before the wait (0: none)
    int tok_dim;      // tensor-map dimension of the token coordinate (1 or 2)
    float scale_log2; // softmax scale * log2(e) (times k_scale for an FP8 cache)
    float v_scale;    // FP8 cache: V = code value * v_scale (unused for BF16)
    unsigned int *status;  // device status word (PD_DEV_* flags)
};

struct MergeParams {
    const int32_t *context_lens;
    const float *ws_o;
    const float *ws_ml;
    __nv_bfloat16 *out;
    int num_seqs, num_q_heads, head_dim, num_splits, block_size, min_kv_per_split;
    int max_tokens;  // max_blocks_per_seq * block_size (context lengths are clamped to it)
    FastDiv fd_hq, fd_split, fd_bs;  // num_q_heads, num_splits, block_size
};

// Record an error message for pd_last_error() and return `code`.
int report_error(int code, const char *message);

// Dynamic shared memory a unit CTA needs (kv8: FP8 cache).
int unit_smem_bytes(int dpad, int rows, int stages, bool kv8);

// Kernel launchers (defined in the per-head-dim translation units).
// layout: 0 = choose from occupancy, 1 = one CTA per unit, 2 = one CTA per part.
// p.stages is the ring depth per warp of a single-wave launch, stages_seq that
// of a launch of several waves of one-CTA units (both must fit the device).
// tmk / tmv: one tensor map each, or p.num_sources of them for a fused tiled run.
template <int DPAD, int GN, bool HL, int MODE, bool PACKED, bool KV8>
cudaError_t launch_unit(const CUtensorMap *tmk, const CUtensorMap *tmv, const UnitParams &p,
                        long long units, int stages_seq, cudaStream_t stream, int layout);

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream, bool programmatic);

// Fold of a fused tiled run's per-call partials, in call order, into the
// running state (from begin's (-inf, 0, 0)), then out = o / l.
struct RunMergeParams {
    const float *ws_o;   // [rows, num_sources, D]
    const float *ws_ml;  // [rows, num_sources, 2]
    const int32_t *src_counts[kMaxRunSources];
    float *st_m, *st_l, *st_o;
    __nv_bfloat16 *out;
    int num_seqs, num_q_heads, head_dim, num_sources, tile_capacity;
};
cudaError_t launch_tiled_run_merge(const RunMergeParams &p, cudaStream_t stream);
cudaError_t launch_tiled_begin(float *m, float *l, float *o, int rows, int head_dim,
                               cudaStream_t stream);
cudaError_t launch_tiled_finalize(const float *l, const float *o, __nv_bfloat16 *out, int rows,
                                  int head_dim, cudaStream_t stream);

// Compile-time values the packed kernel is instantiated with (the kernels'
// own copy of the pack width and head dim, checked against pd.h).
int kernel_pack_width();
int kernel_pack_head_dim();

}  // namespace pd
