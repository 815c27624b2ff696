// pd_small.cu -- the light kernels of libpd: the split-K merge pass and the
// tiled begin / finalize passes.
#include <cuda_bf16.h>
#include <stdint.h>

#include "pd_device.cuh"
#include "pd_internal.h"
#include "pd.h"

namespace pd {

namespace {

constexpr int kMergeWarps = 8;
constexpr int kMergeCols = 128;   // columns of a row one warp merges (4 per lane)
constexpr int kMergeBatch = 16;   // splits whose partials are loaded together
static_assert(PD_MAX_HEAD_DIM <= 2 * kMergeCols, "a row is at most two warps' columns");

// Merge pass (Module attn_splitk page: the split-K workspace of [o, m, l]
// slots and the non-associative merge).  One warp per (sequence, q head, 128
// columns) folds the non-empty splits in split order with the online rule
//   M' = max(M, m_i),  L = L 2^(M - M') + l_i 2^(m_i - M'),  O likewise,
// and writes out = O / L as BF16 (0 when L is 0).  The partials of up to 16
// splits and the context length are loaded in one go, before the length says
// which splits are non-empty (every slot of the workspace is in bounds; slots
// past the non-empty splits are read and ignored), so the pass costs one
// round trip to memory; the row's sequence is found before the wait on the
// partial pass, and the split geometry divides by multiply-highs (FastDiv).
// Split i is non-empty when i * chunk < L.  Sequences with at most one
// non-empty split were written by the partial pass directly and are left
// alone here.
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const __grid_constant__ MergeParams p) {
    const float kNegInf = -__int_as_float(0x7f800000);
    dev::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.head_dim;
    const int N = p.num_splits;
    const int chunks = D > kMergeCols ? 2 : 1;  // head_dim <= PD_MAX_HEAD_DIM = 2 * kMergeCols
    const long long item = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
    if (item >= static_cast<long long>(p.num_seqs) * p.num_q_heads * chunks) return;
    const long long row = item >> (chunks - 1);
    const int d0 = static_cast<int>(item - row * chunks) * kMergeCols + lane * 4;
    const bool cols = d0 < D;  // D is a multiple of 8: the lane's 4 columns are all in range
    const int s = row < 0x7fffffffLL ? fast_div(static_cast<int>(row), p.fd_hq)
                                     : static_cast<int>(row / p.num_q_heads);
    const float *ml = p.ws_ml + row * N * 2;
    const float *ob = p.ws_o + row * N * D + d0;
    // Wait before any global read: the partial pass may have started before the
    // kernel ahead of it (which may write context_lens) finished, and waiting
    // for the partial pass's completion covers that kernel too.
    dev::griddep_wait();
    int L = p.context_lens[s];

    float M = kNegInf, Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    long long chunk = -1;
    for (int i0 = 0; i0 < N; i0 += kMergeBatch) {
        float4 oi[kMergeBatch];
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j)
            oi[j] = (cols && i0 + j < N) ? *reinterpret_cast<const float4 *>(ob + static_cast<long long>(i0 + j) * D)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        // lane j holds (m, l) of split i0 + j
        float2 mlj = make_float2(kNegInf, 0.f);
        if (lane < kMergeBatch && i0 + lane < N) mlj = *reinterpret_cast<const float2 *>(ml + 2 * (i0 + lane));
        if (chunk < 0) {
            L = L < 0 ? 0 : (L > p.max_tokens ? p.max_tokens : L);
            chunk = split_chunk_tokens_fd(L, p.fd_split, p.fd_bs, p.min_kv_per_split);
            if (L <= chunk) return;  // at most one non-empty split: written directly
        }
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j) {
            const float mi = __shfl_sync(0xffffffffu, mlj.x, j);
            const float li = __shfl_sync(0xffffffffu, mlj.y, j);
            if ((i0 + j) * chunk < L && mi != kNegInf) {
                const float Mn = fmaxf(M, mi);
                const float a = M == kNegInf ? 0.f : dev::exp2_approx(M - Mn);
                const float b = dev::exp2_approx(mi - Mn);
                Lsum = Lsum * a + li * b;
                acc.x = acc.x * a + oi[j].x * b;
                acc.y = acc.y * a + oi[j].y * b;
                acc.z = acc.z * a + oi[j].z * b;
                acc.w = acc.w * a + oi[j].w * b;
                M = Mn;
            }
        }
        if ((i0 + kMergeBatch) * chunk >= L) break;  // the rest are empty splits
    }
    if (!cols) return;
    const bool pos = Lsum > 0.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(pos ? __fdiv_rn(acc.x, Lsum) : 0.f,
                                              pos ? __fdiv_rn(acc.y, Lsum) : 0.f);
    __nv_bfloat162 hi = __floats2bfloat162_rn(pos ? __fdiv_rn(acc.z, Lsum) : 0.f,
                                              pos ? __fdiv_rn(acc.w, Lsum) : 0.f);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p.out + row * D + d0) = pk;
}

// A fused tiled run's fold (tiled_attention.rs page: begin_step, one step_tile
// per call, finalize): each row starts from begin's (-inf, 0, 0), folds the
// calls' partials in call order with the same pinned rounding as step_tile's
// own fold, skipping calls whose tile held no block, writes the state and
// then out = o / l as BF16 (0 where l is 0), as finalize does.  One warp per
// (row, 128 columns); every load of a row is issued together.
__global__ void __launch_bounds__(kMergeWarps * 32) tiled_run_merge_kernel(const __grid_constant__ RunMergeParams p) {
    const float kNegInf = -__int_as_float(0x7f800000);
    dev::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.head_dim;
    const int T = p.num_sources;
    const int chunks = D > kMergeCols ? 2 : 1;  // head_dim <= PD_MAX_HEAD_DIM = 2 * kMergeCols
    const long long item = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
    if (item >= static_cast<long long>(p.num_seqs) * p.num_q_heads * chunks) return;
    const long long row = item >> (chunks - 1);
    const int chunk = static_cast<int>(item - row * chunks);
    const int d0 = chunk * kMergeCols + lane * 4;
    const bool cols = d0 < D;  // D is a multiple of 8: the lane's 4 columns are all in range
    const int s = static_cast<int>(row / p.num_q_heads);  // (launch geometry: before the wait)
    dev::griddep_wait();  // the unit pass's partials are complete and visible
    int cnt[kMaxRunSources];
    float2 mli[kMaxRunSources];
    float4 oi[kMaxRunSources];
#pragma unroll
    for (int c = 0; c < kMaxRunSources; ++c) {
        if (c < T) {
            cnt[c] = p.src_counts[c][s];
            mli[c] = *reinterpret_cast<const float2 *>(p.ws_ml + (row * T + c) * 2);
            oi[c] = cols ? *reinterpret_cast<const float4 *>(p.ws_o + (row * T + c) * D + d0)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float m = kNegInf, l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMaxRunSources; ++c) {
        if (c < T && cnt[c] > 0) {
            const float M = mli[c].x;
            const float m_new = fmaxf(m, M);
            const float fa = m == kNegInf ? 0.f : dev::exp2_approx(m - m_new);
            const float fb = M == kNegInf ? 0.f : dev::exp2_approx(M - m_new);
            l = dev::fold_value(l, fa, mli[c].y, fb);
            o.x = dev::fold_value(o.x, fa, oi[c].x, fb);
            o.y = dev::fold_value(o.y, fa, oi[c].y, fb);
            o.z = dev::fold_value(o.z, fa, oi[c].z, fb);
            o.w = dev::fold_value(o.w, fa, oi[c].w, fb);
            m = m_new;
        }
    }
    if (chunk == 0 && lane == 0) {
        p.st_m[row] = m;
        p.st_l[row] = l;
    }
    if (!cols) return;
    *reinterpret_cast<float4 *>(p.st_o + row * D + d0) = o;
    const bool pos = l > 0.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(pos ? __fdiv_rn(o.x, l) : 0.f, pos ? __fdiv_rn(o.y, l) : 0.f);
    __nv_bfloat162 hi = __floats2bfloat162_rn(pos ? __fdiv_rn(o.z, l) : 0.f, pos ? __fdiv_rn(o.w, l) : 0.f);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p.out + row * D + d0) = pk;
}

// TiledAttention::begin_step: (m, l, o) <- (-inf, 0, 0) over `rows` rows.
__global__ void tiled_begin_kernel(float *m, float *l, float *o, long long rows, long long n_o) {
    const float kNegInf = -__int_as_float(0x7f800000);
    dev::griddep_launch_dependents();
    dev::griddep_wait();
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_o;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        o[i] = 0.f;
        if (i < rows) {
            m[i] = kNegInf;
            l[i] = 0.f;
        }
    }
}

// TiledAttention::finalize: out = o / l as BF16, 0 where l is 0.
__global__ void tiled_finalize_kernel(const float *l, const float *o, __nv_bfloat16 *out,
                                      long long n, int head_dim) {
    dev::griddep_launch_dependents();
    dev::griddep_wait();
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float lv = l[i / head_dim];
        out[i] = __float2bfloat16_rn(lv > 0.f ? __fdiv_rn(o[i], lv) : 0.f);
    }
}

int grid_for(long long n, int threads) {
    long long g = (n + threads - 1) / threads;
    if (g > 152 * 32) g = 152 * 32;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream, bool programmatic) {
    const long long items = static_cast<long long>(p.num_seqs) * p.num_q_heads *
                            ((p.head_dim + kMergeCols - 1) / kMergeCols);
    if (items == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((items + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

cudaError_t launch_tiled_run_merge(const RunMergeParams &p, cudaStream_t stream) {
    const long long items = static_cast<long long>(p.num_seqs) * p.num_q_heads *
                            ((p.head_dim + kMergeCols - 1) / kMergeCols);
    if (items == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((items + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tiled_run_merge_kernel, p);
}

cudaError_t launch_tiled_begin(float *m, float *l, float *o, int rows, int head_dim,
                               cudaStream_t stream) {
    const long long n_o = static_cast<long long>(rows) * head_dim;
    if (n_o == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_for(n_o, 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tiled_begin_kernel, m, l, o, static_cast<long long>(rows), n_o);
}

cudaError_t launch_tiled_finalize(const float *l, const float *o, __nv_bfloat16 *out, int rows,
                                  int head_dim, cudaStream_t stream) {
    const long long n = static_cast<long long>(rows) * head_dim;
    if (n == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_for(n, 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tiled_finalize_kernel, l, o, out, n, head_dim);
}

}  // namespace pd
