// pd_small.cu -- the light kernels of libpd: the split-K merge pass and the
// tiled begin / finalize passes.
#include <cuda_bf16.h>
#include <stdint.h>

#include "pd_device.cuh"
#include "pd_internal.h"

namespace pd {

namespace {

constexpr int kMergeWarps = 8;

// Merge pass (Module attn_splitk page: the split-K workspace of [o, m, l]
// slots and the non-associative merge).  One warp per (sequence, q head)
// folds the non-empty splits in split order with the online rule
//   M' = max(M, m_i),  L = L 2^(M - M') + l_i 2^(m_i - M'),  O likewise,
// and writes out = O / L as BF16 (0 when L is 0).  All loads of a row are
// independent of the arithmetic, so they are issued together.  Sequences with
// at most one non-empty split were written by the partial pass directly and
// are skipped here.
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const __grid_constant__ MergeParams p) {
    const float kNegInf = -__int_as_float(0x7f800000);
    dev::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
    if (row >= static_cast<long long>(p.num_seqs) * p.num_q_heads) return;
    const int s = static_cast<int>(row / p.num_q_heads);
    int L = p.context_lens[s];
    L = L < 0 ? 0 : (L > p.max_tokens ? p.max_tokens : L);
    const int chunk = split_chunk_tokens(L, p.num_splits, p.block_size, p.min_kv_per_split);
    const int nsu = splits_used(L, chunk);
    if (nsu <= 1) return;
    dev::griddep_wait();  // the partial pass's workspace is complete and visible

    const float *ml = p.ws_ml + row * p.num_splits * 2;
    const int D = p.head_dim;
    for (int d0 = lane * 4; d0 < D; d0 += 128) {
        float M = kNegInf, Lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int kBatch = 4;
        for (int i0 = 0; i0 < nsu; i0 += kBatch) {
            float mi[kBatch], li[kBatch];
            float4 oi[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = i0 + j;
                if (i < nsu) {
                    const float2 v = *reinterpret_cast<const float2 *>(ml + 2 * i);
                    mi[j] = v.x;
                    li[j] = v.y;
                    oi[j] = *reinterpret_cast<const float4 *>(p.ws_o + (row * p.num_splits + i) * D + d0);
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (i0 + j < nsu && mi[j] != kNegInf) {
                    const float Mn = fmaxf(M, mi[j]);
                    const float a = M == kNegInf ? 0.f : dev::exp2_approx(M - Mn);
                    const float b = dev::exp2_approx(mi[j] - Mn);
                    Lsum = Lsum * a + li[j] * b;
                    acc.x = acc.x * a + oi[j].x * b;
                    acc.y = acc.y * a + oi[j].y * b;
                    acc.z = acc.z * a + oi[j].z * b;
                    acc.w = acc.w * a + oi[j].w * b;
                    M = Mn;
                }
            }
        }
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
    const long long rows = static_cast<long long>(p.num_seqs) * p.num_q_heads;
    if (rows == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps));
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
