// pd_unit.cuh -- the unit kernel: one (sequence, KV head, split) of paged-decode
// attention, serving a whole group of query heads from one read of K and V.
//
// What a unit computes (Module attn_splitk page: split-K partials kept as
// [o, m, l]; tiled_attention.rs page: the running (m, l, o) fold):
//   for the query rows g of the group and the tokens t of the unit's range,
//     x[g,t] = (q[g] . K[t]) * inv_sqrt_d
//     m[g]   = max_t x[g,t],  l[g] = sum_t e^(x[g,t]-m[g]),  o[g] = sum_t e^(x[g,t]-m[g]) V[t]
//   (kept internally in base-2 units: m is max_t x[g,t]*log2(e)).
//
// GB300 mapping:
//   * A CTA of kWarps warps owns a range of 16-token tiles.  Warp w folds tiles
//     w, w+kWarps, ... with its own online-softmax state, then the warps merge
//     in warp order through shared memory.  A unit may span a thread-block
//     cluster of C CTAs that split the range and merge through distributed
//     shared memory in rank order.  The range split, the warp interleave and
//     both merge orders depend only on the unit's own length and build
//     constants, so a sequence's bits never depend on the rest of the batch.
//   * K and V tiles (16 tokens x head_dim BF16) move global -> shared with 4-D
//     TMA tensor loads gathered through the block table (one box per 64
//     columns, 128-byte swizzle), each warp running a private ring of
//     `stages` mbarrier-tracked buffers that it refills itself.
//   * q.K^T and P.V run on the tensor cores (mma.sync m16n8k16 BF16 -> FP32):
//     S[g,t] = q[g,:] K[t,:]^T with q rows as A (rows past the group are zero),
//     then O^T[d,g] += V^T[d,t] P^T[t,g] with P taken straight from the S
//     accumulator registers.  P is split into a BF16 high part and a BF16
//     residual (two mma), which keeps ~16 significant bits of each weight.
//   * Row max and row sums use warp shuffles across the 4 lanes of a row.
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

// Shared-memory plan of a unit CTA (host and device agree on it).
struct UnitSmem {
    int bars;        // offset of the mbarriers (after 1024-byte alignment slack)
    int stages;      // offset of the stage ring (1024-aligned)
    int merge;       // per-warp (m, l, o) for the warp merge: overlaps the ring
    int result;      // CTA result (m, l, o) read by the cluster peers
    int total;
};

__host__ __device__ inline UnitSmem unit_smem_plan(int dpad, int rows, int stages_per_warp) {
    UnitSmem s;
    const int stage_bytes = 2 * kTileTokens * dpad * 2;
    const int ring = kWarps * stages_per_warp * stage_bytes;
    const int ostride = dpad + 4;
    const int merge = kWarps * rows * (ostride + 3) * 4;  // o + m + l + weight
    s.bars = 0;
    const int bar_bytes = kWarps * stages_per_warp * 8;
    s.stages = (bar_bytes + 1023) / 1024 * 1024;
    s.merge = s.stages;
    const int big = ring > merge ? ring : merge;
    s.result = s.stages + (big + 15) / 16 * 16;
    const int result_bytes = rows * (ostride + 4) * 4;  // o + m + l + m_old + l_old
    s.total = 1024 /* alignment slack */ + s.result + result_bytes;
    return s;
}

template <int DPAD, int GN, int MODE, bool PACKED>
__global__ void __launch_bounds__(kThreads)
    unit_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const __grid_constant__ UnitParams p) {
    constexpr int KS = DPAD / 16;      // mma k-steps of q.K^T == m-tiles of V^T.P^T
    constexpr int NBOX = DPAD / kBoxCols;
    constexpr int TILE_BYTES = kTileTokens * DPAD * 2;
    constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    constexpr int RT = 8 * GN;         // query rows per CTA
    constexpr int OSTRIDE = DPAD + 4;  // padded row stride of o in shared memory
    const float kNegInf = -__int_as_float(0x7f800000);

    if constexpr (MODE == kModePaged) dev::griddep_launch_dependents();

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const UnitSmem plan = unit_smem_plan(DPAD, RT, S);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + plan.bars);
    uint8_t *ring = smem + plan.stages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- which unit ---------------------------------------------------------
    const int C = p.cluster;
    const int part = blockIdx.x % C;
    int u = blockIdx.x / C;
    int split = 0;
    if constexpr (MODE == kModePaged) {
        split = u % p.num_splits;
        u /= p.num_splits;
    }
    const int qt = u % p.qtiles;
    u /= p.qtiles;
    const int kvh = u % p.num_kv_heads;
    const int s = u / p.num_kv_heads;
    const int G = PACKED ? PD_GQA : p.group;
    const int D = PACKED ? PD_HDIM : p.head_dim;
    const int Hq = PACKED ? p.num_kv_heads * PD_GQA : p.num_q_heads;
    const int bs = p.block_size;
    const int g0 = qt * RT;                       // first group row of this CTA
    const int Gt = min(RT, G - g0);               // valid rows
    const int h0 = kvh * G + g0;                  // first query head

    // ---- token range of the unit --------------------------------------------
    int tok0 = 0, tok1 = 0;
    bool direct = true;  // paged: write normalised output instead of a partial
    const int32_t *ids_base;
    if constexpr (MODE == kModePaged) {
        int L = p.context_lens[s];
        const int Lmax = p.max_blocks_per_seq * bs;
        if (L < 0 || L > Lmax) {
            if (tid == 0 && part == 0 && split == 0 && qt == 0 && kvh == 0)
                dev::flag_status(p.status, kDevBadContextLen);
            L = L < 0 ? 0 : Lmax;
        }
        const int chunk = split_chunk_tokens(L, p.num_splits, bs, p.min_kv_per_split);
        const long long a = static_cast<long long>(split) * chunk;
        tok0 = static_cast<int>(a < L ? a : L);
        tok1 = static_cast<int>(a + chunk < L ? a + chunk : L);
        direct = splits_used(L, chunk) <= 1;
        ids_base = p.block_table + static_cast<long long>(s) * p.max_blocks_per_seq;
        if (tok0 >= tok1) {
            // Empty split.  Split 0 of an empty sequence owns the zero output.
            if (L == 0 && split == 0 && part == 0) {
                for (int e = tid; e < Gt * D; e += kThreads) {
                    const int g = e / D, d = e - g * D;
                    p.out[(static_cast<long long>(s) * Hq + h0 + g) * D + d] = __float2bfloat16_rn(0.f);
                }
            }
            return;  // uniform across the cluster: every rank sees the same range
        }
    } else {
        int cnt = p.tile_counts[s];
        if (cnt < 0 || cnt > p.tile_capacity) {
            if (tid == 0 && part == 0 && qt == 0 && kvh == 0)
                dev::flag_status(p.status, kDevBadTileCount);
            cnt = cnt < 0 ? 0 : p.tile_capacity;
        }
        if (cnt == 0) return;  // nothing to fold: the state is unchanged
        const int lv = (p.last_valid >= 1 && p.last_valid < bs) ? p.last_valid : bs;
        tok0 = 0;
        tok1 = (cnt - 1) * bs + lv;
        ids_base = p.tile_blocks + static_cast<long long>(s) * p.tile_capacity;
    }

    // 16-token tiles of the range, split across the cluster's CTAs.
    const int tile0 = tok0 / kTileTokens;
    const int ntiles = (tok1 + kTileTokens - 1) / kTileTokens - tile0;
    const int per = (ntiles + C - 1) / C;
    const int my0 = tile0 + min(part * per, ntiles);
    const int my1 = tile0 + min((part + 1) * per, ntiles);
    const int nloc = my1 - my0 > warp ? (my1 - my0 - warp + kWarps - 1) / kWarps : 0;

    // ---- barriers -------------------------------------------------------------
    if (tid == 0) {
        dev::prefetch_tensormap(&tmk);
        dev::prefetch_tensormap(&tmv);
        for (int i = 0; i < kWarps * S; ++i) dev::mbar_init(dev::smem_addr(&bars[i]), 1);
        dev::fence_mbar_init();
    }
    __syncthreads();

    const uint64_t policy = dev::l2_evict_first_policy();
    const int tiles_per_block = bs / kTileTokens;

    // Block id of this warp's local tile r (lane-parallel window loads).
    auto load_id = [&](int r) -> int {
        if (r >= nloc) return -1;
        const int gt = my0 + warp + kWarps * r;
        const int j = gt / tiles_per_block;
        int id = __ldg(ids_base + j);
        // TMA reads zeros outside the tensor map's block extent (num_blocks).
        if (id < 0 || id >= p.num_blocks) dev::flag_status(p.status, kDevBadBlockId);
        return id;
    };
    auto issue = [&](int r, int k, int id) {
        const int gt = my0 + warp + kWarps * r;
        const int sub = (gt % tiles_per_block) * kTileTokens;
        const uint32_t bar = dev::smem_addr(&bars[warp * S + k]);
        const uint32_t dst = dev::smem_addr(ring + (warp * S + k) * STAGE_BYTES);
        const int c1 = p.tok_dim == 1 ? sub : kvh;
        const int c2 = p.tok_dim == 1 ? kvh : sub;
        dev::mbar_arrive_expect_tx(bar, STAGE_BYTES);
#pragma unroll
        for (int b = 0; b < NBOX; ++b)
            dev::tma_load_4d(dst + b * (kTileTokens * 128), &tmk, bar, b * kBoxCols, c1, c2, id,
                             policy);
#pragma unroll
        for (int b = 0; b < NBOX; ++b)
            dev::tma_load_4d(dst + TILE_BYTES + b * (kTileTokens * 128), &tmv, bar, b * kBoxCols,
                             c1, c2, id, policy);
    };

    int id_cur = load_id(lane);
    int id_nxt = load_id(32 + lane);
    const int npro = nloc < S ? nloc : S;
    for (int r = 0; r < npro; ++r) {
        const int id = __shfl_sync(0xffffffffu, id_cur, r);
        if (lane == 0) issue(r, r, id);
    }

    // ---- q fragments (A operand of q.K^T), rows past the group are zero -------
    const int qrow = lane >> 2;        // row within an 8-row half
    const int qcol = (lane & 3) * 2;   // column pair within a 16-column k-step
    uint32_t qa[KS][2 * GN];
    {
        const __nv_bfloat16 *qb = p.q + (static_cast<long long>(s) * Hq + h0) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int r = 0; r < GN; ++r) {
                const int g = qrow + 8 * r;
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int d = ks * 16 + hlf * 8 + qcol;
                    uint32_t v = 0;
                    if (g < Gt && d < D)
                        v = __ldg(reinterpret_cast<const unsigned int *>(qb + static_cast<long long>(g) * D + d));
                    // A register order: {row g k0-7, row g+8 k0-7, row g k8-15, row g+8 k8-15}
                    qa[ks][hlf * GN + r] = v;
                }
            }
        }
    }

    // ---- per-lane ldmatrix offsets (128B swizzle: chunk c of row t at c ^ (t & 7)) ----
    const int lm_j = lane >> 3;
    const int lm_tok = ((lm_j >> 1) << 3) | (lane & 7);
    uint32_t lm_off[4];
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2)
        lm_off[c2] = lm_tok * 128 + ((((2 * c2) + (lm_j & 1)) ^ (lane & 7)) << 4);

    // ---- online-softmax state ---------------------------------------------------
    float o[KS][GN][4];
#pragma unroll
    for (int a = 0; a < KS; ++a)
#pragma unroll
        for (int b = 0; b < GN; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[a][b][c] = 0.f;
    float m_run[GN], l_run[GN];
#pragma unroll
    for (int r = 0; r < GN; ++r) {
        m_run[r] = kNegInf;
        l_run[r] = 0.f;
    }
    const int tokb = (lane & 3) * 2;  // this lane's token pair within an 8-token n-tile
    bool aborted = false;
    int fail_r = 0;

    for (int r = 0; r < nloc; ++r) {
        const int k = r % S;
        const uint32_t par = (r / S) & 1;
        if (!dev::mbar_wait_bounded(dev::smem_addr(&bars[warp * S + k]), par)) {
            dev::flag_status(p.status, kDevWaitTimeout);
            aborted = true;
            fail_r = r;
            break;
        }
        const int gt = my0 + warp + kWarps * r;
        const int nvalid = min(kTileTokens, tok1 - gt * kTileTokens);
        const uint32_t kbase = dev::smem_addr(ring + (warp * S + k) * STAGE_BYTES);
        const uint32_t vbase = kbase + TILE_BYTES;

        // S = q . K^T  (two n-tiles of 8 tokens)
        float sc[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[n][c] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t b0, b1, b2, b3;
            dev::ldsm_x4(kbase + (ks >> 2) * (kTileTokens * 128) + lm_off[ks & 3], b0, b1, b2, b3);
            uint32_t a0, a1, a2, a3;
            if constexpr (GN == 2) {
                a0 = qa[ks][0];
                a1 = qa[ks][1];
                a2 = qa[ks][2];
                a3 = qa[ks][3];
            } else {
                a0 = qa[ks][0];
                a1 = 0u;
                a2 = qa[ks][1];
                a3 = 0u;
            }
            dev::mma_bf16_16816(sc[0], a0, a1, a2, a3, b0, b1);
            dev::mma_bf16_16816(sc[1], a0, a1, a2, a3, b2, b3);
        }

        // scale to base 2, mask tokens past the range, row max
        float alpha[GN];
        float pr[GN][2][2];  // [row half][n-tile][token of the pair]
#pragma unroll
        for (int r2 = 0; r2 < GN; ++r2) {
            float mx = kNegInf;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int t = n * 8 + tokb + j;
                    float x = sc[n][2 * r2 + j] * p.scale_log2;
                    x = t < nvalid ? x : kNegInf;
                    pr[r2][n][j] = x;
                    mx = fmaxf(mx, x);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[r2], mx);
            alpha[r2] = dev::exp2_approx(m_run[r2] - m_new);
            float sum = 0.f;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float e = dev::exp2_approx(pr[r2][n][j] - m_new);
                    pr[r2][n][j] = e;
                    sum += e;
                }
            l_run[r2] = l_run[r2] * alpha[r2] + sum;
            m_run[r2] = m_new;
        }

        // rescale O^T columns (query rows) whose max moved
        bool any = false;
#pragma unroll
        for (int r2 = 0; r2 < GN; ++r2) any |= alpha[r2] != 1.f;
        if (__any_sync(0xffffffffu, any)) {
#pragma unroll
            for (int nt = 0; nt < GN; ++nt) {
                const float a0 = __shfl_sync(0xffffffffu, alpha[nt], (lane & 3) * 8);
                const float a1 = __shfl_sync(0xffffffffu, alpha[nt], (lane & 3) * 8 + 4);
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    o[mt][nt][0] *= a0;
                    o[mt][nt][1] *= a1;
                    o[mt][nt][2] *= a0;
                    o[mt][nt][3] *= a1;
                }
            }
        }

        // P^T as the B operand: high BF16 part and BF16 residual
        uint32_t bh[GN][2], bl[GN][2];
#pragma unroll
        for (int nt = 0; nt < GN; ++nt)
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const float e0 = pr[nt][n][0], e1 = pr[nt][n][1];
                const uint32_t hi = dev::pack_bf16x2(e0, e1);
                bh[nt][n] = hi;
                bl[nt][n] = dev::pack_bf16x2(e0 - dev::bf16_lo_f32(hi), e1 - dev::bf16_hi_f32(hi));
            }

        // token masks for a partial tile (V rows past the range may hold anything)
        uint32_t mask01 = 0xffffffffu, mask89 = 0xffffffffu;
        if (nvalid < kTileTokens) {
            mask01 = (tokb < nvalid ? 0x0000ffffu : 0u) | (tokb + 1 < nvalid ? 0xffff0000u : 0u);
            mask89 = (tokb + 8 < nvalid ? 0x0000ffffu : 0u) | (tokb + 9 < nvalid ? 0xffff0000u : 0u);
        }

        // O^T += V^T . P^T
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a0, a1, a2, a3;
            dev::ldsm_x4_trans(vbase + (mt >> 2) * (kTileTokens * 128) + lm_off[mt & 3], a0, a1, a2, a3);
            a0 &= mask01;
            a1 &= mask01;
            a2 &= mask89;
            a3 &= mask89;
#pragma unroll
            for (int nt = 0; nt < GN; ++nt) {
                dev::mma_bf16_16816(o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
                dev::mma_bf16_16816(o[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
            }
        }

        // refill this stage with the warp's tile r + S
        const int rn = r + S;
        if (rn < nloc) {
            if ((rn & 31) == 0) {
                id_cur = id_nxt;
                id_nxt = load_id(rn + 32 + lane);
            }
            const int id = __shfl_sync(0xffffffffu, id_cur, rn & 31);
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) issue(rn, k, id);
        }
    }
    if (aborted) {
        // Drain whatever this warp still has in flight (bounded) before the
        // ring is reused, so no copy lands after the CTA moves on.
        const int last = fail_r + S < nloc ? fail_r + S : nloc;  // tiles issued so far
        for (int r = fail_r; r < last; ++r)
            dev::mbar_wait_bounded(dev::smem_addr(&bars[warp * S + r % S]), (r / S) & 1, 100000000ull);
    }

    // ---- warp merge (fixed warp order) -------------------------------------------
#pragma unroll
    for (int r2 = 0; r2 < GN; ++r2) {
        l_run[r2] += __shfl_xor_sync(0xffffffffu, l_run[r2], 1);
        l_run[r2] += __shfl_xor_sync(0xffffffffu, l_run[r2], 2);
    }
    __syncthreads();  // every warp is done with the ring; reuse it for the merge
    float *wo = reinterpret_cast<float *>(smem + plan.merge);  // [kWarps][RT][OSTRIDE]
    float *wm = wo + kWarps * RT * OSTRIDE;                    // [kWarps][RT]
    float *wl = wm + kWarps * RT;                              // [kWarps][RT]
    float *ww = wl + kWarps * RT;                              // [kWarps][RT] weights
    if ((lane & 3) == 0) {
#pragma unroll
        for (int r2 = 0; r2 < GN; ++r2) {
            wm[warp * RT + qrow + 8 * r2] = m_run[r2];
            wl[warp * RT + qrow + 8 * r2] = l_run[r2];
        }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < GN; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int g = nt * 8 + tokb + (c & 1);
                const int d = mt * 16 + qrow + (c >> 1) * 8;
                wo[(warp * RT + g) * OSTRIDE + d] = o[mt][nt][c];
            }
    __syncthreads();

    float *co = reinterpret_cast<float *>(smem + plan.result);  // [RT][OSTRIDE]
    float *cm = co + RT * OSTRIDE;                               // [RT]
    float *cl = cm + RT;
    float *xm = cl + RT;  // tiled fold: old m
    float *xl = xm + RT;  // tiled fold: old l
    if (tid < RT) {
        float M = kNegInf;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * RT + tid]);
        float Lsum = 0.f;
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
    for (int e = tid; e < RT * DPAD; e += kThreads) {
        const int g = e / DPAD, d = e - g * DPAD;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += ww[w * RT + g] * wo[(w * RT + g) * OSTRIDE + d];
        co[g * OSTRIDE + d] = acc;
    }

    // ---- cluster merge (rank order) and epilogue -----------------------------------
    // Rows are dealt to the cluster's ranks round-robin; each rank combines its
    // rows over all ranks' results and writes them.
    cg::cluster_group cluster = cg::this_cluster();
    if (C > 1) cluster.sync(); else __syncthreads();

    for (int g = part; g < Gt; g += C) {
        const int h = h0 + g;
        const long long row = static_cast<long long>(s) * Hq + h;
        // combined (M, L) of row g
        float M = kNegInf, Lsum = 0.f;
        for (int rk = 0; rk < C; ++rk) {
            const float *pm = C > 1 ? cluster.map_shared_rank(cm, rk) : cm;
            M = fmaxf(M, pm[g]);
        }
        for (int rk = 0; rk < C; ++rk) {
            const float *pm = C > 1 ? cluster.map_shared_rank(cm, rk) : cm;
            const float *pl = C > 1 ? cluster.map_shared_rank(cl, rk) : cl;
            const float mr = pm[g];
            if (mr != kNegInf) Lsum += dev::exp2_approx(mr - M) * pl[g];
        }
        if constexpr (MODE == kModeTiled) {
            if (tid == 0) {
                xm[g] = p.st_m[row];
                xl[g] = p.st_l[row];
            }
            __syncthreads();
        }
        for (int d = tid; d < D; d += kThreads) {
            float acc = 0.f;
            for (int rk = 0; rk < C; ++rk) {
                const float *pm = C > 1 ? cluster.map_shared_rank(cm, rk) : cm;
                const float *po = C > 1 ? cluster.map_shared_rank(co, rk) : co;
                const float mr = pm[g];
                if (mr != kNegInf) acc += dev::exp2_approx(mr - M) * po[g * OSTRIDE + d];
            }
            if constexpr (MODE == kModePaged) {
                if (direct) {
                    const float v = Lsum > 0.f ? __fdiv_rn(acc, Lsum) : 0.f;
                    p.out[row * D + d] = __float2bfloat16_rn(v);
                } else {
                    p.ws_o[(row * p.num_splits + split) * D + d] = acc;
                }
            } else {
                const float m_old = xm[g];
                const float m_new = fmaxf(m_old, M);
                const float a = m_old == kNegInf ? 0.f : dev::exp2_approx(m_old - m_new);
                const float b = M == kNegInf ? 0.f : dev::exp2_approx(M - m_new);
                float *so = p.st_o + row * D + d;
                *so = *so * a + acc * b;
            }
        }
        if (tid == 0) {
            if constexpr (MODE == kModePaged) {
                if (!direct) {
                    p.ws_ml[(row * p.num_splits + split) * 2 + 0] = M;
                    p.ws_ml[(row * p.num_splits + split) * 2 + 1] = Lsum;
                }
            } else {
                const float m_old = xm[g];
                const float m_new = fmaxf(m_old, M);
                const float a = m_old == kNegInf ? 0.f : dev::exp2_approx(m_old - m_new);
                const float b = M == kNegInf ? 0.f : dev::exp2_approx(M - m_new);
                p.st_l[row] = xl[g] * a + Lsum * b;
                p.st_m[row] = m_new;
            }
        }
    }
    if (C > 1) cluster.sync();  // peers keep their shared memory until every rank has read it
}

}  // namespace pd
