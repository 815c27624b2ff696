// pd_unit_launch.cuh -- host launcher of the unit kernel, included by the
// per-head-dim translation units that instantiate it.
#pragma once

#include <cstring>
#include <mutex>

#include "pd_unit.cuh"

namespace pd {

template <int DPAD, int GN, bool HL, int MODE, bool PACKED, bool KV8>
cudaError_t launch_unit(const CUtensorMap *tmk, const CUtensorMap *tmv, const UnitParams &p_in,
                        long long units, int stages_seq, cudaStream_t stream, int layout) {
    auto kern = unit_kernel<DPAD, GN, HL, MODE, PACKED, KV8, false>;
    // Per device: the dynamic shared-memory limit raised so far (for this kernel
    // and its 128-register twin), the SM count, and how many CTAs of this kernel
    // fit on one SM at each stage count.
    static std::mutex mu;
    static int configured[64] = {0};
    static int configured_cap4[64] = {0};
    static int sm_count[64] = {0};
    static int per_sm[64][kMaxStagesPerWarp + 1] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (p_in.stages < 1 || p_in.stages > kMaxStagesPerWarp || stages_seq < 1 || stages_seq > kMaxStagesPerWarp)
        return cudaErrorInvalidValue;
    auto slots_for = [&](int stages, int *smem_out) -> cudaError_t {
        const int smem = unit_smem_plan(DPAD, 8 * GN, stages, KV8).total;
        *smem_out = smem;
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev] < smem) {
            cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e2 != cudaSuccess) return e2;
            configured[dev] = smem;
        }
        if (!sm_count[dev]) {
            cudaError_t e2 = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e2 != cudaSuccess) return e2;
        }
        if (!per_sm[dev][stages]) {
            int n = 0;
            cudaError_t e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
            if (e2 != cudaSuccess) return e2;
            per_sm[dev][stages] = n > 0 ? n : -1;
        }
        return cudaSuccess;
    };
    int smem_bytes = 0;
    e = slots_for(p_in.stages, &smem_bytes);
    if (e != cudaSuccess) return e;
    const int slots = per_sm[dev][p_in.stages] > 0 ? per_sm[dev][p_in.stages] * sm_count[dev] : 0;
    // Where the parts of a unit run.  Both layouts fold the same parts in the
    // same order, so the choice changes timing only, never the output bits:
    // when one CTA per part still fits in about one wave, a cluster of
    // max_parts CTAs per unit (fills the GPU when units are few); otherwise
    // one CTA per unit walking its parts in sequence.
    UnitParams p = p_in;
    int C = 1;
    if (p.max_parts > 1) {
        if (layout == 2)
            C = p.max_parts;
        else if (layout == 0 && units * p.max_parts * 4 <= static_cast<long long>(slots) * 5)
            C = p.max_parts;
    }
    p.cluster = C;
    const long long grid_x = units * C;
    if (grid_x > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // A grid of many short units (several waves, one CTA per unit) keeps more
    // loads in flight with a deeper ring per warp; a single-wave grid keeps
    // the shallower one and more CTAs per SM.  Stages change no result.
    if (C == 1 && stages_seq != p.stages && grid_x > slots) {
        e = slots_for(stages_seq, &smem_bytes);
        if (e != cudaSuccess) return e;
        p.stages = stages_seq;
    }
    // The early L2 prefetch pays off only for CTAs that are resident while the
    // previous kernel drains, i.e. a grid of about one wave; CTAs of later
    // waves would just read the lengths and the block table twice.
    if (grid_x * 4 > static_cast<long long>(slots) * 5) p.prefetch_tiles = 0;
    // Many waves of one-CTA units over an FP8 cache at head dim 128, groups of
    // up to 4: the 128-register twin (4 CTAs per SM instead of 3; measured
    // 471 -> 413 us on the 256-sequence FP8 step, while the one-wave
    // long-context FP8 step runs 22.4 us on this kernel against 25-26 us on
    // the twin).  Same arithmetic, same bits.
    constexpr bool kHasCap4 = KV8 && DPAD == 128 && GN == 1 && HL && MODE == kModePaged && !PACKED;
    bool cap4 = false;
    if constexpr (kHasCap4) {
        if (C == 1 && grid_x > slots) {
            std::lock_guard<std::mutex> lock(mu);
            if (configured_cap4[dev] < smem_bytes) {
                e = cudaFuncSetAttribute(unit_kernel<DPAD, GN, HL, MODE, PACKED, KV8, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
                if (e != cudaSuccess) return e;
                configured_cap4[dev] = smem_bytes;
            }
            cap4 = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_x));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    // Programmatic dependent launch: this grid may launch while the previous
    // kernel in the stream drains; it waits for it before touching memory.
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (p.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(p.cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    constexpr int NM = MODE == kModeTiledRun ? kMaxRunSources : 1;
    const int nmaps = MODE == kModeTiledRun ? p.num_sources : 1;
    if (nmaps < 1 || nmaps > NM) return cudaErrorInvalidValue;
    KvMaps<NM> maps;
    memset(&maps, 0, sizeof(maps));
    for (int i = 0; i < nmaps; ++i) {
        maps.k[i] = tmk[i];
        maps.v[i] = tmv[i];
    }
    if constexpr (kHasCap4) {
        if (cap4) return cudaLaunchKernelEx(&cfg, unit_kernel<DPAD, GN, HL, MODE, PACKED, KV8, true>, maps, p);
    }
    return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

}  // namespace pd

#define PD_INSTANTIATE_UNIT(DPAD, GN, HL, MODE, PACKED, KV8)                                 \
    template cudaError_t pd::launch_unit<DPAD, GN, HL, MODE, PACKED, KV8>(                   \
        const CUtensorMap *, const CUtensorMap *, const pd::UnitParams &, long long, int,       \
        cudaStream_t, int);
