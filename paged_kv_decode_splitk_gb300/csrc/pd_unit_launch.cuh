// pd_unit_launch.cuh -- host launcher of the unit kernel, included by the
// per-head-dim translation units that instantiate it.
#pragma once

#include <mutex>

#include "pd_unit.cuh"

namespace pd {

int unit_smem_bytes(int dpad, int rows, int stages);

template <int DPAD, int GN, bool HL, int MODE, bool PACKED>
cudaError_t launch_unit(const CUtensorMap &tmk, const CUtensorMap &tmv, const UnitParams &p,
                        int grid_x, int smem_bytes, cudaStream_t stream) {
    auto kern = unit_kernel<DPAD, GN, HL, MODE, PACKED>;
    // Raise the kernel's dynamic shared-memory limit once per device (and
    // again only if a launch asks for more).
    static std::mutex mu;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (configured[dev] < smem_bytes) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
            if (e != cudaSuccess) return e;
            configured[dev] = smem_bytes;
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
    return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, p);
}

}  // namespace pd

#define PD_INSTANTIATE_UNIT(DPAD, GN, HL, MODE, PACKED)                                      \
    template cudaError_t pd::launch_unit<DPAD, GN, HL, MODE, PACKED>(                        \
        const CUtensorMap &, const CUtensorMap &, const pd::UnitParams &, int, int, cudaStream_t);
