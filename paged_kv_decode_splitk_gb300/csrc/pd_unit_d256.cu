// pd_unit_d256.cu -- unit kernels for head dims padded to 256 columns.
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(256, 1, true, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(256, 1, false, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(256, 2, false, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(256, 1, true, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(256, 1, false, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(256, 2, false, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(256, 1, true, pd::kModeTiledRun, false, false)
PD_INSTANTIATE_UNIT(256, 1, false, pd::kModeTiledRun, false, false)
PD_INSTANTIATE_UNIT(256, 2, false, pd::kModeTiledRun, false, false)

// The GQA-packed pass: group width PD_GQA at head dim PD_HDIM, compile-time.
PD_INSTANTIATE_UNIT(PD_HDIM, 1, false, pd::kModePaged, true, false)

namespace pd {
int kernel_pack_width() { return PD_GQA; }
int kernel_pack_head_dim() { return PD_HDIM; }
int unit_smem_bytes(int dpad, int rows, int stages, bool kv8) { return unit_smem_plan(dpad, rows, stages, kv8).total; }
}  // namespace pd
