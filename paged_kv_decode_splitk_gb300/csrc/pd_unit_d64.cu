// pd_unit_d64.cu -- unit kernels for head dims padded to 64 columns.
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(64, 1, true, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(64, 1, false, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(64, 2, false, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(64, 1, true, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(64, 1, false, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(64, 2, false, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(64, 1, true, pd::kModeTiledRun, false, false)
PD_INSTANTIATE_UNIT(64, 1, false, pd::kModeTiledRun, false, false)
PD_INSTANTIATE_UNIT(64, 2, false, pd::kModeTiledRun, false, false)
