// pd_unit_d128.cu -- unit kernels for head dims padded to 128 columns.
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(128, 1, true, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(128, 1, false, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(128, 2, false, pd::kModePaged, false, false)
PD_INSTANTIATE_UNIT(128, 1, true, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(128, 1, false, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(128, 2, false, pd::kModeTiled, false, false)
PD_INSTANTIATE_UNIT(128, 1, true, pd::kModeTiledRun, false, false)
PD_INSTANTIATE_UNIT(128, 1, false, pd::kModeTiledRun, false, false)
PD_INSTANTIATE_UNIT(128, 2, false, pd::kModeTiledRun, false, false)
