// pd_unit_d64.cu -- unit kernels for head dims padded to 64 columns.
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(64, 1, pd::kModePaged, false)
PD_INSTANTIATE_UNIT(64, 2, pd::kModePaged, false)
PD_INSTANTIATE_UNIT(64, 1, pd::kModeTiled, false)
PD_INSTANTIATE_UNIT(64, 2, pd::kModeTiled, false)
