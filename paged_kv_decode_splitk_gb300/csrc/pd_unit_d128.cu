// pd_unit_d128.cu -- unit kernels for head dims padded to 128 columns.
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(128, 1, pd::kModePaged, false)
PD_INSTANTIATE_UNIT(128, 2, pd::kModePaged, false)
PD_INSTANTIATE_UNIT(128, 1, pd::kModeTiled, false)
PD_INSTANTIATE_UNIT(128, 2, pd::kModeTiled, false)
