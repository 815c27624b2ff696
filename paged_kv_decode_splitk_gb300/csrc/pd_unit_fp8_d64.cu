// pd_unit_fp8_d64.cu -- unit kernels over an FP8 E4M3 KV cache, head dims padded
// to 64 columns (paged mode: the split-K partial pass and the GQA-packed pass).
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(64, 1, true, pd::kModePaged, false, true)
PD_INSTANTIATE_UNIT(64, 1, false, pd::kModePaged, false, true)
PD_INSTANTIATE_UNIT(64, 2, false, pd::kModePaged, false, true)
