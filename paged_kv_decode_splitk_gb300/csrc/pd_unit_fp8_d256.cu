// pd_unit_fp8_d256.cu -- unit kernels over an FP8 E4M3 KV cache, head dims padded
// to 256 columns (paged mode: the split-K partial pass and the GQA-packed pass).
#include "pd_unit_launch.cuh"

PD_INSTANTIATE_UNIT(256, 1, true, pd::kModePaged, false, true)
PD_INSTANTIATE_UNIT(256, 1, false, pd::kModePaged, false, true)
PD_INSTANTIATE_UNIT(256, 2, false, pd::kModePaged, false, true)

// The GQA-packed pass over an FP8 cache: group width PD_GQA at head dim PD_HDIM.
PD_INSTANTIATE_UNIT(PD_HDIM, 1, false, pd::kModePaged, true, true)
