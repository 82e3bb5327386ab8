// Instantiation of the tcgen05 W4A16 kernel for 32 rows of X per tile, BF16 activations.
#include "gemm_tc_launch.cuh"
W4A16_INSTANTIATE_TC(32, 4, kFmtW4Bf16)
