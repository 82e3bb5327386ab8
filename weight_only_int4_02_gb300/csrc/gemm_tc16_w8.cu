// Instantiation of the tcgen05 kernel for 8-bit codes (W8A16), 16 rows of X per tile.
#include "gemm_tc_launch.cuh"
W4A16_INSTANTIATE_TC(16, 2, kFmtW8)
