// Instantiation of the tcgen05 W4A16 kernel for 16 rows of X per tile.
#include "gemm_tc_launch.cuh"
W4A16_INSTANTIATE_TC(16, 4, kFmtW4)
