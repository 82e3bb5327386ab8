// Instantiation of the tcgen05 kernel for 2:4 sparse 4-bit codes, 128 rows of X per tile.
#include "gemm_tc_launch.cuh"
W4A16_INSTANTIATE_TC(128, 2, kFmtW4Sp)
