// Instantiation of the tcgen05 W4A16 kernel for 128 rows of X per tile, per-group zero-points.
#include "gemm_tc_launch.cuh"
W4A16_INSTANTIATE_TC(128, 2, kFmtW4Zp)
