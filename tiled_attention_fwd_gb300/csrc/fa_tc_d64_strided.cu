// Tensor-core forward pass on strided tensors (4-D tensor maps), head dimension 64, causal and non-causal.
#include "fa_tc_launch.cuh"

FA_DEFINE_TC_STRIDED_LAUNCHER(64)
