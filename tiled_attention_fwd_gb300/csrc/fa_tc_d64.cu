// Tensor-core forward pass instantiated for head dimension 64 (causal and non-causal).
#include "fa_tc_launch.cuh"

FA_DEFINE_TC_LAUNCHER(64)
