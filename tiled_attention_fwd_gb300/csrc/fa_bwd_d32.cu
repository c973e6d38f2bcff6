// Tensor-core backward pass instantiated for head dimension 32 (causal and non-causal).
#include "fa_bwd_launch.cuh"

FA_DEFINE_BWD_LAUNCHER(32)
