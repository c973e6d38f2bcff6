// Tensor-core backward pass instantiated for head dimension 128 (causal and non-causal).
#include "fa_bwd_launch.cuh"

FA_DEFINE_BWD_LAUNCHER(128)
