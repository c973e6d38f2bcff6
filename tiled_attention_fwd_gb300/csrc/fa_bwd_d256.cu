// Tensor-core backward pass for head dimension 256 (causal and non-causal).
#include "fa_bwd_launch.cuh"

FA_DEFINE_BWD_LAUNCHER(256)
