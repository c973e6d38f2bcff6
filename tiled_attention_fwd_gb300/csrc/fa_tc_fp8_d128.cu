// Tensor-core forward pass on e4m3 Q, K, V (bf16 O), head dimension 128, causal and non-causal.
#include "fa_tc_launch.cuh"

FA_DEFINE_TC_FP8_LAUNCHER(128)
