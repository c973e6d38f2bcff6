// Tensor-core forward pass instantiated for head dimension 256 (causal and non-causal): CTA pairs
// (cta_group::2, M = 256, 128-key tiles) on contiguous tensors.
#include "fa_tc_launch.cuh"

FA_DEFINE_TC_PAIR_LAUNCHER(256)
