// Tensor-core backward pass on strided tensors (4-D tensor maps), head dimension 256.
#include "fa_bwd_launch.cuh"

FA_DEFINE_BWD_STRIDED_LAUNCHER(256)
