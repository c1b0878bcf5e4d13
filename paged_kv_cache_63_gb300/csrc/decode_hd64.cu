// Decode and combine kernels instantiated for head_dim = 64.
#include "decode_launch.cuh"

PA_INSTANTIATE_HD(64)
