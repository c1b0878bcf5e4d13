// Decode and combine kernels instantiated for head_dim = 128.
#include "decode_launch.cuh"

PA_INSTANTIATE_HD(128)
