// Decode and combine kernels instantiated for head_dim = 256.
#include "decode_launch.cuh"

PA_INSTANTIATE_HD(256)
