// decode_launch.cuh -- host-side launchers of the decode and combine kernels for one
// head_dim; each decode_hd*.cu instantiates them for its head_dim.
#pragma once

#include "decode_kernel.cuh"

namespace pa {

constexpr int kMaxDevices = 64;

template <int HD, int T, bool MMA, int NH>
cudaError_t launch_variant(const KernelArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                           int ctas, int warps, size_t smem, cudaStream_t stream) {
  auto kern = decode_kernel<HD, T, MMA, NH>;
  // the opt-in shared-memory size is a per-device function attribute; remember the
  // largest value set on each device
  static int smem_set[kMaxDevices] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || smem_set[dev] < static_cast<int>(smem)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) smem_set[dev] = static_cast<int>(smem);
  }
  kern<<<ctas, warps * 32, smem, stream>>>(a, *tk, *tv);
  return cudaGetLastError();
}

template <int HD, int T>
cudaError_t launch_decode_ht(const KernelArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                             int mma, int nh_inst, int ctas, int warps, size_t smem,
                             cudaStream_t stream) {
  if (mma) return launch_variant<HD, T, true, kMaxHeads>(a, tk, tv, ctas, warps, smem, stream);
  switch (nh_inst) {
    case 1: return launch_variant<HD, T, false, 1>(a, tk, tv, ctas, warps, smem, stream);
    case 2: return launch_variant<HD, T, false, 2>(a, tk, tv, ctas, warps, smem, stream);
    case 4: return launch_variant<HD, T, false, 4>(a, tk, tv, ctas, warps, smem, stream);
    case 6: return launch_variant<HD, T, false, 6>(a, tk, tv, ctas, warps, smem, stream);
    case 8: return launch_variant<HD, T, false, 8>(a, tk, tv, ctas, warps, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Tile sizes instantiated per head_dim: 32 tokens for 64, 16 or 32 for 128, 16 for 256.
template <int HD>
cudaError_t launch_decode_hd(const KernelArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                             int mma, int nh_inst, int tile, int ctas, int warps, size_t smem,
                             cudaStream_t stream) {
  if constexpr (HD == 64) {
    if (tile == 32) return launch_decode_ht<HD, 32>(a, tk, tv, mma, nh_inst, ctas, warps, smem, stream);
  } else if constexpr (HD == 128) {
    if (tile == 16) return launch_decode_ht<HD, 16>(a, tk, tv, mma, nh_inst, ctas, warps, smem, stream);
    if (tile == 32) return launch_decode_ht<HD, 32>(a, tk, tv, mma, nh_inst, ctas, warps, smem, stream);
  } else {
    if (tile == 16) return launch_decode_ht<HD, 16>(a, tk, tv, mma, nh_inst, ctas, warps, smem, stream);
  }
  return cudaErrorInvalidValue;
}

template <int HD, int W>
cudaError_t launch_combine_balanced_hw(const KernelArgs &a, int units, int heads, int tile,
                                       cudaStream_t stream) {
  const long long pairs = static_cast<long long>(units) * heads;
  constexpr int P = 8 / W;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((pairs + P - 1) / P), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_wide_kernel<HD, W>, a, heads, pairs, tile);
}

template <int HD>
cudaError_t launch_combine_balanced_hd(const KernelArgs &a, int units, int heads,
                                       int warps_per_pair, int tile, cudaStream_t stream) {
  if (units == 0 || heads == 0) return cudaSuccess;
  switch (warps_per_pair) {
    case 1: return launch_combine_balanced_hw<HD, 1>(a, units, heads, tile, stream);
    case 2: return launch_combine_balanced_hw<HD, 2>(a, units, heads, tile, stream);
    case 4: return launch_combine_balanced_hw<HD, 4>(a, units, heads, tile, stream);
    case 8: return launch_combine_balanced_hw<HD, 8>(a, units, heads, tile, stream);
  }
  return cudaErrorInvalidValue;
}

template <int HD>
cudaError_t launch_combine_split_hd(const KernelArgs &a, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(a.batch) * a.qh;  // one per (sequence, head)
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  combine_split_kernel<HD><<<static_cast<unsigned>(blocks), kCombineSplitWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa

#define PA_INSTANTIATE_HD(HD)                                                                \
  namespace pa {                                                                             \
  cudaError_t launch_decode_hd##HD(const KernelArgs &a, const CUtensorMap *tk,               \
                                   const CUtensorMap *tv, int mma, int nh_inst, int tile,    \
                                   int ctas, int warps, size_t smem, cudaStream_t stream) {  \
    return launch_decode_hd<HD>(a, tk, tv, mma, nh_inst, tile, ctas, warps, smem, stream);   \
  }                                                                                          \
  cudaError_t launch_combine_balanced_hd##HD(const KernelArgs &a, int units, int heads,      \
                                             int warps_per_pair, int tile,                   \
                                             cudaStream_t stream) {                          \
    return launch_combine_balanced_hd<HD>(a, units, heads, warps_per_pair, tile, stream);    \
  }                                                                                          \
  cudaError_t launch_combine_split_hd##HD(const KernelArgs &a, cudaStream_t stream) {        \
    return launch_combine_split_hd<HD>(a, stream);                                           \
  }                                                                                          \
  }
