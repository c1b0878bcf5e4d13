// launch.cu -- head_dim dispatch of the kernel launchers, the shared-memory sizing they
// need, and the device error word.
#include "device_common.cuh"
#include "internal.h"

namespace pa {

cudaError_t launch_decode_hd64(const KernelArgs &, const CUtensorMap *, const CUtensorMap *, int,
                               int, int, int, int, size_t, cudaStream_t);
cudaError_t launch_decode_hd128(const KernelArgs &, const CUtensorMap *, const CUtensorMap *, int,
                                int, int, int, int, size_t, cudaStream_t);
cudaError_t launch_decode_hd256(const KernelArgs &, const CUtensorMap *, const CUtensorMap *, int,
                                int, int, int, int, size_t, cudaStream_t);
cudaError_t launch_combine_balanced_hd64(const KernelArgs &, int, int, int, int, cudaStream_t);
cudaError_t launch_combine_balanced_hd128(const KernelArgs &, int, int, int, int, cudaStream_t);
cudaError_t launch_combine_balanced_hd256(const KernelArgs &, int, int, int, int, cudaStream_t);
cudaError_t launch_combine_split_hd64(const KernelArgs &, cudaStream_t);
cudaError_t launch_combine_split_hd128(const KernelArgs &, cudaStream_t);
cudaError_t launch_combine_split_hd256(const KernelArgs &, cudaStream_t);

// One word per device: PA_DEVERR_* bits raised by the kernels.
__device__ unsigned g_device_error = 0;

// Tokens per K/V tile. head_dim 128 defaults to 16-token tiles (8 KB stages, three per warp
// by default): on GB300 they beat 32-token tiles by ~2 % on mixed context lengths (less
// imbalance at the end of the balanced split) and are within 0.5 % elsewhere.
int tile_tokens(int head_dim, int requested) {
  if (head_dim == 128 && (requested == 16 || requested == 32)) return requested;
  return head_dim == 64 ? 32 : 16;
}

bool tile_supported(int head_dim, int tile) {
  return tile == tile_tokens(head_dim, tile);
}

int simt_heads_instance(int nh) {
  if (nh <= 1) return 1;
  if (nh <= 2) return 2;
  if (nh <= 4) return 4;
  if (nh <= 6) return 6;
  return 8;
}

int warp_smem_bytes(int head_dim, int mma, int nh_inst, int stages, int t) {
  long long bytes = static_cast<long long>(stages) * t * head_dim * 4;
  if (!mma) {
    const int nhp = (nh_inst + 3) & ~3;
    bytes += static_cast<long long>(nh_inst) * head_dim * 4 + static_cast<long long>(t) * nhp * 4;
  }
  bytes = (bytes + kSmemAlign - 1) / kSmemAlign * kSmemAlign;
  return static_cast<int>(bytes);
}

cudaError_t launch_decode(const KernelArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                          int mma, int nh_inst, int tile, int ctas, int warps_per_cta,
                          size_t smem, cudaStream_t stream) {
  switch (a.hd) {
    case 64:
      return launch_decode_hd64(a, tk, tv, mma, nh_inst, tile, ctas, warps_per_cta, smem, stream);
    case 128:
      return launch_decode_hd128(a, tk, tv, mma, nh_inst, tile, ctas, warps_per_cta, smem, stream);
    case 256:
      return launch_decode_hd256(a, tk, tv, mma, nh_inst, tile, ctas, warps_per_cta, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_balanced(const KernelArgs &a, int units, int heads, int warps_per_pair,
                                    int tile, cudaStream_t stream) {
  switch (a.hd) {
    case 64: return launch_combine_balanced_hd64(a, units, heads, warps_per_pair, tile, stream);
    case 128: return launch_combine_balanced_hd128(a, units, heads, warps_per_pair, tile, stream);
    case 256: return launch_combine_balanced_hd256(a, units, heads, warps_per_pair, tile, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_split(const KernelArgs &a, cudaStream_t stream) {
  switch (a.hd) {
    case 64: return launch_combine_split_hd64(a, stream);
    case 128: return launch_combine_split_hd128(a, stream);
    case 256: return launch_combine_split_hd256(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

unsigned *device_error_word() {
  static unsigned *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned *>(p);
  }
  return addr[dev];
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, uint32_t *flags) {
  unsigned *w = device_error_word();
  if (!w) return cudaErrorInvalidSymbol;
  unsigned v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof(unsigned), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  *flags = v;
  return e;
}

}  // namespace pa
