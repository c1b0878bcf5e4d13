// noalloc.cu -- pa_decode_noalloc: the balanced split-K decode with its scratch in a fixed,
// statically sized device array instead of memory the library or the caller allocates.
//
// Who needs this: a serving engine commonly reserves almost all of HBM for its K/V page
// pool when it starts and then forbids further device allocations, and cudaMalloc and
// cudaFree synchronise the device, which a latency-bound decode loop cannot afford. Code
// running inside such an engine (for example a plugin that is handed only the tensors)
// has no allocator it may call, yet the split-K schedule needs scratch for per-range
// softmax states. This entry point gives those callers a decode call that allocates
// nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "pagedattn.h"

namespace {

// The scratch. It exists in every GPU context that loads this library, from module load
// until the process exits. In host code this name is only a stand-in for the symbol; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_address[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up once per device.
pa_status_t scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_address[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_scratch_address[dev] = p;
  }
  *out = g_scratch_address[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_decode_noalloc(const pa_problem_t *problem, const void *query,
                                         const void *key_cache, const void *value_cache,
                                         const int32_t *block_tables,
                                         const int32_t *context_lengths, float scale, float *out,
                                         void *stream) {
  pa_status_t st = pa::validate_call(problem, nullptr, query, key_cache, value_cache,
                                     block_tables, context_lengths, scale, out);
  if (st != PA_OK) return st;
  if (problem->batch == 0) return PA_OK;
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  // The fused merge's flags in the scratch need no clearing (each call publishes states
  // under its own number); a plan needing more than PA_NOALLOC_SCRATCH_BYTES is refused
  // with PA_ERR_WORKSPACE before anything is launched.
  return pa::decode_into(problem, query, key_cache, value_cache, block_tables, context_lengths,
                         scale, out, nullptr, scratch, PA_NOALLOC_SCRATCH_BYTES,
                         pa::WorkspaceKind::kStatic, static_cast<cudaStream_t>(stream));
}
