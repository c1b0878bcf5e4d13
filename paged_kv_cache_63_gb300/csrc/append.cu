// append.cu -- the cache write before a decode step: one new K and V row per sequence and
// K/V head, written at token index context_lengths[b] through the block table.
#include "device_common.cuh"
#include "internal.h"

namespace pa {

struct AppendArgs {
  const uint16_t *new_k, *new_v;  // [batch][kv_heads][head_dim] fp16 bits
  const int32_t *bt, *ctx;
  uint16_t *k, *v;                // the caches
  unsigned *err;
  int batch, kvh, hd, ps, ps_shift, maxp, num_pages, layout;
};

// One warp per (sequence, K/V head): lanes copy the K and V rows as 16-byte vectors.
__global__ void __launch_bounds__(256) append_kv_kernel(const __grid_constant__ AppendArgs a) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= static_cast<long long>(a.batch) * a.kvh) return;
  const int lane = threadIdx.x & 31;
  const int b = static_cast<int>(w / a.kvh);
  const int kv = static_cast<int>(w % a.kvh);
  const int t = __ldg(a.ctx + b);
  if (t < 0 || t >= (a.maxp << a.ps_shift)) {
    if (lane == 0) atomicOr(a.err, PA_DEVERR_CONTEXT);
    return;
  }
  const int page = __ldg(a.bt + static_cast<long long>(b) * a.maxp + (t >> a.ps_shift));
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) atomicOr(a.err, PA_DEVERR_PAGE_ID);
    return;
  }
  const int slot = t & (a.ps - 1);
  const long long row =
      a.layout == PA_LAYOUT_HEAD_MAJOR
          ? (static_cast<long long>(page) * a.kvh + kv) * a.ps + slot
          : (static_cast<long long>(page) * a.ps + slot) * a.kvh + kv;
  const long long dst = row * a.hd;
  const long long src = w * a.hd;
  const int chunks = a.hd >> 3;  // 16-byte vectors per row
  for (int i = lane; i < 2 * chunks; i += 32) {
    const int c = i < chunks ? i : i - chunks;
    const uint16_t *from = (i < chunks ? a.new_k : a.new_v) + src + c * 8;
    uint16_t *to = (i < chunks ? a.k : a.v) + dst + c * 8;
    *reinterpret_cast<uint4 *>(to) = __ldg(reinterpret_cast<const uint4 *>(from));
  }
}

}  // namespace pa

extern "C" pa_status_t pa_append_kv(const pa_problem_t *problem, const void *new_key,
                                    const void *new_value, const int32_t *block_tables,
                                    const int32_t *context_lengths, void *key_cache,
                                    void *value_cache, void *stream) {
  pa_status_t st = pa::validate_call(problem, nullptr, new_key, key_cache, value_cache,
                                     block_tables, context_lengths, 1.0f,
                                     static_cast<const float *>(new_value));
  if (st != PA_OK) return st;
  if (problem->batch == 0) return PA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_NO_DEVICE;
  pa::AppendArgs a;
  a.new_k = static_cast<const uint16_t *>(new_key);
  a.new_v = static_cast<const uint16_t *>(new_value);
  a.bt = block_tables;
  a.ctx = context_lengths;
  a.k = static_cast<uint16_t *>(key_cache);
  a.v = static_cast<uint16_t *>(value_cache);
  a.err = pa::device_error_word();
  if (!a.err) return PA_ERR_CUDA;
  a.batch = problem->batch;
  a.kvh = problem->kv_heads;
  a.hd = problem->head_dim;
  a.ps = problem->page_size;
  a.ps_shift = 0;
  while ((1 << a.ps_shift) < a.ps) ++a.ps_shift;
  a.maxp = problem->max_pages_per_sequence;
  a.num_pages = problem->num_physical_pages;
  a.layout = problem->cache_layout;
  const long long threads = static_cast<long long>(a.batch) * a.kvh * 32;
  const int blocks = static_cast<int>((threads + 255) / 256);
  pa::append_kv_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
