// prefill.cu -- host entry point of the causal multi-token (prefill) kernel: argument
// checks, tensor maps and the launch.
#include <cmath>

#include "internal.h"
#include "pagedattn.h"
#include "prefill2_kernel.cuh"
#include "prefill_kernel.cuh"

namespace pa {

namespace {

constexpr int kMaxDevicesPrefill = 64;

template <int HD>
cudaError_t launch_prefill_hd(const PrefillArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
  using C = PrefillCfg<HD>;
  auto kern = prefill_kernel<HD>;
  constexpr int smem = C::kSmem + 1024;
  static bool set[kMaxDevicesPrefill] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesPrefill || !set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevicesPrefill) set[dev] = true;
  }
  kern<<<grid, kPrefillThreads, smem, stream>>>(a, tq, tk, tv);
  return cudaGetLastError();
}

// head_dim 64 / 128: two query tiles per CTA (a.n_qtiles counts pairs, grid.z too)
template <int HD>
cudaError_t launch_prefill2_hd(const PrefillArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
  using C = Prefill2Cfg<HD>;
  auto kern = prefill2_kernel<HD>;
  constexpr int smem = C::kSmem + 1024;
  static bool set[kMaxDevicesPrefill] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesPrefill || !set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevicesPrefill) set[dev] = true;
  }
  kern<<<grid, kPrefill2Threads, smem, stream>>>(a, tq, tk, tv);
  return cudaGetLastError();
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace pa

extern "C" pa_status_t pa_prefill(const pa_problem_t *problem, const void *query,
                                  const int32_t *query_start, int64_t total_tokens,
                                  int32_t max_query_len, const void *key_cache,
                                  const void *value_cache, const int32_t *block_tables,
                                  const int32_t *context_lengths, float scale, float *out,
                                  const pa_options_t *options, void *stream) {
  using namespace pa;
  pa_status_t st = check_problem_public(problem);
  if (st != PA_OK) return st;
  if (options && (options->schedule || options->math || options->combine || options->workers ||
                  options->stages || options->warps_per_cta || options->tile_tokens ||
                  (options->test_flags & ~PA_TEST_EXPIRE_WAITS)))
    return PA_ERR_INVALID_ARG;
  if (!query || !query_start || !key_cache || !value_cache || !block_tables ||
      !context_lengths || !out || !std::isfinite(scale))
    return PA_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens >= (int64_t(1) << 31) || max_query_len < 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(query_start) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lengths) & 3u))
    return PA_ERR_MISALIGNED;
  const int g = problem->query_heads / problem->kv_heads;
  if (g > 128) return PA_ERR_UNSUPPORTED;
  if (problem->batch == 0 || total_tokens == 0 || max_query_len == 0) return PA_OK;
  if (problem->batch > 65535 || problem->kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  int smem_optin = 0;
  st = current_device_smem(&smem_optin);
  if (st != PA_OK) return st;

  const int hd = problem->head_dim;
  const int tn = hd == 256 ? 64 : 128;
  const int qt = 128 / g;
  const long long n_qtiles = (static_cast<long long>(max_query_len) + qt - 1) / qt;
  if (n_qtiles > 65535) return PA_ERR_UNSUPPORTED;

  PrefillArgs a = {};
  a.qs = query_start;
  a.bt = block_tables;
  a.ctx = context_lengths;
  a.out = out;
  a.err = device_error_word();
  if (!a.err) return PA_ERR_CUDA;
  a.total = total_tokens;
  a.batch = problem->batch;
  a.qh = problem->query_heads;
  a.kvh = problem->kv_heads;
  a.ps = problem->page_size;
  a.ps_shift = 0;
  while ((1 << a.ps_shift) < a.ps) ++a.ps_shift;
  a.maxp = problem->max_pages_per_sequence;
  a.num_pages = problem->num_physical_pages;
  a.layout = problem->cache_layout;
  a.g = g;
  a.qt = qt;
  a.n_qtiles = static_cast<int>(n_qtiles);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.expire = (options && (options->test_flags & PA_TEST_EXPIRE_WAITS)) ? 1 : 0;
  a.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;

  CUtensorMap tq, tk, tv;
  const int rows = a.ps < tn ? a.ps : tn;
  st = encode_query_map(&tq, query, total_tokens, a.qh, hd, g, qt);
  if (st != PA_OK) return st;
  st = encode_cache_map_rows(&tk, key_cache, problem, rows);
  if (st != PA_OK) return st;
  st = encode_cache_map_rows(&tv, value_cache, problem, rows);
  if (st != PA_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (hd != 256) a.n_qtiles = (a.n_qtiles + 1) / 2;  // pairs of query tiles
  const dim3 grid(a.kvh, a.batch, a.n_qtiles);
  switch (hd) {
    case 64:
      e = launch_prefill2_hd<64>(a, tq, tk, tv, grid, s);
      break;
    case 128:
      e = launch_prefill2_hd<128>(a, tq, tk, tv, grid, s);
      break;
    case 256:
      e = launch_prefill_hd<256>(a, tq, tk, tv, grid, s);
      break;
    default:
      return PA_ERR_UNSUPPORTED;
  }
  (void)smem_optin;
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
