// api.cpp -- the C ABI of libpagedattn: argument checks, the schedule/math heuristic,
// TMA tensor-map encoding, workspace handling and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "pagedattn.h"

namespace {

using namespace pa;

constexpr int32_t kVersion = 100;  // 0.1.0
constexpr int kMaxDev = 64;
// Bytes of shared memory the SM reserves per resident CTA.
constexpr int kSmemReservedPerCta = 1024;
// Static shared memory of the decode kernel (its mbarriers), rounded up.
constexpr int kStaticSmem = 1024;
constexpr int kDefaultWarps = 8;

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

pa_status_t check_problem(const pa_problem_t *p) {
  if (!p) return PA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->query_heads < 1 || p->kv_heads < 1 || p->head_dim < 1 ||
      p->page_size < 1 || p->max_pages_per_sequence < 1 || p->num_physical_pages < 1)
    return PA_ERR_INVALID_ARG;
  if (p->query_heads % p->kv_heads) return PA_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(p->page_size) || p->page_size < 8 || p->page_size > 256) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->num_physical_pages) * p->page_size >= (int64_t(1) << 31))
    return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->max_pages_per_sequence) * p->page_size >= (int64_t(1) << 31))
    return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->batch) * p->query_heads * p->head_dim >= (int64_t(1) << 40))
    return PA_ERR_UNSUPPORTED;
  if (p->cache_layout != PA_LAYOUT_TOKEN_MAJOR && p->cache_layout != PA_LAYOUT_HEAD_MAJOR)
    return PA_ERR_INVALID_ARG;
  if (p->cache_layout == PA_LAYOUT_HEAD_MAJOR &&
      static_cast<int64_t>(p->num_physical_pages) * p->kv_heads >= (int64_t(1) << 31))
    return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

pa_status_t check_options(const pa_options_t *o) {
  if (!o) return PA_OK;
  if (o->schedule < PA_SCHEDULE_AUTO || o->schedule > PA_SCHEDULE_BALANCED) return PA_ERR_INVALID_ARG;
  if (o->math < PA_MATH_AUTO || o->math > PA_MATH_MMA) return PA_ERR_INVALID_ARG;
  if (o->combine < PA_COMBINE_AUTO || o->combine > PA_COMBINE_KERNEL) return PA_ERR_INVALID_ARG;
  if (o->workers < 0 || o->stages < 0 || o->stages > kMaxStages || o->warps_per_cta < 0 ||
      o->warps_per_cta > kMaxWarpsPerCta || o->tile_tokens < 0 ||
      (o->test_flags & ~PA_TEST_EXPIRE_WAITS))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pa_status_t check_tensors(const void *q, const void *k, const void *v, const int32_t *bt,
                          const int32_t *ctx, float scale, const float *out) {
  if (!q || !k || !v || !bt || !ctx || !out) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(bt, 4) || !aligned(ctx, 4))
    return PA_ERR_MISALIGNED;
  return PA_OK;
}

struct DeviceInfo {
  bool valid = false;
  int sm_count = 0, smem_optin = 0, smem_per_sm = 0, major = 0, minor = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDev];

pa_status_t current_device(int *dev, DeviceInfo *info) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDev) return PA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[*dev];
  if (!d.valid) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess)
      return PA_ERR_NO_DEVICE;
    d.valid = true;
  }
  *info = d;
  // the library is built for sm_103a only
  if (d.major != 10 || d.minor != 3) return PA_ERR_NO_DEVICE;
  return PA_OK;
}

// Shared-memory limits used when planning without a device (pa_plan): GB300 values.
constexpr int kPlanSmemOptin = 232448;
constexpr int kPlanSmemPerSm = 233472;

struct Resolved {
  pa_plan_t plan;
  int g, sub, nh_unit, nh_inst, mma, ctas_per_sm;
};

int gcd(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

pa_status_t resolve(const pa_problem_t *p, const pa_options_t *o, int sm_count, int smem_optin,
                    int smem_per_sm, Resolved *r) {
  pa_status_t st = check_problem(p);
  if (st != PA_OK) return st;
  st = check_options(o);
  if (st != PA_OK) return st;
  if (sm_count < 1) return PA_ERR_INVALID_ARG;
  std::memset(r, 0, sizeof(*r));
  pa_plan_t &pl = r->plan;
  r->g = p->query_heads / p->kv_heads;
  r->sub = ceil_div(r->g, kMaxHeads);
  r->nh_unit = ceil_div(r->g, r->sub);
  const int units = p->batch * p->kv_heads * r->sub;
  pl.units = units;
  pl.heads_per_unit = r->nh_unit;

  int math = o ? o->math : PA_MATH_AUTO;
  if (math == PA_MATH_AUTO) math = PA_MATH_MMA;
  r->mma = math == PA_MATH_MMA;
  r->nh_inst = r->mma ? kMaxHeads : simt_heads_instance(r->nh_unit);
  pl.math = math;
  if (o && o->tile_tokens && !tile_supported(p->head_dim, o->tile_tokens))
    return PA_ERR_UNSUPPORTED;
  pl.tile_tokens = tile_tokens(p->head_dim, o ? o->tile_tokens : 0);

  const int stage_bytes = pl.tile_tokens * p->head_dim * 4;
  // Measured on GB300: eight warps per SM with 16 to 24 KB in flight each saturate HBM for
  // this scattered access pattern (three 8 KB stages shorten the tail of gqa4_mid by ~1 %:
  // SMs differ in memory latency by ~5 %, and deeper rings narrow the spread); a ring that
  // costs a warp per SM, or deeper ones, only add queueing.
  int stages = (o && o->stages) ? o->stages : std::max(1, 24576 / stage_bytes);
  if (!(o && o->stages)) {
    const int floor_stages = std::max(1, 16384 / stage_bytes);
    while (stages > floor_stages &&
           kDefaultWarps * warp_smem_bytes(p->head_dim, r->mma, r->nh_inst, stages,
                                           pl.tile_tokens) +
                   kSmemAlign + kStaticSmem >
               smem_optin)
      --stages;
  }
  int per_warp = warp_smem_bytes(p->head_dim, r->mma, r->nh_inst, stages, pl.tile_tokens);
  // Eight warps per CTA: with all of them on neighbouring K/V heads (group below) their
  // reads of a row cover up to 8 * head_dim * 2 contiguous bytes.
  int warps = (o && o->warps_per_cta)
                  ? o->warps_per_cta
                  : std::min(kDefaultWarps, (smem_optin - kSmemAlign - kStaticSmem) / per_warp);
  if (warps < 1) return PA_ERR_UNSUPPORTED;
  if (warps * per_warp + kSmemAlign + kStaticSmem > smem_optin) return PA_ERR_UNSUPPORTED;
  const int smem = warps * per_warp + kSmemAlign;
  pl.stages = stages;
  pl.warps_per_cta = warps;
  pl.smem_bytes = smem;
  r->ctas_per_sm = std::max(1, smem_per_sm / (smem + kStaticSmem + kSmemReservedPerCta));
  const int capacity = sm_count * r->ctas_per_sm * warps;  // workers resident at once

  int sched = o ? o->schedule : PA_SCHEDULE_AUTO;
  if (sched == PA_SCHEDULE_AUTO) {
    // One worker per unit pays off only when the units alone fill the GPU several times
    // over and no context can be long; otherwise cut the tiles evenly across workers.
    const int64_t max_ctx = static_cast<int64_t>(p->max_pages_per_sequence) * p->page_size;
    sched = (units >= 4 * static_cast<int64_t>(capacity) && max_ctx <= 1024) ? PA_SCHEDULE_SINGLE
                                                                            : PA_SCHEDULE_BALANCED;
  }
  pl.schedule = sched;
  // Warps of a CTA are grouped onto neighbouring units (K/V heads) of one sequence and
  // walk the same tokens, so their K/V reads of a row arrive together and cover
  // group * head_dim * 2 contiguous bytes.
  pl.group = gcd(p->kv_heads * r->sub, warps);
  if (sched == PA_SCHEDULE_SINGLE) {
    pl.workers = units;
    pl.combine = PA_COMBINE_FUSED;
    pl.workspace_bytes = 0;
  } else {
    pl.workers = (o && o->workers) ? o->workers : capacity;
    pl.workers = (pl.workers + pl.group - 1) / pl.group * pl.group;
    pl.combine = o ? o->combine : PA_COMBINE_AUTO;
    if (pl.combine == PA_COMBINE_AUTO) {
      // With more units than workers most units are whole in one worker and the few shared
      // ones are merged by their last worker at no cost; with more workers than units most
      // units are shared, and a separate combine kernel (a CTA per (unit, head), launched
      // as a programmatic dependent) keeps one warp from reading every partial state at
      // the end.
      pl.combine = static_cast<int64_t>(pl.workers) >= static_cast<int64_t>(units)
                       ? PA_COMBINE_KERNEL
                       : PA_COMBINE_FUSED;
    }
    const int64_t slots = static_cast<int64_t>(units) + pl.workers;
    auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
    pl.workspace_bytes = al(slots * 4) + al(slots * kMaxHeads * 2 * 4) +
                         al(slots * kMaxHeads * p->head_dim * 4);
  }
  pl.ctas = ceil_div(std::max(pl.workers, 1), warps);
  return PA_OK;
}

// ---- TMA tensor maps ---------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a cache with a box of rows_per_box rows of one head, 64 elements wide, and
// 128-byte swizzle. Token-major caches are viewed as [num_pages * page_size rows][kv_heads]
// [head_dim] (box 64 x 1 x rows), head-major ones as [num_pages * kv_heads][page_size]
// [head_dim] (box 64 x rows x 1); either way a box lands as rows x 128 bytes.
pa_status_t encode_cache_map(CUtensorMap *map, const void *base, const pa_problem_t *p,
                             int rows_per_box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const bool hm = p->cache_layout == PA_LAYOUT_HEAD_MAJOR;
  const cuuint64_t hd = static_cast<cuuint64_t>(p->head_dim);
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3] = {64, 1, 1};
  dims[0] = hd;
  strides[0] = hd * 2;
  if (hm) {
    dims[1] = static_cast<cuuint64_t>(p->page_size);
    dims[2] = static_cast<cuuint64_t>(p->num_physical_pages) * p->kv_heads;
    strides[1] = static_cast<cuuint64_t>(p->page_size) * hd * 2;
    box[1] = static_cast<cuuint32_t>(rows_per_box);
  } else {
    dims[1] = static_cast<cuuint64_t>(p->kv_heads);
    dims[2] = static_cast<cuuint64_t>(p->num_physical_pages) * p->page_size;
    strides[1] = static_cast<cuuint64_t>(p->kv_heads) * hd * 2;
    box[2] = static_cast<cuuint32_t>(rows_per_box);
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult rc = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

namespace pa {

pa_status_t encode_cache_map_rows(CUtensorMap *map, const void *base, const pa_problem_t *p,
                                  int rows_per_box) {
  return encode_cache_map(map, base, p, rows_per_box);
}

pa_status_t encode_query_map(CUtensorMap *map, const void *query, int64_t total_tokens,
                             int query_heads, int head_dim, int heads_per_box, int tokens_per_box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const cuuint64_t hd = static_cast<cuuint64_t>(head_dim);
  cuuint64_t dims[3] = {hd, static_cast<cuuint64_t>(query_heads),
                        static_cast<cuuint64_t>(total_tokens > 0 ? total_tokens : 1)};
  cuuint64_t strides[2] = {hd * 2, static_cast<cuuint64_t>(query_heads) * hd * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(heads_per_box),
                       static_cast<cuuint32_t>(tokens_per_box)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult rc = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(query), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

pa_status_t check_problem_public(const pa_problem_t *p) { return check_problem(p); }

pa_status_t current_device_smem(int *smem_optin) {
  int dev = 0;
  DeviceInfo di;
  pa_status_t st = current_device(&dev, &di);
  if (st == PA_OK) *smem_optin = di.smem_optin;
  return st;
}

}  // namespace pa

namespace {

// ---- fused merge epochs ---------------------------------------------------------------
// Every call gets a number no earlier call in the process had (never 0); its contributors
// publish their partial states by writing it into their slots' flags. A zeroed workspace
// holds no valid number, and flags left by earlier calls (completed, aborted, or through
// another pointer into the same buffer) hold older ones, so no flag ever needs resetting.
std::atomic<uint32_t> g_epoch{0};

uint32_t next_epoch() {
  uint32_t e = ++g_epoch;
  while (e == 0) e = ++g_epoch;
  return e;
}

}  // namespace

namespace {

// ---- library-owned workspace ----------------------------------------------------------
struct Workspace {
  void *ptr = nullptr;
  size_t bytes = 0;
};
Workspace g_ws[kMaxDev];
std::mutex g_ws_mu;

pa_status_t library_workspace(int dev, size_t need, cudaStream_t stream, void **ptr) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace &w = g_ws[dev];
  if (w.bytes < need) {
    if (w.ptr) {
      if (cudaFree(w.ptr) != cudaSuccess) return PA_ERR_CUDA;
      w.ptr = nullptr;
      w.bytes = 0;
    }
    const size_t grow = need + need / 4;
    if (cudaMalloc(&w.ptr, grow) != cudaSuccess) {
      w.ptr = nullptr;
      return PA_ERR_WORKSPACE;
    }
    if (cudaMemsetAsync(w.ptr, 0, grow, stream) != cudaSuccess) return PA_ERR_CUDA;
    w.bytes = grow;
  }
  *ptr = w.ptr;
  return PA_OK;
}

void fill_args(KernelArgs *a, const pa_problem_t *p, const Resolved &r, const void *q,
               const int32_t *bt, const int32_t *ctx, float scale, float *out) {
  std::memset(a, 0, sizeof(*a));
  a->q = static_cast<const uint16_t *>(q);
  a->bt = bt;
  a->ctx = ctx;
  a->out = out;
  a->batch = p->batch;
  a->qh = p->query_heads;
  a->kvh = p->kv_heads;
  a->hd = p->head_dim;
  a->ps = p->page_size;
  a->ps_shift = ilog2(p->page_size);
  a->maxp = p->max_pages_per_sequence;
  a->num_pages = p->num_physical_pages;
  a->layout = p->cache_layout;
  a->g = r.g;
  a->sub = r.sub;
  a->nh_unit = r.nh_unit;
  a->ups = p->kv_heads * r.sub;
  a->group = r.plan.group;
  a->upg = a->ups / a->group;
  a->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a->stages = r.plan.stages;
  a->warp_smem = warp_smem_bytes(p->head_dim, r.mma, r.nh_inst, r.plan.stages, r.plan.tile_tokens);
  a->err = device_error_word();
}

}  // namespace

namespace pa {

pa_status_t validate_call(const pa_problem_t *p, const pa_options_t *o, const void *q,
                          const void *k, const void *v, const int32_t *bt, const int32_t *ctx,
                          float scale, const float *out) {
  pa_status_t st = check_problem(p);
  if (st != PA_OK) return st;
  st = check_options(o);
  if (st != PA_OK) return st;
  return check_tensors(q, k, v, bt, ctx, scale, out);
}

pa_status_t decode_into(const pa_problem_t *p, const void *q, const void *k, const void *v,
                        const int32_t *bt, const int32_t *ctx, float scale, float *out,
                        const pa_options_t *o, void *ws, size_t ws_bytes, WorkspaceKind kind,
                        cudaStream_t stream) {
  pa_status_t st = validate_call(p, o, q, k, v, bt, ctx, scale, out);
  if (st != PA_OK) return st;
  if (p->batch == 0) return PA_OK;
  int dev = 0;
  DeviceInfo di;
  st = current_device(&dev, &di);
  if (st != PA_OK) return st;
  Resolved r;
  st = resolve(p, o, di.sm_count, di.smem_optin, di.smem_per_sm, &r);
  if (st != PA_OK) return st;
  const pa_plan_t &pl = r.plan;

  if (pl.workspace_bytes > 0) {
    if (kind == WorkspaceKind::kLibrary) {
      st = library_workspace(dev, static_cast<size_t>(pl.workspace_bytes), stream, &ws);
      if (st != PA_OK) return st;
    } else if (!ws || ws_bytes < static_cast<size_t>(pl.workspace_bytes)) {
      return PA_ERR_WORKSPACE;
    } else if (!aligned(ws, 256)) {
      return PA_ERR_MISALIGNED;
    }
  }

  alignas(64) CUtensorMap tk, tv;
  const int rows = std::min(p->page_size, pl.tile_tokens);
  st = encode_cache_map(&tk, k, p, rows);
  if (st != PA_OK) return st;
  st = encode_cache_map(&tv, v, p, rows);
  if (st != PA_OK) return st;

  KernelArgs a;
  fill_args(&a, p, r, q, bt, ctx, scale, out);
  if (!a.err) return PA_ERR_CUDA;
  a.mode = pl.schedule == PA_SCHEDULE_SINGLE ? MODE_SINGLE : MODE_BALANCED;
  a.workers = pl.workers / pl.group;
  if (o && (o->test_flags & PA_TEST_EXPIRE_WAITS)) a.tx_extra = 16;
  a.fused = pl.combine == PA_COMBINE_FUSED;
  if (a.mode == MODE_BALANCED) {
    const int64_t units = pl.units;
    const int64_t slots = units + pl.workers;
    auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
    char *base = static_cast<char *>(ws);
    a.ws_flag = reinterpret_cast<unsigned *>(base);
    base += al(slots * 4);
    a.ws_ml = reinterpret_cast<float *>(base);
    base += al(slots * kMaxHeads * 2 * 4);
    a.ws_acc = reinterpret_cast<float *>(base);
  }
  a.epoch = next_epoch();
  if (launch_decode(a, &tk, &tv, r.mma, r.nh_inst, r.plan.tile_tokens, pl.ctas, pl.warps_per_cta,
                    static_cast<size_t>(pl.smem_bytes), stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if (a.mode == MODE_BALANCED && !a.fused) {
    if (launch_combine_balanced(a, pl.units, r.nh_unit,
                                combine_warps_per_pair(pl.units, pl.workers),
                                r.plan.tile_tokens, stream) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

pa_status_t pa_plan(const pa_problem_t *problem, const pa_options_t *options, int32_t sm_count,
                    pa_plan_t *plan) {
  if (!plan) return PA_ERR_INVALID_ARG;
  Resolved r;
  pa_status_t st = resolve(problem, options, sm_count, kPlanSmemOptin, kPlanSmemPerSm, &r);
  if (st != PA_OK) return st;
  *plan = r.plan;
  return PA_OK;
}

pa_status_t pa_workspace_size(const pa_problem_t *problem, const pa_options_t *options,
                              size_t *bytes) {
  if (!bytes) return PA_ERR_INVALID_ARG;
  int dev = 0;
  DeviceInfo di;
  pa_status_t st = current_device(&dev, &di);
  if (st != PA_OK) return st;
  Resolved r;
  st = resolve(problem, options, di.sm_count, di.smem_optin, di.smem_per_sm, &r);
  if (st != PA_OK) return st;
  *bytes = static_cast<size_t>(r.plan.workspace_bytes);
  return PA_OK;
}

pa_status_t pa_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace && workspace_bytes) return PA_ERR_INVALID_ARG;
  if (!workspace_bytes) return PA_OK;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_decode(const pa_problem_t *problem, const void *query, const void *key_cache,
                      const void *value_cache, const int32_t *block_tables,
                      const int32_t *context_lengths, float scale, float *out, void *stream) {
  return decode_into(problem, query, key_cache, value_cache, block_tables, context_lengths, scale,
                     out, nullptr, nullptr, 0, WorkspaceKind::kLibrary,
                     static_cast<cudaStream_t>(stream));
}

pa_status_t pa_decode_ex(const pa_problem_t *problem, const void *query, const void *key_cache,
                         const void *value_cache, const int32_t *block_tables,
                         const int32_t *context_lengths, float scale, float *out,
                         const pa_options_t *options, void *workspace, size_t workspace_bytes,
                         void *stream) {
  return decode_into(problem, query, key_cache, value_cache, block_tables, context_lengths, scale,
                     out, options, workspace, workspace_bytes, WorkspaceKind::kCaller,
                     static_cast<cudaStream_t>(stream));
}

pa_status_t pa_split_kv_partial(const pa_problem_t *problem, const void *query,
                                const void *key_cache, const void *value_cache,
                                const int32_t *block_tables, const int32_t *context_lengths,
                                float scale, int32_t num_splits, int32_t math,
                                float *partial_max, float *partial_sum, float *partial_out,
                                void *stream) {
  pa_status_t st = check_problem(problem);
  if (st != PA_OK) return st;
  if (num_splits < 1 || math < PA_MATH_AUTO || math > PA_MATH_MMA) return PA_ERR_INVALID_ARG;
  if (!partial_max || !partial_sum || !partial_out) return PA_ERR_INVALID_ARG;
  if (!aligned(partial_max, 4) || !aligned(partial_sum, 4) || !aligned(partial_out, 16))
    return PA_ERR_MISALIGNED;
  st = check_tensors(query, key_cache, value_cache, block_tables, context_lengths, scale,
                     partial_out);
  if (st != PA_OK) return st;
  if (problem->batch == 0) return PA_OK;
  int dev = 0;
  DeviceInfo di;
  st = current_device(&dev, &di);
  if (st != PA_OK) return st;
  pa_options_t o;
  std::memset(&o, 0, sizeof(o));
  o.schedule = PA_SCHEDULE_SINGLE;
  o.math = math;
  Resolved r;
  st = resolve(problem, &o, di.sm_count, di.smem_optin, di.smem_per_sm, &r);
  if (st != PA_OK) return st;
  const int64_t workers = static_cast<int64_t>(r.plan.units) * num_splits;
  if (workers >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  alignas(64) CUtensorMap tk, tv;
  const int rows = std::min(problem->page_size, r.plan.tile_tokens);
  st = encode_cache_map(&tk, key_cache, problem, rows);
  if (st != PA_OK) return st;
  st = encode_cache_map(&tv, value_cache, problem, rows);
  if (st != PA_OK) return st;
  KernelArgs a;
  fill_args(&a, problem, r, query, block_tables, context_lengths, scale, nullptr);
  if (!a.err) return PA_ERR_CUDA;
  a.mode = MODE_SPLIT;
  a.num_splits = num_splits;
  a.p_max = partial_max;
  a.p_sum = partial_sum;
  a.p_out = partial_out;
  const int ctas = static_cast<int>((workers + r.plan.warps_per_cta - 1) / r.plan.warps_per_cta);
  if (launch_decode(a, &tk, &tv, r.mma, r.nh_inst, r.plan.tile_tokens, ctas, r.plan.warps_per_cta,
                    static_cast<size_t>(r.plan.smem_bytes),
                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_split_kv_combine(const pa_problem_t *problem, int32_t num_splits,
                                const float *partial_max, const float *partial_sum,
                                const float *partial_out, float *out, void *stream) {
  pa_status_t st = check_problem(problem);
  if (st != PA_OK) return st;
  if (num_splits < 1 || !partial_max || !partial_sum || !partial_out || !out)
    return PA_ERR_INVALID_ARG;
  if (!aligned(partial_max, 4) || !aligned(partial_sum, 4) || !aligned(partial_out, 16) ||
      !aligned(out, 16))
    return PA_ERR_MISALIGNED;
  if (problem->batch == 0) return PA_OK;
  int dev = 0;
  DeviceInfo di;
  st = current_device(&dev, &di);
  if (st != PA_OK) return st;
  KernelArgs a;
  std::memset(&a, 0, sizeof(a));
  a.batch = problem->batch;
  a.qh = problem->query_heads;
  a.hd = problem->head_dim;
  a.num_splits = num_splits;
  a.p_max = const_cast<float *>(partial_max);
  a.p_sum = const_cast<float *>(partial_sum);
  a.p_out = const_cast<float *>(partial_out);
  a.out = out;
  return launch_combine_split(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                  : PA_ERR_CUDA;
}

pa_status_t pa_get_device_error(void *stream, uint32_t *flags) {
  if (!flags) return PA_ERR_INVALID_ARG;
  int dev = 0;
  DeviceInfo di;
  pa_status_t st = current_device(&dev, &di);
  if (st != PA_OK) return st;
  return read_and_clear_device_error(static_cast<cudaStream_t>(stream), flags) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

const char *pa_status_string(pa_status_t status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported problem shape";
    case PA_ERR_MISALIGNED: return "misaligned pointer";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_NO_DEVICE: return "no usable sm_103a device";
  }
  return "unknown status";
}

int32_t pa_version(void) { return kVersion; }

}  // extern "C"
