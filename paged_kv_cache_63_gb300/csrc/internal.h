// internal.h -- types shared by the host API (api.cpp) and the kernel launchers (*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#ifdef __CUDACC__
#define PA_HD __host__ __device__ __forceinline__
#else
#define PA_HD inline
#endif

namespace pa {

// Query heads one worker serves from one K/V read; a group larger than this is split
// into ceil(g / kMaxHeads) units that each read the group's K/V.
constexpr int kMaxHeads = 8;
constexpr int kMaxWarpsPerCta = 8;
constexpr int kMaxStages = 8;
constexpr int kSmemAlign = 1024;  // 128-byte TMA swizzle repeats every 1024 bytes

enum Mode : int {
  MODE_SINGLE = 0,   // one worker per unit, whole context, final output
  MODE_SPLIT = 1,    // one worker per (unit, split): fixed page ranges, partial arrays
  MODE_BALANCED = 2  // equal contiguous ranges of the concatenated tiles, merge by LSE
};

struct KernelArgs {
  const uint16_t *q;  // fp16 bits
  const int32_t *bt;
  const int32_t *ctx;
  float *out;
  // balanced-schedule workspace
  float *ws_ml;   // [slots][kMaxHeads][2]  (max in base-2 units, sum)
  float *ws_acc;  // [slots][kMaxHeads][head_dim]
  unsigned *ws_flag;  // [slots] fused merge: holds the call's epoch once the slot's partial
                      // state is written
  // fixed-split partial arrays: [batch][splits][query_heads]([head_dim])
  float *p_max;
  float *p_sum;
  float *p_out;
  unsigned *err;  // device error word
  int batch, qh, kvh, hd, ps, ps_shift, maxp, num_pages;
  int layout;   // pa_cache_layout_t
  int g;        // query heads per K/V head
  int sub;      // units per K/V head
  int nh_unit;  // heads per unit (ceil(g / sub))
  int ups;      // units per sequence = kvh * sub
  int group;    // warps per worker; warp `member` of a worker serves unit group_unit * group +
                // member, so the warps of a worker read neighbouring K/V heads together
  int upg;      // group units per sequence = ups / group
  float scale_log2;  // scale * log2(e)
  int mode;
  int num_splits;  // MODE_SPLIT
  int workers;     // MODE_BALANCED: number of workers (groups of `group` warps)
  int fused;       // MODE_BALANCED: each shared unit is merged by the worker holding its
                   // first tiles, once the other contributors' flags show `epoch`
  unsigned epoch;  // this call's number (never 0), unique within the process
  int stages;
  int warp_smem;   // bytes of dynamic shared memory per warp (multiple of kSmemAlign)
  unsigned tx_extra;  // bytes the first tile of each warp waits for beyond what it loads
                      // (nonzero only under PA_TEST_EXPIRE_WAITS)
};

// ---- schedule arithmetic shared by the kernels and the host-side checks -------------

PA_HD int tiles_of(int ctx, int tile_tokens) { return (ctx + tile_tokens - 1) / tile_tokens; }

// Balanced schedule: worker c owns global tiles [start(c), start(c+1)) with
// start(c) = floor(c * total / workers), where workers <= total (the kernel uses
// min(launched workers, total)), so every range holds at least one tile and the workers
// that share a unit are consecutive.
PA_HD int64_t worker_start(int64_t c, int64_t total, int64_t workers) {
  return (c * total) / workers;
}

// The worker whose range holds global tile x (0 <= x < total): the largest c with
// start(c) <= x, i.e. floor(((x + 1) * workers - 1) / total).
PA_HD int64_t worker_of(int64_t x, int64_t total, int64_t workers) {
  return ((x + 1) * workers - 1) / total;
}

// Partial-state slot of (unit u, worker c) when workers are groups of `group` warps that
// serve `group` consecutive units of a sequence (unit u = group_unit * group + member).
// Along the monotone path of (group_unit, worker) pairs in tile order each step raises one
// of them, so group_unit + c is unique per member and (group_unit + c) * group + member
// = u + c * group is unique; slots < units + workers * group.
PA_HD int64_t slot_of(int64_t unit, int64_t worker, int64_t group) { return unit + worker * group; }

// Warps that merge one (unit, head) pair in the separate combine kernel: enough that each
// walks at most about 8 of the unit's contributors, of which there are 1 + workers / units
// on average (workers and units both counted in warps).
inline int combine_warps_per_pair(int64_t units, int64_t workers) {
  const int64_t avg = 1 + workers / (units > 0 ? units : 1);
  int w = 1;
  while (w < 8 && avg > 8 * w) w *= 2;
  return w;
}

// ---- launchers (defined in the .cu files) --------------------------------------------

// Tokens per K/V tile for head_dim: `requested` when that size is instantiated, else the
// default (32, or 16 for head_dim 256).
int tile_tokens(int head_dim, int requested);
bool tile_supported(int head_dim, int tile);
// Dynamic shared memory one warp needs (multiple of kSmemAlign).
int warp_smem_bytes(int head_dim, int mma, int nh_inst, int stages, int tile);
// SIMT kernels are instantiated for these head counts per unit; returns the smallest
// instantiation >= nh.
int simt_heads_instance(int nh);

cudaError_t launch_decode(const KernelArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                          int mma, int nh_inst, int tile, int ctas, int warps_per_cta,
                          size_t smem, cudaStream_t stream);
// warps_per_pair: 1, 2, 4 or 8 warps merge one (unit, head) pair (combine_warps_per_pair);
// tile: the decode launch's tokens per tile (the combine redoes its split)
cudaError_t launch_combine_balanced(const KernelArgs &a, int units, int heads, int warps_per_pair,
                                    int tile, cudaStream_t stream);
cudaError_t launch_combine_split(const KernelArgs &a, cudaStream_t stream);
cudaError_t read_and_clear_device_error(cudaStream_t stream, uint32_t *flags);
unsigned *device_error_word();

}  // namespace pa

#include "pagedattn.h"

namespace pa {

// Who owns a decode call's workspace.
enum class WorkspaceKind {
  kLibrary,  // library-owned grow-only buffer, zeroed when allocated (pa_decode)
  kCaller,   // caller buffer zeroed once by pa_workspace_init (pa_decode_ex)
  kStatic    // the library's fixed scratch array, zero at load (pa_decode_noalloc)
};

// Host-side argument checks shared by the entry points (no GPU access).
pa_status_t validate_call(const pa_problem_t *p, const pa_options_t *o, const void *q,
                          const void *k, const void *v, const int32_t *bt, const int32_t *ctx,
                          float scale, const float *out);

// Tensor maps (api.cpp): a cache map whose box is rows_per_box rows of one head; a query map
// over [total_tokens][query_heads][head_dim] whose box is 64 x heads_per_box x tokens_per_box.
pa_status_t encode_cache_map_rows(CUtensorMap *map, const void *base, const pa_problem_t *p,
                                  int rows_per_box);
pa_status_t encode_query_map(CUtensorMap *map, const void *query, int64_t total_tokens,
                             int query_heads, int head_dim, int heads_per_box, int tokens_per_box);
pa_status_t check_problem_public(const pa_problem_t *p);
// The current device's opt-in shared memory per block; PA_ERR_NO_DEVICE unless sm_103.
pa_status_t current_device_smem(int *smem_optin);

// One decode step: validation, plan, workspace checks, tensor maps and launches.
pa_status_t decode_into(const pa_problem_t *p, const void *q, const void *k, const void *v,
                        const int32_t *bt, const int32_t *ctx, float scale, float *out,
                        const pa_options_t *o, void *ws, size_t ws_bytes, WorkspaceKind kind,
                        cudaStream_t stream);

}  // namespace pa
