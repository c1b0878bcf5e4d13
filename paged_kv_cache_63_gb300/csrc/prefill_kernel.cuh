// prefill_kernel.cuh -- causal multi-token attention over the paged K/V cache on the
// tcgen05 tensor cores ("[TIL] Optimizing paged attention", section "Flash Attention":
// scores of a block of query rows against a tile of keys, an online softmax, and the
// weighted sum of the tile's values, applied to the paged cache of section "Paged
// Attention" with a causal limit per query row).
//
// A work item is one (sequence b, K/V head, query tile): 128 MMA rows holding QT new tokens x
// g query heads (row = token * g + head, QT = 128 / g), so the K/V tile in shared memory
// serves every query head that reads it. Per K/V tile of TN tokens:
//   S = Q K^T        128 x TN   fp32 in TMEM (two buffers, so S(j+1) overlaps softmax(j))
//   P = exp2(S*scale*log2e - m)  fp16 in shared memory (two buffers)
//   O += P V         128 x HD   fp32 in TMEM
// The grid has one CTA per item, but CTAs stay resident: warp 7 asks the hardware to cancel
// CTAs that have not started (cluster launch control) and publishes their items, so a CTA
// runs item after item with its TMEM, barriers and rings (counted across items) kept.
// Warp roles (8 warps): 0 loads K with TMA, 6 loads Q and V; 1 owns TMEM and issues the
// MMAs warp-collectively (one elected lane of the converged warp); 2..5 run the softmax, one
// query row per thread (TMEM lane = row), rescale O in TMEM when a row's running maximum
// grows by more than 2^8, and write the output; 7 schedules.
// Every mbarrier wait is bounded; a wait that expires raises PA_DEVERR_TIMEOUT, the other
// roles stop at their next wait, in-flight copies and MMAs are drained and TMEM is freed.
#pragma once

#include "device_common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pa {

struct PrefillArgs {
  const int32_t *qs;   // [batch + 1] first query row of each sequence
  const int32_t *bt;   // [batch][maxp]
  const int32_t *ctx;  // [batch] tokens in the cache, the new ones included
  float *out;          // [total][qh][hd]
  unsigned *err;
  long long total;  // rows of query and out
  int batch, qh, kvh, ps, ps_shift, maxp, num_pages, layout;
  int g;         // query heads per K/V head
  int qt;        // new tokens per query tile (128 / g)
  int n_qtiles;  // grid.z
  float scale_log2;
  int expire;  // PA_TEST_EXPIRE_WAITS: the MMA warp's first wait is on a barrier that
               // completes only at the end, so it runs out
  int out_v8;  // out is 32-byte aligned: the two-tile kernel writes rows in 32-byte stores
};

template <int HD>
struct PrefillCfg {
  static constexpr int kRows = 128;                // MMA M
  static constexpr int KB = HD / 64;               // 64-element (128-byte) column blocks
  static constexpr int TN = HD == 256 ? 64 : 128;  // K/V tokens per tile
  static constexpr int kStages = 2;
  static constexpr int kQBytes = KB * kRows * 128;
  static constexpr int kKVBytes = TN * HD * 2;     // one K (or V) stage
  static constexpr int kPBytes = kRows * TN * 2;   // one P buffer
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kStages * kKVBytes;
  static constexpr int kPOff = kVOff + kStages * kKVBytes;
  static constexpr int kSmem = kPOff + 2 * kPBytes;  // the launch adds 1 KB for alignment
  static constexpr int kOCol = 256;                  // O columns [256, 256 + HD); S at 0 and TN
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = idesc_f16(kRows, TN, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_f16(kRows, HD, 0, 1);
};

constexpr int kPrefillThreads = 256;
constexpr int kPrefillVWarp = 6;
constexpr int kPrefillSchedWarp = 7;
// warps that read each published work item: 0, 1, the softmax warps 2..5 and 6
constexpr int kItemReaders1 = 7;
// O is rescaled only when a row's running maximum grows by more than 2^kPrefillSlackLog2;
// until then every exponent term is at most kPrefillSlackBound, which a tile's row sum may
// therefore be checked against.
constexpr int kPrefillSlackLog2 = 8;
constexpr float kPrefillRescaleSlack = static_cast<float>(kPrefillSlackLog2);  // log2 units
constexpr float kPrefillSlackBound = static_cast<float>(1 << kPrefillSlackLog2);

// Barrier slots.
enum : int {
  kBarQ = 0,
  kBarKFull = 1,   // +stage
  kBarKEmpty = 3,  // +stage
  kBarVFull = 5,
  kBarVEmpty = 7,
  kBarSFull = 9,   // +buffer
  kBarPFull = 11,  // +buffer (128 arrivals: the softmax threads)
  kBarPV = 13,     // +buffer: the P.V MMAs of that buffer completed
  kBarDone = 15,
  kBarQEmpty = 16,     // the item's last score MMA completed: Q may be replaced
  kBarItemFull = 17,   // +entry: a work item is published
  kBarItemEmpty = 19,  // +entry: every reader has taken it (kItemReaders1 arrivals)
  kBarProdStart = 21,  // the K producer started an item: time to ask for the next one
  kBarClc = 22,        // the answer to a cancellation request landed (16 bytes)
  kNumBars = 23
};

// L2 policy for bytes that other CTAs read again soon: keep them ahead of streamed data.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ float prefill_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100 family): one instruction does two FMAs or two adds.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// P = exp2(s * sl2 + nm) over a row of TN scores, in place, with keys past lim (when the row
// is not full) giving exactly 0, and the row's partial sums in rp. Packed fp32 pairs: one
// FFMA2 gives two exponent arguments and one FADD2 adds two terms to the sums.
template <int TN>
__device__ __forceinline__ void exps_row(float (&x)[TN], float sl2, float nm, bool full, int lim,
                                         float (&rp)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) rp[e] = 0.f;
#pragma unroll
  for (int c = 0; c < TN; c += 2) {
    const float2 xx = ffma2(make_float2(x[c], x[c + 1]), make_float2(sl2, sl2), make_float2(nm, nm));
    const float p0 = (full || c <= lim) ? prefill_exp2(xx.x) : 0.f;
    const float p1 = (full || c + 1 <= lim) ? prefill_exp2(xx.y) : 0.f;
    const float2 acc = fadd2(make_float2(rp[c & 7], rp[(c + 1) & 7]), make_float2(p0, p1));
    rp[c & 7] = acc.x;
    rp[(c + 1) & 7] = acc.y;
    x[c] = p0;
    x[c + 1] = p1;
  }
}

// 32-byte store (one full sector) of 8 floats with an L2 eviction-priority policy.
__device__ __forceinline__ void st_global_v8(float *p, float v0, float v1, float v2, float v3,
                                             float v4, float v5, float v6, float v7, uint64_t pol) {
  asm volatile(
      "st.global.L2::cache_hint.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p),
      "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Warp-collective bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool pipe_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *err) {
  bool ok = mbar_try_wait(bar, parity);
  bool expired = false;
  if (!ok) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
      if ((i & 31u) == 0) {
        if (*abort_flag) break;
        if (global_ns() - t0 > kWaitLimitNs) {
          expired = true;
          break;
        }
      }
    }
  }
  ok = __all_sync(0xffffffffu, ok);
  expired = __any_sync(0xffffffffu, expired);
  if (!ok && (threadIdx.x & 31) == 0) {
    if (expired) atomicOr(err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  }
  return ok;
}

// Bounded wait used while draining (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned *err) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
      if ((i & 31u) == 0 && global_ns() - t0 > kWaitLimitNs) break;
    }
  }
  if (!ok) atomicOr(err, PA_DEVERR_TIMEOUT);
}

// ---- cluster launch control -------------------------------------------------------------
// Ask for one CTA of this grid that has not started to be cancelled so that the caller runs
// its work; the 16-byte answer is written to shared memory and completes `bar` with 16 bytes
// of transaction count.
__device__ __forceinline__ void clc_try_cancel(uint32_t answer, uint32_t bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
      " [%0], [%1];" ::"r"(answer), "r"(bar)
      : "memory");
}

// Read an answer: true and the cancelled CTA's index if a CTA was cancelled, false when
// every CTA of the grid has started (no work is left to take).
__device__ __forceinline__ bool clc_query(uint32_t answer, int &x, int &y, int &z) {
  uint32_t ok, cx = 0, cy = 0, cz = 0;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\tld.shared.b128 r, [%4];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %3, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid.v4.b32.b128 {%0, %1, %2, _}, r;\n\t}"
      : "+r"(cx), "+r"(cy), "+r"(cz), "=r"(ok)
      : "r"(answer)
      : "memory");
  x = static_cast<int>(cx);
  y = static_cast<int>(cy);
  z = static_cast<int>(cz);
  return ok != 0;
}

// Geometry of one work item (K/V head kv, sequence b, query tile), computed once by the
// scheduler and published to every role. `live` is 0 when the tile holds no new token or the
// sequence's offsets or length are out of range (those are flagged here); `stop` marks the
// end of the CTA's work.
struct Item1 {
  int kv, b, q0, n, tok0, base_pos, max_pos, kv_len, ntiles;
  int live, stop;
};

template <int TN>
__device__ __forceinline__ Item1 item1_of(const PrefillArgs &a, int kv, int b, int qtile) {
  Item1 it;
  it.kv = kv;
  it.b = b;
  it.live = 0;
  it.stop = 0;
  it.ntiles = 0;
  const int q0 = __ldg(a.qs + b), q1 = __ldg(a.qs + b + 1), ctx = __ldg(a.ctx + b);
  const int n = q1 - q0;
  it.q0 = q0;
  it.n = n;
  if (ctx < 0 || static_cast<long long>(ctx) > static_cast<long long>(a.maxp) << a.ps_shift) {
    atomicOr(a.err, PA_DEVERR_CONTEXT);
    return it;
  }
  if (q0 < 0 || n < 0 || static_cast<long long>(q1) > a.total || n > ctx) {
    atomicOr(a.err, PA_DEVERR_QUERY_START);
    return it;
  }
  it.tok0 = qtile * a.qt;
  if (it.tok0 >= n) return it;
  it.base_pos = ctx - n + it.tok0;                       // position of the tile's token 0
  it.max_pos = ctx - n + min(it.tok0 + a.qt, n) - 1;     // last position any row sees
  it.kv_len = it.max_pos + 1;
  it.ntiles = (it.kv_len + TN - 1) / TN;
  it.live = 1;
  return it;
}

template <int HD>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using C = PrefillCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ __align__(16) uint4 clc_answer;
  __shared__ Item1 items[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_word;
  volatile int *abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q_rows = a.qt * a.g;

  const uint32_t sbase = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t *sgen = smem_raw + (sbase - smem_addr(smem_raw));
  const uint32_t sq = sbase + C::kQOff;
  auto k_stage = [&](int s) { return sbase + C::kKOff + s * C::kKVBytes; };
  auto v_stage = [&](int s) { return sbase + C::kVOff + s * C::kKVBytes; };
  auto p_buf = [&](int s) { return sbase + C::kPOff + s * C::kPBytes; };
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i == kBarPFull || i == kBarPFull + 1) count = 128;
      if (i == kBarItemEmpty || i == kBarItemEmpty + 1) count = kItemReaders1;
      mbar_init(bar(i), count);
    }
    abort_word = 0;
    fence_barrier_init();
  }
  // Rows of Q past q_rows are never loaded: zero them once so their (discarded) results stay
  // finite.
  if (q_rows < C::kRows) {
    const int per_block = (C::kRows - q_rows) * 8;  // 16-byte chunks
    for (int i = threadIdx.x; i < C::KB * per_block; i += kPrefillThreads) {
      const int kb = i / per_block, c = i % per_block;
      *reinterpret_cast<uint4 *>(sgen + C::kQOff + kb * (C::kRows * 128) + q_rows * 128 + c * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Reader side of the item ring: item k sits in entry k & 1. Returns false on abort.
  auto take_item = [&](int k, Item1 &it) {
    if (!pipe_wait(bar(kBarItemFull + (k & 1)), (k >> 1) & 1, abort_flag, a.err)) return false;
    it = items[k & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarItemEmpty + (k & 1)));
    return true;
  };

  // K/V tiles, S and P buffers and their barrier phases are numbered across the work items
  // a CTA runs: tile t (global) uses stage / buffer t & 1 and phase (t >> 1) & 1.
  if (warp == kPrefillSchedWarp) {
    // ================= scheduler: one request per item (as in prefill2_kernel) =================
    int kv = blockIdx.x, b = blockIdx.y, z = blockIdx.z;
    bool stop = false;
    const uint32_t answer = smem_addr(&clc_answer);
    for (int k = 0;; ++k) {
      if (k >= 2 && !pipe_wait(bar(kBarItemEmpty + (k & 1)), ((k >> 1) - 1) & 1, abort_flag, a.err))
        break;
      if (lane == 0) {
        if (stop) {
          items[k & 1].stop = 1;
          items[k & 1].live = 0;
        } else {
          items[k & 1] = item1_of<C::TN>(a, kv, b, a.n_qtiles - 1 - z);  // longest rows first
        }
        mbar_arrive(bar(kBarItemFull + (k & 1)));
      }
      __syncwarp();
      if (stop) break;
      if (!pipe_wait(bar(kBarProdStart), k & 1, abort_flag, a.err)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kBarClc), 16);
        clc_try_cancel(answer, bar(kBarClc));
      }
      __syncwarp();
      if (!pipe_wait(bar(kBarClc), k & 1, abort_flag, a.err)) {
        if (lane == 0) drain_wait(bar(kBarClc), k & 1, a.err);  // the answer's write lands first
        __syncwarp();
        break;
      }
      int x, y, zz;
      // after a failed request (every CTA has started) no other may be made
      stop = !clc_query(answer, x, y, zz) || x >= static_cast<int>(gridDim.x) ||
             y >= static_cast<int>(gridDim.y) || zz >= static_cast<int>(gridDim.z);
      kv = x;
      b = y;
      z = zz;
    }
  } else if (warp == 0 || warp == kPrefillVWarp) {
    // ============ producers: warp 0 the K tiles, warp 6 Q and the V tiles ============
    const bool is_v = warp == kPrefillVWarp;
    if (lane == 0) {
      prefetch_tensormap(is_v ? &tv : &tk);
      if (is_v) prefetch_tensormap(&tq);
    }
    const CUtensorMap *map = is_v ? &tv : &tk;
    // every query tile of the (sequence, K/V head) reads these K/V tiles: keep them in L2
    const uint64_t pol = l2_evict_last_policy();
    const int full = is_v ? kBarVFull : kBarKFull;
    const int empty = is_v ? kBarVEmpty : kBarKEmpty;
    const uint32_t stage0 = is_v ? v_stage(0) : k_stage(0);
    const int rows_per_box = min(a.ps, C::TN);
    const int boxes = C::TN / rows_per_box;
    const uint32_t box_bytes = rows_per_box * 128;
    int g = 0;  // global index of the next tile
    int q_loads = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item1 it;
      ok = take_item(k, it);
      if (!ok || it.stop) break;
      if (!is_v && lane == 0) mbar_arrive(bar(kBarProdStart));
      if (!it.live) continue;
      if (is_v) {
        // Q of this item, once the previous item's last score MMA has read the buffer
        if (q_loads > 0) ok = pipe_wait(bar(kBarQEmpty), (q_loads - 1) & 1, abort_flag, a.err);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(kBarQ), C::KB * q_rows * 128);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sq + kb * (C::kRows * 128), &tq, bar(kBarQ), kb * 64, it.kv * a.g,
                        it.q0 + it.tok0, l2_evict_first_policy());  // read once
        }
        ++q_loads;
      }
      const int32_t *bt_row = a.bt + static_cast<size_t>(it.b) * a.maxp;
      // page of this lane's box of tile j (lanes < boxes); -1 past the last needed token
      auto page_of = [&](int j) {
        const int tok = j * C::TN + lane * rows_per_box;
        return (j < it.ntiles && lane < boxes && tok < it.kv_len)
                   ? __ldg(bt_row + (tok >> a.ps_shift))
                   : -1;
      };
      // the block-table read for tile j + 1 is issued before the waits of tile j
      int page_next = page_of(0);
      for (int j = 0; j < it.ntiles && ok; ++j, ++g) {
        const int st = g & 1;
        const int tok = j * C::TN + lane * rows_per_box;
        int page = page_next;
        page_next = page_of(j + 1);
        if (lane < boxes && tok < it.kv_len && (page < 0 || page >= a.num_pages)) {
          if (!is_v) atomicOr(a.err, PA_DEVERR_PAGE_ID);
          page = -1;
        }
        const uint32_t issue = __ballot_sync(0xffffffffu, page >= 0);
        const int slot = tok & (a.ps - 1);
        int y, z;
        if (a.layout == PA_LAYOUT_HEAD_MAJOR) {
          y = slot;
          z = page * a.kvh + it.kv;
        } else {
          y = it.kv;
          z = (page << a.ps_shift) + slot;
        }
        if (g >= 2) ok = pipe_wait(bar(empty + st), ((g >> 1) - 1) & 1, abort_flag, a.err);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(bar(full + st), __popc(issue) * box_bytes * C::KB);
        __syncwarp();
        if (page >= 0) {
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(stage0 + st * C::kKVBytes + kb * (C::TN * 128) + lane * box_bytes, map,
                        bar(full + st), kb * 64, y, z, pol);
        }
      }
    }
    // drain: the last load issued into each stage, and the last Q, have landed before the CTA
    // exits (older loads of a stage were consumed before it was refilled)
    if (lane == 0) {
      if (is_v && q_loads > 0) drain_wait(bar(kBarQ), (q_loads - 1) & 1, a.err);
      for (int t = max(0, g - 2); t < g; ++t) drain_wait(bar(full + (t & 1)), (t >> 1) & 1, a.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    bool ok = true;
    // PA_TEST_EXPIRE_WAITS: the first wait is on kBarDone, which no one completes before the end
    if (a.expire) ok = pipe_wait(bar(kBarDone), 0, abort_flag, a.err);
    int g = 0, q_waits = 0;
    for (int k = 0; ok; ++k) {
      Item1 it;
      ok = take_item(k, it);
      if (!ok || it.stop) break;
      if (!it.live) continue;
      ok = pipe_wait(bar(kBarQ), q_waits & 1, abort_flag, a.err);
      ++q_waits;
      if (!ok) break;
      tc_fence_after();
      const int rows_last = it.kv_len - (it.ntiles - 1) * C::TN;  // valid rows of the last V tile
      for (int j = 0; j <= it.ntiles && ok; ++j) {
        if (j < it.ntiles) {
          const int t = g + j, st = t & 1;
          ok = pipe_wait(bar(kBarKFull + st), (t >> 1) & 1, abort_flag, a.err);
          if (!ok) break;
          tc_fence_after();
          {
            // issued warp-collectively by one elected lane of the converged warp, with
            // descriptors = base descriptor + step offset / 16 (the empty asm keeps the
            // compiler from hoisting every step's descriptor into registers)
            const uint32_t d = tmem + st * C::TN;
            uint64_t qd = smem_desc_sw128(sq, 16, 1024);
            uint64_t kd = smem_desc_sw128(k_stage(st), 16, 1024);
            asm volatile("" : "+l"(qd), "+l"(kd));
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
              const uint64_t ad = qd + (((ks >> 2) * (C::kRows * 128) + (ks & 3) * 32) >> 4);
              const uint64_t bd = kd + (((ks >> 2) * (C::TN * 128) + (ks & 3) * 32) >> 4);
              mma_f16_ss_warp(d, ad, bd, C::kIdescS, ks > 0);
            }
            mma_commit_warp(bar(kBarSFull + st));
            mma_commit_warp(bar(kBarKEmpty + st));
            if (j == it.ntiles - 1) mma_commit_warp(bar(kBarQEmpty));
          }
        }
        if (j >= 1) {
          const int i = j - 1, t = g + i, st = t & 1;
          ok = pipe_wait(bar(kBarPFull + st), (t >> 1) & 1, abort_flag, a.err);
          if (ok) ok = pipe_wait(bar(kBarVFull + st), (t >> 1) & 1, abort_flag, a.err);
          if (!ok) break;
          tc_fence_after();
          if (i == it.ntiles - 1 && rows_last < C::TN) {
            // V rows past the last needed token hold unread cache slots (possibly never
            // written); P is zero there, but 0 * NaN is not, so clear them.
            const int per_block = (C::TN - rows_last) * 8;
            uint8_t *vg = sgen + C::kVOff + st * C::kKVBytes;
            for (int c = lane; c < C::KB * per_block; c += 32) {
              const int kb = c / per_block, r = c % per_block;
              *reinterpret_cast<uint4 *>(vg + kb * (C::TN * 128) + rows_last * 128 + r * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
            __syncwarp();
          }
          {
            // the item's first P.V overwrites O: the softmax released this P only after it
            // had read the previous item's O
            uint64_t pd = smem_desc_sw128(p_buf(st), 16, 1024);
            uint64_t vd = smem_desc_sw128(v_stage(st), C::TN * 128, 1024);
            asm volatile("" : "+l"(pd), "+l"(vd));
#pragma unroll
            for (int ks = 0; ks < C::TN / 16; ++ks) {
              const uint64_t ad = pd + (((ks >> 2) * (C::kRows * 128) + (ks & 3) * 32) >> 4);
              const uint64_t bd = vd + ((ks * 2048) >> 4);
              mma_f16_ss_warp(tmem + C::kOCol, ad, bd, C::kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit_warp(bar(kBarPV + st));
            mma_commit_warp(bar(kBarVEmpty + st));
          }
        }
      }
      g += it.ntiles;
    }
    // every MMA this warp issued has completed before TMEM is released
    mma_commit_warp(bar(kBarDone));
    if (lane == 0) drain_wait(bar(kBarDone), 0, a.err);
    __syncwarp();
  } else if (warp >= 2 && warp <= 5) {
    // ================= softmax: one query row per thread =================
    const int rg = warp & 3;
    const int row = rg * 32 + lane;
    const int t = row / a.g, h = row - t * a.g;
    const uint32_t trow = tmem + (static_cast<uint32_t>(rg * 32) << 16);
    const float sl2 = a.scale_log2;
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item1 it;
      ok = take_item(k, it);
      if (!ok || it.stop) break;
      if (!it.live) continue;
      const bool valid = row < q_rows && it.tok0 + t < it.n;
      const int pos = min(it.base_pos + t, it.max_pos);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.ntiles; ++j) {
        const int gj = g + j, st = gj & 1;
        ok = pipe_wait(bar(kBarSFull + st), (gj >> 1) & 1, abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        float x[C::TN];
#pragma unroll
        for (int c = 0; c < C::TN / 32; ++c) {
          float v[32];
          tmem_ld32(trow + st * C::TN + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c * 32 + e] = v[e];
        }
        const int lim = pos - j * C::TN;
        const bool full = lim >= C::TN - 1;
        float rp[8];
        // After a row's first tile its running maximum m seldom grows by more than the slack,
        // so a tile first takes its exponents with m as it stands and no maximum pass: the
        // terms are non-negative (masked keys give 0), so the tile's row sum bounds each of
        // them, and a sum of at most 2^slack shows that no score passed m + slack. Only a warp
        // in which some row's sum is larger (or not a number) reloads the scores and takes
        // the plain order: maximum, rescale, exponents.
        bool redo = true;
        if (j > 0) {
          if (__all_sync(0xffffffffu, full))
            exps_row<C::TN>(x, sl2, -m, true, lim, rp);  // no key of the warp's rows masked
          else
            exps_row<C::TN>(x, sl2, -m, full, lim, rp);
          const float tsum =
              ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
          redo = __any_sync(0xffffffffu, !(tsum <= kPrefillSlackBound));
          if (redo) {
#pragma unroll
            for (int c = 0; c < C::TN / 32; ++c) {
              float v[32];
              tmem_ld32(trow + st * C::TN + c * 32, v);
#pragma unroll
              for (int e = 0; e < 32; ++e) x[c * 32 + e] = v[e];
            }
          }
        }
        if (redo) {
          // keys past this row's position are masked out; the row maximum of the scaled scores
          // (log2 units) is the extreme raw score times the scale (the maximum for a
          // non-negative scale, else the minimum), which saves a multiply per score; eight
          // independent partial extremes keep the reduction off one dependency chain
          float mp[8];
          float ext;
          if (sl2 >= 0.f) {
#pragma unroll
            for (int e = 0; e < 8; ++e) mp[e] = -INFINITY;
#pragma unroll
            for (int c = 0; c < C::TN; ++c) mp[c & 7] = fmaxf(mp[c & 7], (full || c <= lim) ? x[c] : -INFINITY);
            ext = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                        fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) mp[e] = INFINITY;
#pragma unroll
            for (int c = 0; c < C::TN; ++c) mp[c & 7] = fminf(mp[c & 7], (full || c <= lim) ? x[c] : INFINITY);
            ext = fminf(fminf(fminf(mp[0], mp[1]), fminf(mp[2], mp[3])),
                        fminf(fminf(mp[4], mp[5]), fminf(mp[6], mp[7])));
          }
          const float mx = ext * sl2;
          const bool grow = mx > m + kPrefillRescaleSlack;
          if (__any_sync(0xffffffffu, grow)) {
            const float mnew = grow ? mx : m;
            // 0 on the first tile (m = -inf); 1 for rows whose maximum did not grow
            const float f = mnew == -INFINITY ? 1.f : prefill_exp2(m - mnew);
            l *= f;
            if (j > 0) {
              // O holds tiles < j: wait for the last P.V, then scale this row of O in TMEM
              ok = pipe_wait(bar(kBarPV + ((gj - 1) & 1)), ((gj - 1) >> 1) & 1, abort_flag, a.err);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int c = 0; c < HD / 32; ++c) {
                float v[32];
                tmem_ld32(trow + C::kOCol + c * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= f;
                tmem_st32(trow + C::kOCol + c * 32, v);
              }
              tmem_wait_st();
            }
            m = mnew;
          }
          // P = exp2(s * scale * log2e - m): the scale is folded into one FMA per score (packed
          // fp32 pairs: one FFMA2 for two exponents, one FADD2 for two sums); masked keys give 0
          exps_row<C::TN>(x, sl2, -m, full, lim, rp);
        }
        l += ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
        // P buffer st was last read by the P.V of global tile gj - 2
        if (gj >= 2) {
          ok = pipe_wait(bar(kBarPV + st), ((gj >> 1) - 1) & 1, abort_flag, a.err);
          if (!ok) break;
        }
        const uint32_t prow = p_buf(st) + row * 128;
#pragma unroll
        for (int c8 = 0; c8 < C::TN / 8; ++c8) {
          uint4 w;
          w.x = pack_half2(x[c8 * 8 + 0], x[c8 * 8 + 1]);
          w.y = pack_half2(x[c8 * 8 + 2], x[c8 * 8 + 3]);
          w.z = pack_half2(x[c8 * 8 + 4], x[c8 * 8 + 5]);
          w.w = pack_half2(x[c8 * 8 + 6], x[c8 * 8 + 7]);
          sts128(prow + (c8 >> 3) * (C::kRows * 128) + (((c8 & 7) ^ (row & 7)) << 4), w);
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + st));
      }
      if (ok) {
        const int tl = g + it.ntiles - 1;
        ok = pipe_wait(bar(kBarPV + (tl & 1)), (tl >> 1) & 1, abort_flag, a.err);
      }
      if (ok) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *dst = a.out + (static_cast<size_t>(it.q0 + it.tok0 + t) * a.qh + it.kv * a.g + h) * HD;
        // whole 32-byte sectors where out allows (L2 then never fills a partly written sector
        // from DRAM); the output is read by no kernel here, so it leaves L2 first. Once these
        // loads have returned, O may be overwritten by the next item's first P.V, which waits
        // for this warp's next P.
        const uint64_t pol = l2_evict_first_policy();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float v[32];
          tmem_ld32(trow + C::kOCol + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= inv;
          if (valid) {
            if (a.out_v8) {
#pragma unroll
              for (int e = 0; e < 32; e += 8)
                st_global_v8(dst + c * 32 + e, v[e], v[e + 1], v[e + 2], v[e + 3], v[e + 4],
                             v[e + 5], v[e + 6], v[e + 7], pol);
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(dst + c * 32 + e) =
                    make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            }
          }
        }
      }
      g += it.ntiles;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace pa
