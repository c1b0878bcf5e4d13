// decode_kernel.cuh -- the paged decode attention kernel for sm_103a.
//
// Method ("[TIL] Optimizing paged attention", retepy.com): for each sequence b and query
// head h, out = softmax(scale * q K^T) V over the sequence's context, where token t is at
// physical page block_tables[b][t / page_size], slot t % page_size (sections "Data Layout"
// and "Baseline"), the softmax is accumulated online (running max, rescaled sum and
// accumulator; section "Baseline"), all query heads of a GQA group are served from one
// K/V read (section "V3 (Shared memory data reuse)"), and long contexts are split across
// workers whose (max, sum, partial output) states are merged by log-sum-exp (section
// "V4 (Context-axis parallelism)").
//
// GB300 design:
//  * A worker is one warp with a private ring of `stages` shared-memory K/V tiles of T
//    tokens. Lane 0 issues TMA tensor loads (3-D map over [rows][kv_heads][head_dim],
//    128-byte swizzle) for each page piece of a tile, one tile per mbarrier; the warp
//    waits on the barrier, computes, and refills the slot S-1 tiles ahead. Warps never
//    synchronise with each other.
//  * Work units are (sequence, K/V head, head subgroup); a unit serves up to 8 query heads
//    from one K/V read. Scores and the online softmax stay in fp32 registers, in base-2
//    units (scale * log2 e folded in), with ex2.approx.
//  * Math variants: SIMT (lanes over tokens for q.k, lanes over head_dim for p.V) and
//    MMA (m16n8k16 fp16 tensor-core tiles: S[8 heads x 16 tokens] = Q K^T with K fragments
//    by ldmatrix, then O += P V with the score fragments reused as the A operand and V
//    fragments by ldmatrix.trans).
//  * Schedules: SINGLE (a worker per unit), SPLIT (a worker per (unit, page range), the
//    pages' fixed split) and BALANCED (the concatenated tiles of all units cut into one
//    equal contiguous range per worker; a unit shared by several workers is merged by
//    log-sum-exp, by the last of its workers or by a separate combine kernel).
#pragma once

#include <type_traits>

#include "device_common.cuh"
#include "internal.h"

namespace pa {

template <int HD, int T>
struct Geom {
  static constexpr int kHalfBytes = T * HD * 2;  // the K (or V) part of a stage
  static constexpr int kStageBytes = 2 * kHalfBytes;
};

// Byte offset of 16-byte chunk `chunk` (0 .. HD/8 - 1) of tile row `row`, as TMA lays a
// [T rows][64 halves] box down with 128-byte swizzle: column block chunk / 8 is a
// [T][128 B] array, and inside every 8-row group the chunk index is XORed with row & 7.
template <int HD, int T>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (T * 128) + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Context length of sequence b, clamped to [0, max_pages * page_size]; a value outside
// that range raises PA_DEVERR_CONTEXT.
__device__ __forceinline__ int load_ctx(const KernelArgs &a, int b) {
  int c = __ldg(a.ctx + b);
  const int cap = a.maxp << a.ps_shift;
  if (c < 0 || c > cap) {
    atomicOr(a.err, PA_DEVERR_CONTEXT);
    c = c < 0 ? 0 : cap;
  }
  return c;
}

// Position of a worker in its token stream.
struct Cursor {
  int b;         // sequence
  int us;        // group unit within the sequence; this warp's unit is us * group + member
  int tok;       // first token of the current tile
  int end;       // exclusive token bound of the current unit segment
  int left;      // tiles still to visit
  long long ug0;  // balanced schedule: global index of the unit's first tile
};

// Balanced schedule: step to the next unit with at least one tile.
__device__ __forceinline__ void next_unit(const KernelArgs &a, Cursor &c, int T) {
  c.ug0 += tiles_of(c.end, T);
  c.tok = 0;
  if (++c.us == a.upg) {
    c.us = 0;
    do {
      ++c.b;
      c.end = (c.b < a.batch) ? load_ctx(a, c.b) : 1;
    } while (c.b < a.batch && c.end == 0);
  }
}

__device__ __forceinline__ void advance(const KernelArgs &a, Cursor &c, int T) {
  c.tok += T;
  --c.left;
  if (a.mode == MODE_BALANCED && c.left > 0 && c.tok >= c.end) next_unit(a, c, T);
}

// Balanced schedule: total tiles over all units, the number of workers that get tiles
// (min(workers, total), so that every such worker's range is non-empty and the workers
// sharing a unit are consecutive), and the cursor at this worker's first tile. Returns
// false when the worker gets no tiles.
__device__ inline bool balanced_start(const KernelArgs &a, int worker, int T, Cursor &c,
                                      long long &total, long long &nworkers) {
  const int lane = threadIdx.x & 31;
  // lane l owns the contiguous sequences [b0, b1); its loads are independent of each
  // other, so the whole scan costs about one memory round trip
  const int blk = (a.batch + 31) >> 5;
  const int b0 = min(lane * blk, a.batch);
  const int b1 = min(b0 + blk, a.batch);
  long long mine = 0;
#pragma unroll 16
  for (int b = b0; b < b1; ++b) mine += tiles_of(load_ctx(a, b), T);
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(0xffffffffu, incl, 31) * a.upg;
  nworkers = total < a.workers ? total : a.workers;
  if (worker >= nworkers) return false;
  const long long s = worker_start(worker, total, nworkers);
  const long long e = worker_start(worker + 1, total, nworkers);
  // the lane whose block holds global tile s, then that block walked 32 sequences at a time
  const int L = __ffs(__ballot_sync(0xffffffffu, incl * a.upg > s)) - 1;
  long long run = __shfl_sync(0xffffffffu, incl - mine, L) * a.upg;
  const int lb0 = min(L * blk, a.batch);
  const int lb1 = min(lb0 + blk, a.batch);
  for (int base = lb0; base < lb1; base += 32) {
    const int b = base + lane;
    const long long t = b < lb1 ? static_cast<long long>(tiles_of(load_ctx(a, b), T)) * a.upg : 0;
    long long in2 = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, in2, o);
      if (lane >= o) in2 += y;
    }
    const long long chunk = __shfl_sync(0xffffffffu, in2, 31);
    if (s < run + chunk) {
      const int M = __ffs(__ballot_sync(0xffffffffu, run + in2 > s)) - 1;
      const long long excl = run + __shfl_sync(0xffffffffu, in2 - t, M);
      c.b = base + M;
      c.end = load_ctx(a, c.b);
      const int tb = tiles_of(c.end, T);
      const long long inner = s - excl;
      c.us = static_cast<int>(inner / tb);
      c.tok = static_cast<int>(inner % tb) * T;
      c.ug0 = excl + static_cast<long long>(c.us) * tb;
      c.left = static_cast<int>(e - s);
      return true;
    }
    run += chunk;
  }
  return false;
}

// A 64-entry window of one sequence's block-table row, held one entry per lane in two
// registers (entries base..base+31 and base+32..base+63); the second half is loaded one
// window ahead so the TMA issue rarely waits on a block-table read. Entries at or past
// `npages` (the pages the context needs) are never read.
struct BtWindow {
  int b, base, cur, nxt;
};

__device__ __forceinline__ int bt_load(const KernelArgs &a, int b, int lp, int npages) {
  return lp < npages ? __ldg(a.bt + static_cast<long long>(b) * a.maxp + lp) : -1;
}

__device__ __forceinline__ int bt_page(const KernelArgs &a, BtWindow &w, int b, int lp,
                                       int npages) {
  const int lane = threadIdx.x & 31;
  if (b != w.b || lp < w.base || lp >= w.base + 64) {
    w.b = b;
    w.base = lp & ~31;
    w.cur = bt_load(a, b, w.base + lane, npages);
    w.nxt = bt_load(a, b, w.base + 32 + lane, npages);
  } else if (lp >= w.base + 32) {
    w.base += 32;
    w.cur = w.nxt;
    w.nxt = bt_load(a, b, w.base + 32 + lane, npages);
  }
  return __shfl_sync(0xffffffffu, w.cur, lp - w.base);
}

// Issue the TMA loads of the tile at cursor c into a stage (warp-uniform call).
template <int HD, int T>
__device__ __forceinline__ void issue_tile(const KernelArgs &a, const CUtensorMap *tk,
                                           const CUtensorMap *tv, const Cursor &c, int member,
                                           BtWindow &w, uint32_t stage, uint32_t bar,
                                           uint64_t pol, uint32_t extra_tx) {
  constexpr int kMaxPieces = T / 8;
  const int R = a.ps < T ? a.ps : T;  // rows per piece: a piece never crosses a page
  const int pieces = T / R;
  const int kv = (c.us * a.group + member) / a.sub;
  const int npages = (c.end + a.ps - 1) >> a.ps_shift;
  // TMA coordinates of each piece: token-major (y, z) = (kv, page * ps + slot),
  // head-major (y, z) = (slot, page * kv_heads + kv); z < 0 marks a piece not loaded
  int yc[kMaxPieces], zc[kMaxPieces];
  uint32_t bytes = 0;
#pragma unroll
  for (int p = 0; p < kMaxPieces; ++p) {
    zc[p] = -1;
    yc[p] = 0;
    const int tok = c.tok + p * R;
    if (p < pieces && tok < c.end) {
      const int page = bt_page(a, w, c.b, tok >> a.ps_shift, npages);
      if (page < 0 || page >= a.num_pages) {
        if ((threadIdx.x & 31) == 0) atomicOr(a.err, PA_DEVERR_PAGE_ID);
      } else {
        const int slot = tok & (a.ps - 1);
        if (a.layout == PA_LAYOUT_HEAD_MAJOR) {
          yc[p] = slot;
          zc[p] = page * a.kvh + kv;
        } else {
          yc[p] = kv;
          zc[p] = (page << a.ps_shift) + slot;
        }
        bytes += static_cast<uint32_t>(R * HD * 4);
      }
    }
  }
  if ((threadIdx.x & 31) == 0) {
    mbar_arrive_expect_tx(bar, bytes + extra_tx);
#pragma unroll
    for (int p = 0; p < kMaxPieces; ++p) {
      if (zc[p] < 0) continue;
#pragma unroll
      for (int blk = 0; blk < HD / 64; ++blk) {
        const uint32_t dst = stage + blk * (T * 128) + p * R * 128;
        tma_load_3d(dst, tk, bar, blk * 64, yc[p], zc[p], pol);
        tma_load_3d(dst + Geom<HD, T>::kHalfBytes, tv, bar, blk * 64, yc[p], zc[p], pol);
      }
    }
  }
}

// ------------------------------------------------------------------ SIMT arithmetic
template <int HD, int NH>
struct SimtState {
  static constexpr int DPL = HD / 32;
  float m[NH], lsum[NH];
  float acc[NH][DPL];
};

template <int NH>
struct Nhp {
  static constexpr int v = (NH + 3) & ~3;
};

template <int HD, int NH>
__device__ __forceinline__ void simt_begin(SimtState<HD, NH> &st, const KernelArgs &a, int b,
                                           int h0, int nh, uint32_t qs) {
  const int lane = threadIdx.x & 31;
  const uint16_t *src = a.q + (static_cast<long long>(b) * a.qh + h0) * HD;
  for (int i = lane; i < NH * HD / 8; i += 32) {
    const int h = i / (HD / 8);
    const int d8 = i % (HD / 8);
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = 0.f;
    if (h < nh) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src + h * HD + d8 * 8));
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 v = half2_bits_to_float2(w4[j]);
        f[2 * j] = v.x * a.scale_log2;
        f[2 * j + 1] = v.y * a.scale_log2;
      }
    }
    const uint32_t dst = qs + (h * HD + d8 * 8) * 4;
    sts128(dst, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                           __float_as_uint(f[3])));
    sts128(dst + 16, make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]),
                                __float_as_uint(f[6]), __float_as_uint(f[7])));
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    st.m[h] = -INFINITY;
    st.lsum[h] = 0.f;
#pragma unroll
    for (int i = 0; i < SimtState<HD, NH>::DPL; ++i) st.acc[h][i] = 0.f;
  }
}

template <int HD, int T, int NH>
__device__ __forceinline__ void simt_tile(SimtState<HD, NH> &st, uint32_t stk, uint32_t qs,
                                          uint32_t pbuf, int tok0, int end) {
  constexpr int LPT = 32 / T;  // lanes per token in the score phase
  constexpr int CH = HD / LPT / 8;  // 16-byte chunks of a row per lane
  constexpr int DPL = HD / 32;
  constexpr int NHP = Nhp<NH>::v;
  const int lane = threadIdx.x & 31;
  const int r = lane % T;
  const int part = lane / T;
  const uint32_t stv = stk + Geom<HD, T>::kHalfBytes;

  // scores: lane (r, part) dots its share of K row r with every head's scaled q
  float s[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) s[h] = 0.f;
#pragma unroll 2
  for (int c = 0; c < CH; ++c) {
    const int chunk = part * CH + c;
    const uint4 raw = lds128(stk + tile_off<HD, T>(r, chunk));
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    float kf[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = half2_bits_to_float2(w4[j]);
      kf[2 * j] = v.x;
      kf[2 * j + 1] = v.y;
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const uint4 q0 = lds128(qs + (h * HD + chunk * 8) * 4);
      const uint4 q1 = lds128(qs + (h * HD + chunk * 8) * 4 + 16);
      float t = s[h];
      t = fmaf(kf[0], __uint_as_float(q0.x), t);
      t = fmaf(kf[1], __uint_as_float(q0.y), t);
      t = fmaf(kf[2], __uint_as_float(q0.z), t);
      t = fmaf(kf[3], __uint_as_float(q0.w), t);
      t = fmaf(kf[4], __uint_as_float(q1.x), t);
      t = fmaf(kf[5], __uint_as_float(q1.y), t);
      t = fmaf(kf[6], __uint_as_float(q1.z), t);
      t = fmaf(kf[7], __uint_as_float(q1.w), t);
      s[h] = t;
    }
  }
  if (LPT == 2) {
#pragma unroll
    for (int h = 0; h < NH; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], 16);
  }

  // online softmax (base 2): tile max, rescale factor, probabilities
  const bool valid = tok0 + r < end;
  float alpha[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float x = valid ? s[h] : -INFINITY;
    float mt = x;
#pragma unroll
    for (int o = T / 2; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    const float mn = fmaxf(st.m[h], mt);
    alpha[h] = fast_exp2(st.m[h] - mn);
    st.m[h] = mn;
    const float p = fast_exp2(x - mn);
    st.lsum[h] = st.lsum[h] * alpha[h] + (lane < T ? p : 0.f);
    s[h] = p;
  }
  if (lane < T) {
#pragma unroll
    for (int h = 0; h < NHP; h += 4) {
      const float p0 = s[h];
      const float p1 = (h + 1 < NH) ? s[h + 1] : 0.f;
      const float p2 = (h + 2 < NH) ? s[h + 2] : 0.f;
      const float p3 = (h + 3 < NH) ? s[h + 3] : 0.f;
      sts128(pbuf + (r * NHP + h) * 4, make_uint4(__float_as_uint(p0), __float_as_uint(p1),
                                                  __float_as_uint(p2), __float_as_uint(p3)));
    }
  }
  __syncwarp();

  // values: lane owns DPL consecutive dims; rows past `end` are never read
#pragma unroll
  for (int h = 0; h < NH; ++h)
#pragma unroll
    for (int i = 0; i < DPL; ++i) st.acc[h][i] *= alpha[h];
  const int nvalid = min(T, end - tok0);
  const int d0 = lane * DPL;
  const uint32_t vcol = static_cast<uint32_t>((d0 & 7) * 2);
#pragma unroll 4
  for (int rr = 0; rr < nvalid; ++rr) {
    const uint32_t va = stv + tile_off<HD, T>(rr, d0 >> 3) + vcol;
    float vf[DPL];
    if constexpr (DPL == 8) {
      const uint4 raw = lds128(va);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 v = half2_bits_to_float2(w4[j]);
        vf[2 * j] = v.x;
        vf[2 * j + 1] = v.y;
      }
    } else if constexpr (DPL == 4) {
      const uint2 raw = lds64(va);
      const float2 v0 = half2_bits_to_float2(raw.x);
      const float2 v1 = half2_bits_to_float2(raw.y);
      vf[0] = v0.x;
      vf[1] = v0.y;
      vf[2] = v1.x;
      vf[3] = v1.y;
    } else {
      const float2 v0 = half2_bits_to_float2(lds32(va));
      vf[0] = v0.x;
      vf[1] = v0.y;
    }
#pragma unroll
    for (int h = 0; h < NHP; h += 4) {
      const uint4 p4 = lds128(pbuf + (rr * NHP + h) * 4);
      const float pv[4] = {__uint_as_float(p4.x), __uint_as_float(p4.y), __uint_as_float(p4.z),
                           __uint_as_float(p4.w)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (h + j < NH) {
#pragma unroll
          for (int i = 0; i < DPL; ++i) st.acc[h + j][i] = fmaf(pv[j], vf[i], st.acc[h + j][i]);
        }
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA arithmetic
template <int HD>
struct MmaState {
  float m, lsum;          // row (head) lane / 4: reference maximum and sum relative to it
  float mx;               // the row's true running maximum (m <= mx <= m + kRescaleSlack)
  float o[HD / 8][2];     // O[lane / 4][8 nt + 2 (lane % 4) + {0, 1}]
  uint32_t qa[HD / 16][2];  // A fragments of q: rows 0..7, k = 16 ks + 2 (lane % 4) (+8)
};

template <int HD>
__device__ __forceinline__ void mma_begin(MmaState<HD> &st, const KernelArgs &a, int b, int h0,
                                          int nh) {
  const int lane = threadIdx.x & 31;
  const int h = lane >> 2;
  const int c = (lane & 3) * 2;
  const uint32_t *src =
      reinterpret_cast<const uint32_t *>(a.q + (static_cast<long long>(b) * a.qh + h0 + h) * HD);
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    st.qa[ks][0] = h < nh ? __ldg(src + (ks * 16 + c) / 2) : 0u;
    st.qa[ks][1] = h < nh ? __ldg(src + (ks * 16 + 8 + c) / 2) : 0u;
  }
  st.m = -INFINITY;
  st.mx = -INFINITY;
  st.lsum = 0.f;
#pragma unroll
  for (int nt = 0; nt < HD / 8; ++nt) st.o[nt][0] = st.o[nt][1] = 0.f;
}

// Zero V rows [from, T) of a stage (all chunks), so that a zero probability can never
// meet a non-finite value left in an unused row.
template <int HD, int T>
__device__ __forceinline__ void zero_v_rows(uint32_t stv, int from) {
  const int lane = threadIdx.x & 31;
  const int n = (T - from) * (HD / 8);
  for (int i = lane; i < n; i += 32) {
    const int row = from + i / (HD / 8);
    const int chunk = i % (HD / 8);
    sts128(stv + (chunk >> 3) * (T * 128) + row * 128 + (chunk & 7) * 16, make_uint4(0, 0, 0, 0));
  }
}

// Per-lane ldmatrix addresses inside a stage, fixed for the whole kernel. For K (score
// phase) the lane supplies row (mi >> 1) * 8 + rr of a 16-token chunk and 16-byte chunk
// 2 j + (mi & 1) of a 64-column block (j = ks & 3); for V (value phase) row
// (mi & 1) * 8 + rr and chunk 2 j + (mi >> 1). Rows of a chunk are 8-aligned, so the
// swizzle term is the lane's rr; the chunk's 64-column block and 16-token offset are
// compile-time constants added at the use.
template <int HD, int T>
struct MmaLane {
  uint32_t k[4], v[4];
  __device__ __forceinline__ void init() {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3;
    const int rr = lane & 7;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      k[j] = static_cast<uint32_t>(((mi >> 1) * 8 + rr) * 128 + (((2 * j + (mi & 1)) ^ rr) << 4));
      v[j] = static_cast<uint32_t>(Geom<HD, T>::kHalfBytes + ((mi & 1) * 8 + rr) * 128 +
                                   (((2 * j + (mi >> 1)) ^ rr) << 4));
    }
  }
};

// Rescale threshold of the online softmax, in base-2 units: the reference maximum of a row
// moves only when a tile's maximum exceeds it by more than this, so the fp16 probabilities
// stay <= 2^8 and most tiles skip rescaling the accumulators.
constexpr float kRescaleSlack = 8.f;

template <int HD, int T>
__device__ __forceinline__ void mma_tile(MmaState<HD> &st, const MmaLane<HD, T> &ln,
                                         uint32_t stage, int tok0, int end, float scale_log2) {
  constexpr int NCH = T / 16;
  const int lane = threadIdx.x & 31;
  uint32_t kb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) kb[j] = stage + ln.k[j];

  // S[h][t] for the tile's 16-token chunks: two n8 tiles per chunk
  float sc[NCH][2][2];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    sc[ch][0][0] = sc[ch][0][1] = sc[ch][1][0] = sc[ch][1][1] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb[ks & 3] + (ks >> 2) * (T * 128) + ch * 2048, b0, b1, b2, b3);
      mma_rows8(sc[ch][0][0], sc[ch][0][1], st.qa[ks][0], st.qa[ks][1], b0, b1);
      mma_rows8(sc[ch][1][0], sc[ch][1][1], st.qa[ks][0], st.qa[ks][1], b2, b3);
    }
  }

  // online softmax (base 2) for row lane / 4; the row's scores live in lanes
  // lane & ~3 .. lane | 3. Tokens past `end` are masked only on a partial tile.
  const bool partial = end - tok0 < T;
  float mt = -INFINITY;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float x = sc[ch][nt][j] * scale_log2;
        if (partial) {
          const int tok = tok0 + ch * 16 + nt * 8 + 2 * (lane & 3) + j;
          x = tok < end ? x : -INFINITY;
        }
        sc[ch][nt][j] = x;
        mt = fmaxf(mt, x);
      }
  mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
  st.mx = fmaxf(st.mx, mt);
  if (__any_sync(0xffffffffu, mt > st.m + kRescaleSlack)) {
    const float mn = fmaxf(st.m, mt);
    const float alpha = fast_exp2(st.m - mn);
    st.m = mn;
    st.lsum *= alpha;
#pragma unroll
    for (int nt = 0; nt < HD / 8; ++nt) {
      st.o[nt][0] *= alpha;
      st.o[nt][1] *= alpha;
    }
  }
  // The P.V products use the probabilities rounded to fp16, so the row sum adds those same
  // rounded values: numerator and denominator then weigh every token alike (a constant V
  // comes back as that constant up to fp32 summation order).
  float psum = 0.f;
  uint32_t pa[NCH][2];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float p0 = fast_exp2(sc[ch][nt][0] - st.m);
      const float p1 = fast_exp2(sc[ch][nt][1] - st.m);
      pa[ch][nt] = pack_half2(p0, p1);
      const float2 pr = half2_bits_to_float2(pa[ch][nt]);
      psum += pr.x + pr.y;
    }
  st.lsum += psum;

  if (partial) {
    zero_v_rows<HD, T>(stage + Geom<HD, T>::kHalfBytes, end - tok0);
    __syncwarp();
  }
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
#pragma unroll
    for (int dt = 0; dt < HD / 16; ++dt) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_trans(stage + ln.v[dt & 3] + (dt >> 2) * (T * 128) + ch * 2048, b0, b1, b2, b3);
      mma_rows8(st.o[2 * dt][0], st.o[2 * dt][1], pa[ch][0], pa[ch][1], b0, b1);
      mma_rows8(st.o[2 * dt + 1][0], st.o[2 * dt + 1][1], pa[ch][0], pa[ch][1], b2, b3);
    }
  }
}

// ------------------------------------------------------------------ merge (log-sum-exp)
// Fused merge flags: a contributor publishes its partial state with a release store of the
// call's epoch; the merger's acquire loads of every other contributor's flag then see the
// states. Each call has its own epoch, so flags from earlier calls never match.
__device__ __forceinline__ void flag_release(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned flag_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The merger of `unit` (contributor c0) waits until contributors c0 + 1 .. c0 + n - 1 have
// published their states. Every lane polls every flag itself (the same addresses, one
// transaction each), so each lane's later loads are ordered after its own acquire. Bounded:
// after kWaitLimitNs it raises PA_DEVERR_TIMEOUT and returns false (the unit's rows are
// then not written).
__device__ __forceinline__ bool merge_wait(const KernelArgs &a, long long unit, long long c0,
                                           int n) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    bool all = true;
    for (int k = 1; k < n && all; ++k)
      all = flag_acquire(a.ws_flag + slot_of(unit, c0 + k, a.group)) == a.epoch;
    if (__all_sync(0xffffffffu, all)) return true;
    __nanosleep(64);
    if ((it & 15u) == 15u && global_ns() - t0 > kWaitLimitNs) {
      if ((threadIdx.x & 31) == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Merge the n partial states of one unit (balanced layout: slots unit + c0 .. unit + c0 +
// n - 1) into normalised rows of `out`, all heads at once, by one warp: out_h = sum_k
// 2^(m_hk - M_h) acc_hk / sum_k 2^(m_hk - M_h) l_hk with M_h the largest m_hk (states with
// l = 0 are empty and skipped). Contributors are taken KB at a time, and for each batch the
// (m, l) pairs (one per lane: lane = head * KB + contributor) and the accumulator rows
// (lanes own head_dim / 32 dims) are loaded together, so a batch costs one memory round
// trip; the running maximum, sum and rows are rescaled when a later batch raises the
// maximum. Contributors are added in their order, so the result is deterministic.
template <int HD>
__device__ __forceinline__ void merge_balanced(const KernelArgs &a, long long unit, long long c0,
                                               int n, int b, int h0, int nh) {
  constexpr int DPL = HD / 32;
  constexpr int KB = HD >= 256 ? 1 : 2;             // contributors per batch (registers)
  constexpr int HG = HD >= 256 ? 4 : kMaxHeads;     // heads per pass (registers)
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int g0 = 0; g0 < kMaxHeads; g0 += HG) {
    if (g0 >= nh) break;
    float O[HG][DPL], L[HG], M[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      L[h] = 0.f;
      M[h] = -INFINITY;
#pragma unroll
      for (int i = 0; i < DPL; ++i) O[h][i] = 0.f;
    }
    for (int k0 = 0; k0 < n; k0 += KB) {
      // loads of the batch: lane (h, k) its (m, l); every lane its dims of every row
      const int lk = lane % KB, lh = lane / KB;
      float2 ml = make_float2(-INFINITY, 0.f);
      if (lh < HG && g0 + lh < nh && k0 + lk < n)
        ml = __ldcg(reinterpret_cast<const float2 *>(
            a.ws_ml + (slot_of(unit, c0 + k0 + lk, a.group) * kMaxHeads + g0 + lh) * 2));
      float2 v[KB][HG][DPL / 2];
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        const bool kin = k0 + k < n;
        const float *acc =
            a.ws_acc + (slot_of(unit, c0 + (kin ? k0 + k : 0), a.group) * kMaxHeads + g0) * HD +
            lane * DPL;
#pragma unroll
        for (int h = 0; h < HG; ++h)
#pragma unroll
          for (int i = 0; i < DPL / 2; ++i)
            v[k][h][i] = (kin && g0 + h < nh)
                             ? __ldcg(reinterpret_cast<const float2 *>(acc + h * HD + 2 * i))
                             : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        // the batch's (m, l) of head h, from lanes h * KB .. h * KB + KB - 1
        float mk[KB], lk2[KB];
        float bm = -INFINITY;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
          mk[k] = __shfl_sync(0xffffffffu, ml.x, (h * KB + k) & 31);
          lk2[k] = __shfl_sync(0xffffffffu, ml.y, (h * KB + k) & 31);
          if (lk2[k] > 0.f) bm = fmaxf(bm, mk[k]);
        }
        if (g0 + h >= nh || bm == -INFINITY) continue;  // warp-uniform
        if (bm > M[h]) {
          const float f = M[h] == -INFINITY ? 0.f : fast_exp2(M[h] - bm);
          L[h] *= f;
#pragma unroll
          for (int i = 0; i < DPL; ++i) O[h][i] *= f;
          M[h] = bm;
        }
#pragma unroll
        for (int k = 0; k < KB; ++k) {
          const float w = lk2[k] > 0.f ? fast_exp2(mk[k] - M[h]) : 0.f;
          L[h] += w * lk2[k];
#pragma unroll
          for (int i = 0; i < DPL / 2; ++i) {
            O[h][2 * i] += w * v[k][h][i].x;
            O[h][2 * i + 1] += w * v[k][h][i].y;
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      if (g0 + h < nh) {
        const float inv = L[h] > 0.f ? 1.f / L[h] : 0.f;
        float *dst = a.out + (static_cast<long long>(b) * a.qh + h0 + g0 + h) * HD + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; i += 2)
          *reinterpret_cast<float2 *>(dst + i) = make_float2(O[h][i] * inv, O[h][i + 1] * inv);
      }
    }
  }
}

// Unit coordinates.
struct UnitInfo {
  int b, us, h0, nh;
};

__device__ __forceinline__ UnitInfo unit_info(const KernelArgs &a, int b, int us) {
  UnitInfo u;
  u.b = b;
  u.us = us;
  const int k = us / a.sub;
  const int sg = us % a.sub;
  u.h0 = k * a.g + sg * a.nh_unit;
  u.nh = min(a.nh_unit, a.g - sg * a.nh_unit);
  return u;
}

// Writes of one finished unit segment. `whole`: this worker saw the unit's full context;
// otherwise a partial state goes to `slot` (balanced) or to split `split` (fixed split).
template <int HD, bool MMA, int NH>
struct Epilogue;

template <int HD, int NH>
struct Epilogue<HD, true, NH> {
  template <typename St>
  __device__ static void final_out(const KernelArgs &a, St &st, const UnitInfo &u) {
    const int lane = threadIdx.x & 31;
    float l = st.lsum;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int h = lane >> 2;
    if (h >= u.nh) return;
    const float inv = 1.f / l;
    float *dst = a.out + (static_cast<long long>(u.b) * a.qh + u.h0 + h) * HD + 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < HD / 8; ++nt)
      *reinterpret_cast<float2 *>(dst + nt * 8) = make_float2(st.o[nt][0] * inv, st.o[nt][1] * inv);
  }
  // Partial state to (max, sum, acc) arrays with per-head strides.
  // Partial state relative to the row's true maximum (the running sum and accumulator are
  // kept against a reference maximum up to kRescaleSlack lower; rebased here).
  template <typename St>
  __device__ static void partial_out(St &st, const UnitInfo &u, float *mx, float *sm, float *acc,
                                     long long head_stride_ml, long long head_stride_acc) {
    const int lane = threadIdx.x & 31;
    float l = st.lsum;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int h = lane >> 2;
    if (h >= u.nh) return;
    const float rebase = fast_exp2(st.m - st.mx);
    if ((lane & 3) == 0) {
      mx[h * head_stride_ml] = st.mx;
      sm[h * head_stride_ml] = l * rebase;
    }
    float *dst = acc + h * head_stride_acc + 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < HD / 8; ++nt)
      *reinterpret_cast<float2 *>(dst + nt * 8) =
          make_float2(st.o[nt][0] * rebase, st.o[nt][1] * rebase);
  }
};

template <int HD, int NH>
struct Epilogue<HD, false, NH> {
  static constexpr int DPL = HD / 32;
  template <typename St>
  __device__ static void final_out(const KernelArgs &a, St &st, const UnitInfo &u) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float l = warp_sum(st.lsum[h]);
      if (h < u.nh) {
        const float inv = 1.f / l;
        float *dst = a.out + (static_cast<long long>(u.b) * a.qh + u.h0 + h) * HD + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; i += 2)
          *reinterpret_cast<float2 *>(dst + i) = make_float2(st.acc[h][i] * inv, st.acc[h][i + 1] * inv);
      }
    }
  }
  template <typename St>
  __device__ static void partial_out(St &st, const UnitInfo &u, float *mx, float *sm, float *acc,
                                     long long head_stride_ml, long long head_stride_acc) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float l = warp_sum(st.lsum[h]);
      if (h < u.nh) {
        if (lane == 0) {
          mx[h * head_stride_ml] = st.m[h];
          sm[h * head_stride_ml] = l;
        }
        float *dst = acc + h * head_stride_acc + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; i += 2)
          *reinterpret_cast<float2 *>(dst + i) = make_float2(st.acc[h][i], st.acc[h][i + 1]);
      }
    }
  }
};

// Warm L2 with the query rows of the unit at cursor c (used when the consuming cursor
// reaches that unit a few tiles later).
template <int HD>
__device__ __forceinline__ void prefetch_q(const KernelArgs &a, const Cursor &c, int member) {
  const int lane = threadIdx.x & 31;
  const UnitInfo u = unit_info(a, c.b, c.us * a.group + member);
  const int lines = u.nh * HD * 2 / 128;
  if (lane < lines) {
    const uint16_t *p = a.q + (static_cast<long long>(c.b) * a.qh + u.h0) * HD + lane * 64;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
  }
}

// Zero the output rows of a unit (a context of length 0).
template <int HD>
__device__ __forceinline__ void zero_unit(const KernelArgs &a, const UnitInfo &u) {
  const int lane = threadIdx.x & 31;
  float *dst = a.out + (static_cast<long long>(u.b) * a.qh + u.h0) * HD;
  for (int i = lane * 2; i < u.nh * HD; i += 64) *reinterpret_cast<float2 *>(dst + i) = make_float2(0.f, 0.f);
}

template <int HD, int T, bool MMA, int NH>
__global__ void __launch_bounds__(kMaxWarpsPerCta * 32, 1)
    decode_kernel(const __grid_constant__ KernelArgs a, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  using G = Geom<HD, T>;
  using Ep = Epilogue<HD, MMA, NH>;
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bars[kMaxWarpsPerCta * kMaxStages];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // warps [group * w, group * (w + 1)) of the grid form worker w; member m serves unit
  // group_unit * group + m of the worker's group units
  const int worker = (blockIdx.x * (blockDim.x >> 5) + warp) / a.group;
  const int member = warp % a.group;
  const int S = a.stages;
  const uint32_t wbase =
      ((smem_addr(dsm) + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1)) +
      warp * a.warp_smem;
  const uint32_t qs = wbase + S * G::kStageBytes;  // SIMT: scaled q, fp32 [NH][HD]
  const uint32_t pbuf = qs + NH * HD * 4;           // SIMT: probabilities [T][NHP]
  const uint32_t bar0 = smem_addr(&bars[warp * kMaxStages]);

  {
    // warm L2 with the small inputs every warp reads first: the context lengths, the block
    // table and the queries, one 128-byte line per lane of the grid (no registers held)
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long ctx_lines = (static_cast<long long>(a.batch) * 4 + 127) / 128;
    const long long bt_lines = (static_cast<long long>(a.batch) * a.maxp * 4 + 127) / 128;
    const long long q_lines = (static_cast<long long>(a.batch) * a.qh * a.hd * 2 + 127) / 128;
    for (long long i = tid; i < ctx_lines + bt_lines + q_lines; i += nthreads) {
      const char *p = i < ctx_lines ? reinterpret_cast<const char *>(a.ctx) + i * 128
                    : i < ctx_lines + bt_lines ? reinterpret_cast<const char *>(a.bt) + (i - ctx_lines) * 128
                    : reinterpret_cast<const char *>(a.q) + (i - ctx_lines - bt_lines) * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
  }

  // ---- the worker's range
  Cursor c;
  long long total = 0, nworkers = 0;
  const int gunits = a.batch * a.upg;
  if (a.mode == MODE_BALANCED) {
    if (worker >= a.workers) return;
    const bool any = balanced_start(a, worker, T, c, total, nworkers);
    // sequences with an empty context: zero their rows (worker b mod workers); lanes test
    // 32 candidate sequences at once
    for (long long base = worker; base < a.batch; base += 32ll * a.workers) {
      const long long bl = base + static_cast<long long>(lane) * a.workers;
      unsigned empty = __ballot_sync(0xffffffffu, bl < a.batch && load_ctx(a, static_cast<int>(bl)) == 0);
      while (empty) {
        const int j = __ffs(empty) - 1;
        empty &= empty - 1;
        const int b = static_cast<int>(base + static_cast<long long>(j) * a.workers);
        for (int us = member; us < a.ups; us += a.group) zero_unit<HD>(a, unit_info(a, b, us));
      }
    }
    if (!any) return;
  } else if (a.mode == MODE_SINGLE) {
    if (worker >= gunits) return;
    c.b = worker / a.upg;
    c.us = worker % a.upg;
    c.end = load_ctx(a, c.b);
    c.tok = 0;
    c.left = tiles_of(c.end, T);
    c.ug0 = 0;
    if (c.left == 0) {
      zero_unit<HD>(a, unit_info(a, c.b, c.us * a.group + member));
      return;
    }
  } else {  // MODE_SPLIT
    if (worker >= gunits * a.num_splits) return;
    const int u = worker / a.num_splits;
    const int sp = worker % a.num_splits;
    c.b = u / a.upg;
    c.us = u % a.upg;
    const int ctx = load_ctx(a, c.b);
    const int pages = (ctx + a.ps - 1) >> a.ps_shift;
    const int pps = (pages + a.num_splits - 1) / a.num_splits;
    const int p0 = min(sp * pps, pages);
    const int p1 = min(p0 + pps, pages);
    c.tok = p0 << a.ps_shift;
    c.end = min(p1 << a.ps_shift, ctx);
    c.left = c.end > c.tok ? tiles_of(c.end - c.tok, T) : 0;
    c.ug0 = 0;
    if (c.left == 0) {
      const UnitInfo ui = unit_info(a, c.b, c.us * a.group + member);
      const long long row = (static_cast<long long>(c.b) * a.num_splits + sp) * a.qh + ui.h0;
      for (int h = 0; h < ui.nh; ++h) {
        if (lane == 0) {
          a.p_max[row + h] = -INFINITY;
          a.p_sum[row + h] = 0.f;
        }
        for (int i = lane * 2; i < HD; i += 64)
          *reinterpret_cast<float2 *>(a.p_out + (row + h) * HD + i) = make_float2(0.f, 0.f);
      }
      return;
    }
  }

  // ---- pipeline set-up
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  __syncwarp();
  const uint64_t pol = l2_evict_first_policy();

  Cursor ic = c;
  BtWindow win;
  win.b = -1;
  win.base = 0;
  win.cur = win.nxt = -1;
  int issued = 0, consumed = 0;
  for (; issued < S - 1 && ic.left > 0; ++issued) {
    issue_tile<HD, T>(a, &tk, &tv, ic, member, win, wbase + issued * G::kStageBytes, bar0 + 8 * issued, pol,
                      issued == 0 ? a.tx_extra : 0u);
    advance(a, ic, T);
  }

  typename std::conditional<MMA, MmaState<HD>, SimtState<HD, NH>>::type st;
  MmaLane<HD, T> lane_addr;
  if constexpr (MMA) lane_addr.init();
  UnitInfo cur;
  cur.b = -1;
  cur.us = -1;
  cur.h0 = cur.nh = 0;
  long long cur_ug0 = 0;
  int cur_end = 0;
  bool aborted = false;

  auto finish_unit = [&]() {
    if (a.mode == MODE_SINGLE) {
      Ep::final_out(a, st, cur);
      return;
    }
    if (a.mode == MODE_SPLIT) {
      const int sp = worker % a.num_splits;
      const long long row = (static_cast<long long>(cur.b) * a.num_splits + sp) * a.qh + cur.h0;
      Ep::partial_out(st, cur, a.p_max + row, a.p_sum + row, a.p_out + row * HD, 1, HD);
      return;
    }
    const long long unit = static_cast<long long>(cur.b) * a.ups + cur.us;
    const int nt = tiles_of(cur_end, T);
    const long long c0 = worker_of(cur_ug0, total, nworkers);
    const long long c1 = worker_of(cur_ug0 + nt - 1, total, nworkers);
    const int n = static_cast<int>(c1 - c0 + 1);
    if (n == 1) {
      Ep::final_out(a, st, cur);
      return;
    }
    const long long slot = slot_of(unit, worker, a.group);
    Ep::partial_out(st, cur, a.ws_ml + slot * kMaxHeads * 2, a.ws_ml + slot * kMaxHeads * 2 + 1,
                    a.ws_acc + slot * kMaxHeads * HD, 2, HD);
    if (!a.fused) return;
    __syncwarp();
    if (worker != c0) {
      // The unit's merger is the worker holding its first tiles: it reaches them at the end
      // of its range, after the others have written their states (at the start of their
      // ranges, or over the whole of them). The flag's release store orders this warp's
      // state writes before it; nothing else waits here.
      if (lane == 0) flag_release(a.ws_flag + slot, a.epoch);
      return;
    }
    if (merge_wait(a, unit, c0, n)) merge_balanced<HD>(a, unit, c0, n, cur.b, cur.h0, cur.nh);
  };

  // ---- main loop: refill the slot freed last iteration, wait for the next tile, compute
  while (c.left > 0) {
    if (c.b != cur.b || c.us * a.group + member != cur.us) {
      if (cur.b >= 0) finish_unit();
      cur = unit_info(a, c.b, c.us * a.group + member);
      cur_ug0 = c.ug0;
      cur_end = c.end;
      if constexpr (MMA)
        mma_begin<HD>(st, a, cur.b, cur.h0, cur.nh);
      else
        simt_begin<HD, NH>(st, a, cur.b, cur.h0, cur.nh, qs);
    }
    if (ic.left > 0) {
      const int s = issued % S;
      issue_tile<HD, T>(a, &tk, &tv, ic, member, win, wbase + s * G::kStageBytes, bar0 + 8 * s, pol,
                        issued == 0 ? a.tx_extra : 0u);
      ++issued;
      const int ib = ic.b, ius = ic.us;
      advance(a, ic, T);
      if (ic.left > 0 && (ic.b != ib || ic.us != ius)) prefetch_q<HD>(a, ic, member);
    }
    const int s = consumed % S;
    if (!mbar_wait(bar0 + 8 * s, static_cast<uint32_t>((consumed / S) & 1), a.err)) {
      aborted = true;
      break;
    }
    const uint32_t stk = wbase + s * G::kStageBytes;
    if constexpr (MMA)
      mma_tile<HD, T>(st, lane_addr, stk, c.tok, c.end, a.scale_log2);
    else
      simt_tile<HD, T, NH>(st, stk, qs, pbuf, c.tok, c.end);
    fence_proxy_async();
    __syncwarp();
    ++consumed;
    advance(a, c, T);
  }
  // the combine kernel launched as this grid's programmatic dependent may come up now: its
  // CTAs prepare during the last warps' tiles and wait for this grid's completion before
  // reading anything it wrote (triggering at the start instead kept them parked beside the
  // whole decode, measured slower)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (aborted) {
    // let the copies still in flight land before the shared memory is given up
    for (int i = consumed; i < issued; ++i)
      mbar_wait(bar0 + 8 * (i % S), static_cast<uint32_t>((i / S) & 1), a.err);
    // Fused merge: this warp's flags stay unset, so a merger waiting on them gives up
    // (bounded) and the call reports the timeout; the next call's epoch differs from every
    // flag written so far, so nothing needs resetting.
    return;
  }
  finish_unit();
}

// Separate log-sum-exp combine for the balanced schedule, for units shared by several
// workers, launched as a programmatic dependent of the decode kernel. W warps (W = 1, 2, 4
// or 8) merge one (unit, head) pair, so a CTA of 8 warps serves 8 / W pairs: one warp per
// pair for a few contributors per unit, W warps sharing tens of them. Its CTAs come up once
// every decode CTA has finished its tiles (the decode triggers the launch there). Before
// griddepcontrol.wait, which returns once the decode grid has finished and its writes are
// visible, a warp reads only inputs: it redoes the decode kernel's balanced split from the
// context lengths to find its unit's contributors, overlapping the decode's last warps.
// After it, the contributors' (m, l) and the first batch of accumulators are loaded
// together, so the merge costs about one memory round trip. Two passes as in
// merge_balanced: the maximum over contributors, then the weighted sums. Warp `sub` of a
// pair takes contributors sub, sub + W, ...; a lane holds one contributor's (m, l) of each
// chunk of 32 and the warp walks the chunk with its weights broadcast by shuffles, KB
// accumulator loads in flight at a time. The W partial sums are added in warp order.
template <int HD, int W>
__global__ void __launch_bounds__(256)
    combine_wide_kernel(const __grid_constant__ KernelArgs a, int heads, long long pairs, int T) {
  static_assert(W == 1 || W == 2 || W == 4 || W == 8, "warps per pair");
  constexpr int DPL = HD / 32;
  constexpr int P = 8 / W;  // pairs per CTA
  constexpr int KB = HD >= 256 ? 4 : 8;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = warp % W;
  const long long pair = static_cast<long long>(blockIdx.x) * P + warp / W;
  const bool valid = pair < pairs;  // warp-uniform
  const long long unit = valid ? pair / heads : 0;
  const int h = valid ? static_cast<int>(pair % heads) : 0;
  const int b = static_cast<int>(unit / a.ups);
  const int us = static_cast<int>(unit % a.ups);
  // the decode kernel's split: total tiles over all group units, workers that got tiles, and
  // the global index of this unit's first tile
  long long all = 0, before = 0;
  for (int bb = lane; bb < a.batch; bb += 32) {
    const long long t = tiles_of(load_ctx(a, bb), T);
    all += t;
    if (bb < b) before += t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    all += __shfl_xor_sync(0xffffffffu, all, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
  }
  const long long total = all * a.upg;
  const long long nworkers = total < a.workers ? total : a.workers;
  const int nt = tiles_of(load_ctx(a, b), T);
  long long c0 = 0;
  int n = 0;
  UnitInfo u = {0, 0, 0, 0};
  if (valid && nt > 0) {
    const long long ug0 = before * a.upg + static_cast<long long>(us / a.group) * nt;
    c0 = worker_of(ug0, total, nworkers);
    n = static_cast<int>(worker_of(ug0 + nt - 1, total, nworkers) - c0 + 1);
    u = unit_info(a, b, us);
    // a unit with one worker was finalised by it; heads past the unit's own do not exist
    if (n <= 1 || h >= u.nh) n = 0;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (W == 1) {
    if (n == 0) return;  // no barrier below for a warp per pair
  }
  // contributors of this warp: sub, sub + W, ... < n
  const int mine = n > sub ? (n - sub + W - 1) / W : 0;
  auto ml_of = [&](int j) {
    const long long slot = slot_of(unit, c0 + sub + W * j, a.group);
    return __ldcg(reinterpret_cast<const float2 *>(a.ws_ml + (slot * kMaxHeads + h) * 2));
  };
  const float *acc_base = a.ws_acc + static_cast<long long>(h) * HD + lane * DPL;
  float2 v[KB][DPL / 2];
  auto load_batch = [&](int j0) {  // accumulators of contributors j0 .. j0 + KB - 1
#pragma unroll
    for (int tt = 0; tt < KB; ++tt) {
      if (j0 + tt < mine) {
        const float *src =
            acc_base + slot_of(unit, c0 + sub + W * (j0 + tt), a.group) * kMaxHeads * HD;
#pragma unroll
        for (int i = 0; i < DPL / 2; ++i)
          v[tt][i] = __ldcg(reinterpret_cast<const float2 *>(src + 2 * i));
      } else {
#pragma unroll
        for (int i = 0; i < DPL / 2; ++i) v[tt][i] = make_float2(0.f, 0.f);
      }
    }
  };
  float2 first = make_float2(-INFINITY, 0.f);  // (m, l) of contributor `lane`
  if (lane < mine) first = ml_of(lane);
  load_batch(0);
  float mx = first.y > 0.f ? first.x : -INFINITY;
  for (int j = lane + 32; j < mine; j += 32) {
    const float2 ml = ml_of(j);
    if (ml.y > 0.f) mx = fmaxf(mx, ml.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __shared__ float s_max[8];
  __shared__ float s_l[8];
  __shared__ __align__(16) float s_acc[W > 1 ? 8 : 1][HD];
  float M = mx;
  if constexpr (W > 1) {
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    M = s_max[warp - sub];
#pragma unroll
    for (int w = 1; w < W; ++w) M = fmaxf(M, s_max[warp - sub + w]);
  }
  float O[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) O[i] = 0.f;
  float L = 0.f;
  for (int j0 = 0; j0 < mine; j0 += 32) {
    float2 ml = first;
    if (j0 > 0) ml = j0 + lane < mine ? ml_of(j0 + lane) : make_float2(-INFINITY, 0.f);
    const float wk = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
    L += wk * ml.y;
    const int cnt = min(32, mine - j0);
    for (int t0 = 0; t0 < cnt; t0 += KB) {
      if (j0 + t0 > 0) load_batch(j0 + t0);
#pragma unroll
      for (int tt = 0; tt < KB; ++tt) {
        // contributors past the end were loaded as zeros
        const float w = __shfl_sync(0xffffffffu, wk, (t0 + tt) & 31);
#pragma unroll
        for (int i = 0; i < DPL / 2; ++i) {
          O[2 * i] += w * v[tt][i].x;
          O[2 * i + 1] += w * v[tt][i].y;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if constexpr (W > 1) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) s_acc[warp][lane * DPL + i] = O[i];
    if (lane == 0) s_l[warp] = L;
    __syncthreads();
    if (sub != 0) return;
    L = s_l[warp];
#pragma unroll
    for (int i = 0; i < DPL; ++i) O[i] = s_acc[warp][lane * DPL + i];
#pragma unroll
    for (int w = 1; w < W; ++w) {
      L += s_l[warp + w];
#pragma unroll
      for (int i = 0; i < DPL; ++i) O[i] += s_acc[warp + w][lane * DPL + i];
    }
  }
  if (n == 0) return;
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float *dst = a.out + (static_cast<long long>(u.b) * a.qh + u.h0 + h) * HD + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; i += 2)
    *reinterpret_cast<float2 *>(dst + i) = make_float2(O[i] * inv, O[i + 1] * inv);
}

// Log-sum-exp combine of the fixed-split arrays (section "V4 (Context-axis parallelism)"'s
// merge: empty splits are skipped, the rest rescaled to a common maximum and normalised).
// One CTA of kCombineSplitWarps warps per (sequence, query head). Every warp first reduces
// the splits' (max, sum) pairs, 32 splits per round, to the common maximum M and the total
// L; warp w then adds the accumulator rows of splits w, w + W, w + 2W, ..., each weighted by
// exp2(m_s - M), with the weights of 32 splits computed at once and the row loads of
// consecutive splits independent of each other; warp 0 adds the W partial rows in warp order
// and divides by L. The summation order is fixed, so results are deterministic.
constexpr int kCombineSplitWarps = 8;

template <int HD>
__global__ void __launch_bounds__(kCombineSplitWarps * 32)
    combine_split_kernel(const __grid_constant__ KernelArgs a) {
  constexpr int DPL = HD / 32;
  constexpr int W = kCombineSplitWarps;
  __shared__ __align__(16) float part[W][HD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long b = blockIdx.x / a.qh;
  const long long h = blockIdx.x % a.qh;
  const int n = a.num_splits;
  auto idx_of = [&](int s) { return (b * n + s) * a.qh + h; };
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) {
    const long long i = idx_of(s);
    if (__ldg(a.p_sum + i) != 0.f) M = fmaxf(M, __ldg(a.p_max + i));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  for (int s = lane; s < n; s += 32) {
    const long long i = idx_of(s);
    const float l = __ldg(a.p_sum + i);
    if (l != 0.f) L += fast_exp2(__ldg(a.p_max + i) - M) * l;
  }
  L = warp_sum(L);
  float O[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) O[i] = 0.f;
  for (int base = warp; base < n; base += 32 * W) {
    // lane j weighs split base + j * W (0 for an empty split or one past the end)
    const int sj = base + lane * W;
    float wj = 0.f;
    if (sj < n) {
      const long long i = idx_of(sj);
      if (__ldg(a.p_sum + i) != 0.f) wj = fast_exp2(__ldg(a.p_max + i) - M);
    }
    const int cnt = min(32, (n - base + W - 1) / W);
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const float wt = __shfl_sync(0xffffffffu, wj, j);
      if (wt == 0.f) continue;
      const float *src = a.p_out + idx_of(base + j * W) * HD + lane * DPL;
#pragma unroll
      for (int i = 0; i < DPL; i += 2) {
        const float2 v = __ldg(reinterpret_cast<const float2 *>(src + i));
        O[i] = fmaf(wt, v.x, O[i]);
        O[i + 1] = fmaf(wt, v.y, O[i + 1]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < DPL; ++i) part[warp][lane * DPL + i] = O[i];
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int w = 1; w < W; ++w)
#pragma unroll
    for (int i = 0; i < DPL; ++i) O[i] += part[w][lane * DPL + i];
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float *dst = a.out + static_cast<long long>(blockIdx.x) * HD + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; i += 2)
    *reinterpret_cast<float2 *>(dst + i) = make_float2(O[i] * inv, O[i + 1] * inv);
}

}  // namespace pa
