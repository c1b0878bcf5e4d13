// prefill2_kernel.cuh -- the multi-token (prefill) kernel for head_dim 64 and 128: two query
// tiles per work item that share every K/V tile and take turns on the tensor cores, and
// CTAs that stay resident and take over work items of CTAs that have not started.
//
// Same computation as prefill_kernel.cuh ("[TIL] Optimizing paged attention", section
// "Flash Attention", over the paged cache of section "Paged Attention", causal per row),
// organised so that the K/V bytes moved per MMA flop are halved and the softmax of one
// query tile overlaps the MMAs of the other:
//   tiles A and B: 2 x 128 MMA rows (consecutive query tiles of one sequence and K/V head)
//   TMEM (512 columns): S_A [0,128)  S_B [128,256)  O_A [256,256+HD)  O_B [384,384+HD)
//   P_X (fp16) overwrites the first 64 columns of S_X once the softmax has read S_X; the
//   P.V MMA reads it from TMEM as its A operand, so P never touches shared memory.
//   shared memory: Q_A, Q_B, and one ring of K/V slots filled in order K0 V0 K1 V1 ...
// MMA order per K/V tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while the tensor cores run
// tile B's MMAs, tile A's softmax runs, and the other way round. Because the tensor core
// executes one thread's MMAs in issue order, the completion of S_X(j+1) also means PV_X(j)
// is done, so the softmax may rescale O_X in TMEM as soon as it sees S_X(j+1).
//
// Work items. The grid has one CTA per item (K/V head, sequence, pair of query tiles), the
// longest pairs first. A CTA keeps its tensor memory, barriers and pipelines and, through
// cluster launch control, cancels CTAs of the grid that have not started and runs their
// items itself, so one item's epilogue and the next item's Q/K loads and first score MMAs
// overlap instead of paying a CTA start, a TMEM allocation and a cold pipeline per item. The
// hardware hands out the items in launch order to whichever CTA asks first, and each item's
// arithmetic does not depend on which CTA runs it, so results stay deterministic.
// Warps: 3 schedules (one request per item, answers published in a two-entry ring); 0 loads
// the K tiles, 2 loads Q and the V tiles, 1 allocates TMEM and issues the MMAs; 4..7 are tile
// A's softmax (TMEM lanes 0..127), 8..11 tile B's. Counters of K/V tiles, Q loads and barrier
// phases run on across items.
#pragma once

#include "prefill_kernel.cuh"

namespace pa {

template <int HD>
struct Prefill2Cfg {
  static constexpr int kRows = 128;
  static constexpr int KB = HD / 64;
  static constexpr int TN = 128;                 // K/V tokens per tile
  static constexpr int kQBytes = KB * kRows * 128;  // one query tile
  static constexpr int kSlotBytes = TN * HD * 2;    // one K or V tile
  static constexpr int kSlots = HD == 64 ? 8 : 5;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kQBytes;
  static constexpr int kSmem = kRingOff + kSlots * kSlotBytes;  // + 1 KB alignment at launch
  static constexpr uint32_t kTmemCols = 512;
  // S_X at column 128 * X, O_X at 256 + 128 * X
  static constexpr uint32_t kIdescS = idesc_f16(kRows, TN, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_f16(kRows, HD, 0, 1);
};

constexpr int kPrefill2Threads = 384;
// Register split between warpgroup 0 (producers, MMA, scheduler) and the two softmax
// warpgroups: 128 * 72 + 256 * 216 <= 384 * 168, the registers the CTA is launched with.
constexpr uint32_t kPrefill2SmallRegs = 72;
constexpr uint32_t kPrefill2BigRegs = 216;
static_assert(128 * kPrefill2SmallRegs + 256 * kPrefill2BigRegs <= 384 * 168,
              "register split exceeds the launch allocation");
// warps that read each published work item: 0, 1, 2 and the eight softmax warps
constexpr int kItemReaders = 11;

enum : int {
  kB2QFull = 0,       // Q of an item landed
  kB2QEmpty = 1,      // the item's last score MMA completed: Q may be replaced
  kB2SFull = 2,       // +tile
  kB2PFull = 4,       // +tile (128 arrivals)
  kB2ODone = 6,       // +tile
  kB2Done = 8,
  kB2ItemFull = 9,    // +entry: a work item is published
  kB2ItemEmpty = 11,  // +entry: every reader has taken it (kItemReaders arrivals)
  kB2ProdStart = 13,  // the K producer started an item: time to ask for the next one
  kB2Clc = 14,        // the answer to a cancellation request landed (16 bytes)
  kB2Full = 15,       // +slot
  kB2Empty = 23,      // +slot
  kNumBars2 = 31
};

// Geometry of one work item (K/V head kv, sequence b, pair of query tiles), computed once by
// the scheduler and published to every role. `live` is 0 when the pair holds no new token
// or the sequence's offsets or length are out of range (those are flagged here); `stop` marks
// the end of the CTA's work.
struct Item2 {
  int kv, b, q0, n, ctx;
  int tok0_a, tok0_b, max_pos_a, max_pos_b, nt_a, nt_b, nt_max, kv_len;
  int live, stop;
};

template <int TN>
__device__ __forceinline__ Item2 item2_of(const PrefillArgs &a, int kv, int b, int pair) {
  Item2 it;
  it.kv = kv;
  it.b = b;
  it.live = 0;
  it.stop = 0;
  it.nt_a = it.nt_b = it.nt_max = 0;
  const int q0 = __ldg(a.qs + b), q1 = __ldg(a.qs + b + 1), ctx = __ldg(a.ctx + b);
  const int n = q1 - q0;
  it.q0 = q0;
  it.n = n;
  it.ctx = ctx;
  if (ctx < 0 || static_cast<long long>(ctx) > static_cast<long long>(a.maxp) << a.ps_shift) {
    atomicOr(a.err, PA_DEVERR_CONTEXT);
    return it;
  }
  if (q0 < 0 || n < 0 || static_cast<long long>(q1) > a.total || n > ctx) {
    atomicOr(a.err, PA_DEVERR_QUERY_START);
    return it;
  }
  // query tile X covers new tokens [tok0_X, tok0_X + qt); tile A has rows whenever B has
  it.tok0_a = 2 * pair * a.qt;
  it.tok0_b = it.tok0_a + a.qt;
  if (it.tok0_a >= n) return it;
  it.max_pos_a = ctx - n + min(it.tok0_a + a.qt, n) - 1;
  it.max_pos_b = it.tok0_b < n ? ctx - n + min(it.tok0_b + a.qt, n) - 1 : -1;
  it.nt_a = (it.max_pos_a + TN) / TN;
  it.nt_b = (it.max_pos_b + TN) / TN;  // 0 when tile B is empty
  it.nt_max = max(it.nt_a, it.nt_b);
  it.kv_len = max(it.max_pos_a, it.max_pos_b) + 1;
  it.live = 1;
  return it;
}

// P = exp2(s * sl2 + nm) over a row of TN scores, written as fp16 pairs over the first TN / 2
// TMEM columns at ts, with the row's partial sums in rp. With kMasked keys past lim give
// exactly 0; without, packed fp32 pairs do two exponent arguments per FFMA2 and two sum terms
// per FADD2.
template <int TN, bool kMasked>
__device__ __forceinline__ void exps_row(const float (&v)[TN], float sl2, float nm, int lim,
                                         uint32_t ts, float (&rp)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) rp[e] = 0.f;
#pragma unroll
  for (int h2 = 0; h2 < TN / 64; ++h2) {
    float pk[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = h2 * 64 + 2 * e;
      float p0, p1;
      if (kMasked) {
        p0 = c <= lim ? prefill_exp2(fmaf(v[c], sl2, nm)) : 0.f;
        p1 = c + 1 <= lim ? prefill_exp2(fmaf(v[c + 1], sl2, nm)) : 0.f;
        rp[c & 7] += p0;
        rp[(c + 1) & 7] += p1;
      } else {
        const float2 xx =
            ffma2(make_float2(v[c], v[c + 1]), make_float2(sl2, sl2), make_float2(nm, nm));
        p0 = prefill_exp2(xx.x);
        p1 = prefill_exp2(xx.y);
        const float2 acc = fadd2(make_float2(rp[c & 7], rp[(c + 1) & 7]), make_float2(p0, p1));
        rp[c & 7] = acc.x;
        rp[(c + 1) & 7] = acc.y;
      }
      pk[e] = __uint_as_float(pack_half2(p0, p1));
    }
    tmem_st32(ts + h2 * 32, pk);
  }
}

template <int HD>
__global__ void __launch_bounds__(kPrefill2Threads, 1)
    prefill2_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
  using C = Prefill2Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars2];
  __shared__ __align__(16) uint4 clc_answer;
  __shared__ Item2 items[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_word;
  __shared__ int drain_last[2];
  volatile int *abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q_rows = a.qt * a.g;

  const uint32_t sbase = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t *sgen = smem_raw + (sbase - smem_addr(smem_raw));
  auto q_tile = [&](int x) { return sbase + C::kQOff + x * C::kQBytes; };
  auto slot_addr = [&](int s) { return sbase + C::kRingOff + s * C::kSlotBytes; };
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars2; ++i) {
      uint32_t count = 1;
      if (i == kB2PFull || i == kB2PFull + 1) count = 128;
      if (i == kB2ItemEmpty || i == kB2ItemEmpty + 1) count = kItemReaders;
      mbar_init(bar(i), count);
    }
    abort_word = 0;
    fence_barrier_init();
  }
  // MMA rows past q_rows (g not dividing 128) are never written by the Q loads: zero once
  if (q_rows < C::kRows) {
    const int per_block = (C::kRows - q_rows) * 8;
    for (int i = threadIdx.x; i < 2 * C::KB * per_block; i += kPrefill2Threads) {
      const int x = i / (C::KB * per_block), r = i % (C::KB * per_block);
      const int kb = r / per_block, c = r % per_block;
      *reinterpret_cast<uint4 *>(sgen + C::kQOff + x * C::kQBytes + kb * (C::kRows * 128) +
                                 q_rows * 128 + c * 16) = make_uint4(0, 0, 0, 0);
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
  auto take_item = [&](int k, Item2 &it) {
    if (!pipe_wait(bar(kB2ItemFull + (k & 1)), (k >> 1) & 1, abort_flag, a.err)) return false;
    it = items[k & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kB2ItemEmpty + (k & 1)));
    return true;
  };

  // registers: the softmax warpgroups hold a 128-column score row per thread; each role
  // changes its own allocation inside its branch so the compiler sees one limit per region
  if (warp < 4) regs_decrease<kPrefill2SmallRegs>();
  if (warp == 3) {
    // ================= scheduler =================
    int kv = blockIdx.x, b = blockIdx.y, z = blockIdx.z;
    bool stop = false;
    const uint32_t answer = smem_addr(&clc_answer);
    for (int k = 0;; ++k) {
      // publish item k once every reader has taken item k - 2 from the same entry
      if (k >= 2 && !pipe_wait(bar(kB2ItemEmpty + (k & 1)), ((k >> 1) - 1) & 1, abort_flag, a.err))
        break;
      if (lane == 0) {
        Item2 it;
        if (stop) {
          it.stop = 1;
          it.live = 0;
        } else {
          it = item2_of<C::TN>(a, kv, b, a.n_qtiles - 1 - z);  // grid.z counts pairs
        }
        items[k & 1] = it;
        mbar_arrive(bar(kB2ItemFull + (k & 1)));
      }
      __syncwarp();
      if (stop) break;
      // ask for item k + 1 when the K producer starts item k
      if (!pipe_wait(bar(kB2ProdStart), k & 1, abort_flag, a.err)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kB2Clc), 16);
        clc_try_cancel(answer, bar(kB2Clc));
      }
      __syncwarp();
      if (!pipe_wait(bar(kB2Clc), k & 1, abort_flag, a.err)) {
        if (lane == 0) drain_wait(bar(kB2Clc), k & 1, a.err);  // the answer's write lands first
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
  } else if (warp == 0 || warp == 2) {
    // ============ producers: warp 2 Q and V(j) (item 2j + 1), warp 0 K(j) (item 2j) ============
    const bool is_v = warp == 2;
    if (lane == 0) {
      prefetch_tensormap(is_v ? &tv : &tk);
      if (is_v) prefetch_tensormap(&tq);
    }
    const CUtensorMap *map = is_v ? &tv : &tk;
    // L2 policies: every pair of query tiles of a (sequence, K/V head) reads its K/V tiles,
    // so they stay (evict last); each Q tile is read once (evict first)
    const uint64_t pol = l2_evict_last_policy();
    const uint64_t pol_q = l2_evict_first_policy();
    const int rows_per_box = min(a.ps, C::TN);
    const int boxes = C::TN / rows_per_box;
    const uint32_t box_bytes = rows_per_box * 128;
    int last_item = -1;  // ring items are numbered across work items: K(j) of the tile with
                         // global index t is 2t, V(j) 2t + 1
    int gt = 0;          // global index of the current item's first tile
    int q_loads = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item2 it;
      ok = take_item(k, it);
      if (!ok || it.stop) break;
      if (!is_v && lane == 0) mbar_arrive(bar(kB2ProdStart));
      if (!it.live) continue;
      if (is_v) {
        // both query tiles, once the previous item's last score MMA has read Q
        if (q_loads > 0) ok = pipe_wait(bar(kB2QEmpty), (q_loads - 1) & 1, abort_flag, a.err);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(kB2QFull), 2 * C::KB * q_rows * 128);
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_3d(q_tile(x) + kb * (C::kRows * 128), &tq, bar(kB2QFull), kb * 64,
                          it.kv * a.g, it.q0 + (x ? it.tok0_b : it.tok0_a), pol_q);
        }
        ++q_loads;
      }
      const int32_t *bt_row = a.bt + static_cast<size_t>(it.b) * a.maxp;
      auto page_of = [&](int j) {
        const int tok = j * C::TN + lane * rows_per_box;
        return (j < it.nt_max && lane < boxes && tok < it.kv_len)
                   ? __ldg(bt_row + (tok >> a.ps_shift))
                   : -1;
      };
      int page_next = page_of(0);
      for (int j = 0; j < it.nt_max && ok; ++j) {
        const int item = 2 * (gt + j) + (is_v ? 1 : 0);
        const int s = item % C::kSlots;
        const int tok = j * C::TN + lane * rows_per_box;
        int page = page_next;
        page_next = page_of(j + 1);
        if (lane < boxes && tok < it.kv_len && (page < 0 || page >= a.num_pages)) {
          if (!is_v) atomicOr(a.err, PA_DEVERR_PAGE_ID);
          page = -1;
        }
        const uint32_t issue = __ballot_sync(0xffffffffu, page >= 0);
        const int slot_in_page = tok & (a.ps - 1);
        int y, z;
        if (a.layout == PA_LAYOUT_HEAD_MAJOR) {
          y = slot_in_page;
          z = page * a.kvh + it.kv;
        } else {
          y = it.kv;
          z = (page << a.ps_shift) + slot_in_page;
        }
        if (item >= C::kSlots)
          ok = pipe_wait(bar(kB2Empty + s), ((item / C::kSlots) - 1) & 1, abort_flag, a.err);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(bar(kB2Full + s), __popc(issue) * box_bytes * C::KB);
        __syncwarp();
        if (page >= 0) {
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(slot_addr(s) + kb * (C::TN * 128) + lane * box_bytes, map,
                        bar(kB2Full + s), kb * 64, y, z, pol);
        }
        last_item = item;
      }
      gt += it.nt_max;
    }
    // drain: the last Q load and, in every slot, the newest item either warp loaded into it
    // have landed (older items of a slot were consumed before the slot was refilled)
    if (lane == 0) drain_last[is_v ? 1 : 0] = last_item;
    asm volatile("bar.sync 1, 64;" ::: "memory");
    if (is_v && lane == 0 && q_loads > 0) drain_wait(bar(kB2QFull), (q_loads - 1) & 1, a.err);
    if (!is_v && lane == 0) {
      const int last_k = drain_last[0], last_v = drain_last[1];
      const int top = max(last_k, last_v);
      for (int s = 0; s < C::kSlots; ++s) {
        int it = top - ((top - s) % C::kSlots + C::kSlots) % C::kSlots;  // newest item in slot s
        for (; it >= 0; it -= C::kSlots)
          if (((it & 1) == 0 && it <= last_k) || ((it & 1) == 1 && it <= last_v)) break;
        if (it >= 0) drain_wait(bar(kB2Full + s), (it / C::kSlots) & 1, a.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    bool ok = true;
    // PA_TEST_EXPIRE_WAITS: the first wait is on the barrier that completes only at the end
    if (a.expire) ok = pipe_wait(bar(kB2Done), 0, abort_flag, a.err);
    int waited = -1;  // ring items are waited for in order; the highest one waited so far
    auto wait_item = [&](int item) {
      if (item <= waited) return true;
      const bool r = pipe_wait(bar(kB2Full + item % C::kSlots), (item / C::kSlots) & 1, abort_flag,
                               a.err);
      if (r) waited = item;
      tc_fence_after();
      return r;
    };
    int gt = 0;
    uint32_t phase = 0;  // parities of the next waits: bit 0 QFull, bit 1 + x PFull[x]
    for (int k = 0; ok; ++k) {
      Item2 it;
      ok = take_item(k, it);
      if (!ok || it.stop) break;
      if (!it.live) continue;
      auto nt_of = [&](int x) { return x ? it.nt_b : it.nt_a; };
      const int last_s_x = it.nt_b == it.nt_max ? 1 : 0;  // tile of the item's last score MMA
      // MMAs and commits are issued warp-collectively (one elected lane), with operands every
      // lane computes identically
      // Descriptors of a K step are the tile's base descriptor plus the step's byte offset / 16
      // (shared-memory addresses stay below 2^18, so the 14-bit address field never carries);
      // the empty asm keeps the compiler from hoisting all steps' descriptors into registers.
      auto issue_s = [&](int x, int j) {  // S_X(j) = Q_X K(j)^T
        uint64_t qd = smem_desc_sw128(q_tile(x), 16, 1024);
        uint64_t kd = smem_desc_sw128(slot_addr((2 * (gt + j)) % C::kSlots), 16, 1024);
        asm volatile("" : "+l"(qd), "+l"(kd));
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint64_t ad = qd + (((ks >> 2) * (C::kRows * 128) + (ks & 3) * 32) >> 4);
          const uint64_t bd = kd + (((ks >> 2) * (C::TN * 128) + (ks & 3) * 32) >> 4);
          mma_f16_ss_warp(tmem + 128u * x, ad, bd, C::kIdescS, ks > 0);
        }
        mma_commit_warp(bar(kB2SFull + x));
        if (j == it.nt_max - 1 && x == last_s_x) mma_commit_warp(bar(kB2QEmpty));
      };
      auto issue_pv = [&](int x, int j) {  // O_X += P_X(j) V(j), P_X from TMEM
        uint64_t vd = smem_desc_sw128(slot_addr((2 * (gt + j) + 1) % C::kSlots), C::TN * 128, 1024);
        asm volatile("" : "+l"(vd));
#pragma unroll
        for (int ks = 0; ks < C::TN / 16; ++ks) {
          const uint64_t bd = vd + ((ks * 2048) >> 4);
          mma_f16_ts_warp(tmem + 256u + 128u * x, tmem + 128u * x + ks * 8, bd, C::kIdescPV,
                          (j > 0 || ks > 0) ? 1u : 0u);
        }
        if (j == nt_of(x) - 1) mma_commit_warp(bar(kB2ODone + x));
      };
      auto release = [&](int item) { mma_commit_warp(bar(kB2Empty + item % C::kSlots)); };
      auto clear_v_tail = [&](int j) {
        // V rows past the last needed token hold unread cache slots (possibly never
        // written): P is zero there, but 0 * NaN is not, so clear them before the first P.V
        // of that tile.
        const int rows_last = it.kv_len - j * C::TN;
        if (j != it.nt_max - 1 || rows_last >= C::TN) return;
        const int per_block = (C::TN - rows_last) * 8;
        uint8_t *vg = sgen + C::kRingOff + ((2 * (gt + j) + 1) % C::kSlots) * C::kSlotBytes;
        for (int c = lane; c < C::KB * per_block; c += 32) {
          const int kb = c / per_block, r = c % per_block;
          *reinterpret_cast<uint4 *>(vg + kb * (C::TN * 128) + rows_last * 128 + r * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
      };
      ok = pipe_wait(bar(kB2QFull), phase & 1u, abort_flag, a.err);
      phase ^= 1u;
      tc_fence_after();
      if (ok) ok = wait_item(2 * gt);
      if (ok) {
        // S_X(0) overwrites the columns from which the previous item's last P.V read P_X:
        // that MMA was issued earlier by this thread and so runs first
        issue_s(0, 0);
        if (it.nt_b > 0) issue_s(1, 0);
        release(2 * gt);
      }
      for (int j = 0; j < it.nt_max && ok; ++j) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok || j >= nt_of(x)) continue;
          // P_X(j) is released only after V(j) and K(j + 1) have landed (see the softmax)
          ok = pipe_wait(bar(kB2PFull + x), (phase >> (1 + x)) & 1u, abort_flag, a.err);
          if (!ok) break;
          phase ^= 2u << x;
          tc_fence_after();
          if (x == 0 || j >= it.nt_a) clear_v_tail(j);
          issue_pv(x, j);
          const bool last_v_user = (x == 1) || (j >= it.nt_b);
          if (last_v_user) release(2 * (gt + j) + 1);
          if (j + 1 < nt_of(x)) {
            issue_s(x, j + 1);
            const bool last_k_user = (x == 1) || (j + 1 >= it.nt_b);
            if (last_k_user) release(2 * (gt + j + 1));
          }
        }
      }
      gt += it.nt_max;
    }
    mma_commit_warp(bar(kB2Done));
    if (lane == 0) drain_wait(bar(kB2Done), 0, a.err);
    __syncwarp();
  } else if (warp >= 4) {
    regs_increase<kPrefill2BigRegs>();
    // ================= softmax: tile x = (warp - 4) / 4, one query row per thread =================
    const int x = (warp - 4) >> 2;
    const int rg = warp & 3;
    const int row = rg * 32 + lane;
    const int t = row / a.g, h = row - t * a.g;
    const uint32_t lane_off = static_cast<uint32_t>(rg * 32) << 16;
    const uint32_t ts = tmem + lane_off + 128u * x;
    const uint32_t to = tmem + lane_off + 256u + 128u * x;
    const float sl2 = a.scale_log2;
    int gt = 0;
    uint32_t phase = 0;  // parities of the next waits: bit 0 SFull[x], bit 1 ODone[x]
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int my_nt, pos, gt0, out_row0, out_head0;
      bool valid;
      {
        Item2 it;
        ok = take_item(k, it);
        if (!ok || it.stop) break;
        if (!it.live) continue;
        const int my_tok0 = x ? it.tok0_b : it.tok0_a;
        my_nt = x ? it.nt_b : it.nt_a;
        valid = row < q_rows && my_tok0 + t < it.n;
        pos = min(it.ctx - it.n + my_tok0 + t, x ? it.max_pos_b : it.max_pos_a);
        out_row0 = it.q0 + my_tok0;  // output row of the tile's first token
        out_head0 = it.kv * a.g;
        gt0 = gt;
        gt += it.nt_max;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < my_nt; ++j) {
        ok = pipe_wait(bar(kB2SFull + x), phase & 1u, abort_flag, a.err);
        if (!ok) break;
        phase ^= 1u;
        tc_fence_after();
        // The MMAs this P releases read V(j) and, for S(j + 1), K(j + 1): one warp of the
        // group confirms they have landed before the group releases P, so the MMA warp waits
        // on P alone. (Neither slot can be recycled first: both are released only after MMAs
        // that need this P.) The probes go out before the score load and are read after it.
        const int iv = 2 * (gt0 + j) + 1, ik = 2 * (gt0 + j) + 2;
        bool kv_ready = true;
        if (rg == 0) {
          const bool rv = mbar_try_wait(bar(kB2Full + iv % C::kSlots), (iv / C::kSlots) & 1);
          const bool rk = j + 1 < my_nt
                              ? mbar_try_wait(bar(kB2Full + ik % C::kSlots), (ik / C::kSlots) & 1)
                              : true;
          kv_ready = rv && rk;
        }
        float v[C::TN];
        tmem_ld128(ts, v);
        if (rg == 0 && !__all_sync(0xffffffffu, kv_ready)) {
          ok = pipe_wait(bar(kB2Full + iv % C::kSlots), (iv / C::kSlots) & 1, abort_flag, a.err);
          if (ok && j + 1 < my_nt)
            ok = pipe_wait(bar(kB2Full + ik % C::kSlots), (ik / C::kSlots) & 1, abort_flag, a.err);
          if (!ok) break;
        }
        const int lim = pos - j * C::TN;
        // warp-uniform: the exponent passes hold tcgen05.st, which the whole warp executes
        const bool full = __all_sync(0xffffffffu, lim >= C::TN - 1);
        float rp[8];
        // After a row's first tile its running maximum m seldom grows by more than the slack,
        // so a tile first takes its exponents with m as it stands and no maximum pass: the
        // terms are non-negative (masked keys give 0), so the tile's row sum bounds each of
        // them, and a sum of at most 2^slack shows that no score passed m + slack. Only a warp
        // in which some row's sum is larger (or not a number) takes the tile again in the
        // plain order: maximum, rescale, exponents.
        bool redo = true;
        if (j > 0) {
          if (full)
            exps_row<C::TN, false>(v, sl2, -m, lim, ts, rp);
          else
            exps_row<C::TN, true>(v, sl2, -m, lim, ts, rp);
          const float tsum =
              ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
          redo = __any_sync(0xffffffffu, !(tsum <= kPrefillSlackBound));
          if (redo) tmem_wait_st();  // the plain pass below rewrites the same columns
        }
        if (redo) {
          // keys past this row's position are masked out (on tiles that reach the diagonal);
          // the row maximum of the scaled scores is the extreme raw score times the scale (the
          // maximum for a non-negative scale, else the minimum), which saves a multiply per score
          float mp[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mp[e] = -INFINITY;
          float ext;
          if (sl2 >= 0.f) {
            if (full) {
#pragma unroll
              for (int c = 0; c < C::TN; ++c) mp[c & 7] = fmaxf(mp[c & 7], v[c]);
            } else {
#pragma unroll
              for (int c = 0; c < C::TN; ++c) mp[c & 7] = fmaxf(mp[c & 7], c <= lim ? v[c] : -INFINITY);
            }
            ext = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                        fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) mp[e] = INFINITY;
#pragma unroll
            for (int c = 0; c < C::TN; ++c) mp[c & 7] = fminf(mp[c & 7], (full || c <= lim) ? v[c] : INFINITY);
            ext = fminf(fminf(fminf(mp[0], mp[1]), fminf(mp[2], mp[3])),
                        fminf(fminf(mp[4], mp[5]), fminf(mp[6], mp[7])));
          }
          const float mx = ext * sl2;
          const bool grow = mx > m + kPrefillRescaleSlack;
          if (__any_sync(0xffffffffu, grow)) {
            const float mnew = grow ? mx : m;
            const float f = mnew == -INFINITY ? 1.f : prefill_exp2(m - mnew);
            l *= f;
            if (j > 0) {
              // S_X(j) completed, so PV_X(j - 1) has too: O_X is stable until P_X(j) is released
#pragma unroll
              for (int c = 0; c < HD / 32; ++c) {
                float o[32];
                tmem_ld32(to + c * 32, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= f;
                tmem_st32(to + c * 32, o);
              }
            }
            m = mnew;
          }
          // P = exp2(s * scale * log2e - m) as fp16 pairs over the first 64 columns of S (the
          // scale is folded into one FFMA per score; masked keys give exactly 0)
          const float nm = -m;
          if (full)
            exps_row<C::TN, false>(v, sl2, nm, lim, ts, rp);
          else
            exps_row<C::TN, true>(v, sl2, nm, lim, ts, rp);
        }
        l += ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kB2PFull + x));
      }
      if (ok && my_nt > 0) {
        ok = pipe_wait(bar(kB2ODone + x), (phase >> 1) & 1u, abort_flag, a.err);
        phase ^= 2u;
      }
      if (ok && my_nt > 0) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        // Each thread writes its row straight from TMEM, 32 columns at a time: 32-byte stores
        // fill whole sectors, so L2 never reads a partly written sector from DRAM first, and
        // no shared memory is involved, so the next item's Q may already be loading. (Staging
        // the rows in shared memory for TMA stores measured no faster: the SM's write path to
        // L2 bounds either form, and the staging buffers cost a K/V ring slot.) Once these
        // loads have returned, O_X may be overwritten, by the next item's first P.V, which
        // waits for this warp's next P. The output is written once and read by no kernel
        // here: it leaves L2 first, ahead of the K/V tiles the other pairs read again.
        const uint64_t pol = l2_evict_first_policy();
        float *dst = a.out + (static_cast<size_t>(out_row0 + t) * a.qh + out_head0 + h) * HD;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float o[32];
          tmem_ld32(to + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv;
          if (valid) {
            if (a.out_v8) {
#pragma unroll
              for (int e = 0; e < 32; e += 8)
                st_global_v8(dst + c * 32 + e, o[e], o[e + 1], o[e + 2], o[e + 3], o[e + 4],
                             o[e + 5], o[e + 6], o[e + 7], pol);
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(dst + c * 32 + e) =
                    make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace pa
