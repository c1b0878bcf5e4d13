// prefill2_kernel.cuh -- the multi-token (prefill) kernel for head_dim 64 and 128: two query
// tiles per CTA that share every K/V tile and take turns on the tensor cores.
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
// Warps: 0 loads Q and the K tiles, 2 loads the V tiles, 1 allocates TMEM and issues the
// MMAs, 3 is idle; 4..7 are tile A's softmax (TMEM lanes 0..127), 8..11 tile B's.
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
// Register split between warpgroup 0 (producers, MMA) and the two softmax warpgroups:
// 128 * 80 + 256 * 208 <= 384 * 168, the registers the CTA is launched with.
constexpr uint32_t kPrefill2SmallRegs = 80;
constexpr uint32_t kPrefill2BigRegs = 208;
static_assert(128 * kPrefill2SmallRegs + 256 * kPrefill2BigRegs <= 384 * 168,
              "register split exceeds the launch allocation");

enum : int {
  kB2Q = 0,
  kB2SFull = 1,   // +tile
  kB2PFull = 3,   // +tile (128 arrivals)
  kB2ODone = 5,   // +tile
  kB2Done = 7,
  kB2Full = 8,    // +slot
  kB2Empty = 16,  // +slot
  kNumBars2 = 24
};

template <int HD>
__global__ void __launch_bounds__(kPrefill2Threads, 1)
    prefill2_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tout) {
  using C = Prefill2Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_word;
  __shared__ int drain_last[2];
  volatile int *abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kv = blockIdx.x, b = blockIdx.y;
  const int pair = a.n_qtiles - 1 - static_cast<int>(blockIdx.z);  // grid.z counts pairs here

  // the first block-table line (the pages of the first key tiles) heads for L2 while the
  // sequence's offsets are read: the K producer's first lookups then hit L2
  if (threadIdx.x == 0)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.bt + static_cast<size_t>(b) * a.maxp));
  const int q0 = __ldg(a.qs + b), q1 = __ldg(a.qs + b + 1), ctx = __ldg(a.ctx + b);
  const int n = q1 - q0;
  if (ctx < 0 || static_cast<long long>(ctx) > static_cast<long long>(a.maxp) << a.ps_shift) {
    if (threadIdx.x == 0) atomicOr(a.err, PA_DEVERR_CONTEXT);
    return;
  }
  if (q0 < 0 || n < 0 || static_cast<long long>(q1) > a.total || n > ctx) {
    if (threadIdx.x == 0) atomicOr(a.err, PA_DEVERR_QUERY_START);
    return;
  }
  // query tile X covers new tokens [tok0_X, tok0_X + qt); tile A has rows whenever B has
  const int tok0_a = 2 * pair * a.qt, tok0_b = tok0_a + a.qt;
  if (tok0_a >= n) return;
  const int max_pos_a = ctx - n + min(tok0_a + a.qt, n) - 1;
  const int max_pos_b = tok0_b < n ? ctx - n + min(tok0_b + a.qt, n) - 1 : -1;
  const int nt_a = (max_pos_a + C::TN) / C::TN;
  const int nt_b = (max_pos_b + C::TN) / C::TN;  // 0 when tile B is empty
  auto nt_of = [&](int x) { return x ? nt_b : nt_a; };
  const int nt_max = max(nt_a, nt_b);
  const int kv_len = max(max_pos_a, max_pos_b) + 1;
  const int q_rows = a.qt * a.g;

  const uint32_t sbase = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t *sgen = smem_raw + (sbase - smem_addr(smem_raw));
  auto q_tile = [&](int x) { return sbase + C::kQOff + x * C::kQBytes; };
  auto slot_addr = [&](int s) { return sbase + C::kRingOff + s * C::kSlotBytes; };
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars2; ++i)
      mbar_init(bar(i), (i == kB2PFull || i == kB2PFull + 1) ? 128 : 1);
    abort_word = 0;
    fence_barrier_init();
  }
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

  // registers: the softmax warpgroups hold a 128-column score row per thread; each role
  // changes its own allocation inside its branch so the compiler sees one limit per region
  if (warp < 4) regs_decrease<kPrefill2SmallRegs>();
  if (warp == 0 || warp == 2) {
    // ============ producers: warp 0 Q and K(j) (item 2j), warp 2 V(j) (item 2j + 1) ============
    const bool is_v = warp == 2;
    if (lane == 0) {
      prefetch_tensormap(is_v ? &tv : &tk);
      if (!is_v) {
        prefetch_tensormap(&tq);
        mbar_arrive_expect_tx(bar(kB2Q), 2 * C::KB * q_rows * 128);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d_plain(q_tile(x) + kb * (C::kRows * 128), &tq, bar(kB2Q), kb * 64,
                              kv * a.g, q0 + (x ? tok0_b : tok0_a));
      }
    }
    const CUtensorMap *map = is_v ? &tv : &tk;
    const int rows_per_box = min(a.ps, C::TN);
    const int boxes = C::TN / rows_per_box;
    const uint32_t box_bytes = rows_per_box * 128;
    const int32_t *bt_row = a.bt + static_cast<size_t>(b) * a.maxp;
    auto page_of = [&](int j) {
      const int tok = j * C::TN + lane * rows_per_box;
      return (j < nt_max && lane < boxes && tok < kv_len) ? __ldg(bt_row + (tok >> a.ps_shift)) : -1;
    };
    int last_item = -1;
    bool ok = true;
    int page_next = page_of(0);
    for (int j = 0; j < nt_max && ok; ++j) {
      const int item = 2 * j + (is_v ? 1 : 0);
      const int s = item % C::kSlots;
      const int tok = j * C::TN + lane * rows_per_box;
      int page = page_next;
      page_next = page_of(j + 1);
      if (lane < boxes && tok < kv_len && (page < 0 || page >= a.num_pages)) {
        if (!is_v) atomicOr(a.err, PA_DEVERR_PAGE_ID);
        page = -1;
      }
      const uint32_t issue = __ballot_sync(0xffffffffu, page >= 0);
      const int slot_in_page = tok & (a.ps - 1);
      int y, z;
      if (a.layout == PA_LAYOUT_HEAD_MAJOR) {
        y = slot_in_page;
        z = page * a.kvh + kv;
      } else {
        y = kv;
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
          tma_load_3d_plain(slot_addr(s) + kb * (C::TN * 128) + lane * box_bytes, map,
                            bar(kB2Full + s), kb * 64, y, z);
      }
      last_item = item;
    }
    // drain: Q and, in every slot, the newest item either warp loaded into it have landed
    // (older items of a slot were consumed before the slot was refilled)
    if (lane == 0) drain_last[is_v ? 1 : 0] = last_item;
    asm volatile("bar.sync 1, 64;" ::: "memory");
    if (!is_v && lane == 0) {
      drain_wait(bar(kB2Q), 0, a.err);
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
    bool ok = pipe_wait(bar(a.expire ? kB2Done : kB2Q), 0, abort_flag, a.err);
    int waited = -1;  // items are waited for in order; the highest one waited so far
    auto wait_item = [&](int item) {
      if (item <= waited) return true;
      const bool r = pipe_wait(bar(kB2Full + item % C::kSlots), (item / C::kSlots) & 1, abort_flag,
                               a.err);
      if (r) waited = item;
      tc_fence_after();
      return r;
    };
    // MMAs and commits are issued warp-collectively (one elected lane), with operands every
    // lane computes identically
    auto issue_s = [&](int x, int j) {  // S_X(j) = Q_X K(j)^T
      const uint32_t kbase = slot_addr((2 * j) % C::kSlots);
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const uint64_t ad = smem_desc_sw128(q_tile(x) + (ks >> 2) * (C::kRows * 128) + (ks & 3) * 32, 16, 1024);
        const uint64_t bd = smem_desc_sw128(kbase + (ks >> 2) * (C::TN * 128) + (ks & 3) * 32, 16, 1024);
        mma_f16_ss_warp(tmem + 128u * x, ad, bd, C::kIdescS, ks > 0);
      }
      mma_commit_warp(bar(kB2SFull + x));
    };
    auto issue_pv = [&](int x, int j) {  // O_X += P_X(j) V(j), P_X from TMEM
      const uint32_t vbase = slot_addr((2 * j + 1) % C::kSlots);
#pragma unroll
      for (int ks = 0; ks < C::TN / 16; ++ks) {
        const uint64_t bd = smem_desc_sw128(vbase + ks * 2048, C::TN * 128, 1024);
        mma_f16_ts_warp(tmem + 256u + 128u * x, tmem + 128u * x + ks * 8, bd, C::kIdescPV,
                        (j > 0 || ks > 0) ? 1u : 0u);
      }
      if (j == nt_of(x) - 1) mma_commit_warp(bar(kB2ODone + x));
    };
    auto release = [&](int item) { mma_commit_warp(bar(kB2Empty + item % C::kSlots)); };
    auto clear_v_tail = [&](int j) {
      // V rows past the last needed token hold unread cache slots (possibly never written):
      // P is zero there, but 0 * NaN is not, so clear them before the first P.V of that tile.
      const int rows_last = kv_len - j * C::TN;
      if (j != nt_max - 1 || rows_last >= C::TN) return;
      const int per_block = (C::TN - rows_last) * 8;
      uint8_t *vg = sgen + C::kRingOff + ((2 * j + 1) % C::kSlots) * C::kSlotBytes;
      for (int c = lane; c < C::KB * per_block; c += 32) {
        const int kb = c / per_block, r = c % per_block;
        *reinterpret_cast<uint4 *>(vg + kb * (C::TN * 128) + rows_last * 128 + r * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
      __syncwarp();
    };
    if (ok) ok = wait_item(0);
    if (ok) {
      issue_s(0, 0);
      if (nt_b > 0) issue_s(1, 0);
      release(0);
    }
    for (int j = 0; j < nt_max && ok; ++j) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (!ok || j >= nt_of(x)) continue;
        // P_X(j) is released only after V(j) and K(j + 1) have landed (see the softmax)
        ok = pipe_wait(bar(kB2PFull + x), j & 1, abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        if (x == 0 || j >= nt_a) clear_v_tail(j);
        issue_pv(x, j);
        const bool last_v_user = (x == 1) || (j >= nt_b);
        if (last_v_user) release(2 * j + 1);
        if (j + 1 < nt_of(x)) {
          issue_s(x, j + 1);
          const bool last_k_user = (x == 1) || (j + 1 >= nt_b);
          if (last_k_user) release(2 * (j + 1));
        }
      }
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
    const int my_tok0 = x ? tok0_b : tok0_a;
    const int my_nt = x ? nt_b : nt_a;
    const bool valid = row < q_rows && my_tok0 + t < n;
    const int pos = min(ctx - n + my_tok0 + t, x ? max_pos_b : max_pos_a);
    const uint32_t lane_off = static_cast<uint32_t>(rg * 32) << 16;
    const uint32_t ts = tmem + lane_off + 128u * x;
    const uint32_t to = tmem + lane_off + 256u + 128u * x;
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < my_nt; ++j) {
      ok = pipe_wait(bar(kB2SFull + x), j & 1, abort_flag, a.err);
      if (!ok) break;
      tc_fence_after();
      // The MMAs this P releases read V(j) and, for S(j + 1), K(j + 1): one warp of the
      // group confirms they have landed before the group releases P, so the MMA warp waits
      // on P alone. (Neither slot can be recycled first: both are released only after MMAs
      // that need this P.) The probes go out before the score load and are read after it.
      const int iv = 2 * j + 1, ik = 2 * j + 2;
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
      // keys past this row's position are masked out (on tiles that reach the diagonal); the
      // row maximum of the scaled scores is the extreme raw score times the scale (the
      // maximum for a non-negative scale, else the minimum), which saves a multiply per score
      const int lim = pos - j * C::TN;
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = -INFINITY;
      // warp-uniform: the exponent pass below holds tcgen05.st, which the whole warp executes
      const bool full = __all_sync(0xffffffffu, lim >= C::TN - 1);
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
      float rp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rp[e] = 0.f;
      const float nm = -m;
      if (full) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = h2 * 64 + 2 * e;
            // packed fp32 pairs: one FFMA2 for both exponents, one FADD2 for both sums
            const float2 xx =
                ffma2(make_float2(v[c], v[c + 1]), make_float2(sl2, sl2), make_float2(nm, nm));
            const float p0 = prefill_exp2(xx.x);
            const float p1 = prefill_exp2(xx.y);
            const float2 acc =
                fadd2(make_float2(rp[(2 * e) & 7], rp[(2 * e + 1) & 7]), make_float2(p0, p1));
            rp[(2 * e) & 7] = acc.x;
            rp[(2 * e + 1) & 7] = acc.y;
            pk[e] = __uint_as_float(pack_half2(p0, p1));
          }
          tmem_st32(ts + h2 * 32, pk);
        }
      } else {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = h2 * 64 + 2 * e;
            const float p0 = c <= lim ? prefill_exp2(fmaf(v[c], sl2, nm)) : 0.f;
            const float p1 = c + 1 <= lim ? prefill_exp2(fmaf(v[c + 1], sl2, nm)) : 0.f;
            rp[(2 * e) & 7] += p0;
            rp[(2 * e + 1) & 7] += p1;
            pk[e] = __uint_as_float(pack_half2(p0, p1));
          }
          tmem_st32(ts + h2 * 32, pk);
        }
      }
      l += ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kB2PFull + x));
    }
    if (ok && my_nt > 0) ok = pipe_wait(bar(kB2ODone + x), 0, abort_flag, a.err);
    if (ok && my_nt > 0) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // This warp's 32 rows are 32 / g whole tokens when g divides 32; when all of them are
      // new tokens of this sequence they leave by TMA stores, staged in the warp's band of
      // its query tile's buffer (free: every MMA that read it has completed), 32 columns
      // (128 bytes) at a time in the 128-byte swizzle. Full-line writes, issued
      // asynchronously; a warp's stores of 16 bytes per row (the other path) leave half
      // sectors that L2 first fills from DRAM.
      const int wtok = a.out_tma ? 32 / a.g : 0;
      if (a.out_tma && my_tok0 + (rg + 1) * wtok <= n) {
        fence_proxy_async();  // the MMAs' reads of the buffer before these writes
#pragma unroll
        for (int r0 = 0; r0 < HD / 32; r0 += C::KB) {
#pragma unroll
          for (int cc = 0; cc < C::KB; ++cc) {
            float v[32];
            tmem_ld32(to + (r0 + cc) * 32, v);
            const uint32_t band = q_tile(x) + cc * (C::kRows * 128) + rg * (32 * 128);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              sts128(band + lane * 128 + ((k ^ (lane & 7)) << 4),
                     make_uint4(__float_as_uint(v[4 * k] * inv), __float_as_uint(v[4 * k + 1] * inv),
                                __float_as_uint(v[4 * k + 2] * inv),
                                __float_as_uint(v[4 * k + 3] * inv)));
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int cc = 0; cc < C::KB; ++cc)
              tma_store_3d(&tout, q_tile(x) + cc * (C::kRows * 128) + rg * (32 * 128),
                           (r0 + cc) * 32, kv * a.g, q0 + my_tok0 + rg * wtok);
            bulk_commit_group();
            bulk_wait_group_read0();
          }
          __syncwarp();
        }
      } else {
        float *dst = a.out + (static_cast<size_t>(q0 + my_tok0 + t) * a.qh + kv * a.g + h) * HD;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float v[32];
          tmem_ld32(to + c * 32, v);
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4 *>(dst + c * 32 + e) =
                  make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
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
