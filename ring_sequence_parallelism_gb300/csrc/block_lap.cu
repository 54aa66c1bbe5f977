// block_lap.cu -- the ring forward in one launch ("lap" schedule, sm_103a).
//
// Each CTA owns two 128-row query tiles of shard r and makes the ring's lap
// itself: at step s = 0 .. P-1 it meets K/V block j = (r - s) mod P, in step
// order, exactly the blocks and order the ring gives shard r ([RA-CN]
// "环是怎样工作的").  The running state (m, l, O~) stays on chip from the first
// step to the last (m and l in the softmax threads' registers, O~ in TMEM),
// so nothing of it crosses HBM between steps, and the CTA's set-up and
// epilogue are paid once per lap instead of once per step.  Inside a block
// the arithmetic is the step kernel's ([RA-CN] "两层分块如何嵌套": update the
// running statistics tile by tile; "局部 Softmax 为什么不能直接相加" and [GRA]
// "Why partial results are allowed to merge" for the rescale): per key tile
//   S = Q K^T, masked by the block's rule;  m' = max(m, rowmax S);
//   P = exp(S - m');  l = l e^{m-m'} + rowsum P;  O~ = O~ e^{m-m'} + P V.
// After the last block: out = O~ / l, lse = m + ln l, in natural order.
//
// The K/V blocks are read in place from the packed (shard-major) buffer,
// slot j holding block j, as rotation mode 0 does: there is no rotation to
// overlap, since no block moves.  This pays off when a step has little work
// per query tile (sliding windows, packed documents): the step schedule then
// spends most of its time moving the running state through HBM.
//
// CTA layout, TMEM and barriers as in the step kernel: warp 0 issues the TMA
// loads (Q once, then K and V through 2-stage rings across all blocks of the
// lap), warps 1 and 2 issue the MMAs of tiles A and B, warps 3..6 and 7..10
// run the softmax of tiles A and B.  Stage and barrier phases count loads
// and tiles over the whole lap.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "block_rules.h"
#include "tc_ptx.h"
#include "tmem_regs.h"

namespace ringattn {
namespace {

constexpr int kThreads = 352;
constexpr int kStages = 2;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct LapLayout {
  static constexpr int kSub = 64;
  static constexpr int kQBytes = kTileM * D * 2;
  static constexpr int kKBytes = kTileN * D * 2;
  static constexpr int kVBytes = kTileN * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  static constexpr int kOffBar = kOffV + kStages * kVBytes;
  static constexpr int kBarQFull = 0;                         // [2]
  static constexpr int kBarKFull = 2;                         // [stage]
  static constexpr int kBarKEmpty = kBarKFull + kStages;      // [stage][tile]
  static constexpr int kBarVFull = kBarKEmpty + 2 * kStages;  // [stage]
  static constexpr int kBarVEmpty = kBarVFull + kStages;      // [stage][tile]
  static constexpr int kBarSFull = kBarVEmpty + 2 * kStages;  // [tile]
  static constexpr int kBarPFull = kBarSFull + 2;             // [tile]
  static constexpr int kBarOFull = kBarPFull + 2;             // [tile]
  static constexpr int kBarDrain = kBarOFull + 2;             // [tile]
  static constexpr int kNumBars = kBarDrain + 2;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kAlloc = (kBytes + 1024) > 122880 ? (kBytes + 1024) : 122880;
  __device__ static constexpr uint32_t tmem_s(int t) { return t == 0 ? 0u : 128u; }
  __device__ static constexpr uint32_t tmem_o(int t) { return t == 0 ? 256u : 256u + D; }
};

// One block of the lap for the CTA's tile pair: key tiles lo .. lo+nk-1 of
// block j are loaded (loop index x = 0 .. nk-1), and every existing query
// tile of the pair computes all of them; a tile masks x < mask_lo and
// x >= mask_from, which covers the key tiles outside its own range (its row
// bounds then exclude every key there).  Both tiles thus consume the lap's
// loads in the same order, one after another, so every wait on a stage's
// full barrier is for the phase right after the last one the tile saw (a
// parity wait cannot tell a phase from the one two before it, which a tile
// skipping loads would risk).
struct Visit {
  int j, lo, nk;
  Tile tile;  // the rule of the query tile the calling warp serves
};

// t: the query tile (0 or 1) whose rule `v.tile` keeps; the union range needs
// both tiles' key-tile ranges, the rest of the other tile is dropped.
template <bool kWin>
__device__ __forceinline__ void block_visit(const StepArgs& a, int r, int j, int u, int t, Visit& v) {
  v.j = j;
  const Tile t0 = tile_work<kWin>(a, r, j, 2 * u);
  const Tile t1 = tile_work<kWin>(a, r, j, 2 * u + 1);
  int lo = a.KT, hi = 0;
  if (t0.kt_hi > t0.kt_lo) lo = min(lo, t0.kt_lo), hi = max(hi, t0.kt_hi);
  if (t1.kt_hi > t1.kt_lo) lo = min(lo, t1.kt_lo), hi = max(hi, t1.kt_hi);
  if (hi == 0) lo = 0;
  v.lo = lo;
  v.nk = hi - lo;
  v.tile = t == 0 ? t0 : t1;
  Tile& tt = v.tile;
  tt.jb = 0;
  tt.je = v.nk;
  const bool own = tt.kt_hi > tt.kt_lo;
  tt.mask_lo = (!own || tt.full_lo >= tt.full_hi) ? v.nk : tt.full_lo - lo;
  tt.mask_from = own ? tt.full_hi - lo : v.nk;
}

__device__ __forceinline__ int block_at_step(int r, int s, int P) {
  int j = (r - s) % P;
  return j < 0 ? j + P : j;
}

// Position in the lap: block s (block v.j), loop index x, and g, the global
// index of the load (and, since every tile consumes every load, of the tile).
struct LapPos {
  int s, x, g;
  Visit v;
};

// The first load at or after block s; false when the lap has no more.
template <bool kWin>
__device__ __forceinline__ bool seek_load(const StepArgs& a, int r, int u, int t, LapPos& p) {
  while (p.s < a.P) {
    block_visit<kWin>(a, r, block_at_step(r, p.s, a.P), u, t, p.v);
    if (p.v.nk > 0) {
      p.x = 0;
      return true;
    }
    ++p.s;
  }
  return false;
}

template <bool kWin>
__device__ __forceinline__ bool next_load(const StepArgs& a, int r, int u, int t, LapPos& p) {
  ++p.g;
  if (++p.x < p.v.nk) return true;
  ++p.s;
  return seek_load<kWin>(a, r, u, t, p);
}

template <int D, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_lap_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map) {
  using L = LapLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kOffBar;
  auto bar = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // blockIdx.x -> (head, tile pair, shard): all CTAs of one head are
  // consecutive, so those running together read the same K/V head and it
  // stays in L2; within a head the heaviest tile pairs (largest u under the
  // causal mask) start first.
  const int U = (a.T + 1) / 2;
  const int per_head = U * a.P;
  const int bh = blockIdx.x / per_head;
  const int rem = blockIdx.x % per_head;
  const int u = U - 1 - rem / a.P;
  const int r = rem % a.P;
  const int kvh = bh / a.G;
  const int nq = 2 * u + 1 < a.T ? 2 : 1;  // query tiles that exist (each has keys: its own position)

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarQFull + 1), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::kBarKFull + s), 1);
      mbar_init(bar(L::kBarVFull + s), 1);
      for (int t = 0; t < 2; ++t) {
        mbar_init(bar(L::kBarKEmpty + 2 * s + t), 1);
        mbar_init(bar(L::kBarVEmpty + 2 * s + t), 1);
      }
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarSFull + t), 1);
      mbar_init(bar(L::kBarPFull + t), 128);
      mbar_init(bar(L::kBarOFull + t), 1);
      mbar_init(bar(L::kBarDrain + t), 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
    // Q tiles before the set-up barrier
    for (int t = 0; t < nq; ++t) {
      const int i0 = (2 * u + t) * kTileM;
      mbar_expect_tx(bar(L::kBarQFull + t), L::kQBytes);
      for (int c = 0; c < D / L::kSub; ++c) {
        const uint32_t dst = sbase + L::kOffQ + t * L::kQBytes + c * (kTileM * 128);
        if (a.q_mode == kQStriped)
          tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, r, i0, bh);
        else if (a.q_mode == kQZigzag)
          tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, i0 < a.n / 2 ? i0 : i0 - a.n / 2,
                      i0 < a.n / 2 ? r : 2 * a.P - 1 - r, bh);
        else
          tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, i0, r, bh);
      }
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Stage st is reloaded once every existing tile has released its last
      // load: the tiles' empty barriers of a stage complete once per load in
      // it, so the wait for the occupant g - 2 has parity ((g - 2) / 2) & 1.
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      LapPos pos{0, 0, 0, {}};
      for (bool more = seek_load<kWin>(a, r, u, 0, pos); more && ok; more = next_load<kWin>(a, r, u, 0, pos)) {
        const int g = pos.g;
        const int st = g % kStages;
        const uint32_t par = ((g - kStages) / kStages) & 1;
        const int key0 = (pos.v.lo + pos.x) * kTileN;
        if (g >= kStages)
          for (int t = 0; t < nq && ok; ++t) ok = mbar_wait(bar(L::kBarKEmpty + 2 * st + t), par, abort_flag, a, 1);
        if (!ok) break;
        mbar_expect_tx(bar(L::kBarKFull + st), L::kKBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(sbase + L::kOffK + st * L::kKBytes + c * (kTileN * 128), &k_map, bar(L::kBarKFull + st),
                      c * L::kSub, key0, kvh, pos.v.j);
        k_issued = g + 1;
        if (g >= kStages)
          for (int t = 0; t < nq && ok; ++t) ok = mbar_wait(bar(L::kBarVEmpty + 2 * st + t), par, abort_flag, a, 2);
        if (!ok) break;
        if (a.debug_drop_v) continue;  // test hook: nothing ever completes v_full
        mbar_expect_tx(bar(L::kBarVFull + st), L::kVBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(sbase + L::kOffV + st * L::kVBytes + c * (kTileN * 128), &v_map, bar(L::kBarVFull + st),
                      c * L::kSub, key0, kvh, pos.v.j);
        v_issued = g + 1;
      }
      // Drain: every load this thread started has landed before the CTA exits.
      const unsigned long long lim = a.wait_limit_ns;
      for (int t = 0; t < nq; ++t) mbar_drain_wait(bar(L::kBarQFull + t), 0, lim);
      for (int x = (k_issued > kStages ? k_issued - kStages : 0); x < k_issued; ++x)
        mbar_drain_wait(bar(L::kBarKFull + x % kStages), (x / kStages) & 1, lim);
      for (int x = (v_issued > kStages ? v_issued - kStages : 0); x < v_issued; ++x)
        mbar_drain_wait(bar(L::kBarVFull + x % kStages), (x / kStages) & 1, lim);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------ MMA issuers (A, B)
    const int t = warp - 1;
    LapPos cur{0, 0, 0, {}};
    if (t < nq && seek_load<kWin>(a, r, u, t, cur)) {
      constexpr uint32_t idesc_qk = instr_desc(kTileM, kTileN, false);
      constexpr uint32_t idesc_pv = instr_desc(kTileM, D, true);
      const uint32_t q_s = sbase + L::kOffQ + t * L::kQBytes;
      auto issue_s = [&](int g) {
        const uint32_t k_s = sbase + L::kOffK + (g % kStages) * L::kKBytes;
        mma_qk<D>(tmem + L::tmem_s(t), smem_desc(q_s, 16, 1024), smem_desc(k_s, 16, 1024), idesc_qk);
        mma_commit_elect(bar(L::kBarSFull + t));
      };
      auto issue_pv = [&](int g) {
        const uint32_t v_s = sbase + L::kOffV + (g % kStages) * L::kVBytes;
        mma_pv(tmem + L::tmem_o(t), tmem + L::tmem_s(t), smem_desc(v_s, kTileN * 128, 1024), idesc_pv,
               g > 0 ? 1u : 0u);
      };
      bool ok = warp_wait(bar(L::kBarQFull + t), 0, abort_flag, a, 3) &&
                warp_wait(bar(L::kBarKFull), 0, abort_flag, a, 4);
      if (ok) {
        issue_s(0);
        mma_commit_elect(bar(L::kBarKEmpty + t));
      }
      while (ok) {
        const int g = cur.g;
        const int st = g % kStages;
        const bool more = next_load<kWin>(a, r, u, t, cur);  // cur is now load g + 1
        ok = warp_wait(bar(L::kBarVFull + st), (g / kStages) & 1, abort_flag, a, 6);
        if (ok && more)
          ok = warp_wait(bar(L::kBarKFull + (g + 1) % kStages), ((g + 1) / kStages) & 1, abort_flag, a, 7);
        ok = ok && warp_wait(bar(L::kBarPFull + t), g & 1, abort_flag, a, 5);
        if (!ok) break;
        tc_fence_after();
        issue_pv(g);
        if (more) {
          issue_s(g + 1);
        } else {
          mma_commit_elect(bar(L::kBarOFull + t));
        }
        mma_commit_elect(bar(L::kBarVEmpty + 2 * st + t));
        if (!more) break;
        mma_commit_elect(bar(L::kBarKEmpty + 2 * ((g + 1) % kStages) + t));
      }
      // Drain: all MMAs this warp issued are complete before TMEM is freed.
      mma_commit_elect(bar(L::kBarDrain + t));
      mbar_drain_wait(bar(L::kBarDrain + t), 0, a.wait_limit_ns);
    }
  } else {
    // -------------------------------------------- softmax and epilogue
    const int t = (warp - 3) / 4;
    const int quad = warp & 3;
    const int ti = 2 * u + t;  // query tile index within the shard
    const long long i_row = (long long)ti * kTileM + quad * 32 + lane;
    const bool valid = i_row < a.nq;
    const long long half_n = a.n / 2;
    const long long gidx =
        (long long)bh * a.row_bh +
        (a.q_mode == kQZigzag ? (i_row < half_n ? (long long)r * half_n + i_row
                                                : (long long)(2 * a.P - 1 - r) * half_n + (i_row - half_n))
                              : (long long)r * a.row_r + i_row * a.row_i);
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + L::tmem_s(t);
    const uint32_t o_addr = tmem + lane_off + L::tmem_o(t);
    float m2 = -INFINITY;  // running max, log2 domain
    float l = 0.0f;
    bool ok = true;
    bool any = false;
    LapPos cur{0, 0, 0, {}};
    if (t < nq && seek_load<kWin>(a, r, u, t, cur)) {
      any = true;
      int cur_s = -1;
      int kmax_row = -1, kmin_row = 0;
      do {
        const int c = cur.g;
        if (cur.s != cur_s) {
          // this row's allowed keys [kmin_row, kmax_row] in block cur.v.j
          cur_s = cur.s;
          row_key_bounds<kWin>(a, cur.v.tile, r, cur.v.j, i_row, kmin_row, kmax_row);
        }
        ok = warp_wait(bar(L::kBarSFull + t), c & 1, abort_flag, a, 8);
        if (!ok) break;
        tc_fence_after();
        float s[kTileN];
        {
          uint32_t x[kTileN];
          tmem_load128(s_addr, x);
#pragma unroll
          for (int e = 0; e < kTileN; ++e) s[e] = __uint_as_float(x[e]);
        }
        const Tile& tw = cur.v.tile;
        if (cur.x < tw.mask_lo || cur.x >= tw.mask_from) {
          const int kbase = (cur.v.lo + cur.x) * kTileN;
#pragma unroll
          for (int e = 0; e < kTileN; ++e) {
            const int key = kbase + e;
            if (key > kmax_row || (kWin && key < kmin_row)) s[e] = -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(s[2 * q], s[2 * q + 1]);
#pragma unroll
        for (int e = 16; e < kTileN; e += 16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) mx[q] = fmax3(mx[q], s[e + 2 * q], s[e + 2 * q + 1]);
        }
        const float m_tile =
            fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7]))) * a.scale_log2;
        const bool need = m_tile > m2;
        const float m_new = need ? m_tile : m2;
        const float alpha = need ? fast_exp2(m2 - m_new) : 1.0f;
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        // p = exp2(s * scale - m) as in the step kernel: P (bf16 pairs) over
        // the first 64 columns of S_t, l summed from the fp32 values, and O~
        // rescaled in TMEM when a row of the warp moved
        const uint64_t sc2 = f2(a.scale_log2, a.scale_log2);
        const uint64_t nm2 = f2(-m_use, -m_use);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pb[kTileN / 2];
#pragma unroll
        for (int e = 0; e < kTileN; e += 2) {
          float t0, t1;
          unf2(ffma2(f2(s[e], s[e + 1]), sc2, nm2), t0, t1);
          const float p0 = fast_exp2(t0);
          const float p1 = fast_exp2(t1);
          pb[e / 2] = pack_bf16(p0, p1);
          acc[(e / 2) & 3] = fadd2(acc[(e / 2) & 3], f2(p0, p1));
        }
        float r0, r1, r2, r3;
        unf2(fadd2(acc[0], acc[1]), r0, r1);
        unf2(fadd2(acc[2], acc[3]), r2, r3);
        l = l * alpha + ((r0 + r1) + (r2 + r3));
        m2 = m_new;
        tmem_store64(s_addr, pb);
        if (c > 0 && __any_sync(0xffffffffu, need)) {
          const uint64_t al2 = f2(alpha, alpha);
          uint32_t x[D];
          if constexpr (D == 128) tmem_load128(o_addr, x);
          else tmem_load64(o_addr, x);
#pragma unroll
          for (int e = 0; e < D; e += 2) {
            float o0, o1;
            unf2(fmul2(f2(__uint_as_float(x[e]), __uint_as_float(x[e + 1])), al2), o0, o1);
            x[e] = __float_as_uint(o0);
            x[e + 1] = __float_as_uint(o1);
          }
          if constexpr (D == 128) tmem_store128(o_addr, x);
          else tmem_store64(o_addr, x);
        }
        tmem_store_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + t));
      } while (next_load<kWin>(a, r, u, t, cur));
    }
    if (ok && any) {
      ok = warp_wait(bar(L::kBarOFull + t), 0, abort_flag, a, 9);
      tc_fence_after();
    }
    if (ok && ti < a.T) {
      // ------------------------------------------------------ epilogue
      const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
      float* dst = a.out + gidx * D;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t x[32];
        if (any) tmem_load32(o_addr + q * 32, x);
        if (valid) {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            float vv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) vv[e] = any ? __uint_as_float(x[q8 * 8 + e]) * inv_l : 0.0f;
            st_global_v8(dst + q * 32 + q8 * 8, vv);
          }
        }
      }
      if (valid) a.lse[gidx] = (l > 0.0f) ? (m2 + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

template <int D>
int prepare_lap_one() {
  int e = (int)cudaFuncSetAttribute(fwd_lap_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    LapLayout<D>::kAlloc);
  if (e) return e;
  return (int)cudaFuncSetAttribute(fwd_lap_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   LapLayout<D>::kAlloc);
}

}  // namespace

int prepare_fwd_lap_kernels() {
  int e = prepare_lap_one<64>();
  if (e) return e;
  return prepare_lap_one<128>();
}

int launch_fwd_lap(const StepArgs& a, const void* q_map, const void* k_map, const void* v_map, int d, void* stream) {
  const long long grid = (long long)((a.T + 1) / 2) * a.P * a.BH;
  if (grid <= 0) return 0;
  if (grid > 0x7fffffffLL) return (int)cudaErrorInvalidValue;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(k_map);
  const CUtensorMap& vm = *static_cast<const CUtensorMap*>(v_map);
  const bool win = (a.causal && a.window > 0) || a.seg_lo != nullptr;  // row-dependent bounds
  if (d == 64) {
    if (win) fwd_lap_kernel<64, true><<<(int)grid, kThreads, LapLayout<64>::kAlloc, s>>>(a, qm, km, vm);
    else fwd_lap_kernel<64, false><<<(int)grid, kThreads, LapLayout<64>::kAlloc, s>>>(a, qm, km, vm);
  } else {
    if (win) fwd_lap_kernel<128, true><<<(int)grid, kThreads, LapLayout<128>::kAlloc, s>>>(a, qm, km, vm);
    else fwd_lap_kernel<128, false><<<(int)grid, kThreads, LapLayout<128>::kAlloc, s>>>(a, qm, km, vm);
  }
  return (int)cudaGetLastError();
}

}  // namespace ringattn
