// block_partial.cu -- blockwise exact attention of query tiles against one
// K/V block, continuing a per-row online-softmax state (sm_103a).
//
// What it computes ([RA-CN] "两层分块如何嵌套": inside a device-level block the
// kernel walks GPU tiles and updates the online-softmax statistics per tile,
// then either emits a mergeable state or updates the running buffer;
// [RA-CN] "局部 Softmax 为什么不能直接相加" for (m, l, O~); [GRA] "Why partial
// results are allowed to merge" for the rescale):
//   for each key tile of the block that has an allowed pair for the tile:
//     S  = Q K^T                                   (tcgen05, bf16 -> fp32 TMEM)
//     S' = S masked with k - i <= delta, k < n     (only tiles that need it)
//     m' = max(m, rowmax S' * scale)
//     P  = exp(S' * scale - m'),  l = l e^{m-m'} + rowsum P
//     O~ = O~ e^{m-m'} + P V                       (tcgen05, P bf16 from TMEM)
// The state (m, l, O~) is loaded from HBM first when `accumulate` is set, so
// the exact merge with the incoming state is the same rescale.  The epilogue
// writes the state back, or the normalised output O~/l and lse = m + ln l.
//
// CTA layout: 352 threads, two 128-row query tiles A and B (rows 256u ..
// 256u+255 of one shard) against the same K/V key tiles.
//   warp 0      TMEM allocation; lane 0 issues the TMA loads (Q_A, Q_B once,
//               then K and V tiles through two 2-stage rings)
//   warp 1      issues the tcgen05.mma of tile A: S_A(0), then per key tile
//               PV_A(j), S_A(j+1); warp 2 does the same for tile B.  The
//               tensor core works on one tile while the other tile's softmax
//               runs.  One issuing warp per tile waits only for its own P:
//               an mbarrier wait costs ~140-270 cycles even on a completed
//               phase, and with one warp serving both tiles those waits sat
//               between one tile's P and its PV.  Each warp releases a K/V
//               stage through its own barrier (tcgen05.commit tracks the
//               MMAs of the issuing thread only).  PV takes P from TMEM (A
//               operand in TMEM, V from shared memory), which keeps
//               shared-memory reads of the MMAs below the 128 B/clk the SM
//               can serve.
//   warps 3..6  softmax + epilogue of tile A, one query row per thread
//   warps 7..10 softmax + epilogue of tile B
// TMEM (512 columns): S_A [0,128), S_B [128,256), O~_A [256,256+d),
// O~_B [256+d, 256+2d).  P_t (bf16 pairs, 64 columns) is written over the
// first half of S_t once the softmax has read S_t into registers; the next
// S_t MMA is issued after the PV MMA that reads P_t, and tcgen05.mma
// instructions from one thread execute in issue order.
//
// Rescale: the reference max follows the running row max exactly (threshold
// 0): the row's largest weight is then exp2(0) = 1, exact in bf16, so a row
// that one key dominates loses nothing to the bf16 rounding of P.  A warp
// rescales its rows of O~ in TMEM only when one of them moved.  The commit
// that signals S_t(j) ready also covers PV_t(j-1), so O~_t is stable then.
//
// Send along the ring (`forward`): the CTA of query tiles 2u, 2u+1 also
// sends key tiles 2u and 2u+1 of its block to slot r+1 of the next step's
// buffer, straight from shared memory with TMA stores, so no separate copy
// rereads the block from HBM ([GRA] "Hiding the ring behind the GEMMs";
// [RA-CN] "双缓冲是重叠成立的基础").  Those two tiles are the last ones the CTA
// loads: a DIAG block ends on its diagonal tiles, and a FULL block walks its
// key tiles in the rotated order 2u+2, .., KT-1, 0, .., 2u+1 (the order of the
// tiles does not change the exact result; every tile's mask uses its own
// key index).  A tile that the mask leaves unused is still loaded for sending.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the thread
// records the error, tells the others to stop, and all warps drain what they
// started (TMA loads, MMAs) before TMEM is freed and the CTA exits.
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
constexpr float kRescaleThreshold = 0.0f;

// Shared-memory map.  Every tile starts on a 1024-byte boundary (the
// 128-byte swizzle pattern repeats every 8 rows of 128 bytes).
template <int D>
struct Layout {
  static constexpr int kSub = 64;                 // bf16 columns per 128-byte row
  static constexpr int kQBytes = kTileM * D * 2;  // one Q tile
  static constexpr int kKBytes = kTileN * D * 2;  // one K tile
  static constexpr int kVBytes = kTileN * D * 2;  // one V tile
  static constexpr int kOffQ = 0;                 // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  static constexpr int kOffBar = kOffV + kStages * kVBytes;
  static constexpr int kBarQFull = 0;  // [2]: tile A, B
  static constexpr int kBarKFull = 2;
  static constexpr int kBarKEmpty = kBarKFull + kStages;      // [stage][tile]
  static constexpr int kBarVFull = kBarKEmpty + 2 * kStages;
  static constexpr int kBarVEmpty = kBarVFull + kStages;      // [stage][tile]
  static constexpr int kBarSFull = kBarVEmpty + 2 * kStages;  // [2]: tile A, B
  static constexpr int kBarPFull = kBarSFull + 2;              // [2]
  static constexpr int kBarOFull = kBarPFull + 2;              // [2]
  static constexpr int kBarDrain = kBarOFull + 2;              // [2]
  static constexpr int kNumBars = kBarDrain + 2;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  // room to align the base to 1024; at least 120 KB so that only one CTA
  // (the owner of all 512 TMEM columns) is resident per SM
  static constexpr int kAlloc = (kBytes + 1024) > 122880 ? (kBytes + 1024) : 122880;
  // TMEM columns of tile t
  __device__ static constexpr uint32_t tmem_s(int t) { return t == 0 ? 0u : 128u; }
  __device__ static constexpr uint32_t tmem_o(int t) { return t == 0 ? 256u : 256u + D; }
};

// Grid (2^head_lg * U * ksplit, head groups, shards) -> (shard, head, tile
// pair, key piece).  blockIdx.x runs over the 2^head_lg heads of a group
// fastest, then the tile pairs from the heaviest (largest u under the causal
// mask) down, then the key pieces; y is the head group, z the shard's slot
// in the step's list.  The CTAs of one group of heads of one shard are
// consecutive, so the K/V blocks they read stay in L2, and the launch order
// puts the heaviest pairs of every group first: the last wave of the launch
// holds light pairs, which shortens its tail.  No division on the way
// without key pieces.
template <bool kWin>
__device__ __forceinline__ WorkItem decode_item(const StepArgs& a) {
  WorkItem w;
  const int U = (a.T + 1) / 2;
  const int x = blockIdx.x;
  const int xi = x >> a.head_lg;
  const int u = U - 1 - (a.ksplit == 1 ? xi : xi % U);
  const int piece = a.ksplit == 1 ? 0 : xi / U;
  w.bh = a.bh0 + ((int)blockIdx.y << a.head_lg) + (x & ((1 << a.head_lg) - 1));
  w.kvh = a.G == 1 ? w.bh : w.bh / a.G;
  const int slot_in_list = a.fixed_r >= 0 ? 0 : (int)blockIdx.z;
  w.r = a.fixed_r >= 0 ? a.fixed_r : (int)a.active[slot_in_list];
  int j = (w.r - a.step) % a.P;
  if (j < 0) j += a.P;
  w.j = j;
  w.tile[0] = tile_work<kWin>(a, w.r, j, 2 * u);
  w.tile[1] = tile_work<kWin>(a, w.r, j, 2 * u + 1);
  w.sr = w.r * a.ksplit + piece;
  if (a.ksplit > 1) {
    // this piece's key tiles only: [p0, p1) of the block's KT
    const int span = (a.KT + a.ksplit - 1) / a.ksplit;
    const int p0 = min(a.KT, piece * span), p1 = min(a.KT, p0 + span);
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      Tile& tt = w.tile[x];
      const int lo_ = max(tt.kt_lo, p0), hi_ = min(tt.kt_hi, p1);
      if (hi_ <= lo_) {
        tt.kt_lo = tt.kt_hi = tt.full_lo = tt.full_hi = 0;
      } else {
        tt.full_lo = min(max(tt.full_lo, lo_), hi_);
        tt.full_hi = min(max(tt.full_hi, lo_), hi_);
        tt.kt_lo = lo_;
        tt.kt_hi = hi_;
      }
    }
  }
  // The CTA loads the union of the two tiles' key-tile ranges (the second
  // tile's range starts and ends no earlier than the first's).
  int lo = a.KT, hi = 0;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (w.tile[x].kt_hi > w.tile[x].kt_lo) {
      lo = min(lo, w.tile[x].kt_lo);
      hi = max(hi, w.tile[x].kt_hi);
    }
  }
  if (hi == 0) lo = 0;
  w.lo = lo;
  w.nk = hi - lo;
  w.fwd_lo = 2 * u;
  w.fwd_hi = min(2 * u + 2, a.KT);
  // Rotating is needed only when the sent tiles are inside a computed prefix
  // but not at its end; then both tiles of a ring block visit the whole
  // prefix (blocks without a diagonal or window), so one order serves both.
  // Short queries (decode) send nothing and keep the natural order.
  w.rot = (a.decode_pos0 < 0 && !(kWin && (a.window > 0 || a.seg_lo)) && lo == 0 && w.fwd_hi < hi) ? w.fwd_hi : 0;
  // Tiles sent along the ring come last: either they end the computed range
  // (after the rotation), possibly followed by the ones beyond it, or they
  // are loaded again after it (a window can leave them inside or below it).
  if (w.fwd_lo >= lo && (w.fwd_hi >= hi || w.rot != 0)) {
    w.ext0 = max(w.fwd_lo, hi);
  } else {
    w.ext0 = w.fwd_lo;
  }
  w.np_send = w.nk + max(0, w.fwd_hi - w.ext0);
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    Tile& tt = w.tile[x];
    if (tt.kt_hi > tt.kt_lo) {
      tt.jb = tt.kt_lo - lo;
      tt.je = tt.kt_hi - lo;
      // With documents the two tiles' ranges can start far apart and leave
      // loaded key tiles that neither uses between them.  A tile whose first
      // loop index is 2 or more would then wait on a stage barrier two
      // phases ahead of its current one (the wait would return at once), and
      // a stage could be reloaded before its unused tile landed.  So each
      // tile with keys runs the CTA's whole range; the masks zero the rest.
      // (A window shifts the second tile's range by at most one tile.  In the
      // zigzag layout the two tiles can lie in different chunks, so a window
      // or documents there take the whole range too.)
      if (kWin && (a.seg_lo || a.layout == RING_LAYOUT_ZIGZAG)) {
        tt.jb = 0;
        tt.je = w.nk;
      }
    } else {
      tt.jb = tt.je = 0;
    }
    // with a rotation (lo = 0, no window) only the ragged last key tile can
    // need the mask; it comes at loop index nk - 1 - rot, and the tiles after
    // it take the mask too, which leaves them unchanged
    tt.mask_lo = tt.full_lo >= tt.full_hi ? tt.je : tt.full_lo - lo;
    tt.mask_from = w.rot == 0 ? tt.full_hi - lo : (tt.full_hi < tt.kt_hi ? w.nk - 1 - w.rot : w.nk);
  }
  w.slot = a.kv_mode == kKvSlotR ? w.r : (a.kv_mode == kKvSlotJ ? j : 0);
  return w;
}

// ------------------------------------------------------------- the kernel
// kWin: row-dependent bounds are in force, a sliding window's lower bound
// and/or the document bounds of sequence packing (instantiated apart so the
// plain kernel carries none of their bookkeeping).
template <int D, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
    block_partial_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                         const __grid_constant__ CUtensorMap k_next, const __grid_constant__ CUtensorMap v_next) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kOffBar;
  auto bar = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // A kernel launched after this one as a programmatic dependent (the
  // decode's merge) may be scheduled now; it waits for this grid's
  // completion itself (griddepcontrol.wait) before reading what it wrote.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const WorkItem w = decode_item<kWin>(a);
  const int nk = w.nk;  // loop indices of computed key tiles
  // Loads for sending only (tiles the mask leaves unused) follow the
  // computed prefix (key_tile), at most two of them, so the MMA warps have
  // released every stage they reuse.
  // With grouped heads, the first query head of each group sends the shared block.
  const bool sends = a.forward && (w.bh % a.G) == 0;
  const int np = sends ? w.np_send : nk;
  const int nq = nk == 0 ? 0 : (w.tile[1].je > w.tile[1].jb ? 2 : 1);  // Q tiles to load (tile A has keys if B has)

  // Softmax threads (warps 3..10, tile (warp-3)/4, one query row each) read
  // their incoming m and l now; the incoming O~ (64 KB a tile) is read once
  // the tile's Q has landed (below), so that the loads the first MMAs need
  // (Q, K(0)) are not queued behind it.
  const int t_sm = warp >= 3 ? (warp - 3) / 4 : 0;
  const Tile tw = t_sm == 0 ? w.tile[0] : w.tile[1];
  const int quad = warp & 3;
  const long long i_row = (long long)tw.t * kTileM + quad * 32 + lane;
  const bool valid = i_row < a.nq;
  const bool in_range = tw.t < a.T;  // the tile exists (its rows may still be partly past n)
  const long long half_n = a.n / 2;
  const long long g =
      (long long)w.bh * a.row_bh +
      (a.q_mode == kQZigzag ? (i_row < half_n ? (long long)w.r * half_n + i_row
                                              : (long long)(2 * a.P - 1 - w.r) * half_n + (i_row - half_n))
                            : (long long)w.sr * a.row_r + i_row * a.row_i);
  // Running state: row-major [row][D] (the C ABI's states), or with
  // state_tiled one block per (head, shard, 128-row tile) laid out
  // [D/8][128 rows][8], so a warp's 32 rows of one 8-column chunk are 1 KB
  // contiguous (row-major rows put each lane of a warp on its own line).
  const long long tile_base = (long long)(w.bh * a.P + w.r) * a.T + tw.t;
  const long long ml_idx = a.state_tiled ? tile_base * kTileM + quad * 32 + lane : g;
  float* const o_row = a.state_tiled ? a.o_state + tile_base * (kTileM * D) + (quad * 32 + lane) * 8 : a.o_state + g * D;
  const int o_stride = a.state_tiled ? kTileM * 8 : 8;  // floats from one 8-column chunk to the next
  float m_in = -INFINITY, l_in = 0.0f;
  const bool load_state = warp >= 3 && a.accumulate && in_range;
  if (load_state && valid) {
    m_in = a.m_state[ml_idx] * kLog2e;
    l_in = a.l_state[ml_idx];
  }

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
    // First loads before the TMEM allocation and the barrier, in the order
    // the first MMA needs them: Q_A and K(0) gate S_A(0).
    if (np > 0) {
      auto load_q = [&](int t) {
        const int i0 = w.tile[t].t * kTileM;
        mbar_expect_tx(bar(L::kBarQFull + t), L::kQBytes);
        for (int c = 0; c < D / L::kSub; ++c) {
          const uint32_t dst = sbase + L::kOffQ + t * L::kQBytes + c * (kTileM * 128);
          if (a.q_mode == kQStriped)
            tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, w.r, i0, w.bh);
          else if (a.q_mode == kQZigzag)
            tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, i0 < a.n / 2 ? i0 : i0 - a.n / 2,
                        i0 < a.n / 2 ? w.r : 2 * a.P - 1 - w.r, w.bh);
          else if (a.q_mode == kQContiguous)
            tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, i0, w.r, w.bh);
          else
            tma_load_4d(dst, &q_map, bar(L::kBarQFull + t), c * L::kSub, i0, 0, w.bh);
        }
      };
      const int key0 = key_tile(a, w, 0) * kTileN;
      if (nq > 0) load_q(0);
      mbar_expect_tx(bar(L::kBarKFull), L::kKBytes);
      for (int c = 0; c < D / L::kSub; ++c)
        tma_load_4d(sbase + L::kOffK + c * (kTileN * 128), &k_map, bar(L::kBarKFull), c * L::kSub, key0, w.kvh,
                    w.slot);
      if (nq > 1) load_q(1);
      if (!a.debug_drop_v) {  // test hook: nothing ever completes v_full
        mbar_expect_tx(bar(L::kBarVFull), L::kVBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(sbase + L::kOffV + c * (kTileN * 128), &v_map, bar(L::kBarVFull), c * L::kSub, key0, w.kvh,
                      w.slot);
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
    // (Q tiles and key tile 0 were issued before the set-up barrier.)
    if (lane == 0 && np > 0) {
      int k_issued = 1, v_issued = a.debug_drop_v ? 0 : 1;
      bool ok = true;
      for (int j = 1; j < np && ok; ++j) {
        const int st = j % kStages;
        const int key0 = key_tile(a, w, j) * kTileN;
        // stage st last held tile j - 2; wait for each tile that used it.
        // A tile's empty barrier of a stage completes once per use by that
        // tile, and a tile's uses start at its own first loop index jb, so
        // the phase of the use at jp is the count of its earlier uses of the
        // stage, (jp - jb) / 2 (jb = 0 without a window).
        const int jp = j - kStages;  // the loop index that last used stage st
        const int jb0 = kWin ? w.tile[0].jb : 0;
        const int jb1 = kWin ? w.tile[1].jb : 0;
        const bool used0 = jp >= w.tile[0].jb && jp < w.tile[0].je;
        const bool used1 = jp >= w.tile[1].jb && jp < w.tile[1].je;
        const uint32_t par0 = ((jp - jb0) >> 1) & 1;
        const uint32_t par1 = ((jp - jb1) >> 1) & 1;
        if (used0) ok = mbar_wait(bar(L::kBarKEmpty + 2 * st), par0, abort_flag, a, 1);
        if (ok && used1) ok = mbar_wait(bar(L::kBarKEmpty + 2 * st + 1), par1, abort_flag, a, 1);
        if (!ok) break;
        mbar_expect_tx(bar(L::kBarKFull + st), L::kKBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(sbase + L::kOffK + st * L::kKBytes + c * (kTileN * 128), &k_map, bar(L::kBarKFull + st),
                      c * L::kSub, key0, w.kvh, w.slot);
        k_issued = j + 1;
        if (used0) ok = mbar_wait(bar(L::kBarVEmpty + 2 * st), par0, abort_flag, a, 2);
        if (ok && used1) ok = mbar_wait(bar(L::kBarVEmpty + 2 * st + 1), par1, abort_flag, a, 2);
        if (!ok) break;
        if (a.debug_drop_v) continue;  // test hook: nothing ever completes v_full
        mbar_expect_tx(bar(L::kBarVFull + st), L::kVBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(sbase + L::kOffV + st * L::kVBytes + c * (kTileN * 128), &v_map, bar(L::kBarVFull + st),
                      c * L::kSub, key0, w.kvh, w.slot);
        v_issued = j + 1;
      }
      if (sends && ok) {
        // Send the last fwd_hi - fwd_lo tiles (still resident in their
        // stages: nothing loads after them) to slot r+1 of the next buffer.
        const int dst = w.r + 1 == a.P ? 0 : w.r + 1;
        const int nf = w.fwd_hi - w.fwd_lo;
        for (int j = np - nf; j < np && ok; ++j) {
          const int st = j % kStages;
          const uint32_t par = (j / kStages) & 1;
          const int key0 = key_tile(a, w, j) * kTileN;
          ok = mbar_wait(bar(L::kBarKFull + st), par, abort_flag, a, 10);
          if (!ok) break;
          for (int c = 0; c < D / L::kSub; ++c)
            tma_store_4d(&k_next, sbase + L::kOffK + st * L::kKBytes + c * (kTileN * 128), c * L::kSub, key0, w.kvh,
                         dst);
          if (a.debug_drop_v) continue;
          ok = mbar_wait(bar(L::kBarVFull + st), par, abort_flag, a, 11);
          if (!ok) break;
          for (int c = 0; c < D / L::kSub; ++c)
            tma_store_4d(&v_next, sbase + L::kOffV + st * L::kVBytes + c * (kTileN * 128), c * L::kSub, key0, w.kvh,
                         dst);
        }
        // the stores have read shared memory before exit
        bulk_commit_and_wait_read();
      }
      // Drain: every load this thread started has landed before the CTA
      // can exit (normally these waits return at once).
      const unsigned long long lim = a.wait_limit_ns;
      for (int t = 0; t < nq; ++t) mbar_drain_wait(bar(L::kBarQFull + t), 0, lim);
      for (int j = (k_issued > kStages ? k_issued - kStages : 0); j < k_issued; ++j)
        mbar_drain_wait(bar(L::kBarKFull + j % kStages), (j / kStages) & 1, lim);
      for (int j = (v_issued > kStages ? v_issued - kStages : 0); j < v_issued; ++j)
        mbar_drain_wait(bar(L::kBarVFull + j % kStages), (j / kStages) & 1, lim);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------ MMA issuers (A, B)
    // The whole warp runs this loop (every lane waits on the barriers);
    // one elected lane issues the MMAs and commits.
    const int t = warp - 1;
    const int jb = t == 0 ? w.tile[0].jb : w.tile[1].jb;  // this tile's loop indices [jb, je)
    const int je = t == 0 ? w.tile[0].je : w.tile[1].je;
    if (je > jb) {
      constexpr uint32_t idesc_qk = instr_desc(kTileM, kTileN, false);
      constexpr uint32_t idesc_pv = instr_desc(kTileM, D, true);
      const uint32_t q_s = sbase + L::kOffQ + t * L::kQBytes;
      auto issue_s = [&](int j) {
        const uint32_t k_s = sbase + L::kOffK + (j % kStages) * L::kKBytes;
        mma_qk<D>(tmem + L::tmem_s(t), smem_desc(q_s, 16, 1024), smem_desc(k_s, 16, 1024), idesc_qk);
        mma_commit_elect(bar(L::kBarSFull + t));
      };
      auto issue_pv = [&](int j) {
        const uint32_t v_s = sbase + L::kOffV + (j % kStages) * L::kVBytes;
        mma_pv(tmem + L::tmem_o(t), tmem + L::tmem_s(t), smem_desc(v_s, kTileN * 128, 1024), idesc_pv,
               (j > jb || a.accumulate) ? 1u : 0u);
      };
      // Waits on TMA data (Q, K, V) need no tcgen05 fence: the mbarrier's
      // transaction count completes only after the bytes are in shared
      // memory.  Only the wait for P (written to TMEM by the softmax warps)
      // is followed by tcgen05.fence::after_thread_sync; a fence issued right
      // after commits measured ~125 cycles of tensor-pipe bubble.  The data
      // waits come first, so the wait for P alone gates the PV + S issue.
      bool ok = warp_wait(bar(L::kBarQFull + t), 0, abort_flag, a, 3) &&
                warp_wait(bar(L::kBarKFull + jb % kStages), (jb / kStages) & 1, abort_flag, a, 4);
      if (ok) {
        issue_s(jb);
        mma_commit_elect(bar(L::kBarKEmpty + 2 * (jb % kStages) + t));
      }
      for (int j = jb; j < je && ok; ++j) {
        const int st = j % kStages;
        const bool more = j + 1 < je;
        ok = warp_wait(bar(L::kBarVFull + st), (j / kStages) & 1, abort_flag, a, 6);
        if (ok && more)
          ok = warp_wait(bar(L::kBarKFull + (j + 1) % kStages), ((j + 1) / kStages) & 1, abort_flag, a, 7);
        ok = ok && warp_wait(bar(L::kBarPFull + t), (j - jb) & 1, abort_flag, a, 5);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j);
        if (more) {
          issue_s(j + 1);
        } else {
          mma_commit_elect(bar(L::kBarOFull + t));
        }
        mma_commit_elect(bar(L::kBarVEmpty + 2 * st + t));
        if (more) mma_commit_elect(bar(L::kBarKEmpty + 2 * ((j + 1) % kStages) + t));
      }
      // Drain: all MMAs this warp issued are complete before TMEM is freed.
      mma_commit_elect(bar(L::kBarDrain + t));
      mbar_drain_wait(bar(L::kBarDrain + t), 0, a.wait_limit_ns);
    }
  } else {
    // -------------------------------------------- softmax and epilogue
    const int t = t_sm;  // 0: tile A (warps 3-6), 1: tile B (warps 7-10)
    // this row's allowed keys [kmin_row, kmax_row] (keys fit in int; the
    // bounds are clamped to it)
    int kmin_row, kmax_row;
    row_key_bounds<kWin>(a, tw, w.r, w.j, i_row, kmin_row, kmax_row);
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + L::tmem_s(t);
    const uint32_t o_addr = tmem + lane_off + L::tmem_o(t);
    float m2 = m_in;  // reference max, log2 domain
    float l = l_in;
    bool ok = true;
    if (load_state) {
      // the incoming O~ into TMEM, after this tile's Q has landed (a tile
      // with keys has its Q loaded; one without reads its state at once)
      if (tw.je > tw.jb) ok = warp_wait(bar(L::kBarQFull + t), 0, abort_flag, a, 12);
      uint32_t o_in[D];
#pragma unroll
      for (int q8 = 0; q8 < D / 8; ++q8) {
        if (valid) {
          ld_global_v8(o_row + q8 * o_stride, o_in + q8 * 8);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) o_in[q8 * 8 + e] = 0u;
        }
      }
      if constexpr (D == 128) tmem_store128(o_addr, o_in);
      else tmem_store64(o_addr, o_in);
      tmem_store_wait();
    }
    for (int j = tw.jb; j < tw.je; ++j) {
      ok = warp_wait(bar(L::kBarSFull + t), (j - tw.jb) & 1, abort_flag, a, 8);
      if (!ok) break;
      tc_fence_after();
      float s[kTileN];
      {
        uint32_t x[kTileN];
        tmem_load128(s_addr, x);
#pragma unroll
        for (int e = 0; e < kTileN; ++e) s[e] = __uint_as_float(x[e]);
      }
      if (j < tw.mask_lo || j >= tw.mask_from) {
        const int kbase = key_tile(a, w, j) * kTileN;
#pragma unroll
        for (int e = 0; e < kTileN; ++e) {
          const int key = kbase + e;
          if (key > kmax_row || (kWin && key < kmin_row)) s[e] = -INFINITY;
        }
      }
      // row max: eight independent chains of 3-input max, then a tree
      float mx[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mx[c] = fmaxf(s[2 * c], s[2 * c + 1]);
#pragma unroll
      for (int e = 16; e < kTileN; e += 16) {
#pragma unroll
        for (int c = 0; c < 8; ++c) mx[c] = fmax3(mx[c], s[e + 2 * c], s[e + 2 * c + 1]);
      }
      const float m_tile =
          fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7]))) * a.scale_log2;
      const bool need = m_tile > m2 + kRescaleThreshold;
      const float m_new = need ? m_tile : m2;
      const float alpha = need ? fast_exp2(m2 - m_new) : 1.0f;
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      // p = exp2(s * scale - m): pairs through one packed FMA, two MUFU ex2,
      // one bf16x2 convert (the PV operand) and one packed add into four
      // independent fp32 pair sums (l sums the fp32 values).
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
      tmem_store64(s_addr, pb);  // P_t over the first 64 columns of S_t
      if ((j > tw.jb || a.accumulate) && __any_sync(0xffffffffu, need)) {
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
    }
    if (ok && tw.je > tw.jb) {
      ok = warp_wait(bar(L::kBarOFull + t), 0, abort_flag, a, 9);
      tc_fence_after();
    }
    if (ok && in_range) {
      // ------------------------------------------------------ epilogue
      const bool have_o = tw.je > tw.jb || a.accumulate;
      if (a.finalize) {
        const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
        float* dst = a.out + g * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          if (have_o) tmem_load32(o_addr + c * 32, x);
          if (valid) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = have_o ? __uint_as_float(x[q8 * 8 + e]) * inv_l : 0.0f;
              st_global_v8(dst + c * 32 + q8 * 8, v);
            }
          }
        }
        if (valid) a.lse[g] = (l > 0.0f) ? (m2 + __log2f(l)) * kLn2 : -INFINITY;
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          if (have_o) tmem_load32(o_addr + c * 32, x);
          if (valid) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = have_o ? __uint_as_float(x[q8 * 8 + e]) : 0.0f;
              st_global_v8(o_row + (c * 4 + q8) * o_stride, v);
            }
          }
        }
        if (valid) {
          a.m_state[ml_idx] = m2 * kLn2;
          a.l_state[ml_idx] = l;
        }
      }
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
int prepare_one() {
  int e = (int)cudaFuncSetAttribute(block_partial_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Layout<D>::kAlloc);
  if (e) return e;
  return (int)cudaFuncSetAttribute(block_partial_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   Layout<D>::kAlloc);
}

}  // namespace

int block_partial_smem_bytes(int d) { return d == 64 ? Layout<64>::kAlloc : Layout<128>::kAlloc; }

int prepare_block_partial_kernels() {
  int e = prepare_one<64>();
  if (e) return e;
  return prepare_one<128>();
}

int block_partial_grid(int T, int n_active, int BH) { return ((T + 1) / 2) * n_active * BH; }

int launch_block_partial(const StepArgs& a, const void* q_map, const void* k_map, const void* v_map, int d,
                         int grid, void* stream, const void* k_next_map, const void* v_next_map) {
  if (grid <= 0) return 0;
  if (a.forward && (!k_next_map || !v_next_map)) return (int)cudaErrorInvalidValue;
  const int U = (a.T + 1) / 2;
  const int per_slot = U * a.ksplit * a.BH;
  if (grid % per_slot != 0) return (int)cudaErrorInvalidValue;
  const int slots = grid / per_slot;
  StepArgs b = a;
  // four heads (two, one) interleave; with key pieces (short queries) one
  b.head_lg = a.ksplit > 1 ? 0 : (a.BH % 4 == 0 ? 2 : (a.BH % 2 == 0 ? 1 : 0));
  const int hg = 1 << b.head_lg;
  const int max_groups = 65535;  // grid y limit
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(k_map);
  const CUtensorMap& vm = *static_cast<const CUtensorMap*>(v_map);
  // without `forward` the kernel never touches the send maps
  const CUtensorMap& kn = *static_cast<const CUtensorMap*>(k_next_map ? k_next_map : k_map);
  const CUtensorMap& vn = *static_cast<const CUtensorMap*>(v_next_map ? v_next_map : v_map);
  // row-dependent bounds: a window or documents
  const bool win = (a.causal && a.window > 0) || a.seg_lo != nullptr;
  for (int h0 = 0; h0 < a.BH; h0 += max_groups * hg) {
    b.bh0 = h0;
    const int groups = (a.BH - h0) / hg < max_groups ? (a.BH - h0) / hg : max_groups;
    const dim3 g3((unsigned)(hg * U * a.ksplit), (unsigned)groups, (unsigned)slots);
    if (d == 64) {
      if (win) block_partial_kernel<64, true><<<g3, kThreads, Layout<64>::kAlloc, s>>>(b, qm, km, vm, kn, vn);
      else block_partial_kernel<64, false><<<g3, kThreads, Layout<64>::kAlloc, s>>>(b, qm, km, vm, kn, vn);
    } else {
      if (win) block_partial_kernel<128, true><<<g3, kThreads, Layout<128>::kAlloc, s>>>(b, qm, km, vm, kn, vn);
      else block_partial_kernel<128, false><<<g3, kThreads, Layout<128>::kAlloc, s>>>(b, qm, km, vm, kn, vn);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  return 0;
}

}  // namespace ringattn
