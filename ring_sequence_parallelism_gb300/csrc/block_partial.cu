// block_partial.cu -- blockwise exact attention of one query tile against one
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
//     m' = max(m, rowmax S' * scale)               (lazily, see below)
//     P  = exp(S' * scale - m'),  l = l e^{m-m'} + rowsum P
//     O~ = O~ e^{m-m'} + P V                       (tcgen05, P bf16, fp32 TMEM)
// The state (m, l, O~) is loaded from HBM first when `accumulate` is set, so
// the exact merge with the incoming state is the same rescale.  The epilogue
// writes the state back, or the normalised output O~/l and lse = m + ln l.
//
// Rescale: the reference max m moves when a tile's max exceeds it by more
// than kRescaleThreshold (exp2 domain), and the warp rescales O~ in TMEM only
// when one of its rows moved.  Any reference max gives the same state (l and
// O~ are scaled by exp(-m) consistently).
//
// CTA layout (192 threads, one 128-row query tile per CTA):
//   warp 0      TMEM allocation; lane 0 issues the TMA loads (Q once, then
//               K and V tiles through a 2-stage ring)
//   warp 1      lane 0 issues tcgen05.mma: S_j = Q K_j^T into one of two TMEM
//               S buffers, then O += P_{j-1} V_{j-1} (software pipelined)
//   warps 2..5  softmax + epilogue, one query row per thread (TMEM lane
//               quadrant = warp % 4); P goes to shared memory in the
//               128-byte-swizzled K-major layout the MMA reads
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the thread
// records the error, tells the others to stop, and all warps drain what they
// started (TMA loads, MMAs) before TMEM is freed and the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace ringattn {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr int kTmemCols = 512;
constexpr int kTmemS0 = 0;    // S buffer 0: columns [0, 128)
constexpr int kTmemS1 = 128;  // S buffer 1: columns [128, 256)
constexpr int kTmemO = 256;   // O~: columns [256, 256 + d)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The reference max follows the running row max exactly (threshold 0): the
// row's largest weight is then exp2(0) = 1, exact in bf16, so a row that one
// key dominates loses nothing to the bf16 rounding of P.  (A lazy threshold
// of 8 halves the rescale work but leaves the dominant weight anywhere in
// [1, 256) with a bf16 rounding error of up to 2^-9 relative.)
constexpr float kRescaleThreshold = 0.0f;

// Shared-memory map.  Every tile starts on a 1024-byte boundary (the
// 128-byte swizzle pattern repeats every 8 rows of 128 bytes).
template <int D>
struct Layout {
  static constexpr int kSub = 64;                 // bf16 columns per 128-byte row
  static constexpr int kQBytes = kTileM * D * 2;  // Q tile
  static constexpr int kKBytes = kTileN * D * 2;  // one K tile
  static constexpr int kVBytes = kTileN * D * 2;  // one V tile
  static constexpr int kPBytes = kTileM * kTileN * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  static constexpr int kOffP = kOffV + kStages * kVBytes;
  static constexpr int kOffBar = kOffP + kPBytes;
  // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full, o_done, drain
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;
  static constexpr int kBarVFull = kBarKFull + kStages;
  static constexpr int kBarKvEmpty = kBarVFull + kStages;
  static constexpr int kBarSFull = kBarKvEmpty + kStages;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarODone = kBarPFull + 1;
  static constexpr int kBarDrain = kBarODone + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  // room to align the base to 1024; at least 120 KB so that only one CTA
  // (the owner of all 512 TMEM columns) is resident per SM
  static constexpr int kAlloc = (kBytes + 1024) > 122880 ? (kBytes + 1024) : 122880;
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (after
// recording the error and raising the CTA abort flag) when the wall-clock
// limit runs out, or when another thread of the CTA has already aborted.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       const StepArgs& a, int site) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer() - t0 > a.wait_limit_ns) {
      *abort_flag = 1;
      atomicOr(a.err, kErrTimeout);
      atomicCAS(a.err + 1, 0, site);
      return false;
    }
  }
}

// Wait used only while draining after an abort: bounded, records nothing.
__device__ __noinline__ bool mbar_drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit) {
  const uint64_t t0 = global_timer();
  while (!mbar_try(bar, parity)) {
    if (global_timer() - t0 > limit) return false;
  }
  return true;
}

// Wait for a whole warp: every lane polls, and the warp continues only if
// all lanes saw the phase complete, so warp-collective tcgen05 instructions
// after it always run with the full warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const StepArgs& a, int site) {
  const bool ok = mbar_wait(bar, parity, abort_flag, a, site);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 version (1), 61-63 swizzle (2 = 128B)
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t desc = 0;
  desc |= (uint64_t)((addr & 0x3FFFF) >> 4);
  desc |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  desc |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  desc |= (uint64_t)1 << 46;
  desc |= (uint64_t)2 << 61;
  return desc;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (0 = K), 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

#define RA_REGS32(x)                                                                                   \
  "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),      \
      "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]),        \
      "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]),      \
      "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]),      \
      "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
#define RA_INREGS32(x)                                                                                  \
  "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]),   \
      "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]), "r"(x[16]),   \
      "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]), "r"(x[24]),  \
      "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31])
#define RA_FIXREGS32(x)                                                                                \
  "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4]), "+r"(x[5]), "+r"(x[6]), "+r"(x[7]),      \
      "+r"(x[8]), "+r"(x[9]), "+r"(x[10]), "+r"(x[11]), "+r"(x[12]), "+r"(x[13]), "+r"(x[14]),        \
      "+r"(x[15]), "+r"(x[16]), "+r"(x[17]), "+r"(x[18]), "+r"(x[19]), "+r"(x[20]), "+r"(x[21]),      \
      "+r"(x[22]), "+r"(x[23]), "+r"(x[24]), "+r"(x[25]), "+r"(x[26]), "+r"(x[27]), "+r"(x[28]),      \
      "+r"(x[29]), "+r"(x[30]), "+r"(x[31])

// 32 consecutive TMEM columns of this thread's lane -> registers.  The wait
// is in the same asm block so no consumer can be scheduled before it.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&x)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : RA_REGS32(x)
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&x)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
      "%31, %32};" ::"r"(taddr),
      RA_INREGS32(x)
      : "memory");
}

__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- the kernel
struct WorkItem {
  int bh, r, j, t, nk, full_kt, slot;
  long long delta;
};

__device__ __forceinline__ WorkItem decode_item(const StepArgs& a) {
  WorkItem w;
  const int item = blockIdx.x;
  w.bh = item % a.BH;
  const int rest = item / a.BH;
  const int nact = a.fixed_r >= 0 ? 1 : a.n_active;
  const int slot_in_list = rest % nact;
  w.t = a.T - 1 - rest / nact;  // heaviest (largest t) tiles first
  w.r = a.fixed_r >= 0 ? a.fixed_r : (int)a.active[slot_in_list];
  int j = (w.r - a.step) % a.P;
  if (j < 0) j += a.P;
  w.j = j;
  // class and diagonal offset (same rule as the host planner)
  const long long n = a.n;
  int cls;
  long long delta;
  if (!a.causal) {
    cls = RING_BLOCK_FULL;
    delta = n;
  } else {
    delta = (a.layout == RING_LAYOUT_STRIPED) ? (j <= w.r ? 0 : -1) : (long long)(w.r - j) * n;
    cls = delta >= n - 1 ? RING_BLOCK_FULL : (delta <= -n ? RING_BLOCK_SKIP : RING_BLOCK_DIAG);
  }
  w.delta = delta;
  const bool ragged = (n % kTileN) != 0;
  if (cls == RING_BLOCK_SKIP) {
    w.nk = 0;
    w.full_kt = 0;
  } else if (cls == RING_BLOCK_FULL) {
    w.nk = a.KT;
    w.full_kt = ragged ? a.KT - 1 : a.KT;
  } else {
    const long long i_min = (long long)w.t * kTileM;
    const long long i_max = min(n - 1, i_min + kTileM - 1);
    const long long last_key = i_max + delta;
    w.nk = last_key < 0 ? 0 : (int)min((long long)a.KT, last_key / kTileN + 1);
    const long long first_keys = i_min + delta + 1;
    int full = first_keys <= 0 ? 0 : (int)min((long long)w.nk, first_keys / kTileN);
    if (ragged && full == a.KT) full = a.KT - 1;
    w.full_kt = full;
  }
  w.slot = a.kv_mode == kKvSlotR ? w.r : (a.kv_mode == kKvSlotJ ? j : 0);
  return w;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    block_partial_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map) {
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
  const WorkItem w = decode_item(a);

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarQFull), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::kBarKFull + s), 1);
      mbar_init(bar(L::kBarVFull + s), 1);
      mbar_init(bar(L::kBarKvEmpty + s), 1);
    }
    mbar_init(bar(L::kBarSFull + 0), 1);
    mbar_init(bar(L::kBarSFull + 1), 1);
    mbar_init(bar(L::kBarPFull), 128);
    mbar_init(bar(L::kBarODone), 1);
    mbar_init(bar(L::kBarDrain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
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

  const int nk = w.nk;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && nk > 0) {
      const uint32_t q_s = sbase + L::kOffQ;
      mbar_expect_tx(bar(L::kBarQFull), L::kQBytes);
      const int i0 = w.t * kTileM;
      for (int c = 0; c < D / L::kSub; ++c) {
        const uint32_t dst = q_s + c * (kTileM * 128);
        if (a.q_mode == kQStriped)
          tma_load_4d(dst, &q_map, bar(L::kBarQFull), c * L::kSub, w.r, i0, w.bh);
        else if (a.q_mode == kQContiguous)
          tma_load_4d(dst, &q_map, bar(L::kBarQFull), c * L::kSub, i0, w.r, w.bh);
        else
          tma_load_4d(dst, &q_map, bar(L::kBarQFull), c * L::kSub, i0, 0, w.bh);
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nk && ok; ++j) {
        const int st = j % kStages;
        if (j >= kStages) ok = mbar_wait(bar(L::kBarKvEmpty + st), ((j / kStages) - 1) & 1, abort_flag, a, 1);
        if (!ok) break;
        const uint32_t k_s = sbase + L::kOffK + st * L::kKBytes;
        const uint32_t v_s = sbase + L::kOffV + st * L::kVBytes;
        mbar_expect_tx(bar(L::kBarKFull + st), L::kKBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(k_s + c * (kTileN * 128), &k_map, bar(L::kBarKFull + st), c * L::kSub, j * kTileN, w.bh,
                      w.slot);
        mbar_expect_tx(bar(L::kBarVFull + st), L::kVBytes);
        for (int c = 0; c < D / L::kSub; ++c)
          tma_load_4d(v_s + c * (kTileN * 128), &v_map, bar(L::kBarVFull + st), c * L::kSub, j * kTileN, w.bh,
                      w.slot);
        issued = j + 1;
      }
      // Drain: every load this thread started has landed before the CTA
      // can exit (normally these waits return at once).
      const unsigned long long lim = a.wait_limit_ns;
      mbar_drain_wait(bar(L::kBarQFull), 0, lim);
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
        const int st = j % kStages;
        mbar_drain_wait(bar(L::kBarKFull + st), (j / kStages) & 1, lim);
        mbar_drain_wait(bar(L::kBarVFull + st), (j / kStages) & 1, lim);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0 && nk > 0) {
      constexpr uint32_t idesc_qk = instr_desc(kTileM, kTileN, false);
      constexpr uint32_t idesc_pv = instr_desc(kTileM, D, true);
      const uint32_t q_s = sbase + L::kOffQ;
      const uint32_t p_s = sbase + L::kOffP;
      bool ok = mbar_wait(bar(L::kBarQFull), 0, abort_flag, a, 2);
      tc_fence_after();
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj % kStages;
        if (!mbar_wait(bar(L::kBarPFull), jj & 1, abort_flag, a, 3)) return false;
        if (!mbar_wait(bar(L::kBarVFull + st), (jj / kStages) & 1, abort_flag, a, 4)) return false;
        tc_fence_after();
        const uint32_t v_s = sbase + L::kOffV + st * L::kVBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          const uint64_t ad = smem_desc(p_s + (kk / 4) * (kTileM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = smem_desc(v_s + kk * 2048, kTileN * 128, 1024);
          mma_bf16(tmem + kTmemO, ad, bd, idesc_pv, (jj > 0 || a.accumulate || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(L::kBarKvEmpty + st));
        mma_commit(bar(L::kBarODone));
        return true;
      };
      for (int j = 0; j < nk && ok; ++j) {
        const int st = j % kStages;
        ok = mbar_wait(bar(L::kBarKFull + st), (j / kStages) & 1, abort_flag, a, 5);
        if (!ok) break;
        tc_fence_after();
        const uint32_t k_s = sbase + L::kOffK + st * L::kKBytes;
        const uint32_t s_t = tmem + ((j & 1) ? kTmemS1 : kTmemS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = smem_desc(q_s + (kk / 4) * (kTileM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = smem_desc(k_s + (kk / 4) * (kTileN * 128) + (kk % 4) * 32, 16, 1024);
          mma_bf16(s_t, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarSFull + (j & 1)));
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(nk - 1);
      // Drain: all MMAs this thread issued are complete before TMEM is freed.
      mma_commit(bar(L::kBarDrain));
      mbar_drain_wait(bar(L::kBarDrain), 0, a.wait_limit_ns);
    }
  } else {
    // -------------------------------------------- softmax and epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const long long i = (long long)w.t * kTileM + row;
    const bool valid = i < a.n;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const long long g = (long long)w.bh * a.row_bh + (long long)w.r * a.row_r + i * a.row_i;
    float m2 = -INFINITY;  // reference max, log2 domain
    float l = 0.0f;
    if (a.accumulate) {
      if (valid) {
        m2 = a.m_state[g] * kLog2e;
        l = a.l_state[g];
      }
      const float4* src = reinterpret_cast<const float4*>(a.o_state + g * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t x[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          float4 v = valid ? src[c * 8 + q4] : make_float4(0.f, 0.f, 0.f, 0.f);
          x[q4 * 4 + 0] = __float_as_uint(v.x);
          x[q4 * 4 + 1] = __float_as_uint(v.y);
          x[q4 * 4 + 2] = __float_as_uint(v.z);
          x[q4 * 4 + 3] = __float_as_uint(v.w);
        }
        tmem_store32(lane_base + kTmemO + c * 32, x);
      }
      tmem_store_wait();
    }
    bool ok = true;
    const uint32_t p_s = sbase + L::kOffP;
    for (int j = 0; j < nk; ++j) {
      ok = warp_wait(bar(L::kBarSFull + (j & 1)), (j >> 1) & 1, abort_flag, a, 6);
      if (!ok) break;
      tc_fence_after();
      float s[kTileN];
      {
        const uint32_t s_t = lane_base + ((j & 1) ? kTmemS1 : kTmemS0);
#pragma unroll
        for (int c = 0; c < kTileN / 32; ++c) {
          uint32_t x[32];
          tmem_load32(s_t + c * 32, x);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(x[e]);
        }
      }
      if (j >= w.full_kt) {
        const long long kbase = (long long)j * kTileN;
#pragma unroll
        for (int e = 0; e < kTileN; ++e) {
          const long long key = kbase + e;
          if (key >= a.n || key - i > w.delta) s[e] = -INFINITY;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < kTileN; ++e) mx = fmaxf(mx, s[e]);
      const float m_tile = mx * a.scale_log2;
      const bool need = m_tile > m2 + kRescaleThreshold;
      const float m_new = need ? m_tile : m2;
      const float alpha = need ? fast_exp2(m2 - m_new) : 1.0f;
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      // P is rounded to bf16 (the PV operand); l sums the fp32 values.
      float rowsum = 0.0f;
      uint32_t pb[kTileN / 2];
#pragma unroll
      for (int e = 0; e < kTileN; e += 2) {
        const float p0 = fast_exp2(fmaf(s[e], a.scale_log2, -m_use));
        const float p1 = fast_exp2(fmaf(s[e + 1], a.scale_log2, -m_use));
        pb[e / 2] = pack_bf16(p0, p1);
        rowsum += p0 + p1;
      }
      l = l * alpha + rowsum;
      m2 = m_new;
      if (j > 0) {
        ok = warp_wait(bar(L::kBarODone), (j - 1) & 1, abort_flag, a, 7);
        if (!ok) break;
        tc_fence_after();
      }
      if ((j > 0 || a.accumulate) && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          tmem_load32(lane_base + kTmemO + c * 32, x);
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) * alpha);
          tmem_store32(lane_base + kTmemO + c * 32, x);
        }
        tmem_store_wait();
      }
      // P (bf16) -> shared memory, K-major with the 128-byte swizzle:
      // keys [64h, 64h+64) form sub-tile h; 16-byte chunk c of row `row`
      // sits at chunk position c ^ (row & 7).
#pragma unroll
      for (int c = 0; c < kTileN / 8; ++c) {
        const uint32_t sub = p_s + (c / 8) * (kTileM * 128) + row * 128;
        const uint32_t addr = sub + (((c % 8) ^ (row & 7)) << 4);
        st_shared_v4(addr, pb[c * 4 + 0], pb[c * 4 + 1], pb[c * 4 + 2], pb[c * 4 + 3]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull));
    }
    if (ok && nk > 0) {
      ok = warp_wait(bar(L::kBarODone), (nk - 1) & 1, abort_flag, a, 8);
      tc_fence_after();
    }
    if (ok) {
      // ------------------------------------------------------ epilogue
      const bool have_o = nk > 0 || a.accumulate;
      if (a.finalize) {
        const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
        float4* dst = reinterpret_cast<float4*>(a.out + g * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          if (have_o) tmem_load32(lane_base + kTmemO + c * 32, x);
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 v;
              v.x = have_o ? __uint_as_float(x[q4 * 4 + 0]) * inv_l : 0.0f;
              v.y = have_o ? __uint_as_float(x[q4 * 4 + 1]) * inv_l : 0.0f;
              v.z = have_o ? __uint_as_float(x[q4 * 4 + 2]) * inv_l : 0.0f;
              v.w = have_o ? __uint_as_float(x[q4 * 4 + 3]) * inv_l : 0.0f;
              dst[c * 8 + q4] = v;
            }
          }
        }
        if (valid) a.lse[g] = (l > 0.0f) ? (m2 + __log2f(l)) * kLn2 : -INFINITY;
      } else {
        float4* dst = reinterpret_cast<float4*>(a.o_state + g * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          if (have_o) tmem_load32(lane_base + kTmemO + c * 32, x);
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 v;
              v.x = have_o ? __uint_as_float(x[q4 * 4 + 0]) : 0.0f;
              v.y = have_o ? __uint_as_float(x[q4 * 4 + 1]) : 0.0f;
              v.z = have_o ? __uint_as_float(x[q4 * 4 + 2]) : 0.0f;
              v.w = have_o ? __uint_as_float(x[q4 * 4 + 3]) : 0.0f;
              dst[c * 8 + q4] = v;
            }
          }
        }
        if (valid) {
          a.m_state[g] = m2 * kLn2;
          a.l_state[g] = l;
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
  return (int)cudaFuncSetAttribute(block_partial_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Layout<D>::kAlloc);
}

}  // namespace

int block_partial_smem_bytes(int d) { return d == 64 ? Layout<64>::kAlloc : Layout<128>::kAlloc; }

int prepare_block_partial_kernels() {
  int e = prepare_one<64>();
  if (e) return e;
  return prepare_one<128>();
}

int launch_block_partial(const StepArgs& a, const void* q_map, const void* k_map, const void* v_map, int d,
                         int grid, void* stream) {
  if (grid <= 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(k_map);
  const CUtensorMap& vm = *static_cast<const CUtensorMap*>(v_map);
  if (d == 64) {
    block_partial_kernel<64><<<grid, kThreads, Layout<64>::kAlloc, s>>>(a, qm, km, vm);
  } else {
    block_partial_kernel<128><<<grid, kThreads, Layout<128>::kAlloc, s>>>(a, qm, km, vm);
  }
  return (int)cudaGetLastError();
}

}  // namespace ringattn
