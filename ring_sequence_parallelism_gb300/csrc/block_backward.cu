// block_backward.cu -- the ring backward of blockwise attention (sm_103a).
//
// What it computes ([RA-CN] "Backward 需要让梯度也沿环传播": every Q-K/V block
// interaction contributes a gradient; the owner of a query shard accumulates
// its dQ from every K/V block; the dK and dV of a travelling K/V block
// accumulate the contributions of the query owners it passes and return to
// the block's owner; the probabilities are recomputed from the forward's
// saved per-row logsumexp, block by block, as in FlashAttention's backward).
// For the allowed pairs (i, k) of query shard r against block j:
//   P_ik  = exp(scale q_i . k_k - lse_i)
//   dP_ik = dO_i . v_k
//   dS_ik = P_ik (dP_ik - D_i),   D_i = dO_i . out_i
//   dV~_k += P_ik dO_i,  dK~_k += dS_ik q_i,  dQ~_i += dS_ik k_k
// and at the end dK = scale dK~, dV = dV~, dQ = scale dQ~.
//
// Kernels of one ring step (every shard r against block j = (r - s) mod P):
//   bwd_dkdv_kernel  one 128-key tile of block j per CTA (keys stationary),
//                    looping over the query tiles of shard r that see it:
//                      S^T  = K Q^T            (tcgen05, K-major operands)
//                      dP^T = V dO^T
//                      P^T, dS^T by the key-row threads, bf16 into TMEM
//                      dV~ += P^T dO,  dK~ += dS^T Q   (A operand in TMEM)
//                    The accumulators enter from slot r of one buffer and
//                    leave to slot r + 1 of the other: they travel with the
//                    block; the last step writes dK and dV in natural order.
//   bwd_dq_kernel    one 128-row query tile of shard r per CTA (queries
//                    stationary), looping over the key tiles of block j:
//                      S = Q K^T,  dP = dO V^T,  dS by the query-row threads,
//                      dQ~ += dS K              (A operand in TMEM)
//                    dQ~ stays with its owner: the running value lives in dq.
// Lap schedule (kLap; one launch of each kernel for the whole ring): a
// dK/dV CTA owns one key tile of block j and makes the block's lap itself,
// visiting the shards j, j + 1, .. in step order, and a dQ CTA owns one
// query tile of shard r and visits the blocks r, r - 1, ..; the
// accumulators stay in TMEM from the first visit to the last.  Same MMAs
// on the same values in the same order as the per-step launches.
// Every MMA shape is one the forward kernel uses (S = Q K^T with both
// operands K-major; O += P V with P in TMEM and V MN-major): each operand
// here is a 128-row tile of a natural-order tensor loaded by TMA with the
// 128-byte swizzle.  S and dP are computed in both kernels (7 MMAs per tile
// pair, 5 of them distinct) so that no gradient needs atomics.
//
// CTA: 320 threads.  warp 0 allocates TMEM and its lane 0 issues the TMA
// loads; warp 1 issues the MMAs (elected lane); warps 2-9 own the rows, two
// warps per TMEM lane quadrant (warp % 4), each thread one row and one half
// of its 128 columns (two warps per SM sub-partition hide each other's TMEM
// and MUFU latency).  Every mbarrier wait is
// bounded; on expiry the CTA drains what it started and frees TMEM.
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

constexpr int kBwdThreads = 320;
constexpr int kBwdTmemCols = 512;
constexpr long long kFar = 1LL << 40;  // "no bound" for the diagonal offsets

// Shared memory of both kernels: two stationary tiles (K, V or Q, dO), two
// stages of two streamed tiles, two stages of 128 nlse2 and nD values (dK/dV
// kernel only), the barriers.  Every tile starts on a 1024-byte boundary.
template <int D>
struct BwdLayout {
  static constexpr int kTile = kTileM * D * 2;      // one 128-row tile
  static constexpr int kOffA = 0;                   // stationary tile 1 (K or Q)
  static constexpr int kOffB = kTile;               // stationary tile 2 (V or dO)
  static constexpr int kOffX = 2 * kTile;           // streamed tile 1, 2 stages (Q or K)
  static constexpr int kOffY = 4 * kTile;           // streamed tile 2, 2 stages (dO or V)
  static constexpr int kOffLse = 6 * kTile;         // [2][128] floats
  static constexpr int kOffD = kOffLse + 1024;      // [2][128] floats
  static constexpr int kOffBar = kOffD + 1024;
  static constexpr int kBarAB = 0;       // stationary tiles landed
  static constexpr int kBarFull = 1;     // [2] stage landed
  static constexpr int kBarEmpty = 3;    // [2] stage released by the MMAs
  static constexpr int kBarS = 5;        // S (or S^T) in TMEM
  static constexpr int kBarDP = 6;       // dP (or dP^T) in TMEM
  static constexpr int kBarP = 7;        // P^T in TMEM (dK/dV) / S read (dQ), 128 arrivals
  static constexpr int kBarDS = 8;       // dS in TMEM, 128 arrivals
  static constexpr int kBarAcc = 9;      // every MMA done: accumulators final
  static constexpr int kBarDrain = 10;
  static constexpr int kNumBars = 11;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  // room to align the base to 1024; at least 120 KB so that only one CTA
  // (the owner of all 512 TMEM columns) is resident per SM
  static constexpr int kAlloc = (kBytes + 1024) > 122880 ? (kBytes + 1024) : 122880;
  // TMEM columns: S/P [0,128), dP/dS [128,256), accumulators from 256
  static constexpr uint32_t kTmS = 0, kTmDP = 128, kTmAcc1 = 256, kTmAcc2 = 256 + D;
};

// D (+)= A B with A (128 x 128 bf16) in TMEM as two halves of 32 packed
// columns: K steps 0-3 (columns 0-63 of A) at a_tmem + 0..31 and K steps 4-7
// (columns 64-127) at a_tmem + 64..95, each half written by its own warps
// over the TMEM columns they read; B MN-major with the 128-byte swizzle
// (+2 KB = 16 rows per K step).
__device__ __forceinline__ void mma_pv_split(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 at, bl;\n\t.reg .b64 bd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t"
      "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "add.u32 at, %1, 16;\n\tadd.u32 bl, %2, 256;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "add.u32 at, %1, 24;\n\tadd.u32 bl, %2, 384;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "add.u32 at, %1, 64;\n\tadd.u32 bl, %2, 512;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "add.u32 at, %1, 72;\n\tadd.u32 bl, %2, 640;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "add.u32 at, %1, 80;\n\tadd.u32 bl, %2, 768;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "add.u32 at, %1, 88;\n\tadd.u32 bl, %2, 896;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, 1;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "r"((uint32_t)b_desc), "r"((uint32_t)(b_desc >> 32)), "r"(idesc),
      "r"(accumulate)
      : "memory");
}

// Shared memory of the dQ kernel: Q and dO stationary, then separate rings
// for K (3 stages: a K tile serves S(x) and, at the end of the tile, dQ(x))
// and V (2 stages: a V tile serves dP(x) only), so the load of a K tile has
// about two tile periods to land; 224 KB at d = 128.
template <int D>
struct DqLayout {
  static constexpr int kTile = kTileM * D * 2;
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTile;
  static constexpr int kOffK = 2 * kTile;
  static constexpr int kOffV = kOffK + kKStages * kTile;
  static constexpr int kOffBar = kOffV + kVStages * kTile;
  static constexpr int kBarAB = 0;                         // Q and dO landed
  static constexpr int kBarKFull = 1;                      // [3]
  static constexpr int kBarKEmpty = kBarKFull + kKStages;  // [3]
  static constexpr int kBarVFull = kBarKEmpty + kKStages;  // [2]
  static constexpr int kBarVEmpty = kBarVFull + kVStages;  // [2]
  static constexpr int kBarS = kBarVEmpty + kVStages;
  static constexpr int kBarDP = kBarS + 1;   // [2]: dP buffer b computed
  static constexpr int kBarP = kBarDP + 2;   // S read, 256 arrivals
  static constexpr int kBarDS = kBarP + 1;   // [2]: dS in dP buffer b, 256 arrivals each
  static constexpr int kBarAcc = kBarDS + 2;
  static constexpr int kBarDrain = kBarAcc + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr bool row_barrier(int x) { return x == kBarP || x == kBarDS || x == kBarDS + 1; }
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kAlloc = (kBytes + 1024) > 122880 ? (kBytes + 1024) : 122880;
  // TMEM columns: S [0,128), dP/dS buffers [128,256) and [384,512), dQ~ from 256
  static constexpr uint32_t kTmS = 0, kTmAcc1 = 256;
  __device__ static constexpr uint32_t tm_dp(int b) { return b ? 384u : 128u; }
};

// Mask of block (shard r, block j) for the contiguous and striped layouts:
// local query i and local key k form an allowed pair iff
//   dlo <= k - i <= dhi  and  k < klim.
// Contiguous: pos_q - pos_k = (r - j) n + i - k; striped: (i - k) P + r - j.
// Causal: pos_k <= pos_q.  Window W: pos_q - pos_k < W.
struct BwdRule {
  long long dhi, dlo, kmax;  // kmax: last key that can be allowed (n - 1, or -1 for none)
  long long dhi1, kmax1;     // zigzag: the rule of the shard's late chunk (rows i >= n/2)
};

__device__ __forceinline__ long long floor_div_ll(long long x, long long q) {
  return x >= 0 ? x / q : -((-x + q - 1) / q);
}

__device__ __forceinline__ BwdRule bwd_rule(const BwdArgs& a, int r, int j) {
  BwdRule w;
  w.kmax = w.kmax1 = a.n - 1;
  w.dhi = w.dhi1 = kFar;
  w.dlo = -kFar;
  if (!a.causal) return w;
  if (a.layout == RING_LAYOUT_ZIGZAG) {
    // chunks of c = n/2: shard r holds chunk r, then chunk 2P-1-r.  j < r:
    // both halves see block j's early chunk entirely; j = r: k - i <= 0;
    // j > r: the early rows see nothing, the late rows every key.
    const long long c = a.n / 2;
    if (j < r) {
      w.kmax = w.kmax1 = c - 1;
    } else if (j == r) {
      w.dhi = w.dhi1 = 0;
    } else {
      w.kmax = -1;
    }
    return w;
  }
  if (a.layout == RING_LAYOUT_STRIPED) {
    w.dhi = j <= r ? 0 : -1;
    if (a.window > 0) w.dlo = floor_div_ll((long long)(r - j) - a.window, a.P) + 1;
  } else {
    w.dhi = (long long)(r - j) * a.n;
    if (a.window > 0) w.dlo = (long long)(r - j) * a.n - a.window + 1;
  }
  return w;
}

// Sequence packing: local row x of shard `sh` sits in a document [ds, de)
// of natural positions; as local indices of shard `other` that document is
// [lo, hi] (contiguous: positions sh n + x and o n + y; striped: x P + sh and
// y P + o).  Non-decreasing in x.
__device__ __forceinline__ void doc_range(const BwdArgs& a, int sh, int other, long long x, long long& lo,
                                          long long& hi) {
  const bool striped = a.layout == RING_LAYOUT_STRIPED;
  const long long pos = striped ? x * a.P + sh : (long long)sh * a.n + x;
  const long long ds = a.seg_lo[pos], de = a.seg_hi[pos];
  if (striped) {
    lo = floor_div_ll(ds - other + a.P - 1, a.P);
    hi = floor_div_ll(de - 1 - other, a.P);
  } else {
    lo = ds - (long long)other * a.n;
    hi = de - 1 - (long long)other * a.n;
  }
}

// Zigzag: the query rows of shard r that key k of block j meets, as one
// range [lo, hi] (lo > hi: none).  Half h of the shard (rows [h c, (h+1) c),
// c = n/2) follows (kmax_h, dhi_h): row i allowed iff k <= kmax_h and
// i >= k - dhi_h.  Under the zigzag rules the two halves' ranges join
// without a gap (j < r: every row; j = r: rows >= k; j > r: the late half).
__device__ __forceinline__ void zig_query_range(const BwdArgs& a, const BwdRule& w, long long k, long long& lo,
                                                long long& hi) {
  const long long c = a.n / 2;
  lo = a.n;
  hi = -1;
  if (k <= w.kmax) {
    const long long s0 = max(0LL, k - w.dhi);
    if (s0 <= c - 1) {
      lo = s0;
      hi = c - 1;
    }
  }
  if (k <= w.kmax1) {
    const long long s1 = max(c, k - w.dhi1);
    if (s1 <= (long long)a.n - 1) {
      lo = min(lo, s1);
      hi = (long long)a.n - 1;
    }
  }
}

// Zigzag with a window or documents: a shard and a block each hold chunk x
// then chunk 2P-1-x (c = n/2 tokens), positions increasing with the local
// index, so the queries a key meets and the keys a query sees are one local
// interval each (zz_local_interval of the forward's rules maps an interval
// of allowed positions to it).
__device__ __forceinline__ long long zz_pos_of(const BwdArgs& a, int sh, long long x) {
  const long long c = a.n / 2;
  return x < c ? (long long)sh * c + x : (long long)(2 * a.P - 1 - sh) * c + (x - c);
}

// Keys of block j (local, inclusive) that query row i of shard r sees.
__device__ __forceinline__ void zz_keys_of_row(const BwdArgs& a, int r, int j, long long i, long long& lo,
                                               long long& hi) {
  const long long c = a.n / 2, t = zz_pos_of(a, r, i);
  long long L = 0, U = a.N - 1;
  if (a.causal) {
    U = t;
    if (a.window > 0) L = t - a.window + 1;
  }
  if (a.seg_lo) {
    L = max(L, (long long)a.seg_lo[t]);
    U = min(U, (long long)a.seg_hi[t] - 1);
  }
  zz_local_interval(c, (long long)j * c, (long long)(2 * a.P - 1 - j) * c, L, U, lo, hi);
}

// Query rows of shard r (local, inclusive) that see key k of block j.
__device__ __forceinline__ void zz_rows_of_key(const BwdArgs& a, int r, int j, long long k, long long& lo,
                                               long long& hi) {
  const long long c = a.n / 2, p = zz_pos_of(a, j, k);
  long long L = 0, U = a.N - 1;
  if (a.causal) {
    L = p;
    if (a.window > 0) U = p + a.window - 1;
  }
  if (a.seg_lo) {
    L = max(L, (long long)a.seg_lo[p]);
    U = min(U, (long long)a.seg_hi[p] - 1);
  }
  zz_local_interval(c, (long long)r * c, (long long)(2 * a.P - 1 - r) * c, L, U, lo, hi);
}

// Row of (shard r, local i) of head bh in a natural-order tensor.
__device__ __forceinline__ long long nat_row(const BwdArgs& a, int bh, int r, long long i) {
  if (a.layout == RING_LAYOUT_ZIGZAG) {
    const long long c = a.n / 2;
    const long long pos = i < c ? (long long)r * c + i : (long long)(2 * a.P - 1 - r) * c + (i - c);
    return (long long)bh * a.N + pos;
  }
  return (long long)bh * a.N + (long long)r * a.row_r + i * a.row_i;
}

// TMA load of a 128-row tile (rows i0.. of shard `sh`, head bh) of a
// natural-order tensor through its shard view, D/64 sub-tiles of 64 columns.
template <int D>
__device__ __forceinline__ void load_rows(const BwdArgs& a, uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                          int sh, int i0, int bh) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint32_t to = dst + c * (kTileM * 128);
    if (a.q_mode == kQStriped) {
      tma_load_4d(to, map, bar, c * 64, sh, i0, bh);
    } else if (a.q_mode == kQZigzag) {
      // map dims (d, n/2, 2P chunks, heads): rows of chunk sh, then 2P-1-sh
      const int half_n = a.n / 2;
      tma_load_4d(to, map, bar, c * 64, i0 < half_n ? i0 : i0 - half_n, i0 < half_n ? sh : 2 * a.P - 1 - sh, bh);
    } else {
      tma_load_4d(to, map, bar, c * 64, i0, sh, bh);
    }
  }
}

// ------------------------------------------------------------ preprocessing
// nlse2 = -lse * log2(e) and nD = -(dO . out) for every query row, written
// shard-major [BH][P][n_pad] (rows n..n_pad-1 of a shard get 0); negated so
// that P = exp2(S scale log2(e) + nlse2) and dP - D = dP + nD take one packed
// FMA or add per column pair in the step kernels.  Eight
// threads per row, 16 columns each (d = 128) or 8 (d = 64).
__global__ void bwd_prep_kernel(const float* __restrict__ out, const float* __restrict__ lse,
                                const __nv_bfloat16* __restrict__ dout, float* __restrict__ nlse2,
                                float* __restrict__ nD, int BH, long long n, int n_pad, int d, int P,
                                long long row_r, long long row_i, long long N, int zigzag) {
  const long long rows = (long long)BH * P * n_pad;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gid / 8;
  const int part = (int)(gid % 8);
  if (row >= rows) return;  // whole groups of 8 leave together (rows are a multiple of 128)
  const long long i = row % n_pad;
  const long long rb = row / n_pad;
  const int r = (int)(rb % P);
  const int bh = (int)(rb / P);
  float acc = 0.0f;
  float l2 = 0.0f;
  if (i < n) {
    const long long c = n / 2;
    const long long pos = !zigzag ? (long long)r * row_r + i * row_i
                                  : (i < c ? (long long)r * c + i : (long long)(2 * P - 1 - r) * c + (i - c));
    const long long g = (long long)bh * N + pos;
    const int cols = d / 8;
    const float* o = out + g * d + part * cols;
    const __nv_bfloat16* x = dout + g * d + part * cols;
    for (int c = 0; c < cols; c += 8) {
      const float4 o0 = *reinterpret_cast<const float4*>(o + c);
      const float4 o1 = *reinterpret_cast<const float4*>(o + c + 4);
      const uint4 xb = *reinterpret_cast<const uint4*>(x + c);
      const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xb);
      const float2 a0 = __bfloat1622float2(x2[0]), a1 = __bfloat1622float2(x2[1]);
      const float2 a2 = __bfloat1622float2(x2[2]), a3 = __bfloat1622float2(x2[3]);
      acc += a0.x * o0.x + a0.y * o0.y + a1.x * o0.z + a1.y * o0.w;
      acc += a2.x * o1.x + a2.y * o1.y + a3.x * o1.z + a3.y * o1.w;
    }
    l2 = lse[g] * 1.4426950408889634f;
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  if (part == 0) {
    nD[row] = i < n ? -acc : 0.0f;
    nlse2[row] = -l2;
  }
}

// ------------------------------------------------------------ dK/dV kernel
// blockIdx.x -> (shard r, head bh, key tile kt); the CTAs of one (shard,
// head) are consecutive so its Q and dO tiles stay in L2, and within it the
// key tiles run in ascending order (under the causal mask the early keys of
// a block meet the most queries).
template <int D, bool kWin, bool kLap>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap do_map, const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kOffBar;
  auto bar = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // the key tile, the K/V head (its G query heads share the block) and the
  // block.  Lap launches go head-major, so the CTAs resident at one time
  // share one head's Q and dO (64 MB at 128K tokens, d = 128), which L2
  // holds; within a head the key tiles go in ascending order across all
  // blocks (the early key tiles meet the most queries), so the last wave
  // holds the lightest tiles.
  const int per_head = a.P * a.KT;
  const int kt = kLap ? (int)(blockIdx.x % per_head) / a.P : (int)(blockIdx.x % a.KT);
  const int kvh = kLap ? (int)(blockIdx.x / per_head) : (int)(blockIdx.x / a.KT) % a.BHkv;
  const int gq = kLap ? (int)(blockIdx.x % a.P) : (int)(blockIdx.x / a.KT) / a.BHkv;
  // Per-step launch: this CTA is shard gq's visit to block (gq - step) mod P.
  // Lap (kLap): the CTA owns block gq and makes the block's whole lap
  // itself, visiting shards gq, gq + 1, .. in step order (shard r holds
  // block j at step (r - j) mod P), with dK~ and dV~ kept in TMEM.
  const int nvis = kLap ? a.P : 1;
  int j = kLap ? gq : (gq - a.step) % a.P;
  if (j < 0) j += a.P;
  const int r = gq;  // the shard of visit 0
  auto visit_r = [&](int s) { return r + s >= a.P ? r + s - a.P : r + s; };
  const long long k0 = (long long)kt * kTileN;
  // the rule of (shard rv, block j) and the query tiles of shard rv that see
  // a key of this tile
  auto range_of = [&](int rv, BwdRule& rule, int& it_lo, int& n_it) {
    const int r = rv;
    rule = bwd_rule(a, r, j);
    if (!kWin) rule.dlo = -kFar;
    // last key of the tile that any row can see (zigzag: either half's rule)
    const long long k1 = min(k0 + kTileN - 1, a.layout == RING_LAYOUT_ZIGZAG ? max(rule.kmax, rule.kmax1) : rule.kmax);
    it_lo = 0;
    n_it = 0;
    if (kWin && a.layout == RING_LAYOUT_ZIGZAG) {
      // the key tile lies in one chunk, so its keys' query ranges are
      // non-decreasing: the first key bounds them from below, the last from above
      long long lo0, hi0, lo1, hi1;
      zz_rows_of_key(a, r, j, k0, lo0, hi0);
      zz_rows_of_key(a, r, j, min(k0 + kTileN - 1, (long long)a.n - 1), lo1, hi1);
      const long long i_lo = max(0LL, lo0), i_hi = min((long long)a.n - 1, hi1);
      if (i_lo <= i_hi) {
        it_lo = (int)(i_lo / kTileM);
        n_it = (int)(i_hi / kTileM) + 1 - it_lo;
      }
      return;
    }
    if (k0 <= k1) {
      long long i_lo = max(0LL, k0 - rule.dhi);
      long long i_hi = min((long long)a.n - 1, k1 - rule.dlo);
      if (a.layout == RING_LAYOUT_ZIGZAG) {
        // (the chunk size is a multiple of the tile: a key tile is in one chunk)
        long long lo1, hi1;
        zig_query_range(a, rule, k0, i_lo, i_hi);
        zig_query_range(a, rule, k1, lo1, hi1);
        i_hi = max(i_hi, hi1);
      }
      if (kWin && a.seg_lo) {
        // queries in the documents of the tile's first and last keys
        long long lo0, hi0, lo1, hi1;
        doc_range(a, j, r, k0, lo0, hi0);
        doc_range(a, j, r, k1, lo1, hi1);
        i_lo = max(i_lo, lo0);
        i_hi = min(i_hi, hi1);
      }
      if (i_lo <= i_hi) {
        it_lo = (int)(i_lo / kTileM);
        n_it = (int)(i_hi / kTileM) + 1 - it_lo;
      }
    }
  };
  // visit 0's rule and query tiles (the only visit of a per-step launch)
  BwdRule rule0;
  int it_lo0, n_it0;
  range_of(r, rule0, it_lo0, n_it0);
  int total = n_it0 * a.G;  // loop indices of all visits (visit s: its query tiles x the G query heads)
  for (int s = 1; s < nvis; ++s) {
    BwdRule rl;
    int lo, cnt;
    range_of(visit_r(s), rl, lo, cnt);
    total += cnt * a.G;
  }

  // key-row threads (warps 2..9): lane quadrant warp % 4, column half
  const int quad = warp & 3;
  const long long k_row = k0 + quad * 32 + lane;  // this thread's key
  const bool k_valid = k_row < a.n;
  const size_t slot_rows = (size_t)a.BHkv * a.n;
  const float* in_k = a.acc_in_k + ((size_t)r * slot_rows + (size_t)kvh * a.n + (size_t)k_row) * D;
  const float* in_v = a.acc_in_v + ((size_t)r * slot_rows + (size_t)kvh * a.n + (size_t)k_row) * D;
  // Row threads issue the loads of their half of both incoming accumulator
  // rows now, so the latency overlaps the set-up; the values reach TMEM
  // after the barrier.
  constexpr int kHalfD = D / 2;  // accumulator columns this thread loads and stores
  const int half = warp >= 2 ? (warp - 2) >> 2 : 0;
  const bool load_acc = warp >= 2 && a.accumulate && k_valid;
  uint32_t acc_in[2 * kHalfD];
  if (warp >= 2 && a.accumulate) {
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float* src = (which == 0 ? in_v : in_k) + half * kHalfD;
#pragma unroll
      for (int q8 = 0; q8 < kHalfD / 8; ++q8) {
        if (load_acc) {
          ld_global_v8(src + q8 * 8, acc_in + which * kHalfD + q8 * 8);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc_in[which * kHalfD + q8 * 8 + e] = 0u;
        }
      }
    }
  }

  if (threadIdx.x == 0) {
    for (int x = 0; x < L::kNumBars; ++x)
      mbar_init(bar(x), (x == L::kBarP || x == L::kBarDS) ? 256 : 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
    if (total > 0) {
      // K and V tiles of block j, then the first query stage
      mbar_expect_tx(bar(L::kBarAB), 2 * L::kTile);
      load_rows<D>(a, sbase + L::kOffA, &k_map, bar(L::kBarAB), j, (int)k0, kvh);
      load_rows<D>(a, sbase + L::kOffB, &v_map, bar(L::kBarAB), j, (int)k0, kvh);
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kBwdTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && total > 0) {
      int issued = 0;
      bool ok = true;
      int x = 0;  // loop index over all visits
      for (int s = 0; s < nvis && ok; ++s) {
        const int rv = visit_r(s);
        BwdRule rl;
        int it_lo, n_it;
        range_of(rv, rl, it_lo, n_it);
        // every query head of the group visits the same query tiles: local
        // index xl is query head kvh G + xl / n_it, query tile it_lo + xl % n_it
        for (int xl = 0; xl < n_it * a.G && ok; ++xl, ++x) {
          const int qh = kvh * a.G + xl / n_it;
          const float* lse_base = a.nlse2 + ((size_t)qh * a.P + rv) * a.n_pad;
          const float* d_base = a.nD + ((size_t)qh * a.P + rv) * a.n_pad;
          const int st = x & 1;
          if (x >= 2) ok = mbar_poll(bar(L::kBarEmpty + st), ((x >> 1) - 1) & 1, abort_flag, a, 21);
          if (!ok) break;
          const int i0 = (it_lo + xl % n_it) * kTileM;
          mbar_expect_tx(bar(L::kBarFull + st), 2 * L::kTile + 1024);
          load_rows<D>(a, sbase + L::kOffX + st * L::kTile, &q_map, bar(L::kBarFull + st), rv, i0, qh);
          load_rows<D>(a, sbase + L::kOffY + st * L::kTile, &do_map, bar(L::kBarFull + st), rv, i0, qh);
          bulk_load(sbase + L::kOffLse + st * 512, lse_base + i0, 512, bar(L::kBarFull + st));
          bulk_load(sbase + L::kOffD + st * 512, d_base + i0, 512, bar(L::kBarFull + st));
          issued = x + 1;
        }
      }
      // drain: every load started has landed before the CTA can exit
      const unsigned long long lim = a.wait_limit_ns;
      mbar_drain_wait(bar(L::kBarAB), 0, lim);
      for (int x = issued > 2 ? issued - 2 : 0; x < issued; ++x)
        mbar_drain_wait(bar(L::kBarFull + (x & 1)), (x >> 1) & 1, lim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (total > 0) {
      constexpr uint32_t idesc_s = instr_desc(kTileM, kTileN, false);
      constexpr uint32_t idesc_acc = instr_desc(kTileM, D, true);
      const uint64_t k_desc = smem_desc(sbase + L::kOffA, 16, 1024);
      const uint64_t v_desc = smem_desc(sbase + L::kOffB, 16, 1024);
      auto q_s = [&](int x) { return sbase + L::kOffX + (x & 1) * L::kTile; };
      auto do_s = [&](int x) { return sbase + L::kOffY + (x & 1) * L::kTile; };
      bool ok = warp_poll(bar(L::kBarAB), 0, abort_flag, a, 22) &&
                warp_poll(bar(L::kBarFull), 0, abort_flag, a, 23);
      if (ok) {
        mma_qk<D>(tmem + L::kTmS, k_desc, smem_desc(q_s(0), 16, 1024), idesc_s);  // S^T(0) = K Q^T
        mma_commit_elect(bar(L::kBarS));
        mma_qk<D>(tmem + L::kTmDP, v_desc, smem_desc(do_s(0), 16, 1024), idesc_s);  // dP^T(0) = V dO^T
        mma_commit_elect(bar(L::kBarDP));
      }
      for (int x = 0; x < total && ok; ++x) {
        const uint32_t acc = (x > 0 || a.accumulate) ? 1u : 0u;
        const bool more = x + 1 < total;
        // dV~ += P^T dO once P^T(x) is in TMEM
        ok = warp_poll(bar(L::kBarP), x & 1, abort_flag, a, 24);
        if (!ok) break;
        tc_fence_after();
        mma_pv_split(tmem + L::kTmAcc1, tmem + L::kTmS, smem_desc(do_s(x), kTileM * 128, 1024), idesc_acc, acc);
        // S^T(x+1) overwrites S/P(x) after that MMA (one thread's MMAs run in order)
        if (more) {
          ok = warp_poll(bar(L::kBarFull + ((x + 1) & 1)), ((x + 1) >> 1) & 1, abort_flag, a, 25);
          if (!ok) break;
          mma_qk<D>(tmem + L::kTmS, k_desc, smem_desc(q_s(x + 1), 16, 1024), idesc_s);
          mma_commit_elect(bar(L::kBarS));
        }
        // dK~ += dS^T Q once dS^T(x) is in TMEM
        ok = warp_poll(bar(L::kBarDS), x & 1, abort_flag, a, 26);
        if (!ok) break;
        tc_fence_after();
        mma_pv_split(tmem + L::kTmAcc2, tmem + L::kTmDP, smem_desc(q_s(x), kTileM * 128, 1024), idesc_acc, acc);
        mma_commit_elect(bar(L::kBarEmpty + (x & 1)));
        if (more) {
          mma_qk<D>(tmem + L::kTmDP, v_desc, smem_desc(do_s(x + 1), 16, 1024), idesc_s);
          mma_commit_elect(bar(L::kBarDP));
        }
      }
      if (ok) mma_commit_elect(bar(L::kBarAcc));
      mma_commit_elect(bar(L::kBarDrain));
      mbar_drain_wait(bar(L::kBarDrain), 0, a.wait_limit_ns);
    }
  } else {
    // ------------------------------------- key-row threads and epilogue
    // Two warps per TMEM lane quadrant: half h owns query columns
    // [64h, 64h + 64) of S^T and dP^T and writes its bf16 P^T and dS^T into
    // the first 32 columns of its own range, so the halves never touch each
    // other's columns (the MMAs read the A operand with a jump at the middle).
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int c0 = half * 64;
    // keep both accumulators in TMEM before the first MMA (dV, then dK)
    if (a.accumulate) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? L::kTmAcc1 : L::kTmAcc2) + half * kHalfD;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t buf[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) buf[e] = acc_in[which * kHalfD + c * 32 + e];
          tmem_store32(tmem + lane_off + col + c * 32, buf);
        }
      }
      tmem_store_wait();
    }
    bool ok = true;
    int x = 0;  // loop index over all visits
    for (int s = 0; s < nvis && ok; ++s) {
      const int rv = visit_r(s);
      BwdRule rule = rule0;
      int it_lo = it_lo0, n_it = n_it0;
      if (s > 0) range_of(rv, rule, it_lo, n_it);
      // this key's allowed queries: i_lo_k <= i <= i_hi_k
      long long i_lo_k = k_row <= rule.kmax ? max(0LL, k_row - rule.dhi) : (long long)a.n;
      long long i_hi_k = min((long long)a.n - 1, k_row - rule.dlo);
      if (a.layout == RING_LAYOUT_ZIGZAG) zig_query_range(a, rule, k_row, i_lo_k, i_hi_k);
      if (kWin && a.layout == RING_LAYOUT_ZIGZAG) {
        zz_rows_of_key(a, rv, j, min(k_row, (long long)a.n - 1), i_lo_k, i_hi_k);
        if (!k_valid) i_hi_k = -1;
      } else if (kWin && a.seg_lo && k_row <= rule.kmax) {
        long long qlo, qhi;
        doc_range(a, j, rv, k_row, qlo, qhi);
        i_lo_k = max(i_lo_k, qlo);
        i_hi_k = min(i_hi_k, qhi);
      }
      // (per-step kernels: x_begin is 0, and the loop is the single visit's)
      const int x_begin = x, x_end = x + n_it * a.G;
      for (; x < x_end; ++x) {
        const int st = x & 1;
        const long long i0 = (long long)(it_lo + (x - x_begin) % n_it) * kTileM + c0;  // first query of this half
        const float* lse_s = reinterpret_cast<const float*>(smem + L::kOffLse + st * 512) + c0;
        const float* d_s = reinterpret_cast<const float*>(smem + L::kOffD + st * 512) + c0;
        // the stage's nlse2 and D landed (TMA writes are visible to the threads
        // that observe this barrier), then S^T(x) is in TMEM
        ok = warp_poll(bar(L::kBarFull + st), (x >> 1) & 1, abort_flag, a, 30);
        if (!ok) break;
        // the first 32 of this half's 64 values of -lse log2(e), read while
        // S^T(x) is computed (all 64 would not fit the register budget)
        float4 nl[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) nl[e4] = reinterpret_cast<const float4*>(lse_s)[e4];
        ok = warp_poll(bar(L::kBarS), x & 1, abort_flag, a, 27);
        if (!ok) break;
        tc_fence_after();
        float p[64];
        {
          uint32_t t[64];
          tmem_load64(tmem + lane_off + L::kTmS + c0, t);
#pragma unroll
          for (int e = 0; e < 64; ++e) p[e] = __uint_as_float(t[e]);
        }
        const bool masked = !(i0 >= i_lo_k && i0 + 63 <= i_hi_k);
        // P^T = exp2(S^T scale log2(e) + nlse2): one packed FMA and two MUFU
        // ex2 per column pair; bf16 pairs over the first 32 columns of the half
        {
          const uint64_t sc2 = f2(a.scale_log2, a.scale_log2);
          uint32_t pb[32];
#pragma unroll
          for (int e4 = 8; e4 < 16; ++e4) nl[e4] = reinterpret_cast<const float4*>(lse_s)[e4];
#pragma unroll
          for (int e4 = 0; e4 < 16; ++e4) {
            float v0, v1, v2, v3;
            unf2(ffma2(f2(p[4 * e4], p[4 * e4 + 1]), sc2, f2(nl[e4].x, nl[e4].y)), v0, v1);
            unf2(ffma2(f2(p[4 * e4 + 2], p[4 * e4 + 3]), sc2, f2(nl[e4].z, nl[e4].w)), v2, v3);
            p[4 * e4] = fast_exp2(v0);
            p[4 * e4 + 1] = fast_exp2(v1);
            p[4 * e4 + 2] = fast_exp2(v2);
            p[4 * e4 + 3] = fast_exp2(v3);
          }
          if (masked) {
            // queries of this half outside [i_lo_k, i_hi_k] get 0 (relative
            // bounds clamped to [-1, 64] fit in 32 bits)
            const int lo = (int)max(-1LL, min(64LL, i_lo_k - i0));
            const int hi = (int)max(-1LL, min(64LL, i_hi_k - i0));
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (e < lo || e > hi) p[e] = 0.0f;
          }
#pragma unroll
          for (int e = 0; e < 64; e += 2) pb[e / 2] = pack_bf16(p[e], p[e + 1]);
          tmem_store32(tmem + lane_off + L::kTmS + c0, pb);
        }
        tmem_store_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarP));
        // dS^T = P^T (dP^T - D), 32 columns at a time, bf16 over the read
        // columns; the first 32 values of -D are read while dP^T(x) finishes
        float4 nd4[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) nd4[e4] = reinterpret_cast<const float4*>(d_s)[e4];
        ok = warp_poll(bar(L::kBarDP), x & 1, abort_flag, a, 28);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t t[32];
          tmem_load32(tmem + lane_off + L::kTmDP + c0 + c * 32, t);
          if (c == 0) {
#pragma unroll
            for (int e4 = 8; e4 < 16; ++e4) nd4[e4] = reinterpret_cast<const float4*>(d_s)[e4];
          }
          uint32_t sb[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 nd = nd4[c * 8 + e4];
            const int e = c * 32 + e4 * 4;
            float s0, s1, s2, s3;
            unf2(fmul2(f2(p[e], p[e + 1]),
                       fadd2(f2(__uint_as_float(t[e4 * 4]), __uint_as_float(t[e4 * 4 + 1])), f2(nd.x, nd.y))),
                 s0, s1);
            unf2(fmul2(f2(p[e + 2], p[e + 3]),
                       fadd2(f2(__uint_as_float(t[e4 * 4 + 2]), __uint_as_float(t[e4 * 4 + 3])), f2(nd.z, nd.w))),
                 s2, s3);
            sb[e4 * 2] = pack_bf16(s0, s1);
            sb[e4 * 2 + 1] = pack_bf16(s2, s3);
          }
          tmem_store16(tmem + lane_off + L::kTmDP + c0 + c * 16, sb);
        }
        tmem_store_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDS));
      }
    }
    if (ok && total > 0) {
      ok = warp_poll(bar(L::kBarAcc), 0, abort_flag, a, 29);
      tc_fence_after();
    }
    if (ok) {
      // ------------------------------------------------------ epilogue
      // (tcgen05.ld is warp-collective: every lane loads, valid keys store;
      // half h stores accumulator columns [h D/2, (h + 1) D/2))
      const bool have = total > 0 || a.accumulate;
      float* dst_v;
      float* dst_k;
      if (a.last) {
        const long long gk = nat_row(a, kvh, j, k_row);
        dst_v = a.dv + gk * D;
        dst_k = a.dk + gk * D;
      } else {
        const int to = r + 1 == a.P ? 0 : r + 1;
        const size_t off = ((size_t)to * slot_rows + (size_t)kvh * a.n + (size_t)k_row) * D;
        dst_v = a.acc_out_v + off;
        dst_k = a.acc_out_k + off;
      }
      const float ks = a.last ? a.scale : 1.0f;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float* dst = (which == 0 ? dst_v : dst_k) + half * kHalfD;
        const float mul = which == 0 ? 1.0f : ks;
        const uint32_t col = (which == 0 ? L::kTmAcc1 : L::kTmAcc2) + half * kHalfD;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t t[32];
          if (have) tmem_load32(tmem + lane_off + col + c * 32, t);
          if (k_valid) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = have ? __uint_as_float(t[q8 * 8 + e]) * mul : 0.0f;
              st_global_v8(dst + c * 32 + q8 * 8, v);
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBwdTmemCols)
                 : "memory");
  }
}

// --------------------------------------------------------------- dQ kernel
// blockIdx.x -> (shard r, head bh, query tile t); consecutive CTAs share a
// (shard, head) so the key block stays in L2, and the query tiles with the
// most keys (the last ones under the causal mask) start first.
template <int D, bool kWin, bool kLap>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap do_map, const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map) {
  using L = DqLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kOffBar;
  auto bar = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // query tile, head and shard.  Lap launches go head-major so that the
  // resident CTAs share one head's K and V in L2; within a head the query
  // tiles go in descending order across all shards (the last ones see the
  // most keys), so the last wave holds the lightest tiles.
  const int per_head = a.P * a.T;
  const int t = a.T - 1 - (kLap ? (int)(blockIdx.x % per_head) / a.P : (int)(blockIdx.x % a.T));
  const int bh = kLap ? (int)(blockIdx.x / per_head) : (int)(blockIdx.x / a.T) % a.BH;
  const int r = kLap ? (int)(blockIdx.x % a.P) : (int)(blockIdx.x / a.T) / a.BH;
  // Per-step launch: the tile's visit to block (r - step) mod P.  Lap
  // (kLap): the tile visits every block in step order, j = r, r - 1, ..,
  // with dQ~ kept in TMEM.
  const int nvis = kLap ? a.P : 1;
  auto visit_j = [&](int s) {
    int jv = (r - (kLap ? s : a.step)) % a.P;
    return jv < 0 ? jv + a.P : jv;
  };
  const long long i0 = (long long)t * kTileM;
  const long long i1 = min(i0 + kTileM - 1, (long long)a.n - 1);
  // the rule of (shard r, block jv) for this tile's rows and the key tiles
  // with an allowed key for one of them
  auto range_of = [&](int jv, BwdRule& rule, int& kt_lo, int& n_kt) {
    const int j = jv;
    rule = bwd_rule(a, r, j);
    if (!kWin) rule.dlo = -kFar;
    if (a.layout == RING_LAYOUT_ZIGZAG && i0 >= a.n / 2) {
      // a zigzag tile lies in one chunk; the late chunk has its own rule
      rule.kmax = rule.kmax1;
      rule.dhi = rule.dhi1;
    }
    kt_lo = 0;
    n_kt = 0;
    long long k_lo = max(0LL, i0 + rule.dlo);
    long long k_hi = min(rule.kmax, i1 + rule.dhi);
    if (kWin && a.layout == RING_LAYOUT_ZIGZAG) {
      // the tile's rows lie in one chunk: non-decreasing key ranges
      long long lo0, hi0, lo1, hi1;
      zz_keys_of_row(a, r, j, i0, lo0, hi0);
      zz_keys_of_row(a, r, j, i1, lo1, hi1);
      k_lo = max(0LL, lo0);
      k_hi = min((long long)a.n - 1, hi1);
    } else if (kWin && a.seg_lo) {
      // keys in the documents of the tile's first and last rows
      long long lo0, hi0, lo1, hi1;
      doc_range(a, r, j, i0, lo0, hi0);
      doc_range(a, r, j, i1, lo1, hi1);
      k_lo = max(k_lo, lo0);
      k_hi = min(k_hi, hi1);
    }
    if (k_lo <= k_hi) {
      kt_lo = (int)(k_lo / kTileN);
      n_kt = (int)(k_hi / kTileN) + 1 - kt_lo;
    }
  };
  int total = 0;  // key tiles of all visits
  for (int s = 0; s < nvis; ++s) {
    BwdRule rl;
    int lo, cnt;
    range_of(visit_j(s), rl, lo, cnt);
    total += cnt;
  }
  const int n_kt = total;

  // query-row threads (warps 2..9): lane quadrant warp % 4, column half
  const int quad = warp & 3;
  const int half = warp >= 2 ? (warp - 2) >> 2 : 0;
  constexpr int kHalfD = D / 2;  // dQ~ columns this thread loads and stores
  const long long i_row = i0 + quad * 32 + lane;
  const bool i_valid = i_row < a.n;
  const long long g_row = nat_row(a, bh, r, i_valid ? i_row : 0);
  float* dq_row = a.dq + g_row * D + half * kHalfD;  // this thread's half of the row
  uint32_t buf[kHalfD];
  float nlse2_i = 0.0f, nD_i = 0.0f;
  const bool rows = warp >= 2;
  if (rows) {
    const size_t v = ((size_t)bh * a.P + r) * a.n_pad + (size_t)i_row;
    if (i_valid && n_kt > 0) {
      nlse2_i = a.nlse2[v];
      nD_i = a.nD[v];
    }
    if (a.accumulate && n_kt > 0) {
#pragma unroll
      for (int q8 = 0; q8 < kHalfD / 8; ++q8) {
        if (i_valid) {
          ld_global_v8(dq_row + q8 * 8, buf + q8 * 8);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) buf[q8 * 8 + e] = 0u;
        }
      }
    }
  }

  if (threadIdx.x == 0) {
    for (int x = 0; x < L::kNumBars; ++x)
      mbar_init(bar(x), L::row_barrier(x) ? 256 : 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
    if (n_kt > 0) {
      mbar_expect_tx(bar(L::kBarAB), 2 * L::kTile);
      load_rows<D>(a, sbase + L::kOffQ, &q_map, bar(L::kBarAB), r, (int)i0, bh);
      load_rows<D>(a, sbase + L::kOffDO, &do_map, bar(L::kBarAB), r, (int)i0, bh);
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kBwdTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && n_kt > 0) {
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      int x = 0;  // key tile index over all visits
      for (int s = 0; s < nvis && ok; ++s) {
      const int j = visit_j(s);
      BwdRule rl;
      int kt_lo, n_vis;
      range_of(j, rl, kt_lo, n_vis);
      for (int xl = 0; xl < n_vis && ok; ++xl, ++x) {
        const int k0 = (kt_lo + xl) * kTileN;
        const int ks = x % L::kKStages, vs = x % L::kVStages;
        // K(x) into its stage once dQ(x - 3) has released it
        if (x >= L::kKStages)
          ok = mbar_poll(bar(L::kBarKEmpty + ks), ((x / L::kKStages) - 1) & 1, abort_flag, a, 31);
        if (!ok) break;
        mbar_expect_tx(bar(L::kBarKFull + ks), L::kTile);
        load_rows<D>(a, sbase + L::kOffK + ks * L::kTile, &k_map, bar(L::kBarKFull + ks), j, k0, bh / a.G);
        k_issued = x + 1;
        // V(x) once dP(x - 2) has released its stage
        if (x >= L::kVStages)
          ok = mbar_poll(bar(L::kBarVEmpty + vs), ((x / L::kVStages) - 1) & 1, abort_flag, a, 41);
        if (!ok) break;
        mbar_expect_tx(bar(L::kBarVFull + vs), L::kTile);
        load_rows<D>(a, sbase + L::kOffV + vs * L::kTile, &v_map, bar(L::kBarVFull + vs), j, k0, bh / a.G);
        v_issued = x + 1;
      }
      }
      const unsigned long long lim = a.wait_limit_ns;
      mbar_drain_wait(bar(L::kBarAB), 0, lim);
      for (int x = k_issued > L::kKStages ? k_issued - L::kKStages : 0; x < k_issued; ++x)
        mbar_drain_wait(bar(L::kBarKFull + x % L::kKStages), (x / L::kKStages) & 1, lim);
      for (int x = v_issued > L::kVStages ? v_issued - L::kVStages : 0; x < v_issued; ++x)
        mbar_drain_wait(bar(L::kBarVFull + x % L::kVStages), (x / L::kVStages) & 1, lim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (n_kt > 0) {
      constexpr uint32_t idesc_s = instr_desc(kTileM, kTileN, false);
      constexpr uint32_t idesc_acc = instr_desc(kTileM, D, true);
      const uint64_t q_desc = smem_desc(sbase + L::kOffQ, 16, 1024);
      const uint64_t do_desc = smem_desc(sbase + L::kOffDO, 16, 1024);
      auto k_s = [&](int x) { return sbase + L::kOffK + (x % L::kKStages) * L::kTile; };
      auto v_s = [&](int x) { return sbase + L::kOffV + (x % L::kVStages) * L::kTile; };
      auto k_full = [&](int x, int site) {
        return warp_poll(bar(L::kBarKFull + x % L::kKStages), (x / L::kKStages) & 1, abort_flag, a, site);
      };
      auto v_full = [&](int x, int site) {
        return warp_poll(bar(L::kBarVFull + x % L::kVStages), (x / L::kVStages) & 1, abort_flag, a, site);
      };
      bool ok = warp_poll(bar(L::kBarAB), 0, abort_flag, a, 32) && k_full(0, 33);
      if (ok) {
        mma_qk<D>(tmem + L::kTmS, q_desc, smem_desc(k_s(0), 16, 1024), idesc_s);  // S(0) = Q K^T
        mma_commit_elect(bar(L::kBarS));
        ok = v_full(0, 42);
      }
      if (ok) {
        mma_qk<D>(tmem + L::tm_dp(0), do_desc, smem_desc(v_s(0), 16, 1024), idesc_s);  // dP(0) = dO V^T
        mma_commit_elect(bar(L::kBarDP));
        mma_commit_elect(bar(L::kBarVEmpty));  // V(0) served its only MMA
      }
      // Per key tile x: S(x+1) and dP(x+1) go ahead of dQ(x), so the row
      // threads find both ready when they finish dS(x).  dP alternates
      // between two TMEM buffers: dP(x+1) overwrites dS(x-1), whose reader
      // dQ(x-1) was issued before it (one thread's MMAs run in order).
      for (int x = 0; x < n_kt && ok; ++x) {
        const bool more = x + 1 < n_kt;
        if (more) {
          // S(x+1) may overwrite S(x) once the row threads have read it
          ok = warp_poll(bar(L::kBarP), x & 1, abort_flag, a, 34) && k_full(x + 1, 35);
          if (!ok) break;
          tc_fence_after();
          mma_qk<D>(tmem + L::kTmS, q_desc, smem_desc(k_s(x + 1), 16, 1024), idesc_s);
          mma_commit_elect(bar(L::kBarS));
          ok = v_full(x + 1, 43);
          if (!ok) break;
          const int b1 = (x + 1) & 1;
          mma_qk<D>(tmem + L::tm_dp(b1), do_desc, smem_desc(v_s(x + 1), 16, 1024), idesc_s);
          mma_commit_elect(bar(L::kBarDP + b1));
          mma_commit_elect(bar(L::kBarVEmpty + (x + 1) % L::kVStages));
        }
        // dQ~ += dS K once dS(x) is in TMEM (over dP buffer x mod 2)
        ok = warp_poll(bar(L::kBarDS + (x & 1)), (x >> 1) & 1, abort_flag, a, 36);
        if (!ok) break;
        tc_fence_after();
        mma_pv_split(tmem + L::kTmAcc1, tmem + L::tm_dp(x & 1), smem_desc(k_s(x), kTileN * 128, 1024), idesc_acc,
                     (x > 0 || a.accumulate) ? 1u : 0u);
        mma_commit_elect(bar(L::kBarKEmpty + x % L::kKStages));  // K(x) served S(x) and dQ(x)
      }
      if (ok) mma_commit_elect(bar(L::kBarAcc));
      mma_commit_elect(bar(L::kBarDrain));
      mbar_drain_wait(bar(L::kBarDrain), 0, a.wait_limit_ns);
    }
  } else {
    // ------------------------------------- query-row threads and epilogue
    // Two warps per TMEM lane quadrant: half h owns key columns [64h, 64h+64)
    // of S and dP and writes its bf16 dS into the first 32 columns of its own
    // dP range (the dQ MMA reads the A operand with a jump at the middle).
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int c0 = half * 64;
    if (a.accumulate && n_kt > 0) {
#pragma unroll
      for (int c = 0; c < kHalfD / 32; ++c) {
        uint32_t x32[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x32[e] = buf[c * 32 + e];
        tmem_store32(tmem + lane_off + L::kTmAcc1 + half * kHalfD + c * 32, x32);
      }
      tmem_store_wait();
    }
    bool ok = true;
    int x = 0;  // key tile index over all visits
    for (int s = 0; s < nvis && ok; ++s) {
      const int j = visit_j(s);
      BwdRule rule;
      int kt_lo, n_vis;
      range_of(j, rule, kt_lo, n_vis);
      // this row's allowed keys: k_lo_i <= k <= k_hi_i
      long long k_lo_i = max(0LL, i_row + rule.dlo);
      long long k_hi_i = i_valid ? min(rule.kmax, i_row + rule.dhi) : -1;
      if (kWin && a.layout == RING_LAYOUT_ZIGZAG) {
        zz_keys_of_row(a, r, j, min(i_row, (long long)a.n - 1), k_lo_i, k_hi_i);
        if (!i_valid) k_hi_i = -1;
      } else if (kWin && a.seg_lo && i_valid) {
        long long klo, khi;
        doc_range(a, r, j, i_row, klo, khi);
        k_lo_i = max(k_lo_i, klo);
        k_hi_i = min(k_hi_i, khi);
      }
    for (int xl = 0; xl < n_vis; ++xl, ++x) {
      const long long kbase = (long long)(kt_lo + xl) * kTileN + c0;  // first key of this half
      ok = warp_poll(bar(L::kBarS), x & 1, abort_flag, a, 37);
      if (!ok) break;
      tc_fence_after();
      float p[64];
      {
        uint32_t tt[64];
        tmem_load64(tmem + lane_off + L::kTmS + c0, tt);
#pragma unroll
        for (int e = 0; e < 64; ++e) p[e] = __uint_as_float(tt[e]);
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarP));  // S(x) read: the S columns are free
      const bool masked = !(kbase >= k_lo_i && kbase + 63 <= k_hi_i);
      // P = exp2(S scale log2(e) + nlse2): one packed FMA, two MUFU ex2 per pair
      {
        const uint64_t sc2 = f2(a.scale_log2, a.scale_log2);
        const uint64_t nl2 = f2(nlse2_i, nlse2_i);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float v0, v1;
          unf2(ffma2(f2(p[e], p[e + 1]), sc2, nl2), v0, v1);
          p[e] = fast_exp2(v0);
          p[e + 1] = fast_exp2(v1);
        }
        if (masked) {
          // keys of this half outside [k_lo_i, k_hi_i] get 0 (relative
          // bounds clamped to [-1, 64] fit in 32 bits)
          const int lo = (int)max(-1LL, min(64LL, k_lo_i - kbase));
          const int hi = (int)max(-1LL, min(64LL, k_hi_i - kbase));
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e < lo || e > hi) p[e] = 0.0f;
        }
      }
      const int b = x & 1;  // dP buffer of this tile
      ok = warp_poll(bar(L::kBarDP + b), (x >> 1) & 1, abort_flag, a, 38);
      if (!ok) break;
      tc_fence_after();
      // dS = P (dP - D), 32 columns at a time, bf16 over the read dP columns
      const uint64_t nd2 = f2(nD_i, nD_i);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t tt[32];
        tmem_load32(tmem + lane_off + L::tm_dp(b) + c0 + c * 32, tt);
        uint32_t sb[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float s0, s1;
          unf2(fmul2(f2(p[c * 32 + e], p[c * 32 + e + 1]),
                     fadd2(f2(__uint_as_float(tt[e]), __uint_as_float(tt[e + 1])), nd2)),
               s0, s1);
          sb[e / 2] = pack_bf16(s0, s1);
        }
        tmem_store16(tmem + lane_off + L::tm_dp(b) + c0 + c * 16, sb);
      }
      tmem_store_wait();
      tc_fence_before();
      mbar_arrive(bar(L::kBarDS + b));
    }
    }
    if (ok && n_kt > 0) {
      ok = warp_poll(bar(L::kBarAcc), 0, abort_flag, a, 39);
      tc_fence_after();
    }
    if (ok) {
      // ------------------------------------------------------ epilogue
      // (tcgen05.ld is warp-collective: every lane loads, valid rows store;
      // half h stores dQ columns [h D/2, (h + 1) D/2))
      const float mul = a.last ? a.scale : 1.0f;
      if (n_kt > 0) {
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t tt[32];
          tmem_load32(tmem + lane_off + L::kTmAcc1 + half * kHalfD + c * 32, tt);
          if (i_valid) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(tt[q8 * 8 + e]) * mul;
              st_global_v8(dq_row + c * 32 + q8 * 8, v);
            }
          }
        }
      } else if (i_valid && (!a.accumulate || a.last)) {
        // no key of this block for the tile: dQ~ stays as it is (zero at
        // step 0), scaled at the last step
#pragma unroll
        for (int q8 = 0; q8 < kHalfD / 8; ++q8) {
          uint32_t x8[8];
          float v[8];
          if (a.accumulate) {
            ld_global_v8(dq_row + q8 * 8, x8);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x8[e] = 0u;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(x8[e]) * mul;
          st_global_v8(dq_row + q8 * 8, v);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBwdTmemCols)
                 : "memory");
  }
}

template <int D, bool kWin, bool kLap>
int prepare_bwd_variant() {
  int e;
  if ((e = (int)cudaFuncSetAttribute(bwd_dkdv_kernel<D, kWin, kLap>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     BwdLayout<D>::kAlloc)))
    return e;
  return (int)cudaFuncSetAttribute(bwd_dq_kernel<D, kWin, kLap>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   DqLayout<D>::kAlloc);
}

template <int D>
int prepare_bwd_one() {
  int e;
  if ((e = prepare_bwd_variant<D, false, false>())) return e;
  if ((e = prepare_bwd_variant<D, true, false>())) return e;
  if ((e = prepare_bwd_variant<D, false, true>())) return e;
  return prepare_bwd_variant<D, true, true>();
}

// one launch of a dK/dV or dQ kernel variant (kDq picks the kernel)
template <bool kDq, int D, bool kWin, bool kLap>
void launch_variant(int grid, cudaStream_t s, const BwdArgs& a, const CUtensorMap& qm, const CUtensorMap& om,
                    const CUtensorMap& km, const CUtensorMap& vm) {
  if (kDq)
    bwd_dq_kernel<D, kWin, kLap><<<grid, kBwdThreads, DqLayout<D>::kAlloc, s>>>(a, qm, om, km, vm);
  else
    bwd_dkdv_kernel<D, kWin, kLap><<<grid, kBwdThreads, BwdLayout<D>::kAlloc, s>>>(a, qm, om, km, vm);
}

template <bool kDq>
int launch_kernel(const BwdArgs& a, int grid, const void* q_map, const void* do_map, const void* k_map,
                  const void* v_map, int d, void* stream) {
  if (grid <= 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& om = *static_cast<const CUtensorMap*>(do_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(k_map);
  const CUtensorMap& vm = *static_cast<const CUtensorMap*>(v_map);
  const bool win = (a.causal && a.window > 0) || a.seg_lo != nullptr;
  const bool lap = a.lap != 0;
  const int sel = (d == 64 ? 0 : 4) + (win ? 2 : 0) + (lap ? 1 : 0);
  switch (sel) {
    case 0: launch_variant<kDq, 64, false, false>(grid, s, a, qm, om, km, vm); break;
    case 1: launch_variant<kDq, 64, false, true>(grid, s, a, qm, om, km, vm); break;
    case 2: launch_variant<kDq, 64, true, false>(grid, s, a, qm, om, km, vm); break;
    case 3: launch_variant<kDq, 64, true, true>(grid, s, a, qm, om, km, vm); break;
    case 4: launch_variant<kDq, 128, false, false>(grid, s, a, qm, om, km, vm); break;
    case 5: launch_variant<kDq, 128, false, true>(grid, s, a, qm, om, km, vm); break;
    case 6: launch_variant<kDq, 128, true, false>(grid, s, a, qm, om, km, vm); break;
    default: launch_variant<kDq, 128, true, true>(grid, s, a, qm, om, km, vm); break;
  }
  return (int)cudaGetLastError();
}

}  // namespace

int prepare_backward_kernels() {
  int e = prepare_bwd_one<64>();
  if (e) return e;
  return prepare_bwd_one<128>();
}

int launch_bwd_prep(const float* out, const float* lse, const void* dout, float* nlse2, float* nD, int BH,
                    long long n, int n_pad, int d, int P, long long row_r, long long row_i, long long N,
                    int zigzag, void* stream) {
  const long long threads = (long long)BH * P * n_pad * 8;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid <= 0) return 0;
  bwd_prep_kernel<<<(unsigned)grid, block, 0, static_cast<cudaStream_t>(stream)>>>(
      out, lse, static_cast<const __nv_bfloat16*>(dout), nlse2, nD, BH, n, n_pad, d, P, row_r, row_i, N, zigzag);
  return (int)cudaGetLastError();
}

int launch_bwd_dkdv(const BwdArgs& a, const void* q_map, const void* do_map, const void* k_map, const void* v_map,
                    int d, void* stream) {
  return launch_kernel<false>(a, a.KT * a.P * a.BHkv, q_map, do_map, k_map, v_map, d, stream);
}

int launch_bwd_dq(const BwdArgs& a, const void* q_map, const void* do_map, const void* k_map, const void* v_map,
                  int d, void* stream) {
  return launch_kernel<true>(a, a.T * a.P * a.BH, q_map, do_map, k_map, v_map, d, stream);
}

}  // namespace ringattn
