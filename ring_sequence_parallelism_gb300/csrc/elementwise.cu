// elementwise.cu -- HBM-bound kernels of the ring: empty state, the exact
// merge of two states, finalize into natural order, and the shard-major
// packing of K/V into the rotation buffer.
//
// They move 16- or 32-byte vectors with consecutive threads on consecutive
// addresses.  Grids are a multiple of the SM count with grid-stride loops.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace ringattn {

int sm_count() {
  static int count = 0;
  if (count == 0) {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        c > 0)
      count = c;
    else
      return 1;
  }
  return count;
}

namespace {

int grid_for(long long work, int threads) {
  long long blocks = (work + threads - 1) / threads;
  long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

// Empty state ([RA-CN] "环是怎样工作的": empty_online_softmax_state):
// m = -inf, l = 0, O~ = 0.
__global__ void state_init_kernel(float* __restrict__ m, float* __restrict__ l, float4* __restrict__ o,
                                  long long rows, int d4) {
  const long long total = rows * d4;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (x % d4 == 0) {
      const long long row = x / d4;
      m[row] = -INFINITY;
      l[row] = 0.0f;
    }
  }
}

// Vector global accesses of V fp32 values: V = 8 (256 bits, one full
// 32-byte sector per lane; needs 32-byte alignment) or V = 4 (128 bits).
template <int V>
__device__ __forceinline__ void ldv(const float* p, float (&x)[V]);
template <>
__device__ __forceinline__ void ldv<8>(const float* p, float (&x)[8]) {
  asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7])
               : "l"(p));
}
template <>
__device__ __forceinline__ void ldv<4>(const float* p, float (&x)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
}
template <int V>
__device__ __forceinline__ void stv(float* p, const float (&x)[V]);
template <>
__device__ __forceinline__ void stv<8>(float* p, const float (&x)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(x[0]), "f"(x[1]),
               "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7])
               : "memory");
}
template <>
__device__ __forceinline__ void stv<4>(float* p, const float (&x)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}

// a <- merge(a, b) ([GRA] "Why partial results are allowed to merge";
// [ZQ]: rescale by exp(old_max - new_max)):
//   m = max(ma, mb); alpha = e^{ma-m}, beta = e^{mb-m} (0 for an -inf side)
//   l = alpha la + beta lb;  O~ = alpha O~a + beta O~b
// D / V lanes share a row, V columns each.  The first lane of the row reads
// the four scalars once, computes alpha and beta and writes m and l; the
// others get alpha and beta by a shuffle.  Each lane issues both O~ loads
// before the scalar loads and the arithmetic; at 40 registers a lane, 6
// blocks of 256 stay resident per SM, which keeps enough bytes in flight.
// The loop is warp-uniform (the shuffles need every lane), with rows past the
// end masked.
template <int D, int V>
__global__ void __launch_bounds__(256, 6) merge_kernel(float* __restrict__ ma, float* __restrict__ la,
                                                    float* __restrict__ oa, const float* __restrict__ mb,
                                                    const float* __restrict__ lb, const float* __restrict__ ob,
                                                    long long rows) {
  constexpr int TPR = D / V;
  constexpr int kRowsPerWarp = 32 / TPR;
  constexpr int kUnroll = 1;
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPR;
  const int leader = lane - sub;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long nwarps = (long long)gridDim.x * blockDim.x / 32;
  const long long step = nwarps * kRowsPerWarp;
  for (long long base = warp * kRowsPerWarp; base < rows; base += step * kUnroll) {
    float xa[kUnroll][V], xb[kUnroll][V];
    float sa[kUnroll], sb[kUnroll], sm[kUnroll], sl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long row = base + u * step + lane / TPR;
      if (row < rows) {
        ldv<V>(oa + row * D + sub * V, xa[u]);
        ldv<V>(ob + row * D + sub * V, xb[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long row = base + u * step + lane / TPR;
      sa[u] = sb[u] = sm[u] = sl[u] = 0.0f;
      if (row < rows && sub == 0) {
        const float m_a = ma[row], m_b = mb[row];
        const float m = fmaxf(m_a, m_b);
        sa[u] = (m_a == -INFINITY) ? 0.0f : expf(m_a - m);
        sb[u] = (m_b == -INFINITY) ? 0.0f : expf(m_b - m);
        sm[u] = m;
        sl[u] = sa[u] * la[row] + sb[u] * lb[row];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float alpha = __shfl_sync(0xffffffffu, sa[u], leader);
      const float beta = __shfl_sync(0xffffffffu, sb[u], leader);
      const long long row = base + u * step + lane / TPR;
      if (row < rows) {
        float r[V];
#pragma unroll
        for (int e = 0; e < V; ++e) r[e] = alpha * xa[u][e] + beta * xb[u][e];
        stv<V>(oa + row * D + sub * V, r);
        if (sub == 0) {
          ma[row] = sm[u];
          la[row] = sl[u];
        }
      }
    }
  }
}

// Natural position of local row i of shard r (see ring_layout_t).
__device__ __forceinline__ long long natural_pos(int layout, long long n, int P, long long r, long long i) {
  if (layout == RING_LAYOUT_STRIPED) return i * P + r;
  if (layout == RING_LAYOUT_ZIGZAG) {
    const long long c = n / 2;
    return i < c ? r * c + i : (2 * P - 1 - r) * c + (i - c);
  }
  return r * n + i;
}

// Finalize shard r ([RA-CN] "环是怎样工作的": local_output = finalize(state)):
// out = O~ / l, lse = m + ln l at natural position pos(r, i).
__global__ void finalize_kernel(const float* __restrict__ m, const float* __restrict__ l,
                                const float4* __restrict__ o, float4* __restrict__ out,
                                float* __restrict__ lse, int BH, long long n, int d4, int P, int r,
                                int layout, long long N) {
  const long long rows = (long long)BH * n;
  const long long total = rows * d4;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const long long row = x / d4;
    const int c = (int)(x % d4);
    const long long bh = row / n, i = row % n;
    const long long dst_row = bh * N + natural_pos(layout, n, P, r, i);
    const float lv = l[row];
    const float inv = lv > 0.0f ? 1.0f / lv : 0.0f;
    float4 v = o[x];
    v.x *= inv;
    v.y *= inv;
    v.z *= inv;
    v.w *= inv;
    out[dst_row * d4 + c] = v;
    if (c == 0) lse[dst_row] = lv > 0.0f ? m[row] + logf(lv) : -INFINITY;
  }
}

// Pack natural-order K and V into the shard-major rotation buffer:
// buf[r][bh][k][:] = src[bh][pos(r, k)][:].  A row is u16 16-byte chunks; a
// 256-thread block copies kPackRows consecutive rows k of one (shard, head)
// of K or V, a chunk per thread and pass, all its loads issued before its
// stores.  Grid (ceil(n / kPackRows) * BH, P, 2): the (head, row block) pair,
// the shard, K or V; the index arithmetic is per block, not per chunk.
constexpr int kPackRows = 64;
constexpr int kPackThreads = 256;
__global__ void __launch_bounds__(kPackThreads) pack_kv_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                               uint4* __restrict__ kb, uint4* __restrict__ vb, int BH,
                                                               long long n, int u16, int P, int layout) {
  const uint4* src = blockIdx.z == 0 ? k : v;
  uint4* dst = blockIdx.z == 0 ? kb : vb;
  const int nblk = (int)((n + kPackRows - 1) / kPackRows);
  const int bh = (int)(blockIdx.x / nblk);
  const long long k0 = (long long)(blockIdx.x % nblk) * kPackRows;
  const int r = blockIdx.y;
  const long long N = n * P;
  const int per_pass = kPackThreads / u16;  // rows per pass: 16 (d = 128) or 32 (d = 64)
  const int passes = kPackRows / per_pass;  // 4 or 2
  const int c = threadIdx.x % u16;
  const int kr = threadIdx.x / u16;
  const uint4* s_head = src + (long long)bh * N * u16 + c;
  uint4* d_rows = dst + ((long long)r * BH + bh) * n * u16 + c;
  uint4 buf[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const long long kk = k0 + p * per_pass + kr;
    if (p < passes && kk < n) buf[p] = s_head[natural_pos(layout, n, P, r, kk) * u16];
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const long long kk = k0 + p * per_pass + kr;
    if (p < passes && kk < n) d_rows[kk * u16] = buf[p];
  }
}

// Split-K/V decode: merge the P shard states of every row and finalize
// ([RA-CN] the query is sent to every K/V shard, each returns a local
// state, and the states are merged exactly; [GRA] "Why partial results are
// allowed to merge"): m = max_s m_s, each side scaled by e^{m_s - m} (0 for
// an empty side), out = O~/l, lse = m + ln l.  One warp per row: the lanes
// first find the row max over the states in parallel, then each lane holds
// d/32 columns and folds the states in groups of kGroup, whose loads are
// all issued before the arithmetic (the states of one row are independent
// reads; one at a time they would cost a memory latency each).  States are
// [P][rows] and [P][rows][d].
template <int D>
__global__ void merge_shards_kernel(const float* __restrict__ m, const float* __restrict__ l,
                                    const float* __restrict__ o, float* __restrict__ out,
                                    float* __restrict__ lse, long long rows, int P) {
  constexpr int kGroup = 16;
  constexpr int per = D / 32;  // 2 or 4 columns per lane
  constexpr int d = D;
  // Launched as a programmatic dependent of the kernel that wrote the
  // states: wait until that grid has completed and its writes are visible
  // (returns at once when launched without the dependency).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long row = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32; row < rows; row += warps) {
    float mx = -INFINITY;
    for (int s = lane; s < P; s += 32) mx = fmaxf(mx, m[(long long)s * rows + row]);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
    float lsum = 0.0f;
    float acc[per];
#pragma unroll
    for (int c = 0; c < per; ++c) acc[c] = 0.0f;
    if (mx != -INFINITY) {
      for (int s0 = 0; s0 < P; s0 += kGroup) {
        float ms[kGroup], ls[kGroup], ov[kGroup][per];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const int s = s0 + u;
          ms[u] = -INFINITY;
          ls[u] = 0.0f;
#pragma unroll
          for (int c = 0; c < per; ++c) ov[u][c] = 0.0f;
          if (s < P) {
            ms[u] = m[(long long)s * rows + row];
            ls[u] = l[(long long)s * rows + row];
            const float* src = o + ((long long)s * rows + row) * d + lane * per;
#pragma unroll
            for (int c = 0; c < per; ++c) ov[u][c] = src[c];
          }
        }
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const float w = ms[u] == -INFINITY ? 0.0f : expf(ms[u] - mx);
          lsum += w * ls[u];
#pragma unroll
          for (int c = 0; c < per; ++c) acc[c] += w * ov[u][c];
        }
      }
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    float* dst = out + row * d + lane * per;
#pragma unroll
    for (int c = 0; c < per; ++c) dst[c] = acc[c] * inv;
    if (lane == 0) lse[row] = lsum > 0.0f ? mx + logf(lsum) : -INFINITY;
  }
}

}  // namespace

int launch_merge_shards(const float* m, const float* l, const float* o, float* out, float* lse, long long rows,
                        int d, int P, void* stream) {
  if (rows <= 0) return 0;
  const long long blocks = (rows + 7) / 8;  // 8 warps a block
  const int grid = (int)(blocks < 65535 * 32 ? blocks : 65535 * 32);
  // programmatic dependent launch: the merge's blocks are scheduled as the
  // previous kernel's blocks exit and wait in griddepcontrol.wait, so the
  // launch latency overlaps the previous kernel's last wave
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = d == 64 ? cudaLaunchKernelEx(&cfg, merge_shards_kernel<64>, m, l, o, out, lse, rows, P)
                          : cudaLaunchKernelEx(&cfg, merge_shards_kernel<128>, m, l, o, out, lse, rows, P);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaGetLastError();
}

int launch_state_init(float* m, float* l, float* o, long long rows, int d, void* stream) {
  const int d4 = d / 4;
  if (rows <= 0) return 0;
  state_init_kernel<<<grid_for(rows * d4, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      m, l, reinterpret_cast<float4*>(o), rows, d4);
  return (int)cudaGetLastError();
}

int launch_merge(float* ma, float* la, float* oa, const float* mb, const float* lb, const float* ob,
                 long long rows, int d, void* stream) {
  if (rows <= 0) return 0;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // 256-bit accesses when both O~ arrays are 32-byte aligned (rows are d
  // floats, a multiple of 8), else 128-bit ones
  const bool wide = reinterpret_cast<uintptr_t>(oa) % 32 == 0 && reinterpret_cast<uintptr_t>(ob) % 32 == 0;
  const long long lanes = rows * (d / (wide ? 8 : 4));
  const int grid = grid_for(lanes, 256);
  if (d == 64) {
    if (wide) merge_kernel<64, 8><<<grid, 256, 0, s>>>(ma, la, oa, mb, lb, ob, rows);
    else merge_kernel<64, 4><<<grid, 256, 0, s>>>(ma, la, oa, mb, lb, ob, rows);
  } else {
    if (wide) merge_kernel<128, 8><<<grid, 256, 0, s>>>(ma, la, oa, mb, lb, ob, rows);
    else merge_kernel<128, 4><<<grid, 256, 0, s>>>(ma, la, oa, mb, lb, ob, rows);
  }
  return (int)cudaGetLastError();
}

int launch_finalize(const float* m, const float* l, const float* o, float* out, float* lse, int BH, long long n,
                    int d, int P, int r, int layout, long long N, void* stream) {
  const int d4 = d / 4;
  const long long rows = (long long)BH * n;
  if (rows <= 0) return 0;
  finalize_kernel<<<grid_for(rows * d4, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      m, l, reinterpret_cast<const float4*>(o), reinterpret_cast<float4*>(out), lse, BH, n, d4, P, r, layout, N);
  return (int)cudaGetLastError();
}

int launch_pack_kv(const void* k, const void* v, void* kbuf, void* vbuf, int BH, long long n, int d, int P,
                   int layout, void* stream) {
  const int u16 = d * 2 / 16;  // 8 or 16: kPackThreads is a multiple, kPackRows * u16 of kPackThreads
  if ((long long)P * BH * n <= 0) return 0;
  const long long blocks = (n + kPackRows - 1) / kPackRows * BH;
  if (blocks > 0x7fffffffLL || P > 65535) return (int)cudaErrorInvalidValue;
  dim3 grid((unsigned)blocks, (unsigned)P, 2);
  pack_kv_kernel<<<grid, kPackThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(kbuf),
      static_cast<uint4*>(vbuf), BH, n, u16, P, layout);
  return (int)cudaGetLastError();
}

}  // namespace ringattn
