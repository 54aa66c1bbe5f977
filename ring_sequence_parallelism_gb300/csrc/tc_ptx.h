// tc_ptx.h -- inline-PTX wrappers for sm_103a shared by the kernels of this
// library: mbarriers with bounded waits, TMA tile loads and stores, tcgen05
// MMA issue (fused K loops), TMEM loads and stores, packed fp32 arithmetic.
// Bounded waits take any argument struct with `wait_limit_ns` and `err`
// (device error words [0] flags, [1] site).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "tmem_regs.h"

namespace ringattn {
namespace {

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
// mbar_poll is expanded at its call site; mbar_wait is the same loop as an
// out-of-line call.  A call site with many live registers pays for saving
// them around the call (the backward's row threads, inlined: 1030 -> 1142
// TFLOP/s); the forward kernel keeps the call (no gain from inlining there).
template <class Args>
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const Args& a, int site) {
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

template <class Args>
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       const Args& a, int site) {
  return mbar_poll(bar, parity, abort_flag, a, site);
}

// Wait used only while draining: bounded, records nothing.
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
template <class Args>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const Args& a, int site) {
  const bool ok = mbar_wait(bar, parity, abort_flag, a, site);
  return __all_sync(0xffffffffu, ok);
}

// warp_wait with the poll expanded at the call site
template <class Args>
__device__ __forceinline__ bool warp_poll(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const Args& a, int site) {
  const bool ok = mbar_poll(bar, parity, abort_flag, a, site);
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

// Global -> shared bulk copy (no tensor map): both addresses 16-byte
// aligned, bytes a multiple of 16; completes on the mbarrier's tx count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Shared -> global tile store through the same kind of map (bulk group).
__device__ __forceinline__ void tma_store_4d(const void* map, uint32_t src, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// Waits until every bulk store this thread issued has read its shared-memory
// source (the writes themselves are complete when the grid is).
__device__ __forceinline__ void bulk_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
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

// Fused MMA issue.  One asm block issues a whole K loop from the elected lane
// of a converged warp; the descriptors keep their high words and advance the
// 14-bit start-address field of the low word (16-byte units) per K step.
// Issuing MMAs one asm statement at a time, with the descriptor arithmetic
// left to the compiler, measured about three times slower per instruction
// than the tensor core's own rate on this part.
//
// S (+)= Q K^T, both operands K-major with the 128-byte swizzle: K steps of
// 16 elements are +32 bytes within a 64-column sub-tile and +16 KB
// (kTileM/kTileN rows x 128 B) to the next sub-tile.
template <int D>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc);
template <>
__device__ __forceinline__ void mma_qk<128>(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 al, bl;\n\t.reg .b64 ad, bd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 0;\n\t"
      "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 1024;\n\tadd.u32 bl, %3, 1024;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 1026;\n\tadd.u32 bl, %3, 1026;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 1028;\n\tadd.u32 bl, %3, 1028;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 1030;\n\tadd.u32 bl, %3, 1030;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "}"
      ::"r"(d_tmem), "r"((uint32_t)a_desc), "r"((uint32_t)(a_desc >> 32)), "r"((uint32_t)b_desc),
      "r"((uint32_t)(b_desc >> 32)), "r"(idesc)
      : "memory");
}
template <>
__device__ __forceinline__ void mma_qk<64>(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 al, bl;\n\t.reg .b64 ad, bd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 0;\n\t"
      "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\tmov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, 1;\n\t"
      "}"
      ::"r"(d_tmem), "r"((uint32_t)a_desc), "r"((uint32_t)(a_desc >> 32)), "r"((uint32_t)b_desc),
      "r"((uint32_t)(b_desc >> 32)), "r"(idesc)
      : "memory");
}

// O~ (+)= P V: P from TMEM (8 columns of bf16 pairs per K step of 16 keys),
// V MN-major with the 128-byte swizzle (+2 KB = 16 key rows per K step).
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 at, bl;\n\t.reg .b64 bd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %5, p;\n\t"
      "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "add.u32 at, %1, 16;\n\tadd.u32 bl, %2, 256;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "add.u32 at, %1, 24;\n\tadd.u32 bl, %2, 384;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "add.u32 at, %1, 32;\n\tadd.u32 bl, %2, 512;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "add.u32 at, %1, 40;\n\tadd.u32 bl, %2, 640;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "add.u32 at, %1, 48;\n\tadd.u32 bl, %2, 768;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "add.u32 at, %1, 56;\n\tadd.u32 bl, %2, 896;\n\tmov.b64 bd, {bl, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %5, 1;\n\t"
      "}"
      ::"r"(d_tmem), "r"(p_tmem), "r"((uint32_t)b_desc), "r"((uint32_t)(b_desc >> 32)), "r"(0u), "r"(idesc),
      "r"(accumulate)
      : "memory");
}

// tcgen05.commit from the elected lane (the lane that issued the MMAs).
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// TMEM -> registers: 32 / 128 consecutive columns of this thread's lane.
// The wait is in the same asm block, so no consumer runs before it.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&x)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " RA_LD_REGS32 ", [%32];\n\t"
               "tcgen05.wait::ld.sync.aligned;"
               : RA_OUT32(x)
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_load128(uint32_t taddr, uint32_t (&x)[128]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x128.b32 " RA_LD_REGS128 ", [%128];\n\t"
               "tcgen05.wait::ld.sync.aligned;"
               : RA_OUT128(x)
               : "r"(taddr)
               : "memory");
}


__device__ __forceinline__ void tmem_store64(uint32_t taddr, const uint32_t (&x)[64]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], " RA_ST_REGS64 ";" ::"r"(taddr), RA_IN64(x)
               : "memory");
}

__device__ __forceinline__ void tmem_load64(uint32_t taddr, uint32_t (&x)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 " RA_LD_REGS64 ", [%64];\n\t"
               "tcgen05.wait::ld.sync.aligned;"
               : RA_OUT64(x)
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_store128(uint32_t taddr, const uint32_t (&x)[128]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x128.b32 [%0], " RA_ST_REGS128 ";" ::"r"(taddr), RA_IN128(x)
               : "memory");
}

__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&x)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], " RA_ST_REGS32 ";" ::"r"(taddr), RA_IN32(x)
               : "memory");
}

__device__ __forceinline__ void tmem_store16(uint32_t taddr, const uint32_t (&x)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]), "r"(x[9]),
      "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15])
      : "memory");
}

__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic: one instruction, two lanes of work).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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

// 256-bit global accesses (8 fp32): one full 32-byte sector per lane.
__device__ __forceinline__ void ld_global_v8(const float* p, uint32_t* x) {
  asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7])
               : "l"(p));
}
__device__ __forceinline__ void st_global_v8(float* p, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]),
               "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace
}  // namespace ringattn
