// Device helpers for the sm_103a kernels: shared-memory barriers, 1-D bulk
// copies (the TMA engine's untiled form), bounded waits, fp16 arithmetic.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

constexpr unsigned kFullMask = 0xffffffffu;
// A wait on the library's own copies gives up after this long (ns) and
// reports PA_ERRBIT_TIMEOUT instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- programmatic dependent launch --------------------------------------
// Every library kernel is launched with programmatic stream serialisation:
// it may start while the previous kernel in the stream is finishing, does
// only CTA-local set-up, and waits here before touching global memory that
// earlier stream work may produce or consume.  Without the launch attribute
// both instructions are no-ops.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream start its own set-up early (it still
// waits for this grid to finish before touching memory).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier (shared::cta) ---------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// kWaitLimitNs.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// ---- 1-D bulk copy global -> shared, completing on an mbarrier ----------
// Both addresses 16-byte aligned, bytes a multiple of 16.

__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_smem),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority policy from createpolicy (streamed data).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst_smem, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Predicated forms for warp-uniform code: every lane executes them with the
// same operands and only the lane with `leader` set performs the operation.
__device__ __forceinline__ void mbar_arrive_expect_tx_if(bool leader, uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n"
      "  .reg .pred e;\n"
      "  setp.ne.b32 e, %2, 0;\n"
      "  @e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
      "}\n" ::"r"(bar),
      "r"(bytes), "r"(leader ? 1u : 0u)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_if(bool leader, uint32_t bar) {
  asm volatile(
      "{\n"
      "  .reg .pred e;\n"
      "  setp.ne.b32 e, %1, 0;\n"
      "  @e mbarrier.arrive.shared::cta.b64 _, [%0];\n"
      "}\n" ::"r"(bar),
      "r"(leader ? 1u : 0u)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint_if(bool leader, uint32_t dst_smem, const void* src,
                                                 uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n"
      "  .reg .pred e;\n"
      "  setp.ne.b32 e, %5, 0;\n"
      "  @e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;\n"
      "}\n" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy), "r"(leader ? 1u : 0u)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- asynchronous 4-byte global -> shared copies (block-table prefetch) --

__device__ __forceinline__ void cp_async_4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- arithmetic ----------------------------------------------------------

// 2^x (the SFU's approximate exponential; relative error about 2^-22).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (2^a, 2^b) as a packed fp16 pair (low half = 2^a): both exponentials in
// fp32 (ex2.approx.ftz.f32), then rounded once to fp16 (a weight's relative
// error is then that rounding, at most 2^-11).
__device__ __forceinline__ uint32_t exp2_f32_to_f16x2(float a, float b) {
  uint32_t r;
  asm("{\n"
      "  .reg .f32 ea, eb;\n"
      "  ex2.approx.ftz.f32 ea, %1;\n"
      "  ex2.approx.ftz.f32 eb, %2;\n"
      "  cvt.rn.f16x2.f32 %0, eb, ea;\n"
      "}\n"
      : "=r"(r)
      : "f"(a), "f"(b));
  return r;
}

// acc + lo(h) + hi(h) for a packed fp16 pair, in fp32 (each add rounded once).
__device__ __forceinline__ float add_f16x2_f32(uint32_t h, float acc) {
  asm("{\n"
      "  .reg .f16 h0, h1, one;\n"
      "  mov.b32 {h0, h1}, %1;\n"
      "  mov.b16 one, 0x3C00;\n"
      "  fma.rn.f32.f16 %0, h0, one, %0;\n"
      "  fma.rn.f32.f16 %0, h1, one, %0;\n"
      "}\n"
      : "+f"(acc)
      : "r"(h));
  return acc;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// acc + a.lo*b.lo + a.hi*b.hi for two packed fp16 pairs, each product added
// with one fp32 rounding (fp16 x fp16 products are exact in fp32).
__device__ __forceinline__ float dot2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{\n"
      "  .reg .f16 a0, a1, b0, b1;\n"
      "  mov.b32 {a0, a1}, %1;\n"
      "  mov.b32 {b0, b1}, %2;\n"
      "  fma.rn.f32.f16 %0, a0, b0, %0;\n"
      "  fma.rn.f32.f16 %0, a1, b1, %0;\n"
      "}\n"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// Dot product of 8 fp16 pairs (one 16-byte vector each), fp32 accumulate,
// dimensions in increasing order.
__device__ __forceinline__ float dot8_f16(const uint4& a, const uint4& b) {
  float acc = 0.f;
  acc = dot2_f16_f32(a.x, b.x, acc);
  acc = dot2_f16_f32(a.y, b.y, acc);
  acc = dot2_f16_f32(a.z, b.z, acc);
  acc = dot2_f16_f32(a.w, b.w, acc);
  return acc;
}

// o0 += p * lo(v), o1 += p * hi(v): fp16 x fp16 products added in fp32 with
// one rounding each (the products are exact in fp32).  p: fp16 bits.
__device__ __forceinline__ void fma2_f16_f32(uint16_t p, uint32_t v, float& o0, float& o1) {
  asm("{\n"
      "  .reg .f16 v0, v1;\n"
      "  mov.b32 {v0, v1}, %2;\n"
      "  fma.rn.f32.f16 %0, %3, v0, %0;\n"
      "  fma.rn.f32.f16 %1, %3, v1, %1;\n"
      "}\n"
      : "+f"(o0), "+f"(o1)
      : "r"(v), "h"(p));
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t u) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = u;
  return __half22float2(h);
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  return *reinterpret_cast<const uint2*>(p);
}

// ---- FP8 E4M3 ------------------------------------------------------------

// Two E4M3 codes (low byte = first element) -> packed fp16 pair (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes16) {
  uint32_t r;
  const unsigned short c = (unsigned short)codes16;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
  return r;
}

// (a0 * b0 + c0, a1 * b1 + c1) as one packed fp32 fused multiply-add
// (sm_100 family): each lane is an IEEE fma rounded to nearest, so the
// result is bit-identical to two fmaf calls in half the instructions.
__device__ __forceinline__ float2 ffma2(float a0, float a1, uint64_t b, uint64_t c) {
  uint64_t a, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  float2 out;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(out.x), "=f"(out.y) : "l"(r));
  return out;
}

// The same value in both halves of a packed fp32 pair.
__device__ __forceinline__ uint64_t f32x2_splat(float v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}

// Eight E4M3 codes (element order in memory) -> 4 packed fp16 pairs.
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(const uint2& c) {
  uint4 r;
  r.x = e4m3x2_to_f16x2(c.x & 0xffffu);
  r.y = e4m3x2_to_f16x2(c.x >> 16);
  r.z = e4m3x2_to_f16x2(c.y & 0xffffu);
  r.w = e4m3x2_to_f16x2(c.y >> 16);
  return r;
}

// Nearest E4M3 codes of two floats (ties to even, saturating to +-448);
// `first` goes to the low byte, matching element order in memory.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float first, float second) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core, TMA, bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 E4M3 codes of 16 fp16 values (the 32 bytes lo, hi): each value is
// divided by the tensor's scale in IEEE binary32 (round to nearest) and the
// quotient rounded to the nearest E4M3 code, saturating to +-448.  The one
// quantisation every FP8 cache write uses.
__device__ __forceinline__ uint4 quantize16(const uint4& lo, const uint4& hi, float scale) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f = half2_bits_to_float2(w[j]);
    c[j] = f32x2_to_e4m3x2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
  }
  return make_uint4(c[0] | c[1] << 16, c[2] | c[3] << 16, c[4] | c[5] << 16, c[6] | c[7] << 16);
}

// 8 E4M3 codes of 8 fp16 values (16 bytes), elementwise as quantize16.
__device__ __forceinline__ uint2 quantize8(const uint4& v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = half2_bits_to_float2(w[j]);
    c[j] = f32x2_to_e4m3x2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
  }
  return make_uint2(c[0] | c[1] << 16, c[2] | c[3] << 16);
}

}  // namespace pa