// pkd_device.cuh -- inline-PTX building blocks for the sm_103a decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pkd_internal.h"

namespace pkd {
namespace dev {

// A pipeline wait that has not completed after this long gives up (status bit 0).  The decode
// kernel's pipeline waits take their limit from the launch (DecodeParams::wait_ns); the waits
// that let copies in flight land before a CTA exits always keep this one.
constexpr unsigned long long kWaitTimeoutNs = kWaitLimitNs;
// Status word bits.  A timeout makes every later launch on the same status word return at
// once (until the host clears it); a page id outside the pool is reported and read as zeros.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBadPage = 2u;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Whether phase `parity` of `bar` has completed, without waiting.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete.  Gives up (returns false) when *abort is
// set by another warp or after limit_ns; every wait in these kernels is bounded.  A limit of
// 0 tests the phase once and gives up at once if it has not completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned long long limit_ns = kWaitTimeoutNs) {
  if (limit_ns == 0) return mbar_test(bar, parity);
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (the consumer warps), id 1..15, that also returns the OR
// of every participant's `pred`: one decision all of them share.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Named barrier over `count` threads (the consumer warps), id 1..15.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tmap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Streaming policy for K/V: each byte is read once per call, so let it leave L2 first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, int c0, int c1, int c2,
                                            int c3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------ tensor-core fragments
// Shared-memory reads of a pipeline stage.  They are not volatile, so the compiler may issue
// them early (ahead of earlier MMAs); callers make the stage address depend on the stage's
// barrier wait (stage_after_wait) so no read moves above it, and every value read feeds an
// MMA, which stays ordered before the stage is released.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(addr));
  return v;
}

// An opaque copy of a stage address taken after the stage's barrier wait: reads addressed
// through it cannot be scheduled before the wait.
__device__ __forceinline__ uint32_t stage_after_wait(uint32_t addr) {
  asm volatile("" : "+r"(addr)::"memory");
  return addr;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Four e4m3 bytes of a word to two half2 (bytes 0,1 -> lo; bytes 2,3 -> hi), exactly: every
// e4m3 value is an fp16 value.  The word's halves are split without arithmetic.
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

template <typename T>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1);

template <>
__device__ __forceinline__ void mma_16816<__half>(float (&c)[4], const uint32_t (&a)[4],
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma_16816<__nv_bfloat16>(float (&c)[4], const uint32_t (&a)[4],
                                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ element conversions
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t v);

template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t v) {
  return __half22float2(*reinterpret_cast<__half2*>(&v));
}

template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
}

// Two e4m3 bytes (low byte first) to a half2 bit pattern, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint16_t v) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  uint32_t out;
  out = static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
  return out;
}

// sin and cos of the RoPE angle t * rate, where rate = hi + lo is a double held as a float
// pair and t an integer position (exact as a float below 2^24).  The product is kept exact
// (t * hi rounded, its rounding error by FMA, plus t * lo), the nearest multiple of 2*pi is
// removed in two parts (Cody and Waite's reduction, 2*pi = 6.28125 + 0.0019353071795864769),
// and only the reduced angle, within about [-pi, pi], goes to the fast sine and cosine.
// Angle error about 1e-6 rad for positions below 2^24.
__device__ __forceinline__ void rope_sincos(float t, float hi, float lo, float& s, float& c) {
  const float p = t * hi;
  const float e = fmaf(t, hi, -p) + t * lo;
  const float k = rintf(p * 0.15915494309189535f);
  float r = fmaf(-k, 6.28125f, p);
  r = fmaf(-k, 0.0019353071795864769f, r);
  __sincosf(r + e, &s, &c);
}

// Rotation of two complex numbers held as fp16 pairs: (x, y) -> (x c - y s, y c + x s) per
// half, where x holds the real parts, y the imaginary parts and (c, s) the two phasors.  Each
// output is one fp16 product and one fused multiply-add (two roundings).
__device__ __forceinline__ void rot_h2(uint32_t& x, uint32_t& y, uint32_t c, uint32_t s) {
  const __half2 X = *reinterpret_cast<const __half2*>(&x), Y = *reinterpret_cast<const __half2*>(&y);
  const __half2 C = *reinterpret_cast<const __half2*>(&c), S = *reinterpret_cast<const __half2*>(&s);
  const __half2 nx = __hfma2(X, C, __hneg2(__hmul2(Y, S)));
  const __half2 ny = __hfma2(Y, C, __hmul2(X, S));
  x = *reinterpret_cast<const uint32_t*>(&nx);
  y = *reinterpret_cast<const uint32_t*>(&ny);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk `c` of row `r` in a tile stored as 128-byte column blocks of
// `rows_per_block` rows each, with the 128-byte TMA swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz_off(int r, int c, int rows_per_block) {
  return static_cast<uint32_t>((c >> 3) * rows_per_block * 128 + r * 128 +
                               (((c & 7) ^ (r & 7)) << 4));
}

}  // namespace dev
}  // namespace pkd
