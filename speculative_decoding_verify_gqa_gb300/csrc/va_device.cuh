// Small device helpers (inline PTX) used by the kernels of libverify_attn.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace va {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared async copy; bytes < 16 zero-fills the rest (0 reads nothing).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: block until the grids this one depends on
// have completed and their writes are visible (a no-op when the kernel was
// launched without the programmatic-serialization attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
// Allow the next kernel in the stream (if launched with programmatic
// serialization) to be scheduled now; it still waits for our completion
// before touching memory.
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Two fp32 lanes in one 64-bit register (low word = first) and the packed
// fp32x2 FMA / add of sm_100+: one instruction for two elements.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 2^x via the SFU instruction (denormal results flushed to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two fp8-e4m3 codes (low byte first) -> two bf16 (exact: every e4m3 value is
// a bf16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t codes) {
  __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  __half2 hv = *reinterpret_cast<__half2*>(&hr);
  float2 f = __half22float2(hv);
  return pack_bf16x2(f.x, f.y);
}

// Two fp8-e4m3 codes (low byte first) -> two f16 (exact), one instruction.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// Four floats -> four fp8-e4m3 codes (first in the low byte), round to
// nearest even, finite overflow and infinities saturated to +-448.
__device__ __forceinline__ uint32_t e4m3x4_rn_satfinite(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Both halves of a packed bf16 / f16 pair times a (a power of two in the
// softmax, so exact down to the formats' subnormal range).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float a) {
  return pack_bf16x2(__uint_as_float(v << 16) * a, __uint_as_float(v & 0xffff0000u) * a);
}
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t v, float a) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  const float2 f = __half22float2(h);
  return pack_f16x2(f.x * a, f.y * a);
}

// bf16x2 -> f16x2 (exact for values inside f16's normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
  return pack_f16x2(lo, hi);
}

// cos and sin of one RoPE angle, position * (hi + lo), where hi + lo is a
// frequency held as a float pair.  The product keeps ~46 bits (its rounding
// error recovered exactly by an FMA) and is reduced modulo 2 pi by the
// Cody-Waite method (Cody and Waite, "Software Manual for the Elementary
// Functions", 1980: 2 pi split into a float head and tail, each product
// with the multiple k taken exactly inside an FMA) before sincosf sees it,
// so for positions below 2^24 the reduced angle is good to ~1e-7 rad where a
// plain float product would be off by up to position * 2^-24 (4e-3 rad at
// position 32768).
__device__ __forceinline__ void rope_cos_sin(int pos, float hi, float lo, float* c, float* s) {
  constexpr float kTwoPiHi = 6.2831854820251465f;      // float nearest to 2 pi
  constexpr float kTwoPiLo = -1.7484555314695172e-07f;  // 2 pi - kTwoPiHi
  constexpr float kInvTwoPi = 0.15915493667125702f;
  const float p = (float)pos;                           // exact below 2^24
  const float a_hi = p * hi;
  const float a_err = fmaf(p, hi, -a_hi);               // p * hi - a_hi, exactly
  const float a_lo = fmaf(p, lo, a_err);
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r);
  r += a_lo;
  // |r| <= pi + a few ulps: the hardware approximations are good to ~4e-7
  // absolute there, far below the 2^-9 relative rounding of the bf16 result
  __sincosf(r, s, c);
}

// Byte offset of 16-byte chunk `ch` of row `r` in a row-major shared tile of
// `row_bytes` per row, XOR-swizzled so that 8 consecutive rows' same chunk
// fall in 8 different bank groups (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t swz(int r, int ch, int row_bytes) {
  return static_cast<uint32_t>(r * row_bytes + ((ch ^ (r & 7)) << 4));
}

}  // namespace va
