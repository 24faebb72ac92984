// Device helpers shared by the kernels: 3D RoPE pair rotation, dtype loads
// and stores, error recording.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "la_internal.h"

namespace la {

__device__ __forceinline__ void record_error(DevError* e, int code, int kernel, int d0, int d1) {
  if (atomicCAS(&e->code, 0, code) == 0) {
    e->kernel = kernel;
    e->detail0 = d0;
    e->detail1 = d1;
  }
}

// 3D RoPE ("SoulX-LiveAct" 技术内核 names RoPE positions; the (t, h, w)
// split and interleaved pairing are the standard 3D RoPE reading): dims are
// [t | h | w]; the pair (2i, 2i+1) of an axis part turns by pos * freq_i.
// Returns (cos, sin) of the pair that starts at head dim `d` (even) for the
// position (pt, ph, pw).
__device__ __forceinline__ float2 rope_cs(const RopeDims& r, int d, int pt, int ph, int pw) {
  if (d < r.dt) return r.tab_t[pt * (r.dt >> 1) + (d >> 1)];
  d -= r.dt;
  if (d < r.dh) return r.tab_h[ph * (r.dh >> 1) + (d >> 1)];
  d -= r.dh;
  return r.tab_w[pw * (r.dw >> 1) + (d >> 1)];
}

// Single-rounding rotation (no contraction), so the stored fp32 value is
// reproducible bit for bit: x0' = x0 c - x1 s, x1' = x0 s + x1 c.
__device__ __forceinline__ float2 rot_exact(float x0, float x1, float2 cs) {
  float a = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
  float b = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
  return make_float2(a, b);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// Two fp32 -> bf16 (round to nearest even) in one instruction; lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// e4m3 with round-to-nearest-even and saturation to +-448 (cvt.rn.satfinite).
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  __nv_fp8_storage_t s = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  return (uint8_t)s;
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(n, f.m) + n) >> f.l;
}

// Token index (raster order) -> (frame, row, column).
__device__ __forceinline__ void token_pos(const RopeDims& r, int t, int& f, int& h, int& w) {
  f = (int)fdiv((uint32_t)t, r.div_hw);
  const int rem = t - f * (int)r.div_hw.d;
  h = (int)fdiv((uint32_t)rem, r.div_w);
  w = rem - h * r.GW;
}

}  // namespace la
