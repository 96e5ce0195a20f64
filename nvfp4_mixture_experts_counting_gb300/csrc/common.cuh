// Device helpers shared by the ftmoe kernels: NVFP4 encode/decode through the
// sm_100-family conversion instructions, bf16 conversions, warp reductions and
// the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace ftmoe {

constexpr int kBlock = 16;           // NVFP4 scale block (elements)
constexpr float kE2M1Max = 6.0f;
constexpr float kWeightGlobalDiv = 2688.0f;  // 448 * 6

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- NVFP4 codes

// E4M3 ("fn") byte of a non-negative fp32 value: round to nearest even,
// saturating at 448 (cvt .satfinite).
__device__ __forceinline__ uint8_t e4m3_encode(float u) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(u));
  return (uint8_t)(r & 0xFF);
}

// fp32 value of an E4M3 byte (exact).
__device__ __forceinline__ float e4m3_decode(uint8_t c) {
  uint32_t r;
  uint16_t in = c;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  __half2 h = *reinterpret_cast<__half2*>(&r);
  return __low2float(h);
}

// Two E2M1 codes (low nibble = a, high nibble = b) of fp32 values, round to
// nearest even, saturating at 6; a zero magnitude gets sign bit 0.
__device__ __forceinline__ uint8_t e2m1x2_encode(float a, float b) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(b), "f"(a));
  uint32_t lo = r & 0xF, hi = (r >> 4) & 0xF;
  if ((lo & 7) == 0) lo = 0;
  if ((hi & 7) == 0) hi = 0;
  return (uint8_t)(lo | (hi << 4));
}

// Exact half2 of a byte holding two E2M1 codes (x = low nibble).
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
  uint32_t r;
  uint16_t in = (uint16_t)(byte & 0xFF);
  asm("{ .reg .b8 t; cvt.u8.u16 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "h"(in));
  return *reinterpret_cast<__half2*>(&r);
}

// Quantise one 16-element block of fp32 values with row global g (1.0 for
// activations).  Writes 8 code bytes and returns the scale byte.
// Steps: t = fp32(amax/6); u = fp32(t/g); s = E4M3(u); d = fp32(dec(s)*g);
// code_i = E2M1(fp32(v_i/d)); g == 0, s == 0 or d == 0 give zero codes.
__device__ __forceinline__ uint8_t quantize_block16(const float v[16], float g, uint8_t codes[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  uint8_t s = 0;
  if (g != 0.f) {
    float t = __fdiv_rn(amax, kE2M1Max);
    float u = __fdiv_rn(t, g);
    s = e4m3_encode(u);
  }
  float d = __fmul_rn(e4m3_decode(s), g);
  if (s == 0 || d == 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0;
    return 0;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) codes[i] = e2m1x2_encode(__fdiv_rn(v[2 * i], d), __fdiv_rn(v[2 * i + 1], d));
  return s;
}

// ---------------------------------------------------------------- misc

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// 32 bytes of read-only global data at a 32-byte-aligned address, one
// 256-bit load.
__device__ __forceinline__ void ldg_nc_32B(const void* p, uint32_t* r) {
  asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "l"(p));
}

// ---------------------------------------------------------------- double-fp32

// A number hi + lo held as two fp32 values.  Built from error-free
// transformations (two-sum of Knuth, FMA two-product), so a router logit is
// carried to about twice fp32's precision on the fp32 pipes.  The explicit
// _rn intrinsics keep the compiler from fusing the steps.
struct df32 {
  float hi, lo;
};

__device__ __forceinline__ df32 df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float z = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
  return {s, e};
}

__device__ __forceinline__ df32 df_add(df32 a, df32 b) {
  const df32 s = df_two_sum(a.hi, b.hi);
  return df_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

// Strict order of logits: larger value first (hi, then lo), then lower index.
__device__ __forceinline__ bool df_before(df32 a, int ea, df32 b, int eb) {
  if (a.hi != b.hi) return a.hi > b.hi;
  if (a.lo != b.lo) return a.lo > b.lo;
  return ea < eb;
}

// Compensated router logit of one token (bf16 row x) and one expert (fp32 row
// w), + bias, by a warp: every product is split exactly (x*w = p + pe) and
// accumulated with two-sum, lane sums are combined in double-fp32.  The
// absolute error is a few units of 2^-48 times sum |x*w|.
__device__ __forceinline__ df32 logit_df32(const uint16_t* x, const float* w, int H, float bias, int lane) {
  float s = 0.f, c = 0.f;
  const uint2* x4 = reinterpret_cast<const uint2*>(x);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const int n4 = H / 4;
  // eight chunks' loads in flight before their (in-order) accumulation
  for (int i0 = lane; i0 < n4; i0 += 32 * 8) {
    uint2 xv[8];
    float4 wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u;
      if (i < n4) {
        xv[u] = __ldg(x4 + i);
        wv[u] = __ldg(w4 + i);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (i0 + 32 * u < n4) {
        const float xs[4] = {__uint_as_float(xv[u].x << 16), __uint_as_float(xv[u].x & 0xffff0000u),
                             __uint_as_float(xv[u].y << 16), __uint_as_float(xv[u].y & 0xffff0000u)};
        const float ws[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float p = __fmul_rn(xs[k], ws[k]);
          const float pe = __fmaf_rn(xs[k], ws[k], -p);
          const df32 t = df_two_sum(s, p);
          s = t.hi;
          c = __fadd_rn(c, __fadd_rn(t.lo, pe));
        }
      }
    }
  }
  df32 v = df_two_sum(s, c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const df32 u = {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    v = df_add(v, u);
  }
  return df_add(v, {bias, 0.f});
}

}  // namespace ftmoe
