// W4A16 numerics mode of the routed experts: NVFP4 weights dequantised in
// registers against bf16 activations, on the CUDA cores.
//
// The pages' own kernel choice for the offload backend on its GPUs is a
// weight-only 4-bit kernel (PR #385 "feat(qwen4_exp): tensor parallelism for
// Qwen3.8-Flash-Next (offload backend)", review thread, the kernel-selection
// fix naming the marlin kernel): activations stay 16-bit and only the
// weights are 4-bit.  This mode computes that: for each pair of a routed
// expert, G = g_row * sum_b s_b * sum_16 e2m1(q) * x over the window's gate
// and up rows with x the bf16 hidden state, h = bf16(silu(G_gate) * G_up)
// (the intermediate kept 16-bit, as the shared expert keeps it), and
// Y = g_h * sum_b s_b * sum_16 e2m1(q) * h over the window's down columns.
// Every sum runs in a fixed order; the combine with the shared expert is the
// forward's own.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace ftmoe {

namespace {

constexpr int kWMT = 8;  // pairs staged per pass

__device__ __forceinline__ void e2m1x16(uint2 c, float s, float w[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = __half22float2(e2m1x2_to_half2((c.x >> (8 * i)) & 0xFF));
    const float2 b = __half22float2(e2m1x2_to_half2((c.y >> (8 * i)) & 0xFF));
    w[2 * i] = a.x * s;
    w[2 * i + 1] = a.y * s;
    w[8 + 2 * i] = b.x * s;
    w[8 + 2 * i + 1] = b.y * s;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Dot of 16 dequantised weights with 16 bf16 values at p (16-byte aligned).
__device__ __forceinline__ float dot16_bf16(const float w[16], const uint16_t* p) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint4 b = *reinterpret_cast<const uint4*>(p + 8);
  const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    acc = fmaf(w[2 * i], bf16_lo(v[i]), acc);
    acc = fmaf(w[2 * i + 1], bf16_hi(v[i]), acc);
  }
  return acc;
}

}  // namespace

// Work item = (touched expert, 8 window indices).  Warp w owns window index
// i = 8 * block + w: gate row i and up row i; its lanes split the rows'
// 16-blocks.  The expert's pairs go in passes of up to 8 tokens whose bf16
// rows are staged in shared memory.
__global__ void __launch_bounds__(256) k_w16_gate_up(ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  uint16_t* s_x = reinterpret_cast<uint16_t*>(sm);  // [kWMT][H]
  __shared__ int s_tok[kWMT];
  const RouteArgs& r = a.r;
  const int H = a.H, NB = H / kBlock, HC = H / 2;
  const int I_loc = a.win.I_loc, nblk = (I_loc + 7) / 8;
  const int n_items = r.n_touched[0] * nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = r.touched[item / nblk];
    const int i = (item % nblk) * 8 + warp;
    const bool live = i < I_loc;
    const uint8_t* rec = a.rec[e];
    const int gr = a.win.row0 + (live ? i : 0), ur = a.win.Iw + gr;
    const uint8_t* gc = rec + a.lay.gu_codes + (int64_t)gr * HC;
    const uint8_t* uc = rec + a.lay.gu_codes + (int64_t)ur * HC;
    const uint8_t* gs = rec + a.lay.gu_scales + (int64_t)gr * NB;
    const uint8_t* us = rec + a.lay.gu_scales + (int64_t)ur * NB;
    const float* glob = reinterpret_cast<const float*>(rec + a.lay.gu_global);
    const float gg = glob[gr], gu = glob[ur];
    const int s0 = r.offsets[e], s1 = r.offsets[e + 1];
    for (int c0 = s0; c0 < s1; c0 += kWMT) {
      const int mc = min(kWMT, s1 - c0);
      __syncthreads();
      if (threadIdx.x < mc) s_tok[threadIdx.x] = r.perm[c0 + threadIdx.x] / a.top_k;
      __syncthreads();
      for (int q = threadIdx.x; q < mc * (H / 8); q += blockDim.x) {
        const int m = q / (H / 8), c = q % (H / 8);
        reinterpret_cast<uint4*>(s_x)[m * (H / 8) + c] =
            __ldg(reinterpret_cast<const uint4*>(r.x + (int64_t)s_tok[m] * H) + c);
      }
      __syncthreads();
      float ag[kWMT], au[kWMT];
#pragma unroll
      for (int m = 0; m < kWMT; ++m) { ag[m] = 0.f; au[m] = 0.f; }
      if (live) {
        for (int b = lane; b < NB; b += 32) {
          float wg[16], wu[16];
          e2m1x16(*reinterpret_cast<const uint2*>(gc + b * 8), e4m3_decode(gs[b]), wg);
          e2m1x16(*reinterpret_cast<const uint2*>(uc + b * 8), e4m3_decode(us[b]), wu);
#pragma unroll
          for (int m = 0; m < kWMT; ++m) {
            if (m < mc) {
              ag[m] += dot16_bf16(wg, s_x + m * H + 16 * b);
              au[m] += dot16_bf16(wu, s_x + m * H + 16 * b);
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kWMT; ++m) {
        const float g = warp_sum(ag[m]) * gg, u = warp_sum(au[m]) * gu;
        if (lane == 0 && live && m < mc) {
          const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * u);
          reinterpret_cast<uint16_t*>(a.hq_codes)[(int64_t)(c0 + m) * I_loc + i] =
              *reinterpret_cast<const uint16_t*>(&hb);
        }
      }
    }
  }
}

// Work item = (touched expert, 32 output rows).  Warp w owns rows 4w..4w+3;
// 8 lanes share a row and split the window's 16-blocks.
// Y[pos][h] = g_h * sum_b s_b * sum_16 e2m1(q) * h_pos for every pair.
__global__ void __launch_bounds__(256) k_w16_down(ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int K = a.win.I_loc, nbk = K / kBlock;
  uint16_t* s_h = reinterpret_cast<uint16_t*>(sm);  // [kWMT][K]
  const RouteArgs& r = a.r;
  const int H = a.H, n_hb = (H + 31) / 32;
  const int n_items = r.n_touched[0] * n_hb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = warp * 4 + (lane >> 3), sub = lane & 7;
  const int col0 = a.win.row0;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = r.touched[item / n_hb];
    const int h = (item % n_hb) * 32 + rr;
    const bool live = h < H;
    const int hh = live ? h : 0;
    const uint8_t* rec = a.rec[e];
    const uint8_t* wc = rec + a.lay.dn_codes + (int64_t)hh * (a.win.Iw / 2) + col0 / 2;
    const uint8_t* ws = rec + a.lay.dn_scales + (int64_t)hh * (a.win.Iw / kBlock) + col0 / kBlock;
    const float gd = reinterpret_cast<const float*>(rec + a.lay.dn_global)[hh];
    const int s0 = r.offsets[e], s1 = r.offsets[e + 1];
    for (int c0 = s0; c0 < s1; c0 += kWMT) {
      const int mc = min(kWMT, s1 - c0);
      __syncthreads();
      const uint16_t* hb = reinterpret_cast<const uint16_t*>(a.hq_codes);
      for (int q = threadIdx.x; q < mc * (K / 8); q += blockDim.x) {
        const int m = q / (K / 8), c = q % (K / 8);
        reinterpret_cast<uint4*>(s_h)[m * (K / 8) + c] =
            *reinterpret_cast<const uint4*>(hb + (int64_t)(c0 + m) * K + 8 * c);
      }
      __syncthreads();
      float acc[kWMT];
#pragma unroll
      for (int m = 0; m < kWMT; ++m) acc[m] = 0.f;
      if (live) {
        for (int b = sub; b < nbk; b += 8) {
          float w[16];
          e2m1x16(*reinterpret_cast<const uint2*>(wc + b * 8), e4m3_decode(ws[b]), w);
#pragma unroll
          for (int m = 0; m < kWMT; ++m)
            if (m < mc) acc[m] += dot16_bf16(w, s_h + m * K + 16 * b);
        }
      }
#pragma unroll
      for (int m = 0; m < kWMT; ++m) {
        float v = acc[m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (sub == 0 && m < mc && live) a.Y[(int64_t)(c0 + m) * H + h] = v * gd;
      }
    }
  }
}

cudaError_t w16_set_smem_limits(int H, int I) {
  cudaError_t e = cudaFuncSetAttribute(k_w16_gate_up, cudaFuncAttributeMaxDynamicSharedMemorySize, kWMT * H * 2);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_w16_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kWMT * I * 2);
}

cudaError_t launch_w16_routed(const ExpertArgs& a, cudaStream_t s) {
  const int grid = a.num_sms * 4;
  FTMOE_PROF_BEGIN("k_w16_gate_up", s);
  k_w16_gate_up<<<grid, 256, (size_t)kWMT * a.H * 2, s>>>(a);
  FTMOE_PROF_END(s);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  FTMOE_PROF_BEGIN("k_w16_down", s);
  k_w16_down<<<grid, 256, (size_t)kWMT * a.win.I_loc * 2, s>>>(a);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

}  // namespace ftmoe
