// Expert kernels on CUDA cores (any T): shared-expert gate_up + SwiGLU,
// routed gate_up + SwiGLU + NVFP4 quantisation of the intermediate, routed
// down, shared down, and the deterministic weighted combine.
//
// Pages: Issue #62 "Offloaded MoE ignores tensor parallelism ...", "What it
// touches" (gate_up [2I, H] with gate rows [0, I) and up rows [I, 2I); down
// [H, I] sliced by columns); PR #385 "feat(qwen4_exp): tensor parallelism for
// Qwen3.8-Flash-Next (offload backend)", "What this adds" (routed +
// sigmoid(gate) * shared before one reduce) and "Correctness" (no value
// atomics: every sum here runs in a fixed order).
#include "common.cuh"
#include "tma.cuh"
#include "kernels.h"

namespace ftmoe {

constexpr int kMT = 8;  // tokens (pairs) staged per pass

// ------------------------------------------------------------------ NVFP4 block dot

// Sum over one 16-block of q_w * q_a, exact: each half2 lane sums 8 products
// of E2M1 values (multiples of 1/4, |sum| <= 288), which half precision holds
// exactly, and the two lanes add exactly in fp32.
__device__ __forceinline__ float block_dot(const __half2 w[8], const __half2* a) {
  __half2 acc = __hmul2(w[0], a[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) acc = __hfma2(w[i], a[i], acc);
  return __low2float(acc) + __high2float(acc);
}

__device__ __forceinline__ void decode_codes8(uint2 c, __half2 w[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i] = e2m1x2_to_half2((c.x >> (8 * i)) & 0xFF);
    w[4 + i] = e2m1x2_to_half2((c.y >> (8 * i)) & 0xFF);
  }
}

// Stage the NVFP4 activations of up to kMT rows into shared memory as exact
// half2 code values plus fp32 scales.  rows[m] is the source row of slot m.
__device__ void stage_act(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                          int K, const int* rows, int mc, __half2* s_codes, float* s_scales) {
  const int nb = K / kBlock;
  for (int i = threadIdx.x; i < mc * (K / 2); i += blockDim.x) {
    const int m = i / (K / 2), c = i % (K / 2);
    s_codes[m * (K / 2) + c] = e2m1x2_to_half2(codes[(int64_t)rows[m] * (K / 2) + c]);
  }
  for (int i = threadIdx.x; i < mc * nb; i += blockDim.x) {
    const int m = i / nb, b = i % nb;
    s_scales[m * nb + b] = e4m3_decode(scales[(int64_t)rows[m] * nb + b]);
  }
}

// ------------------------------------------------------------------ routed gate_up

// Work item = (touched expert, 16-wide block ib of the window): 16 gate rows
// and the matching 16 up rows.  Warp w owns rows 4w..4w+3 (0..15 gate,
// 16..31 up); 8 lanes share a row and split its 16-blocks.  For every pair of
// the expert: G = g_row * sum_b s_w * s_a * dot_b, h = silu(G_gate) * G_up,
// then h is NVFP4-quantised (global 1.0) into the pair's sorted row.
__global__ void __launch_bounds__(256) k_gate_up(ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int H = a.H, nbh = H / kBlock;
  __half2* s_codes = reinterpret_cast<__half2*>(sm);              // [kMT][H/2]
  float* s_scales = reinterpret_cast<float*>(s_codes + kMT * (H / 2));  // [kMT][nbh]
  float* s_G = s_scales + kMT * nbh;                               // [kMT][32]
  __shared__ int s_rows[kMT];
  __shared__ int s_pos[kMT];
  const RouteArgs& r = a.r;
  const int n_ib = a.win.I_loc / kBlock;
  const int n_items = r.n_touched[0] * n_ib;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = warp * 4 + (lane >> 3);  // 0..31
  const int sub = lane & 7;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = r.touched[item / n_ib];
    const int ib = item % n_ib;
    const uint8_t* rec = a.rec[e];
    const int i_local = a.win.row0 + ib * kBlock + (rr & 15);
    const int brow = (rr < 16) ? i_local : a.win.Iw + i_local;  // row inside the record's gate_up
    const uint8_t* wc = rec + a.lay.gu_codes + (int64_t)brow * (H / 2);
    const uint8_t* ws = rec + a.lay.gu_scales + (int64_t)brow * nbh;
    const float gw = reinterpret_cast<const float*>(rec + a.lay.gu_global)[brow];
    const int s0 = r.offsets[e], s1 = r.offsets[e + 1];
    for (int c0 = s0; c0 < s1; c0 += kMT) {
      const int mc = min(kMT, s1 - c0);
      __syncthreads();
      if (threadIdx.x < mc) {
        const int p = r.perm[c0 + threadIdx.x];
        s_rows[threadIdx.x] = p / a.top_k;
        s_pos[threadIdx.x] = c0 + threadIdx.x;
      }
      __syncthreads();
      stage_act(r.xq_codes, r.xq_scales, H, s_rows, mc, s_codes, s_scales);
      __syncthreads();
      float acc[kMT];
#pragma unroll
      for (int m = 0; m < kMT; ++m) acc[m] = 0.f;
      for (int b = sub; b < nbh; b += 8) {
        const uint2 c = *reinterpret_cast<const uint2*>(wc + b * 8);
        const float sw = e4m3_decode(ws[b]);
        __half2 w[8];
        decode_codes8(c, w);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          if (m < mc) {
            const float d = block_dot(w, s_codes + m * (H / 2) + b * 8);
            acc[m] = fmaf(d, sw * s_scales[m * nbh + b], acc[m]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kMT; ++m) {
        float v = acc[m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (sub == 0 && m < mc) s_G[m * 32 + rr] = v * gw;
      }
      __syncthreads();
      // SwiGLU + quantisation: one thread per staged pair
      if (threadIdx.x < mc) {
        const int m = threadIdx.x;
        float h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) h[i] = silu(s_G[m * 32 + i]) * s_G[m * 32 + 16 + i];
        uint8_t q[8];
        const uint8_t s = quantize_block16(h, 1.0f, q);
        const int64_t pos = s_pos[m];
        uint2 packed;
        packed.x = q[0] | (q[1] << 8) | (q[2] << 16) | ((uint32_t)q[3] << 24);
        packed.y = q[4] | (q[5] << 8) | (q[6] << 16) | ((uint32_t)q[7] << 24);
        *reinterpret_cast<uint2*>(a.hq_codes + pos * (a.win.I_loc / 2) + ib * 8) = packed;
        a.hq_scales[pos * n_ib + ib] = s;
      }
    }
  }
}

// ------------------------------------------------------------------ routed down

// Work item = (touched expert, block of 32 output rows).  Warp w owns rows
// 4w..4w+3; 8 lanes share a row and split its 16-blocks of the window.
// Y[pos][h] = g_h * sum_b s_w * s_h * dot_b for every pair of the expert.
__global__ void __launch_bounds__(256) k_down(ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int K = a.win.I_loc, nbk = K / kBlock;
  __half2* s_codes = reinterpret_cast<__half2*>(sm);               // [kMT][K/2]
  float* s_scales = reinterpret_cast<float*>(s_codes + kMT * (K / 2));  // [kMT][nbk]
  __shared__ int s_rows[kMT];
  const RouteArgs& r = a.r;
  const int H = a.H;
  const int n_hb = (H + 31) / 32;
  const int n_items = r.n_touched[0] * n_hb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = warp * 4 + (lane >> 3);
  const int sub = lane & 7;
  const int col0 = a.win.row0;  // first window column inside the loaded down rows
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = r.touched[item / n_hb];
    const int h = (item % n_hb) * 32 + rr;
    const bool live = h < H;
    const uint8_t* rec = a.rec[e];
    const int hh = live ? h : 0;
    const uint8_t* wc = rec + a.lay.dn_codes + (int64_t)hh * (a.win.Iw / 2) + col0 / 2;
    const uint8_t* ws = rec + a.lay.dn_scales + (int64_t)hh * (a.win.Iw / kBlock) + col0 / kBlock;
    const float gd = reinterpret_cast<const float*>(rec + a.lay.dn_global)[hh];
    const int s0 = r.offsets[e], s1 = r.offsets[e + 1];
    for (int c0 = s0; c0 < s1; c0 += kMT) {
      const int mc = min(kMT, s1 - c0);
      __syncthreads();
      if (threadIdx.x < mc) s_rows[threadIdx.x] = c0 + threadIdx.x;
      __syncthreads();
      stage_act(a.hq_codes, a.hq_scales, K, s_rows, mc, s_codes, s_scales);
      __syncthreads();
      float acc[kMT];
#pragma unroll
      for (int m = 0; m < kMT; ++m) acc[m] = 0.f;
      if (live) {
        for (int b = sub; b < nbk; b += 8) {
          // window columns start at a multiple of 16, i.e. 8-byte aligned
          const uint2 c = *reinterpret_cast<const uint2*>(wc + b * 8);
          const float sw = e4m3_decode(ws[b]);
          __half2 w[8];
          decode_codes8(c, w);
#pragma unroll
          for (int m = 0; m < kMT; ++m) {
            if (m < mc) {
              const float d = block_dot(w, s_codes + m * (K / 2) + b * 8);
              acc[m] = fmaf(d, sw * s_scales[m * nbk + b], acc[m]);
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kMT; ++m) {
        float v = acc[m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (sub == 0 && m < mc && live) a.Y[(int64_t)(c0 + m) * H + h] = v * gd;
      }
    }
  }
}

// ------------------------------------------------------------------ shared expert

// Work item = (8 window indices, token chunk of kMT).  Warp w owns index
// i = 8*item + w: gate row i and up row i (bf16), dotted with x in fp32;
// hs[t][i] = bf16(silu(G_gate) * G_up).
__global__ void __launch_bounds__(256) k_shared_gate_up(ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  const RouteArgs& r = a.r;
  const int H = a.H;
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);  // [kMT][H]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kMT;
  const int tn = min(kMT, a.T - t0);
  {
    const uint4* src = reinterpret_cast<const uint4*>(r.x + (int64_t)t0 * H);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < tn * H / 8; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const int i = blockIdx.x * 8 + warp;
  if (i >= a.s_I_loc) return;
  const uint16_t* g_row = a.sh_gate_up + (int64_t)(a.s_row0 + i) * H;
  const uint16_t* u_row = a.sh_gate_up + (int64_t)(a.s_Iw + a.s_row0 + i) * H;
  float ag[kMT], au[kMT];
#pragma unroll
  for (int m = 0; m < kMT; ++m) { ag[m] = 0.f; au[m] = 0.f; }
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 gv = *reinterpret_cast<const uint4*>(g_row + c * 8);
    const uint4 uv = *reinterpret_cast<const uint4*>(u_row + c * 8);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      if (m < tn) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + m * H + c * 8);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float x0 = __uint_as_float(xw[q] << 16), x1 = __uint_as_float(xw[q] & 0xffff0000u);
          ag[m] = fmaf(x0, __uint_as_float(gw[q] << 16), ag[m]);
          ag[m] = fmaf(x1, __uint_as_float(gw[q] & 0xffff0000u), ag[m]);
          au[m] = fmaf(x0, __uint_as_float(uw[q] << 16), au[m]);
          au[m] = fmaf(x1, __uint_as_float(uw[q] & 0xffff0000u), au[m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kMT; ++m) {
    const float g = warp_sum(ag[m]);
    const float u = warp_sum(au[m]);
    if (lane == 0 && m < tn) {
      const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * u);
      a.hs[(int64_t)(t0 + m) * a.s_I_loc + i] = *reinterpret_cast<const uint16_t*>(&hb);
    }
  }
}

// Work item = (32 output rows, token chunk).  Warp w owns rows 4w..4w+3, 8
// lanes per row split the window columns in 8-element chunks.
// S[t][h] = sum_i W_sd[h][i] * hs[t][i] (fp32).
__global__ void __launch_bounds__(256) k_shared_down(ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int K = a.s_I_loc, H = a.H;
  float* hsf = reinterpret_cast<float*>(sm);  // [kMT][K]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kMT;
  const int tn = min(kMT, a.T - t0);
  for (int i = threadIdx.x; i < tn * K; i += blockDim.x)
    hsf[i] = bf16_bits_to_float(a.hs[(int64_t)t0 * K + i]);
  __syncthreads();
  const int h = blockIdx.x * 32 + warp * 4 + (lane >> 3);
  const int sub = lane & 7;
  if (h >= H) return;  // whole 8-lane groups leave together
  const uint16_t* row = a.sh_down + (int64_t)h * a.s_Iw + a.s_row0;
  float acc[kMT];
#pragma unroll
  for (int m = 0; m < kMT; ++m) acc[m] = 0.f;
  for (int c = sub; c < K / 8; c += 8) {
    // the window starts at a multiple of 16 columns: 16-byte aligned chunks
    const uint4 wv = *reinterpret_cast<const uint4*>(row + c * 8);
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      if (m < tn) {
        const float* hp = hsf + m * K + c * 8;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[m] = fmaf(__uint_as_float(ww[q] << 16), hp[2 * q], acc[m]);
          acc[m] = fmaf(__uint_as_float(ww[q] & 0xffff0000u), hp[2 * q + 1], acc[m]);
        }
      }
    }
  }
  const unsigned gmask = 0xffu << (lane & 24);
#pragma unroll
  for (int m = 0; m < kMT; ++m) {
    float v = acc[m];
    v += __shfl_xor_sync(gmask, v, 1);
    v += __shfl_xor_sync(gmask, v, 2);
    v += __shfl_xor_sync(gmask, v, 4);
    if (sub == 0 && m < tn) a.S[(int64_t)(t0 + m) * H + h] = v;
  }
}

// ------------------------------------------------------------------ combine

// out[t][h] = sum_j w_tj * Y[inv[t*k+j]][h] + sigma_t * S[t][h], in slot
// order, fp32, rounded once (or added to an fp32 out under ACCUMULATE).
__global__ void k_combine(ExpertArgs a) {
  const RouteArgs& r = a.r;
  const int H = a.H, k = a.top_k;
  const int64_t n = (int64_t)a.T * H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H), h = (int)(i % H);
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int64_t yt = (((int64_t)t * (H / 128) + h / 128) * k + j) * 128 + (h & 127);
      const float y =
          a.y_tiles == 2 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(a.Y)[yt] << 16)
          : a.y_tiles == 1 ? a.Y[yt]
                           : a.Y[(int64_t)r.inv[(int64_t)t * k + j] * H + h];
      // a slot of weight zero (an expert left out of the computed subset)
      // adds nothing, whatever its stale Y holds
      const float wv = r.topk_w[(int64_t)t * k + j];
      if (wv != 0.f) acc = fmaf(wv, y, acc);
    }
    if (a.sh_gate_up) acc = fmaf(r.sigma[t], a.S[i], acc);
    if ((a.out_flags & 0xff) == 0) {
      const __nv_bfloat16 b = __float2bfloat16_rn(acc);
      reinterpret_cast<__nv_bfloat16*>(a.out)[i] = b;
    } else if (a.out_flags & 0x100) {
      reinterpret_cast<float*>(a.out)[i] += acc;
    } else {
      reinterpret_cast<float*>(a.out)[i] = acc;
    }
  }
}

// ------------------------------------------------------------------ RMS renorm

__global__ void k_rms_renorm(const float* __restrict__ y, uint16_t* __restrict__ x, int H) {
  // launched programmatically: the next layer's router may start streaming
  // its tiles now, and this grid waits for the one that wrote y
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const float* yr = y + (int64_t)t * H;
  __shared__ float red[32];
  float s = 0.f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) s = fmaf(yr[h], yr[h], s);
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[0] / (float)H + 1e-6f);
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(yr[h] * inv);
    x[(int64_t)t * H + h] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

// ------------------------------------------------------------------ launchers

// Per-function maxima shared by every handle in the process: always the
// request of the largest accepted sizes (H, I <= 8192, I_shared <= 4096).
cudaError_t experts_set_smem_limits(int H, int I) {
  (void)H;
  (void)I;
  const int Hm = 8192, Im = 8192, Ism = 4096;
  cudaError_t e;
  const int gu = kMT * (Hm / 2) * 4 + kMT * (Hm / kBlock) * 4 + kMT * 32 * 4;
  if ((e = cudaFuncSetAttribute(k_gate_up, cudaFuncAttributeMaxDynamicSharedMemorySize, gu)) != cudaSuccess)
    return e;
  const int dn = kMT * (Im / 2) * 4 + kMT * (Im / kBlock) * 4;
  if ((e = cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, dn)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_shared_gate_up, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kMT * Hm * 2)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_shared_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kMT * Ism * 4);
}

cudaError_t launch_experts(const ExpertArgs& a, cudaStream_t s, int parts) {
  cudaError_t err;
  const int grid = a.num_sms * 4;
  if ((parts & kPartSharedGateUp) && a.sh_gate_up) {
    dim3 g1((a.s_I_loc + 7) / 8, (a.T + kMT - 1) / kMT);
    FTMOE_PROF_BEGIN("k_shared_gate_up", s);
    k_shared_gate_up<<<g1, 256, (size_t)kMT * a.H * 2, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (parts & kPartRouted) {
    const size_t smem = (size_t)kMT * (a.H / 2) * 4 + kMT * (a.H / kBlock) * 4 + kMT * 32 * 4;
    FTMOE_PROF_BEGIN("k_gate_up", s);
    k_gate_up<<<grid, 256, smem, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (parts & kPartRouted) {
    const size_t smem = (size_t)kMT * (a.win.I_loc / 2) * 4 + kMT * (a.win.I_loc / kBlock) * 4;
    FTMOE_PROF_BEGIN("k_down", s);
    k_down<<<grid, 256, smem, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if ((parts & kPartTail) && a.sh_gate_up) {
    dim3 g2((a.H + 31) / 32, (a.T + kMT - 1) / kMT);
    FTMOE_PROF_BEGIN("k_shared_down", s);
    k_shared_down<<<g2, 256, (size_t)kMT * a.s_I_loc * 4, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (parts & kPartTail) {
    const int64_t n = (int64_t)a.T * a.H;
    int64_t nblk = (n + 255) / 256;
    if (nblk > (int64_t)a.num_sms * 16) nblk = (int64_t)a.num_sms * 16;
    int blocks = (int)nblk;
    FTMOE_PROF_BEGIN("k_combine", s);
    k_combine<<<blocks, 256, 0, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

__global__ void k_store_out(const float* __restrict__ y, void* out, int out_flags, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = y[i];
    if ((out_flags & 0xff) == 0) {
      reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
    } else if (out_flags & 0x100) {
      reinterpret_cast<float*>(out)[i] += v;
    } else {
      reinterpret_cast<float*>(out)[i] = v;
    }
  }
}

cudaError_t launch_store_out(const float* y, void* out, int out_flags, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  FTMOE_PROF_BEGIN("k_store_out", s);
  k_store_out<<<(int)blocks, 256, 0, s>>>(y, out, out_flags, n);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

// out = sum over r of parts[r] (fp32 [n_parts][n], rank order), rounded once
// to the output type (or added to an fp32 out): the combine of the window
// partials that the ranks of an intermediate-sharded layer exchange.  Four
// elements per thread; every element sums its partials in rank order.
__global__ void k_reduce_partials(const float* __restrict__ parts, int n_parts, int64_t n, void* out,
                                  int out_flags) {
  // whole float4s while every partial starts 16-byte aligned (n % 4 == 0)
  const int64_t n4 = (n & 3) == 0 ? n / 4 : 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (n + 3) / 4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (i < n4) {
      for (int r = 0; r < n_parts; ++r) {
        const float4 p = __ldg(reinterpret_cast<const float4*>(parts + (int64_t)r * n) + i);
        v[0] += p.x; v[1] += p.y; v[2] += p.z; v[3] += p.w;
      }
    } else {
      for (int r = 0; r < n_parts; ++r)
        for (int c = 0; c < 4 && 4 * i + c < n; ++c) v[c] += parts[(int64_t)r * n + 4 * i + c];
    }
    for (int c = 0; c < 4 && 4 * i + c < n; ++c) {
      const int64_t j = 4 * i + c;
      if ((out_flags & 0xff) == 0) reinterpret_cast<__nv_bfloat16*>(out)[j] = __float2bfloat16_rn(v[c]);
      else if (out_flags & 0x100) reinterpret_cast<float*>(out)[j] += v[c];
      else reinterpret_cast<float*>(out)[j] = v[c];
    }
  }
}

cudaError_t launch_reduce_partials(const float* parts, int n_parts, int64_t n, void* out, int out_flags,
                                   cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = ((n + 3) / 4 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  FTMOE_PROF_BEGIN("k_reduce_partials", s);
  k_reduce_partials<<<(int)blocks, 256, 0, s>>>(parts, n_parts, n, out, out_flags);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

// w_out[p] = w[p] if pair p's expert is in the mask, else 0 (the combine of
// an expert subset's pairs).
__global__ void k_mask_weights(const int32_t* __restrict__ idx, const float* __restrict__ w,
                               const uint8_t* __restrict__ mask, float* __restrict__ w_out, int64_t P) {
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < P; p += (int64_t)gridDim.x * blockDim.x)
    w_out[p] = mask[idx[p]] ? w[p] : 0.f;
}

cudaError_t launch_mask_weights(const int32_t* idx, const float* w, const uint8_t* mask, float* w_out, int64_t P,
                                cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  int64_t blocks = (P + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  FTMOE_PROF_BEGIN("k_mask_weights", s);
  k_mask_weights<<<(int)blocks, 256, 0, s>>>(idx, w, mask, w_out, P);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

cudaError_t launch_rms_renorm(const float* y, uint16_t* x, int T, int H, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  FTMOE_PROF_BEGIN("k_rms_renorm", s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_rms_renorm, y, x, H);
  FTMOE_PROF_END(s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ftmoe
