// Routing kernels: activation quantisation + shared gate, router logits with
// a certified error bound, top-k with compensated re-ranking of uncertain
// candidates, and the counting-sort permutation.
//
// Pages: PR #385 "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
// (offload backend)", "What this adds" (replicated router; the shared gate of
// the combine); Issue #62 "Offloaded MoE ignores tensor parallelism ...",
// first comment (norm_topk_prob defaults to True; the fused expert kernels are
// dense-in/dense-out, so tokens are grouped per expert by a permutation).
#include "common.cuh"
#include "kernels.h"

namespace ftmoe {

// ------------------------------------------------------------------ quantisers

// One warp per row: row amax -> global, then every 16-block.
__global__ void k_quantize_weights(const float* __restrict__ w, int64_t rows, int K,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                   float* __restrict__ globals) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* wr = w + row * K;
  float amax = 0.f;
  for (int i = lane; i < K; i += 32) amax = fmaxf(amax, fabsf(wr[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float g = __fdiv_rn(amax, kWeightGlobalDiv);
  if (lane == 0) globals[row] = g;
  const int nb = K / kBlock;
  for (int b = lane; b < nb; b += 32) {
    float v[16];
    const float4* src = reinterpret_cast<const float4*>(wr + b * kBlock);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 f = src[q];
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
    uint8_t c[8];
    uint8_t s = quantize_block16(v, g, c);
    uint2 packed;
    packed.x = c[0] | (c[1] << 8) | (c[2] << 16) | ((uint32_t)c[3] << 24);
    packed.y = c[4] | (c[5] << 8) | (c[6] << 16) | ((uint32_t)c[7] << 24);
    *reinterpret_cast<uint2*>(codes + row * (K / 2) + b * 8) = packed;
    scales[row * nb + b] = s;
  }
}

// Quantise one block of 16 bf16 values (global 1.0) at src; returns the scale.
__device__ __forceinline__ uint8_t quant_bf16_block(const uint16_t* src, uint8_t* dst_codes,
                                                    float* dot_with = nullptr,
                                                    const uint16_t* g = nullptr) {
  float v[16];
  const uint4* p = reinterpret_cast<const uint4*>(src);
  uint4 a = p[0], b = p[1];
  uint32_t words[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(words[i] << 16);
    v[2 * i + 1] = __uint_as_float(words[i] & 0xffff0000u);
  }
  if (dot_with) {
    const uint4* gp = reinterpret_cast<const uint4*>(g);
    uint4 ga = gp[0], gb = gp[1];
    uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    float acc = *dot_with;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc = fmaf(v[2 * i], __uint_as_float(gw[i] << 16), acc);
      acc = fmaf(v[2 * i + 1], __uint_as_float(gw[i] & 0xffff0000u), acc);
    }
    *dot_with = acc;
  }
  uint8_t c[8];
  uint8_t s = quantize_block16(v, 1.0f, c);
  uint2 packed;
  packed.x = c[0] | (c[1] << 8) | (c[2] << 16) | ((uint32_t)c[3] << 24);
  packed.y = c[4] | (c[5] << 8) | (c[6] << 16) | ((uint32_t)c[7] << 24);
  *reinterpret_cast<uint2*>(dst_codes) = packed;
  return s;
}

// One thread per 16-block.
__global__ void k_quantize_act(const uint16_t* __restrict__ a, int64_t nblocks, int K,
                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  scales[b] = quant_bf16_block(a + b * kBlock, codes + b * 8);
}

// One warp per token: quantise x_t (global 1.0) and sigma_t = sigmoid(g . x_t).
__global__ void k_xquant_sigma(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int nb = a.H / kBlock;
  float z = 0.f;
  for (int b = lane; b < nb; b += 32) {
    int64_t blk = (int64_t)t * nb + b;
    a.xq_scales[blk] = quant_bf16_block(a.x + blk * kBlock, a.xq_codes + blk * 8,
                                        a.sh_gate ? &z : nullptr,
                                        a.sh_gate ? a.sh_gate + b * kBlock : nullptr);
  }
  if (a.sh_gate) {
    z = warp_sum(z);
    if (lane == 0) a.sigma[t] = 1.0f / (1.0f + expf(-z));
  } else if (lane == 0) {
    a.sigma[t] = 0.f;
  }
  if (a.xnorm) {
    // sum of squares of the bf16 values (exact products, fp32 sums), with a
    // relative margin far above the sum's rounding error
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + (int64_t)t * a.H);
    float q = 0.f;
    for (int i = lane; i < a.H / 8; i += 32) {
      const uint4 v = xr[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
        q = fmaf(lo, lo, q);
        q = fmaf(hi, hi, q);
      }
    }
    q = warp_sum(q);
    if (lane == 0) a.xnorm[t] = sqrtf(q) * (1.0f + 1e-5f);
  }
}

// ------------------------------------------------------------------ router logits

constexpr int kRouterTT = 8;     // tokens per CTA
constexpr int kRouterWarps = 8;  // experts per CTA (one per warp)

// logits[t][e] = sum_h x[t][h] * W[e][h] (+ b[e]) in fp32, and a rigorous
// bound err[t][e] on its distance from the exact value.  Each lane sums its
// products with FMAs in a fixed order (n = 4*ceil(H/128) roundings), then a
// 5-level butterfly and the bias add follow, so |l - exact| <= gamma_D * A
// + u*|l| with D = n + 6, u = 2^-24 and A = sum |x*w| (also accumulated here;
// the factor 1.01 covers A's own rounding).
__global__ void __launch_bounds__(kRouterWarps * 32) k_router_logits(RouteArgs a) {
  extern __shared__ __align__(16) uint16_t xs[];  // [kRouterTT][H]
  const int H = a.H;
  const int t0 = blockIdx.y * kRouterTT;
  const int tn = min(kRouterTT, a.T - t0);
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (int64_t)t0 * H);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n16 = tn * H / 8;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  if (e >= a.E) return;
  float acc[kRouterTT], ab[kRouterTT];
#pragma unroll
  for (int m = 0; m < kRouterTT; ++m) { acc[m] = 0.f; ab[m] = 0.f; }
  const float4* wr = reinterpret_cast<const float4*>(a.router_w + (int64_t)e * H);
  for (int c = lane; c < H / 4; c += 32) {
    const float4 w = __ldg(wr + c);
#pragma unroll
    for (int m = 0; m < kRouterTT; ++m) {
      if (m < tn) {
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + m * H + 4 * c);
        const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xffff0000u);
        const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xffff0000u);
        acc[m] = fmaf(x0, w.x, acc[m]);
        acc[m] = fmaf(x1, w.y, acc[m]);
        acc[m] = fmaf(x2, w.z, acc[m]);
        acc[m] = fmaf(x3, w.w, acc[m]);
        ab[m] = fmaf(fabsf(x0), fabsf(w.x), ab[m]);
        ab[m] = fmaf(fabsf(x1), fabsf(w.y), ab[m]);
        ab[m] = fmaf(fabsf(x2), fabsf(w.z), ab[m]);
        ab[m] = fmaf(fabsf(x3), fabsf(w.w), ab[m]);
      }
    }
  }
  const float bias = a.router_bias ? a.router_bias[e] : 0.f;
  const int n_seq = 4 * ((H / 4 + 31) / 32);
  const float gamma = (float)((double)(n_seq + 6) * 5.9604644775390625e-8 * 1.01);
#pragma unroll
  for (int m = 0; m < kRouterTT; ++m) {
    float s = warp_sum(acc[m]);
    float b = warp_sum(ab[m]);
    if (lane == 0 && m < tn) {
      float l = s + bias;
      a.logits[(int64_t)(t0 + m) * a.E + e] = l;
      a.err[(int64_t)(t0 + m) * a.E + e] = gamma * b + 1.2e-7f * fabsf(l) + 1e-30f;
    }
  }
}

// ------------------------------------------------------------------ top-k

constexpr int kTopkWarps = 4;

// Key order: larger logit first, then lower expert index.
__device__ __forceinline__ bool before(float la, int ea, float lb, int eb) {
  return la > lb || (la == lb && ea < eb);
}
// One warp per token.  Select the k best by fp32 logit; certify the set and
// its order with the error bounds; if not certified, recompute compensated
// double-fp32 logits (about 2^-48 relative; FP64 is far slower on this GPU)
// for every expert that could belong to the top-k and select among those.
// The recomputations of all the CTA's uncertain tokens are spread over its
// warps.
__global__ void __launch_bounds__(kTopkWarps * 32) k_topk(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ int s_nc[kTopkWarps];
  const int E = a.E, k = a.top_k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* lw = reinterpret_cast<float*>(sm) + warp * E;                // working logits
  int* cand = reinterpret_cast<int*>(sm) + kTopkWarps * E + warp * E;  // candidate list
  df32* l64 = reinterpret_cast<df32*>(sm + (size_t)kTopkWarps * E * 8) + warp * E;
  // the token's logits and bounds, copied once: every later read is in
  // shared memory (the selection's reads depend on the previous round's
  // winner, so from global memory each would wait a full load latency)
  float* lg = reinterpret_cast<float*>(sm + (size_t)kTopkWarps * E * 16) + warp * E;
  float* er = reinterpret_cast<float*>(sm + (size_t)kTopkWarps * E * 20) + warp * E;
  const int t = blockIdx.x * kTopkWarps + warp;
  const bool have = t < a.T;
  {
    const float* lgg = a.logits + (int64_t)(have ? t : 0) * E;
    const float* erg = a.err + (int64_t)(have ? t : 0) * E;
    for (int e = lane; e < E; e += 32) {
      const float l = lgg[e];
      lw[e] = l;
      lg[e] = l;
      er[e] = erg[e];
    }
  }
  __syncwarp();

  int chosen[32];
  float lmax = -INFINITY;
  bool certified = true;
  float prev_lo = INFINITY;
  float lmin_lo = INFINITY;
  for (int j = 0; j < k; ++j) {
    float bl = -INFINITY;
    int be = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      float v = lw[e];
      if (before(v, e, bl, be)) { bl = v; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ol = __shfl_xor_sync(0xffffffffu, bl, o);
      int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (before(ol, oe, bl, be)) { bl = ol; be = oe; }
    }
    chosen[j] = be;
    if (j == 0) lmax = bl;
    const float lo = bl - er[be], hi = bl + er[be];
    if (!(hi < prev_lo)) certified = false;  // order against the previous slot
    prev_lo = lo;
    lmin_lo = fminf(lmin_lo, lo);
    __syncwarp();
    if (lane == 0) lw[be] = -INFINITY;
    __syncwarp();
  }
  // any unchosen expert whose interval reaches the lowest chosen lower end?
  bool reach = false;
  for (int e = lane; e < E; e += 32)
    if (lw[e] != -INFINITY && lg[e] + er[e] >= lmin_lo) reach = true;
  if (__any_sync(0xffffffffu, reach)) certified = false;

  float w64[32];
  if (!have) certified = true;
  // candidates: the chosen plus every unchosen expert that may outrank one
  int nc = 0;
  if (!certified) {
    if (lane == 0 && a.n_rerank) atomicAdd(a.n_rerank, 1ull);  // telemetry only
    for (int base = 0; base < E; base += 32) {
      int e = base + lane;
      bool c = false;
      if (e < E) c = (lw[e] == -INFINITY) || (lg[e] + er[e] >= lmin_lo);
      unsigned m = __ballot_sync(0xffffffffu, c);
      if (c) cand[nc + __popc(m & ((1u << lane) - 1))] = e;
      nc += __popc(m);
    }
  }
  // Only a candidate whose interval meets another candidate's needs its
  // compensated logit: one whose interval is apart from every other
  // candidate's already ranks right against all of them by its fp32 logit
  // (and an expert outside the candidates ranks below every chosen one).
  // The list of those that need it reuses the warp's working logits.
  int* need = reinterpret_cast<int*>(lw);
  int nn = 0;
  __syncwarp();
  if (!certified) {
    for (int base = 0; base < nc; base += 32) {
      const int c = base + lane;
      bool nd = false;
      if (c < nc) {
        const int e = cand[c];
        const float l = lg[e], r = er[e];
        for (int c2 = 0; c2 < nc && !nd; ++c2) {
          const int e2 = cand[c2];
          if (c2 != c && fabsf(l - lg[e2]) <= r + er[e2]) nd = true;
        }
        l64[c] = df32{l, 0.f};  // the fp32 logit, unless computed again below
      }
      const unsigned m = __ballot_sync(0xffffffffu, nd);
      if (nd) need[nn + __popc(m & ((1u << lane) - 1))] = c;
      nn += __popc(m);
    }
  }
  if (lane == 0) s_nc[warp] = nn;
  __syncthreads();
  {
    // every warp computes compensated logits of the CTA's needed candidates in turn
    int total = 0;
    for (int w = 0; w < kTopkWarps; ++w) total += s_nc[w];
    for (int item = warp; item < total; item += kTopkWarps) {
      int w = 0, i = item;
      while (i >= s_nc[w]) { i -= s_nc[w]; ++w; }
      const int tw = blockIdx.x * kTopkWarps + w;
      const int c = reinterpret_cast<const int*>(sm)[w * E + i];
      const int e = reinterpret_cast<const int*>(sm)[kTopkWarps * E + w * E + c];
      const df32 v = logit_df32(a.x + (int64_t)tw * a.H, a.router_w + (int64_t)e * a.H, a.H,
                                a.router_bias ? a.router_bias[e] : 0.f, lane);
      if (lane == 0) reinterpret_cast<df32*>(sm + (size_t)kTopkWarps * E * 8)[w * E + c] = v;
    }
  }
  __syncthreads();
  if (!have) return;
  if (!certified) {
    // select k among the candidates by (compensated logit desc, index asc)
    const df32 none = {-INFINITY, 0.f};
    for (int j = 0; j < k; ++j) {
      df32 bl = none;
      int be = 0x7fffffff, bc = -1;
      for (int c = lane; c < nc; c += 32) {
        const df32 v = l64[c];
        const int e = cand[c];
        if (v.hi != -INFINITY && df_before(v, e, bl, be)) { bl = v; be = e; bc = c; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const df32 ol = {__shfl_xor_sync(0xffffffffu, bl.hi, o), __shfl_xor_sync(0xffffffffu, bl.lo, o)};
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
        if (df_before(ol, oe, bl, be)) { bl = ol; be = oe; bc = oc; }
      }
      chosen[j] = be;
      w64[j] = bl.hi;
      __syncwarp();
      if (lane == 0) l64[bc] = none;
      __syncwarp();
    }
    lmax = w64[0];
  }
  // routing weights
  float wt[32];
  if (a.norm_topk_prob) {
    float den = 0.f;
    for (int j = 0; j < k; ++j) {
      float l = certified ? lg[chosen[j]] : (float)w64[j];
      wt[j] = expf(l - lmax);
      den += wt[j];
    }
    for (int j = 0; j < k; ++j) wt[j] = wt[j] / den;
  } else {
    float den = 0.f;
    for (int e = lane; e < E; e += 32) den += expf(lg[e] - lmax);
    den = warp_sum(den);
    for (int j = 0; j < k; ++j) {
      float l = certified ? lg[chosen[j]] : (float)w64[j];
      wt[j] = expf(l - lmax) / den;
    }
  }
  if (lane < k) {
    int idx = chosen[0];
    float ww = wt[0];
    for (int j = 1; j < k; ++j)
      if (lane == j) { idx = chosen[j]; ww = wt[j]; }
    a.topk_idx[(int64_t)t * k + lane] = idx;
    a.topk_w[(int64_t)t * k + lane] = ww;
  }
}

// ------------------------------------------------------------------ counting sort

constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortChunk = 4096;  // pairs per CTA of the many-CTA sort

// Exclusive scan of v over the CTA's 1024 threads; returns the prefix and
// writes the total to *total.
__device__ int block_exclusive_scan(int v, int* scratch /*[32]*/, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    scratch[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  int res = scratch[warp] + inc - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// Single CTA.  Histogram per warp chunk -> exclusive scan over experts ->
// per-(warp, expert) cursors -> each warp scatters its chunk in order, so the
// pairs of every expert come out in increasing pair id (a stable sort).
__global__ void __launch_bounds__(kSortThreads) k_sort(RouteArgs a) {
  extern __shared__ int hist[];  // [kSortWarps][E]
  __shared__ int scratch[33];
  const int E = a.E;
  const int P = a.T * a.top_k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSortWarps * E; i += kSortThreads) hist[i] = 0;
  __syncthreads();
  const int CH = (P + kSortWarps - 1) / kSortWarps;
  const int c0 = min(P, warp * CH), c1 = min(P, c0 + CH);
  // eight of the lane's loads in flight at a time
  for (int p0 = c0; p0 < c1; p0 += 32 * 8) {
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = p0 + 32 * u + lane;
      ev[u] = p < c1 ? __ldg(a.topk_idx + p) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (p0 + 32 * u + lane < c1) {
        int e = ev[u];
        if ((unsigned)e >= (unsigned)E) { set_status(a.status, kStatusRange); e = 0; }
        atomicAdd(&hist[warp * E + e], 1);
      }
    }
  }
  __syncthreads();
  for (int base = 0; base < E; base += kSortThreads) {
    const int e = base + threadIdx.x;
    int cnt = 0;
    if (e < E)
      for (int w = 0; w < kSortWarps; ++w) cnt += hist[w * E + e];
    int total;
    int off = block_exclusive_scan(cnt, scratch, &total);
    int prev_total = base == 0 ? 0 : a.offsets[base];  // running offset of earlier chunks
    off += prev_total;
    int tflag;
    int tpos = block_exclusive_scan((e < E && cnt > 0) ? 1 : 0, scratch, &tflag);
    int prev_touched = base == 0 ? 0 : a.n_touched[0];
    if (e < E) {
      a.offsets[e] = off;
      if (cnt > 0) a.touched[prev_touched + tpos] = e;
      int cur = off;
      for (int w = 0; w < kSortWarps; ++w) {
        int h = hist[w * E + e];
        hist[w * E + e] = cur;
        cur += h;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      a.offsets[min(base + kSortThreads, E)] = prev_total + total;
      a.n_touched[0] = prev_touched + tflag;
    }
    __threadfence_block();
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.offsets[E] = P;
    if (a.touched_total) atomicAdd(a.touched_total, (unsigned long long)a.n_touched[0]);
  }
  __syncthreads();
  for (int p8 = c0; p8 < c1; p8 += 32 * 8) {
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = p8 + 32 * u + lane;
      ev[u] = p < c1 ? __ldg(a.topk_idx + p) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p0 = p8 + 32 * u;
      if (p0 >= c1) break;  // uniform across the warp
      const int p = p0 + lane;
      const bool valid = p < c1;
      int e = valid ? ev[u] : -1 - lane;
      if (valid && (unsigned)e >= (unsigned)E) e = 0;
      const unsigned mask = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(mask & ((1u << lane) - 1));
      int pos = 0;
      if (valid) pos = hist[warp * E + e] + rank;
      __syncwarp();
      if (valid) {
        a.perm[pos] = p;
        a.inv[p] = pos;
        if (rank == 0) hist[warp * E + e] += __popc(mask);
      }
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------------ counting sort over many CTAs

// The same stable counting sort for large P, in three grids: each CTA c
// counts its chunk of pairs [c * kSortChunk, ...) per expert; one CTA turns
// the counts into the expert offsets and, per (chunk, expert), the first
// sorted position of that chunk's pairs (chunks in order); each CTA then
// scatters its chunk exactly as k_sort does (warps in order, lanes in order
// within a warp), so every expert's pairs still come out in increasing pair
// id.

// Per-warp histogram of the warp's part of [c0, c1) into hist[warp][e].
__device__ void sort_warp_hist(const RouteArgs& a, int E, int c0, int c1, int* hist) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSortWarps * E; i += kSortThreads) hist[i] = 0;
  __syncthreads();
  const int CH = (c1 - c0 + kSortWarps - 1) / kSortWarps;
  const int w0 = min(c1, c0 + warp * CH), w1 = min(c1, w0 + CH);
  for (int p = w0 + lane; p < w1; p += 32) {
    int e = __ldg(a.topk_idx + p);
    if ((unsigned)e >= (unsigned)E) { set_status(a.status, kStatusRange); e = 0; }
    atomicAdd(&hist[warp * E + e], 1);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kSortThreads) k_sort_count(RouteArgs a) {
  extern __shared__ int hist[];  // [kSortWarps][E]
  const int E = a.E, P = a.T * a.top_k;
  const int c0 = min(P, (int)blockIdx.x * kSortChunk), c1 = min(P, c0 + kSortChunk);
  sort_warp_hist(a, E, c0, c1, hist);
  for (int e = threadIdx.x; e < E; e += kSortThreads) {
    int cnt = 0;
    for (int w = 0; w < kSortWarps; ++w) cnt += hist[w * E + e];
    a.sort_cnt[(int64_t)blockIdx.x * E + e] = cnt;
  }
}

// One CTA: offsets, the touched list, and sort_cnt[c][e] replaced by the
// first sorted position of chunk c's pairs of expert e.
__global__ void __launch_bounds__(kSortThreads) k_sort_scan(RouteArgs a, int n_chunks) {
  __shared__ int scratch[33];
  const int E = a.E, P = a.T * a.top_k;
  for (int base = 0; base < E; base += kSortThreads) {
    const int e = base + threadIdx.x;
    int cnt = 0;
    if (e < E)
      for (int c = 0; c < n_chunks; ++c) cnt += a.sort_cnt[(int64_t)c * E + e];
    int total;
    int off = block_exclusive_scan(cnt, scratch, &total);
    const int prev_total = base == 0 ? 0 : a.offsets[base];
    off += prev_total;
    int tflag;
    const int tpos = block_exclusive_scan((e < E && cnt > 0) ? 1 : 0, scratch, &tflag);
    const int prev_touched = base == 0 ? 0 : a.n_touched[0];
    if (e < E) {
      a.offsets[e] = off;
      if (cnt > 0) a.touched[prev_touched + tpos] = e;
      int cur = off;
      for (int c = 0; c < n_chunks; ++c) {
        int* q = a.sort_cnt + (int64_t)c * E + e;
        const int h = *q;
        *q = cur;
        cur += h;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      a.offsets[min(base + kSortThreads, E)] = prev_total + total;
      a.n_touched[0] = prev_touched + tflag;
    }
    __threadfence_block();
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.offsets[E] = P;
    if (a.touched_total) atomicAdd(a.touched_total, (unsigned long long)a.n_touched[0]);
  }
}

__global__ void __launch_bounds__(kSortThreads) k_sort_scatter(RouteArgs a) {
  extern __shared__ int hist[];  // [kSortWarps][E]: counts, then each warp's cursors
  const int E = a.E, P = a.T * a.top_k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = min(P, (int)blockIdx.x * kSortChunk), c1 = min(P, c0 + kSortChunk);
  sort_warp_hist(a, E, c0, c1, hist);
  for (int e = threadIdx.x; e < E; e += kSortThreads) {
    int cur = a.sort_cnt[(int64_t)blockIdx.x * E + e];
    for (int w = 0; w < kSortWarps; ++w) {
      const int h = hist[w * E + e];
      hist[w * E + e] = cur;
      cur += h;
    }
  }
  __syncthreads();
  const int CH = (c1 - c0 + kSortWarps - 1) / kSortWarps;
  const int w0 = min(c1, c0 + warp * CH), w1 = min(c1, w0 + CH);
  for (int p0 = w0; p0 < w1; p0 += 32) {
    const int p = p0 + lane;
    const bool valid = p < w1;
    int e = valid ? __ldg(a.topk_idx + p) : -1 - lane;
    if (valid && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(mask & ((1u << lane) - 1));
    int pos = 0;
    if (valid) pos = hist[warp * E + e] + rank;
    __syncwarp();
    if (valid) {
      a.perm[pos] = p;
      a.inv[p] = pos;
      if (rank == 0) hist[warp * E + e] += __popc(mask);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_quantize_weights(const float* w, int64_t rows, int K, uint8_t* codes,
                                    uint8_t* scales, float* globals, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int wpb = 8;
  FTMOE_PROF_BEGIN("k_quantize_weights", s);
  k_quantize_weights<<<(unsigned)((rows + wpb - 1) / wpb), wpb * 32, 0, s>>>(w, rows, K, codes, scales,
                                                                            globals);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

cudaError_t launch_quantize_act_bf16(const uint16_t* a, int64_t rows, int K, uint8_t* codes,
                                     uint8_t* scales, cudaStream_t s) {
  const int64_t nb = rows * (K / kBlock);
  if (nb == 0) return cudaSuccess;
  FTMOE_PROF_BEGIN("k_quantize_act", s);
  k_quantize_act<<<(unsigned)((nb + 255) / 256), 256, 0, s>>>(a, nb, K, codes, scales);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, int parts) {
  cudaError_t err;
  if (parts & kRouteXq) {
    const int wpb = 8;
    FTMOE_PROF_BEGIN("k_xquant_sigma", s);
    k_xquant_sigma<<<(a.T + wpb - 1) / wpb, wpb * 32, 0, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (parts & kRouteLogits) {
    dim3 grid((a.E + kRouterWarps - 1) / kRouterWarps, (a.T + kRouterTT - 1) / kRouterTT);
    size_t smem = (size_t)kRouterTT * a.H * 2;
    FTMOE_PROF_BEGIN("k_router_logits", s);
    k_router_logits<<<grid, kRouterWarps * 32, smem, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (parts & kRouteTopk) {
    size_t smem = (size_t)kTopkWarps * a.E * (4 + 4 + 8 + 4 + 4);
    FTMOE_PROF_BEGIN("k_topk", s);
    k_topk<<<(a.T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, smem, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (parts & kRouteSort) {
    size_t smem = (size_t)kSortWarps * a.E * 4;
    const int64_t P = (int64_t)a.T * a.top_k;
    const int n_chunks = (int)((P + kSortChunk - 1) / kSortChunk);
    // the many-CTA sort (three launches) pays off above four chunks; below,
    // the one-CTA sort's single launch is faster
    if (a.sort_cnt && n_chunks > 4 && n_chunks <= a.sort_max_chunks) {
      FTMOE_PROF_BEGIN("k_sort_count", s);
      k_sort_count<<<n_chunks, kSortThreads, smem, s>>>(a);
      FTMOE_PROF_END(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
      FTMOE_PROF_BEGIN("k_sort_scan", s);
      k_sort_scan<<<1, kSortThreads, 0, s>>>(a, n_chunks);
      FTMOE_PROF_END(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
      FTMOE_PROF_BEGIN("k_sort_scatter", s);
      k_sort_scatter<<<n_chunks, kSortThreads, smem, s>>>(a);
      FTMOE_PROF_END(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
    } else {
      FTMOE_PROF_BEGIN("k_sort", s);
      k_sort<<<1, kSortThreads, smem, s>>>(a);
      FTMOE_PROF_END(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
  }
  return cudaSuccess;
}

// Opt the kernels that need more than 48 KB of dynamic shared memory in.
// The limit is a per-function maximum shared by every handle in the process,
// so it is always set to what the largest accepted sizes (H <= 8192,
// E <= 1024) can request; the arguments only have to stay within those.
cudaError_t route_set_smem_limits(int H, int E) {
  (void)H;
  (void)E;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_router_logits, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kRouterTT * 8192 * 2)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTopkWarps * 1024 * 24)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_sort_count, cudaFuncAttributeMaxDynamicSharedMemorySize, kSortWarps * 1024 * 4)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_sort_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSortWarps * 1024 * 4)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_sort, cudaFuncAttributeMaxDynamicSharedMemorySize, kSortWarps * 1024 * 4);
}

}  // namespace ftmoe
