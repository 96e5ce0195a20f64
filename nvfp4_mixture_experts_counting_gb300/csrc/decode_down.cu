// k_dec_down: routed down projection of the decode path fused with the
// shared expert's down projection and the combine
//   out_t = sum_e w_(t,e) * Y_(t,e) + sigma_t * S_t
// (PR #385 "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
// (offload backend)", "What this adds": routed + sigmoid(gate) * shared
// before one reduce; down is [H, I], read by columns of the window, Issue #62
// "Offloaded MoE ignores tensor parallelism ...", "What it touches").
//
// One CTA owns 16 output rows.  A producer warp streams those rows of every
// touched expert (and that expert's quantised intermediates) into a ring of
// stages; 8 consumer warps add w * Y into per-row accumulators in a fixed
// expert order, then add sigma * S from the shared expert's rows.  No atomics
// on values, so the result is the same on every run (PR #385, "Correctness",
// traces run-to-run divergence to atomics in the expert kernels).
#include "decode_common.cuh"

namespace ftmoe {

// One pass over the up-to-MC pairs of an item: thread (row r, lane sub of 16)
// accumulates its row's dot products over the window's blocks sub, sub+16, ...
// The intermediates are decoded already: hv holds each pair's values as half
// (pitch hcp2 half2), hs each block's scale as fp32 (pitch hsp4 floats).
template <int MC>
__device__ __forceinline__ void dn_pass(const uint8_t* wrow, const uint8_t* wsc, const __half2* hv,
                                        const float* hs, int hcp2, int hsp4, int NBK, int sub, int mc,
                                        float acc[MC]) {
#pragma unroll
  for (int m = 0; m < MC; ++m) acc[m] = 0.f;
  for (int bb = sub; bb < NBK; bb += 16) {
    const uint2 wc = *reinterpret_cast<const uint2*>(wrow + bb * 8);
    const float sw = e4m3_decode(wsc[bb]);
    __half2 w[8];
    decode8(wc, w);
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      if (MC == 1 || m < mc) {
        const float d = dot16_h(w, hv + m * hcp2 + bb * 8);
        acc[m] = fmaf(d, sw * hs[m * hsp4 + bb], acc[m]);
      }
    }
  }
}

template <int MC>
__device__ __forceinline__ void dn_accumulate(const float acc[MC], int sub, int mc, int r, float gd, int c0,
                                              const int* s_tok, const float* s_w, float* out_s) {
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    float v = acc[m];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    if (sub == 0 && m < mc) {
      const int t = s_tok[c0 + m];
      out_s[t * kDnRows + r] = fmaf(s_w[c0 + m], v * gd, out_s[t * kDnRows + r]);
    }
  }
}

__global__ void __launch_bounds__(kDnThreads + 32) k_dec_down(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ int s_abort;
  const int I_loc = a.win.I_loc, NBK = I_loc / kBlock, T = a.T, E = a.r.E;
  const int P = T * a.top_k;
  const DnSmem L = dn_smem_choose(a.win.Iw, a.win.row0, I_loc, a.s_I_loc, T, E, P);
  const int NST = L.nst;
  constexpr int kConsumerWarps = kDnThreads / 32;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bar_off);
  uint64_t* empty = full + 8;
  uint64_t* shbar = full + 16;
  uint16_t* shw = reinterpret_cast<uint16_t*>(sm + L.shw_off);
  float* out_s = reinterpret_cast<float*>(sm + L.out_off);
  int* s_touched = reinterpret_cast<int*>(sm + L.touched_off);
  int* s_off = reinterpret_cast<int*>(sm + L.off_off);
  int* s_tok = reinterpret_cast<int*>(sm + L.tok_off);
  float* s_w = reinterpret_cast<float*>(sm + L.w_off);
  int* p_touched = reinterpret_cast<int*>(sm + L.ptouched_off);  // producer's own copies
  int* p_off = reinterpret_cast<int*>(sm + L.poff_off);
  const uint8_t** s_rec = reinterpret_cast<const uint8_t**>(sm + L.rec_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h0 = blockIdx.x * kDnRows;
  const int cbytes = align16(kDnRows * L.cpitch);
  const int hcp = a.hq_cpitch, hsp = a.hq_spitch;
  if (tid == 0) {
    // a stage is released once every consumer warp is done with it
    for (int s = 0; s < NST; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumerWarps); }
    mbar_init(shbar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool has_shared = a.sh_down != nullptr;
  if (warp == kConsumerWarps) {
    // ---- producer warp.  The shared expert's rows do not depend on the
    // previous kernel: start them before waiting for it.
    if (has_shared) {
      const uint32_t rb = a.s_I_loc * 2;
      if (lane == 0) mbar_arrive_expect_tx(shbar, kDnRows * rb);
      __syncwarp();
      if (lane < kDnRows)
        bulk_g2s(shw + lane * a.s_I_loc, a.sh_down + (int64_t)(h0 + lane) * a.s_Iw + a.s_row0, rb, shbar);
    }
    pdl_wait();
    const int nt = a.r.n_touched[0];
    for (int j = lane; j < nt; j += 32) {
      const int e = a.r.touched[j];
      s_rec[j] = a.rec[e];
      p_touched[j] = e;
    }
    for (int e = lane; e <= E; e += 32) p_off[e] = a.r.offsets[e];
    __syncwarp();
    if (lane == 0) {
      int k = 0;  // items issued
      bool stop = false;
      for (int kk = 0; kk < nt && !stop; ++kk) {
        const int e = p_touched[kk];
        const int s0 = p_off[e], s1 = p_off[e + 1];
        const uint8_t* rec = s_rec[kk];
        for (int c0 = s0; c0 < s1; c0 += kDnPairs) {
          const int s = k % NST;
          if (k >= NST && !mbar_wait(&empty[s], ((k / NST) - 1) & 1, a.r.status)) { s_abort = 1; stop = true; break; }
          if (*(volatile int*)&s_abort) { stop = true; break; }
          uint8_t* st = sm + s * L.stage_bytes;
          // 16 rows x Iw/2 code bytes, 16 x Iw/16 scale bytes, 16 globals and
          // the item's m decoded intermediate rows: every size a multiple of
          // 16 bytes and every source 16-byte aligned (Iw and h0 multiples of
          // 16, intermediate pitches multiples of 16 bytes)
          const uint32_t cb = kDnRows * L.cpitch, sb = kDnRows * L.spitch;
          const uint32_t m = min(kDnPairs, s1 - c0);
          mbar_arrive_expect_tx(&full[s], cb + sb + 64 + m * (hcp + hsp));
          bulk_g2s(st, rec + a.lay.dn_codes + (int64_t)h0 * L.cpitch, cb, &full[s]);
          bulk_g2s(st + cbytes, rec + a.lay.dn_scales + (int64_t)h0 * L.spitch, sb, &full[s]);
          bulk_g2s(st + cbytes + align16(sb), rec + a.lay.dn_global + (int64_t)h0 * 4, 64, &full[s]);
          bulk_g2s(st + L.hq_off, a.hq_codes + (int64_t)c0 * hcp, m * hcp, &full[s]);
          bulk_g2s(st + L.hs_off, a.hq_scales + (int64_t)c0 * hsp, m * hsp, &full[s]);
          ++k;
        }
      }
      // drain: nothing may be landing in shared memory when the CTA exits
      for (int j = k - NST > 0 ? k - NST : 0; j < k; ++j) mbar_wait(&full[j % NST], (j / NST) & 1, a.r.status);
      if (has_shared) mbar_wait(shbar, 0, a.r.status);
    }
    return;
  }
  // ---- consumers: thread -> row r (16 rows), 16 lanes per row; warp w owns
  // rows 2w and 2w+1 and every accumulator of them, so warps only meet at the
  // stage barriers.  A wait that runs out sets s_abort; the remaining items
  // are walked without waiting and the kernel writes nothing.
  const int r = tid >> 4, sub = tid & 15;
  for (int i = tid; i < T * kDnRows; i += kDnThreads) out_s[i] = 0.f;
  pdl_wait();
  const int nt = a.r.n_touched[0];
  for (int j = tid; j < nt; j += kDnThreads) s_touched[j] = a.r.touched[j];
  for (int e = tid; e <= E; e += kDnThreads) s_off[e] = a.r.offsets[e];
  for (int p = tid; p < P; p += kDnThreads) {
    const int pp = a.r.perm[p];
    s_tok[p] = pp / a.top_k;
    s_w[p] = a.r.topk_w[pp];
  }
  named_barrier(1, kDnThreads);
  const int hcp2 = hcp / 4, hsp4 = hsp / 4;
  int k = 0;
  for (int kk = 0; kk < nt; ++kk) {
    const int e = s_touched[kk];
    const int s0 = s_off[e], s1 = s_off[e + 1];
    for (int c0 = s0; c0 < s1; c0 += kDnPairs, ++k) {
      const int s = k % NST;
      if (!*(volatile int*)&s_abort && !mbar_wait(&full[s], (k / NST) & 1, a.r.status)) s_abort = 1;
      const uint8_t* st = sm + s * L.stage_bytes;
      const uint8_t* wrow = st + r * L.cpitch + L.coff;
      const uint8_t* wsc = st + cbytes + r * L.spitch + L.soff;
      const float gd = reinterpret_cast<const float*>(st + cbytes + align16(kDnRows * L.spitch))[r];
      const __half2* hv = reinterpret_cast<const __half2*>(st + L.hq_off);
      const float* hs = reinterpret_cast<const float*>(st + L.hs_off);
      const int mc = min(kDnPairs, s1 - c0);
      if (mc == 1) {
        float acc[1];
        dn_pass<1>(wrow, wsc, hv, hs, hcp2, hsp4, NBK, sub, mc, acc);
        dn_accumulate<1>(acc, sub, mc, r, gd, c0, s_tok, s_w, out_s);
      } else if (mc == 2) {
        float acc[2];
        dn_pass<2>(wrow, wsc, hv, hs, hcp2, hsp4, NBK, sub, mc, acc);
        dn_accumulate<2>(acc, sub, mc, r, gd, c0, s_tok, s_w, out_s);
      } else {
        float acc[kDnPairs];
        dn_pass<kDnPairs>(wrow, wsc, hv, hs, hcp2, hsp4, NBK, sub, mc, acc);
        dn_accumulate<kDnPairs>(acc, sub, mc, r, gd, c0, s_tok, s_w, out_s);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
    }
  }
  if (*(volatile int*)&s_abort) return;
  // ---- shared expert down rows and the combine (out_s[t][r] is owned by
  // the lane-0 thread of row r, which wrote every routed term of it)
  if (has_shared && !mbar_wait(shbar, 0, a.r.status)) return;
  const int nch = a.s_I_loc / 8;
  for (int t0 = 0; t0 < T; t0 += kDecMT) {
    float acc[kDecMT];
#pragma unroll
    for (int m = 0; m < kDecMT; ++m) acc[m] = 0.f;
    if (has_shared) {
      for (int c = sub; c < nch; c += 16) {
        const uint4 wv = *reinterpret_cast<const uint4*>(shw + r * a.s_I_loc + c * 8);
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int m = 0; m < kDecMT; ++m) {
          if (t0 + m < T) {
            const uint4 hv = __ldg(reinterpret_cast<const uint4*>(a.hs + (int64_t)(t0 + m) * a.s_I_loc) + c);
            const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[m] = fmaf(__uint_as_float(ww[q] << 16), __uint_as_float(hw[q] << 16), acc[m]);
              acc[m] = fmaf(__uint_as_float(ww[q] & 0xffff0000u), __uint_as_float(hw[q] & 0xffff0000u), acc[m]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kDecMT; ++m) {
      float v = acc[m];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      const int t = t0 + m;
      if (sub == 0 && t < T) {
        float o = out_s[t * kDnRows + r];
        if (has_shared) o = fmaf(a.r.sigma[t], v, o);
        const int64_t idx = (int64_t)t * a.H + h0 + r;
        if ((a.out_flags & 0xff) == 0) {
          reinterpret_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(o);
        } else if (a.out_flags & 0x100) {
          reinterpret_cast<float*>(a.out)[idx] += o;
        } else {
          reinterpret_cast<float*>(a.out)[idx] = o;
        }
      }
    }
  }
}

}  // namespace ftmoe
