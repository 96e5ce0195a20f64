// k_dec_gate_up: routed gate_up of the decode path, fused with SwiGLU and the
// NVFP4 quantisation of the intermediate.
//
// Persistent, one CTA per SM, each with a contiguous range of work items
// (touched expert, 16-wide block ib of the window: 16 gate rows [i0+16ib,
// +16) and the matching 16 up rows [I+i0+16ib, +16), Issue #62 "Offloaded MoE
// ignores tensor parallelism ...", "What it touches").  A producer warp
// streams each item's codes, scales and globals into a ring of shared-memory
// stages with bulk-async copies; 16 consumer warps form, for every pair of
// the expert, G = g_row * sum_b s_w * s_x * dot_b; then half-warps apply
// h = silu(G_gate) * G_up and quantise each pair's 16 values.
#include "decode_common.cuh"

namespace ftmoe {

// One pass of up to MC tokens over one item: the warp of window index i
// covers gate row i and up row i; lane sub takes blocks sub, sub+32, ... of
// both rows, so each activation block it loads serves two rows.
template <int MC>
__device__ __forceinline__ void gu_pass(const uint8_t* grow, const uint8_t* urow, const uint8_t* gsc,
                                        const uint8_t* usc, const __half2* xh, const float* xsf, int HC, int NB,
                                        int sub, int mc, float ag[MC], float au[MC]) {
#pragma unroll
  for (int m = 0; m < MC; ++m) { ag[m] = 0.f; au[m] = 0.f; }
  for (int bb = sub; bb < NB; bb += 32) {
    const uint2 gc = *reinterpret_cast<const uint2*>(grow + bb * 8);
    const uint2 uc = *reinterpret_cast<const uint2*>(urow + bb * 8);
    const float sg = e4m3_decode(gsc[bb]), su = e4m3_decode(usc[bb]);
    __half2 wg[8], wu[8];
    decode8(gc, wg);
    decode8(uc, wu);
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      if (MC == 1 || m < mc) {
        const __half2* xp = xh + m * HC + bb * 8;
        const float sx = xsf[m * NB + bb];
        ag[m] = fmaf(dot16_h(wg, xp), sg * sx, ag[m]);
        au[m] = fmaf(dot16_h(wu, xp), su * sx, au[m]);
      }
    }
  }
}

template <int MC>
__device__ __forceinline__ void gu_reduce(const float ag[MC], const float au[MC], int sub, int mc, int i,
                                          float gwg, float gwu, float* G) {
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    const float g = warp_sum(ag[m]), u = warp_sum(au[m]);
    if (sub == 0 && m < mc) {
      G[m * kGuRows + i] = g * gwg;
      G[m * kGuRows + 16 + i] = u * gwu;
    }
  }
}

__global__ void __launch_bounds__(kGuThreads + 32, 1) k_dec_gate_up(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ int s_abort;
  const int H = a.H, NB = H / kBlock, HC = H / 2, T = a.T, E = a.r.E;
  const int P = T * a.top_k;
  const GuSmem L = gu_smem_layout(H, T, E, P);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bar_off);
  uint64_t* empty = full + 4;
  uint64_t* xbar = full + 8;
  uint8_t* xs = sm + L.xs_off;
  uint8_t* xsc = sm + L.xsc_off;
  __half2* xh = reinterpret_cast<__half2*>(sm + L.xh_off);
  float* xsf = reinterpret_cast<float*>(sm + L.xsf_off);
  int* s_touched = reinterpret_cast<int*>(sm + L.touched_off);
  int* s_off = reinterpret_cast<int*>(sm + L.off_off);
  int* s_tok = reinterpret_cast<int*>(sm + L.tok_off);
  const uint8_t** s_rec = reinterpret_cast<const uint8_t**>(sm + L.rec_off);
  float* Gs = reinterpret_cast<float*>(sm + L.g_off);  // [2][kDecMT][32]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < L.nst; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(xbar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const int n_ib = a.win.I_loc / kBlock;
  const int n_items = a.r.n_touched[0] * n_ib;
  // this CTA's items, balanced by cost by the routing kernel
  const int it0 = min(n_items, a.gu_split[blockIdx.x]), it1 = min(n_items, a.gu_split[blockIdx.x + 1]);
  if (it0 >= it1) return;
  const int e_first = it0 / n_ib, e_last = (it1 - 1) / n_ib;  // touched indices this CTA uses
  if (warp == kGuThreads / 32) {
    // ---- producer warp: record pointers of its experts, then the copies
    for (int j = e_first + lane; j <= e_last; j += 32) s_rec[j] = a.rec[a.r.touched[j]];
    __syncwarp();
    if (lane == 0) {
      // every token's quantised activations (contiguous rows)
      const uint32_t xb = T * HC, sb = T * NB;
      mbar_arrive_expect_tx(xbar, xb + sb);
      bulk_g2s(xs, a.r.xq_codes, xb, xbar);
      bulk_g2s(xsc, a.r.xq_scales, sb, xbar);
      int issued = 0;
      for (int it = it0, k = 0; it < it1; ++it, ++k) {
        const int s = k % L.nst;
        if (k >= L.nst && !mbar_wait(&empty[s], ((k / L.nst) - 1) & 1, a.r.status)) { s_abort = 1; break; }
        if (*(volatile int*)&s_abort) break;
        const uint8_t* rec = s_rec[it / n_ib];
        const int g0 = a.win.row0 + (it % n_ib) * kBlock;  // first gate row of the item
        const int u0 = a.win.Iw + g0;                         // first up row
        uint8_t* st = sm + s * L.item_bytes;
        const uint32_t cb = 16 * HC, scb = 16 * NB;
        mbar_arrive_expect_tx(&full[s], 2 * cb + 2 * scb + 128);
        bulk_g2s(st, rec + a.lay.gu_codes + (int64_t)g0 * HC, cb, &full[s]);
        bulk_g2s(st + cb, rec + a.lay.gu_codes + (int64_t)u0 * HC, cb, &full[s]);
        bulk_g2s(st + 2 * cb, rec + a.lay.gu_scales + (int64_t)g0 * NB, scb, &full[s]);
        bulk_g2s(st + 2 * cb + scb, rec + a.lay.gu_scales + (int64_t)u0 * NB, scb, &full[s]);
        bulk_g2s(st + 2 * cb + 2 * scb, rec + a.lay.gu_global + (int64_t)g0 * 4, 64, &full[s]);
        bulk_g2s(st + 2 * cb + 2 * scb + 64, rec + a.lay.gu_global + (int64_t)u0 * 4, 64, &full[s]);
        issued = k + 1;
      }
      // nothing may still be landing in this CTA's shared memory when it
      // exits: wait (bounded) for the activations and the last use of every
      // stage
      mbar_wait(xbar, 0, a.r.status);
      for (int k = issued - L.nst > 0 ? issued - L.nst : 0; k < issued; ++k)
        mbar_wait(&full[k % L.nst], (k / L.nst) & 1, a.r.status);
    }
    return;
  }
  // ---- consumers: routing metadata once, then the items.  A wait that runs
  // out sets s_abort; every consumer still walks the same barriers (without
  // waiting again), so none is left behind at a barrier.
  for (int j = e_first + tid; j <= e_last; j += kGuThreads) s_touched[j] = a.r.touched[j];
  for (int e = tid; e <= E; e += kGuThreads) s_off[e] = a.r.offsets[e];
  for (int p = tid; p < P; p += kGuThreads) s_tok[p] = a.r.perm[p] / a.top_k;
  if (!mbar_wait(xbar, 0, a.r.status)) s_abort = 1;
  named_barrier(1, kGuThreads);
  // warp i -> window index i of the item (gate row i, up row 16 + i)
  const int i = warp, sub = lane;
  int staged_e = -1;  // expert whose (single) pass is in xh
  int pass = 0;
  for (int it = it0, k = 0; it < it1; ++it, ++k) {
    const int s = k % L.nst;
    const int e = s_touched[it / n_ib], ib = it % n_ib;
    const int s0 = s_off[e], s1 = s_off[e + 1];
    if (!*(volatile int*)&s_abort && !mbar_wait(&full[s], (k / L.nst) & 1, a.r.status)) s_abort = 1;
    const uint8_t* st = sm + s * L.item_bytes;
    const uint8_t* grow = st + i * HC;
    const uint8_t* urow = st + (16 + i) * HC;
    const uint8_t* gsc = st + kGuRows * HC + i * NB;
    const uint8_t* usc = st + kGuRows * HC + (16 + i) * NB;
    const float* glob = reinterpret_cast<const float*>(st + kGuRows * HC + kGuRows * NB);
    const float gwg = glob[i], gwu = glob[16 + i];
    const bool multi = (s1 - s0) > kDecMT;
    for (int c0 = s0; c0 < s1; c0 += kDecMT, ++pass) {
      const int mc = min(kDecMT, s1 - c0);
      float* G = Gs + (pass & 1) * kDecMT * kGuRows;
      if (multi || e != staged_e) {
        // half2 code values and fp32 scales of this pass's tokens (every
        // reader of the previous pass's values passed the last barrier)
        for (int i = tid; i < mc * HC; i += kGuThreads) {
          const int m = i / HC, c = i - m * HC;
          xh[m * HC + c] = e2m1x2_to_half2(xs[s_tok[c0 + m] * HC + c]);
        }
        for (int i = tid; i < mc * NB; i += kGuThreads) {
          const int m = i / NB, bb = i - m * NB;
          xsf[m * NB + bb] = e4m3_decode(xsc[s_tok[c0 + m] * NB + bb]);
        }
        staged_e = multi ? -1 : e;
        named_barrier(1, kGuThreads);
      }
      if (mc == 1) {
        float ag[1], au[1];
        gu_pass<1>(grow, urow, gsc, usc, xh, xsf, HC, NB, sub, mc, ag, au);
        gu_reduce<1>(ag, au, sub, mc, i, gwg, gwu, G);
      } else if (mc == 2) {
        float ag[2], au[2];
        gu_pass<2>(grow, urow, gsc, usc, xh, xsf, HC, NB, sub, mc, ag, au);
        gu_reduce<2>(ag, au, sub, mc, i, gwg, gwu, G);
      } else if (mc <= 4) {
        float ag[4], au[4];
        gu_pass<4>(grow, urow, gsc, usc, xh, xsf, HC, NB, sub, mc, ag, au);
        gu_reduce<4>(ag, au, sub, mc, i, gwg, gwu, G);
      } else {
        float ag[8], au[8];
        gu_pass<8>(grow, urow, gsc, usc, xh, xsf, HC, NB, sub, mc, ag, au);
        gu_reduce<8>(ag, au, sub, mc, i, gwg, gwu, G);
      }
      named_barrier(1, kGuThreads);  // G written; stage and xh read by every consumer
      if (tid == 0 && c0 + kDecMT >= s1) mbar_arrive(&empty[s]);  // item done: stage free
      if (warp < kDecMT / 2) {
        // half-warp per pair: SwiGLU and quantisation of its 16 values
        const int m = 2 * warp + (lane >> 4), l = lane & 15;
        const int64_t pos = c0 + m;
        const bool w = m < mc;
        swiglu_quant16(G[m * kGuRows + l], G[m * kGuRows + 16 + l], l, w,
                       reinterpret_cast<__half*>(a.hq_codes + (w ? pos : 0) * a.hq_cpitch) + ib * kBlock,
                       reinterpret_cast<float*>(a.hq_scales + (w ? pos : 0) * a.hq_spitch) + ib);
      }
    }
  }
}

}  // namespace ftmoe
