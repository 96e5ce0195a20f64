// Shared pieces of the decode path (1 <= T <= 32): sizes, shared-memory
// layouts of its three kernels, and the NVFP4 block helpers they use.
//
// At decode sizes the layer is a read of the touched expert bytes (Issue #62
// "Offloaded MoE ignores tensor parallelism ...", "Why TP=2 loses today": the
// step streams experts; PR #385 "feat(qwen4_exp): tensor parallelism for
// Qwen3.8-Flash-Next (offload backend)", "Measurements": the decode step is
// dominated by weight reads).  Each 16-element block product is formed
// exactly in half precision from E2M1 codes and scaled in fp32.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace ftmoe {

constexpr int kGuThreads = 512;  // k_dec_gate_up consumers (16 warps); +1 producer warp
constexpr int kDnThreads = 256;  // k_dec_down consumers (8 warps); +1 producer warp
constexpr int kRtThreads = 256;  // k_dec_route
constexpr int kDecMT = 8;        // tokens / pairs per compute pass
constexpr int kGuRows = 32;      // 16 gate + 16 up rows per item
constexpr int kDnRows = 16;      // output rows per down CTA
constexpr int kDecMaxT = 32;
// dynamic shared memory a decode kernel may request (below the 227 KB opt-in
// limit, leaving room for the static variables)
constexpr int kDecSmemMax = 220 * 1024;

__global__ void k_dec_route(DecodeArgs a);
__global__ void k_dec_topk(DecodeArgs a);
__global__ void k_dec_gate_up(DecodeArgs a);
__global__ void k_dec_down(DecodeArgs a);

// ------------------------------------------------------------------ helpers

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

__device__ __forceinline__ void decode8(uint2 c, __half2 w[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i] = e2m1x2_to_half2((c.x >> (8 * i)) & 0xFF);
    w[4 + i] = e2m1x2_to_half2((c.y >> (8 * i)) & 0xFF);
  }
}

// Exact sum of 16 products of E2M1 values, w as 8 half2 and a pointing at 8
// half2 (16-byte aligned).  Two chains of 4 products: a lane of a chain stays
// within 144 in magnitude and the combined lane within 288, all multiples of
// 1/4, which half precision holds exactly; the two lanes add exactly in fp32.
__device__ __forceinline__ float dot16_h(const __half2 w[8], const __half2* a) {
  const uint4 a0 = *reinterpret_cast<const uint4*>(a);
  const uint4 a1 = *reinterpret_cast<const uint4*>(a + 4);
  const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  __half2 c0 = __hmul2(w[0], *reinterpret_cast<const __half2*>(&aw[0]));
  __half2 c1 = __hmul2(w[1], *reinterpret_cast<const __half2*>(&aw[1]));
#pragma unroll
  for (int i = 2; i < 8; i += 2) {
    c0 = __hfma2(w[i], *reinterpret_cast<const __half2*>(&aw[i]), c0);
    c1 = __hfma2(w[i + 1], *reinterpret_cast<const __half2*>(&aw[i + 1]), c1);
  }
  const __half2 acc = __hadd2(c0, c1);
  return __low2float(acc) + __high2float(acc);
}

__device__ __forceinline__ uint2 pack8(const uint8_t q[8]) {
  uint2 p;
  p.x = q[0] | (q[1] << 8) | (q[2] << 16) | ((uint32_t)q[3] << 24);
  p.y = q[4] | (q[5] << 8) | (q[6] << 16) | ((uint32_t)q[7] << 24);
  return p;
}

// SwiGLU of one 16-block of a pair and its NVFP4 quantisation (global 1.0),
// by the 16 lanes of a half-warp, lane l holding element l: element by
// element the arithmetic of quantize_block16.  The result is stored decoded,
// for the down kernel to use as is: the code's value as a half (values[l])
// and the E4M3 scale's value as an fp32 (*scale).  All 32 lanes of the warp
// must call it; `write` selects the half-warps whose result is stored.
__device__ __forceinline__ void swiglu_quant16(float g, float u, int l, bool write, __half* values,
                                               float* scale) {
  const float h = silu(g) * u;
  float amax = fabsf(h);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o, 16));
  const uint8_t s = e4m3_encode(__fdiv_rn(__fdiv_rn(amax, kE2M1Max), 1.0f));
  const float d = __fmul_rn(e4m3_decode(s), 1.0f);
  uint32_t code = 0;
  if (s != 0 && d != 0.f) code = e2m1x2_encode(__fdiv_rn(h, d), 0.0f) & 0xF;
  if (write) {
    values[l] = __low2half(e2m1x2_to_half2(code));
    if (l == 0) *scale = e4m3_decode(s);
  }
}

// ------------------------------------------------------------------ layouts

// k_dec_route: the router CTAs' quarter partial sums, or, in the last router
// CTA, every logit and bound plus the top-k and sort working sets: per-warp
// token rows, a shared list of (token, candidate expert, compensated logit)
// for the tokens whose top-k needs re-ranking (capacity 4E), and per-token
// bookkeeping.
struct RtSmem {
  int logits_off, err_off, ch_off, le_off, lt_off, lv_off, idx_off, hist_off, scan_off, tok_off, total, cap;
};

__host__ __device__ inline RtSmem rt_smem_layout(int T, int E, int top_k) {
  RtSmem L;
  int o = 0;
  L.cap = 4 * E;
  L.logits_off = o; o += align16(8 * E * 4);      // one token's logits, per warp
  L.err_off = o;    o += align16(8 * E * 4);      // and their bounds
  L.ch_off = o;     o += align16(8 * E);          // chosen flags, per warp
  L.le_off = o;     o += align16(L.cap * 4);      // re-rank list: expert
  L.lt_off = o;     o += align16(L.cap * 4);      //               token
  L.lv_off = o;     o += L.cap * 8;               //               compensated logit
  L.idx_off = o;    o += align16(T * top_k * 4);  // chosen experts of every pair
  L.hist_off = o;   o += align16(8 * E * 4);      // sort histograms
  L.scan_off = o;   o += 32 * 4;
  L.tok_off = o;    o += 32 * 16 + 16;            // per token: state, start, count, lower end
  const int router = 8 * T * 2 * 4;               // quarter partial sums of the router CTAs
  L.total = o > router ? o : router;
  return L;
}

// k_dec_topk: one CTA per token (its logits and bounds, the chosen slots by
// rank, the re-rank candidates), and in the last CTA the counting sort over
// every token (chosen experts of every pair, histograms, scan).
struct TkSmem {
  int lg_off, er_off, sl_off, le_off, lv_off, idx_off, hist_off, scan_off, total;
};

__host__ __device__ inline TkSmem tk_smem_layout(int T, int E, int top_k) {
  TkSmem L;
  int o = 0;
  L.lg_off = o;   o += align16(E * 4);            // logits of the CTA's token
  L.er_off = o;   o += align16(E * 4);            // their bounds
  L.sl_off = o;   o += 4 * 32 * 4;                // chosen by rank: logit, bound, expert, count
  L.le_off = o;   o += align16(E * 4);            // re-rank candidates: expert
  L.lv_off = o;   o += E * 8;                     //                     compensated logit
  L.idx_off = o;  o += align16(T * top_k * 4);    // chosen experts of every pair (sort)
  L.hist_off = o; o += align16(8 * E * 4);        // sort histograms
  L.scan_off = o; o += 32 * 4 + 64;               // scan, flags
  L.total = o;
  return L;
}

// k_dec_gate_up.  A stage holds one item: 16 gate and 16 up rows (codes,
// scales, globals).  Beside it: every token's raw activations (bulk-copied
// once), the current pass's activations as half2 code values and fp32 scales,
// the routing metadata, the touched experts' record pointers and two buffers
// of gate/up dot products.
struct GuSmem {
  int item_bytes, nst;
  int xs_off, xsc_off, xh_off, xsf_off, touched_off, off_off, tok_off, rec_off, g_off, bar_off, total;
};

__host__ __device__ inline GuSmem gu_smem_layout(int H, int T, int E, int P) {
  GuSmem L;
  const int HC = H / 2, NB = H / kBlock;
  L.item_bytes = kGuRows * HC + kGuRows * NB + 128;
  const int fixed = align16(T * HC) + align16(T * NB) + kDecMT * HC * 4 + align16(kDecMT * NB * 4) +
                    align16(E * 4) + align16((E + 1) * 4) + align16(P * 4) + E * 8 + 2 * kDecMT * kGuRows * 4 + 256;
  const int nst = (kDecSmemMax - fixed) / L.item_bytes;
  L.nst = nst > 4 ? 4 : nst;
  int o = (L.nst > 0 ? L.nst : 0) * L.item_bytes;
  L.xs_off = o;      o += align16(T * HC);
  L.xsc_off = o;     o += align16(T * NB);
  L.xh_off = o;      o += kDecMT * HC * 4;
  L.xsf_off = o;     o += align16(kDecMT * NB * 4);
  L.touched_off = o; o += align16(E * 4);
  L.off_off = o;     o += align16((E + 1) * 4);
  L.tok_off = o;     o += align16(P * 4);
  o = (o + 7) & ~7;
  L.rec_off = o;     o += E * 8;
  o = align16(o);
  L.g_off = o;       o += 2 * kDecMT * kGuRows * 4;
  L.bar_off = o;     o += (2 * 4 + 1) * 8;
  L.total = o;
  return L;
}

// k_dec_down.  Work items are (touched expert, up to kDnPairs of its pairs).
// A stage holds the CTA's 16 down rows of the item's expert across the whole
// loaded window (codes, scales, globals) and the item's decoded intermediates
// (half values and fp32 scales); a narrower forward window is read from
// inside the rows.
constexpr int kDnPairs = 4;
struct DnSmem {
  int cpitch, spitch;  // bytes per row of codes / scales in a stage (loaded pitch)
  int coff, soff;      // where the forward window starts inside a staged row
  int hq_off, hs_off;  // intermediates' values / scales inside a stage
  int stage_bytes, nst;
  int shw_off, out_off, touched_off, off_off, tok_off, w_off, ptouched_off, poff_off, rec_off, bar_off, total;
};

__host__ __device__ inline DnSmem dn_smem_layout(int Iw, int row0, int I_loc, int s_I_loc, int T, int E, int P,
                                                 int budget) {
  DnSmem L;
  L.cpitch = Iw / 2;
  L.spitch = Iw / kBlock;
  L.coff = row0 / 2;
  L.soff = row0 / kBlock;
  const int hcp = align16(I_loc * 2), hsp = align16((I_loc / kBlock) * 4);
  const int cbytes = align16(kDnRows * L.cpitch), sbytes = align16(kDnRows * L.spitch);
  L.hq_off = cbytes + sbytes + 64;
  L.hs_off = L.hq_off + kDnPairs * hcp;
  L.stage_bytes = align16(L.hs_off + kDnPairs * hsp);
  const int fixed = align16(kDnRows * s_I_loc * 2) + align16(T * kDnRows * 4) + align16(E * 4) +
                    align16((E + 1) * 4) + align16(P * 4) + align16(P * 4) + align16(E * 4) +
                    align16((E + 1) * 4) + E * 8 + 256;
  const int nst = (budget - fixed) / L.stage_bytes;
  L.nst = nst > 8 ? 8 : nst;
  int o = (L.nst > 0 ? L.nst : 0) * L.stage_bytes;
  L.shw_off = o;      o += align16(kDnRows * s_I_loc * 2);
  L.out_off = o;      o += align16(T * kDnRows * 4);
  L.touched_off = o;  o += align16(E * 4);
  L.off_off = o;      o += align16((E + 1) * 4);
  L.tok_off = o;      o += align16(P * 4);
  L.w_off = o;        o += align16(P * 4);
  L.ptouched_off = o; o += align16(E * 4);
  L.poff_off = o;     o += align16((E + 1) * 4);
  o = (o + 7) & ~7;
  L.rec_off = o;      o += E * 8;
  o = align16(o);
  L.bar_off = o;      o += (2 * 8 + 1) * 8;
  L.total = o;
  return L;
}

__host__ __device__ inline DnSmem dn_smem_choose(int Iw, int row0, int I_loc, int s_I_loc, int T, int E, int P) {
  // two CTAs per SM when three or more stages fit in half the shared memory
  DnSmem L = dn_smem_layout(Iw, row0, I_loc, s_I_loc, T, E, P, 110 * 1024);
  if (L.nst >= 3) return L;
  return dn_smem_layout(Iw, row0, I_loc, s_I_loc, T, E, P, kDecSmemMax);
}

}  // namespace ftmoe
