// Prefill path: routed gate_up and down as grouped block-scaled NVFP4 GEMMs
// on the fifth-generation tensor cores.
//
// For every touched expert e with m_e pairs (sorted positions
// [off_e, off_e + m_e)), the pairs are laid out in a padded order: expert e
// owns rows [pad_e, pad_e + round128(m_e)), so each 128-row tile belongs to
// one expert.
//   gate_up: G[pair][r] = sum_k xq[pair][k] * W_gu[r][k] over r in 64 gate
//            rows and the matching 64 up rows of the window (Issue #62
//            "Offloaded MoE ignores tensor parallelism ...", "What it
//            touches": gate and up rows split as two disjoint row ranges);
//            the epilogue applies the row globals, SwiGLU and the NVFP4
//            quantisation of the intermediate (global 1.0).
//   down:    Y[pair][h] = sum_k hq[pair][k] * W_dn[h][window k] over the
//            window's columns, times the down row global.
// Both are D = A * B^T with the pairs as the 128-row A operand and 128
// weight rows as B: E2M1 codes in shared memory (TMA, 128-byte swizzle),
// E4M3 16-block scales copied into TMEM, fp32 accumulators in TMEM.  The
// products of E2M1 values are exact; scaling and accumulation are fp32.
//
// Kernel roles (one persistent CTA per SM): warp 0 issues TMA, warp 1 owns
// TMEM and issues the MMAs, warps 2-9 drain the accumulators.  Two TMEM
// accumulators let the epilogue of one tile run under the next tile's MMAs.
// Every mbarrier wait is bounded; a wait that runs out stops every role,
// drains what is in flight and frees TMEM.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace ftmoe {

namespace {

constexpr int kPfStages = 5;
constexpr int kPfThreads = 384;    // two producers, MMA, 8 epilogue warps, scale-factor copier
constexpr int kPfEpiWarps = 8;
// The routed gate_up's epilogue (globals, SwiGLU, NVFP4 quantisation of the
// intermediate) is long chains of dependent arithmetic per value; with 8
// warps it, not the copies or the tensor pipe, set the kernel's pace, so that
// mode drains its accumulators with 16 warps, one 16-wide block each.
__host__ __device__ constexpr int pf_epi_warps(int mode) { return mode == 0 ? 16 : kPfEpiWarps; }
// warps: 0 and 3 + epilogue warps the TMA producers (alternate stages), 1
// MMA, 2 .. 1 + epilogue warps the epilogue, 2 + epilogue warps the
// scale-factor copies
__host__ __device__ constexpr int pf_threads(int mode) { return 32 * (4 + pf_epi_warps(mode)); }
constexpr int kTile = 16384;        // one 128 x 128-byte operand tile
constexpr int kSfStage = 2048;      // four 512-byte scale blocks
// shared-memory layout of the 128 x 128 kernels (NS stages)
template <int NS>
struct PfLay {
  static constexpr int A = 0;
  static constexpr int B = NS * kTile;
  static constexpr int Sfa = 2 * NS * kTile;
  static constexpr int Sfb = Sfa + NS * kSfStage;
  static constexpr int Bar = Sfb + NS * kSfStage;
  static constexpr int Glob = Bar + 256;  // per epilogue warp: 128 row globals
  static constexpr int Tab = Glob + kPfEpiWarps * 512;
};
constexpr int kPfOffTab = PfLay<kPfStages>::Tab;
constexpr int kPfMaxE = 1024;
constexpr int kPfMaxK = 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;   // scale-factor columns start after the two accumulators

__host__ __device__ inline int pf_smem_bytes(int E) { return 1024 + kPfOffTab + 3 * 4 * (E + 1); }

// Exclusive scan over n values val(i) by one warp: out[i] = sum_{j<i} val(j),
// out[n] = the total.
template <class F>
__device__ void warp_excl_scan(int n, F val, int* out) {
  const int lane = threadIdx.x & 31;
  const int c = (n + 31) / 32, i0 = lane * c, i1 = min(n, i0 + c);
  int s = 0;
  for (int i = i0; i < i1; ++i) s += val(i);
  int inc = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  int run = inc - s;
  for (int i = i0; i < i1; ++i) {
    out[i] = run;
    run += val(i);
  }
  if (lane == 31) out[n] = inc;
}

// Largest index i in [0, n] with tab[i] <= v (tab non-decreasing, tab[0] <= v).
__device__ __forceinline__ int find_le(const int* tab, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Byte offset of row r's 4 scale bytes inside a 512-byte scale block of 128
// rows: rows r, r+32, r+64, r+96 share a 16-byte line (the order tcgen05.cp
// .32x128b.warpx4 places into TMEM lanes r % 32, columns r / 32).
__host__ __device__ constexpr int sf_slot(int r) { return (r & 31) * 16 + ((r & 127) >> 5) * 4; }

// SiLU with the hardware exponential and reciprocal: the intermediate is
// formed in fp32 (the oracle forms it in fp64), a few ulp either way; the
// quantisation that follows keeps the quantiser's own order.
__device__ __forceinline__ float silu_fast(float z) { return z * __frcp_rn(1.0f + __expf(-z)); }

// 32 bytes to a 32-byte-aligned global address, one 256-bit store (a whole
// sector per lane when the lanes write different rows).
__device__ __forceinline__ void stg_32B(void* p, const uint32_t (&r)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]),
               "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// NVFP4 quantisation of 16 activation values with global 1.0, in the
// quantiser's own order: scale = E4M3(fp32(amax / 6)), then each code =
// E2M1(fp32(v / dec(scale))) with IEEE divisions, so the codes are those the
// same fp32 values give in any other implementation of that order.
__device__ __forceinline__ uint8_t quantize_act16(const float v[16], uint8_t codes[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint8_t s = e4m3_encode(__fdiv_rn(amax, kE2M1Max));
  const float d = e4m3_decode(s);
  if (s == 0 || d == 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0;
    return 0;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) codes[i] = e2m1x2_encode(__fdiv_rn(v[2 * i], d), __fdiv_rn(v[2 * i + 1], d));
  return s;
}

}  // namespace

// ------------------------------------------------------------------ weight scale repack

// Row-major weight scales -> 512-byte blocks for the MMA, per expert:
//   gate_up: tile j = window gate rows [64j, 64j+64) then the matching up
//            rows; blocks [tile][H/64]
//   down:    tile j = rows [128j, 128j+128); blocks [tile][Iw/64]
__global__ void k_repack_sf(uint8_t* bank, RecLayout lay, int H, int Iw, int E) {
  const int gtiles = Iw / 64, gks = H / 64, dtiles = H / 128, dks = Iw / 64;
  const int64_t n_gu = (int64_t)gtiles * gks * 128, n_dn = (int64_t)dtiles * dks * 128;
  const int64_t per = n_gu + n_dn, total = per * E;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / per);
    int64_t k = i % per;
    uint8_t* rec = bank + lay.bytes * e;
    if (k < n_gu) {
      const int n = (int)(k % 128), ks = (int)((k / 128) % gks), j = (int)(k / (128 * gks));
      const int row = n < 64 ? 64 * j + n : Iw + 64 * j + (n - 64);
      const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + lay.gu_scales + (int64_t)row * (H / 16) + 4 * ks);
      *reinterpret_cast<uint32_t*>(rec + lay.gu_sf + ((int64_t)j * gks + ks) * 512 + sf_slot(n)) = w;
    } else {
      k -= n_gu;
      const int n = (int)(k % 128), ks = (int)((k / 128) % dks), j = (int)(k / (128 * dks));
      const int row = 128 * j + n;
      const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + lay.dn_scales + (int64_t)row * (Iw / 16) + 4 * ks);
      *reinterpret_cast<uint32_t*>(rec + lay.dn_sf + ((int64_t)j * dks + ks) * 512 + sf_slot(n)) = w;
    }
  }
}

// ------------------------------------------------------------------ prep

// Padded group starts, and every padded row's activation codes and scale
// blocks in padded order (padding rows get zero scales).
__global__ void __launch_bounds__(256) k_pf_prep(PfArgs a) {
  __shared__ int s_off[kPfMaxE + 1], s_pad[kPfMaxE + 1];
  const int E = a.E, H = a.H;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = a.offsets[e];
  __syncthreads();
  if (threadIdx.x < 32)
    warp_excl_scan(
        E, [&](int e) { return (!a.active || a.active[e]) ? (s_off[e + 1] - s_off[e] + 127) & ~127 : 0; }, s_pad);
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) a.pad_off[e] = s_pad[e];
  const int total = s_pad[E], hc = H / 2, nks = H / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  // codes: eight lanes per padded row, four rows per warp at a time, each
  // lane's loads of its row in flight together (rows past an expert's pairs
  // stay as they are: their MMA rows are never read)
  {
    const int sub = lane >> 3, l8 = lane & 7, n16 = hc / 16;
    for (int p0 = (blockIdx.x * nw + warp) * 4; p0 < total; p0 += gridDim.x * nw * 4) {
      const int pp = p0 + sub;
      int t = -1;
      if (pp < total) {
        const int e = find_le(s_pad, E, pp);
        const int local = pp - s_pad[e];
        if (local < s_off[e + 1] - s_off[e]) t = __ldg(a.perm + s_off[e] + local) / a.top_k;
      }
      if (t >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(a.xq_codes + (int64_t)t * hc);
        uint4* dst = reinterpret_cast<uint4*>(a.xg + (int64_t)pp * hc);
        for (int i0 = l8; i0 < n16; i0 += 8 * 8) {
          uint4 v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (i0 + 8 * c < n16) v[c] = __ldg(src + i0 + 8 * c);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (i0 + 8 * c < n16) dst[i0 + 8 * c] = v[c];
        }
      }
    }
  }
  // scales: a 128-row tile per 128 threads, a thread per row: its token's
  // scales (16-byte loads in flight together), one 4-byte word into each
  // K step's 512-byte block, so every block is written whole; padding rows
  // get zero scales
  const int ntile = total >> 7;
  for (int tile = blockIdx.x * 2 + (threadIdx.x >> 7); tile < ntile; tile += gridDim.x * 2) {
    const int pp = tile * 128 + (threadIdx.x & 127);
    const int e = find_le(s_pad, E, pp);
    const int local = pp - s_pad[e], m = s_off[e + 1] - s_off[e];
    const uint4* src = nullptr;
    if (local < m) src = reinterpret_cast<const uint4*>(a.xq_scales + (int64_t)(a.perm[s_off[e] + local] / a.top_k) * (H / 16));
    uint8_t* dst = a.xg_sf + (int64_t)tile * nks * 512 + sf_slot(pp);
    for (int c0 = 0; c0 < nks / 4; c0 += 8) {  // nks / 4 16-byte groups of 4 K steps
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = (src && c0 + c < nks / 4) ? __ldg(src + c0 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (c0 + c < nks / 4) {
          uint8_t* d = dst + (int64_t)4 * (c0 + c) * 512;
          *reinterpret_cast<uint32_t*>(d) = v[c].x;
          *reinterpret_cast<uint32_t*>(d + 512) = v[c].y;
          *reinterpret_cast<uint32_t*>(d + 1024) = v[c].z;
          *reinterpret_cast<uint32_t*>(d + 1536) = v[c].w;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ grouped GEMM

// One kernel body, four problems (all D = A * B^T, A = 128 token or pair
// rows, B = 128 weight rows, K-major operands in 128-byte swizzled tiles);
// each is also, or only, served by a 128 x 256 kernel where the shapes allow:
//   MODE 0  routed gate_up, NVFP4, grouped by expert; epilogue: row globals,
//           SwiGLU, NVFP4 quantisation of the intermediate (padded order)
//   MODE 1  routed down, NVFP4, grouped; epilogue: down row global -> Y
//   MODE 2  shared gate_up, bf16, one group of T tokens; epilogue: SwiGLU,
//           rounded to bf16 -> hs
//   MODE 4  router logits, bf16: x . (W1 + W2 + W3) with K = 3H (the three
//           exact bf16 parts of the fp32 router rows, x repeated along K);
//           epilogue: bias and the error bound the top-k certificate uses
// A K step is 32 bytes of a row (64 E2M1 or 16 bf16 elements), a K tile 4
// steps (one 128-byte swizzle row).
template <int MODE>
__global__ void __launch_bounds__(pf_threads(MODE), 1)
    k_pf_mma(const __grid_constant__ PfArgs a, const __grid_constant__ CUtensorMap mapA,
             const __grid_constant__ CUtensorMap mapB) {
  constexpr int NS = kPfStages;
  using L = PfLay<NS>;
  constexpr bool kF4 = MODE < 2;
  constexpr int EW = pf_epi_warps(MODE), NT = pf_threads(MODE);
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::Bar);
  uint64_t* empty = full + NS;
  uint64_t* acc_full = empty + NS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* sf_ready = drain + 1;  // [NS] stage landed and its scale blocks are in TMEM
  uint64_t* sf_drain = sf_ready + NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int E = kF4 ? a.E : 1, H = a.H;
  int* s_off = reinterpret_cast<int*>(sm + L::Tab);
  int* s_pad = s_off + (E + 1);
  int* s_up = s_pad + (E + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int I_loc = a.win.I_loc, row0 = a.win.row0, Iw = a.win.Iw;
  static_assert(MODE != 3, "the shared down runs on k_pf_bf16w<3>, the combine on k_pf_combine");
  const int kbytes = MODE == 0 ? H / 2 : MODE == 1 ? I_loc / 2 : MODE == 2 ? 2 * H : 6 * H;
  const int nks_all = kbytes / 32;
  const int nkt = (nks_all + 3) / 4;
  const int J = MODE == 0 ? I_loc / 64 : MODE == 2 ? a.s_I_loc / 64 : MODE == 4 ? a.E / 128 : H / 128;  // weight tiles per row tile

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], EW); }
    mbar_init(drain, 1);
    for (int s = 0; s < NS; ++s) mbar_init(&sf_ready[s], 1);
    mbar_init(sf_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if ((warp == 0 || warp == 3 + EW) && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  if (kF4) {
    for (int e = tid; e <= E; e += NT) {
      s_off[e] = a.offsets[e];
      s_pad[e] = a.pad_off[e];
    }
  } else if (tid == 0) {
    s_off[0] = 0;
    s_off[1] = a.T;
    s_pad[0] = 0;
    s_pad[1] = (a.T + 127) & ~127;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) warp_excl_scan(E, [&](int e) { return ((s_pad[e + 1] - s_pad[e]) >> 7) * J; }, s_up);
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  const int n_units = s_up[E];

  if (warp == 0 || warp == 3 + EW) {
    // ---------------- TMA producers: warp 0 issues the even stages, the
    // other producer the odd ones (a thread's per-stage work -- the wait
    // for the stage to come free, the barrier's expected bytes, the copies
    // one after another -- is longer than the MMA thread's)
    const int pw = warp == 0 ? 0 : 1;
    if (lane == 0) {
      int k = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        const int e = find_le(s_up, E, u), r = u - s_up[e];
        const int nt = r / J, j = r % J;
        const int pp0 = s_pad[e] + nt * 128;
        const int z = kF4 && a.rec_z ? a.rec_z[e] : e;  // record index in the bank / slot pool
        const uint8_t* rec = kF4 ? a.bank + a.lay.bytes * z : nullptr;
        for (int kt = 0; kt < nkt; ++kt, ++k) {
          if ((k & 1) != pw) continue;
          const int s = k % NS;
          if (k >= NS && !mbar_wait(&empty[s], ((k / NS) - 1) & 1, a.status)) {
            *abort_flag = 1;
            break;
          }
          const int nks = min(4, nks_all - 4 * kt);
          unsigned char* sa = sm + L::A + s * kTile;
          unsigned char* sb = sm + L::B + s * kTile;
          unsigned char* sfa = sm + L::Sfa + s * kSfStage;
          unsigned char* sfb = sm + L::Sfb + s * kSfStage;
          mbar_arrive_expect_tx(&full[s], 2 * kTile + (kF4 ? 2 * nks * 512 : 0));
          tma_load_2d(sa, &mapA, MODE == 4 ? (kt * 128) % (2 * H) : kt * 128, pp0, &full[s]);
          if (MODE == 0) {
            tma_load_3d(sb, &mapB, kt * 128, row0 + 64 * j, z, &full[s]);
            tma_load_3d(sb + kTile / 2, &mapB, kt * 128, Iw + row0 + 64 * j, z, &full[s]);
            bulk_g2s(sfa, a.xg_sf + ((int64_t)(pp0 >> 7) * nks_all + 4 * kt) * 512, nks * 512, &full[s]);
            bulk_g2s(sfb, rec + a.lay.gu_sf + ((int64_t)(row0 / 64 + j) * nks_all + 4 * kt) * 512, nks * 512,
                     &full[s]);
          } else if (MODE == 1) {
            tma_load_3d(sb, &mapB, row0 / 2 + kt * 128, 128 * j, z, &full[s]);
            bulk_g2s(sfa, a.hq_sf + ((int64_t)(pp0 >> 7) * nks_all + 4 * kt) * 512, nks * 512, &full[s]);
            bulk_g2s(sfb, rec + a.lay.dn_sf + ((int64_t)j * (Iw / 64) + row0 / 64 + 4 * kt) * 512, nks * 512,
                     &full[s]);
          } else if (MODE == 2) {
            tma_load_2d(sb, &mapB, kt * 128, a.s_row0 + 64 * j, &full[s]);
            tma_load_2d(sb + kTile / 2, &mapB, kt * 128, a.s_Iw + a.s_row0 + 64 * j, &full[s]);
          } else {
            tma_load_2d(sb, &mapB, kt * 128, 128 * j, &full[s]);
          }
        }
      }
      // nothing this warp issued may still be landing when the CTA exits
      for (int q = k - NS > 0 ? k - NS : 0; q < k; ++q)
        if ((q & 1) == pw) mbar_wait(&full[q % NS], (q / NS) & 1, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = kF4 ? idesc_nvf4(128, 128) : idesc_bf16(128, 128);
      int k = 0, ui = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x, ++ui) {
        const int buf = ui & 1;
        if (ui >= 2 && !mbar_wait(&acc_empty[buf], ((ui >> 1) - 1) & 1, a.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d = tmem + buf * 128;
        bool ok = true;
        for (int kt = 0; kt < nkt; ++kt, ++k) {
          const int s = k % NS;
          // NVFP4: the scale-factor warp completes sf_ready[s] once the stage
          // has landed and its scale blocks are in TMEM
          if (!mbar_wait(kF4 ? &sf_ready[s] : &full[s], (k / NS) & 1, a.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const int nks = min(4, nks_all - 4 * kt);
          const uint64_t adesc = sdesc_k_sw128(smem_u32(sm + L::A + s * kTile));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(sm + L::B + s * kTile));
          if (kF4) {
            const uint32_t sfa_col = tmem + kSfCol0 + s * 32, sfb_col = sfa_col + 16;
            for (int ks = 0; ks < nks; ++ks)
              tc_mma_nvf4(d, adesc + 2 * ks, bdesc + 2 * ks, idesc, sfa_col + 4 * ks, sfb_col + 4 * ks,
                          (kt | ks) != 0);
          } else {
            for (int ks = 0; ks < nks; ++ks) tc_mma_bf16(d, adesc + 2 * ks, bdesc + 2 * ks, idesc, (kt | ks) != 0);
          }
          tc_commit(&empty[s]);  // stage free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      // every MMA this thread issued has completed before TMEM is released
      tc_commit(drain);
      mbar_wait(drain, 0, a.status);
    }
  } else if (warp == 2 + EW) {
    // ---------------- scale factors (NVFP4 modes): once a stage has landed,
    // its scale blocks go into that stage's TMEM columns
    if (kF4 && lane == 0) {
      int k = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        for (int kt = 0; kt < nkt; ++kt, ++k) {
          const int s = k % NS;
          if (!mbar_wait(&full[s], (k / NS) & 1, a.status)) { *abort_flag = 1; break; }
          tc_fence_after();
          const int nks = min(4, nks_all - 4 * kt);
          const uint32_t sfa_col = tmem + kSfCol0 + s * 32, sfb_col = sfa_col + 16;
          const uint32_t sfa_smem = smem_u32(sm + L::Sfa + s * kSfStage);
          const uint32_t sfb_smem = smem_u32(sm + L::Sfb + s * kSfStage);
          for (int ks = 0; ks < nks; ++ks) {
            tc_cp_sf(sfa_col + 4 * ks, sdesc_sf(sfa_smem + 512 * ks));
            tc_cp_sf(sfb_col + 4 * ks, sdesc_sf(sfb_smem + 512 * ks));
          }
          tc_commit(&sf_ready[s]);
        }
      }
      tc_commit(sf_drain);
      mbar_wait(sf_drain, 0, a.status);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + EW) {
    // ---------------- epilogue: warp w reads TMEM lanes 32 * (w % 4) ...;
    // the two warps of a lane quarter split the columns in halves
    const int q = warp & 3, hf = (warp - 2) >> 2;
    float* wglob = reinterpret_cast<float*>(sm + L::Glob) + (warp - 2) * 128;
    int ui = 0;
    for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x, ++ui) {
      const int buf = ui & 1;
      const int e = find_le(s_up, E, u), r = u - s_up[e];
      const int nt = r / J, j = r % J;
      const int pp0 = s_pad[e] + nt * 128;
      const int local = nt * 128 + 32 * q + lane;
      const bool valid = local < s_off[e + 1] - s_off[e];
      // the unit's loads that do not need the accumulator are issued before
      // its wait, so their latency overlaps the unit's MMAs: the down
      // rows' globals and the lane's pair index (mode 1)
      float4 pre_g = make_float4(0.f, 0.f, 0.f, 0.f);
      int pre_pr = 0;
      if (MODE == 1) {
        const uint8_t* rec = a.bank + a.lay.bytes * (a.rec_z ? a.rec_z[e] : e);
        pre_g = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(rec + a.lay.dn_global) + 128 * j) +
                      lane);
        if (valid) pre_pr = __ldg(a.perm + s_off[e] + local);
      }
      if (!mbar_wait(&acc_full[buf], (ui >> 1) & 1, a.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * 128;
      if (MODE == 0) {
        // warp (q, cb): pair rows 32q.. and the unit's 16-wide block cb, gate
        // columns 16cb.. and up columns 64 + 16cb..; the rows' globals are
        // read where they are (every lane the same sixteen)
        const int cb = (warp - 2) >> 2;
        const uint8_t* rec = a.bank + a.lay.bytes * (a.rec_z ? a.rec_z[e] : e);
        const float* gglob = reinterpret_cast<const float*>(rec + a.lay.gu_global) + row0 + 64 * j + 16 * cb;
        const float* uglob = gglob + Iw;
        const int pp = pp0 + 32 * q + lane;
        uint32_t g[16], v[16];
        tc_ld16(taddr + 16 * cb, g);
        tc_ld16(taddr + 64 + 16 * cb, v);
        tc_wait16x2(g, v);
        float h[16];
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 gg = __ldg(reinterpret_cast<const float4*>(gglob + i));
          const float4 ug = __ldg(reinterpret_cast<const float4*>(uglob + i));
          h[i] = silu_fast(__uint_as_float(g[i]) * gg.x) * (__uint_as_float(v[i]) * ug.x);
          h[i + 1] = silu_fast(__uint_as_float(g[i + 1]) * gg.y) * (__uint_as_float(v[i + 1]) * ug.y);
          h[i + 2] = silu_fast(__uint_as_float(g[i + 2]) * gg.z) * (__uint_as_float(v[i + 2]) * ug.z);
          h[i + 3] = silu_fast(__uint_as_float(g[i + 3]) * gg.w) * (__uint_as_float(v[i + 3]) * ug.w);
        }
        uint8_t codes[8];
        const uint8_t sc = quantize_act16(h, codes);
        if (valid) {
          uint2 pk;
          pk.x = codes[0] | (codes[1] << 8) | (codes[2] << 16) | ((uint32_t)codes[3] << 24);
          pk.y = codes[4] | (codes[5] << 8) | (codes[6] << 16) | ((uint32_t)codes[7] << 24);
          *reinterpret_cast<uint2*>(a.hq + (int64_t)pp * a.hq_pitch + 32 * j + 8 * cb) = pk;
        }
        a.hq_sf[((int64_t)(pp0 >> 7) * (I_loc / 64) + j) * 512 + lane * 16 + q * 4 + cb] = valid ? sc : 0;
      } else if (MODE == 1) {
        reinterpret_cast<float4*>(wglob)[lane] = pre_g;
        __syncwarp();
        // Y is [token][H / 128 column tiles][slot][128]: a lane's row is
        // pair p = t * k + slot, its tile-j segment at (t * H/128 + j) * k + slot;
        // bf16 when the forward's output is bf16, else fp32
        if (a.y_bf16) {
          uint16_t* Yb = reinterpret_cast<uint16_t*>(a.Y);
          {
            int yseg = 0;
            if (valid) yseg = ((pre_pr / a.top_k) * (H / 128) + j) * a.top_k + pre_pr % a.top_k;
            uint16_t* yrow = Yb + (int64_t)yseg * 128;
#pragma unroll 1
            for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
              uint32_t v[16];
              tc_ld16(taddr + 16 * c, v);
              tc_wait16(v);
              if (valid) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                  const float2 gd = *reinterpret_cast<const float2*>(wglob + 16 * c + i);
                  const __nv_bfloat162 b =
                      __floats2bfloat162_rn(__uint_as_float(v[i]) * gd.x, __uint_as_float(v[i + 1]) * gd.y);
                  pk[i / 2] = *reinterpret_cast<const uint32_t*>(&b);
                }
                stg_32B(yrow + 16 * c, pk);
              }
            }
          }
        } else {
          float* Yf = reinterpret_cast<float*>(a.Y);
          {
            int yseg = 0;
            if (valid) yseg = ((pre_pr / a.top_k) * (H / 128) + j) * a.top_k + pre_pr % a.top_k;
            float* yrow = Yf + (int64_t)yseg * 128;
#pragma unroll 1
            for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
              uint32_t v[16];
              tc_ld16(taddr + 16 * c, v);
              tc_wait16(v);
              if (valid) {
                uint32_t lo[8], hi[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  lo[i] = __float_as_uint(__uint_as_float(v[i]) * wglob[16 * c + i]);
                  hi[i] = __float_as_uint(__uint_as_float(v[8 + i]) * wglob[16 * c + 8 + i]);
                }
                stg_32B(yrow + 16 * c, lo);
                stg_32B(yrow + 16 * c + 8, hi);
              }
            }
          }
        }
      } else if (MODE == 2) {
        const int t = local;
        uint16_t* hrow = a.hs + (int64_t)t * a.s_I_loc + 64 * j;
#pragma unroll 1
        for (int b = 2 * hf; b < 2 * hf + 2; ++b) {
          uint32_t g[16], v[16];
          tc_ld16(taddr + 16 * b, g);
          tc_ld16(taddr + 64 + 16 * b, v);
          tc_wait16x2(g, v);
          if (valid) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(v[2 * i]);
              const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(v[2 * i + 1]);
              const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
              pk[i] = *reinterpret_cast<const uint32_t*>(&hb);
            }
            uint4* dst = reinterpret_cast<uint4*>(hrow + 16 * b);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else if (MODE == 4) {
        // logits of token t for experts [128 j, 128 j + 128) and their bounds
        const int t = local;
        const float xn = valid ? a.xnorm[t] : 0.f;
#pragma unroll 1
        for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
          uint32_t v[16];
          tc_ld16(taddr + 16 * c, v);
          tc_wait16(v);
          if (valid) {
            const int e0 = 128 * j + 16 * c;
            float* lrow = a.logits + (int64_t)t * a.E + e0;
            float* erow = a.err + (int64_t)t * a.E + e0;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 wn = __ldg(reinterpret_cast<const float4*>(a.wnorm + e0 + i));
              float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
              if (a.router_bias) b = __ldg(reinterpret_cast<const float4*>(a.router_bias + e0 + i));
              float4 l, er;
              l.x = __uint_as_float(v[i]) + b.x;
              l.y = __uint_as_float(v[i + 1]) + b.y;
              l.z = __uint_as_float(v[i + 2]) + b.z;
              l.w = __uint_as_float(v[i + 3]) + b.w;
              er.x = a.kappa * xn * wn.x + 2.4e-7f * fabsf(l.x) + 1e-30f;
              er.y = a.kappa * xn * wn.y + 2.4e-7f * fabsf(l.y) + 1e-30f;
              er.z = a.kappa * xn * wn.z + 2.4e-7f * fabsf(l.z) + 1e-30f;
              er.w = a.kappa * xn * wn.w + 2.4e-7f * fabsf(l.w) + 1e-30f;
              *reinterpret_cast<float4*>(lrow + i) = l;
              *reinterpret_cast<float4*>(erow + i) = er;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ routed gate_up, 128 x 256 tiles

// Scale columns stored from registers (tcgen05.st, this warp's 32 TMEM
// lanes).  A block-scaled MMA reads A row m's scales from lane m, column
// base + m/32, and B row n's from lane n % 32 of every lane quarter, column
// base + n/32: a warp of quarter q stores, per K step, its A rows' word
// (atom word q of row `lane`) into all 4 columns of the step, and the whole
// 16-byte atom row `lane` of each B block.
// 16 columns: column 4k + j = a[k].
__device__ __forceinline__ void tc_st_sfa4(uint32_t taddr, const uint32_t (&a)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%2,%2,%2,%2,%3,%3,%3,%3,%4,%4,%4,%4};" ::"r"(taddr),
      "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3])
      : "memory");
}

// 8 columns: b0's four words, then b1's.
__device__ __forceinline__ void tc_st_sfb2(uint32_t taddr, uint4 b0, uint4 b1) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(b0.x),
               "r"(b0.y), "r"(b0.z), "r"(b0.w), "r"(b1.x), "r"(b1.y), "r"(b1.z), "r"(b1.w)
               : "memory");
}

// Wait for this thread's TMEM stores.
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Per-warpgroup register budgets (all four warps of the warpgroup execute
// it).  The increases draw on what the decreases released within the
// block's launch-time registers, so the shares must add up to them.
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// The routed gate_up with 256 weight rows per tile: two consecutive 64 + 64
// (gate, up) window tiles against one 128-row pair tile, one MMA of N = 256
// per K step.  The operand ring's turn-around (TMA latency, the scale and
// MMA hops: about 2.1 us for four stages, about 100 GB/s per SM) bounds an
// SM's intake, so operand bytes per product set the pace: a stage brings
// 48 KB of codes for twice the products of a 128 x 128 tile's 32 KB.  Four
// stages of 54 KB; one accumulator of 256
// TMEM columns, drained into registers by 16 epilogue warps (two 16-wide
// blocks each) before they compute, so the next tile's MMAs start early.
//
// Scale factors go into TMEM by tcgen05.st from four warps, one per lane
// quarter, not by tcgen05.cp: a copy costs about 43 ns of the SM's tensor
// pipe per instruction, and a stage needs twelve, in the same pipe as the
// stage's MMAs.  The 24 warps are six warpgroups: 0 = the TMA producers
// (warps 0 and 2, alternate stages), the MMA thread (warp 1) and an idle
// warp, 1 = the scale warps, 2-5 = the epilogue.  Launched at 80
// registers a thread; warpgroups 0 and 1 give theirs down to 48 so the
// epilogue's rise to 96 (what its drain of 64 accumulator values needs)
// comes out of the same launch budget: 2 x 128 x 48 + 4 x 128 x 96 =
// 768 x 80.
namespace {
constexpr int kGuStages = 4;
constexpr int kGuTileB = 32768;    // 256 x 128-byte weight tile
constexpr int kGuSfb = 4096;       // two tiles' four 512-byte scale blocks
constexpr int kGuEpi = 16;
constexpr int kGuSfW0 = 4;         // first scale warp (warpgroup 1)
constexpr int kGuEpiW0 = 8;        // first epilogue warp (warpgroups 2-5)
constexpr int kGuThreads = 32 * (kGuEpiW0 + kGuEpi);
constexpr int kGuLaunchRegs = 80, kGuLowRegs = 48, kGuEpiRegs = 96;
static_assert(kGuThreads * kGuLaunchRegs == 2 * 128 * kGuLowRegs + kGuEpi * 32 * kGuEpiRegs,
              "the warpgroups' register shares add up to the launch's registers");
constexpr int kGuOffA = 0;
constexpr int kGuOffB = kGuStages * kTile;
constexpr int kGuOffSfa = kGuOffB + kGuStages * kGuTileB;
constexpr int kGuOffSfb = kGuOffSfa + kGuStages * kSfStage;
constexpr int kGuOffBar = kGuOffSfb + kGuStages * kGuSfb;
constexpr int kGuOffTab = kGuOffBar + 256;
constexpr uint32_t kGuSfCol0 = 256;  // after the accumulator; 48 columns per stage
__host__ __device__ inline int gu256_smem_bytes(int E) { return 1024 + kGuOffTab + 3 * 4 * (E + 1); }
}  // namespace

__global__ void __launch_bounds__(kGuThreads, 1)
    k_pf_gu256(const __grid_constant__ PfArgs a, const __grid_constant__ CUtensorMap mapA,
               const __grid_constant__ CUtensorMap mapB) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kGuOffBar);
  uint64_t* empty = full + kGuStages;
  uint64_t* acc_full = empty + kGuStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* sf_ready = drain + 1;  // [kGuStages]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_ready + kGuStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int E = a.E, H = a.H;
  int* s_off = reinterpret_cast<int*>(sm + kGuOffTab);
  int* s_pad = s_off + (E + 1);
  int* s_up = s_pad + (E + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int I_loc = a.win.I_loc, row0 = a.win.row0, Iw = a.win.Iw;
  const int nks_all = H / 64;            // 64-element K steps
  const int nkt = (nks_all + 3) / 4;     // 128-byte K tiles
  const int J2 = I_loc / 128;            // 256-row weight tiles per pair tile

  if (tid == 0) {
    for (int s = 0; s < kGuStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kGuEpi);
    mbar_init(drain, 1);
    for (int s = 0; s < kGuStages; ++s) mbar_init(&sf_ready[s], 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if ((warp == 0 || warp == 2) && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  for (int e = tid; e <= E; e += kGuThreads) {
    s_off[e] = a.offsets[e];
    s_pad[e] = a.pad_off[e];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) warp_excl_scan(E, [&](int e) { return ((s_pad[e + 1] - s_pad[e]) >> 7) * J2; }, s_up);
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  const int n_units = s_up[E];
  if (warp < kGuEpiW0) {
  setmaxnreg_dec<kGuLowRegs>();
  if (warp == 0 || warp == 2) {
    // ---------------- TMA producers: warp 0 issues the even stages, warp 2
    // the odd ones
    const int pw = warp == 0 ? 0 : 1;
    if (lane == 0) {
      int k = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        const int e = find_le(s_up, E, u), r = u - s_up[e];
        const int nt = r / J2, jj = r % J2;
        const int pp0 = s_pad[e] + nt * 128;
        const int z = a.rec_z ? a.rec_z[e] : e;
        const uint8_t* rec = a.bank + a.lay.bytes * z;
        const int t0 = row0 / 64 + 2 * jj;  // first of the unit's two 64 + 64-row window tiles
        for (int kt = 0; kt < nkt; ++kt, ++k) {
          if ((k & 1) != pw) continue;
          const int s = k % kGuStages;
          if (k >= kGuStages && !mbar_wait(&empty[s], ((k / kGuStages) - 1) & 1, a.status)) {
            *abort_flag = 1;
            break;
          }
          const int nks = min(4, nks_all - 4 * kt);
          unsigned char* sa = sm + kGuOffA + s * kTile;
          unsigned char* sb = sm + kGuOffB + s * kGuTileB;
          unsigned char* sfa = sm + kGuOffSfa + s * kSfStage;
          unsigned char* sfb = sm + kGuOffSfb + s * kGuSfb;
          mbar_arrive_expect_tx(&full[s], kTile + kGuTileB + 3 * nks * 512);
          tma_load_2d(sa, &mapA, kt * 128, pp0, &full[s]);
          for (int h = 0; h < 2; ++h) {
            // B rows: gate tile, then its up tile, for each of the two tiles
            tma_load_3d(sb + h * kTile, &mapB, kt * 128, 64 * (t0 + h), z, &full[s]);
            tma_load_3d(sb + h * kTile + kTile / 2, &mapB, kt * 128, Iw + 64 * (t0 + h), z, &full[s]);
            bulk_g2s(sfb + h * kSfStage, rec + a.lay.gu_sf + ((int64_t)(t0 + h) * nks_all + 4 * kt) * 512,
                     nks * 512, &full[s]);
          }
          bulk_g2s(sfa, a.xg_sf + ((int64_t)(pp0 >> 7) * nks_all + 4 * kt) * 512, nks * 512, &full[s]);
        }
      }
      // nothing this warp issued may still be landing when the CTA exits
      for (int q = k - kGuStages > 0 ? k - kGuStages : 0; q < k; ++q)
        if ((q & 1) == pw) mbar_wait(&full[q % kGuStages], (q / kGuStages) & 1, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: one accumulator, N = 256
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4(128, 256);
      int k = 0, ui = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x, ++ui) {
        if (ui >= 1 && !mbar_wait(acc_empty, (ui - 1) & 1, a.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        bool ok = true;
        for (int kt = 0; kt < nkt; ++kt, ++k) {
          const int s = k % kGuStages;
          if (!mbar_wait(&sf_ready[s], (k / kGuStages) & 1, a.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const int nks = min(4, nks_all - 4 * kt);
          const uint64_t adesc = sdesc_k_sw128(smem_u32(sm + kGuOffA + s * kTile));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(sm + kGuOffB + s * kGuTileB));
          const uint32_t sfa_col = tmem + kGuSfCol0 + s * 48, sfb_col = sfa_col + 16;
          for (int ks = 0; ks < nks; ++ks)
            tc_mma_nvf4(tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, sfa_col + 4 * ks, sfb_col + 8 * ks,
                        (kt | ks) != 0);
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(acc_full);
      }
      tc_commit(drain);
      mbar_wait(drain, 0, a.status);
    }
  } else if (warp >= kGuSfW0 && warp < kGuSfW0 + 4) {
    // ---------------- scale factors: warp q = warp % 4 stores, for each K
    // step, its 32 pair rows' scale word into the step's 4 A columns and
    // the 16-byte atom row `lane` of both weight-row blocks into its 8 B
    // columns, once the stage has landed
    const int q = warp & 3;
    int k = 0;
    for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
      bool ok = true;
      for (int kt = 0; kt < nkt; ++kt, ++k) {
        const int s = k % kGuStages;
        bool landed = true;
        if (lane == 0) landed = mbar_wait(&full[s], (k / kGuStages) & 1, a.status);
        if (!__shfl_sync(0xffffffffu, landed, 0)) {
          if (lane == 0) *abort_flag = 1;
          ok = false;
          break;
        }
        // every lane's own acquire of the completed phase (returns at once)
        mbar_wait(&full[s], (k / kGuStages) & 1, a.status);
        const uint32_t* fa = reinterpret_cast<const uint32_t*>(sm + kGuOffSfa + s * kSfStage) + 4 * lane + q;
        const uint4* fb = reinterpret_cast<const uint4*>(sm + kGuOffSfb + s * kGuSfb) + lane;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + kGuSfCol0 + s * 48;
        uint32_t va[4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) va[ks] = fa[128 * ks];
        tc_st_sfa4(tq, va);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) tc_st_sfb2(tq + 16 + 8 * ks, fb[32 * ks], fb[kSfStage / 16 + 32 * ks]);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[s]);
      }
      if (!ok) break;
    }
  }
  } else {
  setmaxnreg_inc<kGuEpiRegs>();
  {
    // ---------------- epilogue: warp (q, part) holds TMEM lanes 32q.. (pair
    // rows) and two 16-wide blocks of window tile t0 + (part >> 1): gate
    // columns 16b.. and up columns 64 + 16b.. for b = 2 (part & 1) + {0, 1}
    const int q = warp & 3, part = (warp - kGuEpiW0) >> 2;
    const int hf = part >> 1, b0 = 2 * (part & 1);
    int ui = 0;
    for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x, ++ui) {
      if (!mbar_wait(acc_full, ui & 1, a.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const int e = find_le(s_up, E, u), r = u - s_up[e];
      const int nt = r / J2, jj = r % J2;
      const int pp0 = s_pad[e] + nt * 128;
      const int local = nt * 128 + 32 * q + lane;
      const bool valid = local < s_off[e + 1] - s_off[e];
      const int tw = 2 * jj + hf;  // the warp's window tile, counted from the forward's window start
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + 128 * hf;
      // the warp's slice into registers, then the accumulator is free
      uint32_t g[2][16], v[2][16];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        tc_ld16(taddr + 16 * (b0 + i), g[i]);
        tc_ld16(taddr + 64 + 16 * (b0 + i), v[i]);
      }
      tc_wait16x2(g[0], v[0]);
      tc_wait16x2(g[1], v[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      const uint8_t* rec = a.bank + a.lay.bytes * (a.rec_z ? a.rec_z[e] : e);
      const float* gglob = reinterpret_cast<const float*>(rec + a.lay.gu_global) + row0 + 64 * tw;
      const float* uglob = gglob + Iw;
      const int pp = pp0 + 32 * q + lane;
      uint32_t sfw = 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int b = b0 + i;
        float h[16];
#pragma unroll
        for (int c = 0; c < 16; c += 4) {
          const float4 gg = __ldg(reinterpret_cast<const float4*>(gglob + 16 * b + c));
          const float4 ug = __ldg(reinterpret_cast<const float4*>(uglob + 16 * b + c));
          h[c] = silu_fast(__uint_as_float(g[i][c]) * gg.x) * (__uint_as_float(v[i][c]) * ug.x);
          h[c + 1] = silu_fast(__uint_as_float(g[i][c + 1]) * gg.y) * (__uint_as_float(v[i][c + 1]) * ug.y);
          h[c + 2] = silu_fast(__uint_as_float(g[i][c + 2]) * gg.z) * (__uint_as_float(v[i][c + 2]) * ug.z);
          h[c + 3] = silu_fast(__uint_as_float(g[i][c + 3]) * gg.w) * (__uint_as_float(v[i][c + 3]) * ug.w);
        }
        uint8_t codes[8];
        const uint8_t sc = quantize_act16(h, codes);
        sfw |= (uint32_t)sc << (8 * i);
        if (valid) {
          uint2 pk;
          pk.x = codes[0] | (codes[1] << 8) | (codes[2] << 16) | ((uint32_t)codes[3] << 24);
          pk.y = codes[4] | (codes[5] << 8) | (codes[6] << 16) | ((uint32_t)codes[7] << 24);
          *reinterpret_cast<uint2*>(a.hq + (int64_t)pp * a.hq_pitch + 32 * tw + 8 * b) = pk;
        }
      }
      *reinterpret_cast<uint16_t*>(a.hq_sf + ((int64_t)(pp0 >> 7) * (I_loc / 64) + tw) * 512 + lane * 16 + q * 4 +
                                   b0) = valid ? (uint16_t)sfw : (uint16_t)0;
    }
  }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

int64_t pf_pad_max(int64_t P, int E) {
  const int64_t groups = P < E ? P : E;
  return ((P + 127 * groups) + 127) / 128 * 128;
}

bool prefill_supported(int H, int E, int I_loc, int Iw, int row0) {
  if (E > kPfMaxE || H % 256 || H > 16384) return false;
  if (I_loc % 64 || row0 % 64 || Iw % 64) return false;
  // every operand row is at least one 128-byte TMA box wide
  if (I_loc < 256 || Iw < 256) return false;
  return pf_smem_bytes(E) <= 227 * 1024;
}

// ------------------------------------------------------------------ bf16 products, 128 x 256 tiles

// The shared expert's gate_up (mode 2) and the router logits (mode 4) with
// 256 weight rows per tile.  One thread issues a tile's MMAs, and at N = 128
// its four MMAs per stage plus the stage's wait and commit take longer than
// the tensor pipe needs for them; at N = 256 the same issue work moves twice
// the products.  No scale factors, so two 256-column accumulators fit in
// TMEM and the epilogue of one tile overlaps the next tile's MMAs.
namespace {
constexpr int kBwStages = 4;
constexpr int kBwTileB = 32768;  // 256 x 128-byte weight tile
constexpr int kBwOffA = 0;
constexpr int kBwOffB = kBwStages * kTile;
constexpr int kBwOffBar = kBwOffB + kBwStages * kBwTileB;
constexpr int kBwThreads = 32 * (2 + kPfEpiWarps);
constexpr int kBwSmem = 1024 + kBwOffBar + 256;
}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kBwThreads, 1)
    k_pf_bf16w(const __grid_constant__ PfArgs a, const __grid_constant__ CUtensorMap mapA,
               const __grid_constant__ CUtensorMap mapB) {
  static_assert(MODE == 2 || MODE == 3 || MODE == 4, "bf16 modes only");
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kBwOffBar);
  uint64_t* empty = full + kBwStages;
  uint64_t* acc_full = empty + kBwStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int nks_all = MODE == 2 ? 2 * H / 32 : MODE == 3 ? 2 * a.s_I_loc / 32 : 6 * H / 32;  // 32-byte K steps
  const int nkt = (nks_all + 3) / 4;
  const int J = MODE == 2 ? a.s_I_loc / 128 : MODE == 3 ? H / 256 : a.E / 256;  // weight tiles per row tile
  // router with few tokens: each (row tile, weight tile) split into KS
  // contiguous K ranges, one unit each
  const int KS = MODE == 4 && a.r_ksplit > 1 ? a.r_ksplit : 1;
  const int n_units = ((a.T + 127) / 128) * J * KS;

  if (tid == 0) {
    for (int s = 0; s < kBwStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], kPfEpiWarps); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int k = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        const int mn = u / KS, ks = u % KS;
        const int nt = mn / J, j = mn % J;
        for (int kt = ks * nkt / KS; kt < (ks + 1) * nkt / KS; ++kt, ++k) {
          const int s = k % kBwStages;
          if (k >= kBwStages && !mbar_wait(&empty[s], ((k / kBwStages) - 1) & 1, a.status)) {
            *abort_flag = 1;
            break;
          }
          unsigned char* sa = sm + kBwOffA + s * kTile;
          unsigned char* sb = sm + kBwOffB + s * kBwTileB;
          mbar_arrive_expect_tx(&full[s], kTile + kBwTileB);
          tma_load_2d(sa, &mapA, MODE == 4 ? (kt * 128) % (2 * H) : kt * 128, nt * 128, &full[s]);
          if (MODE == 2) {
            // gate rows, then the matching up rows, for each of the two 64-row tiles
            for (int h = 0; h < 2; ++h) {
              tma_load_2d(sb + h * kTile, &mapB, kt * 128, a.s_row0 + 128 * j + 64 * h, &full[s]);
              tma_load_2d(sb + h * kTile + kTile / 2, &mapB, kt * 128, a.s_Iw + a.s_row0 + 128 * j + 64 * h,
                          &full[s]);
            }
          } else if (MODE == 3) {
            // output rows [256 j, 256 j + 256) of the shared down, the window's columns
            tma_load_2d(sb, &mapB, 2 * a.s_row0 + kt * 128, 256 * j, &full[s]);
            tma_load_2d(sb + kTile, &mapB, 2 * a.s_row0 + kt * 128, 256 * j + 128, &full[s]);
          } else {
            tma_load_2d(sb, &mapB, kt * 128, 256 * j, &full[s]);
            tma_load_2d(sb + kTile, &mapB, kt * 128, 256 * j + 128, &full[s]);
          }
        }
      }
      for (int q = k - kBwStages > 0 ? k - kBwStages : 0; q < k; ++q)
        mbar_wait(&full[q % kBwStages], (q / kBwStages) & 1, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: two 256-column accumulators
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 256);
      int k = 0, ui = 0;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x, ++ui) {
        const int buf = ui & 1;
        if (ui >= 2 && !mbar_wait(&acc_empty[buf], ((ui >> 1) - 1) & 1, a.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        const int ks = u % KS, kt0 = ks * nkt / KS;
        bool ok = true;
        for (int kt = kt0; kt < (ks + 1) * nkt / KS; ++kt, ++k) {
          const int s = k % kBwStages;
          if (!mbar_wait(&full[s], (k / kBwStages) & 1, a.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const int nks = min(4, nks_all - 4 * kt);
          const uint64_t adesc = sdesc_k_sw128(smem_u32(sm + kBwOffA + s * kTile));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(sm + kBwOffB + s * kBwTileB));
          for (int q = 0; q < nks; ++q) tc_mma_bf16(d, adesc + 2 * q, bdesc + 2 * q, idesc, (kt != kt0) || q != 0);
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      tc_commit(drain);
      mbar_wait(drain, 0, a.status);
    }
  } else {
    // ---------------- epilogue: warp (q, hf) reads TMEM lanes 32q.. and the
    // accumulator's columns [128 hf, 128 hf + 128)
    const int q = warp & 3, hf = (warp - 2) >> 2;
    int ui = 0;
    for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x, ++ui) {
      const int buf = ui & 1;
      if (!mbar_wait(&acc_full[buf], (ui >> 1) & 1, a.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const int mn = u / KS, ks = u % KS;
      const int nt = mn / J, j = mn % J;
      const int t = nt * 128 + 32 * q + lane;
      const bool valid = t < a.T;
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * 256 + 128 * hf;
      if (MODE == 2) {
        // h = silu(gate) * up for intermediate columns [128 j + 64 hf, +64):
        // gate in the half's first 64 columns, up in its last 64
        uint16_t* hrow = a.hs + (int64_t)t * a.s_I_loc + 128 * j + 64 * hf;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          uint32_t g[16], v[16];
          tc_ld16(taddr + 16 * b, g);
          tc_ld16(taddr + 64 + 16 * b, v);
          tc_wait16x2(g, v);
          if (valid) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(v[2 * i]);
              const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(v[2 * i + 1]);
              const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
              pk[i] = *reinterpret_cast<const uint32_t*>(&hb);
            }
            uint4* dst = reinterpret_cast<uint4*>(hrow + 16 * b);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else if (MODE == 3) {
        // the shared expert's output for columns [256 j + 128 hf, +128), in
        // Y's precision (bf16 when the forward's output is bf16), each lane's
        // 16 values of a chunk in whole 32-byte stores
        const int64_t so = (int64_t)t * H + 256 * j + 128 * hf;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[16];
          tc_ld16(taddr + 16 * c, v);
          tc_wait16(v);
          if (valid) {
            if (a.y_bf16) {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const __nv_bfloat162 hb = __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                pk[i] = *reinterpret_cast<const uint32_t*>(&hb);
              }
              stg_32B(reinterpret_cast<uint16_t*>(a.S) + so + 16 * c, pk);
            } else {
              uint32_t lo[8], hi[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                lo[i] = v[i];
                hi[i] = v[8 + i];
              }
              stg_32B(a.S + so + 16 * c, lo);
              stg_32B(a.S + so + 16 * c + 8, hi);
            }
          }
        }
      } else if (KS > 1) {
        // this K range's partial sums for experts [256 j + 128 hf, +128)
        float* prow = a.rpart + ((int64_t)ks * a.T + t) * a.E + 256 * j + 128 * hf;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[16];
          tc_ld16(taddr + 16 * c, v);
          tc_wait16(v);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(prow + 16 * c + i) =
                  make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                              __uint_as_float(v[i + 3]));
          }
        }
      } else {
        // logits of token t for experts [256 j + 128 hf, +128) and their bounds
        const float xn = valid ? a.xnorm[t] : 0.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[16];
          tc_ld16(taddr + 16 * c, v);
          tc_wait16(v);
          if (valid) {
            const int e0 = 256 * j + 128 * hf + 16 * c;
            float* lrow = a.logits + (int64_t)t * a.E + e0;
            float* erow = a.err + (int64_t)t * a.E + e0;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 wn = __ldg(reinterpret_cast<const float4*>(a.wnorm + e0 + i));
              float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
              if (a.router_bias) b = __ldg(reinterpret_cast<const float4*>(a.router_bias + e0 + i));
              float4 l, er;
              l.x = __uint_as_float(v[i]) + b.x;
              l.y = __uint_as_float(v[i + 1]) + b.y;
              l.z = __uint_as_float(v[i + 2]) + b.z;
              l.w = __uint_as_float(v[i + 3]) + b.w;
              er.x = a.kappa * xn * wn.x + 2.4e-7f * fabsf(l.x) + 1e-30f;
              er.y = a.kappa * xn * wn.y + 2.4e-7f * fabsf(l.y) + 1e-30f;
              er.z = a.kappa * xn * wn.z + 2.4e-7f * fabsf(l.z) + 1e-30f;
              er.w = a.kappa * xn * wn.w + 2.4e-7f * fabsf(l.w) + 1e-30f;
              *reinterpret_cast<float4*>(lrow + i) = l;
              *reinterpret_cast<float4*>(erow + i) = er;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The combine, after the shared down wrote S (in Y's precision):
//   out_t = sum_j w_tj * Y[t, slot j] + sigma_t * S_t
// the slots in order (a slot of weight zero adds nothing, whatever its stale
// Y holds), then the shared term, in fp32 (the pages' combine: PR #385
// "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next (offload
// backend)", "What this adds").  A thread takes 8 consecutive columns of a
// token: each slot's piece is one 16-byte load (bf16 Y), and a warp's loads
// cover whole runs of the token's slot segments, so the reads stream
// instead of gathering 32 rows per load.
__global__ void __launch_bounds__(256) k_pf_combine(PfArgs a) {
  const int H = a.H, k = a.top_k;
  const int64_t n8 = (int64_t)a.T * (H / 8);
  for (int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i8 < n8;
       i8 += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = i8 * 8;
    const int t = (int)(i / H), h = (int)(i % H);
    // slot 0's 8 values; slot j's are 128 further
    const int64_t y0 = ((int64_t)t * (H / 128) + h / 128) * k * 128 + (h & 127);
    const float* w = a.topk_w + (int64_t)t * k;
    float o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = 0.f;
    if (k <= 8) {
      float wj[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) wj[q] = q < k ? __ldg(w + q) : 0.f;
      if (a.y_bf16) {
        const uint16_t* Yb = reinterpret_cast<const uint16_t*>(a.Y);
        uint4 y[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          y[q] = q < k ? __ldg(reinterpret_cast<const uint4*>(Yb + y0 + q * 128)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (q < k && wj[q] != 0.f) {
            const uint32_t u[4] = {y[q].x, y[q].y, y[q].z, y[q].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              o[2 * c] = fmaf(wj[q], __uint_as_float(u[c] << 16), o[2 * c]);
              o[2 * c + 1] = fmaf(wj[q], __uint_as_float(u[c] & 0xffff0000u), o[2 * c + 1]);
            }
          }
        }
      } else {
        const float* Yf = reinterpret_cast<const float*>(a.Y);
#pragma unroll
        for (int q0 = 0; q0 < 8; q0 += 4) {
          float4 y[4][2];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q0 + q < k) {
              y[q][0] = __ldg(reinterpret_cast<const float4*>(Yf + y0 + (q0 + q) * 128));
              y[q][1] = __ldg(reinterpret_cast<const float4*>(Yf + y0 + (q0 + q) * 128 + 4));
            } else {
              y[q][0] = y[q][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q0 + q < k && wj[q0 + q] != 0.f) {
              const float v8[8] = {y[q][0].x, y[q][0].y, y[q][0].z, y[q][0].w,
                                   y[q][1].x, y[q][1].y, y[q][1].z, y[q][1].w};
#pragma unroll
              for (int c = 0; c < 8; ++c) o[c] = fmaf(wj[q0 + q], v8[c], o[c]);
            }
          }
        }
      }
    } else {
      for (int q = 0; q < k; ++q) {
        const float wv = __ldg(w + q);
        if (wv == 0.f) continue;
        if (a.y_bf16) {
          const uint4 yv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.Y) + y0 + q * 128));
          const uint32_t u[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            o[2 * c] = fmaf(wv, __uint_as_float(u[c] << 16), o[2 * c]);
            o[2 * c + 1] = fmaf(wv, __uint_as_float(u[c] & 0xffff0000u), o[2 * c + 1]);
          }
        } else {
          const float* yp = reinterpret_cast<const float*>(a.Y) + y0 + q * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) o[c] = fmaf(wv, __ldg(yp + c), o[c]);
        }
      }
    }
    const float sg = __ldg(a.sigma + t);
    float sv[8];
    if (a.y_bf16) {
      const uint4 sb = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.S) + i));
      const uint32_t u[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        sv[2 * c] = __uint_as_float(u[c] << 16);
        sv[2 * c + 1] = __uint_as_float(u[c] & 0xffff0000u);
      }
    } else {
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(a.S + i));
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(a.S + i) + 1);
      sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w;
      sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = fmaf(sg, sv[c], o[c]);
    if ((a.out_flags & 0xff) == 0) {
      uint32_t pk[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(o[2 * c], o[2 * c + 1]);
        pk[c] = *reinterpret_cast<const uint32_t*>(&hb);
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + i) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + i);
      float4 v0 = make_float4(o[0], o[1], o[2], o[3]), v1 = make_float4(o[4], o[5], o[6], o[7]);
      if (a.out_flags & 0x100) {
        const float4 p0 = dst[0], p1 = dst[1];
        v0.x += p0.x; v0.y += p0.y; v0.z += p0.z; v0.w += p0.w;
        v1.x += p1.x; v1.y += p1.y; v1.z += p1.z; v1.w += p1.w;
      }
      dst[0] = v0;
      dst[1] = v1;
    }
  }
}

static cudaError_t encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                          const uint32_t* box) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return cudaErrorNotSupported;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), d, st, b, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool prefill_shared_supported(int H, int s_I_loc, int s_Iw, int s_row0, int top_k) {
  // bf16 rows of at least one 128-byte box, windows in 64-element tiles
  return H % 128 == 0 && s_I_loc % 64 == 0 && s_row0 % 64 == 0 && s_Iw % 64 == 0 && top_k <= kPfMaxK;
}

cudaError_t prefill_make_maps(const PfArgs& a, PfMaps* m) {
  cudaError_t e;
  if (a.x) {
    const uint64_t dims[2] = {(uint64_t)2 * a.H, (uint64_t)a.T}, st[1] = {(uint64_t)2 * a.H};
    const uint32_t box[2] = {128, 128};
    if ((e = encode(&m->x, a.x, 2, dims, st, box)) != cudaSuccess) return e;
  }
  if (a.wcat) {
    const uint64_t dims[2] = {(uint64_t)6 * a.H, (uint64_t)a.E}, st[1] = {(uint64_t)6 * a.H};
    const uint32_t box[2] = {128, 128};
    if ((e = encode(&m->wr, a.wcat, 2, dims, st, box)) != cudaSuccess) return e;
  }
  if (a.sh_gu) {
    const int H = a.H;
    {
      const uint64_t dims[2] = {(uint64_t)2 * H, (uint64_t)2 * a.s_Iw}, st[1] = {(uint64_t)2 * H};
      const uint32_t box[2] = {128, 64};
      if ((e = encode(&m->sgu, a.sh_gu, 2, dims, st, box)) != cudaSuccess) return e;
    }
    {
      const uint64_t dims[2] = {(uint64_t)2 * a.s_I_loc, (uint64_t)a.T}, st[1] = {(uint64_t)2 * a.s_I_loc};
      const uint32_t box[2] = {128, 128};
      if ((e = encode(&m->hs, a.hs, 2, dims, st, box)) != cudaSuccess) return e;
    }
    {
      const uint64_t dims[2] = {(uint64_t)2 * a.s_Iw, (uint64_t)H}, st[1] = {(uint64_t)2 * a.s_Iw};
      const uint32_t box[2] = {128, 128};
      if ((e = encode(&m->sdn, a.sh_dn, 2, dims, st, box)) != cudaSuccess) return e;
    }
  }
  const int H = a.H, Iw = a.win.Iw, I_loc = a.win.I_loc;
  {
    const uint64_t dims[2] = {(uint64_t)H / 2, (uint64_t)a.P_pad_max}, st[1] = {(uint64_t)H / 2};
    const uint32_t box[2] = {128, 128};
    if ((e = encode(&m->xg, a.xg, 2, dims, st, box)) != cudaSuccess) return e;
  }
  {
    const uint64_t dims[3] = {(uint64_t)H / 2, (uint64_t)2 * Iw, (uint64_t)a.n_records};
    const uint64_t st[2] = {(uint64_t)H / 2, (uint64_t)a.lay.bytes};
    const uint32_t box[3] = {128, 64, 1};
    if ((e = encode(&m->gu, a.bank + a.lay.gu_codes, 3, dims, st, box)) != cudaSuccess) return e;
  }
  {
    const uint64_t dims[2] = {(uint64_t)I_loc / 2, (uint64_t)a.P_pad_max}, st[1] = {(uint64_t)a.hq_pitch};
    const uint32_t box[2] = {128, 128};
    if ((e = encode(&m->hq, a.hq, 2, dims, st, box)) != cudaSuccess) return e;
  }
  {
    const uint64_t dims[3] = {(uint64_t)Iw / 2, (uint64_t)H, (uint64_t)a.n_records};
    const uint64_t st[2] = {(uint64_t)Iw / 2, (uint64_t)a.lay.bytes};
    const uint32_t box[3] = {128, 128, 1};
    if ((e = encode(&m->dn, a.bank + a.lay.dn_codes, 3, dims, st, box)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t prefill_set_smem_limits() {
  cudaError_t e;
  const int bytes = pf_smem_bytes(kPfMaxE);
  if ((e = cudaFuncSetAttribute(k_pf_mma<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf_mma<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf_gu256, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf_mma<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf_bf16w<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf_bf16w<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf_bf16w<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwSmem)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_pf_mma<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_repack_sf(uint8_t* bank, const RecLayout& lay, int H, int Iw, int E, cudaStream_t s) {
  if (!lay.gu_sf_bytes) return cudaSuccess;
  k_repack_sf<<<1024, 256, 0, s>>>(bank, lay, H, Iw, E);
  return cudaGetLastError();
}

// The 128 x 256 gate_up kernel divides its launch registers between
// warpgroups; it runs only when compiled at exactly the registers a thread
// that the division adds up to (a larger increase than the launch holds
// would wait forever), else the 128 x 128 kernel takes the routed gate_up.
static bool gu256_launchable() {
  static int state = 0;  // 0 unknown, 1 yes, 2 no
  if (state == 0) {
    cudaFuncAttributes attr;
    const bool ok = cudaFuncGetAttributes(&attr, k_pf_gu256) == cudaSuccess && attr.numRegs == kGuLaunchRegs &&
                    attr.maxThreadsPerBlock >= kGuThreads;
    if (!ok) (void)cudaGetLastError();
    state = ok ? 1 : 2;
  }
  return state == 1;
}

cudaError_t launch_prefill_routed(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s) {
  cudaError_t err;
  {
    int64_t blocks = (a.P_pad_max + 7) / 8;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    FTMOE_PROF_BEGIN("k_pf_prep", s);
    k_pf_prep<<<(int)blocks, 256, 0, s>>>(a);
    FTMOE_PROF_END(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  const int smem = pf_smem_bytes(a.E);
  FTMOE_PROF_BEGIN("k_pf_gate_up", s);
  if (a.win.I_loc % 128 == 0 && gu256_smem_bytes(a.E) <= 227 * 1024 && gu256_launchable())
    k_pf_gu256<<<num_sms, kGuThreads, gu256_smem_bytes(a.E), s>>>(a, m.xg, m.gu);
  else
    k_pf_mma<0><<<num_sms, pf_threads(0), smem, s>>>(a, m.xg, m.gu);
  FTMOE_PROF_END(s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  FTMOE_PROF_BEGIN("k_pf_down", s);
  k_pf_mma<1><<<num_sms, pf_threads(1), smem, s>>>(a, m.hq, m.dn);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

// Each pair's intermediate codes and scales in sorted-position order, from
// the padded pair rows the gate_up epilogue wrote (a scale lives in its
// row tile's 512-byte block of the 64-wide window tile, at sf_slot(row)).
// One warp per sorted position.
__global__ void __launch_bounds__(256) k_pf_export_h(PfArgs a, uint8_t* codes, uint8_t* scales) {
  const int P = a.T * a.top_k, I_loc = a.win.I_loc, hc = I_loc / 2, nb = I_loc / 16;
  const int lane = threadIdx.x & 31;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < P; p += (gridDim.x * blockDim.x) >> 5) {
    const int e = find_le(a.offsets, a.E - 1, p);
    const int pp = a.pad_off[e] + p - a.offsets[e];
    if (codes)
      for (int i = lane; i < hc; i += 32) codes[(int64_t)p * hc + i] = a.hq[(int64_t)pp * a.hq_pitch + i];
    if (scales)
      for (int kb = lane; kb < nb; kb += 32)
        scales[(int64_t)p * nb + kb] =
            a.hq_sf[((int64_t)(pp >> 7) * (I_loc / 64) + kb / 4) * 512 + sf_slot(pp) + (kb & 3)];
  }
}

cudaError_t launch_prefill_export_h(const PfArgs& a, uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t s) {
  if (!codes && !scales) return cudaSuccess;
  k_pf_export_h<<<num_sms * 4, 256, 0, s>>>(a, codes, scales);
  return cudaGetLastError();
}

bool prefill_router_supported(int H, int E) { return E % 128 == 0 && E <= kPfMaxE && H % 64 == 0; }

// Exact split of each fp32 router row into three bf16 parts (w - W1 and
// (w - W1) - W2 are exact in fp32, and the last remainder has at most 8
// significant bits, so W1 + W2 + W3 == w), and an upper bound of its norm.
__global__ void __launch_bounds__(256) k_router_split(const float* __restrict__ w, int H, uint16_t* __restrict__ wcat,
                                                      float* __restrict__ wnorm) {
  const int e = blockIdx.x;
  __shared__ float red[8];
  float q = 0.f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float v = w[(int64_t)e * H + h];
    const __nv_bfloat16 b1 = __float2bfloat16_rn(v);
    const float r1 = __fsub_rn(v, __bfloat162float(b1));
    const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(b2));
    const __nv_bfloat16 b3 = __float2bfloat16_rn(r2);
    uint16_t* row = wcat + (int64_t)e * 3 * H;
    row[h] = *reinterpret_cast<const uint16_t*>(&b1);
    row[H + h] = *reinterpret_cast<const uint16_t*>(&b2);
    row[2 * H + h] = *reinterpret_cast<const uint16_t*>(&b3);
    q = fmaf(v, v, q);
  }
  q = warp_sum(q);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = q;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += red[i];
    wnorm[e] = sqrtf(t) * (1.0f + 1e-5f);
  }
}

cudaError_t launch_router_split(const float* w, int E, int H, uint16_t* wcat, float* wnorm, cudaStream_t s) {
  k_router_split<<<E, 256, 0, s>>>(w, H, wcat, wnorm);
  return cudaGetLastError();
}

// Router logits from the K-split partials: l = sum over the ranges in range
// order + bias, and the bound of the tensor-core sums plus that of the
// KS - 1 fp32 additions (each at most 2^-24 of the sum of the partials'
// magnitudes, which sum to at most ||[x x x]|| ||[W1 W2 W3]|| <= 1.75
// ||x|| ||w|| upper bounds).
__global__ void __launch_bounds__(256) k_router_finish(PfArgs a, int KS) {
  const int E = a.E;
  const int64_t n = (int64_t)a.T * E;
  const float add = (float)(KS - 1) * 1.05e-7f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / E), e = (int)(i % E);
    float l = 0.f;
    for (int ks = 0; ks < KS; ++ks) l += __ldg(a.rpart + (int64_t)ks * n + i);
    if (a.router_bias) l += __ldg(a.router_bias + e);
    const float xw = a.xnorm[t] * __ldg(a.wnorm + e);
    a.logits[i] = l;
    a.err[i] = a.kappa * xw + add * xw + 2.4e-7f * fabsf(l) + 1e-30f;
  }
}

cudaError_t launch_prefill_router(const PfArgs& a0, const PfMaps& m, int num_sms, cudaStream_t s) {
  PfArgs a = a0;
  a.r_ksplit = 1;
  if (a.E % 256 == 0 && a.rpart) {
    // enough units for the SMs: split each tile's K range while there are
    // fewer tiles than SMs (at most 16 ranges, and as many as the buffer holds)
    const int tiles = ((a.T + 127) / 128) * (a.E / 256);
    const int nkt = (6 * a.H / 32 + 3) / 4;
    int ks = num_sms / tiles;
    if (ks > 16) ks = 16;
    if (ks > nkt) ks = nkt;
    while (ks > 1 && (int64_t)ks * a.T * a.E > a.rpart_cap) --ks;
    a.r_ksplit = ks < 1 ? 1 : ks;
  }
  FTMOE_PROF_BEGIN("k_pf_router", s);
  if (a.E % 256 == 0) {
    k_pf_bf16w<4><<<num_sms, kBwThreads, kBwSmem, s>>>(a, m.x, m.wr);
    if (a.r_ksplit > 1 && cudaPeekAtLastError() == cudaSuccess) {
      const int64_t n = (int64_t)a.T * a.E;
      int blocks = (int)((n + 255) / 256);
      if (blocks > num_sms * 8) blocks = num_sms * 8;
      k_router_finish<<<blocks, 256, 0, s>>>(a, a.r_ksplit);
    }
  } else {
    k_pf_mma<4><<<num_sms, kPfThreads, pf_smem_bytes(1), s>>>(a, m.x, m.wr);
  }
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

cudaError_t launch_prefill_shared_gate_up(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s) {
  FTMOE_PROF_BEGIN("k_pf_shared_gate_up", s);
  if (a.s_I_loc % 128 == 0)
    k_pf_bf16w<2><<<num_sms, kBwThreads, kBwSmem, s>>>(a, m.x, m.sgu);
  else
    k_pf_mma<2><<<num_sms, kPfThreads, pf_smem_bytes(1), s>>>(a, m.x, m.sgu);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

// The shared down on 128 x 256 tiles into S (H is a multiple of 256 on the
// prefill path).
cudaError_t launch_prefill_shared_down(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s) {
  if (!a.S || a.H % 256) return cudaErrorInvalidValue;
  FTMOE_PROF_BEGIN("k_pf_shared_down", s);
  k_pf_bf16w<3><<<num_sms, kBwThreads, kBwSmem, s>>>(a, m.hs, m.sdn);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

// The combine, streaming Y, S and the output.
cudaError_t launch_prefill_combine(const PfArgs& a, int num_sms, cudaStream_t s) {
  const int64_t n8 = (int64_t)a.T * (a.H / 8);
  int64_t blocks = (n8 + 255) / 256;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  FTMOE_PROF_BEGIN("k_pf_combine", s);
  k_pf_combine<<<(int)blocks, 256, 0, s>>>(a);
  FTMOE_PROF_END(s);
  return cudaGetLastError();
}

cudaError_t launch_prefill_shared_down_combine(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s) {
  cudaError_t e = launch_prefill_shared_down(a, m, num_sms, s);
  return e != cudaSuccess ? e : launch_prefill_combine(a, num_sms, s);
}

}  // namespace ftmoe
