// Decode path on the tensor cores (1 <= T <= 32 tokens).
//
// At decode sizes the layer is a read of the touched experts' bytes (Issue
// #62 "Offloaded MoE ignores tensor parallelism ...", "Why TP=2 loses
// today"; PR #385 "feat(qwen4_exp): tensor parallelism for
// Qwen3.8-Flash-Next (offload backend)", "Measurements").  Here the weights
// are the 128-row A operand of a block-scaled NVFP4 MMA and the (at most 32)
// tokens are N, so the SMs only issue TMA copies and MMAs while the weight
// bytes stream; E2M1 values never pass through the CUDA cores.
//
//   k_dtc_router     router logits per K chunk on the tensor cores, the
//                    activation codes, sigma and the x-norm bound (or, where
//                    the chunks do not fit, k_dec_route in decode_route.cu)
//   k_dec_topk       (decode_route.cu) one CTA per token: top-k, certificate,
//                    the token's bits in the expert masks
//   k_dtc_gate_up    work units: (touched expert, 64 gate + 64 up window rows)
//                    against every token's resident activation codes, and
//                    (shared expert, 64 + 64 bf16 rows) against bf16 x; the
//                    epilogue picks each pair's column, applies SwiGLU and
//                    quantises the intermediate (NVFP4, global 1.0), or rounds
//                    the shared intermediate to bf16
//   k_dtc_down       CTA (128 output rows, expert group): the group's down
//                    rows against each expert's intermediates, accumulated per
//                    token in a fixed order; one more group holds the shared
//                    expert (bf16) times sigmoid(gate).  The last CTA of an
//                    output tile adds the groups' partials in group order, so
//                    the result does not depend on timing (PR #385,
//                    "Correctness": no value atomics).
#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "tc_common.cuh"

namespace ftmoe {

namespace {

constexpr int kDtThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kDgThreads = 224;  // gate_up: warp 0 TMA, 1 MMA, 2-5 epilogue, 6 scale factors into TMEM
constexpr int kDdThreads = 256;  // down: warp 7 joins only the group reduction
constexpr int kDtSmem = 220 * 1024;
// the down kernel runs two CTAs per SM (each issues its own MMAs), so it
// keeps to half of the shared memory and of TMEM
constexpr int kDdSmem = 112 * 1024;
constexpr uint32_t kDdTmemCols = 256;
// Arrival mark of a down CTA that gave up (a bounded wait ran out): the
// low 16 bits of a tile's counter count arrivals, the high bits count
// CTAs that gave up.
constexpr int kDnGaveUp = 1 << 16;
constexpr int kDtA = 16384;      // 128 weight rows x 128 bytes
constexpr int kDtB = 4096;       // up to 32 token / pair rows x 128 bytes

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return p + ((1024 - (smem_u32(p) & 1023)) & 1023);
}

// ---- k_dtc_gate_up shared memory: stages (A tile, B tile for shared units,
// A scale blocks), every token's activation codes (one [npad][128] box per
// 256-element K tile), their scale blocks, the up values of the epilogue.
// Routing metadata staged once per CTA: touched experts and their record
// pointers, expert offsets, and per sorted position the token (and, for the
// down kernel, the routing weight).
struct Meta {
  int touched_off, z_off, rec_off, off_off, tok_off, w_off, mask_off, scan_off, bytes;
};

__host__ __device__ inline Meta meta_layout(int E, int P, int base) {
  Meta M;
  int o = base;
  M.rec_off = o;     o += E * 8;
  M.touched_off = o; o += align16(E * 4);
  M.z_off = o;       o += align16(E * 4);
  M.off_off = o;     o += align16((E + 1) * 4);
  M.tok_off = o;     o += align16(P * 4);
  M.w_off = o;       o += align16(P * 4);
  M.mask_off = o;    o += align16(E * 4);
  M.scan_off = o;    o += 80 * 4;
  M.bytes = o - base;
  return M;
}

struct DgLayout {
  int npad, nkt, nks, stage, nst, xres_off, sfb_off, u_off, meta_off, bar_off, total;
};

__host__ __device__ inline DgLayout dg_layout(int H, int T, int E, int P) {
  DgLayout L;
  L.npad = T <= 16 ? 16 : 32;
  L.nkt = H / 256;
  L.nks = H / 64;
  // the A tile, then one region: a routed stage's A scale blocks (2 KB) or a
  // shared stage's x tile (npad rows of 128 bytes); 18 or 20 KB, multiples
  // of 1024
  L.stage = kDtA + (L.npad * 128 > 2048 ? L.npad * 128 : 2048);
  const int xres = L.nkt * L.npad * 128, sfb = L.nks * 512, u = 2 * 32 * 64 * 4;
  const int meta = meta_layout(E, P, 0).bytes;
  const int nst = (kDtSmem - 1024 - xres - sfb - u - meta - 512) / L.stage;
  L.nst = nst > 8 ? 8 : nst;
  int o = (L.nst > 0 ? L.nst : 0) * L.stage;
  L.xres_off = o; o += xres;
  L.sfb_off = o;  o += sfb;
  L.u_off = o;    o += u;
  L.meta_off = o; o += meta;
  L.bar_off = o;  o += 512;
  L.total = o + 1024;
  return L;
}

// All threads: stage the routing metadata (after the routing kernels).
// Loads go to L2 (the producing grid ran on other SMs), first-level ones
// together, so a thread waits for two round trips.
__device__ __forceinline__ void stage_meta(const DecodeArgs& a, unsigned char* sm, const Meta& M, int nt) {
  const int E = a.r.E, P = a.T * a.top_k, k = a.top_k;
  int* s_touched = reinterpret_cast<int*>(sm + M.touched_off);
  int* s_z = reinterpret_cast<int*>(sm + M.z_off);
  const uint8_t** s_rec = reinterpret_cast<const uint8_t**>(sm + M.rec_off);
  int* s_off = reinterpret_cast<int*>(sm + M.off_off);
  int* s_tok = reinterpret_cast<int*>(sm + M.tok_off);
  float* s_w = reinterpret_cast<float*>(sm + M.w_off);
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = __ldcg(a.r.offsets + i);
  for (int i = threadIdx.x; i < nt || i < P; i += blockDim.x) {
    const int e = i < nt ? __ldcg(a.r.touched + i) : 0;
    const int p = i < P ? __ldcg(a.r.perm + i) : 0;
    if (i < nt) {
      const int z = a.rec_z ? __ldcg(a.rec_z + e) : e;
      s_touched[i] = e;
      s_z[i] = z;
      s_rec[i] = a.bank + (int64_t)z * a.lay.bytes;
    }
    if (i < P) {
      s_tok[i] = p / k;
      s_w[i] = __ldcg(a.r.topk_w + p);
    }
  }
}

// All threads: the routing tables from the token masks of the top-k kernel
// and the chosen experts.  A token picks an expert at most once, so expert
// e's pairs are its mask's tokens in increasing order: the count is the
// mask's population and pair (t, j) goes to offsets[e] + the mask's tokens
// before t -- the same stable order as a counting sort.  With `globals`
// (one CTA) the offsets, touched list, pair order and telemetry also go to
// HBM.  Returns the number of touched experts.
__device__ int build_meta(const DecodeArgs& a, unsigned char* sm, const Meta& M, bool globals) {
  const int E = a.r.E, k = a.top_k, P = a.T * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  int* s_touched = reinterpret_cast<int*>(sm + M.touched_off);
  int* s_z = reinterpret_cast<int*>(sm + M.z_off);
  const uint8_t** s_rec = reinterpret_cast<const uint8_t**>(sm + M.rec_off);
  int* s_off = reinterpret_cast<int*>(sm + M.off_off);
  int* s_tok = reinterpret_cast<int*>(sm + M.tok_off);
  float* s_w = reinterpret_cast<float*>(sm + M.w_off);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(sm + M.mask_off);
  int* s_scan = reinterpret_cast<int*>(sm + M.scan_off);  // [32] pairs, [32] touched, [1] total touched
  // first-level loads together: the masks and this thread's pairs
  constexpr int kPairs = 8;  // P <= 1024 pairs over at least 128 threads
  int pe[kPairs];
  float pw[kPairs];
#pragma unroll
  for (int m = 0; m < kPairs; ++m) {
    const int p = tid + m * nthr;
    pe[m] = p < P ? __ldcg(a.r.topk_idx + p) : 0;
    pw[m] = p < P ? __ldcg(a.r.topk_w + p) : 0.f;
  }
  for (int e = tid; e < E; e += nthr) s_mask[e] = __ldcg(a.r.emask + e);
  // each thread owns experts [e0, e1) (at most 5: E <= 1024 over >= 224
  // threads); their record indices load with the masks (an offloaded
  // forward's slots; resident, the index is the expert), and a record
  // starts at bank + index * record size
  const int per = (E + nthr - 1) / nthr;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  constexpr int kPer = 5;
  int rz[kPer];
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int e = e0 + m;
    rz[m] = e < e1 ? (a.rec_z ? __ldcg(a.rec_z + e) : e) : 0;
  }
  __syncthreads();
  // pair and touched counts, block scan
  int cnt = 0, tcnt = 0;
  for (int e = e0; e < e1; ++e) {
    const uint32_t msk = s_mask[e];
    cnt += __popc(msk);
    tcnt += msk != 0u;
  }
  int inc = cnt, tinc = tcnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o), tn = __shfl_up_sync(0xffffffffu, tinc, o);
    if (lane >= o) { inc += n; tinc += tn; }
  }
  if (lane == 31) { s_scan[warp] = inc; s_scan[32 + warp] = tinc; }
  __syncthreads();
  int run = inc - cnt, toff = tinc - tcnt;
  for (int w = 0; w < warp; ++w) { run += s_scan[w]; toff += s_scan[32 + w]; }
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int e = e0 + m;
    if (e >= e1) break;
    const uint32_t msk = s_mask[e];
    s_off[e] = run;
    if (globals) a.r.offsets[e] = run;
    if (msk) {
      s_touched[toff] = e;
      s_z[toff] = rz[m];
      s_rec[toff] = a.bank + (int64_t)rz[m] * a.lay.bytes;
      if (globals) a.r.touched[toff] = e;
      ++toff;
    }
    run += __popc(msk);
  }
  if (tid == nthr - 1) {
    s_off[E] = run;
    s_scan[64] = toff;
    if (globals) {
      a.r.offsets[E] = run;
      a.r.n_touched[0] = toff;
      if (a.r.touched_total) atomicAdd(a.r.touched_total, (unsigned long long)toff);
    }
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < kPairs; ++m) {
    const int p = tid + m * nthr;
    if (p < P) {
      int e = pe[m];
      if ((unsigned)e >= (unsigned)E) { set_status(a.r.status, kStatusRange); e = 0; }
      const int t = p / k;
      const int pos = s_off[e] + __popc(s_mask[e] & ((1u << t) - 1u));
      s_tok[pos] = t;
      s_w[pos] = pw[m];
      if (globals) {
        a.r.perm[pos] = p;
        a.r.inv[p] = pos;
      }
    }
  }
  __syncthreads();
  return s_scan[64];
}

// ---- k_dtc_down shared memory: stages (A tile, B tile, A and B scale
// blocks) and the per-token partial sums of the CTA's 128 output rows.
struct DdLayout {
  int npad, stage, nst, part_off, meta_off, bar_off, total;
};

__host__ __device__ inline DdLayout dd_layout(int T, int E, int P) {
  DdLayout L;
  L.npad = T <= 16 ? 16 : 32;
  // A tile, B tile (npad rows of 128 bytes), A and B scale blocks: 22 or 24 KB
  L.stage = kDtA + L.npad * 128 + 2048 + 2048;
  const int part = L.npad * 128 * 4;
  const int meta = meta_layout(E, P, 0).bytes;
  const int nst = (kDdSmem - 1024 - part - meta - 512) / L.stage;
  L.nst = nst > 8 ? 8 : nst;
  int o = (L.nst > 0 ? L.nst : 0) * L.stage;
  L.part_off = o; o += part;
  L.meta_off = o; o += meta;
  L.bar_off = o;  o += 512;
  L.total = o + 1024;
  return L;
}

}  // namespace

// ------------------------------------------------------------------ gate_up

// First routed unit of CTA b (of G) when the CTAs' whole loads are balanced
// in K tiles: the R routed units cost nkt tiles each, and the Js shared
// units (nkt_s tiles each) went round-robin to the CTAs first, so CTAs
// before b ran cum(b) = (Js / G) * b + min(b, Js % G) of them.  With the
// cumulative target b * total / G, the routed units before CTA b are
// (b * total / G - nkt_s * cum(b)) / nkt, clamped to [0, R]; that is
// non-decreasing in b (where it falls, it is below zero) and reaches R at
// b = G.
__device__ __forceinline__ int dtc_split(int b, int G, int R, int nkt, int Js, int nkt_s) {
  if (b >= G) return R;
  const int64_t total = (int64_t)R * nkt + (int64_t)Js * nkt_s;
  const int rem = Js % G;
  const int64_t cum = (int64_t)(Js / G) * b + (b < rem ? b : rem);
  const int64_t num = (int64_t)b * total - (int64_t)G * nkt_s * cum;
  if (num <= 0) return 0;
  const int64_t r = num / ((int64_t)G * nkt);
  return r < R ? (int)r : R;
}

__global__ void __launch_bounds__(kDgThreads, 1)
    k_dtc_gate_up(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap map_gu,
                  const __grid_constant__ CUtensorMap map_xq, const __grid_constant__ CUtensorMap map_sgu,
                  const __grid_constant__ CUtensorMap map_x) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = align1024(sm_raw);
  const int H = a.H, T = a.T, E = a.r.E;
  const DgLayout L = dg_layout(H, T, E, T * a.top_k);
  const Meta M = meta_layout(E, T * a.top_k, L.meta_off);
  const int* s_touched = reinterpret_cast<const int*>(sm + M.touched_off);
  const int* s_z = reinterpret_cast<const int*>(sm + M.z_off);
  const uint8_t* const* s_rec = reinterpret_cast<const uint8_t* const*>(sm + M.rec_off);
  const int* s_off = reinterpret_cast<const int*>(sm + M.off_off);
  const int* s_tok = reinterpret_cast<const int*>(sm + M.tok_off);
  const int NST = L.nst, npad = L.npad;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bar_off);
  uint64_t* empty = full + 8;
  uint64_t* acc_full = empty + 8;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* xbar = acc_empty + 2;
  uint64_t* drain = xbar + 1;
  uint64_t* u_full = drain + 1;   // [2] up values written (the two up warps arrive)
  uint64_t* u_free = u_full + 2;  // [2] up values consumed (the two gate warps arrive)
  uint64_t* sf_ready = u_free + 2;  // [8] stage landed and its weight scales are in TMEM
  uint64_t* sf_drain = sf_ready + 8;
  uint64_t* uq_full = sf_drain + 1;  // [8] phase-1 unit queue: entry written
  volatile int* uq = reinterpret_cast<volatile int*>(uq_full + 8);  // [8] routed unit, -1 = none left
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uq_full + 12);  // after the 8 queue entries
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* U0 = reinterpret_cast<float*>(sm + L.u_off);  // [2][32 pairs][64]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // TMEM columns: accumulators [0, 2 npad), activation scales (4 per K
  // step), then 16 per stage for the weight scales
  const uint32_t kSfbCol = 64, kSfaCol = 64 + 4 * L.nks;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 4); }
    mbar_init(xbar, 1);
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) { mbar_init(&u_full[b], 2); mbar_init(&u_free[b], 2); }
    for (int s = 0; s < NST; ++s) mbar_init(&sf_ready[s], 1);
    mbar_init(sf_drain, 1);
    for (int q = 0; q < 8; ++q) mbar_init(&uq_full[q], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_gu);
    tma_prefetch_desc(&map_xq);
    tma_prefetch_desc(&map_sgu);
    tma_prefetch_desc(&map_x);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int J = a.win.I_loc / 64, Js = (a.sh_gate_up && !a.skip_shared) ? a.s_I_loc / 64 : 0;
  const int nkt_q = H / 64;  // bf16 K tiles of a shared unit (its whole K)
  const int Us = Js;         // shared units: window tiles of 64 gate + 64 up rows
  const int row0 = a.win.row0, Iw = a.win.Iw;
  const uint32_t id_f4 = idesc_nvf4(128, npad), id_bf = idesc_bf16(128, npad);
  // Two phases.  0: the shared expert's units, one whole-K unit per 64 + 64
  // window rows on the first CTAs (they need only x, so they run while the
  // routing kernels still work); 1: after the routing is known, the routed
  // units (touched expert, 64-row window tile), handed out as below.  Ring
  // positions carry over.
  int kk = 0, ui = 0, uu = 0, nt = 0, r0 = 0, R = 0;
  int qn = 0;  // phase-1 unit queue entries this thread has produced or consumed
  // When a whole forward has more routed units than CTAs it hands them out
  // dynamically: each CTA's first unit is fixed (CTAs without a shared unit
  // first), the rest come from a global counter, so CTAs that start late or
  // ran a shared unit simply take fewer.  The producer draws them and passes
  // them to the other roles through a queue of 8 entries (at most about 3
  // units are in flight in a CTA: the ring holds less than a unit and the
  // accumulators two).  With fewer units than CTAs (one token), and for
  // offload batches, a contiguous range per CTA that balances the CTAs'
  // whole loads (dtc_split).
  bool dyn_units = false;
  // the next unit of this role: the static range, or the queue
  auto next_unit = [&](int it, int phase, int* rr) -> bool {
    if (phase == 0 || !dyn_units) {
      if (it >= 0x7fffffff) return false;
      *rr = r0 + it;
      return true;
    }
    const int q = qn & 7;
    if (!mbar_wait(&uq_full[q], (qn >> 3) & 1, a.r.status)) { *abort_flag = 1; return false; }
    ++qn;
    *rr = uq[q];
    return *rr >= 0;
  };
  int rs = 0;         // ring stage of kk (kk mod NST) and its phase parity, kept
  uint32_t rph = 0;   // incrementally: NST is a run-time value and divisions cost
  const int q = warp & 3;
  const bool up = q >= 2;
  const int i = 32 * (q & 1) + lane;
  for (int phase = 0; phase < 2; ++phase) {
    int n_my;
    if (phase == 0) {
      n_my = (int)blockIdx.x < Us ? (Us - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    } else {
      pdl_wait();  // routing and the activation codes
      pdl_launch_dependents();
      if (warp == 0 && lane == 0) {
        // every token's activation codes (they do not depend on the tables)
        mbar_arrive_expect_tx(xbar, L.nkt * npad * 128);
        for (int kt = 0; kt < L.nkt; ++kt)
          tma_load_2d(sm + L.xres_off + kt * npad * 128, &map_xq, kt * 128, 0, xbar);
      }
      if (a.meta_masks) {
        nt = build_meta(a, sm, M, blockIdx.x == 0);
      } else {
        nt = __ldcg(a.r.n_touched);
        stage_meta(a, sm, M, nt);
        __syncthreads();
      }
      if (warp == 6) {
        // activation scale blocks into TMEM (once): lane t stages token t's
        // scales (H/16 bytes, 16-byte loads all in flight) as word t of
        // each K step's block
        unsigned char* sfb = sm + L.sfb_off;
        const uint4* src = reinterpret_cast<const uint4*>(a.r.xq_scales + (int64_t)lane * (H / 16));
        for (int c0 = 0; c0 < L.nks / 4; c0 += 8) {
          uint4 v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) v[c] = (lane < T && c0 + c < L.nks / 4) ? __ldg(src + c0 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (c0 + c < L.nks / 4) {
              const int ks = 4 * (c0 + c);
              *reinterpret_cast<uint32_t*>(sfb + (ks + 0) * 512 + lane * 16) = v[c].x;
              *reinterpret_cast<uint32_t*>(sfb + (ks + 1) * 512 + lane * 16) = v[c].y;
              *reinterpret_cast<uint32_t*>(sfb + (ks + 2) * 512 + lane * 16) = v[c].z;
              *reinterpret_cast<uint32_t*>(sfb + (ks + 3) * 512 + lane * 16) = v[c].w;
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        // the first scale-factor commit of phase 1 covers these copies too
        // (the MMA thread waits for it before its first MMA, so nothing
        // else waits for this warp here)
        if (lane == 0)
          for (int ks = 0; ks < L.nks; ++ks) tc_cp_sf(tmem + kSfbCol + 4 * ks, sdesc_sf(smem_u32(sfb) + 512 * ks));
        __syncwarp();
      }
      R = nt * J;
      dyn_units = a.meta_masks != 0 && R > (int)gridDim.x;
      r0 = dtc_split(blockIdx.x, gridDim.x, R, L.nkt, Us, nkt_q);
      n_my = dyn_units ? 0x7fffffff : dtc_split(blockIdx.x + 1, gridDim.x, R, L.nkt, Us, nkt_q) - r0;
    }
    if (warp == 0) {
      // ---------------- TMA producer
      if (lane == 0) {
        int drawn = 0;  // the counter's answer for the next unit, asked one unit ahead
        for (int it = 0; it < n_my && !*abort_flag; ++it) {
          const bool shared = phase == 0;
          int rr = r0 + it;
          if (!shared && dyn_units) {
            // this CTA's fixed first unit, then draws from the counter (the
            // draw for unit it + 1 goes out when unit it starts, so its round
            // trip overlaps the unit's loads); the unit goes to the other
            // roles through the queue
            const int G = gridDim.x, b = blockIdx.x, Un = min(Us, G);
            if (it == 0) rr = b >= Un ? b - Un : (G - Un) + b;
            else rr = G + drawn;
            if (rr >= R) rr = -1;
            uq[qn & 7] = rr;
            mbar_arrive(&uq_full[qn & 7]);  // release: the entry is visible
            ++qn;
            if (rr < 0) break;
            // the next unit's draw; the stage barriers below arrive without
            // release semantics, so nothing waits for it before the next unit
            drawn = atomicAdd(a.counter, 1);
          }
          const int us = (int)blockIdx.x + it * (int)gridDim.x;  // shared unit
          const int j = shared ? us : rr % J;
          const int z = shared ? 0 : s_z[rr / J];  // record index in the bank / slot pool
          const uint8_t* rec = shared ? nullptr : s_rec[rr / J];
          const int nkt_u = shared ? nkt_q : L.nkt;
          for (int kt = 0; kt < nkt_u; ++kt, ++kk) {
            const int s = rs;
            const uint32_t ph = rph;
            if (++rs == NST) { rs = 0; rph ^= 1; }
            if (kk >= NST && !mbar_wait(&empty[s], ph ^ 1, a.r.status)) { *abort_flag = 1; break; }
            unsigned char* sa = sm + s * L.stage;
            if (shared) {
              mbar_arrive_expect_tx(&full[s], kDtA + npad * 128);
              tma_load_2d(sa, &map_sgu, kt * 128, a.s_row0 + 64 * j, &full[s]);
              tma_load_2d(sa + kDtA / 2, &map_sgu, kt * 128, a.s_Iw + a.s_row0 + 64 * j, &full[s]);
              tma_load_2d(sa + kDtA, &map_x, kt * 128, 0, &full[s]);
            } else {
              mbar_arrive_expect_tx_relaxed(&full[s], kDtA + 2048);
              tma_load_3d(sa, &map_gu, kt * 128, row0 + 64 * j, z, &full[s]);
              tma_load_3d(sa + kDtA / 2, &map_gu, kt * 128, Iw + row0 + 64 * j, z, &full[s]);
              bulk_g2s(sa + kDtA, rec + a.lay.gu_sf + ((int64_t)(row0 / 64 + j) * L.nks + 4 * kt) * 512,
                       2048, &full[s]);
            }
          }
        }
      }
      // the other lanes wait here for lane 0: a lane that went ahead to the
      // next phase's dependency wait would hold the whole warp there
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer
      if (lane == 0) {
        bool ok = phase == 0 || mbar_wait(xbar, 0, a.r.status);
        if (!ok) *abort_flag = 1;
        for (int it = 0; ok && it < n_my && !*abort_flag; ++it, ++ui) {
          const bool shared = phase == 0;
          int rr_unused;
          if (!shared && !next_unit(it, phase, &rr_unused)) break;
          const int nkt_u = shared ? nkt_q : L.nkt;
          const int buf = ui & 1;
          if (ui >= 2 && !mbar_wait(&acc_empty[buf], ((ui >> 1) - 1) & 1, a.r.status)) { *abort_flag = 1; break; }
          tc_fence_after();
          const uint32_t d = tmem + buf * npad;
          for (int kt = 0; kt < nkt_u; ++kt, ++kk) {
            const int s = rs;
            const uint32_t ph = rph;
            if (++rs == NST) { rs = 0; rph ^= 1; }
            if (!mbar_wait(&sf_ready[s], ph, a.r.status)) { *abort_flag = 1; ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(sm + s * L.stage);
            const uint64_t adesc = sdesc_k_sw128(sa);
            if (shared) {
              const uint64_t bdesc = sdesc_k_sw128(sa + kDtA);
              for (int ks = 0; ks < 4; ++ks) tc_mma_bf16(d, adesc + 2 * ks, bdesc + 2 * ks, id_bf, (kt | ks) != 0);
            } else {
              const uint32_t sfa_col = tmem + kSfaCol + 16 * s;
              const uint64_t bdesc = sdesc_k_sw128(smem_u32(sm + L.xres_off + kt * npad * 128));
              for (int ks = 0; ks < 4; ++ks)
                tc_mma_nvf4(d, adesc + 2 * ks, bdesc + 2 * ks, id_f4, sfa_col + 4 * ks,
                            tmem + kSfbCol + 4 * (4 * kt + ks), (kt | ks) != 0);
            }
            tc_commit(&empty[s]);
          }
          if (!ok) break;
          tc_commit(&acc_full[buf]);
        }
      }
      __syncwarp();  // as for the producer warp
    } else if (warp == 6) {
      // ---------------- scale factors: once a stage has landed, its weight
      // scale blocks go into that stage's TMEM columns and sf_ready[s]
      // completes when they are there (for a shared unit's stage, as soon
      // as it has landed), so the MMA thread only issues MMAs
      if (lane == 0) {
        for (int it = 0; it < n_my && !*abort_flag; ++it) {
          const bool shared = phase == 0;
          int rr_unused;
          if (!shared && !next_unit(it, phase, &rr_unused)) break;
          const int nkt_u = shared ? nkt_q : L.nkt;
          for (int kt = 0; kt < nkt_u; ++kt, ++kk) {
            const int s = rs;
            const uint32_t ph = rph;
            if (++rs == NST) { rs = 0; rph ^= 1; }
            if (!mbar_wait(&full[s], ph, a.r.status)) { *abort_flag = 1; break; }
            if (shared) {
              mbar_arrive(&sf_ready[s]);
              continue;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(sm + s * L.stage);
            const uint32_t sfa_col = tmem + kSfaCol + 16 * s;
            for (int ks = 0; ks < 4; ++ks) tc_cp_sf(sfa_col + 4 * ks, sdesc_sf(sa + kDtA + 512 * ks));
            tc_commit(&sf_ready[s]);
          }
        }
      }
      __syncwarp();
    } else {
      // ---------------- epilogue: warp q = w % 4 holds TMEM lanes 32q..32q+31:
      // gate rows (q = 0, 1) and up rows (q = 2, 3) of window index i.
      // The up warps hand their values to the gate warps through a double
      // buffer guarded by mbarriers (bounded waits, so a timeout anywhere
      // cannot strand a warp).  A shared unit's columns are the tokens and
      // its SwiGLU output goes to hs in bf16; a routed unit's columns are its
      // expert's pairs, and the output is quantised to NVFP4.
      for (int it = 0; it < n_my && !*abort_flag; ++it, ++ui) {
        const int buf = ui & 1;
        const bool sh = phase == 0;
        int rr = r0 + it;
        if (!sh && !next_unit(it, phase, &rr)) break;
        const int us = (int)blockIdx.x + it * (int)gridDim.x;
        const int ti = sh ? 0 : rr / J, j = sh ? us : rr % J;
        const int e = sh ? 0 : s_touched[ti];
        const int s0 = sh ? 0 : s_off[e];
        const int m = sh ? T : s_off[e + 1] - s0;  // columns this unit uses
        // the row global is loaded before the accumulator wait
        const float gl =
            sh ? 1.f : reinterpret_cast<const float*>(s_rec[ti] + a.lay.gu_global)[(up ? Iw : 0) + row0 + 64 * j + i];
        if (!mbar_wait(&acc_full[buf], (ui >> 1) & 1, a.r.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * npad;
        bool ok = true;
        const int ub = uu & 1;
        float* U = U0 + ub * 32 * 64;
        if (up) {
          if (uu >= 2 && !mbar_wait(&u_free[ub], ((uu >> 1) - 1) & 1, a.r.status)) ok = false;
          if (ok)
            for (int r = 0; r < m; ++r) U[r * 64 + i] = tc_ld1_wait(taddr + (sh ? r : s_tok[s0 + r])) * gl;
          __syncwarp();
          if (lane == 0) mbar_arrive(&u_full[ub]);
        } else {
          if (!mbar_wait(&u_full[ub], (uu >> 1) & 1, a.r.status)) ok = false;
          if (ok && sh) {
            for (int t = 0; t < m; ++t) {
              const __nv_bfloat16 hb = __float2bfloat16_rn(silu(tc_ld1_wait(taddr + t)) * U[t * 64 + i]);
              a.hs[(int64_t)t * a.s_I_loc + 64 * j + i] = *reinterpret_cast<const uint16_t*>(&hb);
            }
          } else if (ok) {
            for (int r = 0; r < m; ++r) {
              const int pos = s0 + r;
              const float g = tc_ld1_wait(taddr + s_tok[pos]) * gl;
              const float h = silu(g) * U[r * 64 + i];
              // NVFP4 quantisation of the 16-element block held by this half-warp
              float amax = fabsf(h);
#pragma unroll
              for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o, 16));
              const uint8_t sc = e4m3_encode(__fdiv_rn(amax, kE2M1Max));
              const float dsc = e4m3_decode(sc);
              uint32_t code = 0;
              if (sc != 0 && dsc != 0.f) code = e2m1x2_encode(__fdiv_rn(h, dsc), 0.0f) & 0xF;
              // gather the half-warp's 16 nibbles into 8 bytes held by its first lane
              const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
              const uint32_t byte = (code | (hi << 4)) & 0xFF;  // valid on even lanes
              uint32_t w0 = 0, w1 = 0;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                w0 |= (__shfl_sync(0xffffffffu, byte, (lane & 16) + 2 * b) & 0xFF) << (8 * b);
                w1 |= (__shfl_sync(0xffffffffu, byte, (lane & 16) + 8 + 2 * b) & 0xFF) << (8 * b);
              }
              if ((lane & 15) == 0) {
                const int half = lane >> 4;
                *reinterpret_cast<uint2*>(a.hq_codes + (int64_t)pos * a.hq_cpitch + 32 * j + 16 * (q & 1) +
                                          8 * half) = make_uint2(w0, w1);
                a.hsf[((int64_t)ti * J + j) * 512 + r * 16 + 2 * (q & 1) + half] = sc;
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&u_free[ub]);
        }
        ++uu;
        if (!ok) *abort_flag = 1;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
    }
  }
  // drain: nothing may be landing in shared memory, and every MMA and scale
  // copy must be complete, before TMEM is released and the CTA exits
  if (warp == 0 && lane == 0) {
    for (int qq = kk - NST > 0 ? kk - NST : 0; qq < kk; ++qq) mbar_wait(&full[qq % NST], (qq / NST) & 1, a.r.status);
    mbar_wait(xbar, 0, a.r.status);
  }
  if (warp == 1 && lane == 0) {
    tc_commit(drain);
    mbar_wait(drain, 0, a.r.status);
  }
  if (warp == 6 && lane == 0) {
    tc_commit(sf_drain);
    mbar_wait(sf_drain, 0, a.r.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ down

__global__ void __launch_bounds__(kDdThreads, 2)
    k_dtc_down(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap map_dn,
               const __grid_constant__ CUtensorMap map_hq, const __grid_constant__ CUtensorMap map_sdn,
               const __grid_constant__ CUtensorMap map_hs) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = align1024(sm_raw);
  __shared__ int s_last;
  const int H = a.H, T = a.T, E = a.r.E;
  const DdLayout L = dd_layout(T, E, T * a.top_k);
  const Meta M = meta_layout(E, T * a.top_k, L.meta_off);
  const int* s_touched = reinterpret_cast<const int*>(sm + M.touched_off);
  const int* s_z = reinterpret_cast<const int*>(sm + M.z_off);
  const uint8_t* const* s_rec = reinterpret_cast<const uint8_t* const*>(sm + M.rec_off);
  const int* s_off = reinterpret_cast<const int*>(sm + M.off_off);
  const int* s_tok = reinterpret_cast<const int*>(sm + M.tok_off);
  const float* s_w = reinterpret_cast<const float*>(sm + M.w_off);
  const int NST = L.nst, npad = L.npad;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bar_off);
  uint64_t* empty = full + 8;
  uint64_t* acc_full = empty + 8;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* sf_ready = drain + 1;  // [8] stage landed and its scale blocks are in TMEM
  uint64_t* sf_drain = sf_ready + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* part = reinterpret_cast<float*>(sm + L.part_off);  // [32 tokens][128 rows]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ht = blockIdx.x, g = blockIdx.y;
  const uint64_t wlim = a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs;
  const bool withhold = a.withhold_first_stage && ht == 0 && g == 0;  // test of the failure path
  const bool has_shared = a.sh_down != nullptr && !a.skip_shared;
  const int G = gridDim.y - (has_shared ? 1 : 0);  // routed expert groups
  const bool shared = has_shared && g == G;
  const int I_loc = a.win.I_loc, row0 = a.win.row0, Iw = a.win.Iw;
  const int nks_r = I_loc / 64, nkt_r = (nks_r + 3) / 4;
  const int nkt_s = a.s_I_loc / 64;  // bf16 K tiles of the shared down (K = s_I_loc)
  const uint32_t kSfCol = 64;         // after the accumulators; 32 per stage

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 4); }
    mbar_init(drain, 1);
    for (int s = 0; s < NST; ++s) mbar_init(&sf_ready[s], 1);
    mbar_init(sf_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_dn);
    tma_prefetch_desc(&map_hq);
    tma_prefetch_desc(&map_sdn);
    tma_prefetch_desc(&map_hs);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kDdTmemCols);
  for (int i2 = tid; i2 < npad * 128; i2 += blockDim.x) part[i2] = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the next grid (the next forward's router) may launch once every CTA here
  // holds its TMEM; it waits for this grid before it touches anything this
  // grid reads or writes
  pdl_launch_dependents();
  // The routing metadata is read before this grid's dependency wait: the
  // routing kernels completed (and their writes were made visible) before
  // the gate_up kernel that launched this grid passed its own wait.
  int nt;
  if (a.meta_masks) {
    nt = build_meta(a, sm, M, false);
  } else {
    nt = __ldcg(a.r.n_touched);
    stage_meta(a, sm, M, nt);
    __syncthreads();
  }
  const int ti0 = shared ? 0 : (int)((int64_t)g * nt / G), ti1 = shared ? 1 : (int)((int64_t)(g + 1) * nt / G);
  const int n_items = ti1 - ti0;

  if (warp == 0) {
    if (lane == 0) {
      // Stage s of K tile kt of item it: the weight part (down rows and their
      // scales; the shared expert's bf16 columns) and the activation part
      // (the item's intermediates and their scales; the bf16 hs).
      auto issue = [&](int s, int it, int kt, bool expect, bool weights, bool acts) {
        const int ti = ti0 + it;
        unsigned char* sa = sm + s * L.stage;
        if (shared) {
          if (expect) mbar_arrive_expect_tx(&full[s], kDtA + npad * 128);
          if (weights) tma_load_2d(sa, &map_sdn, 2 * a.s_row0 + kt * 128, 128 * ht, &full[s]);
          if (acts) tma_load_2d(sa + kDtA, &map_hs, kt * 128, 0, &full[s]);
        } else {
          const int nks = min(4, nks_r - 4 * kt);
          if (expect) mbar_arrive_expect_tx(&full[s], kDtA + npad * 128 + 2 * nks * 512);
          if (weights) {
            tma_load_3d(sa, &map_dn, row0 / 2 + kt * 128, 128 * ht, s_z[ti], &full[s]);
            bulk_g2s(sa + kDtA + npad * 128, s_rec[ti] + a.lay.dn_sf + ((int64_t)ht * (Iw / 64) + row0 / 64 + 4 * kt) * 512,
                     nks * 512, &full[s]);
          }
          if (acts) {
            tma_load_2d(sa + kDtA, &map_hq, kt * 128, s_off[s_touched[ti]], &full[s]);
            bulk_g2s(sa + kDtA + npad * 128 + 2048, a.hsf + ((int64_t)ti * nks_r + 4 * kt) * 512, nks * 512, &full[s]);
          }
        }
      };
      const int nkt_u = shared ? nkt_s : nkt_r;
      // the weights of the first NST K tiles stream before the dependency
      // wait (they do not depend on the gate_up kernel) ...
      const int pre = min(NST, n_items * nkt_u);
      // (a withheld first stage gets no arrival and no copy at all: every
      // wait on it runs out)
      for (int k2 = withhold ? 1 : 0; k2 < pre; ++k2) issue(k2, k2 / nkt_u, k2 % nkt_u, true, true, false);
      pdl_wait();  // the intermediates of the gate_up kernel
      // ... their activations after it, then the ring as usual
      for (int k2 = withhold ? 1 : 0; k2 < pre; ++k2) issue(k2, k2 / nkt_u, k2 % nkt_u, false, false, true);
      int kk = pre, rs = pre == NST ? 0 : pre;  // ring position, its stage and phase parity
      uint32_t rph = pre == NST ? 1 : 0;
      for (int it = kk / nkt_u; it < n_items && !*abort_flag; ++it) {
        for (int kt = (it == pre / nkt_u) ? pre % nkt_u : 0; kt < nkt_u; ++kt, ++kk) {
          const int s = rs;
          const uint32_t ph = rph;
          if (++rs == NST) { rs = 0; rph ^= 1; }
          if (kk >= NST && !mbar_wait(&empty[s], ph ^ 1, a.r.status, wlim)) { *abort_flag = 1; break; }
          issue(s, it, kt, true, true, true);
        }
      }
      for (int q = kk - NST > 0 ? kk - NST : 0; q < kk; ++q) mbar_wait(&full[q % NST], (q / NST) & 1, a.r.status, wlim);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_f4 = idesc_nvf4(128, npad), id_bf = idesc_bf16(128, npad);
      int kk = 0, rs = 0;
      uint32_t rph = 0;
      bool ok = true;
      for (int it = 0; it < n_items && !*abort_flag; ++it) {
        const int buf = it & 1;
        if (it >= 2 && !mbar_wait(&acc_empty[buf], ((it >> 1) - 1) & 1, a.r.status, wlim)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d = tmem + buf * npad;
        const int nkt_u = shared ? nkt_s : nkt_r;
        for (int kt = 0; kt < nkt_u; ++kt, ++kk) {
          const int s = rs;
          const uint32_t ph = rph;
          if (++rs == NST) { rs = 0; rph ^= 1; }
          if (!mbar_wait(&sf_ready[s], ph, a.r.status, wlim)) { *abort_flag = 1; ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(sm + s * L.stage);
          const uint64_t adesc = sdesc_k_sw128(sa), bdesc = sdesc_k_sw128(sa + kDtA);
          if (shared) {
            for (int ks = 0; ks < 4; ++ks) tc_mma_bf16(d, adesc + 2 * ks, bdesc + 2 * ks, id_bf, (kt | ks) != 0);
          } else {
            const int nks = min(4, nks_r - 4 * kt);
            const uint32_t sfa_col = tmem + kSfCol + 32 * s, sfb_col = sfa_col + 16;
            for (int ks = 0; ks < nks; ++ks)
              tc_mma_nvf4(d, adesc + 2 * ks, bdesc + 2 * ks, id_f4, sfa_col + 4 * ks, sfb_col + 4 * ks,
                          (kt | ks) != 0);
          }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      tc_commit(drain);
      mbar_wait(drain, 0, a.r.status, wlim);
    }
  } else if (warp == 6) {
    // ---------------- scale factors: once a stage has landed, its weight
    // and intermediate scale blocks go into that stage's TMEM columns and
    // sf_ready[s] completes when they are there (for the shared group's
    // stages, as soon as they have landed)
    if (lane == 0) {
      int kk = 0, rs = 0;
      uint32_t rph = 0;
      for (int it = 0; it < n_items && !*abort_flag; ++it) {
        const int nkt_u = shared ? nkt_s : nkt_r;
        for (int kt = 0; kt < nkt_u; ++kt, ++kk) {
          const int s = rs;
          const uint32_t ph = rph;
          if (++rs == NST) { rs = 0; rph ^= 1; }
          if (!mbar_wait(&full[s], ph, a.r.status, wlim)) { *abort_flag = 1; break; }
          if (shared) {
            mbar_arrive(&sf_ready[s]);
            continue;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sm + s * L.stage);
          const int nks = min(4, nks_r - 4 * kt);
          const uint32_t sfa_col = tmem + kSfCol + 32 * s, sfb_col = sfa_col + 16;
          for (int ks = 0; ks < nks; ++ks) {
            tc_cp_sf(sfa_col + 4 * ks, sdesc_sf(sa + kDtA + npad * 128 + 512 * ks));
            tc_cp_sf(sfb_col + 4 * ks, sdesc_sf(sa + kDtA + npad * 128 + 2048 + 512 * ks));
          }
          tc_commit(&sf_ready[s]);
        }
      }
      tc_commit(sf_drain);
      mbar_wait(sf_drain, 0, a.r.status, wlim);
    }
    __syncwarp();
  } else if (warp == 7) {
    // only the group reduction below (its loads spread over one more warp)
  } else {
    // ---------------- epilogue: thread = output row h of the tile, TMEM lane h
    const int q = warp & 3, h = 32 * q + lane;
    const int hg = 128 * ht + h;
    const float sig = (shared && lane < T) ? a.r.sigma[lane] : 0.f;
    for (int it = 0; it < n_items && !*abort_flag; ++it) {
      const int buf = it & 1;
      const int e = shared ? 0 : s_touched[ti0 + it];
      const int s0 = shared ? 0 : s_off[e], m = shared ? 0 : s_off[e + 1] - s0;
      // the row global is loaded before the accumulator wait
      const float gd = shared ? 0.f : reinterpret_cast<const float*>(s_rec[ti0 + it] + a.lay.dn_global)[hg];
      if (!mbar_wait(&acc_full[buf], (it >> 1) & 1, a.r.status, wlim)) { *abort_flag = 1; break; }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * npad;
      if (shared) {
        for (int t = 0; t < T; ++t) part[t * 128 + h] = __shfl_sync(0xffffffffu, sig, t) * tc_ld1_wait(taddr + t);
      } else {
        for (int r = 0; r < m; ++r) {
          const int t = s_tok[s0 + r];
          part[t * 128 + h] = fmaf(s_w[s0 + r], gd * tc_ld1_wait(taddr + r), part[t * 128 + h]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    // this group's partials gpart[g][tile][t][128], then the last CTA of
    // the tile adds all groups in group order.  Whether this CTA gave up is
    // decided once (the flag may still be raised by another role), and every
    // CTA arrives on the tile's counter, a CTA that gave up with a mark in
    // the high half: the count always reaches the number of groups, so the
    // last arriver always clears the counter for the next launch, and it
    // writes the output only if no group of the tile gave up.
    named_barrier(1, 128);
    if (tid == 64) s_last = *abort_flag;
    named_barrier(1, 128);
    const bool gave_up = s_last != 0;
    if (!gave_up) {
      float* gp = a.gpart + ((int64_t)g * gridDim.x + ht) * T * 128;
      for (int t = 0; t < T; ++t) gp[t * 128 + h] = part[t * 128 + h];
      __threadfence();
    }
    named_barrier(1, 128);
    if (tid == 64) {
      const int old = atomicAdd(&a.dn_counter[ht], gave_up ? (1 + kDnGaveUp) : 1);
      const bool last = (old & (kDnGaveUp - 1)) == (int)gridDim.y - 1;
      const bool clean = old < kDnGaveUp && !gave_up;
      s_last = last ? (clean ? 1 : 2) : 0;
    }
    named_barrier(1, 128);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kDdTmemCols);
  }
  if (s_last == 2) {
    // a group of this tile gave up (its timeout is in the status word): no
    // output, only the counter cleared for the next launch
    if (tid == 64) a.dn_counter[ht] = 0;
  } else if (s_last == 1) {
    // every thread of the last CTA: items (token, 4 output rows), each the
    // sum over the groups in group order, with the groups' loads in flight
    // together
    __threadfence();
    const int ng = gridDim.y;
    const float4* g4 = reinterpret_cast<const float4*>(a.gpart);
    const int64_t gstride = (int64_t)gridDim.x * T * 32;  // float4s per group
    for (int item = tid; item < T * 32; item += blockDim.x) {
      const int t = item >> 5, c4 = item & 31;
      const float4* src = g4 + ((int64_t)ht * T + t) * 32 + c4;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int g0 = 0; g0 < ng; g0 += 16) {
        float4 v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (g0 + k < ng) v[k] = __ldcg(src + (g0 + k) * gstride);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (g0 + k < ng) { o.x += v[k].x; o.y += v[k].y; o.z += v[k].z; o.w += v[k].w; }
      }
      const int64_t idx = (int64_t)t * H + 128 * ht + 4 * c4;
      if ((a.out_flags & 0xff) == 0) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + idx) = pk;
      } else if (a.out_flags & 0x100) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx);
        float4 c = *dst;
        c.x += o.x; c.y += o.y; c.z += o.z; c.w += o.w;
        *dst = c;
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx) = o;
      }
    }
    if (tid == 64) a.dn_counter[ht] = 0;  // ready for the next launch
  }
}

// ------------------------------------------------------------------ router

// Router logits on the tensor cores, split over K: CTA (128-expert tile m,
// K chunk c) forms rpart[c][t][128 m + r] = sum over the chunk of
// x[t] . [W1 | W2 | W3][128 m + r] (x repeated along K; the three bf16 parts
// add up to the fp32 router row exactly).  Further CTAs quantise the
// activations (global 1.0), and the last ones compute, one warp per token,
// sigma = sigmoid(g . x) and an upper bound of ||x||.
constexpr int kRtKc = 4;  // K tiles per router CTA (all in flight at once)
constexpr int kSgBatch = 12;  // 16-byte pieces of x and g per lane in flight (sigma CTAs; H <= 3072 in one go)

__device__ __forceinline__ int rt_units(int H, int E) {
  const int nkt = 6 * H / 128;
  return (E / 128) * ((nkt + kRtKc - 1) / kRtKc);
}
__host__ __device__ inline int rt_xq_ctas(int T, int H) {
  const int nb = T * (H / kBlock);
  const int n = (nb + kDtThreads - 1) / kDtThreads;
  return n < 1 ? 1 : (n > 64 ? 64 : n);
}

__global__ void __launch_bounds__(kDtThreads)
    k_dtc_router(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap map_wr,
                 const __grid_constant__ CUtensorMap map_x) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = align1024(sm_raw);
  const int H = a.H, T = a.T, E = a.r.E;
  const int npad = T <= 16 ? 16 : 32;
  const int nkt = 6 * H / 128, C = (nkt + kRtKc - 1) / kRtKc;
  const int n_units = (E / 128) * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  // Every CTA lets the next kernels launch only after its own dependency
  // wait: the expert kernel launched after the top-k kernel reads x and
  // writes its shared-expert buffers before its own wait, so the grid
  // before this one (which may have written x, or still read those
  // buffers) must have ended by then.  (Unit CTAs also hold their TMEM by
  // then, so no CTA of a later grid can take it first.)
  if (b < n_units) {
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kRtKc * (kDtA + kDtB));
    uint64_t* accb = full + kRtKc;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
    const int m = b / C, c = b % C;
    const int kt0 = c * kRtKc, nk = min(kRtKc, nkt - kt0);
    if (tid == 0) {
      for (int i = 0; i < kRtKc; ++i) mbar_init(&full[i], 1);
      mbar_init(accb, 1);
      fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // every tile of the chunk at once: the router tiles before this grid's
    // dependency wait (they are weights), x after it
    if (warp == 0 && lane == 0) {
      for (int i = 0; i < nk; ++i) {
        mbar_arrive_expect_tx(&full[i], kDtA + npad * 128);
        tma_load_2d(sm + i * (kDtA + kDtB), &map_wr, (kt0 + i) * 128, 128 * m, &full[i]);
      }
    }
    __syncwarp();
    pdl_wait();  // x, and rpart (the grid before this one may still read it)
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
      for (int i = 0; i < nk; ++i)
        tma_load_2d(sm + i * (kDtA + kDtB) + kDtA, &map_x, ((kt0 + i) * 128) % (2 * H), 0, &full[i]);
    } else if (warp == 1 && lane == 0) {
      const uint32_t id = idesc_bf16(128, npad);
      for (int i = 0; i < nk; ++i) {
        if (!mbar_wait(&full[i], 0, a.r.status)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(sm + i * (kDtA + kDtB));
        const uint64_t adesc = sdesc_k_sw128(sa), bdesc = sdesc_k_sw128(sa + kDtA);
        for (int ks = 0; ks < 4; ++ks) tc_mma_bf16(tmem, adesc + 2 * ks, bdesc + 2 * ks, id, (i | ks) != 0);
      }
      tc_commit(accb);  // every MMA this thread issued
    } else if (warp >= 2) {
      const int q = warp & 3, row = 32 * q + lane;
      const bool ok = mbar_wait(accb, 0, a.r.status);
      tc_fence_after();
      if (ok) {
        float* dst = a.rpart + (int64_t)c * T * E + 128 * m + row;
        for (int t = 0; t < T; ++t) dst[(int64_t)t * E] = tc_ld1_wait(tmem + ((uint32_t)(32 * q) << 16) + t);
      }
    }
    if (warp == 0 && lane == 0)  // nothing may still be landing when the CTA exits
      for (int i = 0; i < nk; ++i) mbar_wait(&full[i], 0, a.r.status);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, 32);
    }
    return;
  }
  pdl_wait();  // x, and the buffers below, belong to the grid before this one until it ends
  pdl_launch_dependents();
  const int nxq = rt_xq_ctas(T, H);
  if (b < n_units + nxq) {
    // a slice of the activation quantisation
    const int nb = T * (H / kBlock);
    const int per = (nb + nxq - 1) / nxq;
    const int q0 = (b - n_units) * per, q1 = min(nb, q0 + per);
    for (int blk = q0 + tid; blk < q1; blk += kDtThreads) {
      float v[16];
      const uint4* p = reinterpret_cast<const uint4*>(a.r.x + (int64_t)blk * kBlock);
      const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
      const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) {
        v[2 * qq] = __uint_as_float(words[qq] << 16);
        v[2 * qq + 1] = __uint_as_float(words[qq] & 0xffff0000u);
      }
      uint8_t cq[8];
      const uint8_t sc = quantize_block16(v, 1.0f, cq);
      *reinterpret_cast<uint2*>(a.r.xq_codes + (int64_t)blk * 8) = pack8(cq);
      a.r.xq_scales[blk] = sc;
    }
    return;
  }
  // the token masks of the top-k kernel start empty, and so does the
  // gate_up kernel's unit counter
  const int b0 = b - n_units - nxq;  // sigma CTA index
  if (b0 == 0) {
    if (a.r.emask)
      for (int e = tid; e < E; e += kDtThreads) a.r.emask[e] = 0u;
    if (a.meta_masks && tid == 0) *a.counter = 0;
  }
  // sigma_t = sigmoid(g . x_t) and an upper bound of ||x_t||, one warp per
  // token (kDtThreads / 32 tokens per CTA), kSgBatch 16-byte pieces of x
  // and of g per lane in flight at a time
  const int t = b0 * (kDtThreads / 32) + warp;
  if (t >= T) return;
  const uint4* xr = reinterpret_cast<const uint4*>(a.r.x + (int64_t)t * H);
  const uint4* gr = reinterpret_cast<const uint4*>(a.r.sh_gate);
  float z = 0.f, q = 0.f;
  for (int i0 = 0; i0 < H / 8; i0 += 32 * kSgBatch) {
    uint4 xv[kSgBatch], gv[kSgBatch];
#pragma unroll
    for (int k = 0; k < kSgBatch; ++k) {
      const int i = i0 + 32 * k + lane;
      xv[k] = i < H / 8 ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
      gv[k] = (gr && i < H / 8) ? __ldg(gr + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kSgBatch; ++k) {
      const uint32_t xw[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
      const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        const float lo = __uint_as_float(xw[k2] << 16), hi = __uint_as_float(xw[k2] & 0xffff0000u);
        z = fmaf(lo, __uint_as_float(gw[k2] << 16), z);
        z = fmaf(hi, __uint_as_float(gw[k2] & 0xffff0000u), z);
        q = fmaf(lo, lo, q);
        q = fmaf(hi, hi, q);
      }
    }
  }
  z = warp_sum(z);
  q = warp_sum(q);
  if (lane == 0) {
    a.r.sigma[t] = gr ? 1.0f / (1.0f + expf(-z)) : 0.f;
    a.r.xnorm[t] = sqrtf(q) * (1.0f + 1e-5f);
  }
}

// ------------------------------------------------------------------ host side

int decode_tc_groups(int H, int num_sms) {
  const int tiles = H / 128;
  int g = 2 * num_sms / tiles - 1;  // routed groups (two CTAs per SM); one more CTA row for the shared expert
  return g < 1 ? 1 : g;
}

int decode_tc_router_chunks(int H) { return (6 * H / 128 + kRtKc - 1) / kRtKc; }

bool decode_tc_router_supported(int H, int E) {
  // the tensor-core router's K chunks (kRtKc tiles of 128 bytes of 3H bf16
  // each) are summed by the top-k kernel, which takes at most 32 of them;
  // larger H routes on the CUDA cores (k_dec_route) ahead of the same expert
  // kernels
  return E % 128 == 0 && E <= 1024 && decode_tc_router_chunks(H) <= 32;
}

bool decode_tc_supported(int H, int E, int I_loc, int Iw, int row0, int s_I_loc, int s_Iw, int s_row0, int T,
                         int top_k, bool has_sf) {
  if (!has_sf || T < 1 || T > 32 || E > 1024 || top_k > 32) return false;
  if (H % 256 || I_loc % 64 || row0 % 64 || Iw % 64 || I_loc < 256 || Iw < 256) return false;
  if (s_I_loc % 64 || s_row0 % 64 || s_Iw % 64) return false;
  const DgLayout g = dg_layout(H, T, E, T * top_k);
  if (g.nst < 3 || g.total > kDtSmem) return false;
  // TMEM columns of the gate_up kernel: accumulators, activation scales,
  // weight scales per stage
  if (64 + 4 * g.nks + 16 * g.nst > 512) return false;
  const DdLayout d = dd_layout(T, E, T * top_k);
  return d.nst >= 3 && d.total <= kDdSmem && 64 + 32 * d.nst <= (int)kDdTmemCols;
}

cudaError_t decode_tc_set_smem_limits() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_dtc_router, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                1024 + kRtKc * (kDtA + kDtB) + 256)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_dec_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemMax)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_dtc_gate_up, cudaFuncAttributeMaxDynamicSharedMemorySize, kDtSmem)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_dtc_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kDdSmem);
}

static cudaError_t encode_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
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

static cudaError_t launch_tc(void (*kern)(DecodeArgs, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap), dim3 grid,
                             int threads, int smem, cudaStream_t s, bool pdl, const DecodeArgs& a,
                             const CUtensorMap& m0, const CUtensorMap& m1, const CUtensorMap& m2,
                             const CUtensorMap& m3) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, m0, m1, m2, m3);
}

cudaError_t launch_decode_tc(DecodeArgs a, cudaStream_t s, int parts) {
  cudaError_t err;
  const int H = a.H, T = a.T, P = T * a.top_k, E = a.r.E;
  const int Iw = a.win.Iw, I_loc = a.win.I_loc;
  const int npad = T <= 16 ? 16 : 32;
  CUtensorMap m_gu, m_xq, m_sgu, m_x, m_dn, m_hq, m_sdn, m_hs;
  const uint8_t* bank = a.bank;
  {
    const uint64_t dims[3] = {(uint64_t)H / 2, (uint64_t)2 * Iw, (uint64_t)a.n_records},
                   st[2] = {(uint64_t)H / 2, (uint64_t)a.lay.bytes};
    const uint32_t box[3] = {128, 64, 1};
    if ((err = encode_u8(&m_gu, bank + a.lay.gu_codes, 3, dims, st, box)) != cudaSuccess) return err;
  }
  {
    const uint64_t dims[2] = {(uint64_t)H / 2, (uint64_t)T}, st[1] = {(uint64_t)H / 2};
    const uint32_t box[2] = {128, (uint32_t)npad};
    if ((err = encode_u8(&m_xq, a.r.xq_codes, 2, dims, st, box)) != cudaSuccess) return err;
  }
  {
    const uint64_t dims[3] = {(uint64_t)Iw / 2, (uint64_t)H, (uint64_t)a.n_records},
                   st[2] = {(uint64_t)Iw / 2, (uint64_t)a.lay.bytes};
    const uint32_t box[3] = {128, 128, 1};
    if ((err = encode_u8(&m_dn, bank + a.lay.dn_codes, 3, dims, st, box)) != cudaSuccess) return err;
  }
  {
    const uint64_t dims[2] = {(uint64_t)I_loc / 2, (uint64_t)P}, st[1] = {(uint64_t)a.hq_cpitch};
    const uint32_t box[2] = {128, (uint32_t)npad};
    if ((err = encode_u8(&m_hq, a.hq_codes, 2, dims, st, box)) != cudaSuccess) return err;
  }
  m_sgu = m_gu;
  m_x = m_xq;
  m_sdn = m_dn;
  m_hs = m_hq;
  if (a.sh_gate_up) {
    {
      const uint64_t dims[2] = {(uint64_t)2 * H, (uint64_t)2 * a.s_Iw}, st[1] = {(uint64_t)2 * H};
      const uint32_t box[2] = {128, 64};
      if ((err = encode_u8(&m_sgu, a.sh_gate_up, 2, dims, st, box)) != cudaSuccess) return err;
    }
    {
      const uint64_t dims[2] = {(uint64_t)2 * H, (uint64_t)T}, st[1] = {(uint64_t)2 * H};
      const uint32_t box[2] = {128, (uint32_t)npad};
      if ((err = encode_u8(&m_x, a.r.x, 2, dims, st, box)) != cudaSuccess) return err;
    }
    {
      const uint64_t dims[2] = {(uint64_t)2 * a.s_Iw, (uint64_t)H}, st[1] = {(uint64_t)2 * a.s_Iw};
      const uint32_t box[2] = {128, 128};
      if ((err = encode_u8(&m_sdn, a.sh_down, 2, dims, st, box)) != cudaSuccess) return err;
    }
    {
      const uint64_t dims[2] = {(uint64_t)2 * a.s_I_loc, (uint64_t)T}, st[1] = {(uint64_t)2 * a.s_I_loc};
      const uint32_t box[2] = {128, (uint32_t)npad};
      if ((err = encode_u8(&m_hs, a.hs, 2, dims, st, box)) != cudaSuccess) return err;
    }
  }
  // routing (no shared gate_up CTAs: the shared expert runs on the tensor
  // cores), then top-k and the sort in one CTA
  a.n_router_ctas = (E + 1) / 2;
  a.n_shared_ctas = 0;
  a.split_tail = 1;
  // a whole forward: the expert kernels sort from the token masks; routing
  // alone (offload): the top-k kernel sorts, for the host to read
  a.meta_masks = parts == 3;
  if (parts & 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    if (a.wcat) {
      // router logits on the tensor cores (split K), activation codes, sigma
      CUtensorMap m_wr, m_xr;
      {
        const uint64_t dims[2] = {(uint64_t)6 * H, (uint64_t)E}, st[1] = {(uint64_t)6 * H};
        const uint32_t box[2] = {128, 128};
        if ((err = encode_u8(&m_wr, a.wcat, 2, dims, st, box)) != cudaSuccess) return err;
      }
      {
        const uint64_t dims[2] = {(uint64_t)2 * H, (uint64_t)T}, st[1] = {(uint64_t)2 * H};
        const uint32_t box[2] = {128, (uint32_t)npad};
        if ((err = encode_u8(&m_xr, a.r.x, 2, dims, st, box)) != cudaSuccess) return err;
      }
      const int nkt = 6 * H / 128;
      a.n_rparts = (nkt + kRtKc - 1) / kRtKc;
      const int units = (E / 128) * a.n_rparts;
      cfg.gridDim = dim3(units + rt_xq_ctas(T, H) + (T + kDtThreads / 32 - 1) / (kDtThreads / 32));
      cfg.blockDim = dim3(kDtThreads);
      cfg.dynamicSmemBytes = 1024 + kRtKc * (kDtA + kDtB) + 256;
      // programmatic launch: the router tiles stream while the grid before
      // this one (the previous forward's down kernel) finishes
      cudaLaunchAttribute rattr[1];
      rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      rattr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = rattr;
      cfg.numAttrs = a.pdl ? 1 : 0;
      FTMOE_PROF_BEGIN("k_dtc_router", s);
      err = cudaLaunchKernelEx(&cfg, k_dtc_router, a, m_wr, m_xr);
      FTMOE_PROF_END(s);
    } else {
      cfg.gridDim = dim3(a.n_router_ctas + 1);
      cfg.blockDim = dim3(kRtThreads);
      cfg.dynamicSmemBytes = 8 * T * 2 * 4;
      FTMOE_PROF_BEGIN("k_dec_route", s);
      err = cudaLaunchKernelEx(&cfg, k_dec_route, a);
      FTMOE_PROF_END(s);
    }
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(T);  // one CTA per token; the last one sorts
    cfg.blockDim = dim3(kRtThreads);
    cfg.dynamicSmemBytes = tk_smem_layout(T, E, a.top_k).total;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    FTMOE_PROF_BEGIN("k_dec_topk", s);
    err = cudaLaunchKernelEx(&cfg, k_dec_topk, a);
    FTMOE_PROF_END(s);
    if (err != cudaSuccess) return err;
  }
  if (!(parts & 2)) return cudaSuccess;
  if (a.wcat) a.n_rparts = (6 * H / 128 + kRtKc - 1) / kRtKc;
  {
    const DgLayout L = dg_layout(H, T, E, P);
    FTMOE_PROF_BEGIN("k_dtc_gate_up", s);
    err = launch_tc(k_dtc_gate_up, dim3(a.num_sms), kDgThreads, L.total, s, a.pdl, a, m_gu, m_xq, m_sgu, m_x);
    FTMOE_PROF_END(s);
    if (err != cudaSuccess) return err;
  }
  {
    const DdLayout L = dd_layout(T, E, P);
    const int rows = a.n_groups + ((a.sh_down && !a.skip_shared) ? 1 : 0);
    FTMOE_PROF_BEGIN("k_dtc_down", s);
    err = launch_tc(k_dtc_down, dim3(H / 128, rows), kDdThreads, L.total, s, a.pdl, a, m_dn, m_hq, m_sdn, m_hs);
    FTMOE_PROF_END(s);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace ftmoe
