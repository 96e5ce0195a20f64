// k_dec_route: routing for the decode path.  Router CTAs quantise a slice of
// the activations and compute the fp32 logits of 2 experts each (H split
// over 4 warps) with a rigorous error bound; optional CTAs run the shared
// expert's gate_up + SwiGLU (the CUDA-core decode path); one CTA computes
// the shared gate sigma; the last router CTA to finish stages every logit
// and bound in shared memory, runs top-k (certified; the whole CTA re-ranks
// uncertain tokens with compensated sums) and the counting sort.
//
// Pages: PR #385 "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
// (offload backend)", "What this adds" (replicated router; shared expert and
// its sigmoid gate); Issue #62 "Offloaded MoE ignores tensor parallelism ...",
// first comment (norm_topk_prob defaults to True).
#include "decode_common.cuh"

namespace ftmoe {

__device__ __forceinline__ bool key_before(float la, int ea, float lb, int eb) {
  return la > lb || (la == lb && ea < eb);
}
// Top-k of token t by one warp, from logits lg and bounds er in shared
// memory.  The fp32 ranking is certified with the error bounds (every chosen
// expert's interval lies above the next one's and above every unchosen
// expert's).  A certified token's slots and weights are written here;
// otherwise the lowest lower end of the chosen intervals is returned in
// *lmin_out (every expert whose interval reaches it is a candidate) and the
// token is re-ranked afterwards.  Ties go to the lower index.
__device__ __forceinline__ void dec_write_slots(const DecodeArgs& a, int t, int lane, int my_idx, float my_l,
                                                float lmax, const float* lg, int* s_idx) {
  const int E = a.r.E, k = a.r.top_k;
  // routing weights: softmax over the chosen (norm_topk_prob) or over all
  const float ex = (lane < k) ? expf(my_l - lmax) : 0.f;
  float den;
  if (a.r.norm_topk_prob) {
    den = warp_sum(ex);
  } else {
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += expf(lg[e] - lmax);
    den = warp_sum(s);
  }
  if (lane < k) {
    a.r.topk_idx[(int64_t)t * k + lane] = my_idx;
    a.r.topk_w[(int64_t)t * k + lane] = ex / den;
    s_idx[t * k + lane] = my_idx;
  }
}

__device__ bool dec_topk_fast(const DecodeArgs& a, int t, int lane, const float* lg, const float* er, uint8_t* ch,
                              int* s_idx, float* lmin_out) {
  const int E = a.r.E, k = a.r.top_k;
  for (int e = lane; e < E; e += 32) ch[e] = 0;
  __syncwarp();
  int my_idx = 0;  // lane j keeps slot j
  float my_l = 0.f;
  float lmax = -INFINITY;
  bool certified = true;
  float prev_lo = INFINITY, lmin_lo = INFINITY;
  for (int j = 0; j < k; ++j) {
    float bl = -INFINITY;
    int be = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = lg[e];
      if (!ch[e] && key_before(v, e, bl, be)) { bl = v; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (key_before(ol, oe, bl, be)) { bl = ol; be = oe; }
    }
    if (lane == j) { my_idx = be; my_l = bl; }
    if (j == 0) lmax = bl;
    const float eb = er[be];
    const float lo = bl - eb, hi = bl + eb;
    if (!(hi < prev_lo)) certified = false;
    prev_lo = lo;
    lmin_lo = fminf(lmin_lo, lo);
    __syncwarp();
    if (lane == 0) ch[be] = 1;
    __syncwarp();
  }
  bool reach = false;
  for (int e = lane; e < E; e += 32)
    if (!ch[e] && lg[e] + er[e] >= lmin_lo) reach = true;
  if (__any_sync(0xffffffffu, reach)) certified = false;
  *lmin_out = lmin_lo;
  if (certified) dec_write_slots(a, t, lane, my_idx, my_l, lmax, lg, s_idx);
  return certified;
}

// Re-rank of the uncertain tokens by the whole CTA, in rounds: each warp
// lists the candidates of its pending tokens (every expert whose interval
// reaches the token's lowest chosen lower end) while the shared list has
// room; then every warp computes compensated logits of list entries in turn
// (one warp per entry, about 2^-48 relative; FP64 is far slower on this
// GPU); then each token's warp selects its k among its candidates.
__device__ void dec_rerank(const DecodeArgs& a, const RtSmem& L, unsigned char* sm, int* s_idx) {
  const int E = a.r.E, k = a.r.top_k, T = a.T, H = a.r.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* le = reinterpret_cast<int*>(sm + L.le_off);
  int* lt = reinterpret_cast<int*>(sm + L.lt_off);
  df32* lv = reinterpret_cast<df32*>(sm + L.lv_off);
  int* state = reinterpret_cast<int*>(sm + L.tok_off);  // 0 done, 1 pending, 2 listed
  int* start = state + 32;
  int* cnt = start + 32;
  float* lmin = reinterpret_cast<float*>(cnt + 32);
  int* s_cnt = reinterpret_cast<int*>(lmin + 32);
  int* s_any = s_cnt + 1;
  // nothing to do in the common case: every token certified
  bool any = false;
  for (int t = 0; t < T; ++t) any |= state[t] != 0;
  if (!any) return;
  // every round lists at least one pending token (a token has at most E
  // candidates and the list holds 4E), so T rounds always suffice
  for (int round = 0; round <= T; ++round) {
    if (tid == 0) { *s_cnt = 0; *s_any = 0; }
    for (int i = tid; i < L.cap; i += kRtThreads) lt[i] = -1;
    __syncthreads();
    for (int t = warp; t < T; t += 8) {
      if (state[t] != 1) continue;
      if (lane == 0) *s_any = 1;
      const float* lg = a.r.logits + (int64_t)t * E;
      const float* er = a.r.err + (int64_t)t * E;
      int nc = 0;
      for (int e = lane; e < E; e += 32) nc += (__ldcg(lg + e) + __ldcg(er + e) >= lmin[t]) ? 1 : 0;
      nc = __reduce_add_sync(0xffffffffu, nc);
      int st = 0;
      if (lane == 0) st = atomicAdd(s_cnt, nc);
      st = __shfl_sync(0xffffffffu, st, 0);
      if (st + nc > L.cap) break;  // no room left this round
      int w = st;
      for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        const bool c = e < E && (__ldcg(lg + e) + __ldcg(er + e) >= lmin[t]);
        const unsigned m = __ballot_sync(0xffffffffu, c);
        if (c) {
          le[w + __popc(m & ((1u << lane) - 1))] = e;
          lt[w + __popc(m & ((1u << lane) - 1))] = t;
        }
        w += __popc(m);
      }
      if (lane == 0) { start[t] = st; cnt[t] = nc; state[t] = 2; }
      __syncwarp();
    }
    __syncthreads();
    if (!*s_any) break;
    const int n = min(*s_cnt, L.cap);
    for (int i = warp; i < n; i += 8) {
      if (lt[i] < 0) continue;
      const int e = le[i];
      const df32 v = logit_df32(a.r.x + (int64_t)lt[i] * H, a.r.router_w + (int64_t)e * H, H,
                                a.r.router_bias ? a.r.router_bias[e] : 0.f, lane);
      if (lane == 0) lv[i] = v;
    }
    __syncthreads();
    for (int t = warp; t < T; t += 8) {
      if (state[t] != 2) continue;
      const int c0 = start[t], nc = cnt[t];
      int my_idx = 0;
      float my_l = 0.f, lmax = -INFINITY;
      const df32 none = {-INFINITY, 0.f};
      for (int j = 0; j < k; ++j) {
        df32 bl = none;
        int be = 0x7fffffff, bc = -1;
        for (int c = lane; c < nc; c += 32) {
          const df32 v = lv[c0 + c];
          const int e = le[c0 + c];
          if (v.hi != -INFINITY && df_before(v, e, bl, be)) { bl = v; be = e; bc = c; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const df32 ol = {__shfl_xor_sync(0xffffffffu, bl.hi, o), __shfl_xor_sync(0xffffffffu, bl.lo, o)};
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
          if (df_before(ol, oe, bl, be)) { bl = ol; be = oe; bc = oc; }
        }
        if (lane == j) { my_idx = be; my_l = bl.hi; }
        if (j == 0) lmax = bl.hi;
        __syncwarp();
        if (lane == 0 && bc >= 0) lv[c0 + bc] = none;
        __syncwarp();
      }
      dec_write_slots(a, t, lane, my_idx, my_l, lmax, a.r.logits + (int64_t)t * E, s_idx);
      if (lane == 0) state[t] = 0;
      __syncwarp();
    }
    __syncthreads();
  }
}

// Counting sort of the P = T * k <= 1024 pairs (T <= 32) by one CTA of
// kRtThreads threads.  A token picks an expert at most once, so expert e's
// pairs are fixed by the mask of tokens that picked it: its count is the
// mask's population, and pair (t, j) of expert e goes to offsets[e] + the
// number of earlier tokens in the mask -- every expert's pairs in
// increasing pair id.  hist holds [E] masks and [E] offsets.
__device__ void dec_sort(const DecodeArgs& a, const int* s_idx, int* hist /*[8][E]*/, int* scan /*[32]*/) {
  const int E = a.r.E, k = a.top_k, P = a.T * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* mask = reinterpret_cast<uint32_t*>(hist);
  int* off = hist + E;
  for (int e = tid; e < E; e += kRtThreads) mask[e] = 0u;
  __syncthreads();
  for (int p = tid; p < P; p += kRtThreads) {
    int e = s_idx[p];
    if ((unsigned)e >= (unsigned)E) { set_status(a.r.status, kStatusRange); e = 0; }
    atomicOr(&mask[e], 1u << (p / k));
  }
  __syncthreads();
  // each thread owns experts [e0, e1): pair and touched counts, block scan
  const int per = (E + kRtThreads - 1) / kRtThreads;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int cnt = 0, tcnt = 0;
  for (int e = e0; e < e1; ++e) {
    const uint32_t m = mask[e];
    cnt += __popc(m);
    tcnt += m != 0u;
  }
  int inc = cnt, tinc = tcnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o), tn = __shfl_up_sync(0xffffffffu, tinc, o);
    if (lane >= o) { inc += n; tinc += tn; }
  }
  if (lane == 31) { scan[warp] = inc; scan[16 + warp] = tinc; }
  __syncthreads();
  int wbase = 0, twbase = 0;
  for (int w = 0; w < warp; ++w) { wbase += scan[w]; twbase += scan[16 + w]; }
  int run = wbase + inc - cnt, toff = twbase + tinc - tcnt;
  for (int e = e0; e < e1; ++e) {
    const uint32_t m = mask[e];
    off[e] = run;
    a.r.offsets[e] = run;
    if (m) a.r.touched[toff++] = e;
    run += __popc(m);
  }
  if (tid == kRtThreads - 1) {
    a.r.offsets[E] = P;
    a.r.n_touched[0] = toff;
    if (a.r.touched_total) atomicAdd(a.r.touched_total, (unsigned long long)toff);
  }
  __syncthreads();
  for (int p = tid; p < P; p += kRtThreads) {
    int e = s_idx[p];
    if ((unsigned)e >= (unsigned)E) e = 0;
    const int t = p / k;
    const int pos = off[e] + __popc(mask[e] & ((1u << t) - 1u));
    a.r.perm[pos] = p;
    a.r.inv[p] = pos;
  }
}

// Work split of k_dec_gate_up over its CTAs (one per SM), balanced by cost.
// An item (touched expert j, 16-wide block) costs kItemCost units of weight
// work plus one unit per pair of the expert.  gu_split[b] is the first item
// whose cost interval starts at or after b * C / G (C the total cost, G the
// number of CTAs), so CTA b takes items [gu_split[b], gu_split[b+1]).
// Runs in the CTA that did the sort; pre[] holds nt + 1 ints of scratch.
constexpr int kItemCost = 2;
__device__ void dec_split(const DecodeArgs& a, int* pre, int* scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = __ldcg(a.r.n_touched), n_ib = a.win.I_loc / kBlock, G = a.num_sms;
  // exclusive prefix of per-expert costs, 4 consecutive experts per thread
  const int j0 = tid * 4;
  int c[4], sum = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = j0 + q;
    int cj = 0;
    if (j < nt) {
      const int e = __ldcg(a.r.touched + j);
      cj = n_ib * (kItemCost + __ldcg(a.r.offsets + e + 1) - __ldcg(a.r.offsets + e));
    }
    c[q] = cj;
    sum += cj;
  }
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scan[warp] = inc;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += scan[w];
  int run = base + inc - sum;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (j0 + q <= nt) pre[j0 + q] = run;
    run += c[q];
  }
  __syncthreads();
  const int64_t C = pre[nt];
  for (int b = tid; b <= G; b += kRtThreads) {
    int item;
    if (b == G || nt == 0) {
      item = nt * n_ib;
    } else {
      const int64_t X = C * b / G;
      int lo = 0, hi = nt - 1;  // last expert whose prefix is <= X
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= X) lo = mid; else hi = mid - 1;
      }
      const int per_item = (pre[lo + 1] - pre[lo]) / n_ib;
      const int64_t into = (X - pre[lo] + per_item - 1) / per_item;
      item = lo * n_ib + (int)(into < n_ib ? into : n_ib);
    }
    a.gu_split[b] = item;
  }
}

// Largest number of K-chunk partials of the tensor-core router; the top-k
// kernel adds them in four contiguous runs of at most kRpRun.
constexpr int kMaxRparts = 32;
constexpr int kRpRun = kMaxRparts / 4;

// Top-k of every token (certified; uncertain tokens re-ranked by the whole
// CTA), the counting sort and the gate_up work split, by one CTA.
__device__ void dec_tail(const DecodeArgs& a, unsigned char* sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, E = a.r.E;
  const RtSmem L = rt_smem_layout(T, E, a.top_k);
  float* s_lg = reinterpret_cast<float*>(sm + L.logits_off) + warp * E;  // one token row per warp
  float* s_er = reinterpret_cast<float*>(sm + L.err_off) + warp * E;
  uint8_t* ch = sm + L.ch_off + warp * E;
  int* s_idx = reinterpret_cast<int*>(sm + L.idx_off);
  int* state = reinterpret_cast<int*>(sm + L.tok_off);
  float* lmin = reinterpret_cast<float*>(state + 96);
  // (the tensor-core router always runs the split tail, k_dec_topk, so the
  // logits and their bounds are in a.r.logits / a.r.err here)
  for (int t = warp; t < T; t += 8) {
    for (int e = lane; e < E; e += 32) {
      s_lg[e] = __ldcg(a.r.logits + (int64_t)t * E + e);
      s_er[e] = __ldcg(a.r.err + (int64_t)t * E + e);
    }
    __syncwarp();
    float lo;
    const bool cert = dec_topk_fast(a, t, lane, s_lg, s_er, ch, s_idx, &lo);
    if (lane == 0) {
      state[t] = cert ? 0 : 1;
      lmin[t] = lo;
      if (!cert && a.r.n_rerank) atomicAdd(a.r.n_rerank, 1ull);  // telemetry only
    }
    __syncwarp();
  }
  __syncthreads();
  dec_rerank(a, L, sm, s_idx);
  int* hist = reinterpret_cast<int*>(sm + L.hist_off);
  int* scan = reinterpret_cast<int*>(sm + L.scan_off);
  dec_sort(a, s_idx, hist, scan);
  if (!a.split_tail) {  // the CUDA-core gate_up kernel's work split
    __syncthreads();
    dec_split(a, hist, scan);
  }
}

// ---- the routing tail as its own kernel: one CTA per token, then the sort
// in the last CTA to finish.

// Ranking key of a logit: NaN orders as -infinity, so the order (logit
// descending, then index ascending) stays total.
__device__ __forceinline__ float tk_key(float v) { return v != v ? -INFINITY : v; }

// Logits and bounds of token t into shared memory: from the tensor-core
// router's K-chunk partials, added in chunk order (the bound is the
// accumulation bound kappa ||x|| ||w|| plus the rounding of these fp32
// additions and of the bias), else as the CUDA-core router wrote them.
// lg is padded with -infinity to a multiple of 4 entries.
__device__ void tk_logits(const DecodeArgs& a, int t, float* lg, float* er, float* scratch) {
  const int tid = threadIdx.x, T = a.T, E = a.r.E;
  if (a.n_rparts > 0) {
    // the K-chunk partials of every expert in four contiguous runs (thread
    // = (expert quad, run), the run's loads in flight together), then the
    // runs added in order; the bound is the accumulation bound
    // kappa ||x|| ||w|| plus the rounding of these fp32 additions (at most
    // C + 2 of them along any path) and of the bias
    const float gam = (float)(a.n_rparts + 2) * 5.9604645e-8f;
    const int C = a.n_rparts;  // at most kMaxRparts
    const int Q = E / 4;       // expert quads, at most kRtThreads
    const float xn = __ldcg(a.r.xnorm + t);
    const float4 wn = tid < Q ? __ldg(reinterpret_cast<const float4*>(a.wnorm) + tid) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4* ps = reinterpret_cast<float4*>(scratch);  // [4][Q] run sums, then [4][Q] run sums of |.|
    for (int w = tid; w < 4 * Q; w += kRtThreads) {
      const int g = w % Q, r = w / Q;
      const int c0 = r * C / 4, c1 = (r + 1) * C / 4;
      const float4* pp = reinterpret_cast<const float4*>(a.rpart + (int64_t)t * E) + g;
      float4 v[kRpRun];
#pragma unroll
      for (int c = 0; c < kRpRun; ++c)
        if (c0 + c < c1) v[c] = __ldcg(pp + (int64_t)(c0 + c) * T * Q);
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f), sa = s;
#pragma unroll
      for (int c = 0; c < kRpRun; ++c) {
        if (c0 + c < c1) {
          s.x += v[c].x; s.y += v[c].y; s.z += v[c].z; s.w += v[c].w;
          sa.x += fabsf(v[c].x); sa.y += fabsf(v[c].y); sa.z += fabsf(v[c].z); sa.w += fabsf(v[c].w);
        }
      }
      ps[r * Q + g] = s;
      ps[(4 + r) * Q + g] = sa;
    }
    __syncthreads();
    if (tid < Q) {
      const int e = 4 * tid;
      float s[4] = {0.f, 0.f, 0.f, 0.f}, sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 u = ps[r * Q + tid], ua = ps[(4 + r) * Q + tid];
        s[0] += u.x; s[1] += u.y; s[2] += u.z; s[3] += u.w;
        sa[0] += ua.x; sa[1] += ua.y; sa[2] += ua.z; sa[3] += ua.w;
      }
      const float w4[4] = {wn.x, wn.y, wn.z, wn.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float bias = a.r.router_bias ? a.r.router_bias[e + q] : 0.f;
        const float l = s[q] + bias;
        const float b = a.kappa * xn * w4[q] + gam * (sa[q] + fabsf(bias)) + 1.2e-7f * fabsf(l) + 1e-30f;
        a.r.logits[(int64_t)t * E + e + q] = l;
        a.r.err[(int64_t)t * E + e + q] = b;
        lg[e + q] = tk_key(l);
        er[e + q] = b;
      }
    }
  } else {
    for (int e = tid; e < E; e += kRtThreads) {
      lg[e] = tk_key(__ldcg(a.r.logits + (int64_t)t * E + e));
      er[e] = __ldcg(a.r.err + (int64_t)t * E + e);
    }
  }
  for (int e = E + tid; e < ((E + 3) & ~3); e += kRtThreads) lg[e] = -INFINITY;
  __syncthreads();
}

// Top-k of the CTA's token with the certificate of the fp32 ranking, and the
// compensated re-rank when the bounds cannot certify it.  Every thread ranks
// its experts against all E (ranks < k are the chosen slots, in order); the
// ranking is certified when each chosen interval lies above the next one and
// no unchosen interval reaches the lowest chosen lower end.  Otherwise every
// expert whose interval reaches it is a candidate: its logit is recomputed
// with compensated sums (one warp per candidate) and the k best candidates
// are taken in (logit, index) order.
__device__ void tk_select(const DecodeArgs& a, const TkSmem& L, unsigned char* sm, int t) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.r.E, k = a.r.top_k, H = a.r.H;
  float* lg = reinterpret_cast<float*>(sm + L.lg_off);
  float* er = reinterpret_cast<float*>(sm + L.er_off);
  float* sl_l = reinterpret_cast<float*>(sm + L.sl_off);
  float* sl_r = sl_l + 32;
  int* sl_e = reinterpret_cast<int*>(sl_r + 32);
  int* le = reinterpret_cast<int*>(sm + L.le_off);
  df32* lv = reinterpret_cast<df32*>(sm + L.lv_off);
  int* s_idx = reinterpret_cast<int*>(sm + L.idx_off);
  int* flags = reinterpret_cast<int*>(sm + L.scan_off) + 32;  // [2] number of re-rank candidates
  // ---- ranks (at most 4 experts per thread: E <= 1024).  Fast pass: the
  // number of keys strictly above each key (four independent counts); it is
  // the rank unless keys tie, which shows as a chosen rank held by other
  // than exactly one expert, and then the exact pass ranks ties by index.
  int* sl_cnt = sl_e + 32;  // zeroed by the caller before the logits' barrier
  int rk[4];
  const float4* k4 = reinterpret_cast<const float4*>(lg);
  const int E4 = (E + 3) >> 2;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int e = tid + m * kRtThreads;
    rk[m] = k;
    if (e < E) {
      const float v = lg[e];
      int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll 8
      for (int f4 = 0; f4 < E4; ++f4) {
        const float4 u = k4[f4];
        c0 += u.x > v;
        c1 += u.y > v;
        c2 += u.z > v;
        c3 += u.w > v;
      }
      const int r = c0 + c1 + c2 + c3;
      rk[m] = r;
      if (r < k) {
        atomicAdd(&sl_cnt[r], 1);
        sl_l[r] = v; sl_r[r] = er[e]; sl_e[r] = e;
      }
    }
  }
  __syncthreads();
  if (__syncthreads_or(tid < k && sl_cnt[tid] != 1)) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kRtThreads;
      rk[m] = k;
      if (e < E) {
        const float v = lg[e];
        int r = 0;
#pragma unroll 4
        for (int f4 = 0; f4 < E4; ++f4) {
          const float4 u = k4[f4];
          const int f = 4 * f4;
          r += (u.x > v) | ((u.x == v) & (f < e));
          r += (u.y > v) | ((u.y == v) & (f + 1 < e));
          r += (u.z > v) | ((u.z == v) & (f + 2 < e));
          r += (u.w > v) | ((u.w == v) & (f + 3 < e));
        }
        rk[m] = r;
        if (r < k) { sl_l[r] = v; sl_r[r] = er[e]; sl_e[r] = e; }
      }
    }
    __syncthreads();
  }
  // ---- certificate, every warp for itself (the chosen intervals are in
  // shared memory since the last barrier): each chosen interval above the
  // next one, and the lowest chosen lower end
  float lmin;
  bool chain_ok;
  {
    float lo = INFINITY, hi = -INFINITY;
    if (lane < k) { lo = sl_l[lane] - sl_r[lane]; hi = sl_l[lane] + sl_r[lane]; }
    const float prev_lo = __shfl_up_sync(0xffffffffu, lo, 1);
    chain_ok = __all_sync(0xffffffffu, lane >= k || hi < (lane == 0 ? INFINITY : prev_lo));
    lmin = lo;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmin = fminf(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
  }
  bool reach = false;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int e = tid + m * kRtThreads;
    if (e < E && rk[m] >= k && lg[e] + er[e] >= lmin) reach = true;
  }
  const bool cert = __syncthreads_or(reach) == 0 && chain_ok;
  if (cert) {
    if (warp == 0)
      dec_write_slots(a, t, lane, lane < k ? sl_e[lane] : 0, lane < k ? sl_l[lane] : 0.f, sl_l[0], lg, s_idx);
    return;
  }
  // ---- re-rank: candidates in index order
  if (tid == 0 && a.r.n_rerank) atomicAdd(a.r.n_rerank, 1ull);  // telemetry only
  if (warp == 0) {
    int w = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const bool c = e < E && lg[e] + er[e] >= lmin;
      const unsigned msk = __ballot_sync(0xffffffffu, c);
      if (c) le[w + __popc(msk & ((1u << lane) - 1))] = e;
      w += __popc(msk);
    }
    if (lane == 0) flags[2] = w;
  }
  __syncthreads();
  const int nc = flags[2];
  for (int i = warp; i < nc; i += kRtThreads / 32) {
    const int e = le[i];
    const df32 v = logit_df32(a.r.x + (int64_t)t * H, a.r.router_w + (int64_t)e * H, H,
                              a.r.router_bias ? a.r.router_bias[e] : 0.f, lane);
    if (lane == 0) lv[i] = v;
  }
  __syncthreads();
  if (warp == 0) {
    int my_idx = 0;
    float my_l = 0.f, lmax = -INFINITY;
    const df32 none = {-INFINITY, 0.f};
    for (int j = 0; j < k; ++j) {
      df32 bl = none;
      int be = 0x7fffffff, bc = -1;
      for (int c = lane; c < nc; c += 32) {
        const df32 v = lv[c];
        const int e = le[c];
        if (v.hi != -INFINITY && df_before(v, e, bl, be)) { bl = v; be = e; bc = c; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const df32 ol = {__shfl_xor_sync(0xffffffffu, bl.hi, o), __shfl_xor_sync(0xffffffffu, bl.lo, o)};
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
        if (df_before(ol, oe, bl, be)) { bl = ol; be = oe; bc = oc; }
      }
      if (lane == j) { my_idx = be; my_l = bl.hi; }
      if (j == 0) lmax = bl.hi;
      __syncwarp();
      if (lane == 0 && bc >= 0) lv[bc] = none;
      __syncwarp();
    }
    dec_write_slots(a, t, lane, my_idx, my_l, lmax, lg, s_idx);
  }
}

// After the router kernel: CTA t selects token t's experts; the last CTA to
// finish (arrival counter) runs the counting sort over every token.
__global__ void __launch_bounds__(kRtThreads) k_dec_topk(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ int s_last;
  // let the gate_up kernel launch now: its first phase (the shared expert)
  // needs no routing
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, t = blockIdx.x;
  const TkSmem L = tk_smem_layout(a.T, a.r.E, a.top_k);
  if (tid < 32) reinterpret_cast<int*>(sm + L.sl_off)[3 * 32 + tid] = 0;  // rank counts of tk_select
  tk_logits(a, t, reinterpret_cast<float*>(sm + L.lg_off), reinterpret_cast<float*>(sm + L.er_off),
            reinterpret_cast<float*>(sm + L.hist_off));
  tk_select(a, L, sm, t);
  if (a.meta_masks) {
    // token t's bit in each chosen expert's mask (lane j of warp 0 wrote
    // slot j); the expert kernels build the sorted tables from the masks
    if (tid < a.top_k) atomicOr(a.r.emask + reinterpret_cast<const int*>(sm + L.idx_off)[t * a.top_k + tid], 1u << t);
    return;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.counter, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int* s_idx = reinterpret_cast<int*>(sm + L.idx_off);
  for (int i = tid; i < a.T * a.top_k; i += kRtThreads) s_idx[i] = __ldcg(a.r.topk_idx + i);
  dec_sort(a, s_idx, reinterpret_cast<int*>(sm + L.hist_off), reinterpret_cast<int*>(sm + L.scan_off));
  if (tid == 0) *a.counter = 0;  // ready for the next launch
}

__global__ void __launch_bounds__(kRtThreads) k_dec_route(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ int s_last;
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.r.H, T = a.T, E = a.r.E;
  const int b = blockIdx.x;
  if (b < a.n_router_ctas) {
    // ---- this CTA's slice of the activation quantisation (global 1.0)
    {
      const int nb = T * (H / kBlock);
      const int per = (nb + a.n_router_ctas - 1) / a.n_router_ctas;
      const int q0 = b * per, q1 = min(nb, q0 + per);
      for (int blk = q0 + tid; blk < q1; blk += kRtThreads) {
        float v[16];
        const uint4* p = reinterpret_cast<const uint4*>(a.r.x + (int64_t)blk * kBlock);
        const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
        const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          v[2 * qq] = __uint_as_float(words[qq] << 16);
          v[2 * qq + 1] = __uint_as_float(words[qq] & 0xffff0000u);
        }
        uint8_t c[8];
        const uint8_t sc = quantize_block16(v, 1.0f, c);
        *reinterpret_cast<uint2*>(a.r.xq_codes + (int64_t)blk * 8) = pack8(c);
        a.r.xq_scales[blk] = sc;
      }
    }
    // ---- router: experts 2b (warps 0-3) and 2b+1 (warps 4-7), H in quarters
    float* part = reinterpret_cast<float*>(sm);  // [8 warps][T][2]
    const int e = 2 * b + (warp >> 2);
    const int q = warp & 3;
    const int Hq = H / 4;
    if (e < E) {
      const float4* wr = reinterpret_cast<const float4*>(a.r.router_w + (int64_t)e * H + q * Hq);
      const int nq = Hq / 4;  // float4 chunks of the quarter row
      for (int t0 = 0; t0 < T; t0 += 8) {
        float acc[8], ab[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) { acc[m] = 0.f; ab[m] = 0.f; }
        for (int g0 = 0; g0 < nq; g0 += 8 * 32) {
          // all of this lane's chunks of the group in flight at once
          float4 wv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = g0 + lane + 32 * j;
            wv[j] = c < nq ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = g0 + lane + 32 * j;
            if (c < nq) {
              const float4 w = wv[j];
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                if (t0 + m < T) {
                  const uint2 xv =
                      __ldg(reinterpret_cast<const uint2*>(a.r.x + (int64_t)(t0 + m) * H + q * Hq) + c);
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
          }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float s = warp_sum(acc[m]);
          const float bb = warp_sum(ab[m]);
          if (lane == 0 && t0 + m < T) {
            part[(warp * T + t0 + m) * 2] = s;
            part[(warp * T + t0 + m) * 2 + 1] = bb;
          }
        }
      }
    }
    __syncthreads();
    // combine the quarters in a fixed order.  The sequential roundings of a
    // logit: 4*ceil(H/512) FMAs per lane, 5 butterfly levels, 3 quarter adds
    // and the bias, so |l - exact| <= (D+1) u A (1.01 covers A's own error)
    const int n_seq = 4 * ((Hq / 4 + 31) / 32);
    const float gamma = (float)((double)(n_seq + 10) * 5.9604644775390625e-8 * 1.01);
    for (int i = tid; i < 2 * T; i += kRtThreads) {
      const int ex = i / T, t = i % T;
      const int ee = 2 * b + ex;
      if (ee < E) {
        const int w0 = ex * 4;
        float s = part[(w0 * T + t) * 2];
        float bb = part[(w0 * T + t) * 2 + 1];
        for (int qq = 1; qq < 4; ++qq) {
          s += part[((w0 + qq) * T + t) * 2];
          bb += part[((w0 + qq) * T + t) * 2 + 1];
        }
        const float l = s + (a.r.router_bias ? a.r.router_bias[ee] : 0.f);
        a.r.logits[(int64_t)t * E + ee] = l;
        a.r.err[(int64_t)t * E + ee] = gamma * bb + 1.2e-7f * fabsf(l) + 1e-30f;
      }
    }
    if (a.split_tail) return;  // top-k and the sort run in k_dec_topk
    // the last router CTA to arrive runs top-k and the sort
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(a.counter, 1) == a.n_router_ctas - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    dec_tail(a, sm);
    if (tid == 0) *a.counter = 0;  // ready for the next launch
    return;
  }
  if (b < a.n_router_ctas + a.n_shared_ctas) {
    // ---- shared expert gate_up + SwiGLU: two window indices per CTA, a
    // quarter of H per warp (warps 0-3 index 2b', warps 4-7 index 2b'+1);
    // the quarters' partial sums add in a fixed order
    float* part = reinterpret_cast<float*>(sm);  // [8 warps][T][2]
    const int i = (b - a.n_router_ctas) * 2 + (warp >> 2);
    const int q = warp & 3;
    const int Hq = H / 4, nq = Hq / 8;  // uint4 chunks (8 bf16) of a quarter row
    if (i < a.s_I_loc) {
      const uint4* g_row = reinterpret_cast<const uint4*>(a.sh_gate_up + (int64_t)(a.s_row0 + i) * H + q * Hq);
      const uint4* u_row =
          reinterpret_cast<const uint4*>(a.sh_gate_up + (int64_t)(a.s_Iw + a.s_row0 + i) * H + q * Hq);
      for (int t0 = 0; t0 < T; t0 += 8) {
        float ag[8], au[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) { ag[m] = 0.f; au[m] = 0.f; }
        for (int g0 = 0; g0 < nq; g0 += 4 * 32) {
          uint4 gv[4], uv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = g0 + lane + 32 * j;
            gv[j] = c < nq ? __ldg(g_row + c) : make_uint4(0, 0, 0, 0);
            uv[j] = c < nq ? __ldg(u_row + c) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = g0 + lane + 32 * j;
            if (c < nq) {
              const uint32_t gw[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
              const uint32_t uw[4] = {uv[j].x, uv[j].y, uv[j].z, uv[j].w};
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                if (t0 + m < T) {
                  const uint4 xv =
                      __ldg(reinterpret_cast<const uint4*>(a.r.x + (int64_t)(t0 + m) * H + q * Hq) + c);
                  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                  for (int qq = 0; qq < 4; ++qq) {
                    const float x0 = __uint_as_float(xw[qq] << 16), x1 = __uint_as_float(xw[qq] & 0xffff0000u);
                    ag[m] = fmaf(x0, __uint_as_float(gw[qq] << 16), ag[m]);
                    ag[m] = fmaf(x1, __uint_as_float(gw[qq] & 0xffff0000u), ag[m]);
                    au[m] = fmaf(x0, __uint_as_float(uw[qq] << 16), au[m]);
                    au[m] = fmaf(x1, __uint_as_float(uw[qq] & 0xffff0000u), au[m]);
                  }
                }
              }
            }
          }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float g = warp_sum(ag[m]), u = warp_sum(au[m]);
          if (lane == 0 && t0 + m < T) {
            part[(warp * T + t0 + m) * 2] = g;
            part[(warp * T + t0 + m) * 2 + 1] = u;
          }
        }
      }
    }
    __syncthreads();
    for (int k2 = tid; k2 < 2 * T; k2 += kRtThreads) {
      const int ii = k2 / T, t = k2 % T;
      const int idx = (b - a.n_router_ctas) * 2 + ii;
      if (idx < a.s_I_loc) {
        const int w0 = ii * 4;
        float g = part[(w0 * T + t) * 2], u = part[(w0 * T + t) * 2 + 1];
        for (int qq = 1; qq < 4; ++qq) {
          g += part[((w0 + qq) * T + t) * 2];
          u += part[((w0 + qq) * T + t) * 2 + 1];
        }
        const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * u);
        a.hs[(int64_t)t * a.s_I_loc + idx] = *reinterpret_cast<const uint16_t*>(&hb);
      }
    }
    return;
  }
  // ---- the token masks of the top-k kernel start empty, and so does the
  // gate_up kernel's unit counter
  if (a.r.emask)
    for (int e = tid; e < E; e += kRtThreads) a.r.emask[e] = 0u;
  if (a.meta_masks && tid == 0) *a.counter = 0;
  // ---- sigma_t = sigmoid(g . x_t), one warp per token
  for (int t = warp; t < T; t += 8) {
    float z = 0.f;
    if (a.r.sh_gate) {
      const uint4* xr = reinterpret_cast<const uint4*>(a.r.x + (int64_t)t * H);
      const uint4* gr = reinterpret_cast<const uint4*>(a.r.sh_gate);
      for (int c = lane; c < H / 8; c += 32) {
        const uint4 xv = __ldg(xr + c), gv = __ldg(gr + c);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          z = fmaf(__uint_as_float(xw[qq] << 16), __uint_as_float(gw[qq] << 16), z);
          z = fmaf(__uint_as_float(xw[qq] & 0xffff0000u), __uint_as_float(gw[qq] & 0xffff0000u), z);
        }
      }
    }
    z = warp_sum(z);
    if (lane == 0) a.r.sigma[t] = a.r.sh_gate ? 1.0f / (1.0f + expf(-z)) : 0.f;
  }
}

}  // namespace ftmoe
