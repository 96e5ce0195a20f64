// Host-side declarations of the ftmoe kernel launchers (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ftmoe {

// Device status word bits (set with atomicOr, read by ftmoe_check_status).
constexpr uint32_t kStatusRange = 1u;    // an in-kernel range check failed
constexpr uint32_t kStatusTimeout = 2u;  // a bounded wait ran out

// Optional per-launch timing: when set for the calling thread, launchers
// bracket each kernel with begin/end (CUDA events on the launch stream).
struct Profiler {
  virtual void begin(const char* name, cudaStream_t s) = 0;
  virtual void end(cudaStream_t s) = 0;
  virtual ~Profiler() = default;
};
extern thread_local Profiler* g_prof;
#define FTMOE_PROF_BEGIN(name, s) \
  do { if (::ftmoe::g_prof) ::ftmoe::g_prof->begin(name, s); } while (0)
#define FTMOE_PROF_END(s) \
  do { if (::ftmoe::g_prof) ::ftmoe::g_prof->end(s); } while (0)

// Byte offsets of the sections of one expert record (one expert's bank
// restricted to a loaded window of width Iw).  Sections are 256-byte aligned.
struct RecLayout {
  int64_t gu_codes, gu_scales, gu_global;  // [2Iw][H/2], [2Iw][H/16], [2Iw] fp32
  int64_t dn_codes, dn_scales, dn_global;  // [H][Iw/2], [H][Iw/16], [H] fp32
  // The same scales in 512-byte blocks for the tensor-core path (present
  // when H % 256 == 0 and Iw % 64 == 0, else gu_sf_bytes == 0):
  //   gu_sf [Iw/64][H/64][512]: tile j = gate rows [64j, 64j+64) then the
  //                             matching up rows, 64-element K steps
  //   dn_sf [H/128][Iw/64][512]: tile j = rows [128j, 128j+128)
  int64_t gu_sf, dn_sf, gu_sf_bytes;
  int64_t bytes;                           // record size (multiple of 256)
};
RecLayout make_rec_layout(int H, int Iw);

// Window of a forward relative to the loaded records.
struct Window {
  int row0;   // first intermediate index of the window inside the loaded window
  int I_loc;  // window width
  int Iw;     // loaded window width (row pitch of down codes is Iw/2)
};

struct RouteArgs {
  const uint16_t* x;      // [T][H] bf16
  const float* router_w;  // [E][H]
  const float* router_bias;  // [E] or null
  const uint16_t* sh_gate;   // [H] bf16 or null
  int T, H, E, top_k, norm_topk_prob;
  // workspace outputs
  float* logits;     // [T][E]
  float* err;        // [T][E]
  int32_t* topk_idx; // [T][k]
  float* topk_w;     // [T][k]
  uint8_t* xq_codes; // [T][H/2]
  uint8_t* xq_scales;  // [T][H/16]
  float* sigma;      // [T]
  float* xnorm;      // [T] upper bound of ||x_t||_2 (may be null)
  int32_t* offsets;  // [E+1]
  int32_t* perm;     // [P]
  int32_t* inv;      // [P]
  int32_t* touched;  // [E] touched experts, increasing
  int32_t* n_touched;  // [1]
  uint32_t* emask;   // [E] decode: bit t set when token t picked expert e (zeroed by the router kernels)
  unsigned long long* n_rerank;  // [1] cumulative count of re-ranked tokens (may be null)
  unsigned long long* touched_total;  // [1] cumulative touched experts over forwards (may be null)
  uint32_t* status;
  // counting sort over many CTAs (large T): per (chunk of 4096 pairs,
  // expert) counts, then first positions; null: the one-CTA sort
  int32_t* sort_cnt;   // [sort_max_chunks][E]
  int sort_max_chunks;
};

cudaError_t launch_quantize_weights(const float* w, int64_t rows, int K, uint8_t* codes,
                                    uint8_t* scales, float* globals, cudaStream_t s);
cudaError_t launch_quantize_act_bf16(const uint16_t* a, int64_t rows, int K, uint8_t* codes,
                                     uint8_t* scales, cudaStream_t s);

// x quantisation + shared gate, router logits, top-k, counting sort (parts
// selectable so another router-logit kernel can take the second's place).
constexpr int kRouteXq = 1, kRouteLogits = 2, kRouteTopk = 4, kRouteSort = 8, kRouteAll = 15;
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, int parts = kRouteAll);

struct ExpertArgs {
  RouteArgs r;  // routing workspace and inputs (by value: kernels read it)
  const uint8_t* const* rec;  // [E] device pointers to expert records
  RecLayout lay;
  Window win;
  int H, T, top_k;
  // shared expert (null sh_gate_up => none)
  const uint16_t* sh_gate_up;  // [2*sIw][H] bf16 (loaded window)
  const uint16_t* sh_down;     // [H][sIw] bf16
  int s_row0, s_I_loc, s_Iw;
  // workspace
  uint16_t* hs;        // [T][s_I_loc] bf16 shared intermediate
  uint8_t* hq_codes;   // [P][I_loc/2]
  uint8_t* hq_scales;  // [P][I_loc/16]
  float* Y;            // [P][H] fp32, rows in sorted order (y_tiles == 0); the tensor-core prefill
                       // down kernel's [T][H/128][k][128] fp32 (y_tiles == 1) or bf16 (y_tiles == 2)
  int y_tiles;
  float* S;            // [T][H] fp32
  void* out;
  int out_flags;
  int num_sms;
};

// Parts of the any-T expert stage: shared gate_up; routed gate_up + down on
// CUDA cores; shared down + combine.
constexpr int kPartSharedGateUp = 1, kPartRouted = 2, kPartTail = 4, kPartAll = 7;
cudaError_t launch_experts(const ExpertArgs& a, cudaStream_t s, int parts = kPartAll);

// Decode path (T <= 32): routing kernel, streamed gate_up, fused down+combine.
struct DecodeArgs {
  RouteArgs r;
  const uint8_t* const* rec;  // [E] device pointers to expert records
  RecLayout lay;
  Window win;
  int H, T, top_k;
  const uint16_t* sh_gate_up;  // null => no shared expert
  const uint16_t* sh_down;
  int s_row0, s_I_loc, s_Iw;
  uint16_t* hs;        // [T][s_I_loc] bf16
  // The quantised SwiGLU output, stored decoded: each E2M1 code as its half
  // value ([P][I_loc] half, pitch hq_cpitch bytes) and each block's E4M3
  // scale as fp32 ([P][I_loc/16], pitch hq_spitch bytes); pitches are
  // multiples of 16 bytes.
  uint8_t* hq_codes;
  uint8_t* hq_scales;
  int hq_cpitch, hq_spitch;
  void* out;
  int out_flags;
  int* counter;        // arrival counter of the router CTAs (zero between launches)
  int* gu_split;       // [num_sms + 1] first gate_up work item of each CTA (cost-balanced)
  int n_router_ctas, n_shared_ctas;
  int num_sms;
  int pdl;             // chain the kernels with programmatic dependent launch
  // tensor-core decode kernels (decode_tc.cu)
  const uint8_t* bank; // expert records, lay.bytes apart (rec[e] == bank + rec_z[e] * lay.bytes)
  const int32_t* rec_z;  // [E] record index of each expert in `bank` (null: the expert index)
  int n_records;         // records in `bank` (E when resident, the slot count when offloaded)
  uint8_t* hsf;        // [E][I_loc/64][512] intermediate scale blocks per touched expert
  float* gpart;        // [groups][T][H] partial outputs of the down kernel
  int* dn_counter;     // [H/128] arrival counters (zero between launches)
  int n_groups;        // down kernel: expert groups per 128-row output tile (+1 for the shared expert)
  int split_tail;      // 1: top-k and the sort run in k_dec_topk instead of the last router CTA
  int skip_shared;     // 1: leave the shared expert out (a later expert batch of an offloaded forward)
  int meta_masks;      // 1: the top-k kernel only sets emask; the expert kernels build the sorted tables
  // router logits on the tensor cores (split K): partial sums rpart[c][t][e]
  // of x . (W1 + W2 + W3) over K chunk c; the top-k kernel adds them in order
  const uint16_t* wcat;  // [E][3H] bf16 parts of the router rows, or null (CUDA-core router)
  const float* wnorm;    // [E] upper bound of ||w_e||
  float* rpart;          // [n_rparts][T][E]
  int n_rparts;
  float kappa;           // bound of the tensor-core accumulation: kappa * ||x|| * ||w||
  // test hook of the down kernel's failure path: CTA (0, 0) never issues its
  // first stage, and its bounded waits give up after wait_limit_ns (0: the
  // default limit), so its waits run out, it marks the status word and the
  // tile's counter and leaves cleanly
  int withhold_first_stage;
  uint64_t wait_limit_ns;
};

int decode_hq_cpitch(int I_loc);
int decode_hq_spitch(int I_loc);
bool decode_supported(int H, int E, int I_loc, int Iw, int row0, int s_I_loc, int s_Iw, int s_row0, int T,
                      int top_k);
cudaError_t decode_set_smem_limits();
cudaError_t launch_decode(DecodeArgs a, cudaStream_t s);
bool decode_tc_router_supported(int H, int E);
int decode_tc_router_chunks(int H);  // K chunks (partial logits) of the tensor-core router
bool decode_tc_supported(int H, int E, int I_loc, int Iw, int row0, int s_I_loc, int s_Iw, int s_row0, int T,
                         int top_k, bool has_sf);
int decode_tc_groups(int H, int num_sms);
cudaError_t decode_tc_set_smem_limits();
// parts: 1 = routing (router, top-k, sort), 2 = the expert kernels
cudaError_t launch_decode_tc(DecodeArgs a, cudaStream_t s, int parts = 3);
// out (bf16, fp32 or fp32 += per out_flags) <- fp32 y [T][H]
cudaError_t launch_store_out(const float* y, void* out, int out_flags, int64_t n, cudaStream_t s);

// Prefill path: grouped block-scaled NVFP4 GEMMs on tcgen05 (prefill.cu).
// Pairs are regrouped in a padded order where expert e owns rows
// [pad_off[e], pad_off[e] + round128(m_e)).
struct PfArgs {
  const int32_t* offsets;     // [E+1] sorted-position starts
  const int32_t* perm;        // [P]
  const uint8_t* xq_codes;    // [T][H/2]
  const uint8_t* xq_scales;   // [T][H/16]
  const uint8_t* bank;        // expert records, lay.bytes apart
  const int32_t* rec_z;       // [E] record index of each expert in `bank` (null: the expert index)
  const uint8_t* active;      // [E] experts this call computes (null: all); others keep Y as is
  int n_records;              // records in `bank` (E when resident, the slot count when offloaded)
  RecLayout lay;
  Window win;
  int H, T, E, top_k;
  int P_pad_max;              // rows of the padded buffers (multiple of 128)
  int32_t* pad_off;           // [E+1]
  uint8_t* xg;                // [P_pad_max][H/2] activation codes, padded order
  uint8_t* xg_sf;             // [P_pad_max/128][H/64][512] activation scale blocks
  uint8_t* hq;                // [P_pad_max][hq_pitch] intermediate codes (I_loc/2 used)
  uint8_t* hq_sf;             // [P_pad_max/128][I_loc/64][512]
  int hq_pitch;
  void* Y;                    // [T][H/128][k][128]: pair (t, slot)'s output, per column tile
  int y_bf16;                 // Y in bf16 (the forward's output is bf16), else fp32
  uint32_t* status;
  // shared expert on the tensor cores, fused with the combine
  const uint16_t* x;          // [T][H] bf16
  const uint16_t* sh_gu;      // [2*s_Iw][H] bf16 (loaded window: gate rows, then up rows)
  const uint16_t* sh_dn;      // [H][s_Iw] bf16
  int s_row0, s_I_loc, s_Iw;
  uint16_t* hs;               // [T][s_I_loc] bf16 shared intermediate
  const int32_t* inv;         // [P]
  const float* topk_w;        // [P]
  const float* sigma;         // [T]
  void* out;
  int out_flags;
  float* S;                   // [T][H] fp32 shared-expert output, when the combine runs as its own kernel
  // router logits on the tensor cores: W = W1 + W2 + W3 exactly (bf16 parts)
  const uint16_t* wcat;       // [E][3H] bf16: W1 | W2 | W3
  const float* wnorm;         // [E] upper bound of ||w_e||_2
  const float* xnorm;         // [T] upper bound of ||x_t||_2
  const float* router_bias;   // [E] or null
  float* logits;              // [T][E]
  float* err;                 // [T][E] bound on |logit - exact|
  float kappa;                // err = kappa * ||x|| * ||w|| + 2^-22 |logit|
  // few tokens: the router's K range split over r_ksplit CTAs per tile, whose
  // partial sums ([r_ksplit][T][E] fp32, in a buffer of rpart_cap floats
  // that routing does not otherwise use) a second kernel adds in order
  float* rpart;
  int64_t rpart_cap;
  int r_ksplit;
};
struct PfMaps {
  CUtensorMap xg, gu, hq, dn;   // routed operands
  CUtensorMap x, sgu, hs, sdn;  // shared-expert operands
  CUtensorMap wr;               // router parts
};

int64_t pf_pad_max(int64_t P, int E);
bool prefill_supported(int H, int E, int I_loc, int Iw, int row0);
bool prefill_shared_supported(int H, int s_I_loc, int s_Iw, int s_row0, int top_k);
bool prefill_router_supported(int H, int E);
cudaError_t launch_router_split(const float* w, int E, int H, uint16_t* wcat, float* wnorm, cudaStream_t s);
cudaError_t launch_prefill_router(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_shared_gate_up(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_shared_down(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_combine(const PfArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_shared_down_combine(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s);
cudaError_t prefill_make_maps(const PfArgs& a, PfMaps* m);
cudaError_t prefill_set_smem_limits();
cudaError_t launch_repack_sf(uint8_t* bank, const RecLayout& lay, int H, int Iw, int E, cudaStream_t s);
cudaError_t launch_prefill_routed(const PfArgs& a, const PfMaps& m, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_export_h(const PfArgs& a, uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t s);

// W4A16 routed experts (w4a16.cu): bf16 x, NVFP4 weights dequantised in
// registers, bf16 intermediate in hq_codes ([P][I_loc] bf16), Y [P][H] in
// sorted order (ExpertArgs y_tiles == 0)
cudaError_t w16_set_smem_limits(int H, int I);
cudaError_t launch_w16_routed(const ExpertArgs& a, cudaStream_t s);

// w_out[p] = mask[idx[p]] ? w[p] : 0 over P pairs
cudaError_t launch_mask_weights(const int32_t* idx, const float* w, const uint8_t* mask, float* w_out, int64_t P,
                                cudaStream_t s);

// out <- sum of n_parts fp32 partials [n_parts][n] in rank order (out_flags as a forward's)
cudaError_t launch_reduce_partials(const float* parts, int n_parts, int64_t n, void* out, int out_flags,
                                   cudaStream_t s);

// y fp32 [T][H] -> bf16(y / sqrt(mean(y^2) + eps)) [T][H]
cudaError_t launch_rms_renorm(const float* y, uint16_t* x, int T, int H, cudaStream_t s);

}  // namespace ftmoe
