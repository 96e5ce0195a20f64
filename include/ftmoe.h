/*
 * ftmoe.h -- C ABI of libftmoe.so, a routed NVFP4 mixture-of-experts FFN layer
 * for one GB300 (sm_103a).
 *
 * The layer (pages, by title):
 *   [PR385] "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
 *           (offload backend)"
 *   [I62]   "Offloaded MoE ignores tensor parallelism: TP=2 is a regression,
 *           and the fix is not expert parallelism"
 *
 *   out_t = sum_j w_tj * Y_{t,j} + sigmoid(g . x_t) * S_t
 *
 * with a replicated router (softmax -> top-k, renormalised over the k chosen
 * when norm_topk_prob is set), NVFP4 expert banks (packed E2M1 codes, 16-wide
 * E4M3 scale blocks, per-row fp32 globals), SwiGLU experts whose gate_up is
 * [2I, H] (gate rows [0, I), up rows [I, 2I)) and down is [H, I], a bf16
 * shared expert, and the combine routed + sigmoid(gate) * shared formed
 * before any reduction ([PR385] "What this adds").  An intermediate window
 * [i0, i0 + I_loc) computes the partial sum that a rank owning that slice of
 * I would compute; partials over windows that cover I once add up to the
 * whole layer ([I62] "The fix that fits: TP-shard the offload banks").
 *
 * Numerics (the pages leave these open; the readings taken):
 *   - Activations are NVFP4 too: x per token and the SwiGLU output per pair
 *     are quantised in 16-blocks with E4M3 scale = RNE(amax / 6) and a global
 *     of 1.0, so each expert contraction is W4A4 with exact block products.
 *   - Top-k ties go to the lower expert index; slots are ordered by logit
 *     descending.  Indices are those of the exact logits: the kernel
 *     ranks fp32 logits, certifies the ranking with a rigorous error bound,
 *     and re-ranks uncertain candidates from compensated double-fp32 sums
 *     (about 2^-48 relative error).
 *   - Reductions are in a fixed order with no atomics on values, so results
 *     are bit-identical run to run ([PR385] "Correctness" traces run-to-run
 *     divergence to bf16 atomics in the expert kernels).
 *
 * Conventions for every entry point:
 *   - Return FTMOE_OK (0) or a negative ftmoe_status; nothing traps or aborts.
 *   - "device" pointers are CUDA device memory of the handle's device;
 *     "host" pointers are ordinary host memory.  All arrays are row-major and
 *     contiguous.  Device pointers must be 16-byte aligned.
 *   - ftmoe_stream_t is a cudaStream_t (NULL = the legacy default stream).
 *   - The caller owns x, out, the aux buffers and the stream; the library
 *     owns the banks and its workspace.
 */
#ifndef FTMOE_H_
#define FTMOE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FTMOE_ABI_VERSION 3

typedef void* ftmoe_stream_t; /* a cudaStream_t */

typedef enum {
  FTMOE_OK = 0,
  FTMOE_ERR_INVALID_ARG = -1,      /* bad size, NULL pointer, T > max_tokens, ... */
  FTMOE_ERR_ALIGNMENT = -2,        /* i0 or I_loc not a multiple of 16, unaligned pointer */
  FTMOE_ERR_NOT_LOADED = -3,       /* forward on a layer whose bank was never loaded */
  FTMOE_ERR_SLICE_OUT_OF_RANGE = -4, /* forward window not inside the loaded window */
  FTMOE_ERR_OOM = -5,              /* a device or pinned allocation failed */
  FTMOE_ERR_CUDA = -6,             /* a CUDA runtime call failed (details: ftmoe_last_cuda_error) */
  FTMOE_ERR_TIMEOUT = -7,          /* a bounded device-side wait ran out */
  FTMOE_ERR_FAULT_INJECTED = -8,   /* FTMOE_FAULT selected this call to fail */
  FTMOE_ERR_DEVICE = -9,           /* no device, or not a compute capability 10.3 device */
  FTMOE_ERR_DEVICE_CHECK = -10,    /* an in-kernel range check failed (see ftmoe_check_status) */
  FTMOE_ERR_TOO_LARGE = -11        /* sizes exceed the fixed scratch of ftmoe_route_static */
} ftmoe_status;

/* out_flags of ftmoe_forward: the output type, optionally OR-ed with
 * ACCUMULATE and with ACT_BF16 */
enum {
  FTMOE_OUT_BF16 = 0,        /* out is bf16 [T, H] */
  FTMOE_OUT_FP32 = 1,        /* out is fp32 [T, H] */
  FTMOE_OUT_ACCUMULATE = 0x100, /* fp32 only: out += this window's partial, one rounding per add */
  FTMOE_ACT_BF16 = 0x200     /* W4A16 numerics: the routed experts take the bf16 x as it is and keep
                                their intermediate in bf16, weights dequantised in registers (the
                                weight-only 4-bit kernel the pages' review thread selects, [PR385]
                                mirror, kernel-selection fix); CUDA cores, meant for decode sizes;
                                resident mode only.  Default (flag clear): W4A4, activations NVFP4. */
};

typedef struct ftmoe_handle ftmoe_handle; /* opaque; library-owned */

typedef struct {
  int32_t abi_version;     /* = FTMOE_ABI_VERSION */
  int32_t H;               /* hidden size, multiple of 16 */
  int32_t I;               /* routed intermediate size, multiple of 16 */
  int32_t E;               /* routed experts, 1..1024 */
  int32_t top_k;           /* 1..min(E, 32) */
  int32_t I_shared;        /* shared-expert intermediate size, multiple of 16 (0 = no shared expert) */
  int32_t num_layers;      /* layers this handle holds banks for */
  int32_t max_tokens;      /* largest T a forward accepts; sizes the workspace once */
  int32_t norm_topk_prob;  /* 1: renormalise over the k chosen; 0: full-softmax probabilities */
  int32_t has_router_bias; /* 1: banks carry a per-expert router bias [E] */
  int64_t hbm_slot_bytes;  /* 0: all banks resident in HBM; > 0: offload mode.  The banks stay in
                              pinned host memory and the handle keeps
                              floor(hbm_slot_bytes / expert window bytes) expert slots in HBM,
                              shared by all layers, filled least-recently-used first (PR #385
                              "What this adds": a fraction of the experts resident, the rest
                              streamed every step).  Expert window bytes = 2*Iw*(H/2 + H/16 + 4)
                              + H*(Iw/2 + Iw/16 + 4) for the loaded window Iw; a slot physically
                              also holds the tensor-core copy of the scales (about 1/8 more). */
} ftmoe_config;

/* One layer's weights, as given to ftmoe_load_bank.  Every array is the full
 * (unsliced) tensor; the loader keeps only the window it is asked for.
 * Pointers are host memory when on_device == 0, else device memory. */
typedef struct {
  const float* router_w;       /* [E, H] fp32 */
  const float* router_bias;    /* [E] fp32, or NULL (required iff has_router_bias) */
  const uint8_t* gu_codes;     /* [E, 2I, H/2]  E2M1 pairs, element 2j in the low nibble */
  const uint8_t* gu_scales;    /* [E, 2I, H/16] E4M3 (fn) scale per 16-block */
  const float* gu_global;      /* [E, 2I]       fp32 per-row global */
  const uint8_t* dn_codes;     /* [E, H, I/2] */
  const uint8_t* dn_scales;    /* [E, H, I/16] */
  const float* dn_global;      /* [E, H] */
  const uint16_t* sh_gate_up;  /* [2*I_shared, H] bf16, gate rows first (NULL iff I_shared == 0) */
  const uint16_t* sh_down;     /* [H, I_shared] bf16 */
  const uint16_t* sh_gate;     /* [H] bf16 shared-expert gate vector */
  int32_t on_device;           /* 0 = host pointers, 1 = device pointers */
} ftmoe_bank_desc;

/* Optional outputs of ftmoe_forward (caller-owned device buffers; any may be NULL). */
typedef struct {
  int32_t* topk_idx;  /* [T, top_k] expert of each slot, slots by logit descending */
  float* topk_w;      /* [T, top_k] routing weight of each slot */
  int32_t* offsets;   /* [E + 1] first sorted position of each expert; offsets[E] = T*top_k */
  int32_t* perm;      /* [T*top_k] pair id p = t*top_k + j at each sorted position */
  int32_t* inv;       /* [T*top_k] sorted position of each pair id */
  float* logits;      /* [T, E] router logits (bias included) as the fast pass computed them,
                         before any re-rank of uncertain tokens */
  /* Each pair's quantised intermediate h = SiLU(G_gate) * G_up (NVFP4, global
     1.0, 16-blocks along the window), rows in sorted-position order:
     h_codes [T*top_k, I_loc/2] (two E2M1 codes a byte, low nibble first),
     h_scales [T*top_k, I_loc/16] (E4M3).  Written by ftmoe_forward's
     tensor-core prefill path only (resident banks, T > 32 and the shapes it
     takes); other paths and calls leave them untouched. */
  uint8_t* h_codes;
  uint8_t* h_scales;
} ftmoe_aux;

typedef struct {
  int32_t touched_experts;  /* distinct experts routed to by the last forward of this layer */
  int32_t resident_slots;   /* offload mode: HBM expert slots; resident mode: E */
  int64_t touched_bytes;    /* routed expert bytes the last forward read (window-restricted) */
  int64_t hits, misses;     /* offload mode: cumulative slot hits / misses of this layer */
  int64_t h2d_bytes;        /* offload mode: cumulative host->device expert bytes of this layer */
  double residency;         /* offload mode: resident slots / E; resident mode: 1.0 */
  int32_t device_status;    /* last device status word read by ftmoe_check_status */
  int64_t reranked_tokens;  /* cumulative tokens (all layers) whose top-k needed re-ranking */
  int64_t touched_total;    /* cumulative touched experts over every forward (all layers) */
} ftmoe_stats;

/* Create a handle on CUDA device `device` for layers of the given shape.
 * The shape is that of one MoE layer of the pages' model: E routed experts
 * with top_k chosen per token, gate_up [2I, H] and down [H, I] per expert,
 * a shared expert of intermediate I_shared gated by sigmoid(g . x)
 * ([PR385] "What this adds", first and third bullets; [I62] "What it
 * touches" for the [2I, H] / [H, I] shapes).  hbm_slot_bytes > 0 selects the
 * offload backend the pages are about: banks in pinned host memory and a
 * fraction of the experts resident in HBM slots ([PR385] "What this adds";
 * [I62] "Why TP=2 loses today").
 * Allocates the workspace for config->max_tokens (offload mode: also the
 * copy stream; the HBM slot pool follows at the first ftmoe_load_bank, once
 * the record size is known), so that a forward allocates nothing and, in
 * resident mode, can be captured in a CUDA graph ([I62] "The fix that
 * fits": "CUDA graphs unaffected. Shapes stay static").  Validates the config
 * (INVALID_ARG, ALIGNMENT) and the device (DEVICE).  On success *out owns
 * everything until ftmoe_destroy; on failure *out is NULL and nothing is
 * left allocated. */
int ftmoe_create(const ftmoe_config* config, int device, ftmoe_handle** out);

/* Load layer `layer`'s weights, keeping the intermediate window
 * [i0, i0 + I_loc) of every routed expert and of the shared expert: gate rows
 * [i0, i0+I_loc) and up rows [I+i0, I+i0+I_loc) of gate_up with their scales
 * and globals, and columns [i0, i0+I_loc) of down with their scale columns;
 * down keeps all H of its per-row globals ([I62] "What it touches": two
 * disjoint row ranges and a column slice; I/tp must stay a multiple of the
 * block size).  i0 and I_loc must be multiples of 16 (ALIGNMENT) and the
 * window inside [0, I) (INVALID_ARG).  The router and the shared gate vector
 * are loaded whole.  The call copies what it keeps (to HBM, or in offload mode
 * to pinned host memory) and synchronises `stream` before returning, so the
 * caller may free its buffers afterwards.  Loading a layer again replaces it. */
int ftmoe_load_bank(ftmoe_handle* h, int layer, const ftmoe_bank_desc* desc, int i0, int I_loc,
                    ftmoe_stream_t stream);

/* One forward of layer `layer` over T tokens (0 <= T <= max_tokens) for the
 * intermediate window [i0, i0 + I_loc), which must lie inside the loaded
 * window (SLICE_OUT_OF_RANGE) and be 16-aligned (ALIGNMENT).
 * It computes the partial output that a tensor-parallel rank owning that
 * window of every expert and of the shared expert would compute: the
 * replicated router, softmax and top-k (renormalised when norm_topk_prob is
 * set), the windowed gate_up rows, SwiGLU, the windowed down columns, and
 * routed + sigmoid(gate) * shared formed before any reduction ([PR385] "What
 * this adds", first to third bullets; [I62] "The fix that fits": the down
 * projection yields partial sums, and its first comment: norm_topk_prob and
 * a replicated router make the plain SUM of the partials exact).  The sums
 * run in a fixed order with no atomics on values, so a repeated call gives
 * the same bits ([PR385] "Correctness").
 *   x:   device, bf16 [T, H]
 *   out: device, [T, H] of the type out_flags names; must not alias x.
 *        With FTMOE_OUT_ACCUMULATE (fp32 only) the window's partial is added
 *        to out, so running the windows of a partition of I one after another
 *        into one buffer gives the full layer in a fixed order.
 *   aux: NULL or optional routing outputs (see ftmoe_aux).
 * Routing always uses the full replicated router.  Asynchronous on `stream`;
 * at prefill sizes the shared expert's products run on a stream of the
 * handle that waits for `stream`'s earlier work and that `stream` waits for
 * before the combine, so the call's work stays ordered within `stream`.
 * Resident mode does no host synchronisation and may be captured in a CUDA
 * graph (the capture follows the fork and the join).  Offload mode reads the step's routing back to the host once per
 * call (one synchronisation) to plan its slot copies; a forward touching more
 * experts than there are slots runs its experts in batches of at most the
 * slot count; offload needs the tensor-core shapes (H a multiple of 256,
 * windows multiples of 64 and at least 256 wide; INVALID_ARG otherwise) and
 * is not capturable.  T == 0 returns OK and does nothing. */
int ftmoe_forward(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags,
                  int i0, int I_loc, const ftmoe_aux* aux, ftmoe_stream_t stream);

/* Layers [0, num_layers) in sequence over T tokens, each on the previous
 * one's output renormalised by its RMS (x <- bf16(y / sqrt(mean(y^2) + 1e-6)),
 * no residual), as in a stack of MoE layers with nothing in between.
 *   x:   device bf16 [T, H] (read only)
 *   out: device bf16 [T, H], the last layer's output
 * Uses the whole loaded window of every layer.  Asynchronous; capturable in a
 * CUDA graph in resident mode. */
int ftmoe_forward_stack(ftmoe_handle* h, const void* x, int T, void* out, ftmoe_stream_t stream);

/* The renorm between the layers of ftmoe_forward_stack, on its own (the same
 * kernel): x[t] = bf16(y[t] / sqrt(mean_h(y[t][h]^2) + 1e-6)) for t < T,
 * sum of squares in fp32 (stack workload: "renormalised by RMS between
 * layers, with no attention").
 *   y: device fp32 [T, H];  x: device bf16 [T, H] (must not alias y)
 * Asynchronous on `stream`.  Returns FTMOE_ERR_INVALID_ARG for null pointers
 * or H, T < 0. */
int ftmoe_rms_renorm(const float* y, void* x, int T, int H, ftmoe_stream_t stream);

/* One rank's share of an expert-parallel layer: the routed slots of a
 * subset of the experts, plus optionally a window of the shared expert:
 *   out_t = sum over the slots j of token t whose expert is in the subset of
 *           w_tj * Y_(t,j)  +  sigmoid(g . x_t) * S_t over the shared window
 * (routing over all experts; shared_I_loc == 0 leaves the shared expert out).
 * expert_mask: host [E], nonzero for the experts of the subset.  Rank r of an
 * expert-parallel layer owns the experts e with e % world == r, the
 * alternative the pages weigh and reject for its all-to-all, its capture at
 * static shapes and its load imbalance under skewed routing ([I62] "Why not
 * expert parallelism proper"); giving rank r also window r of the shared
 * expert keeps the shared work evenly split, and the shares over a partition
 * of the experts and of the shared window add up to the whole layer.  It
 * exists to measure that alternative against the intermediate split on the
 * same GPU.  The routed experts use the whole loaded window; the shared
 * window [shared_i0, shared_i0 + shared_I_loc) must lie in the loaded shared
 * window (SLICE_OUT_OF_RANGE) and be 16-aligned (ALIGNMENT).  Reads the
 * routing back to the host once (one synchronisation); resident mode only;
 * T <= 32 on the tensor-core decode shapes and T > 32 on the prefill shapes
 * (INVALID_ARG otherwise). */
int ftmoe_forward_experts(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags,
                          const uint8_t* expert_mask, int shared_i0, int shared_I_loc, const ftmoe_aux* aux,
                          ftmoe_stream_t stream);

/* The combine of an intermediate-sharded layer: each of n_parts ranks (or
 * windows) computed its fp32 partial of the same T tokens (ftmoe_forward
 * with FTMOE_OUT_FP32 on its window), the partials were exchanged into one
 * device buffer parts [n_parts][n] in rank order (n = T * H), and this sums
 * every element over the ranks in rank order and rounds it once to the
 * output type of out_flags (FTMOE_OUT_BF16, FTMOE_OUT_FP32, optionally
 * FTMOE_OUT_ACCUMULATE).  The pages' TP patch combines the ranks' partials
 * of routed + sigmoid(gate) * shared with one SUM per MoE layer ([PR385]
 * "What this adds", third bullet; [I62] "The fix that fits": "No new
 * collectives"); a fixed rank order keeps that sum identical run to run
 * ([PR385] "Correctness").  parts must be 16-byte aligned.  Asynchronous. */
int ftmoe_reduce_partials(const float* parts, int n_parts, int64_t n, void* out, int out_flags,
                          ftmoe_stream_t stream);

/* Release everything the handle owns (device workspace, banks, pinned host
 * banks and HBM slots of the offload backend, its copy stream).  Safe on
 * NULL.  Synchronises nothing: the caller makes sure no forward of this
 * handle is still running on its streams. */
int ftmoe_destroy(ftmoe_handle* h);

/* Static description of a status code. */
const char* ftmoe_error_string(int code);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* ftmoe_last_cuda_error(void);

/* Per-layer counters (see ftmoe_stats): the touched experts and bytes of the
 * last forward, and, for the offload backend, the slot residency, hits,
 * misses and host-to-device bytes the pages measure the backend by ([PR385]
 * "Measurements": residency and cache slots; [I62] "Why TP=2 loses today":
 * slot counts per rank).  The routing-dependent fields are read back from
 * the device, so this call synchronises the handle's device. */
int ftmoe_get_stats(ftmoe_handle* h, int layer, ftmoe_stats* out);

/* Synchronise `stream`, read the device status word that the kernels set on a
 * failed range check or an expired bounded wait, clear it, and return OK,
 * DEVICE_CHECK or TIMEOUT.  After TIMEOUT the handle's cross-CTA counters
 * are cleared too, so the next forward starts clean.  The pages have no
 * counterpart; it is how a failure inside a kernel reaches the caller
 * without trapping the GPU. */
int ftmoe_check_status(ftmoe_handle* h, ftmoe_stream_t stream);

/* Test hook of the device-side failure path, off by default; the pages have
 * no counterpart.  While enabled (enable = 1), one CTA of every forward's
 * tensor-core decode down kernel never issues its first pipeline stage, so
 * its bounded waits give up after wait_limit_ns (0: the default limit of one
 * second): the kernel sets the status word's timeout bit, drains its copies,
 * frees its tensor memory and returns, and its output tile is not written.
 * ftmoe_check_status then returns FTMOE_ERR_TIMEOUT.  No GPU fault or trap
 * is involved.  INVALID_ARG if the handle has no tensor-core decode path. */
int ftmoe_test_withhold_stage(ftmoe_handle* h, int enable, int64_t wait_limit_ns);

/* Per-kernel timing.  While enabled, every kernel the handle launches is
 * bracketed by two CUDA events recorded on its launch stream.  Reading
 * synchronises those events, returns one entry per kernel name (launches,
 * summed event time in ms) in first-launch order, and clears the record.
 * Recording stays off by default; the events cost a few microseconds of host
 * time per launch.  n_out receives the number of entries (<= max_entries). */
typedef struct {
  char name[48];
  int64_t launches;
  double total_ms;
} ftmoe_kernel_time;

int ftmoe_profile_enable(ftmoe_handle* h, int enable);
int ftmoe_profile_read(ftmoe_handle* h, ftmoe_kernel_time* out, int max_entries, int* n_out);

/* NVFP4-quantise fp32 weight rows on the device (a load-time tool; the same
 * block arithmetic the forward applies to activations):
 *   g = fp32(row_amax / 2688); per 16-block s = E4M3(fp32(fp32(amax / 6) / g));
 *   code = E2M1(fp32(w / fp32(dec(s) * g))), round-to-nearest-even and
 *   saturating; zero rows, zero scales and zero denominators give zero codes.
 *   w:       device fp32 [rows, K], K a multiple of 16
 *   codes:   device [rows, K/2]; scales: device [rows, K/16]; globals: device fp32 [rows]
 * Asynchronous on `stream`. */
int ftmoe_quantize_weights(const float* w, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                           float* globals, ftmoe_stream_t stream);

/* Routing that allocates nothing.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot call cudaMalloc when they
 * route: a serving runtime that has given all free device memory to its KV
 * cache and graph pools up front, a host that forbids device allocations
 * from plugins, or code running while a CUDA graph is captured.
 *
 * It runs the same router, top-k and counting-sort kernels as ftmoe_forward
 * and returns what ftmoe_forward's aux outputs return, with no handle.  All
 * pointers are device memory of the current device:
 *   x:        bf16 [T, H] (16-byte aligned), H a multiple of 16
 *   router_w: fp32 [E, H] (16-byte aligned); router_bias: fp32 [E] or NULL
 *   topk_idx [T, top_k], topk_w [T, top_k], offsets [E + 1],
 *   perm [T*top_k], inv [T*top_k]: outputs, as in ftmoe_aux.
 * Its scratch is one fixed array in the library's device image (287 KB per
 * device that loads the library, held until the process exits),
 * which bounds the sizes: T <= 1024, E <= 1024, T*E <= 16384,
 * T*H <= 262144 and H <= 8192; larger problems return FTMOE_ERR_TOO_LARGE.
 * The first call on a device looks up that array's device address (and sets
 * the kernels' shared-memory limits); make that first call before any stream
 * capture.  Every call shares the one array, so calls whose kernels overlap
 * on the GPU (different streams, or several threads) race: serialise them.
 * Asynchronous on `stream`; calls no allocating routine. */
int ftmoe_route_static(const void* x, int T, int H, const float* router_w, const float* router_bias, int E,
                       int top_k, int norm_topk_prob, int32_t* topk_idx, float* topk_w, int32_t* offsets,
                       int32_t* perm, int32_t* inv, ftmoe_stream_t stream);

/* Device-side checks of the latest ftmoe_route_static call on the current
 * device (the kernels' range checks: an expert index out of range is routed
 * to expert 0 and marked here).  Synchronises `stream`, reads and clears the
 * status word kept in the same fixed array, and returns OK, DEVICE_CHECK or
 * TIMEOUT.  Allocates nothing.  The pages have no counterpart. */
int ftmoe_route_static_status(ftmoe_stream_t stream);

/* Bank formats that ftmoe_slice_format slices (the pages' loader handles
 * several; [I62] "What it touches" and "Suggested staging").  Per expert, a
 * matrix W [N, K] (gate_up: N = 2I, K = H; down: N = H, K = I) is held as:
 *   NVFP4      arrays {codes [N][K/2], E4M3 scales [N][K/16], fp32 globals [N]}
 *   FP8_BLOCK  arrays {E4M3 q [N][K], fp32 scale [ceil(N/128)][ceil(K/128)]},
 *              W[n][k] = q[n][k] * scale[n/128][k/128]
 *   Q4_0       array  {blocks [N][K/32][18]}: fp16 scale d, then 16 bytes of
 *              4-bit codes (byte j: element j low nibble, j+16 high nibble),
 *              value = d * (code - 8)
 *   MXFP4      arrays {blocks_t [K/2][N], UE8M0 scales_t [K/32][N]}: stored
 *              transposed, byte [j][n] holds elements (n, 2j) low and
 *              (n, 2j+1) high, value = e2m1 * 2^(scale - 127) */
typedef enum {
  FTMOE_FMT_NVFP4 = 0,
  FTMOE_FMT_FP8_BLOCK = 1,
  FTMOE_FMT_Q4_0 = 2,
  FTMOE_FMT_MXFP4 = 3
} ftmoe_format;

enum { FTMOE_MAT_GATE_UP = 0, FTMOE_MAT_DOWN = 1 };

/* Slice E experts' gate_up or down matrix, held in `format`, to the
 * intermediate window [i0, i0 + I_loc) ([I62] "What it touches": gate_up
 * keeps two disjoint row ranges, gate rows [i0, i0+I_loc) then up rows
 * [I+i0, I+i0+I_loc); down keeps the columns [i0, i0+I_loc); mxfp4, stored
 * transposed, slices gate_up along its columns and down along its rows; the
 * NVFP4 down row globals stay whole).  src[i] / dst[i] are device pointers
 * to the format's arrays in the order listed above, for all E experts back
 * to back; the sliced arrays have the same layout at I_loc in place of I
 * (fp8_block: whole 128-row scale tiles of each part).  i0, I_loc, I and H
 * must be multiples of the format's block size (16 NVFP4, 128 FP8_BLOCK,
 * 32 Q4_0 and MXFP4: [I62] "Divisibility"), else FTMOE_ERR_ALIGNMENT; a
 * window outside [0, I) is FTMOE_ERR_INVALID_ARG.  Asynchronous on
 * `stream`; a load-time step, not part of the forward. */
int ftmoe_slice_format(int format, int matrix, int E, int H, int I, int i0, int I_loc, const void* const* src,
                       void* const* dst, ftmoe_stream_t stream);

/* NVFP4-quantise bf16 activation rows with the global fixed at 1.0 (the
 * forward's own activation quantiser, exposed for testing):
 *   a: device bf16 [rows, K]; codes [rows, K/2]; scales [rows, K/16]. */
int ftmoe_quantize_activations(const void* a, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                               ftmoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FTMOE_H_ */
