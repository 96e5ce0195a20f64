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

#define FTMOE_ABI_VERSION 2

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

/* out_flags of ftmoe_forward: the output type, optionally OR-ed with ACCUMULATE */
enum {
  FTMOE_OUT_BF16 = 0,        /* out is bf16 [T, H] */
  FTMOE_OUT_FP32 = 1,        /* out is fp32 [T, H] */
  FTMOE_OUT_ACCUMULATE = 0x100 /* fp32 only: out += this window's partial, one rounding per add */
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
 * Allocates the workspace for config->max_tokens (offload mode: also the
 * copy stream; the HBM slot pool follows at the first ftmoe_load_bank, once
 * the record size is known).  Validates the config (INVALID_ARG, ALIGNMENT)
 * and the device (DEVICE).  On success *out owns everything until
 * ftmoe_destroy. */
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
 *   x:   device, bf16 [T, H]
 *   out: device, [T, H] of the type out_flags names; must not alias x.
 *        With FTMOE_OUT_ACCUMULATE (fp32 only) the window's partial is added
 *        to out, so running the windows of a partition of I one after another
 *        into one buffer gives the full layer in a fixed order.
 *   aux: NULL or optional routing outputs (see ftmoe_aux).
 * Routing always uses the full replicated router.  Asynchronous on `stream`;
 * resident mode does no host synchronisation and may be captured in a CUDA
 * graph.  Offload mode reads the step's routing back to the host once per
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

/* Release everything the handle owns.  Safe on NULL. */
int ftmoe_destroy(ftmoe_handle* h);

/* Static description of a status code. */
const char* ftmoe_error_string(int code);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* ftmoe_last_cuda_error(void);

/* Per-layer counters (see ftmoe_stats).  The routing-dependent fields are
 * read back from the device, so this call synchronises the handle's device. */
int ftmoe_get_stats(ftmoe_handle* h, int layer, ftmoe_stats* out);

/* Synchronise `stream`, read the device status word that the kernels set on a
 * failed range check or an expired bounded wait, clear it, and return OK,
 * DEVICE_CHECK or TIMEOUT. */
int ftmoe_check_status(ftmoe_handle* h, ftmoe_stream_t stream);

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

/* NVFP4-quantise bf16 activation rows with the global fixed at 1.0 (the
 * forward's own activation quantiser, exposed for testing):
 *   a: device bf16 [rows, K]; codes [rows, K/2]; scales [rows, K/16]. */
int ftmoe_quantize_activations(const void* a, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                               ftmoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FTMOE_H_ */
