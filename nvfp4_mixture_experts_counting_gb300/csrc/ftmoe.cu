// Host side of the ftmoe C ABI: handle, validation, bank loading (window
// slicing), workspace, forward orchestration, stats and status.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/ftmoe.h"
#include "kernels.h"
#include "slot_cache.h"

namespace ftmoe {
cudaError_t route_set_smem_limits(int H, int E);
cudaError_t experts_set_smem_limits(int H, int I);
thread_local Profiler* g_prof = nullptr;
}  // namespace ftmoe

using namespace ftmoe;

namespace {

// Records a pair of CUDA events around each launch; events are pooled.
class EventProfiler final : public Profiler {
 public:
  struct Rec { std::string name; cudaEvent_t a, b; };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  std::string pending;
  cudaEvent_t pending_ev = nullptr;

  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void begin(const char* name, cudaStream_t s) override {
    pending = name;
    pending_ev = get();
    cudaEventRecord(pending_ev, s);
  }
  void end(cudaStream_t s) override {
    cudaEvent_t b = get();
    cudaEventRecord(b, s);
    recs.push_back({pending, pending_ev, b});
    pending_ev = nullptr;
  }
  ~EventProfiler() override {
    for (auto& r : recs) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
    for (auto e : pool) cudaEventDestroy(e);
  }
};

// Sets the thread's profiler for the duration of one entry-point call.
struct ProfScope {
  Profiler* saved;
  explicit ProfScope(Profiler* p) : saved(g_prof) { g_prof = p; }
  ~ProfScope() { g_prof = saved; }
};

thread_local std::string g_last_cuda_error;

int cuda_fail(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  g_last_cuda_error = buf;
  return FTMOE_ERR_CUDA;
}

#define CK(call)                                          \
  do {                                                    \
    cudaError_t _e = (call);                              \
    if (_e != cudaSuccess) return cuda_fail(_e, #call);   \
  } while (0)

// Host-side fault injection: FTMOE_FAULT is a comma-separated list of names.
bool fault(const char* name) {
  const char* f = getenv("FTMOE_FAULT");
  if (!f || !*f) return false;
  std::string s(f);
  size_t pos = 0;
  while (pos <= s.size()) {
    size_t c = s.find(',', pos);
    if (c == std::string::npos) c = s.size();
    if (s.compare(pos, c - pos, name) == 0) return true;
    pos = c + 1;
  }
  return false;
}

inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

struct Layer {
  bool loaded = false;
  int li0 = 0, lIw = 0;    // loaded routed window
  int sli0 = 0, slIw = 0;  // loaded shared window
  RecLayout lay{};
  float* router_w = nullptr;
  float* router_bias = nullptr;
  uint8_t* bank = nullptr;  // E records
  uint8_t** rec_dev = nullptr;  // [E] record pointers (device)
  uint16_t* sh_gu = nullptr;
  uint16_t* sh_dn = nullptr;
  uint16_t* sh_gate = nullptr;
  uint16_t* router_wcat = nullptr;  // [E][3H] bf16 parts of the router rows (tensor-core router)
  float* router_wnorm = nullptr;    // [E]
  // offload mode
  uint8_t* host_bank = nullptr;     // pinned host: E records
  int32_t* rec_z_dev = nullptr;     // [E] slot of each expert in the current batch
  uint8_t* active_dev = nullptr;    // [E] experts of the current batch
  int last_T = 0;
  int last_I_loc = 0;
  int last_touched = 0;  // offload mode: touched experts of the last forward (read on the host)
};

}  // namespace

struct ftmoe_handle {
  ftmoe_config cfg{};
  int device = 0;
  int num_sms = 0;
  std::vector<Layer> layers;
  // workspace
  unsigned char* ws = nullptr;
  size_t ws_bytes = 0;
  RouteArgs r{};  // workspace pointers for routing (inputs filled per call)
  uint16_t* hs = nullptr;
  uint8_t* hq_codes = nullptr;
  uint8_t* hq_scales = nullptr;
  float* Y = nullptr;
  float* S = nullptr;
  float* stack_y = nullptr;
  uint16_t* stack_x[2] = {nullptr, nullptr};
  uint32_t* status = nullptr;
  int* counter = nullptr;  // arrival counter of the decode routing kernel
  int* gu_split = nullptr;  // decode gate_up work split, one entry per SM + 1
  // prefill (tensor-core) path buffers, present when the shapes allow it
  int64_t pf_pad_max = 0;
  int32_t* pf_pad_off = nullptr;
  uint8_t* pf_xg = nullptr;
  uint8_t* pf_xg_sf = nullptr;
  uint8_t* pf_hq = nullptr;
  uint8_t* pf_hq_sf = nullptr;
  bool pf_enabled = false;
  // offload mode: HBM slot pool, LRU placement, copy stream, pinned staging
  bool offload = false;
  SlotCache cache;
  uint8_t* slot_pool = nullptr;
  int64_t slot_rec_bytes = 0;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ev_compute = nullptr, ev_copied = nullptr;
  // prefill: the shared expert's GEMMs on a side stream, forked at the start
  // of a forward and joined before the combine
  cudaStream_t side_stream = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  int32_t* h_touched = nullptr;   // pinned [E + 1]: touched experts, then their count
  unsigned char* h_stage = nullptr;  // pinned per-batch tables
  size_t stage_bytes = 0;
  int max_batches = 0;
  float* off_y = nullptr;         // [T][H] fp32 sum of a batched decode forward
  std::vector<int64_t> h2d_bytes;
  // tensor-core decode buffers
  bool dtc_enabled = false;
  uint8_t* dtc_hsf = nullptr;
  float* dtc_gpart = nullptr;
  int* dtc_counter = nullptr;
  float* dtc_rpart = nullptr;  // router K-chunk partial logits [chunks][T][E]
  int dtc_groups = 0;
  uint32_t last_status = 0;
  EventProfiler* prof = nullptr;  // non-null while per-kernel timing is enabled
  // expert-subset forwards (ftmoe_forward_experts), made at the first call
  int32_t* ep_host = nullptr;   // pinned [2E + 4]: touched experts and count, then the subset list
  uint8_t* ep_mask = nullptr;   // device [E]: experts of the subset
  float* ep_w = nullptr;        // device [P]: routing weights with the other experts' slots zeroed
  // test hook of the device-side failure path (ftmoe_test_withhold_stage)
  int test_withhold = 0;
  uint64_t test_wait_ns = 0;
};

namespace ftmoe {
// Bound on the tensor-core router's error relative to ||x|| * ||w|| (tokens
// whose top-k the bounds cannot certify are re-ranked with compensated
// sums).  Empirical: the largest relative error measured against fp64
// logits on the prefill layer (T = 4096 and 16384, four seeds) was 2^-19.5;
// 2^-15 leaves a margin above 16.
constexpr float kRouterKappa = 1.0f / 32768.0f;
// The same bound for the decode router, whose tensor-core sums run over
// chunks of 256 products and are then added in fp32 (that addition has its
// own rigorous term in the top-k kernel).  Empirical: the largest error of
// the whole logit measured against fp64 on the decode layer (T = 32, 40
// seeds) was 2^-24.6 ||x|| ||w||; 2^-20 leaves a margin above 16.
constexpr float kRouterKappaSplit = 1.0f / 1048576.0f;

RecLayout make_rec_layout(int H, int Iw) {
  RecLayout L{};
  int64_t o = 0;
  L.gu_codes = o;  o = align_up(o + (int64_t)2 * Iw * (H / 2), 256);
  L.gu_scales = o; o = align_up(o + (int64_t)2 * Iw * (H / 16), 256);
  L.dn_codes = o;  o = align_up(o + (int64_t)H * (Iw / 2), 256);
  L.dn_scales = o; o = align_up(o + (int64_t)H * (Iw / 16), 256);
  L.gu_global = o; o = align_up(o + (int64_t)2 * Iw * 4, 256);
  L.dn_global = o; o = align_up(o + (int64_t)H * 4, 256);
  if (H % 256 == 0 && Iw % 64 == 0) {
    L.gu_sf_bytes = (int64_t)2 * Iw * (H / 16);
    L.gu_sf = o; o = align_up(o + L.gu_sf_bytes, 256);
    L.dn_sf = o; o = align_up(o + (int64_t)H * (Iw / 16), 256);
  }
  L.bytes = o;
  return L;
}
}  // namespace ftmoe

namespace {

void free_layer(Layer& L) {
  cudaFree(L.router_w);
  cudaFree(L.router_bias);
  cudaFree(L.bank);
  cudaFree(L.rec_dev);
  cudaFree(L.sh_gu);
  cudaFree(L.sh_dn);
  cudaFree(L.sh_gate);
  cudaFree(L.router_wcat);
  cudaFree(L.router_wnorm);
  if (L.host_bank) cudaFreeHost(L.host_bank);
  cudaFree(L.rec_z_dev);
  cudaFree(L.active_dev);
  L = Layer{};
}

int validate_config(const ftmoe_config* c) {
  if (!c || c->abi_version != FTMOE_ABI_VERSION) return FTMOE_ERR_INVALID_ARG;
  if (c->H <= 0 || c->I <= 0 || c->E <= 0 || c->top_k <= 0 || c->num_layers <= 0 ||
      c->max_tokens < 0 || c->I_shared < 0)
    return FTMOE_ERR_INVALID_ARG;
  if (c->H % 16 || c->I % 16 || c->I_shared % 16) return FTMOE_ERR_ALIGNMENT;
  if (c->H > 8192 || c->I > 8192 || c->I_shared > 4096 || c->E > 1024 || c->top_k > 32 ||
      c->top_k > c->E || c->max_tokens > (1 << 20))
    return FTMOE_ERR_INVALID_ARG;
  if (c->hbm_slot_bytes < 0) return FTMOE_ERR_INVALID_ARG;
  return FTMOE_OK;
}

// Shared window for a routed window (I_s may differ from I).
bool shared_window(const ftmoe_config& c, int i0, int I_loc, int* si0, int* sI) {
  if (c.I_shared == 0) { *si0 = 0; *sI = 0; return true; }
  if (c.I_shared == c.I) { *si0 = i0; *sI = I_loc; return true; }
  int64_t a = (int64_t)i0 * c.I_shared, b = (int64_t)I_loc * c.I_shared;
  if (a % c.I || b % c.I) return false;
  *si0 = (int)(a / c.I);
  *sI = (int)(b / c.I);
  return (*si0 % 16 == 0) && (*sI % 16 == 0);
}

}  // namespace

extern "C" {

const char* ftmoe_error_string(int code) {
  switch (code) {
    case FTMOE_OK: return "ok";
    case FTMOE_ERR_INVALID_ARG: return "invalid argument";
    case FTMOE_ERR_ALIGNMENT: return "misaligned size or pointer (sizes and windows must be multiples of 16, pointers 16-byte aligned)";
    case FTMOE_ERR_NOT_LOADED: return "layer bank not loaded";
    case FTMOE_ERR_SLICE_OUT_OF_RANGE: return "forward window is not inside the loaded window";
    case FTMOE_ERR_OOM: return "out of memory";
    case FTMOE_ERR_CUDA: return "CUDA runtime error";
    case FTMOE_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case FTMOE_ERR_FAULT_INJECTED: return "fault injected (FTMOE_FAULT)";
    case FTMOE_ERR_DEVICE: return "no usable device (needs compute capability 10.3)";
    case FTMOE_ERR_DEVICE_CHECK: return "an in-kernel range check failed";
    case FTMOE_ERR_TOO_LARGE: return "sizes exceed the fixed scratch of the allocation-free routing entry point";
    default: return "unknown status";
  }
}

const char* ftmoe_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int ftmoe_create(const ftmoe_config* config, int device, ftmoe_handle** out) {
  if (!out) return FTMOE_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_config(config);
  if (rc) return rc;
  if (fault("oom")) return FTMOE_ERR_OOM;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return FTMOE_ERR_DEVICE;
  }
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, device));
  if (prop.major != 10 || prop.minor != 3) return FTMOE_ERR_DEVICE;
  CK(cudaSetDevice(device));
  auto* h = new ftmoe_handle();
  h->cfg = *config;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->layers.resize(config->num_layers);
  const ftmoe_config& c = *config;
  const int64_t T = c.max_tokens > 0 ? c.max_tokens : 1;
  const int64_t P = T * c.top_k;
  // workspace carve-up
  struct Part { void** p; int64_t bytes; };
  std::vector<Part> parts = {
      {(void**)&h->r.logits, T * c.E * 4},   {(void**)&h->r.err, T * c.E * 4},
      {(void**)&h->r.topk_idx, P * 4},       {(void**)&h->r.topk_w, P * 4},
      {(void**)&h->r.xq_codes, T * c.H / 2}, {(void**)&h->r.xq_scales, T * c.H / 16},
      {(void**)&h->r.sigma, T * 4},          {(void**)&h->r.offsets, (int64_t)(c.E + 1) * 4},
      {(void**)&h->r.xnorm, T * 4},
      {(void**)&h->r.perm, P * 4},           {(void**)&h->r.inv, P * 4},
      {(void**)&h->r.touched, (int64_t)c.E * 4}, {(void**)&h->r.n_touched, 16},
      {(void**)&h->r.emask, (int64_t)c.E * 4},
      {(void**)&h->hs, T * (c.I_shared > 0 ? c.I_shared : 16) * 2},
      // intermediate rows padded to 16 bytes (the decode path copies them in bulk)
      {(void**)&h->hq_codes, P * align_up(c.I * 2, 16)}, {(void**)&h->hq_scales, P * align_up(c.I / 16 * 4, 16)},
      {(void**)&h->Y, P * c.H * 4},          {(void**)&h->S, T * c.H * 4},
      {(void**)&h->stack_y, T * c.H * 4},    {(void**)&h->stack_x[0], T * c.H * 2},
      {(void**)&h->stack_x[1], T * c.H * 2}, {(void**)&h->status, 16},
      {(void**)&h->counter, 16},             {(void**)&h->r.n_rerank, 16},
      {(void**)&h->r.touched_total, 16},
      {(void**)&h->off_y, c.hbm_slot_bytes > 0 ? T * c.H * 4 : 16},
      {(void**)&h->gu_split, (int64_t)(prop.multiProcessorCount + 1) * 4},
  };
  // counts of the many-CTA counting sort (chunks of 4096 pairs)
  h->r.sort_max_chunks = (int)((P + 4095) / 4096);
  if (h->r.sort_max_chunks > 1)
    parts.push_back({(void**)&h->r.sort_cnt, (int64_t)h->r.sort_max_chunks * c.E * 4});
  // tensor-core decode buffers
  const char* no_tc = getenv("FTMOE_NO_TC");
  if (c.H % 256 == 0 && c.I % 64 == 0 && c.E <= 1024 && !(no_tc && no_tc[0] == '1')) {
    h->dtc_enabled = true;
    h->dtc_groups = decode_tc_groups(c.H, prop.multiProcessorCount);
    const int64_t Td = T < 32 ? T : 32;
    parts.push_back({(void**)&h->dtc_hsf, (int64_t)c.E * (c.I / 64) * 512});
    parts.push_back({(void**)&h->dtc_gpart, (int64_t)(h->dtc_groups + 1) * Td * c.H * 4});
    parts.push_back({(void**)&h->dtc_counter, (int64_t)(c.H / 128 + 1) * 4});
    if (decode_tc_router_supported(c.H, c.E))  // partial logits per K chunk of [W1 | W2 | W3]
      parts.push_back({(void**)&h->dtc_rpart, (int64_t)decode_tc_router_chunks(c.H) * Td * c.E * 4});
  }
  // tensor-core prefill buffers (padded pair order), for shapes it accepts
  if (c.max_tokens > 32 && c.H % 256 == 0 && c.I % 64 == 0 && c.E <= 1024 && !(no_tc && no_tc[0] == '1')) {
    h->pf_enabled = true;
    h->pf_pad_max = pf_pad_max(P, c.E);
    const int64_t R = h->pf_pad_max;
    parts.push_back({(void**)&h->pf_pad_off, (int64_t)(c.E + 1) * 4});
    parts.push_back({(void**)&h->pf_xg, R * c.H / 2});
    parts.push_back({(void**)&h->pf_xg_sf, R * c.H / 16});
    parts.push_back({(void**)&h->pf_hq, R * align_up(c.I / 2, 16)});
    parts.push_back({(void**)&h->pf_hq_sf, R * (c.I / 16)});
  }
  int64_t total = 0;
  for (auto& p : parts) total += align_up(p.bytes, 256);
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return FTMOE_ERR_OOM;
  }
  h->ws_bytes = total;
  int64_t off = 0;
  for (auto& p : parts) {
    *p.p = h->ws + off;
    off += align_up(p.bytes, 256);
  }
  cudaError_t e = cudaMemset(h->ws, 0, total);
  if (e == cudaSuccess) e = route_set_smem_limits(c.H, c.E);
  if (e == cudaSuccess) e = experts_set_smem_limits(c.H, c.I > c.I_shared ? c.I : c.I_shared);
  if (e == cudaSuccess) e = decode_set_smem_limits();
  if (e == cudaSuccess) e = prefill_set_smem_limits();
  if (e == cudaSuccess) e = decode_tc_set_smem_limits();
  if (e == cudaSuccess) e = w16_set_smem_limits(8192, 8192);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->side_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
  if (e == cudaSuccess && c.hbm_slot_bytes > 0) {
    h->offload = true;
    h->h2d_bytes.assign(c.num_layers, 0);
    e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_compute, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_copied, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaHostAlloc((void**)&h->h_touched, (size_t)(c.E + 1) * 4, cudaHostAllocDefault);
  }
  if (e != cudaSuccess) {
    cuda_fail(e, "create");
    ftmoe_destroy(h);  // the workspace, and the copy stream, events and pinned buffer made so far
    return FTMOE_ERR_CUDA;
  }
  h->r.status = h->status;
  *out = h;
  return FTMOE_OK;
}

int ftmoe_destroy(ftmoe_handle* h) {
  if (!h) return FTMOE_OK;
  cudaSetDevice(h->device);
  for (auto& L : h->layers) free_layer(L);
  if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
  if (h->side_stream) cudaStreamDestroy(h->side_stream);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->ev_compute) cudaEventDestroy(h->ev_compute);
  if (h->ev_copied) cudaEventDestroy(h->ev_copied);
  if (h->h_touched) cudaFreeHost(h->h_touched);
  if (h->ep_host) cudaFreeHost(h->ep_host);
  cudaFree(h->ep_mask);
  cudaFree(h->ep_w);
  if (h->h_stage) cudaFreeHost(h->h_stage);
  cudaFree(h->slot_pool);
  delete h->prof;
  cudaFree(h->ws);
  delete h;
  return FTMOE_OK;
}

int ftmoe_load_bank(ftmoe_handle* h, int layer, const ftmoe_bank_desc* d, int i0, int I_loc,
                    ftmoe_stream_t stream) {
  if (!h || !d || layer < 0 || layer >= h->cfg.num_layers) return FTMOE_ERR_INVALID_ARG;
  const ftmoe_config& c = h->cfg;
  if (i0 % 16 || I_loc % 16) return FTMOE_ERR_ALIGNMENT;
  if (I_loc <= 0 || i0 < 0 || i0 + I_loc > c.I) return FTMOE_ERR_INVALID_ARG;
  int si0, sI;
  if (!shared_window(c, i0, I_loc, &si0, &sI)) return FTMOE_ERR_ALIGNMENT;
  if (!d->router_w || !d->gu_codes || !d->gu_scales || !d->gu_global || !d->dn_codes ||
      !d->dn_scales || !d->dn_global)
    return FTMOE_ERR_INVALID_ARG;
  if ((c.has_router_bias != 0) != (d->router_bias != nullptr)) return FTMOE_ERR_INVALID_ARG;
  if (c.I_shared > 0 && (!d->sh_gate_up || !d->sh_down || !d->sh_gate)) return FTMOE_ERR_INVALID_ARG;
  if (fault("bad_bank")) return FTMOE_ERR_FAULT_INJECTED;
  CK(cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  Layer& L = h->layers[layer];
  free_layer(L);
  const int H = c.H, E = c.E, I = c.I, Iw = I_loc;
  L.lay = make_rec_layout(H, Iw);
  // resident: every record in HBM; offload: records built one at a time in
  // HBM and kept in pinned host memory, HBM slots shared by all layers
  const bool off = h->offload;
  if (off) {
    if (h->slot_pool && h->slot_rec_bytes != L.lay.bytes) return FTMOE_ERR_INVALID_ARG;  // one layout per handle
    if (!h->slot_pool) {
      const int64_t per = (int64_t)2 * Iw * (H / 2 + H / 16 + 4) + (int64_t)H * (Iw / 2 + Iw / 16 + 4);
      int64_t n = c.hbm_slot_bytes / per;
      n = std::min<int64_t>(n, (int64_t)E * c.num_layers);
      if (n < 1) return FTMOE_ERR_INVALID_ARG;
      if (cudaMalloc(&h->slot_pool, n * L.lay.bytes) != cudaSuccess) { cudaGetLastError(); return FTMOE_ERR_OOM; }
      h->slot_rec_bytes = L.lay.bytes;
      h->max_batches = (int)((E + n - 1) / n);
      h->stage_bytes = (size_t)align_up((int64_t)E * 8 + (int64_t)E * 4 + (int64_t)(E + 4) * 4 + E, 256);
      if (cudaHostAlloc((void**)&h->h_stage, h->stage_bytes * h->max_batches, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        return FTMOE_ERR_OOM;
      }
      h->cache.reset((int)n, c.num_layers, E);
    }
    h->cache.reset(h->cache.slots(), c.num_layers, E);  // a reload empties every slot
  }
  const int64_t bank_bytes = off ? L.lay.bytes : L.lay.bytes * E;
  if (cudaMalloc(&L.bank, bank_bytes) != cudaSuccess || cudaMalloc(&L.rec_dev, E * sizeof(void*)) != cudaSuccess ||
      cudaMalloc(&L.router_w, (size_t)E * H * 4) != cudaSuccess) {
    cudaGetLastError();
    free_layer(L);
    return FTMOE_ERR_OOM;
  }
  if (off && (cudaHostAlloc((void**)&L.host_bank, (size_t)L.lay.bytes * E, cudaHostAllocDefault) != cudaSuccess ||
              cudaMalloc(&L.rec_z_dev, (size_t)E * 4) != cudaSuccess ||
              cudaMalloc(&L.active_dev, (size_t)E) != cudaSuccess)) {
    cudaGetLastError();
    free_layer(L);
    return FTMOE_ERR_OOM;
  }
  const cudaMemcpyKind K = cudaMemcpyDefault;
  CK(cudaMemcpyAsync(L.router_w, d->router_w, (size_t)E * H * 4, K, s));
  if (d->router_bias) {
    if (cudaMalloc(&L.router_bias, E * 4) != cudaSuccess) { free_layer(L); return FTMOE_ERR_OOM; }
    CK(cudaMemcpyAsync(L.router_bias, d->router_bias, E * 4, K, s));
  }
  const int64_t gcb = H / 2, gsb = H / 16;  // gate_up row bytes (codes, scales)
  for (int e = 0; e < E; ++e) {
    uint8_t* rec = off ? L.bank : L.bank + L.lay.bytes * e;
    const int64_t r_gate = (int64_t)e * 2 * I + i0, r_up = (int64_t)e * 2 * I + I + i0;
    CK(cudaMemcpyAsync(rec + L.lay.gu_codes, d->gu_codes + r_gate * gcb, Iw * gcb, K, s));
    CK(cudaMemcpyAsync(rec + L.lay.gu_codes + Iw * gcb, d->gu_codes + r_up * gcb, Iw * gcb, K, s));
    CK(cudaMemcpyAsync(rec + L.lay.gu_scales, d->gu_scales + r_gate * gsb, Iw * gsb, K, s));
    CK(cudaMemcpyAsync(rec + L.lay.gu_scales + Iw * gsb, d->gu_scales + r_up * gsb, Iw * gsb, K, s));
    CK(cudaMemcpyAsync(rec + L.lay.gu_global, d->gu_global + r_gate, Iw * 4, K, s));
    CK(cudaMemcpyAsync(rec + L.lay.gu_global + Iw * 4, d->gu_global + r_up, Iw * 4, K, s));
    CK(cudaMemcpy2DAsync(rec + L.lay.dn_codes, Iw / 2, d->dn_codes + (int64_t)e * H * (I / 2) + i0 / 2, I / 2,
                         Iw / 2, H, K, s));
    CK(cudaMemcpy2DAsync(rec + L.lay.dn_scales, Iw / 16, d->dn_scales + (int64_t)e * H * (I / 16) + i0 / 16,
                         I / 16, Iw / 16, H, K, s));
    CK(cudaMemcpyAsync(rec + L.lay.dn_global, d->dn_global + (int64_t)e * H, H * 4, K, s));
    if (off) {
      CK(launch_repack_sf(L.bank, L.lay, H, Iw, 1, s));
      CK(cudaMemcpyAsync(L.host_bank + (int64_t)e * L.lay.bytes, L.bank, L.lay.bytes, cudaMemcpyDeviceToHost, s));
      CK(cudaStreamSynchronize(s));  // the one staging record is reused
    }
  }
  if (off) {
    cudaFree(L.bank);
    L.bank = nullptr;
  } else {
    CK(launch_repack_sf(L.bank, L.lay, H, Iw, E, s));
  }
  if ((h->pf_enabled || h->dtc_enabled) && prefill_router_supported(H, E)) {
    if (cudaMalloc(&L.router_wcat, (size_t)E * 3 * H * 2) != cudaSuccess ||
        cudaMalloc(&L.router_wnorm, (size_t)E * 4) != cudaSuccess) {
      cudaGetLastError();
      free_layer(L);
      return FTMOE_ERR_OOM;
    }
    CK(launch_router_split(L.router_w, E, H, L.router_wcat, L.router_wnorm, s));
  }
  std::vector<uint8_t*> ptrs(E);
  for (int e = 0; e < E; ++e) ptrs[e] = off ? h->slot_pool : L.bank + L.lay.bytes * e;
  CK(cudaMemcpyAsync(L.rec_dev, ptrs.data(), E * sizeof(void*), cudaMemcpyHostToDevice, s));
  if (c.I_shared > 0) {
    if (cudaMalloc(&L.sh_gu, (size_t)2 * sI * H * 2) != cudaSuccess ||
        cudaMalloc(&L.sh_dn, (size_t)H * sI * 2) != cudaSuccess || cudaMalloc(&L.sh_gate, (size_t)H * 2) != cudaSuccess) {
      cudaGetLastError();
      free_layer(L);
      return FTMOE_ERR_OOM;
    }
    const int Is = c.I_shared;
    CK(cudaMemcpyAsync(L.sh_gu, d->sh_gate_up + (int64_t)si0 * H, (size_t)sI * H * 2, K, s));
    CK(cudaMemcpyAsync(L.sh_gu + (int64_t)sI * H, d->sh_gate_up + (int64_t)(Is + si0) * H, (size_t)sI * H * 2, K, s));
    CK(cudaMemcpy2DAsync(L.sh_dn, sI * 2, d->sh_down + si0, (size_t)Is * 2, sI * 2, H, K, s));
    CK(cudaMemcpyAsync(L.sh_gate, d->sh_gate, (size_t)H * 2, K, s));
  }
  CK(cudaStreamSynchronize(s));
  L.li0 = i0;
  L.lIw = Iw;
  L.sli0 = si0;
  L.slIw = sI;
  L.loaded = true;
  return FTMOE_OK;
}

// ---- argument builders shared by the resident and offloaded forwards

static RouteArgs route_args(ftmoe_handle* h, Layer& L, const void* x, int T) {
  const ftmoe_config& c = h->cfg;
  RouteArgs r = h->r;
  r.x = (const uint16_t*)x;
  r.router_w = L.router_w;
  r.router_bias = L.router_bias;
  r.sh_gate = c.I_shared > 0 ? L.sh_gate : nullptr;
  r.T = T;
  r.H = c.H;
  r.E = c.E;
  r.top_k = c.top_k;
  r.norm_topk_prob = c.norm_topk_prob;
  return r;
}

static ExpertArgs expert_args(ftmoe_handle* h, Layer& L, const RouteArgs& r, int T, void* out, int out_flags,
                              int i0, int I_loc) {
  const ftmoe_config& c = h->cfg;
  ExpertArgs a{};
  a.r = r;
  a.rec = L.rec_dev;
  a.lay = L.lay;
  a.win.row0 = i0 - L.li0;
  a.win.I_loc = I_loc;
  a.win.Iw = L.lIw;
  a.H = c.H;
  a.T = T;
  a.top_k = c.top_k;
  if (c.I_shared > 0) {
    int si0 = 0, sI = 0;
    shared_window(c, i0, I_loc, &si0, &sI);
    a.sh_gate_up = L.sh_gu;
    a.sh_down = L.sh_dn;
    a.s_row0 = si0 - L.sli0;
    a.s_I_loc = sI;
    a.s_Iw = L.slIw;
  }
  a.hs = h->hs;
  a.hq_codes = h->hq_codes;
  a.hq_scales = h->hq_scales;
  a.Y = h->Y;
  a.S = h->S;
  a.out = out;
  a.out_flags = out_flags;
  a.num_sms = h->num_sms;
  return a;
}

static DecodeArgs decode_args(ftmoe_handle* h, const ExpertArgs& a) {
  DecodeArgs d{};
  d.r = a.r;
  d.rec = a.rec;
  d.lay = a.lay;
  d.win = a.win;
  d.H = a.H;
  d.T = a.T;
  d.top_k = a.top_k;
  d.sh_gate_up = a.sh_gate_up;
  d.sh_down = a.sh_down;
  d.s_row0 = a.s_row0;
  d.s_I_loc = a.s_I_loc;
  d.s_Iw = a.s_Iw;
  d.hs = h->hs;
  d.hq_codes = h->hq_codes;
  d.hq_scales = h->hq_scales;
  d.hq_cpitch = decode_hq_cpitch(a.win.I_loc);
  d.hq_spitch = decode_hq_spitch(a.win.I_loc);
  d.out = a.out;
  d.out_flags = a.out_flags;
  d.counter = h->counter;
  d.gu_split = h->gu_split;
  d.num_sms = h->num_sms;
  d.pdl = 1;
  return d;
}

// The tensor-core decode kernels' extra arguments.
static void decode_tc_args(ftmoe_handle* h, Layer& L, DecodeArgs& d) {
  d.bank = h->offload ? h->slot_pool : L.bank;
  d.rec_z = h->offload ? L.rec_z_dev : nullptr;
  d.n_records = h->offload ? h->cache.slots() : h->cfg.E;
  d.hsf = h->dtc_hsf;
  d.gpart = h->dtc_gpart;
  d.dn_counter = h->dtc_counter;
  d.n_groups = h->dtc_groups;
  d.hq_cpitch = (int)align_up(d.win.I_loc / 2, 16);
  d.withhold_first_stage = h->test_withhold;
  d.wait_limit_ns = h->test_withhold ? h->test_wait_ns : 0;
  if (L.router_wcat && h->dtc_rpart && decode_tc_router_supported(h->cfg.H, h->cfg.E)) {
    d.wcat = L.router_wcat;
    d.wnorm = L.router_wnorm;
    d.rpart = h->dtc_rpart;
    d.kappa = kRouterKappaSplit;
  }
}

static PfArgs prefill_args(ftmoe_handle* h, Layer& L, const ExpertArgs& a, const void* x, void* out, int out_flags,
                           bool tc_shared, bool tc_router) {
  const ftmoe_config& c = h->cfg;
  const RouteArgs& r = a.r;
  PfArgs p{};
  p.offsets = r.offsets;
  p.perm = r.perm;
  p.xq_codes = r.xq_codes;
  p.xq_scales = r.xq_scales;
  p.bank = h->offload ? h->slot_pool : L.bank;
  p.rec_z = h->offload ? L.rec_z_dev : nullptr;
  p.n_records = h->offload ? h->cache.slots() : c.E;
  p.lay = L.lay;
  p.win = a.win;
  p.H = c.H;
  p.T = a.T;
  p.E = c.E;
  p.top_k = c.top_k;
  p.P_pad_max = (int)h->pf_pad_max;
  p.pad_off = h->pf_pad_off;
  p.xg = h->pf_xg;
  p.xg_sf = h->pf_xg_sf;
  p.hq = h->pf_hq;
  p.hq_sf = h->pf_hq_sf;
  p.hq_pitch = (int)align_up(a.win.I_loc / 2, 16);
  // the pairs' outputs in the output's precision: bf16 for a bf16 output
  // (half the bytes of the write and the read back), fp32 for an fp32 one,
  // so that fp32 window partials still add up to the full layer
  p.Y = h->Y;
  p.y_bf16 = (out_flags & 0xff) == FTMOE_OUT_BF16;
  p.status = h->status;
  if (tc_shared || tc_router) p.x = (const uint16_t*)x;
  if (tc_shared) {
    p.sh_gu = a.sh_gate_up;
    p.sh_dn = a.sh_down;
    p.s_row0 = a.s_row0;
    p.s_I_loc = a.s_I_loc;
    p.s_Iw = a.s_Iw;
    p.hs = h->hs;
    p.inv = r.inv;
    p.topk_w = r.topk_w;
    p.sigma = r.sigma;
    p.out = out;
    p.out_flags = out_flags;
    p.S = h->S;  // the any-T path's buffer, unused by the prefill path otherwise
  }
  if (tc_router) {
    p.wcat = L.router_wcat;
    p.wnorm = L.router_wnorm;
    p.xnorm = r.xnorm;
    p.router_bias = L.router_bias;
    p.logits = r.logits;
    p.err = r.err;
    p.kappa = kRouterKappa;
    // Y is not written before the routed down kernel, so the router's
    // K-split partials may use it
    p.rpart = h->Y;
    p.rpart_cap = (int64_t)(c.max_tokens > 0 ? c.max_tokens : 1) * c.top_k * c.H;
  }
  return p;
}

static int copy_aux(ftmoe_handle* h, const RouteArgs& r, int T, const ftmoe_aux* aux, cudaStream_t s) {
  if (!aux) return FTMOE_OK;
  const ftmoe_config& c = h->cfg;
  const int64_t P = (int64_t)T * c.top_k;
  if (aux->topk_idx) CK(cudaMemcpyAsync(aux->topk_idx, r.topk_idx, P * 4, cudaMemcpyDeviceToDevice, s));
  if (aux->topk_w) CK(cudaMemcpyAsync(aux->topk_w, r.topk_w, P * 4, cudaMemcpyDeviceToDevice, s));
  if (aux->offsets) CK(cudaMemcpyAsync(aux->offsets, r.offsets, (c.E + 1) * 4, cudaMemcpyDeviceToDevice, s));
  if (aux->perm) CK(cudaMemcpyAsync(aux->perm, r.perm, P * 4, cudaMemcpyDeviceToDevice, s));
  if (aux->inv) CK(cudaMemcpyAsync(aux->inv, r.inv, P * 4, cudaMemcpyDeviceToDevice, s));
  if (aux->logits) CK(cudaMemcpyAsync(aux->logits, r.logits, (int64_t)T * c.E * 4, cudaMemcpyDeviceToDevice, s));
  return FTMOE_OK;
}

static bool prefill_path(ftmoe_handle* h, Layer& L, int T, int I_loc, int row0) {
  return h->pf_enabled && T > 32 && L.lay.gu_sf_bytes && prefill_supported(h->cfg.H, h->cfg.E, I_loc, L.lIw, row0);
}

static bool decode_tc_path(ftmoe_handle* h, Layer& L, const ExpertArgs& a, int T) {
  const ftmoe_config& c = h->cfg;
  return h->dtc_enabled && decode_tc_supported(c.H, c.E, a.win.I_loc, L.lIw, a.win.row0, a.s_I_loc, a.s_Iw,
                                               a.s_row0, T, c.top_k, L.lay.gu_sf_bytes != 0);
}

static int forward_offload(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags, int i0,
                           int I_loc, const ftmoe_aux* aux, cudaStream_t s);

static int forward_impl(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags, int i0,
                        int I_loc, const ftmoe_aux* aux, cudaStream_t s) {
  if (h->offload) return forward_offload(h, layer, x, T, out, out_flags, i0, I_loc, aux, s);
  const ftmoe_config& c = h->cfg;
  Layer& L = h->layers[layer];
  RouteArgs r = route_args(h, L, x, T);
  ExpertArgs a = expert_args(h, L, r, T, out, out_flags & ~FTMOE_ACT_BF16, i0, I_loc);
  if (out_flags & FTMOE_ACT_BF16) {
    // W4A16: routing, shared gate_up, the routed experts on bf16 activations
    // (Y in sorted order), shared down + combine
    CK(launch_route(r, s));
    CK(launch_experts(a, s, kPartSharedGateUp));
    CK(launch_w16_routed(a, s));
    a.y_tiles = 0;
    CK(launch_experts(a, s, kPartTail));
    int rc = copy_aux(h, r, T, aux, s);
    if (rc) return rc;
    L.last_T = T;
    L.last_I_loc = I_loc;
    return FTMOE_OK;
  }
  const bool dtc = decode_tc_path(h, L, a, T);
  if (dtc || decode_supported(c.H, c.E, I_loc, L.lIw, a.win.row0, a.s_I_loc, a.s_Iw, a.s_row0, T, c.top_k)) {
    // decode sizes: routing, streamed gate_up, fused down + combine
    DecodeArgs d = decode_args(h, a);
    if (dtc) {
      // weights through the tensor cores: intermediates as packed codes
      decode_tc_args(h, L, d);
      CK(launch_decode_tc(d, s));
    } else {
      CK(launch_decode(d, s));
    }
  } else if (prefill_path(h, L, T, I_loc, a.win.row0)) {
    // prefill sizes: router logits, the routed GEMMs and the shared expert
    // on the tensor cores where the shapes fit them.  The shared expert needs
    // only x, so its two GEMMs (gate_up, then down into S) run on the side
    // stream while the routing and the routed GEMMs run here, and the
    // combine waits for both; the fork's event also orders them after this
    // stream's earlier work (the previous combine read S).  While the
    // per-kernel profiler is on, everything stays on one stream.
    const bool tc_shared = a.sh_gate_up && prefill_shared_supported(c.H, a.s_I_loc, a.s_Iw, a.s_row0, c.top_k);
    const bool tc_router = L.router_wcat != nullptr;
    PfArgs p = prefill_args(h, L, a, x, out, out_flags, tc_shared, tc_router);
    PfMaps maps;
    CK(prefill_make_maps(p, &maps));
    const bool fork = tc_shared && !g_prof;
    cudaStream_t ss = fork ? h->side_stream : s;
    if (fork) {
      CK(cudaEventRecord(h->ev_fork, s));
      CK(cudaStreamWaitEvent(ss, h->ev_fork, 0));
    }
    if (tc_shared) {
      CK(launch_prefill_shared_gate_up(p, maps, h->num_sms, ss));
      CK(launch_prefill_shared_down(p, maps, h->num_sms, ss));
    }
    if (fork) CK(cudaEventRecord(h->ev_join, ss));
    if (tc_router) {
      CK(launch_route(r, s, kRouteXq));
      CK(launch_prefill_router(p, maps, h->num_sms, s));
      CK(launch_route(r, s, kRouteTopk | kRouteSort));
    } else {
      CK(launch_route(r, s));
    }
    if (!tc_shared) CK(launch_experts(a, s, kPartSharedGateUp));
    CK(launch_prefill_routed(p, maps, h->num_sms, s));
    if (aux) CK(launch_prefill_export_h(p, aux->h_codes, aux->h_scales, h->num_sms, s));
    if (tc_shared) {
      if (fork) CK(cudaStreamWaitEvent(s, h->ev_join, 0));
      CK(launch_prefill_combine(p, h->num_sms, s));
    } else {
      a.y_tiles = p.y_bf16 ? 2 : 1;  // the tensor-core down kernel's layout of Y
      CK(launch_experts(a, s, kPartTail));
    }
  } else {
    CK(launch_route(r, s));
    CK(launch_experts(a, s));
  }
  int rc = copy_aux(h, r, T, aux, s);
  if (rc) return rc;
  L.last_T = T;
  L.last_I_loc = I_loc;
  return FTMOE_OK;
}

// Offload mode: route, read the touched experts back (one host
// synchronisation), then for each batch of at most slots() touched experts
// place them in HBM slots (copying the missed records from pinned host
// memory on the copy stream), point the layer's record tables at the slots
// and run the expert kernels on that batch.  With several batches the routed
// outputs add up in an fp32 buffer, converted to the caller's output at the
// end (prefill keeps every pair's Y and combines once).
static int forward_offload(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags, int i0,
                           int I_loc, const ftmoe_aux* aux, cudaStream_t s) {
  const ftmoe_config& c = h->cfg;
  Layer& L = h->layers[layer];
  const int E = c.E;
  RouteArgs r = route_args(h, L, x, T);
  ExpertArgs a = expert_args(h, L, r, T, out, out_flags, i0, I_loc);
  const bool dec = T <= 32;
  if (dec ? !decode_tc_path(h, L, a, T) : !prefill_path(h, L, T, I_loc, a.win.row0)) return FTMOE_ERR_INVALID_ARG;
  DecodeArgs d{};
  PfArgs p{};
  PfMaps maps;
  bool tc_shared = false, tc_router = false;
  // ---- routing
  if (dec) {
    d = decode_args(h, a);
    decode_tc_args(h, L, d);
    CK(launch_decode_tc(d, s, 1));
  } else {
    tc_shared = a.sh_gate_up && prefill_shared_supported(c.H, a.s_I_loc, a.s_Iw, a.s_row0, c.top_k);
    tc_router = L.router_wcat != nullptr;
    p = prefill_args(h, L, a, x, out, out_flags, tc_shared, tc_router);
    CK(prefill_make_maps(p, &maps));
    if (tc_router) {
      CK(launch_route(r, s, kRouteXq));
      CK(launch_prefill_router(p, maps, h->num_sms, s));
      CK(launch_route(r, s, kRouteTopk | kRouteSort));
    } else {
      CK(launch_route(r, s));
    }
  }
  CK(cudaMemcpyAsync(h->h_touched, r.touched, (size_t)E * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(h->h_touched + E, r.n_touched, 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  const int nt = h->h_touched[E];
  if (nt < 0 || nt > E) return FTMOE_ERR_DEVICE_CHECK;
  // the device's count is overwritten by every batch below; keep the step's
  L.last_touched = nt;
  const int S = h->cache.slots();
  const int nb = (nt + S - 1) / S;
  if (nb > h->max_batches) return FTMOE_ERR_INVALID_ARG;
  // experts already resident go first (in expert order), then the rest: when
  // the touched experts need several batches, the resident ones are all hits
  // of the first batch instead of being evicted by earlier misses
  std::vector<int> order;
  order.reserve(nt);
  for (int i = 0; i < nt; ++i)
    if (h->cache.slot_of(layer, h->h_touched[i]) >= 0) order.push_back(h->h_touched[i]);
  for (int i = 0; i < nt; ++i)
    if (h->cache.slot_of(layer, h->h_touched[i]) < 0) order.push_back(h->h_touched[i]);
  // within a batch the kernels take the experts in expert order, as a
  // resident forward does (the same sums in the same order)
  for (int b = 0; b < nb; ++b)
    std::sort(order.begin() + (int64_t)b * S, order.begin() + std::min<int64_t>((int64_t)(b + 1) * S, nt));
  if (!dec && tc_shared) CK(launch_prefill_shared_gate_up(p, maps, h->num_sms, s));
  if (!dec && !tc_shared) CK(launch_experts(a, s, kPartSharedGateUp));
  for (int b = 0; b < nb; ++b) {
    const int* batch = order.data() + (int64_t)b * S;
    const int n = std::min(S, nt - b * S);
    const std::vector<SlotCache::Placement> pl = h->cache.place(layer, batch, n);
    // kernels already queued may still read the slots about to be filled
    CK(cudaEventRecord(h->ev_compute, s));
    CK(cudaStreamWaitEvent(h->copy_stream, h->ev_compute, 0));
    for (int i = 0; i < n; ++i) {
      if (!pl[i].miss) continue;
      CK(cudaMemcpyAsync(h->slot_pool + (int64_t)pl[i].slot * L.lay.bytes,
                         L.host_bank + (int64_t)batch[i] * L.lay.bytes, L.lay.bytes, cudaMemcpyHostToDevice,
                         h->copy_stream));
      h->h2d_bytes[layer] += L.lay.bytes;
    }
    CK(cudaEventRecord(h->ev_copied, h->copy_stream));
    CK(cudaStreamWaitEvent(s, h->ev_copied, 0));
    // this batch's tables, staged in pinned memory of their own
    unsigned char* st = h->h_stage + (size_t)b * h->stage_bytes;
    const uint8_t** rec = reinterpret_cast<const uint8_t**>(st);
    int32_t* z = reinterpret_cast<int32_t*>(st + (size_t)E * 8);
    int32_t* list = z + E;
    uint8_t* active = reinterpret_cast<uint8_t*>(list + E + 4);
    for (int e = 0; e < E; ++e) { rec[e] = h->slot_pool; z[e] = 0; active[e] = 0; }
    for (int i = 0; i < n; ++i) {
      rec[batch[i]] = h->slot_pool + (int64_t)pl[i].slot * L.lay.bytes;
      z[batch[i]] = pl[i].slot;
      active[batch[i]] = 1;
      list[i] = batch[i];
    }
    list[E] = n;
    CK(cudaMemcpyAsync(L.rec_dev, rec, (size_t)E * 8, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(L.rec_z_dev, z, (size_t)E * 4, cudaMemcpyHostToDevice, s));
    if (dec) {
      CK(cudaMemcpyAsync(r.touched, list, (size_t)n * 4, cudaMemcpyHostToDevice, s));
      CK(cudaMemcpyAsync(r.n_touched, list + E, 4, cudaMemcpyHostToDevice, s));
      d.skip_shared = b > 0;
      d.out = nb == 1 ? out : (void*)h->off_y;
      d.out_flags = nb == 1 ? out_flags : (b == 0 ? FTMOE_OUT_FP32 : (FTMOE_OUT_FP32 | FTMOE_OUT_ACCUMULATE));
      CK(launch_decode_tc(d, s, 2));
    } else {
      CK(cudaMemcpyAsync(L.active_dev, active, (size_t)E, cudaMemcpyHostToDevice, s));
      p.active = L.active_dev;
      CK(launch_prefill_routed(p, maps, h->num_sms, s));
    }
  }
  if (dec && nb > 1) CK(launch_store_out(h->off_y, out, out_flags, (int64_t)T * c.H, s));
  if (dec && nb == 0) {
    // nothing routed (cannot happen with T >= 1): still the shared expert
    return FTMOE_ERR_DEVICE_CHECK;
  }
  if (!dec) {
    if (tc_shared) {
      CK(launch_prefill_shared_down_combine(p, maps, h->num_sms, s));
    } else {
      a.y_tiles = p.y_bf16 ? 2 : 1;  // the tensor-core down kernel's layout of Y
      CK(launch_experts(a, s, kPartTail));
    }
  }
  int rc = copy_aux(h, r, T, aux, s);
  if (rc) return rc;
  L.last_T = T;
  L.last_I_loc = I_loc;
  return FTMOE_OK;
}

int ftmoe_forward(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags, int i0, int I_loc,
                  const ftmoe_aux* aux, ftmoe_stream_t stream) {
  if (!h || layer < 0 || layer >= h->cfg.num_layers) return FTMOE_ERR_INVALID_ARG;
  const ftmoe_config& c = h->cfg;
  if (T < 0 || T > c.max_tokens) return FTMOE_ERR_INVALID_ARG;
  const int otype = out_flags & 0xff;
  if ((out_flags & ~0x3ff) || otype > FTMOE_OUT_FP32) return FTMOE_ERR_INVALID_ARG;
  if ((out_flags & FTMOE_ACT_BF16) && h->offload) return FTMOE_ERR_INVALID_ARG;
  if ((out_flags & FTMOE_OUT_ACCUMULATE) && otype != FTMOE_OUT_FP32) return FTMOE_ERR_INVALID_ARG;
  Layer& L = h->layers[layer];
  if (!L.loaded) return FTMOE_ERR_NOT_LOADED;
  if (i0 % 16 || I_loc % 16) return FTMOE_ERR_ALIGNMENT;
  if (I_loc <= 0 || i0 < L.li0 || i0 + I_loc > L.li0 + L.lIw) return FTMOE_ERR_SLICE_OUT_OF_RANGE;
  int si0, sI;
  if (!shared_window(c, i0, I_loc, &si0, &sI)) return FTMOE_ERR_ALIGNMENT;
  if (T == 0) return FTMOE_OK;
  if (!x || !out || x == out) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return FTMOE_ERR_ALIGNMENT;
  if (fault("forward")) return FTMOE_ERR_FAULT_INJECTED;
  CK(cudaSetDevice(h->device));
  ProfScope ps(h->prof);
  return forward_impl(h, layer, x, T, out, out_flags, i0, I_loc, aux, (cudaStream_t)stream);
}

int ftmoe_forward_stack(ftmoe_handle* h, const void* x, int T, void* out, ftmoe_stream_t stream) {
  if (!h) return FTMOE_ERR_INVALID_ARG;
  const ftmoe_config& c = h->cfg;
  if (T < 0 || T > c.max_tokens) return FTMOE_ERR_INVALID_ARG;
  for (auto& L : h->layers)
    if (!L.loaded) return FTMOE_ERR_NOT_LOADED;
  if (T == 0) return FTMOE_OK;
  if (!x || !out || x == out) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return FTMOE_ERR_ALIGNMENT;
  CK(cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  ProfScope ps(h->prof);
  const void* cur = x;
  for (int l = 0; l < c.num_layers; ++l) {
    Layer& L = h->layers[l];
    const bool last = l == c.num_layers - 1;
    int rc = forward_impl(h, l, cur, T, last ? out : (void*)h->stack_y, last ? FTMOE_OUT_BF16 : FTMOE_OUT_FP32,
                          L.li0, L.lIw, nullptr, s);
    if (rc) return rc;
    if (!last) {
      uint16_t* nx = h->stack_x[l & 1];
      CK(launch_rms_renorm(h->stack_y, nx, T, c.H, s));
      cur = nx;
    }
  }
  return FTMOE_OK;
}

int ftmoe_rms_renorm(const float* y, void* x, int T, int H, ftmoe_stream_t stream) {
  if (!y || !x || T < 0 || H <= 0 || (const void*)y == x) return FTMOE_ERR_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  CK(launch_rms_renorm(y, (uint16_t*)x, T, H, (cudaStream_t)stream));
  return FTMOE_OK;
}

int ftmoe_forward_experts(ftmoe_handle* h, int layer, const void* x, int T, void* out, int out_flags,
                          const uint8_t* expert_mask, int shared_i0, int shared_I_loc, const ftmoe_aux* aux,
                          ftmoe_stream_t stream) {
  if (!h || layer < 0 || layer >= h->cfg.num_layers || !expert_mask) return FTMOE_ERR_INVALID_ARG;
  const ftmoe_config& c = h->cfg;
  if (h->offload || T < 0 || T > c.max_tokens) return FTMOE_ERR_INVALID_ARG;
  const int otype = out_flags & 0xff;
  if ((out_flags & ~0x1ff) || otype > FTMOE_OUT_FP32) return FTMOE_ERR_INVALID_ARG;
  if ((out_flags & FTMOE_OUT_ACCUMULATE) && otype != FTMOE_OUT_FP32) return FTMOE_ERR_INVALID_ARG;
  Layer& L = h->layers[layer];
  if (!L.loaded) return FTMOE_ERR_NOT_LOADED;
  if (shared_i0 % 16 || shared_I_loc % 16) return FTMOE_ERR_ALIGNMENT;
  if (shared_I_loc < 0 || (shared_I_loc > 0 && (c.I_shared == 0 || shared_i0 < L.sli0 ||
                                                shared_i0 + shared_I_loc > L.sli0 + L.slIw)))
    return FTMOE_ERR_SLICE_OUT_OF_RANGE;
  if (T == 0) return FTMOE_OK;
  if (!x || !out || x == out) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return FTMOE_ERR_ALIGNMENT;
  CK(cudaSetDevice(h->device));
  ProfScope ps(h->prof);
  cudaStream_t s = (cudaStream_t)stream;
  const int E = c.E;
  if (!h->ep_host) {
    if (cudaHostAlloc((void**)&h->ep_host, (size_t)(2 * E + 4) * 4, cudaHostAllocDefault) != cudaSuccess ||
        cudaMalloc(&h->ep_mask, (size_t)E) != cudaSuccess ||
        cudaMalloc(&h->ep_w, (size_t)(c.max_tokens > 0 ? c.max_tokens : 1) * c.top_k * 4) != cudaSuccess) {
      cudaGetLastError();
      return FTMOE_ERR_OOM;
    }
  }
  const int i0 = L.li0, I_loc = L.lIw;
  RouteArgs r = route_args(h, L, x, T);
  ExpertArgs a = expert_args(h, L, r, T, out, out_flags, i0, I_loc);
  // the shared expert on its own window (or not at all)
  const bool with_shared = shared_I_loc > 0;
  if (with_shared) {
    a.s_row0 = shared_i0 - L.sli0;
    a.s_I_loc = shared_I_loc;
  } else {
    a.sh_gate_up = nullptr;
    a.sh_down = nullptr;
  }
  const bool dec = T <= 32;
  bool ok;
  if (dec) {
    ok = h->dtc_enabled && decode_tc_supported(c.H, E, I_loc, L.lIw, a.win.row0, a.s_I_loc, a.s_Iw, a.s_row0, T,
                                               c.top_k, L.lay.gu_sf_bytes != 0);
  } else {
    ok = prefill_path(h, L, T, I_loc, a.win.row0) &&
         (!with_shared || prefill_shared_supported(c.H, a.s_I_loc, a.s_Iw, a.s_row0, c.top_k));
  }
  if (!ok) return FTMOE_ERR_INVALID_ARG;
  DecodeArgs d{};
  PfArgs p{};
  PfMaps maps;
  // routing over every expert, then the touched list on the host
  if (dec) {
    d = decode_args(h, a);
    decode_tc_args(h, L, d);
    CK(launch_decode_tc(d, s, 1));
  } else {
    const bool tc_router = L.router_wcat != nullptr;
    p = prefill_args(h, L, a, x, out, out_flags, with_shared, tc_router);
    CK(prefill_make_maps(p, &maps));
    if (tc_router) {
      CK(launch_route(r, s, kRouteXq));
      CK(launch_prefill_router(p, maps, h->num_sms, s));
      CK(launch_route(r, s, kRouteTopk | kRouteSort));
    } else {
      CK(launch_route(r, s));
    }
  }
  int32_t* ht = h->ep_host;
  CK(cudaMemcpyAsync(ht, r.touched, (size_t)E * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(ht + E, r.n_touched, 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  const int nt = ht[E];
  if (nt < 0 || nt > E) return FTMOE_ERR_DEVICE_CHECK;
  int32_t* list = ht + E + 1;   // [E] the subset's touched experts, in expert order
  int32_t* count = list + E;    // their number
  int n = 0;
  for (int i = 0; i < nt; ++i)
    if (expert_mask[ht[i]]) list[n++] = ht[i];
  *count = n;
  if (dec) {
    // the expert kernels on the subset's list (and the shared window)
    if (n == 0 && !with_shared) {
      CK(cudaMemsetAsync(out, 0, (size_t)T * c.H * (otype == FTMOE_OUT_FP32 ? 4 : 2), s));
    } else {
      CK(cudaMemcpyAsync(r.touched, list, (size_t)(n > 0 ? n : 1) * 4, cudaMemcpyHostToDevice, s));
      CK(cudaMemcpyAsync(r.n_touched, count, 4, cudaMemcpyHostToDevice, s));
      d.skip_shared = with_shared ? 0 : 1;
      CK(launch_decode_tc(d, s, 2));
    }
  } else {
    // the subset's experts only, then the combine of their slots (the other
    // slots' weights zeroed) with the shared window
    CK(cudaMemcpyAsync(h->ep_mask, expert_mask, (size_t)E, cudaMemcpyHostToDevice, s));
    CK(launch_mask_weights(r.topk_idx, r.topk_w, h->ep_mask, h->ep_w, (int64_t)T * c.top_k, s));
    if (with_shared) CK(launch_prefill_shared_gate_up(p, maps, h->num_sms, s));
    p.active = h->ep_mask;
    CK(launch_prefill_routed(p, maps, h->num_sms, s));
    if (with_shared) {
      p.topk_w = h->ep_w;
      CK(launch_prefill_shared_down_combine(p, maps, h->num_sms, s));
    } else {
      a.r.topk_w = h->ep_w;
      a.y_tiles = p.y_bf16 ? 2 : 1;
      CK(launch_experts(a, s, kPartTail));
    }
  }
  int rc = copy_aux(h, r, T, aux, s);
  if (rc) return rc;
  L.last_T = T;
  L.last_I_loc = I_loc;
  return FTMOE_OK;
}

int ftmoe_reduce_partials(const float* parts, int n_parts, int64_t n, void* out, int out_flags,
                          ftmoe_stream_t stream) {
  if (n_parts < 1 || n < 0 || !parts || !out) return FTMOE_ERR_INVALID_ARG;
  const int otype = out_flags & 0xff;
  if ((out_flags & ~0x1ff) || otype > FTMOE_OUT_FP32) return FTMOE_ERR_INVALID_ARG;
  if ((out_flags & FTMOE_OUT_ACCUMULATE) && otype != FTMOE_OUT_FP32) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(parts)) return FTMOE_ERR_ALIGNMENT;
  if (n == 0) return FTMOE_OK;
  CK(launch_reduce_partials(parts, n_parts, n, out, out_flags, (cudaStream_t)stream));
  return FTMOE_OK;
}

int ftmoe_get_stats(ftmoe_handle* h, int layer, ftmoe_stats* out) {
  if (!h || !out || layer < 0 || layer >= h->cfg.num_layers) return FTMOE_ERR_INVALID_ARG;
  CK(cudaSetDevice(h->device));
  CK(cudaDeviceSynchronize());
  memset(out, 0, sizeof *out);
  Layer& L = h->layers[layer];
  int32_t nt = 0;
  CK(cudaMemcpy(&nt, h->r.n_touched, 4, cudaMemcpyDeviceToHost));
  out->touched_experts = L.last_T > 0 ? (h->offload ? L.last_touched : nt) : 0;
  const int H = h->cfg.H, W = L.last_I_loc;
  const int64_t per_expert = (int64_t)2 * W * (H / 2 + H / 16 + 4) + (int64_t)H * (W / 2 + W / 16) + (int64_t)H * 4;
  out->touched_bytes = out->touched_experts * per_expert;
  out->resident_slots = h->offload ? h->cache.slots() : h->cfg.E;
  out->residency = h->offload ? (double)h->cache.slots() / ((double)h->cfg.E * h->cfg.num_layers) : 1.0;
  if (h->offload && h->cache.slots() > 0) {
    out->hits = h->cache.hits(layer);
    out->misses = h->cache.misses(layer);
    out->h2d_bytes = h->h2d_bytes[layer];
  }
  out->device_status = (int32_t)h->last_status;
  unsigned long long nr = 0;
  CK(cudaMemcpy(&nr, h->r.n_rerank, 8, cudaMemcpyDeviceToHost));
  out->reranked_tokens = (int64_t)nr;
  unsigned long long tt = 0;
  CK(cudaMemcpy(&tt, h->r.touched_total, 8, cudaMemcpyDeviceToHost));
  out->touched_total = (int64_t)tt;
  return FTMOE_OK;
}

int ftmoe_check_status(ftmoe_handle* h, ftmoe_stream_t stream) {
  if (!h) return FTMOE_ERR_INVALID_ARG;
  CK(cudaSetDevice(h->device));
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  uint32_t st = 0;
  CK(cudaMemcpy(&st, h->status, 4, cudaMemcpyDeviceToHost));
  CK(cudaMemset(h->status, 0, 4));
  h->last_status = st;
  if (st & kStatusTimeout) {
    // a kernel gave up mid-launch: clear the cross-CTA counters it may have
    // left behind, so the next forward starts from a clean state
    if (h->dtc_counter) CK(cudaMemset(h->dtc_counter, 0, (size_t)(h->cfg.H / 128 + 1) * 4));
    CK(cudaMemset(h->counter, 0, 16));
    CK(cudaDeviceSynchronize());
    return FTMOE_ERR_TIMEOUT;
  }
  if (st & kStatusRange) return FTMOE_ERR_DEVICE_CHECK;
  return FTMOE_OK;
}

int ftmoe_test_withhold_stage(ftmoe_handle* h, int enable, int64_t wait_limit_ns) {
  if (!h || wait_limit_ns < 0) return FTMOE_ERR_INVALID_ARG;
  if (enable && !h->dtc_enabled) return FTMOE_ERR_INVALID_ARG;  // the hook lives in the tensor-core decode kernel
  h->test_withhold = enable ? 1 : 0;
  h->test_wait_ns = (uint64_t)wait_limit_ns;
  return FTMOE_OK;
}

int ftmoe_profile_enable(ftmoe_handle* h, int enable) {
  if (!h) return FTMOE_ERR_INVALID_ARG;
  CK(cudaSetDevice(h->device));
  if (enable && !h->prof) h->prof = new EventProfiler();
  if (!enable && h->prof) {
    CK(cudaDeviceSynchronize());
    delete h->prof;
    h->prof = nullptr;
  }
  return FTMOE_OK;
}

int ftmoe_profile_read(ftmoe_handle* h, ftmoe_kernel_time* out, int max_entries, int* n_out) {
  if (!h || !n_out || max_entries < 0 || (max_entries > 0 && !out)) return FTMOE_ERR_INVALID_ARG;
  *n_out = 0;
  if (!h->prof) return FTMOE_OK;
  CK(cudaSetDevice(h->device));
  EventProfiler& P = *h->prof;
  std::vector<std::string> names;
  std::vector<ftmoe_kernel_time> acc;
  for (auto& r : P.recs) {
    CK(cudaEventSynchronize(r.b));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, r.a, r.b));
    size_t i = 0;
    while (i < names.size() && names[i] != r.name) ++i;
    if (i == names.size()) {
      names.push_back(r.name);
      ftmoe_kernel_time kt{};
      snprintf(kt.name, sizeof kt.name, "%s", r.name.c_str());
      acc.push_back(kt);
    }
    acc[i].launches += 1;
    acc[i].total_ms += ms;
  }
  for (auto& r : P.recs) { P.pool.push_back(r.a); P.pool.push_back(r.b); }
  P.recs.clear();
  const int n = (int)acc.size() < max_entries ? (int)acc.size() : max_entries;
  for (int i = 0; i < n; ++i) out[i] = acc[i];
  *n_out = n;
  return FTMOE_OK;
}

int ftmoe_quantize_weights(const float* w, int64_t rows, int K, uint8_t* codes, uint8_t* scales, float* globals,
                           ftmoe_stream_t stream) {
  if (rows < 0 || K <= 0) return FTMOE_ERR_INVALID_ARG;
  if (K % 16) return FTMOE_ERR_ALIGNMENT;
  if (rows == 0) return FTMOE_OK;
  if (!w || !codes || !scales || !globals) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(w) || ((uintptr_t)codes & 7)) return FTMOE_ERR_ALIGNMENT;
  CK(launch_quantize_weights(w, rows, K, codes, scales, globals, (cudaStream_t)stream));
  return FTMOE_OK;
}

int ftmoe_quantize_activations(const void* a, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                               ftmoe_stream_t stream) {
  if (rows < 0 || K <= 0) return FTMOE_ERR_INVALID_ARG;
  if (K % 16) return FTMOE_ERR_ALIGNMENT;
  if (rows == 0) return FTMOE_OK;
  if (!a || !codes || !scales) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(a) || ((uintptr_t)codes & 7)) return FTMOE_ERR_ALIGNMENT;
  CK(launch_quantize_act_bf16((const uint16_t*)a, rows, K, codes, scales, (cudaStream_t)stream));
  return FTMOE_OK;
}

}  // extern "C"
