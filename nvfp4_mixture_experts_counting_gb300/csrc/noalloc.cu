// Routing without any device allocation: the same router, top-k and
// counting-sort kernels that ftmoe_forward runs, with their scratch in a
// fixed-size array that lives in the library's own device image.
//
// Some callers cannot call cudaMalloc at the time they need routing: a
// serving runtime that has handed all free device memory to its KV cache and
// graph memory pools up front, a host that forbids allocations from plugins,
// or code that runs while a CUDA graph is being captured (an allocation call
// there is an error).  This entry point lets them route tokens with only the
// buffers they already own.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ftmoe.h"
#include "kernels.h"

namespace ftmoe {
cudaError_t route_set_smem_limits(int H, int E);
}  // namespace ftmoe

using namespace ftmoe;

namespace {

// Limits of the static scratch (see ftmoe_route_static in ftmoe.h).
constexpr int64_t kMaxTE = 16384;    // T * E: logits and their error bounds
constexpr int64_t kMaxTH = 262144;   // T * H: quantised activations
constexpr int kMaxT = 1024;
constexpr int kMaxE = 1024;

constexpr int64_t kOffLogits = 0;
constexpr int64_t kOffErr = kOffLogits + kMaxTE * 4;
constexpr int64_t kOffXqCodes = kOffErr + kMaxTE * 4;
constexpr int64_t kOffXqScales = kOffXqCodes + kMaxTH / 2;
constexpr int64_t kOffSigma = kOffXqScales + kMaxTH / 16;
constexpr int64_t kOffTouched = kOffSigma + kMaxT * 4;
constexpr int64_t kOffNTouched = kOffTouched + kMaxE * 4;
constexpr int64_t kOffStatus = kOffNTouched + 256;
constexpr int64_t kScratchBytes = kOffStatus + 256;

// The scratch itself: one copy per device that loads the library, held until
// the process exits.  Host code must not use this name as a device address.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: the device address of the
// scratch array, and the shared-memory limits of the routing kernels.
int scratch_for_current_device(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FTMOE_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) { cudaGetLastError(); return FTMOE_ERR_DEVICE; }
    if (prop.major != 10 || prop.minor != 3) return FTMOE_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FTMOE_ERR_CUDA;
    }
    // largest shared-memory requests the routing kernels may make
    if (route_set_smem_limits(8192, kMaxE) != cudaSuccess) {
      cudaGetLastError();
      return FTMOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return FTMOE_OK;
}

}  // namespace

extern "C" int ftmoe_route_static(const void* x, int T, int H, const float* router_w, const float* router_bias,
                                  int E, int top_k, int norm_topk_prob, int32_t* topk_idx, float* topk_w,
                                  int32_t* offsets, int32_t* perm, int32_t* inv, ftmoe_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || top_k <= 0 || top_k > 32 || top_k > E) return FTMOE_ERR_INVALID_ARG;
  if (H % 16) return FTMOE_ERR_ALIGNMENT;
  if (H > 8192 || E > kMaxE || T > kMaxT || (int64_t)T * E > kMaxTE || (int64_t)T * H > kMaxTH)
    return FTMOE_ERR_TOO_LARGE;
  if (T == 0) return FTMOE_OK;
  if (!x || !router_w || !topk_idx || !topk_w || !offsets || !perm || !inv) return FTMOE_ERR_INVALID_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)router_w & 15)) return FTMOE_ERR_ALIGNMENT;
  unsigned char* s = nullptr;
  int rc = scratch_for_current_device(&s);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  RouteArgs a{};
  a.x = (const uint16_t*)x;
  a.router_w = router_w;
  a.router_bias = router_bias;
  a.sh_gate = nullptr;
  a.T = T;
  a.H = H;
  a.E = E;
  a.top_k = top_k;
  a.norm_topk_prob = norm_topk_prob;
  a.logits = reinterpret_cast<float*>(s + kOffLogits);
  a.err = reinterpret_cast<float*>(s + kOffErr);
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.xq_codes = s + kOffXqCodes;
  a.xq_scales = s + kOffXqScales;
  a.sigma = reinterpret_cast<float*>(s + kOffSigma);
  a.offsets = offsets;
  a.perm = perm;
  a.inv = inv;
  a.touched = reinterpret_cast<int32_t*>(s + kOffTouched);
  a.n_touched = reinterpret_cast<int32_t*>(s + kOffNTouched);
  a.status = reinterpret_cast<uint32_t*>(s + kOffStatus);
  // the status word is OR-ed into by the kernels: start each call from zero
  if (cudaMemsetAsync(a.status, 0, 4, st) != cudaSuccess) { cudaGetLastError(); return FTMOE_ERR_CUDA; }
  if (launch_route(a, st) != cudaSuccess) { cudaGetLastError(); return FTMOE_ERR_CUDA; }
  return FTMOE_OK;
}

extern "C" int ftmoe_route_static_status(ftmoe_stream_t stream) {
  unsigned char* s = nullptr;
  int rc = scratch_for_current_device(&s);
  if (rc) return rc;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) { cudaGetLastError(); return FTMOE_ERR_CUDA; }
  uint32_t st = 0;
  // a plain copy out of the library's own array: no allocation
  if (cudaMemcpy(&st, s + kOffStatus, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(s + kOffStatus, 0, 4) != cudaSuccess) {
    cudaGetLastError();
    return FTMOE_ERR_CUDA;
  }
  if (st & kStatusTimeout) return FTMOE_ERR_TIMEOUT;
  if (st & kStatusRange) return FTMOE_ERR_DEVICE_CHECK;
  return FTMOE_OK;
}
