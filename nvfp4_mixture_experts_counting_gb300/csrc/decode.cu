// Decode path (1 <= T <= 32): the three kernels chained with programmatic
// dependent launch, and the test of whether a forward's shapes fit it.
//   k_dec_route    (decode_route.cu)    routing, shared gate_up, x quantisation
//   k_dec_gate_up  (decode_gate_up.cu)  routed gate_up + SwiGLU + quantisation
//   k_dec_down     (decode_down.cu)     routed down + shared down + combine
#include "decode_common.cuh"

namespace ftmoe {

// Row pitches of the decoded intermediates (half per element, fp32 per block).
int decode_hq_cpitch(int I_loc) { return align16(I_loc * 2); }
int decode_hq_spitch(int I_loc) { return align16((I_loc / kBlock) * 4); }

static cudaError_t launch_pdl(void (*kern)(DecodeArgs), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              bool pdl, const DecodeArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t decode_set_smem_limits() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_dec_route, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemMax)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_dec_gate_up, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemMax)) !=
      cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_dec_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemMax);
}

bool decode_supported(int H, int E, int I_loc, int Iw, int row0, int s_I_loc, int s_Iw, int s_row0, int T,
                      int top_k) {
  (void)s_Iw;
  (void)s_row0;
  if (T < 1 || T > kDecMaxT || E > 1024 || top_k > 32) return false;
  // 16-blocks per row a multiple of 16: the activation scale rows copy in
  // 16-byte multiples and 16 lanes split every row evenly
  if (H % 256) return false;
  if (I_loc % kBlock || s_I_loc % kBlock) return false;
  const int P = T * top_k;
  if (rt_smem_layout(T, E, top_k).total > kDecSmemMax) return false;
  const GuSmem g = gu_smem_layout(H, T, E, P);
  if (g.nst < 2 || g.total > kDecSmemMax) return false;
  const DnSmem d = dn_smem_choose(Iw, row0, I_loc, s_I_loc, T, E, P);
  if (d.nst < 2 || d.total > kDecSmemMax) return false;
  return true;
}

cudaError_t launch_decode(DecodeArgs a, cudaStream_t s) {
  cudaError_t err;
  const int T = a.T, E = a.r.E, P = T * a.top_k;
  a.n_router_ctas = (E + 1) / 2;
  a.n_shared_ctas = a.sh_gate_up ? (a.s_I_loc + 1) / 2 : 0;
  {
    const RtSmem L = rt_smem_layout(T, E, a.top_k);
    FTMOE_PROF_BEGIN("k_dec_route", s);
    err = launch_pdl(k_dec_route, dim3(a.n_router_ctas + a.n_shared_ctas + 1), dim3(kRtThreads), L.total, s,
                     false, a);
    FTMOE_PROF_END(s);
    if (err != cudaSuccess) return err;
  }
  {
    const GuSmem L = gu_smem_layout(a.H, T, E, P);
    FTMOE_PROF_BEGIN("k_dec_gate_up", s);
    err = launch_pdl(k_dec_gate_up, dim3(a.num_sms), dim3(kGuThreads + 32), L.total, s, a.pdl, a);
    FTMOE_PROF_END(s);
    if (err != cudaSuccess) return err;
  }
  {
    const DnSmem L = dn_smem_choose(a.win.Iw, a.win.row0, a.win.I_loc, a.s_I_loc, T, E, P);
    FTMOE_PROF_BEGIN("k_dec_down", s);
    err = launch_pdl(k_dec_down, dim3(a.H / kDnRows), dim3(kDnThreads + 32), L.total, s, a.pdl, a);
    FTMOE_PROF_END(s);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace ftmoe
