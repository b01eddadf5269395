// Temporary: bf16 entry points on the CUDA-core kernels until the tcgen05 kernels land.
#include "tg_tc.h"

namespace tg {
cudaError_t launch_proj_tc(const ProjArgs& a, cudaStream_t s) {
  cudaError_t e = launch_gemm_simt(TG_BF16, a.x, a.Wq, a.q, nullptr, a.M, a.dqk, a.d, a.dqk, kEpiStore, s);
  if (e == cudaSuccess) e = launch_gemm_simt(TG_BF16, a.x, a.Wk, a.k, nullptr, a.M, a.dqk, a.d, a.dqk, kEpiStore, s);
  if (e == cudaSuccess) e = launch_qk_prep(TG_BF16, a.q, a.q, a.M, a.T, a.H, a.dqk, a.rope_base, true, s);
  if (e == cudaSuccess) e = launch_qk_prep(TG_BF16, a.k, a.k, a.M, a.T, a.H, a.dqk, a.rope_base, true, s);
  if (e == cudaSuccess) e = launch_gemm_simt(TG_BF16, a.x, a.Wg, a.g, nullptr, a.M, a.m, a.d, a.m, kEpiSilu, s);
  if (e == cudaSuccess) e = launch_gemm_simt(TG_BF16, a.x, a.Wv, a.v, nullptr, a.M, a.m, a.d, a.m, kEpiStore, s);
  return e;
}
cudaError_t launch_out_tc(const void* u, const void* Wo, const void* h, void* h_out, int M, int d, int m,
                          unsigned*, cudaStream_t s) {
  return launch_gemm_simt(TG_BF16, u, Wo, h_out, h, M, d, m, d, kEpiResidual, s);
}
cudaError_t launch_tango_tc(const AggArgs& a, cudaStream_t s) { return launch_tango_simt(a, s); }
cudaError_t launch_wango_tc(const AggArgs& a, cudaStream_t s) { return launch_wango_simt(a, s); }
}  // namespace tg
