// Temporary: bf16 aggregation on the CUDA-core kernels until the tcgen05 kernels land.
#include "tg_tc.h"
namespace tg {
cudaError_t launch_tango_tc(const AggArgs& a, cudaStream_t s) { return launch_tango_simt(a, s); }
cudaError_t launch_wango_tc(const AggArgs& a, cudaStream_t s) { return launch_wango_simt(a, s); }
}  // namespace tg
