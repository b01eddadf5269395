// Temporary: bf16 WANGO on the CUDA-core kernel until the tcgen05 kernel lands.
#include "tg_tc.h"
namespace tg {
cudaError_t launch_wango_tc(const AggArgs& a, cudaStream_t s) { return launch_wango_simt(a, s); }
}  // namespace tg
