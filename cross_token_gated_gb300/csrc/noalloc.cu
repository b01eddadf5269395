// tango_aggregate_noalloc: the full-prefix aggregation for callers that cannot
// allocate device memory themselves.
//
// Some callers have no allocator to hand: a host runtime that forbids cudaMalloc
// after start-up, code that runs inside a pre-sized memory pool it does not own, or
// a driver that must not fail on out-of-memory in the middle of its work.  For them
// this entry point needs no workspace argument.  Its scratch (the unit-normalised
// copies of q and k) lives in one fixed array in device memory that the library
// declares at file scope; every GPU that loads the library holds that array until
// the process exits.
//
// The entry point itself allocates nothing: it calls no cudaMalloc, cudaFree or
// allocating library routine, and it hands the array's device address to the
// regular tango_aggregate as its workspace, so the kernels and the results are the
// ones of tango_aggregate.
#include <cuda_runtime.h>

#include <mutex>

#include "tango.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TG_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" tg_status tango_aggregate_noalloc(const tg_agg_params* p, const void* q, const void* k,
                                             const void* g, const void* v, void* out, tg_stream_t stream) {
  if (!p) return TG_ERR_INVALID_ARG;
  // 0 for invalid parameters (tango_aggregate then returns the precise error) and
  // for pre-normalised q/k, which need no scratch.
  const size_t need = tg_workspace_size(TG_WS_TANGO, p);
  if (need > TG_NOALLOC_SCRATCH_BYTES) return TG_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0 && scratch_address(&ws) != cudaSuccess) return TG_ERR_CUDA;
  return tango_aggregate(p, q, k, g, v, out, ws, need > 0 ? (size_t)TG_NOALLOC_SCRATCH_BYTES : 0, stream);
}
