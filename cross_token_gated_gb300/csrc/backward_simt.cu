// CUDA-core kernels of the aggregation backward, "TANGO: Token-Aggregated Nonlinear
// Gating Operators ...", sec. 2.1 eq. 5 with the weights of sec. 2.2 eqs. 6-9:
//   bwd_prep_kernel   E = dU * v / den, dv = dU * gbar, D = E . gbar per (row, head)
// All arithmetic is f32; tensors are bf16.
#include "tg_common.cuh"
#include "tg_kernels.h"
#include "tg_ptx.cuh"

namespace tg {
namespace {

using namespace ptx;

constexpr int kPrepThreads = 256;

__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();  // red is reused across calls
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < (int)(blockDim.x / 32); ++w) s += red[w];
  return s;
}

// One CTA per row (b, t).  Rows are m wide in memory, H heads at a pitch of m / H of
// which the first m_h columns are gates.  den and dp have a row pitch of T_pad (dp) and
// den_pitch (den).
__device__ __forceinline__ void prep8(const uint4 du, const uint4 gb, const uint4 vv, float inv, uint4& eo, uint4& dvo,
                                      float& acc) {
  const uint32_t dus[4] = {du.x, du.y, du.z, du.w}, gbs[4] = {gb.x, gb.y, gb.z, gb.w}, vs[4] = {vv.x, vv.y, vv.z, vv.w};
  uint32_t es[4], dvs[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float d0 = bf16lo(dus[k]), d1 = bf16hi(dus[k]);
    const float g0 = bf16lo(gbs[k]), g1 = bf16hi(gbs[k]);
    es[k] = pack_bf16x2(d0 * bf16lo(vs[k]) * inv, d1 * bf16hi(vs[k]) * inv);
    acc = fmaf(bf16lo(es[k]), g0, acc);
    acc = fmaf(bf16hi(es[k]), g1, acc);
    dvs[k] = pack_bf16x2(d0 * g0, d1 * g1);
  }
  eo = make_uint4(es[0], es[1], es[2], es[3]);
  dvo = make_uint4(dvs[0], dvs[1], dvs[2], dvs[3]);
}

__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(
    const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ gbar,
    const float* __restrict__ den, __nv_bfloat16* __restrict__ E, __nv_bfloat16* __restrict__ dv, float* __restrict__ dp,
    int T, int T_pad, int H, int m, int m_h, int den_pitch) {
  __shared__ float red[kPrepThreads / 32];
  const int b = blockIdx.x / T, t = blockIdx.x % T;
  const int m_hp = m / H;
  const size_t off = ((size_t)b * T + t) * m;
  const bool vec = m_h % 8 == 0;
  for (int a = 0; a < H; ++a) {
    const float inv = 1.f / den[(size_t)(b * H + a) * den_pitch + t];
    float acc = 0.f;
    const size_t h0 = off + (size_t)a * m_hp;
    if (vec) {
      for (int c = threadIdx.x; c < m_h / 8; c += blockDim.x) {
        const size_t o = h0 + 8 * (size_t)c;
        const uint4 vv = v ? *reinterpret_cast<const uint4*>(v + o)
                           : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);  // 1.0
        uint4 eo, dvo;
        prep8(*reinterpret_cast<const uint4*>(dout + o), *reinterpret_cast<const uint4*>(gbar + o), vv, inv, eo, dvo,
              acc);
        *reinterpret_cast<uint4*>(E + o) = eo;
        if (dv) *reinterpret_cast<uint4*>(dv + o) = dvo;
      }
    } else {  // a head width that is not a multiple of 8: one column at a time
      for (int c = threadIdx.x; c < m_h; c += blockDim.x) {
        const size_t o = h0 + c;
        const float d = __bfloat162float(dout[o]), gb = __bfloat162float(gbar[o]);
        const __nv_bfloat16 e = __float2bfloat16_rn(d * (v ? __bfloat162float(v[o]) : 1.f) * inv);
        acc = fmaf(__bfloat162float(e), gb, acc);
        E[o] = e;
        if (dv) dv[o] = __float2bfloat16_rn(d * gb);
      }
    }
    const float tot = block_sum(acc, red);
    if (threadIdx.x == 0) dp[(size_t)(b * H + a) * T_pad + t] = tot;
  }
}

}  // namespace

cudaError_t launch_bwd_prep(const void* dout, const void* v, const void* gbar, const float* den, int den_pitch,
                            void* E, void* dv, float* dp, int B, int T, int T_pad, int H, int m, int m_h,
                            cudaStream_t s) {
  const long long n = (long long)B * T;
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd_prep_kernel<<<(unsigned)n, kPrepThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(v),
      static_cast<const __nv_bfloat16*>(gbar), den, static_cast<__nv_bfloat16*>(E), static_cast<__nv_bfloat16*>(dv),
      dp, T, T_pad, H, m, m_h, den_pitch);
  return cudaGetLastError();
}

}  // namespace tg
