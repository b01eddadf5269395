// CUDA-core kernels of the aggregation backward, "TANGO: Token-Aggregated Nonlinear
// Gating Operators ...", sec. 2.1 eq. 5 with the weights of sec. 2.2 eqs. 6-9:
//   bwd_prep_kernel   E = dU * v / den, dv = dU * gbar, D = E . gbar per (row, head)
//   reverse_rows_kernel  a sequence's rows in reverse order (the WANGO gate gradient is
//                     the forward numerator of the time-reversed problem)
//   bwd_qk_kernel     dqhat = sum_j X_ij khat_j and dkhat = sum_i X_ij qhat_i over the
//                     window pairs; over the older pairs (WANGO) the feature-map
//                     gradients sum_j X_ij phi(k~_j) and sum_i X_ij e^-tau phi(q~_i),
//                     taken through phi' and sqrt(tau); then through the unit
//                     normalisation q^ = q / max(|q|, 1e-12) of sec. 2.1
// All arithmetic is f32; tensors are bf16.
#include <math.h>

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

// One CTA per row (b, t) of `rows` per sequence (T, or T_pad with a reversed copy, whose
// rows t >= T only clear their slot of it).  den and dp have a row pitch of T_pad.
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(
    const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ gbar,
    const float* __restrict__ den, __nv_bfloat16* __restrict__ E, __nv_bfloat16* __restrict__ dv, float* __restrict__ dp,
    __nv_bfloat16* __restrict__ e_rev, int T, int T_pad, int rows, int H, int m) {
  __shared__ float red[kPrepThreads / 32];
  const int b = blockIdx.x / rows, t = blockIdx.x % rows;
  const int nvec = m / 8, m_h = m / H;
  uint4* rev_row = e_rev ? reinterpret_cast<uint4*>(e_rev + ((size_t)b * T_pad + (T_pad - 1 - t)) * m) : nullptr;
  if (t >= T) {
    for (int c = threadIdx.x; c < nvec; c += blockDim.x) rev_row[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  const size_t off = ((size_t)b * T + t) * m;
  const uint4* du4 = reinterpret_cast<const uint4*>(dout + off);
  const uint4* v4 = v ? reinterpret_cast<const uint4*>(v + off) : nullptr;
  const uint4* gb4 = reinterpret_cast<const uint4*>(gbar + off);
  uint4* e4 = reinterpret_cast<uint4*>(E + off);
  uint4* dv4 = dv ? reinterpret_cast<uint4*>(dv + off) : nullptr;
  for (int a = 0; a < H; ++a) {
    const float inv = 1.f / den[(size_t)(b * H + a) * T_pad + t];
    float acc = 0.f;
    const int c0 = a * (m_h / 8), c1 = (a + 1) * (m_h / 8);
    for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
      const uint4 du = du4[c];
      const uint4 gb = gb4[c];
      const uint4 vv = v4 ? v4[c] : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);  // 1.0
      const uint32_t dus[4] = {du.x, du.y, du.z, du.w}, gbs[4] = {gb.x, gb.y, gb.z, gb.w},
                     vs[4] = {vv.x, vv.y, vv.z, vv.w};
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
      const uint4 eo = make_uint4(es[0], es[1], es[2], es[3]);
      e4[c] = eo;
      if (rev_row) rev_row[c] = eo;
      if (dv4) dv4[c] = make_uint4(dvs[0], dvs[1], dvs[2], dvs[3]);
    }
    const float tot = block_sum(acc, red);
    if (threadIdx.x == 0) dp[(size_t)(b * H + a) * T_pad + t] = tot;
  }
}

// One CTA per destination row; 16-byte vectors (width % 8 == 0).
__global__ void reverse_rows_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int T,
                                    int T_pad, int width, int to_padded) {
  const int rows_dst = to_padded ? T_pad : T;
  const int b = blockIdx.x / rows_dst, t = blockIdx.x % rows_dst;
  const int nvec = width / 8;
  uint4* d = reinterpret_cast<uint4*>(dst + ((size_t)b * rows_dst + t) * width);
  int ts;  // source row, or -1 for a zero row
  if (to_padded) ts = (t >= T_pad - T) ? T_pad - 1 - t : -1;
  else ts = T_pad - 1 - t;
  const int rows_src = to_padded ? T : T_pad;
  const uint4* s = ts >= 0 ? reinterpret_cast<const uint4*>(src + ((size_t)b * rows_src + ts) * width) : nullptr;
  for (int c = threadIdx.x; c < nvec; c += blockDim.x) d[c] = s ? s[c] : make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------- dq / dk
constexpr int kQKThreads = 256;
constexpr int kRB = 64;  // own rows per CTA, partner rows per step

// phi (eq. 8 with mode 0, plain ELU + 1 with mode 1) and its derivative
__device__ __forceinline__ float phi_f(float u, int mode, float inv_sqrt_dh) {
  const float e = u > 0.f ? u + 1.f : expf(u);
  return mode == 0 ? fmaxf(e + 1e-4f, 1e-4f) * inv_sqrt_dh : e;
}
__device__ __forceinline__ float dphi_f(float u, int mode, float inv_sqrt_dh) {
  const float d = u > 0.f ? 1.f : expf(u);
  return mode == 0 ? d * inv_sqrt_dh : d;
}

template <int DH>
__global__ void __launch_bounds__(kQKThreads) bwd_qk_kernel(BwdQKArgs a) {
  extern __shared__ float sm[];
  float* xs = sm;                    // [kRB][kRB + 1]: X of (own, partner)
  float* pv = xs + kRB * (kRB + 1);  // [kRB][DH] partner unit vectors
  float* fv = pv + kRB * DH;         // [kRB][DH] partner feature maps (WANGO)
  constexpr int DG = DH / 4;         // 4-dim groups
  constexpr int R = DH / 16;         // own rows per thread (64 rows / (256 / DG) groups)
  const int side = blockIdx.z;       // 0: dq (own = destinations), 1: dk (own = sources)
  const int bh = blockIdx.y, b = bh / a.H, head = bh % a.H;
  const int own0 = blockIdx.x * kRB;
  const int tid = threadIdx.x, dg = tid % DG, rg = tid / DG;
  const float tau = head_tau(a.tau, a.s, head, a.err, kKernBackward);
  const float st = sqrtf(tau), inv_sqrt_dh = rsqrtf((float)DH), etau = expf(-tau);
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.X) + (size_t)bh * a.T_pad * a.T_pad;
  const __nv_bfloat16* partner = static_cast<const __nv_bfloat16*>(side == 0 ? a.khat : a.qhat);
  const int nblk = (a.T + kRB - 1) / kRB;
  const int p_lo = side == 0 ? 0 : blockIdx.x, p_hi = side == 0 ? blockIdx.x : nblk - 1;

  float accA[R][4], accB[R][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int d = 0; d < 4; ++d) accA[r][d] = accB[r][d] = 0.f;

  for (int pb = p_lo; pb <= p_hi; ++pb) {
    const int p0 = pb * kRB;
    __syncthreads();
    // X tile: rows of destinations, columns of sources; stored as xs[own][partner]
    for (int e = tid; e < kRB * kRB / 8; e += blockDim.x) {
      const int rr = e / (kRB / 8), c8 = (e % (kRB / 8)) * 8;
      const int i = side == 0 ? own0 + rr : p0 + rr;   // destination row of X
      const int j0 = side == 0 ? p0 + c8 : own0 + c8;  // first source column
      uint4 x = make_uint4(0, 0, 0, 0);
      if (i < a.T) x = *reinterpret_cast<const uint4*>(X + (size_t)i * a.T_pad + j0);
      const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float f = (k & 1) ? bf16hi(xv[k / 2]) : bf16lo(xv[k / 2]);
        if (side == 0) xs[rr * (kRB + 1) + c8 + k] = f;
        else xs[(c8 + k) * (kRB + 1) + rr] = f;
      }
    }
    // partner unit vectors (and their feature maps)
    for (int e = tid; e < kRB * DH; e += blockDim.x) {
      const int rr = e / DH, c = e % DH, t = p0 + rr;
      const float u = t < a.T ? __bfloat162float(partner[((size_t)b * a.T + t) * a.dqk + head * DH + c]) : 0.f;
      pv[e] = u;
      if (a.wango) {
        const float f = phi_f(st * u, a.phi_mode, inv_sqrt_dh);
        fv[e] = t < a.T ? (side == 0 ? f : etau * f) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int p = 0; p < kRB; ++p) {
      const float4 pvv = *reinterpret_cast<const float4*>(pv + p * DH + 4 * dg);
      if (!a.wango) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float x = xs[(rg * R + r) * (kRB + 1) + p];
          accA[r][0] = fmaf(x, pvv.x, accA[r][0]);
          accA[r][1] = fmaf(x, pvv.y, accA[r][1]);
          accA[r][2] = fmaf(x, pvv.z, accA[r][2]);
          accA[r][3] = fmaf(x, pvv.w, accA[r][3]);
        }
      } else {
        const float4 fvv = *reinterpret_cast<const float4*>(fv + p * DH + 4 * dg);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float x = xs[(rg * R + r) * (kRB + 1) + p];
          const int own = own0 + rg * R + r, par = p0 + p;
          const int dist = side == 0 ? own - par : par - own;  // i - j
          const float xw = dist < a.window ? x : 0.f, xo = x - xw;
          accA[r][0] = fmaf(xw, pvv.x, accA[r][0]);
          accA[r][1] = fmaf(xw, pvv.y, accA[r][1]);
          accA[r][2] = fmaf(xw, pvv.z, accA[r][2]);
          accA[r][3] = fmaf(xw, pvv.w, accA[r][3]);
          accB[r][0] = fmaf(xo, fvv.x, accB[r][0]);
          accB[r][1] = fmaf(xo, fvv.y, accB[r][1]);
          accB[r][2] = fmaf(xo, fvv.z, accB[r][2]);
          accB[r][3] = fmaf(xo, fvv.w, accB[r][3]);
        }
      }
    }
  }
  // gather the own rows' sums: sA [kRB][DH], sB [kRB][DH]
  __syncthreads();
  float* sA = sm;
  float* sB = sm + kRB * DH;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      sA[(rg * R + r) * DH + 4 * dg + d] = accA[r][d];
      sB[(rg * R + r) * DH + 4 * dg + d] = accB[r][d];
    }
  __syncthreads();
  // per own row (four threads, DH / 4 dims each): feature-map chain rule, then the
  // unit normalisation
  const int row = tid / 4, part = tid % 4;
  const int t = own0 + row;
  const bool ok = t < a.T;
  const __nv_bfloat16* unit = static_cast<const __nv_bfloat16*>(side == 0 ? a.qhat : a.khat);
  const __nv_bfloat16* raw = static_cast<const __nv_bfloat16*>(side == 0 ? a.raw_q : a.raw_k);
  const size_t roff = ((size_t)b * a.T + (ok ? t : 0)) * a.dqk + head * DH;
  constexpr int PD = DH / 4;
  float u[PD], dh[PD];
  float n2 = 0.f;
#pragma unroll
  for (int c = 0; c < PD; ++c) {
    const int col = part * PD + c;
    u[c] = ok ? __bfloat162float((raw ? raw : unit)[roff + col]) : 0.f;
    n2 = fmaf(u[c], u[c], n2);
  }
  n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
  n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
  const float nrm = sqrtf(n2);
  const float inv_n = 1.f / fmaxf(nrm, 1e-12f);
  float pr = 0.f;
#pragma unroll
  for (int c = 0; c < PD; ++c) {
    const int col = part * PD + c;
    const float uh = raw ? u[c] * inv_n : u[c];  // the unit vector
    float g = sA[row * DH + col];
    if (a.wango) {
      const float fac = side == 0 ? st * etau : st;
      g = fmaf(fac * dphi_f(st * uh, a.phi_mode, inv_sqrt_dh), sB[row * DH + col], g);
    }
    dh[c] = g;
    u[c] = uh;
    pr = fmaf(uh, g, pr);
  }
  pr += __shfl_xor_sync(0xffffffffu, pr, 1);
  pr += __shfl_xor_sync(0xffffffffu, pr, 2);
  if (!ok) return;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(side == 0 ? a.dq : a.dk) + roff;
#pragma unroll
  for (int c = 0; c < PD; ++c) {
    float y = dh[c];
    if (raw) y = nrm < 1e-12f ? y * 1e12f : (y - u[c] * pr) * inv_n;
    out[part * PD + c] = __float2bfloat16_rn(y);
  }
}

template <int DH>
cudaError_t launch_qk_dh(const BwdQKArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (kRB * (kRB + 1) + 2 * kRB * DH);
  cudaError_t e = cudaFuncSetAttribute(bwd_qk_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.T + kRB - 1) / kRB, a.B * a.H, 2);
  bwd_qk_kernel<DH><<<grid, kQKThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prep(const void* dout, const void* v, const void* gbar, const float* den, void* E, void* dv,
                            float* dp, void* e_rev, int B, int T, int T_pad, int H, int m, cudaStream_t s) {
  const int rows = e_rev ? T_pad : T;
  const long long n = (long long)B * rows;
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd_prep_kernel<<<(unsigned)n, kPrepThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(v),
      static_cast<const __nv_bfloat16*>(gbar), den, static_cast<__nv_bfloat16*>(E), static_cast<__nv_bfloat16*>(dv),
      dp, static_cast<__nv_bfloat16*>(e_rev), T, T_pad, rows, H, m);
  return cudaGetLastError();
}

cudaError_t launch_reverse_rows(const void* src, void* dst, int B, int T, int T_pad, int width, bool to_padded,
                                cudaStream_t s) {
  const long long rows = (long long)B * (to_padded ? T_pad : T);
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  reverse_rows_kernel<<<(unsigned)rows, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src),
                                                     static_cast<__nv_bfloat16*>(dst), T, T_pad, width,
                                                     to_padded ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_bwd_qk(const BwdQKArgs& a, cudaStream_t s) {
  const int d_h = a.dqk / a.H;
  if (d_h == 64) return launch_qk_dh<64>(a, s);
  if (d_h == 32) return launch_qk_dh<32>(a, s);
  if (d_h == 16) return launch_qk_dh<16>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace tg
