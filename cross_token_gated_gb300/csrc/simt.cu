// CUDA-core kernels: the full-fp32 aggregation path (no TF32) and the row
// kernels shared by both precisions (RoPE + unit normalisation, RMSNorm).
//
// Definitions follow "TANGO: Token-Aggregated Nonlinear Gating Operators for
// Natural and Formal Language Modeling": eq. 2 (SwiGLU gate, features), sec. 2.1
// (RoPE then unit-normalised q/k), eq. 4 (logit), eq. 5 (null gate), eq. 6 (TANGO
// weights), eqs. 7-10 (WANGO window, feature map, running sums), eq. 3 (residual).
//
// Every weight is evaluated with a static shift: exp(tau (cos - 1)) instead of
// exp(tau cos), and the feature-map and null weights are multiplied by the same
// e^-tau.  Eq. 5 is a ratio, so the shift cancels exactly; with |cos| <= 1 and
// tau <= 20 every shifted weight lies in [e^-40, 1] and no running maximum is needed.
#include <math.h>

#include "tg_common.cuh"
#include "tg_kernels.h"

namespace tg {
namespace {


// ---------------------------------------------------------------- row kernels

template <typename T>
__global__ void qk_prep_kernel(const T* in, T* out, long long rows, int T_len, int H, int dqk, float rope_base,
                               int normalize) {
  long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * H) return;
  const long long r = idx / H;
  const int a = (int)(idx % H);
  const int d_h = dqk / H;
  const T* src = in + r * dqk + (long long)a * d_h;
  T* dst = out + r * dqk + (long long)a * d_h;
  float x[128];
  for (int c = 0; c < d_h; ++c) x[c] = io<T>::ld(src + c);
  if (rope_base > 0.f) {
    // Rotate-half pairing (c, c + d_h/2); angle t * base^(-2c/d_h) in double so
    // that long positions keep full fp32 accuracy.
    const int half = d_h / 2;
    const double t = (double)(r % T_len);
    for (int c = 0; c < half; ++c) {
      double th = t * pow((double)rope_base, -2.0 * c / (double)d_h);
      double sn, cs;
      sincos(th, &sn, &cs);
      float x1 = x[c], x2 = x[c + half];
      x[c] = (float)(x1 * cs - x2 * sn);
      x[c + half] = (float)(x1 * sn + x2 * cs);
    }
  }
  if (normalize) {
    float ss = 0.f;
    for (int c = 0; c < d_h; ++c) ss = fmaf(x[c], x[c], ss);
    float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
    for (int c = 0; c < d_h; ++c) x[c] *= inv;
  }
  for (int c = 0; c < d_h; ++c) io<T>::st(dst + c, x[c]);
}

template <typename T>
__global__ void rmsnorm_kernel(const T* h, const T* gamma, T* x, long long rows, int d, float eps) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const T* hr = h + r * d;
  float ss = 0.f;
  for (int c = lane; c < d; c += 32) {
    float t = io<T>::ld(hr + c);
    ss = fmaf(t, t, ss);
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)d + eps);
  for (int c = lane; c < d; c += 32) io<T>::st(x + r * d + c, io<T>::ld(hr + c) * inv * io<T>::ld(gamma + c));
}

// ---------------------------------------------------------------------- GEMM

// 64x64 output tile, 256 threads, 4x4 outputs per thread, K in steps of 16.
template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ A, const T* __restrict__ B,
                                                        T* C, const T* R, int M, int N, int K, int ldc,
                                                        int epi) {
  __shared__ float As[16][65];
  __shared__ float Bs[16][65];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tr = (tid / 16) * 4, tc = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int e = tid; e < 64 * 16; e += 256) {
      const int rr = e / 16, kk = e % 16;
      const int gm = m0 + rr, gn = n0 + rr, gk = k0 + kk;
      As[kk][rr] = (gm < M && gk < K) ? io<T>::ld(A + (long long)gm * K + gk) : 0.f;
      Bs[kk][rr] = (gn < N && gk < K) ? io<T>::ld(B + (long long)gn * K + gk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = As[kk][tr + u];
        b[u] = Bs[kk][tc + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(a[u], b[w], acc[u][w]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int gm = m0 + tr + u;
    if (gm >= M) continue;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int gn = n0 + tc + w;
      if (gn >= N) continue;
      float y = acc[u][w];
      const long long off = (long long)gm * ldc + gn;
      if (epi == kEpiSilu) y = y / (1.f + expf(-y));
      else if (epi == kEpiResidual) y += io<T>::ld(R + off);
      io<T>::st(C + off, y);
    }
  }
}

// ---------------------------------------------------------------- aggregation

constexpr int kRows = 32;  // destinations per tile
constexpr int kSrc = 32;   // sources per inner step
constexpr int kCols = 64;  // gate columns per tile
constexpr int kThreads = 256;

// Feature map of eq. 8 (mode 0) or plain ELU + 1 (mode 1), fp32.
__device__ __forceinline__ float phi_f32(float u, float inv_sqrt_dh, int mode) {
  const float elu = u > 0.f ? u : expm1f(u);
  if (mode == 1) return elu + 1.f;
  return fmaxf(elu + 1.f + 1e-4f, 1e-4f) * inv_sqrt_dh;
}

// Thread layout inside a tile: row r = tid / 8 owns 8 gate columns starting at
// (tid % 8) * 8 and 4 source columns starting at (tid % 8) * 4 of each score block.
struct TileThread {
  int r, c0, j0;
  __device__ TileThread() : r(threadIdx.x / 8), c0((threadIdx.x % 8) * 8), j0((threadIdx.x % 8) * 4) {}
};

__device__ __forceinline__ float row_group_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  return x;
}

template <typename T>
__device__ void load_rows(float* dst, const T* src, long long row0, int nrows_valid, int width, int ld,
                          int col0, int ncols_valid) {
  // dst[r * width + c] = src[(row0 + r) * ld + col0 + c] (zero outside the valid box)
  for (int e = threadIdx.x; e < kSrc * width; e += kThreads) {
    const int r = e / width, c = e % width;
    dst[e] = (r < nrows_valid && c < ncols_valid) ? io<T>::ld(src + (row0 + r) * ld + col0 + c) : 0.f;
  }
}

template <typename T>
__device__ void finish_rows(const AggArgs& p, const TileThread& tt, const float* acc, float den, int b, int i,
                            int a, int n0, int m_h, float tau) {
  if (i >= p.T) return;
  if (p.null_bias) den += (float)(i + 1) * expf(p.null_bias[a] - tau);
  const float inv = 1.f / den;
  const long long rowoff = ((long long)b * p.T + i) * p.m + (long long)a * (p.m / p.H) + n0;
  const T* v = static_cast<const T*>(p.v);
  T* out = static_cast<T*>(p.out);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int n = tt.c0 + c;
    if (n0 + n >= m_h) break;
    float y = acc[c] * inv;
    if (v) y *= io<T>::ld(v + rowoff + n);
    io<T>::st(out + rowoff + n, y);
  }
}

// TANGO: grid (H * ceil(m_h / 64), ceil(T / 32), B).
template <typename T>
__global__ void __launch_bounds__(kThreads) tango_simt_kernel(AggArgs p) {
  extern __shared__ float sm[];
  const int d_h = p.dqk / p.H, m_hp = p.m / p.H, m_h = p.m_h ? p.m_h : m_hp;
  const int ntile = (m_h + kCols - 1) / kCols;
  const int a = blockIdx.x / ntile, n0 = (blockIdx.x % ntile) * kCols;
  const int i0 = blockIdx.y * kRows, b = blockIdx.z;
  float* Qs = sm;                   // [32][d_h]
  float* Ks = Qs + kRows * d_h;     // [32][d_h]
  float* Gs = Ks + kSrc * d_h;      // [32][64]
  float* Ps = Gs + kSrc * kCols;    // [32][33]
  const float tau = head_tau(p.tau, p.s, a, p.err, kKernTango);
  const float c = tau * kLog2e;
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* g = static_cast<const T*>(p.g);
  const long long seq = (long long)b * p.T;
  const int rows_valid = min(kRows, p.T - i0);
  load_rows<T>(Qs, q, seq + i0, rows_valid, d_h, p.dqk, a * d_h, d_h);
  TileThread tt;
  const int i = i0 + tt.r;
  float acc[8] = {};
  float den = 0.f;
  const int i_last = min(i0 + kRows, p.T) - 1;
  for (int j0 = 0; j0 <= i_last; j0 += kSrc) {
    __syncthreads();
    const int src_valid = min(kSrc, p.T - j0);
    load_rows<T>(Ks, k, seq + j0, src_valid, d_h, p.dqk, a * d_h, d_h);
    load_rows<T>(Gs, g, seq + j0, src_valid, kCols, p.m, a * m_hp + n0, m_h - n0);
    __syncthreads();
    float part = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jj = tt.j0 + u, j = j0 + jj;
      float w = 0.f;
      if (j <= i && i < p.T) {
        float s = 0.f;
        for (int e = 0; e < d_h; ++e) s = fmaf(Qs[tt.r * d_h + e], Ks[jj * d_h + e], s);
        w = exp2f(c * (s - 1.f));  // eq. 6, shifted by e^-tau
      }
      Ps[tt.r * 33 + jj] = w;
      part += w;
    }
    den += row_group_sum(part);
    __syncthreads();
    for (int jj = 0; jj < kSrc; ++jj) {
      const float w = Ps[tt.r * 33 + jj];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, Gs[jj * kCols + tt.c0 + e], acc[e]);
    }
  }
  finish_rows<T>(p, tt, acc, den, b, i, a, n0, m_h, tau);
}

// WANGO: grid (H * ceil(m_h / 64), 1, B).  One block walks the sequence in
// tiles of 32 destinations.  The running sums S (d_h x 64) and z (d_h) hold every
// source j < state_lo, where state_lo = max(0, i0 - W + 1) for the tile at i0;
// those sources are older than the window for every destination of the tile.
// Sources in [state_lo, i0 + 31] are weighted pair by pair: exp for the window,
// the feature-map product for the older ones.
template <typename T>
__global__ void __launch_bounds__(kThreads) wango_simt_kernel(AggArgs p) {
  extern __shared__ float sm[];
  const int d_h = p.dqk / p.H, m_hp = p.m / p.H, m_h = p.m_h ? p.m_h : m_hp;
  const int ntile = (m_h + kCols - 1) / kCols;
  const int a = blockIdx.x / ntile, n0 = (blockIdx.x % ntile) * kCols;
  const int b = blockIdx.z;
  float* S = sm;                      // [d_h][64]
  float* z = S + d_h * kCols;         // [d_h]
  float* Qs = z + d_h;                // [32][d_h]
  float* FQ = Qs + kRows * d_h;       // [32][d_h]
  float* Ks = FQ + kRows * d_h;       // [32][d_h]
  float* FK = Ks + kSrc * d_h;        // [32][d_h]
  float* Gs = FK + kSrc * d_h;        // [32][64]
  float* Ps = Gs + kSrc * kCols;      // [32][33]
  const float tau = head_tau(p.tau, p.s, a, p.err, kKernWango);
  const float c = tau * kLog2e;
  const float sq = sqrtf(tau), inv_sqrt_dh = rsqrtf((float)d_h), shift = expf(-tau);
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* g = static_cast<const T*>(p.g);
  const long long seq = (long long)b * p.T;
  const int W = p.window;
  for (int e = threadIdx.x; e < d_h * kCols + d_h; e += kThreads) S[e] = 0.f;  // also clears z
  TileThread tt;
  int state_lo = 0;
  for (int i0 = 0; i0 < p.T; i0 += kRows) {
    __syncthreads();
    const int rows_valid = min(kRows, p.T - i0);
    load_rows<T>(Qs, q, seq + i0, rows_valid, d_h, p.dqk, a * d_h, d_h);
    __syncthreads();
    for (int e = threadIdx.x; e < kRows * d_h; e += kThreads) FQ[e] = phi_f32(sq * Qs[e], inv_sqrt_dh, p.phi_mode);
    __syncthreads();
    const int i = i0 + tt.r;
    // Older prefix through the running sums (eq. 10), scaled by the shift.
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float den = 0.f;
    for (int cc = 0; cc < d_h; ++cc) {
      const float f = FQ[tt.r * d_h + cc];
      den = fmaf(f, z[cc], den);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(f, S[cc * kCols + tt.c0 + e], acc[e]);
    }
    den *= shift;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= shift;
    const int i_last = i0 + rows_valid - 1;
    for (int j0 = state_lo; j0 <= i_last; j0 += kSrc) {
      __syncthreads();
      const int src_valid = min(kSrc, p.T - j0);
      load_rows<T>(Ks, k, seq + j0, src_valid, d_h, p.dqk, a * d_h, d_h);
      load_rows<T>(Gs, g, seq + j0, src_valid, kCols, p.m, a * m_hp + n0, m_h - n0);
      __syncthreads();
      for (int e = threadIdx.x; e < kSrc * d_h; e += kThreads) FK[e] = phi_f32(sq * Ks[e], inv_sqrt_dh, p.phi_mode);
      __syncthreads();
      float part = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jj = tt.j0 + u, j = j0 + jj;
        float w = 0.f;
        if (j <= i && i < p.T) {
          float s = 0.f;
          if (j >= i - W + 1) {  // window (eq. 7): eq. 6 weight
            for (int e = 0; e < d_h; ++e) s = fmaf(Qs[tt.r * d_h + e], Ks[jj * d_h + e], s);
            w = exp2f(c * (s - 1.f));
          } else {  // older source: eq. 9 weight
            for (int e = 0; e < d_h; ++e) s = fmaf(FQ[tt.r * d_h + e], FK[jj * d_h + e], s);
            w = shift * s;
          }
        }
        Ps[tt.r * 33 + jj] = w;
        part += w;
      }
      den += row_group_sum(part);
      __syncthreads();
      for (int jj = 0; jj < kSrc; ++jj) {
        const float w = Ps[tt.r * 33 + jj];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, Gs[jj * kCols + tt.c0 + e], acc[e]);
      }
    }
    finish_rows<T>(p, tt, acc, den, b, i, a, n0, m_h, tau);
    // Sources that leave the window before the next tile enter the running sums.
    const int new_lo = min(p.T, max(0, i0 + kRows - W + 1));
    for (int j0 = state_lo; j0 < new_lo; j0 += kSrc) {
      __syncthreads();
      const int src_valid = min(kSrc, new_lo - j0);
      load_rows<T>(Ks, k, seq + j0, src_valid, d_h, p.dqk, a * d_h, d_h);
      load_rows<T>(Gs, g, seq + j0, src_valid, kCols, p.m, a * m_hp + n0, m_h - n0);
      __syncthreads();
      for (int e = threadIdx.x; e < kSrc * d_h; e += kThreads) {
        const int jj = e / d_h;
        FK[e] = jj < src_valid ? phi_f32(sq * Ks[e], inv_sqrt_dh, p.phi_mode) : 0.f;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < d_h * kCols; e += kThreads) {
        const int cc = e / kCols, n = e % kCols;
        float s = S[e];
        for (int jj = 0; jj < src_valid; ++jj) s = fmaf(FK[jj * d_h + cc], Gs[jj * kCols + n], s);
        S[e] = s;
      }
      for (int cc = threadIdx.x; cc < d_h; cc += kThreads) {
        float s = z[cc];
        for (int jj = 0; jj < src_valid; ++jj) s += FK[jj * d_h + cc];
        z[cc] = s;
      }
    }
    state_lo = max(state_lo, new_lo);
  }
}

template <typename T>
cudaError_t launch_agg(const AggArgs& p, cudaStream_t s, bool wango) {
  const int d_h = p.dqk / p.H, m_hp = p.m / p.H, m_h = p.m_h ? p.m_h : m_hp;
  const int ntile = (m_h + kCols - 1) / kCols;
  if (!wango) {
    const size_t smem = sizeof(float) * (size_t)(kRows * d_h + kSrc * d_h + kSrc * kCols + kRows * 33);
    auto kern = tango_simt_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.H * ntile, (p.T + kRows - 1) / kRows, p.B);
    kern<<<grid, kThreads, smem, s>>>(p);
  } else {
    const size_t smem = sizeof(float) * (size_t)(d_h * kCols + d_h + 2 * kRows * d_h + 2 * kSrc * d_h +
                                                 kSrc * kCols + kRows * 33);
    auto kern = wango_simt_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.H * ntile, 1, p.B);
    kern<<<grid, kThreads, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_prep(tg_dtype dt, const void* in, void* out, long long rows, int T, int H, int dqk,
                           float rope_base, bool normalize, cudaStream_t s) {
  const long long n = rows * H;
  const int threads = 128;
  const unsigned blocks = (unsigned)((n + threads - 1) / threads);
  if (dt == TG_F32)
    qk_prep_kernel<float><<<blocks, threads, 0, s>>>(static_cast<const float*>(in), static_cast<float*>(out),
                                                     rows, T, H, dqk, rope_base, normalize ? 1 : 0);
  else
    qk_prep_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(in),
                                                             static_cast<__nv_bfloat16*>(out), rows, T, H, dqk,
                                                             rope_base, normalize ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(tg_dtype dt, const void* h, const void* gamma, void* x, long long rows, int d,
                           float eps, cudaStream_t s) {
  const int warps = 8;
  const unsigned blocks = (unsigned)((rows + warps - 1) / warps);
  if (dt == TG_F32)
    rmsnorm_kernel<float><<<blocks, warps * 32, 0, s>>>(static_cast<const float*>(h),
                                                        static_cast<const float*>(gamma), static_cast<float*>(x),
                                                        rows, d, eps);
  else
    rmsnorm_kernel<__nv_bfloat16><<<blocks, warps * 32, 0, s>>>(
        static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(gamma),
        static_cast<__nv_bfloat16*>(x), rows, d, eps);
  return cudaGetLastError();
}

// ------------------------------------------------------------- model helpers

// Token-embedding lookup (sec. 2.3): h[r, :] = E[ids[r], :], one warp per row.  An id
// outside [0, vocab) is flagged in the error word and its row is written as zeros.
template <typename T>
__global__ void embed_kernel(const int* ids, const T* E, T* h, long long rows, int d, int vocab, unsigned* err) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int id = ids[r];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && lane == 0) record_error(err, kErrValue | kKernModel);
  const T* src = E + (long long)(ok ? id : 0) * d;
  T* dst = h + r * d;
  for (int c = lane; c < d; c += 32) dst[c] = ok ? src[c] : T(0.f);
}

// Copy of a gate-indexed weight with each head's block of m_h entries moved to a
// pitch of m_hp (>= m_h) entries, zeros after it.  axis 0: src [H*m_h, C] -> dst
// [H*m_hp, C] (W_g, W_v); axis 1: src [R, H*m_h] -> dst [R, H*m_hp] (W_o).  R, C are
// the destination's extents.  A plain element copy; no arithmetic.
// Destination rows blockIdx.y, + gridDim.y, ...; each thread takes 8 consecutive
// destination elements (2048 per block along a row), written as one 16-byte vector when
// `vec` (row pitch and bases allow it).  W_g/W_v rows copy whole source rows; a W_o row
// gathers each head's columns, whose source offsets need not be aligned.
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const T* v, int n, bool vec) {
  if (vec && n == 8) {
    static_assert(sizeof(T) == 2 || sizeof(T) == 4, "element size");
    if constexpr (sizeof(T) == 2) {
      *reinterpret_cast<uint4*>(p) =
          make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    } else {
      *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
  } else {
    for (int e = 0; e < n; ++e) p[e] = v[e];
  }
}
template <typename T>
__global__ void __launch_bounds__(256) pad_gate_kernel(const T* src, T* dst, int R, int C, int axis, int H,
                                                       int m_h, int m_hp, bool vec) {
  const int c = (blockIdx.x * 256 + threadIdx.x) * 8;
  if (c >= C) return;
  const int n = C - c < 8 ? C - c : 8;
  for (int r = blockIdx.y; r < R; r += gridDim.y) {
    T v[8];
    if (axis == 0) {
      // the whole row comes from one source row, or is zero
      const int head = r / m_hp, j = r - head * m_hp;
      const T* srow = src + ((size_t)head * m_h + (j < m_h ? j : 0)) * C;
      if (vec && n == 8 && j < m_h) {
        *reinterpret_cast<uint4*>(dst + (size_t)r * C + c) = *reinterpret_cast<const uint4*>(srow + c);
        if (sizeof(T) == 4)
          *reinterpret_cast<uint4*>(dst + (size_t)r * C + c + 4) = *reinterpret_cast<const uint4*>(srow + c + 4);
        continue;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (e < n && j < m_h) ? srow[c + e] : T(0.f);
    } else {
      const T* srow = src + (size_t)r * ((size_t)H * m_h);
      int head = c / m_hp, j = c - head * m_hp;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[e] = (e < n && j < m_h) ? srow[head * m_h + j] : T(0.f);
        if (++j == m_hp) {
          j = 0;
          ++head;
        }
      }
    }
    store8(dst + (size_t)r * C + c, v, n, vec);
  }
}

cudaError_t launch_embed(tg_dtype dt, const int* ids, const void* E, void* h, long long rows, int d, int vocab,
                         unsigned* err, cudaStream_t s) {
  const int warps = 8;
  const unsigned blocks = (unsigned)((rows + warps - 1) / warps);
  if (dt == TG_F32)
    embed_kernel<float><<<blocks, warps * 32, 0, s>>>(ids, static_cast<const float*>(E), static_cast<float*>(h),
                                                      rows, d, vocab, err);
  else
    embed_kernel<__nv_bfloat16><<<blocks, warps * 32, 0, s>>>(ids, static_cast<const __nv_bfloat16*>(E),
                                                              static_cast<__nv_bfloat16*>(h), rows, d, vocab, err);
  return cudaGetLastError();
}

cudaError_t launch_pad_gate(tg_dtype dt, const void* src, void* dst, long long R, long long C, int axis, int H,
                            int m_h, int m_hp, cudaStream_t s) {
  if (R * C == 0) return cudaSuccess;
  if (R > 0x7fffffffLL || C > 0x7fffffffLL - 2048) return cudaErrorInvalidValue;
  const size_t es = dt == TG_F32 ? 4 : 2;
  const bool vec = ((size_t)C * es) % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
  const dim3 grid((unsigned)((C + 2047) / 2048), (unsigned)(R < 65535 ? R : 65535));  // 2048 elements per block
  if (dt == TG_F32)
    pad_gate_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(src), static_cast<float*>(dst), (int)R,
                                                (int)C, axis, H, m_h, m_hp, vec);
  else
    pad_gate_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src),
                                                        static_cast<__nv_bfloat16*>(dst), (int)R, (int)C, axis, H,
                                                        m_h, m_hp, vec);
  return cudaGetLastError();
}

cudaError_t launch_gemm_simt(tg_dtype dt, const void* A, const void* B, void* C, const void* R, int M, int N,
                             int K, int ldc, int epi, cudaStream_t s) {
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  if (dt == TG_F32)
    gemm_simt_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(A), static_cast<const float*>(B),
                                                 static_cast<float*>(C), static_cast<const float*>(R), M, N, K,
                                                 ldc, epi);
  else
    gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
        static_cast<__nv_bfloat16*>(C), static_cast<const __nv_bfloat16*>(R), M, N, K, ldc, epi);
  return cudaGetLastError();
}

cudaError_t launch_tango_simt(const AggArgs& a, cudaStream_t s) {
  return a.dtype == TG_F32 ? launch_agg<float>(a, s, false) : launch_agg<__nv_bfloat16>(a, s, false);
}

cudaError_t launch_wango_simt(const AggArgs& a, cudaStream_t s) {
  return a.dtype == TG_F32 ? launch_agg<float>(a, s, true) : launch_agg<__nv_bfloat16>(a, s, true);
}

}  // namespace tg
