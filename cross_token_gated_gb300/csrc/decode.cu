// WANGO autoregressive decode step, "TANGO: Token-Aggregated Nonlinear Gating
// Operators ...", sec. 2.2 eqs. 7-10: destination i = pos takes exp(tau (qhat.khat_j - 1))
// weights over its window j = i-W+1 .. i and, for every older source, the running sums
//   S = sum_{j <= i-W} phi(k~_j) g_j^T   (d_h x m_h per head),   z = sum phi(k~_j),
// read out as e^-tau phi(q~_i)^T S and e^-tau phi(q~_i)^T z (eq. 10).  After the
// output, source i-W+1 leaves the window and enters S and z, and the current token joins
// the ring of the last W tokens.  One call per token; the state is constant-size in T.
//
// Two kernels per step:
//   wango_decode_scores_kernel  per (head, batch): unit q and k, the window weights, the
//       feature maps, the denominator, z's update and the ring's khat slot.
//   wango_decode_gate_kernel    per 256 gate columns and batch (HBM-bound): the window
//       sum over the ring of g, the older-prefix read-out from S, u = gbar * v, the
//       leaving token's rank-1 update of S and the ring's g slot.
#include <math.h>

#include "tg_common.cuh"
#include "tg_kernels.h"

namespace tg {
namespace {

constexpr int kMaxDh = 128;

template <typename T>
struct DecodeArgs {
  int B, H, dqk, m, d_h, m_h, W;
  long long pos;
  float s;
  const float* tau;
  const float* null_bias;
  int phi_mode;
  int qk_normalized;
  const T *q, *k, *g, *v;
  T* out;
  DecodeState st;
  unsigned* err;
};

__device__ __forceinline__ float phi_of(float u, float inv_sqrt_dh, int mode) {
  const float e1 = u > 0.f ? u + 1.f : expf(u);  // ELU(u) + 1
  if (mode == 1) return e1;
  return fmaxf(e1 + 1e-4f, 1e-4f) * inv_sqrt_dh;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

// grid (H, B), 256 threads.
template <typename T>
__global__ void __launch_bounds__(256) wango_decode_scores_kernel(const DecodeArgs<T> a) {
  __shared__ float qh[kMaxDh], kh[kMaxDh], red[8];
  const int head = blockIdx.x, bb = blockIdx.y, t = threadIdx.x;
  const int d_h = a.d_h, W = a.W;
  const long long i = a.pos;
  const int bh = bb * a.H + head;
  const float tau = head_tau(a.tau, a.s, head, a.err, kKernWango);
  const float sq = sqrtf(tau), shift = expf(-tau), inv_sqrt_dh = rsqrtf((float)d_h);
  // unit q and k of this head (sec. 2.1)
  const T* qr = a.q + (size_t)bb * a.dqk + (size_t)head * d_h;
  const T* kr = a.k + (size_t)bb * a.dqk + (size_t)head * d_h;
  const float qv = t < d_h ? io<T>::ld(qr + t) : 0.f, kv = t < d_h ? io<T>::ld(kr + t) : 0.f;
  const float qn = a.qk_normalized ? 1.f : fmaxf(sqrtf(block_sum(qv * qv, red)), 1e-12f);
  const float kn = a.qk_normalized ? 1.f : fmaxf(sqrtf(block_sum(kv * kv, red)), 1e-12f);
  if (t < d_h) {
    qh[t] = qv / qn;
    kh[t] = kv / kn;
  }
  __syncthreads();
  // the current token's khat into its ring slot (slot i mod W held source i - W, which is
  // already in the state and outside the window)
  T* ring_k = static_cast<T*>(a.st.ring_k) + (size_t)bh * W * d_h;
  const int cur = (int)(i % W);
  const long long jl = i - W + 1;  // the source that leaves the window after this step
  const int lslot = jl >= 0 ? (int)(jl % W) : -1;
  // feature map of the leaving source, read before its slot could be overwritten
  float* fkl = a.st.fk_leave + (size_t)bh * d_h;
  if (t < d_h && lslot >= 0) {
    const float kl = lslot == cur ? kh[t] : io<T>::ld(ring_k + (size_t)lslot * d_h + t);
    fkl[t] = phi_of(sq * kl, inv_sqrt_dh, a.phi_mode);
  }
  __syncthreads();
  if (t < d_h) io<T>::st(ring_k + (size_t)cur * d_h + t, kh[t]);
  __syncthreads();
  // window weights, one ring slot per thread: slot s holds source j = the largest j <= i
  // with j = s (mod W)
  float* wv = a.st.w + (size_t)bh * W;
  float wsum = 0.f;
  for (int s = t; s < W; s += blockDim.x) {
    const long long j = i - (long long)((cur - s + W) % W);
    float w = 0.f;
    if (j >= 0) {
      float dot = 0.f;
      for (int c = 0; c < d_h; ++c) dot = fmaf(qh[c], io<T>::ld(ring_k + (size_t)s * d_h + c), dot);
      w = expf(tau * (dot - 1.f));
    }
    wv[s] = w;
    wsum += w;
  }
  wsum = block_sum(wsum, red);
  // older prefix: e^-tau phi(q~) . z, then z += phi(k~_leave)
  float* z = a.st.z + (size_t)bh * d_h;
  float* fq = a.st.fq + (size_t)bh * d_h;
  const float fqv = t < d_h ? shift * phi_of(sq * qh[t], inv_sqrt_dh, a.phi_mode) : 0.f;
  const float older = block_sum(t < d_h ? fqv * z[t] : 0.f, red);
  if (t < d_h) {
    fq[t] = fqv;
    if (lslot >= 0) z[t] += fkl[t];
  }
  if (t == 0) {
    const float null_w = a.null_bias ? expf(a.null_bias[head] - tau) : 0.f;
    a.st.inv_den[bh] = 1.f / (wsum + older + (float)(i + 1) * null_w);
  }
}

// grid (ceil(m / 128), B), 128 threads, one gate column per thread.
template <typename T>
__global__ void __launch_bounds__(128) wango_decode_gate_kernel(const DecodeArgs<T> a) {
  const int bb = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= a.m) return;
  const int head = c / a.m_h, cl = c % a.m_h;
  const int bh = bb * a.H + head, d_h = a.d_h, W = a.W;
  const long long i = a.pos;
  const int cur = (int)(i % W);
  const long long jl = i - W + 1;
  const int lslot = jl >= 0 ? (int)(jl % W) : -1;
  const T* ring_g = static_cast<const T*>(a.st.ring_g) + (size_t)bb * W * a.m + c;
  const float gi = io<T>::ld(a.g + (size_t)bb * a.m + c);
  const float* wv = a.st.w + (size_t)bh * W;
  // window: the current token from its input, the others from the ring (four
  // independent sums, so that many loads are in flight)
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  int s = 0;
#pragma unroll 2
  for (; s + 4 <= W; s += 4) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float gv = s + e == cur ? gi : io<T>::ld(ring_g + (size_t)(s + e) * a.m);
      acc[e] = fmaf(wv[s + e], gv, acc[e]);
    }
  }
  for (; s < W; ++s) acc[0] = fmaf(wv[s], s == cur ? gi : io<T>::ld(ring_g + (size_t)s * a.m), acc[0]);
  // older prefix and the leaving source's update of S (after its read-out)
  float* S = a.st.S + (size_t)bh * d_h * a.m_h + cl;
  const float* fq = a.st.fq + (size_t)bh * d_h;
  const float* fkl = a.st.fk_leave + (size_t)bh * d_h;
  const float gl = lslot < 0 ? 0.f : (lslot == cur ? gi : io<T>::ld(ring_g + (size_t)lslot * a.m));
  int d = 0;
  for (; d + 4 <= d_h; d += 4) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float sv = S[(size_t)(d + e) * a.m_h];
      acc[e] = fmaf(fq[d + e], sv, acc[e]);
      if (lslot >= 0) S[(size_t)(d + e) * a.m_h] = fmaf(fkl[d + e], gl, sv);
    }
  }
  for (; d < d_h; ++d) {
    const float sv = S[(size_t)d * a.m_h];
    acc[0] = fmaf(fq[d], sv, acc[0]);
    if (lslot >= 0) S[(size_t)d * a.m_h] = fmaf(fkl[d], gl, sv);
  }
  const float num = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  const float gbar = num * a.st.inv_den[bh];
  const float u = a.v ? gbar * io<T>::ld(a.v + (size_t)bb * a.m + c) : gbar;
  io<T>::st(a.out + (size_t)bb * a.m + c, u);
  // the current token's g into its ring slot
  io<T>::st(const_cast<T*>(ring_g) + (size_t)cur * a.m, gi);
}

template <typename T>
cudaError_t launch(const DecodeArgs<T>& a, cudaStream_t s) {
  wango_decode_scores_kernel<T><<<dim3(a.H, a.B), 256, 0, s>>>(a);
  wango_decode_gate_kernel<T><<<dim3((a.m + 127) / 128, a.B), 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_wango_decode(tg_dtype dt, int B, int H, int dqk, int m, int W, long long pos, float s,
                                const float* tau, const float* null_bias, int phi_mode, int qk_normalized,
                                const void* q, const void* k, const void* g, const void* v, void* out,
                                const DecodeState& st, unsigned* err, cudaStream_t stream) {
  if (dt == TG_F32) {
    DecodeArgs<float> a{B, H, dqk, m, dqk / H, m / H, W, pos, s, tau, null_bias, phi_mode, qk_normalized,
                        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(g),
                        static_cast<const float*>(v), static_cast<float*>(out), st, err};
    return launch(a, stream);
  }
  DecodeArgs<__nv_bfloat16> a{B, H, dqk, m, dqk / H, m / H, W, pos, s, tau, null_bias, phi_mode, qk_normalized,
                              static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                              static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(v),
                              static_cast<__nv_bfloat16*>(out), st, err};
  return launch(a, stream);
}

}  // namespace tg
