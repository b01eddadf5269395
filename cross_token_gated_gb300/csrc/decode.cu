// WANGO autoregressive decode step, "TANGO: Token-Aggregated Nonlinear Gating
// Operators ...", sec. 2.2 eqs. 7-10: destination i = pos takes exp(tau (qhat.khat_j - 1))
// weights over its window j = i-W+1 .. i and, for every older source, the running sums
//   S = sum_{j <= i-W} phi(k~_j) g_j^T   (d_h x m_h per head),   z = sum phi(k~_j),
// read out as e^-tau phi(q~_i)^T S and e^-tau phi(q~_i)^T z (eq. 10).  After the
// output, source i-W+1 leaves the window and enters S and z, and the current token joins
// the ring of the last W tokens.  One call per token; the state is constant-size in T.
//
// Two kernels per step:
//   wango_decode_scores_kernel  per (head, batch, part of the ring): unit q and k, the
//       window weights of its ring slots and their partial sum; the first part also the
//       feature maps, the older-prefix term, z's update and the ring's khat slot.  At
//       one or two sequences the ring is split over 8 CTAs per head, so that the chain
//       of dependent steps in one CTA is short.
//   wango_decode_gate_kernel    per 128 gate columns and batch (HBM-bound): the
//       denominator from the partial sums, the window sum over the ring of g, the
//       older-prefix read-out from S, u = gbar * v, the leaving token's rank-1 update of
//       S and the ring's g slot.  At one or two sequences it is launched as a
//       programmatic dependent of the score kernel: it asks its rows of the ring and of
//       S into L2 while the score kernel runs, and waits for the scores only then.
#include <math.h>

#include "tg_common.cuh"
#include "tg_kernels.h"

namespace tg {
namespace {

constexpr int kMaxDh = 128;
constexpr int kMaxParts = 8;  // ring parts of the score kernel (the partial sums' stride)

// Programmatic dependent launch: the score kernel lets the gate kernel of the same step
// start early; the gate kernel waits for the score kernel's results (and memory) only
// where it first needs them.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ uint32_t smem_u32_of(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

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

// grid (H, B, parts), 256 threads; part p takes ring slots [p * ceil(W / parts), ...).
template <typename T>
__global__ void __launch_bounds__(256) wango_decode_scores_kernel(const DecodeArgs<T> a) {
  __shared__ float qh[kMaxDh], kh[kMaxDh], red[8];
  __shared__ __align__(16) unsigned char kstage[32768];  // a chunk of the ring's keys
  const int head = blockIdx.x, bb = blockIdx.y, part = blockIdx.z, t = threadIdx.x;
  const int d_h = a.d_h, W = a.W;
  const long long i = a.pos;
  const int bh = bb * a.H + head;
  const int per = (W + gridDim.z - 1) / gridDim.z;
  const int s_lo = min(W, part * per), s_hi = min(W, s_lo + per);
  griddep_launch_dependents();  // the gate kernel may start fetching its rows now
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
    // as the ring stores it (the storage type): the current slot's weight uses this value
    T kr1;
    io<T>::st(&kr1, kv / kn);
    kh[t] = io<T>::ld(&kr1);
  }
  __syncthreads();
  // the current token's khat into its ring slot (slot i mod W held source i - W, which is
  // already in the state and outside the window)
  T* ring_k = static_cast<T*>(a.st.ring_k) + (size_t)bh * W * d_h;
  const int cur = (int)(i % W);
  const long long jl = i - W + 1;  // the source that leaves the window after this step
  const int lslot = jl >= 0 ? (int)(jl % W) : -1;
  // part 0: feature map of the leaving source (its slot is not rewritten this step), and
  // the current key into its slot.  No part reads slot cur from the ring: its weight
  // comes from kh.
  float* fkl = a.st.fk_leave + (size_t)bh * d_h;
  if (part == 0 && t < d_h) {
    if (lslot >= 0) {
      const float kl = lslot == cur ? kh[t] : io<T>::ld(ring_k + (size_t)lslot * d_h + t);
      fkl[t] = phi_of(sq * kl, inv_sqrt_dh, a.phi_mode);
    }
    io<T>::st(ring_k + (size_t)cur * d_h + t, kh[t]);
  }
  // window weights: the ring's keys pass through shared memory in chunks (one coalesced
  // copy each), then one ring slot per thread; slot s holds source j = the largest
  // j <= i with j = s (mod W).  The dot product starts at column s (mod d_h), so the
  // threads of a warp read different banks.
  float* wv = a.st.w + (size_t)bh * W;
  T* ks = reinterpret_cast<T*>(kstage);
  const int chunk = (int)(sizeof(kstage) / ((size_t)d_h * sizeof(T)));  // slots per chunk
  float wsum = 0.f;
  for (int s0 = s_lo; s0 < s_hi; s0 += chunk) {
    const int n = min(chunk, s_hi - s0);
    const T* src = ring_k + (size_t)s0 * d_h;
    const size_t bytes = (size_t)n * d_h * sizeof(T);
    __syncthreads();  // the previous chunk has been read
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && bytes % 16 == 0) {
      for (size_t x = t; x < bytes / 16; x += blockDim.x)
        reinterpret_cast<uint4*>(kstage)[x] = reinterpret_cast<const uint4*>(src)[x];
    } else {
      for (int x = t; x < n * d_h; x += blockDim.x) ks[x] = src[x];
    }
    __syncthreads();
    for (int sl = t; sl < n; sl += blockDim.x) {
      const int s = s0 + sl;
      const long long j = i - (long long)((cur - s + W) % W);
      float w = 0.f;
      if (j >= 0) {
        const T* kr = ks + (size_t)sl * d_h;
        float dot = 0.f;
        if (s == cur) {
          for (int c = 0; c < d_h; ++c) dot = fmaf(qh[c], kh[c], dot);
        } else {
          for (int cc = 0, c = s % d_h; cc < d_h; ++cc, c = c + 1 == d_h ? 0 : c + 1)
            dot = fmaf(qh[c], io<T>::ld(kr + c), dot);
        }
        w = expf(tau * (dot - 1.f));
      }
      wv[s] = w;
      wsum += w;
    }
  }
  wsum = block_sum(wsum, red);
  if (t == 0) a.st.wpart[(size_t)bh * kMaxParts + part] = wsum;
  if (part != 0) return;
  // part 0: older prefix e^-tau phi(q~) . z, then z' = z + phi(k~_leave) into the other
  // buffer (the sums alternate between two buffers by step parity)
  const float* z = a.st.z + ((size_t)(i & 1) * a.B * a.H + bh) * d_h;
  float* z_next = a.st.z + ((size_t)((i + 1) & 1) * a.B * a.H + bh) * d_h;
  float* fq = a.st.fq + (size_t)bh * d_h;
  const float fqv = t < d_h ? shift * phi_of(sq * qh[t], inv_sqrt_dh, a.phi_mode) : 0.f;
  __syncthreads();  // fkl written above by this CTA
  const float older = block_sum(t < d_h ? fqv * z[t] : 0.f, red);
  if (t < d_h) {
    fq[t] = fqv;
    z_next[t] = lslot >= 0 ? z[t] + fkl[t] : z[t];
  }
  if (t == 0) a.st.older[bh] = older;
}

// Gate kernel layout: a CTA takes 128 gate columns of one sequence as 16 groups of 8
// columns, and its 256 threads split each group's work 16 ways ("slices"): slice r sums
// the ring slots r, r + 16, ... and the state rows r, r + 16, ...  The slices' partial
// sums meet in shared memory.  A thread moves 8 columns at a time (16-byte loads of
// bf16, two of f32) when every row pitch and base allows it and no group straddles a
// head; otherwise it takes its 8 columns one by one.
constexpr int kGateCols = 128, kGroup = 8, kSlices = 16;

template <typename T, bool VEC>
struct Cols8 {
  // the 8 columns [c0, c0 + 8) of row p (columns at or past `lim` read as 0)
  static __device__ __forceinline__ void ld(const T* p, int c0, int lim, float* x) {
#pragma unroll
    for (int e = 0; e < kGroup; ++e) x[e] = c0 + e < lim ? io<T>::ld(p + c0 + e) : 0.f;
  }
};
template <>
struct Cols8<__nv_bfloat16, true> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, int c0, int, float* x) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + c0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
};
template <>
struct Cols8<float, true> {
  static __device__ __forceinline__ void ld(const float* p, int c0, int, float* x) {
    const float4 u = *reinterpret_cast<const float4*>(p + c0), v = *reinterpret_cast<const float4*>(p + c0 + 4);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
  }
};
template <bool VEC>
__device__ __forceinline__ void ld_f32x8(const float* p, int c0, int lim, float* x) {
  Cols8<float, VEC>::ld(p, c0, lim, x);
}
template <bool VEC>
__device__ __forceinline__ void st_f32x8(float* p, int c0, int lim, const float* x) {
  if (VEC) {
    *reinterpret_cast<float4*>(p + c0) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + c0 + 4) = make_float4(x[4], x[5], x[6], x[7]);
  } else {
#pragma unroll
    for (int e = 0; e < kGroup; ++e)
      if (c0 + e < lim) p[c0 + e] = x[e];
  }
}

// grid (ceil(m / 128), B), 256 threads.
template <typename T, bool VEC, int C>
__global__ void __launch_bounds__(256) wango_decode_gate_kernel(const DecodeArgs<T> a, int parts) {
  constexpr int kG = C / kGroup;  // 8-column groups
  constexpr int kSl = 256 / kG;   // slices per group
  __shared__ float red[kSl][C + 4];
  __shared__ float inv_den[TG_MAX_HEADS];
  const int bb = blockIdx.y, grp = threadIdx.x % kG, sl = threadIdx.x / kG;
  const int col0 = blockIdx.x * C, d_h = a.d_h, W = a.W, m = a.m;
  const int c0 = col0 + grp * kGroup;  // first of this thread's 8 columns
  const long long i = a.pos;
  const int cur = (int)(i % W);
  const long long jl = i - W + 1;
  const int lslot = jl >= 0 ? (int)(jl % W) : -1;
  const T* gin = a.g + (size_t)bb * m;
  const T* ring_g = static_cast<const T*>(a.st.ring_g) + (size_t)bb * W * m;
  // while the score kernel runs: this thread's ring and state rows into L2 (the previous
  // step's gate kernel, which wrote them, has completed before the score kernel began)
  if (parts > 1 && c0 < m) {  // launched early (one or two sequences)
    for (int s = sl; s < W; s += kSl)
      if (s != cur) prefetch_l2(ring_g + (size_t)s * m + c0);
    const int hd = c0 / a.m_h;
    for (int d = sl; d < d_h; d += kSl)
      prefetch_l2(a.st.S + (((size_t)bb * a.H + hd) * d_h + d) * a.m_h + (c0 - hd * a.m_h));
  }
  griddep_wait();  // the window weights, feature maps and partial sums of this step
  if (threadIdx.x < a.H) {  // this sequence's denominators
    const int hd = threadIdx.x, bh = bb * a.H + hd;
    float wsum = 0.f;
    for (int p = 0; p < parts; ++p) wsum += a.st.wpart[(size_t)bh * kMaxParts + p];
    const float tau = head_tau(a.tau, a.s, hd, a.err, kKernWango);
    const float null_w = a.null_bias ? expf(a.null_bias[hd] - tau) : 0.f;
    inv_den[hd] = 1.f / (wsum + a.st.older[bh] + (float)(i + 1) * null_w);
  }
  __syncthreads();
  float acc[kGroup];
#pragma unroll
  for (int e = 0; e < kGroup; ++e) acc[e] = 0.f;
  if (c0 < m) {
    // the head of the group's first column; with VEC the whole group shares it, and
    // otherwise each column takes its own head below
    const int head0 = c0 / a.m_h;
    const int lim = m;
    // window: ring slots sl, sl + 16, ...; the current token's slot from the input.  With
    // bf16 vectors and one or two sequences, eight slots' loads are issued before their
    // products, so that one thread keeps eight loads in flight (a single sequence has
    // few threads to hide HBM latency with)
    float x[kGroup];
    int s_begin = sl;
    if constexpr (VEC && sizeof(T) == 2) if (parts > 1) {
      const float* wrow = a.st.w + (size_t)(bb * a.H + head0) * W;
      for (; s_begin + 7 * kSl < W; s_begin += 8 * kSl) {
        uint4 r[8];
        float wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int s = s_begin + u * kSl;
          r[u] = *reinterpret_cast<const uint4*>((s == cur ? gin : ring_g + (size_t)s * m) + c0);
          wv[u] = wrow[s];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t gw[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(wv[u], __uint_as_float(gw[e] << 16), acc[2 * e]);
            acc[2 * e + 1] = fmaf(wv[u], __uint_as_float(gw[e] & 0xFFFF0000u), acc[2 * e + 1]);
          }
        }
      }
    }
#pragma unroll 2
    for (int s = s_begin; s < W; s += kSl) {
      Cols8<T, VEC>::ld(s == cur ? gin : ring_g + (size_t)s * m, c0, lim, x);
      if (VEC) {
        const float w = a.st.w[(size_t)(bb * a.H + head0) * W + s];
#pragma unroll
        for (int e = 0; e < kGroup; ++e) acc[e] = fmaf(w, x[e], acc[e]);
      } else {
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int hd = min(c0 + e, m - 1) / a.m_h;
          acc[e] = fmaf(a.st.w[(size_t)(bb * a.H + hd) * W + s], x[e], acc[e]);
        }
      }
    }
    // older prefix: rows sl, sl + 16, ... of S, read out and then updated by the source
    // that leaves the window
    float gl[kGroup];
    if (lslot >= 0) Cols8<T, VEC>::ld(lslot == cur ? gin : ring_g + (size_t)lslot * m, c0, lim, gl);
#pragma unroll 1
    for (int d = sl; d < d_h; d += kSl) {
      if (VEC) {
        const size_t bh = (size_t)bb * a.H + head0;
        float* Srow = a.st.S + (bh * d_h + d) * a.m_h;
        const int cl = c0 - head0 * a.m_h;
        float sv[kGroup];
        ld_f32x8<true>(Srow, cl, a.m_h, sv);
        const float fq = a.st.fq[bh * d_h + d];
#pragma unroll
        for (int e = 0; e < kGroup; ++e) acc[e] = fmaf(fq, sv[e], acc[e]);
        if (lslot >= 0) {
          const float fk = a.st.fk_leave[bh * d_h + d];
#pragma unroll
          for (int e = 0; e < kGroup; ++e) sv[e] = fmaf(fk, gl[e], sv[e]);
          st_f32x8<true>(Srow, cl, a.m_h, sv);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int c = c0 + e;
          if (c >= m) break;
          const int hd = c / a.m_h;
          const size_t bh = (size_t)bb * a.H + hd;
          float* sp = a.st.S + (bh * d_h + d) * a.m_h + (c - hd * a.m_h);
          const float sv = *sp;
          acc[e] = fmaf(a.st.fq[bh * d_h + d], sv, acc[e]);
          if (lslot >= 0) *sp = fmaf(a.st.fk_leave[bh * d_h + d], gl[e], sv);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < kGroup; ++e) red[sl][grp * kGroup + e] = acc[e];
  __syncthreads();
  // one column per thread: the slices' sums, the denominator, u = gbar * v, and the
  // current token's g into its ring slot
  if (threadIdx.x < C) {
    const int c = col0 + threadIdx.x;
    if (c < m) {
      float num = 0.f;
#pragma unroll
      for (int r = 0; r < kSl; ++r) num += red[r][threadIdx.x];
      const int hd = c / a.m_h;
      const float gbar = num * inv_den[hd];
      const float u = a.v ? gbar * io<T>::ld(a.v + (size_t)bb * m + c) : gbar;
      io<T>::st(a.out + (size_t)bb * m + c, u);
      io<T>::st(const_cast<T*>(ring_g) + (size_t)cur * m + c, io<T>::ld(gin + c));
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T>
cudaError_t launch(const DecodeArgs<T>& a, cudaStream_t s) {
  // one or two sequences: the ring split over up to 8 CTAs per head (a short dependent
  // chain per CTA) and the gate kernel launched early
  const bool few = a.B <= 2;
  const int parts = few ? min(kMaxParts, (a.W + 31) / 32) : 1;
  wango_decode_scores_kernel<T><<<dim3(a.H, a.B, parts), 256, 0, s>>>(a);
  // 8-column vectors when every row of g, the ring and S starts 16-byte aligned and no
  // 8-column group straddles a head
  const bool vec = (a.m * sizeof(T)) % 16 == 0 && a.m_h % kGroup == 0 && aligned16(a.g) &&
                   aligned16(a.st.ring_g) && aligned16(a.st.S);
  if (!few) {  // enough CTAs to hide latency: 128-column blocks and a plain launch
    const dim3 grid((a.m + kGateCols - 1) / kGateCols, a.B);
    if (vec) wango_decode_gate_kernel<T, true, kGateCols><<<grid, 256, 0, s>>>(a, parts);
    else wango_decode_gate_kernel<T, false, kGateCols><<<grid, 256, 0, s>>>(a, parts);
    return cudaGetLastError();
  }
  // one or two sequences: launched as a programmatic dependent of the score kernel; for
  // one sequence in 64-column blocks (twice the CTAs, spread more evenly over the SMs)
  const int cols = a.B == 1 ? 64 : kGateCols;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.m + cols - 1) / cols, a.B);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cols == 64)
    return vec ? cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, true, 64>, a, parts)
               : cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, false, 64>, a, parts);
  return vec ? cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, true, kGateCols>, a, parts)
             : cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, false, kGateCols>, a, parts);
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
