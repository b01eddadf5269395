// WANGO autoregressive decode step, "TANGO: Token-Aggregated Nonlinear Gating
// Operators ...", sec. 2.2 eqs. 7-10: destination i = pos takes exp(tau (qhat.khat_j - 1))
// weights over its window j = i-W+1 .. i and, for every older source, the feature-map
// weight e^-tau phi(q~_i) . phi(k~_j), summed through the running sums
//   S = sum_j phi(k~_j) g_j^T   (d_h x m_h per head),   z = sum_j phi(k~_j)
// and read out as e^-tau phi(q~_i)^T S and e^-tau phi(q~_i)^T z (eq. 10).  One call per
// token; the state is constant-size in T.
//
// Sources enter S and z in groups of kDecodeFold: a source that leaves the window stays
// in the ring (W + kDecodeFold slots) with its feature-map weight computed directly until
// its group is complete, and the step that completes a group adds the whole group to S
// and z.  S is therefore rewritten on one step in kDecodeFold instead of on every step
// (S is about a quarter of a step's bytes at W = 256, d_h = 64); the sums are the same.
//
// Two kernels per step:
//   wango_decode_scores_kernel  per (head, batch, part of the ring): unit q and k, the
//       weights of its ring slots (window, or left the window and not yet folded) and
//       their partial sum; the first part also the feature maps, the older-prefix term
//       Fq . z, the current key into its ring slot, and on a fold step the group's feature
//       maps and z's update.  At one or two sequences the ring is split over 8 CTAs per
//       head, so that the chain of dependent steps in one CTA is short.
//   wango_decode_gate_kernel    per 128 (or 64) gate columns and batch (HBM-bound): the
//       denominator from the partial sums, the weighted sum over the ring of g, the
//       read-out Fq^T S, u = gbar * v, on a fold step S's update by the group, and the
//       current token's g into its ring slot.  At one or two sequences it is launched as a
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
// 16 bytes global -> shared without a register round trip (completes at cp_async_wait)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <typename T>
struct DecodeArgs {
  int B, H, dqk, m, d_h, m_h, W;
  int R;  // ring slots, W + kDecodeFold
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

// Two block-wide sums in one pass (red: 16 floats).
__device__ __forceinline__ void block_sum2(float& x, float& y, float* red) {
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) {
    red[2 * w] = x;
    red[2 * w + 1] = y;
  }
  __syncthreads();
  x = 0.f;
  y = 0.f;
  for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
    x += red[2 * k];
    y += red[2 * k + 1];
  }
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

// Which sources a step sees where (i = pos): the window i-W+1 .. i; the sources from
// `first` (the oldest not yet in S, a multiple of kDecodeFold) to i-W through the ring with
// their feature-map weight; everything older through S and z.  The step folds when the
// source that leaves after it, i-W+1, completes a group.
__device__ __forceinline__ long long first_unfolded(long long i, int W) {
  const long long lo = i - W + 1;
  return lo > 0 ? (long long)kDecodeFold * (lo / kDecodeFold) : 0;
}
__host__ __device__ __forceinline__ bool fold_step(long long i, int W) {
  const long long lo = i - W + 1;
  return lo >= 0 && (lo + 1) % kDecodeFold == 0;
}

// grid (H, B, parts), 256 threads; part p takes ring slots [p * ceil(R / parts), ...).
template <typename T>
__global__ void __launch_bounds__(256) wango_decode_scores_kernel(const DecodeArgs<T> a) {
  __shared__ float qh[kMaxDh], kh[kMaxDh], fqs[kMaxDh], red[16];
  __shared__ __align__(16) unsigned char kstage[40960];  // a chunk of the ring's keys
  const int head = blockIdx.x, bb = blockIdx.y, part = blockIdx.z, t = threadIdx.x;
  const int d_h = a.d_h, W = a.W, R = a.R;
  const long long i = a.pos;
  const int bh = bb * a.H + head;
  const int per = (R + gridDim.z - 1) / gridDim.z;
  const int s_lo = min(R, part * per), s_hi = min(R, s_lo + per);
  griddep_launch_dependents();  // the gate kernel may start fetching its rows now
  // the ring's keys (written by earlier steps) start on their way to shared memory at
  // once: the first chunk by asynchronous copies when it is 16-byte aligned
  T* ring_k = static_cast<T*>(a.st.ring_k) + (size_t)bh * R * d_h;
  T* ks = reinterpret_cast<T*>(kstage);
  const int chunk = (int)(sizeof(kstage) / ((size_t)d_h * sizeof(T)));  // slots per chunk
  bool first_async = false;
  if (s_lo < s_hi) {
    const T* src = ring_k + (size_t)s_lo * d_h;
    const size_t bytes = (size_t)min(chunk, s_hi - s_lo) * d_h * sizeof(T);
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && bytes % 16 == 0) {
      for (size_t x = t; x < bytes / 16; x += blockDim.x)
        cp_async16(kstage + 16 * x, reinterpret_cast<const uint8_t*>(src) + 16 * x);
      cp_async_commit();
      first_async = true;
    }
  }
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
    fqs[t] = shift * phi_of(sq * qh[t], inv_sqrt_dh, a.phi_mode);  // e^-tau phi(q~)
  }
  __syncthreads();
  // the current token's khat into its ring slot (slot i mod R held source i - R, which is
  // already in the state; no part uses what its copy reads there)
  const int cur = (int)(i % R);
  const long long lo_win = i - W + 1, first = first_unfolded(i, W);
  if (part == 0 && t < d_h) io<T>::st(ring_k + (size_t)cur * d_h + t, kh[t]);
  // weights: the ring's keys pass through shared memory in chunks (one coalesced copy
  // each), then one ring slot per thread; slot s holds source j = the largest j <= i with
  // j = s (mod R).  No part reads slot cur from the ring: its weight comes from kh.  The
  // dot products start at column s (mod d_h), so the threads of a warp read different banks.
  float* wv = a.st.w + (size_t)bh * R;
  float wsum = 0.f;
  for (int s0 = s_lo; s0 < s_hi; s0 += chunk) {
    const int n = min(chunk, s_hi - s0);
    const T* src = ring_k + (size_t)s0 * d_h;
    const size_t bytes = (size_t)n * d_h * sizeof(T);
    if (s0 == s_lo && first_async) {
      cp_async_wait();
    } else if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && bytes % 16 == 0) {
      __syncthreads();  // the previous chunk has been read
      for (size_t x = t; x < bytes / 16; x += blockDim.x)
        reinterpret_cast<uint4*>(kstage)[x] = reinterpret_cast<const uint4*>(src)[x];
    } else {
      __syncthreads();
      for (int x = t; x < n * d_h; x += blockDim.x) ks[x] = src[x];
    }
    __syncthreads();
    for (int sl = t; sl < n; sl += blockDim.x) {
      const int s = s0 + sl;
      const long long j = i - (long long)((cur - s + R) % R);
      float w = 0.f;
      if (j >= 0 && j >= first) {
        const T* kr = ks + (size_t)sl * d_h;
        if (j >= lo_win) {  // in the window
          float dot = 0.f;
          if (s == cur) {
            for (int c = 0; c < d_h; ++c) dot = fmaf(qh[c], kh[c], dot);
          } else {
            for (int cc = 0, c = s % d_h; cc < d_h; ++cc, c = c + 1 == d_h ? 0 : c + 1)
              dot = fmaf(qh[c], io<T>::ld(kr + c), dot);
          }
          w = expf(tau * (dot - 1.f));
        } else {  // left the window, not yet in S: e^-tau phi(q~) . phi(k~_j)
          const float* fk = a.st.fk_fold + ((size_t)bh * kDecodeFold + (int)(j % kDecodeFold)) * d_h;
          for (int cc = 0, c = s % d_h; cc < d_h; ++cc, c = c + 1 == d_h ? 0 : c + 1) w = fmaf(fqs[c], fk[c], w);
        }
      }
      wv[s] = w;
      wsum += w;
    }
  }
  // the partial sum of the weights, and in part 0 the older prefix Fq . z, in one pass
  const float* z = a.st.z + ((size_t)(i & 1) * a.B * a.H + bh) * d_h;
  float* z_next = a.st.z + ((size_t)((i + 1) & 1) * a.B * a.H + bh) * d_h;
  float older = part == 0 && t < d_h ? fqs[t] * z[t] : 0.f;
  block_sum2(wsum, older, red);
  if (t == 0) a.st.wpart[(size_t)bh * kMaxParts + part] = wsum;
  if (part != 0) return;
  // part 0: the feature map of the source that leaves the window after this step
  // (i - W + 1) into its slot of the feature-map ring (slot j mod kDecodeFold, which no
  // pending source holds now); z' into the other buffer (the sums alternate between two
  // buffers by step parity): z plus, on a fold step, the group's feature maps, which the
  // gate kernel also takes for S
  if (t < d_h) {
    float* fkf = a.st.fk_fold + (size_t)bh * kDecodeFold * d_h;
    if (lo_win >= 0) {
      const float kj = lo_win == i ? kh[t] : io<T>::ld(ring_k + (size_t)(lo_win % R) * d_h + t);
      fkf[(int)(lo_win % kDecodeFold) * d_h + t] = phi_of(sq * kj, inv_sqrt_dh, a.phi_mode);
    }
    float zs = z[t];
    if (fold_step(i, W))
      for (int u = 0; u < kDecodeFold; ++u) zs += fkf[u * d_h + t];
    a.st.fq[(size_t)bh * d_h + t] = fqs[t];
    z_next[t] = zs;
  }
  if (t == 0) a.st.older[bh] = older;
}

// Gate kernel layout: a CTA takes C (128 or 64) gate columns of one sequence as C / 8
// groups of 8 columns, and its 256 threads split each group's work kSl = 2048 / C ways
// ("slices"): slice r sums the ring slots r, r + kSl, ... and the state rows r, r + kSl,
// ...  The slices' partial
// sums meet in shared memory.  A thread moves 8 columns at a time (16-byte loads of
// bf16, two of f32) when every row pitch and base allows it and no group straddles a
// head; otherwise it takes its 8 columns one by one.
constexpr int kGateCols = 128, kGroup = 8;

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

// grid (ceil(m / C), B), 256 threads.  FOLD: this step completes a group (fold_step).
// FEW: one or two sequences (launched early, the ring read in batches of 9 slots, three
// CTAs an SM so that one sequence's 64-column blocks fit in one wave).  Each is a
// separate instance so that the other launches keep a lean register budget.
template <typename T, bool VEC, int C, bool FOLD, bool FEW>
__global__ void __launch_bounds__(256, (VEC && sizeof(T) == 2) || FEW ? 3 : 6)
    wango_decode_gate_kernel(const DecodeArgs<T> a, int parts) {
  constexpr int kG = C / kGroup;  // 8-column groups
  constexpr int kSl = 256 / kG;   // slices per group
  // bf16 vectors: the ring is read kB slots a thread at a time, and for one or two
  // sequences the first kB are loaded into registers before the scores are waited for
  // (the ring rows and the inputs do not depend on them)
  constexpr bool kPre = VEC && sizeof(T) == 2;
  constexpr int kB = 9;  // W + 8 slots of W = 256 are 9 a thread at 64 columns
  __shared__ float red[kSl][C + 4];
  __shared__ float inv_den[TG_MAX_HEADS];
  // a fold step's group of kDecodeFold g rows over this block's columns, staged once and
  // read by every state row's update
  __shared__ __align__(16) T fold_g[FOLD ? kDecodeFold : 1][FOLD ? C : kGroup];
  const int bb = blockIdx.y, grp = threadIdx.x % kG, sl = threadIdx.x / kG;
  const int col0 = blockIdx.x * C, d_h = a.d_h, W = a.W, R = a.R, m = a.m;
  const int c0 = col0 + grp * kGroup;  // first of this thread's 8 columns
  const bool col_ok = c0 < m;
  const long long i = a.pos;
  const int cur = (int)(i % R);
  const long long j0 = i - W + 1 - (kDecodeFold - 1);  // a fold step's first source
  const T* gin = a.g + (size_t)bb * m;
  const T* ring_g = static_cast<const T*>(a.st.ring_g) + (size_t)bb * R * m;
  // ---- before the scores: what the previous steps (completed before the score kernel
  // began) and the inputs fix
  uint4 r[kPre ? kB : 1];
  if constexpr (kPre) {
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int s = sl + u * kSl;
      r[u] = make_uint4(0, 0, 0, 0);
      if (col_ok && s < R) r[u] = *reinterpret_cast<const uint4*>((s == cur ? gin : ring_g + (size_t)s * m) + c0);
    }
  }
  if constexpr (FOLD) {  // the group's rows (written by earlier steps, or this step's input)
    constexpr int kPer = 16 / (int)sizeof(T);  // elements of a 16-byte chunk
    for (int e = threadIdx.x; e < kDecodeFold * (C / kPer); e += blockDim.x) {
      const int u = e / (C / kPer), x = (e % (C / kPer)) * kPer;
      const long long j = j0 + u;
      const T* row = j == i ? gin : ring_g + (size_t)(j % R) * m;
      if (VEC && col0 + x < m) {
        cp_async16(&fold_g[u][x], row + col0 + x);
      } else {
#pragma unroll
        for (int y = 0; y < kPer; ++y) io<T>::st(&fold_g[u][x + y], col0 + x + y < m ? io<T>::ld(row + col0 + x + y) : 0.f);
      }
    }
    cp_async_commit();
  }
  if (FEW && col_ok) {  // this thread's state rows (and any further ring rows) into L2
    for (int s = sl + (kPre ? kB * kSl : 0); s < R; s += kSl)
      if (s != cur) prefetch_l2(ring_g + (size_t)s * m + c0);
    const int hd = c0 / a.m_h;
    for (int d = sl; d < d_h; d += kSl)
      prefetch_l2(a.st.S + (((size_t)bb * a.H + hd) * d_h + d) * a.m_h + (c0 - hd * a.m_h));
  }
  const int oc = col0 + (int)threadIdx.x;  // the output stage's column
  const bool o_ok = (int)threadIdx.x < C && oc < m;
  float v_o = 1.f, g_o = 0.f;
  if (o_ok) {
    if (a.v) v_o = io<T>::ld(a.v + (size_t)bb * m + oc);
    g_o = io<T>::ld(gin + oc);
  }
  griddep_wait();  // the weights, feature maps and partial sums of this step
  // ---- after: this sequence's denominators (loaded now, used at the end)
  float wsum = 0.f, older = 0.f;
  if ((int)threadIdx.x < a.H) {
    const int bh = bb * a.H + (int)threadIdx.x;
    for (int p = 0; p < parts; ++p) wsum += a.st.wpart[(size_t)bh * kMaxParts + p];
    older = a.st.older[bh];
  }
  if constexpr (FOLD) {
    cp_async_wait();
    __syncthreads();
  }
  float acc[kGroup];
#pragma unroll
  for (int e = 0; e < kGroup; ++e) acc[e] = 0.f;
  if (col_ok) {
    // the head of the group's first column; with VEC the whole group shares it, and
    // otherwise each column takes its own head below
    const int head0 = c0 / a.m_h;
    const int lim = m;
    // the ring: slots sl, sl + kSl, ... with the score kernel's weights (0 for a slot whose
    // source is already in S); the current token's slot from the input
    int s_begin = sl;
    if constexpr (kPre) {
      const float* wrow = a.st.w + (size_t)(bb * a.H + head0) * R;
      for (int batch = 0;; ++batch) {
        float wv[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int s = s_begin + u * kSl;
          wv[u] = s < R ? wrow[s] : 0.f;
          if (batch > 0) {
            r[u] = make_uint4(0, 0, 0, 0);
            if (s < R) r[u] = *reinterpret_cast<const uint4*>((s == cur ? gin : ring_g + (size_t)s * m) + c0);
          }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const uint32_t gw[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(wv[u], __uint_as_float(gw[e] << 16), acc[2 * e]);
            acc[2 * e + 1] = fmaf(wv[u], __uint_as_float(gw[e] & 0xFFFF0000u), acc[2 * e + 1]);
          }
        }
        s_begin += kB * kSl;
        if (s_begin >= R) break;
      }
    }
    float x[kGroup];
#pragma unroll 2
    for (int s = s_begin; s < R; s += kSl) {
      Cols8<T, VEC>::ld(s == cur ? gin : ring_g + (size_t)s * m, c0, lim, x);
      if (VEC) {
        const float w = a.st.w[(size_t)(bb * a.H + head0) * R + s];
#pragma unroll
        for (int e = 0; e < kGroup; ++e) acc[e] = fmaf(w, x[e], acc[e]);
      } else {
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int hd = min(c0 + e, m - 1) / a.m_h;
          acc[e] = fmaf(a.st.w[(size_t)(bb * a.H + hd) * R + s], x[e], acc[e]);
        }
      }
    }
    // older prefix: rows sl, sl + kSl, ... of S read out, and on a fold step updated by the
    // group of kDecodeFold sources that completes now (its g rows from shared memory).
    // With 16-byte vectors a thread has kSB of its state rows in flight at once (all loads
    // first, then the read-out, the update and the stores): 4 in the plain launches that
    // leave registers for them, 2 on their fold steps (which also store the rows) and in
    // the early launches for one or two sequences (whose rows are already on their way to
    // L2, and whose chain after the wait is the step's).
    if (VEC) {
      constexpr int kSB = FEW ? 2 : (kPre ? (FOLD ? 2 : 4) : 1);
      const size_t bh = (size_t)bb * a.H + head0;
      const int cl = c0 - head0 * a.m_h;
#pragma unroll 1
      for (int d0 = sl; d0 < d_h; d0 += kSB * kSl) {
        float sv[kSB][kGroup], fq[kSB];
#pragma unroll
        for (int b = 0; b < kSB; ++b) {
          const int d = d0 + b * kSl;
          fq[b] = 0.f;
          if (d < d_h) {
            ld_f32x8<true>(a.st.S + (bh * d_h + d) * a.m_h, cl, a.m_h, sv[b]);
            fq[b] = a.st.fq[bh * d_h + d];
          } else {
#pragma unroll
            for (int e = 0; e < kGroup; ++e) sv[b][e] = 0.f;
          }
        }
#pragma unroll
        for (int b = 0; b < kSB; ++b)
#pragma unroll
          for (int e = 0; e < kGroup; ++e) acc[e] = fmaf(fq[b], sv[b][e], acc[e]);
        if constexpr (FOLD) {
#pragma unroll
          for (int b = 0; b < kSB; ++b) {
            const int d = d0 + b * kSl;
            if (d >= d_h) break;
            const float* fkf = a.st.fk_fold + bh * kDecodeFold * d_h + d;
#pragma unroll 2
            for (int u = 0; u < kDecodeFold; ++u) {
              const float fk = fkf[u * d_h];
              float x[kGroup];
              Cols8<T, true>::ld(&fold_g[u][0], grp * kGroup, C, x);
#pragma unroll
              for (int e = 0; e < kGroup; ++e) sv[b][e] = fmaf(fk, x[e], sv[b][e]);
            }
            st_f32x8<true>(a.st.S + (bh * d_h + d) * a.m_h, cl, a.m_h, sv[b]);
          }
        }
      }
    } else {
#pragma unroll 1
      for (int d = sl; d < d_h; d += kSl) {
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int c = c0 + e;
          if (c >= m) break;
          const int hd = c / a.m_h;
          const size_t bh = (size_t)bb * a.H + hd;
          float* sp = a.st.S + (bh * d_h + d) * a.m_h + (c - hd * a.m_h);
          float sv = *sp;
          acc[e] = fmaf(a.st.fq[bh * d_h + d], sv, acc[e]);
          if constexpr (FOLD) {
#pragma unroll
            for (int u = 0; u < kDecodeFold; ++u)
              sv = fmaf(a.st.fk_fold[(bh * kDecodeFold + u) * d_h + d], io<T>::ld(&fold_g[u][grp * kGroup + e]), sv);
            *sp = sv;
          }
        }
      }
    }
  }
  if ((int)threadIdx.x < a.H) {
    const int hd = (int)threadIdx.x;
    const float tau = head_tau(a.tau, a.s, hd, a.err, kKernWango);
    const float null_w = a.null_bias ? expf(a.null_bias[hd] - tau) : 0.f;
    inv_den[hd] = 1.f / (wsum + older + (float)(i + 1) * null_w);
  }
#pragma unroll
  for (int e = 0; e < kGroup; ++e) red[sl][grp * kGroup + e] = acc[e];
  __syncthreads();
  // one column per thread: the slices' sums, the denominator, u = gbar * v, and the
  // current token's g into its ring slot
  if (o_ok) {
    float num = 0.f;
#pragma unroll
    for (int q = 0; q < kSl; ++q) num += red[q][threadIdx.x];
    const float gbar = num * inv_den[oc / a.m_h];
    io<T>::st(a.out + (size_t)bb * m + oc, a.v ? gbar * v_o : gbar);
    T gs;
    io<T>::st(&gs, g_o);
    const_cast<T*>(ring_g)[(size_t)cur * m + oc] = gs;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T, bool FOLD>
cudaError_t launch_gate(const DecodeArgs<T>& a, int parts, bool few, bool vec, cudaStream_t s) {
  if (!few) {  // enough CTAs to hide latency: 128-column blocks and a plain launch
    const dim3 grid((a.m + kGateCols - 1) / kGateCols, a.B);
    if (vec) wango_decode_gate_kernel<T, true, kGateCols, FOLD, false><<<grid, 256, 0, s>>>(a, parts);
    else wango_decode_gate_kernel<T, false, kGateCols, FOLD, false><<<grid, 256, 0, s>>>(a, parts);
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
    return vec ? cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, true, 64, FOLD, true>, a, parts)
               : cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, false, 64, FOLD, true>, a, parts);
  return vec ? cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, true, kGateCols, FOLD, true>, a, parts)
             : cudaLaunchKernelEx(&cfg, wango_decode_gate_kernel<T, false, kGateCols, FOLD, true>, a, parts);
}

template <typename T>
cudaError_t launch(const DecodeArgs<T>& a, cudaStream_t s) {
  // one or two sequences: the ring split over up to 8 CTAs per head (a short dependent
  // chain per CTA) and the gate kernel launched early
  const bool few = a.B <= 2;
  const int parts = few ? min(kMaxParts, (a.R + 31) / 32) : min(kMaxParts, (a.R + 127) / 128);
  wango_decode_scores_kernel<T><<<dim3(a.H, a.B, parts), 256, 0, s>>>(a);
  // 8-column vectors when every row of g, the ring and S starts 16-byte aligned and no
  // 8-column group straddles a head
  const bool vec = (a.m * sizeof(T)) % 16 == 0 && a.m_h % kGroup == 0 && aligned16(a.g) &&
                   aligned16(a.st.ring_g) && aligned16(a.st.S);
  return fold_step(a.pos, a.W) ? launch_gate<T, true>(a, parts, few, vec, s)
                               : launch_gate<T, false>(a, parts, few, vec, s);
}

}  // namespace

cudaError_t launch_wango_decode(tg_dtype dt, int B, int H, int dqk, int m, int W, long long pos, float s,
                                const float* tau, const float* null_bias, int phi_mode, int qk_normalized,
                                const void* q, const void* k, const void* g, const void* v, void* out,
                                const DecodeState& st, unsigned* err, cudaStream_t stream) {
  if (dt == TG_F32) {
    DecodeArgs<float> a{B, H, dqk, m, dqk / H, m / H, W, W + kDecodeFold, pos, s, tau, null_bias, phi_mode,
                        qk_normalized, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(g),
                        static_cast<const float*>(v), static_cast<float*>(out), st, err};
    return launch(a, stream);
  }
  DecodeArgs<__nv_bfloat16> a{B, H, dqk, m, dqk / H, m / H, W, W + kDecodeFold, pos, s, tau, null_bias, phi_mode,
                              qk_normalized, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                              static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(v),
                              static_cast<__nv_bfloat16*>(out), st, err};
  return launch(a, stream);
}

}  // namespace tg
