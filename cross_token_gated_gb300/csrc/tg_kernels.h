// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tango.h"

namespace tg {

// Arguments of one aggregation launch.  q/k are unit-normalised per head.
struct AggArgs {
  int B, T, H, dqk, m;
  float s;
  const float* tau;
  const float* null_bias;
  int window;  // WANGO only
  int phi_mode;
  unsigned flags;
  tg_dtype dtype;
  const void* q;
  const void* k;
  const void* g;
  const void* v;  // may be NULL
  void* out;
  unsigned* err;  // device error word
  void* aux;      // WANGO, tensor-core path: feature-map scratch (wango_aux_bytes)
  // m is the row width in memory, H gate blocks of m / H columns (the per-head pitch);
  // m_h the gates of a head that are read and written (0: m / H)
  int m_h = 0;
  // Backward helpers (tensor-core kernels):
  int rev = 0;              // TANGO: sources j >= i instead of j <= i
  int mirror = 0;           // WANGO: the time-reversed problem on the tensors as they lie
                            // (see launch_wango_tc); needs no_norm, v and null_bias NULL
  int no_norm = 0;          // TANGO and WANGO: the numerator alone, no division by the denominator
  float* den_out = nullptr; // TANGO: every row's denominator, [B * H, den_pitch]
  int den_pitch = 0;        // 0: ceil(T / 128) * 128
  void* gbar_out = nullptr; // TANGO and WANGO (tensor cores): gbar in the storage type, laid out as out
  // WANGO with v fused: v = x W_v^T is formed inside the aggregation (then v == NULL)
  const void* fuse_x = nullptr;   // [B, T, fuse_d] bf16, the block's normalised input
  const void* fuse_wv = nullptr;  // [m, fuse_d] bf16
  int fuse_d = 0;                 // a multiple of 64
};

enum Epi : int { kEpiStore = 0, kEpiSilu = 1, kEpiResidual = 2 };

// WANGO decode state (one buffer, regions 256-byte aligned): the running sums S
// [B, H, d_h, m_h] and z [2, B, H, d_h] in f32 (z alternates between its two buffers by
// step parity: a step reads buffer pos % 2 and writes the other), the ring of the last
// W + kDecodeFold tokens' unit k [B, H, R, d_h] and g [B, R, m] (both in the storage
// type), and per-step scratch: the ring weights [B, H, R], e^-tau phi(q~) [B, H, d_h],
// the feature maps of the sources waiting to be folded [B, H, kDecodeFold, d_h], the
// weights' partial sums [B, H, 8] and the older-prefix term [B, H].
// Sources that leave the window are folded into S and z in groups of this many; until
// then they stay in the ring (of W + kDecodeFold slots) with their feature-map weight.
constexpr int kDecodeFold = 8;
struct DecodeState {
  float* S;
  float* z;
  void* ring_k;   // [B * H, W + kDecodeFold, d_h]
  void* ring_g;   // [B, W + kDecodeFold, m]
  float* w;       // [B * H, W + kDecodeFold]
  float* fq;
  float* fk_fold; // [B * H, kDecodeFold, d_h]: phi(k~_j) of pending source j in slot j mod kDecodeFold
  float* wpart;
  float* older;
};
cudaError_t launch_wango_decode(tg_dtype dt, int B, int H, int dqk, int m, int W, long long pos, float s,
                                const float* tau, const float* null_bias, int phi_mode, int qk_normalized,
                                const void* q, const void* k, const void* g, const void* v, void* out,
                                const DecodeState& st, unsigned* err, cudaStream_t stream);

// ---- CUDA-core kernels (simt.cu) -------------------------------------------
// Per (row, head): optional RoPE at position row % T, then optional unit
// normalisation.  in may equal out.
cudaError_t launch_qk_prep(tg_dtype dt, const void* in, void* out, long long rows, int T, int H, int dqk,
                           float rope_base, bool normalize, cudaStream_t s);
// x = gamma * h / sqrt(mean(h^2) + eps), per row of width d.
cudaError_t launch_rmsnorm(tg_dtype dt, const void* h, const void* gamma, void* x, long long rows, int d,
                           float eps, cudaStream_t s);
// C[M, N] (row pitch ldc) = epi(A[M, K] * B[N, K]^T), fp32 accumulation.
cudaError_t launch_gemm_simt(tg_dtype dt, const void* A, const void* B, void* C, const void* R, int M, int N,
                             int K, int ldc, int epi, cudaStream_t s);
// h[r, :] = E[ids[r], :] (sec. 2.3); ids outside [0, vocab) give zero rows and an error flag.
cudaError_t launch_embed(tg_dtype dt, const int* ids, const void* E, void* h, long long rows, int d, int vocab,
                         unsigned* err, cudaStream_t s);
// Gate-indexed weight with each head's m_h entries at a pitch of m_hp, zero-padded;
// axis 0 pads rows (W_g, W_v), axis 1 columns (W_o).  R, C: destination extents.
cudaError_t launch_pad_gate(tg_dtype dt, const void* src, void* dst, long long R, long long C, int axis, int H,
                            int m_h, int m_hp, cudaStream_t s);
cudaError_t launch_tango_simt(const AggArgs& a, cudaStream_t s);

// ---- backward helpers (backward_simt.cu), bf16 storage --------------------
// Per (row, head): E = dout * v / den (v == NULL: dout / den) in bf16, dv = dout * gbar
// (if dv), and D = sum_c E_c gbar_c over the head's columns into dp [B * H, T_pad].
cudaError_t launch_bwd_prep(const void* dout, const void* v, const void* gbar, const float* den, int den_pitch,
                            void* E, void* dv, float* dp, int B, int T, int T_pad, int H, int m, int m_h,
                            cudaStream_t s);

cudaError_t launch_wango_simt(const AggArgs& a, cudaStream_t s);

}  // namespace tg
