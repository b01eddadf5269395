// Internal launchers of the tensor-core (tcgen05) kernels.
#pragma once
#include <cuda_runtime.h>

#include "tg_kernels.h"

namespace tg {

// Projection GEMM of one block: x [M, d] against W_q, W_k [dqk, d] and W_g, W_v
// [m, d]; epilogues: RoPE + unit norm per head (q, k), SiLU (g), identity (v).
struct ProjArgs {
  const void *x, *Wq, *Wk, *Wg, *Wv;
  void *q, *k, *g, *v;
  int M, d, T, H, dqk, m;
  float rope_base;
  unsigned* err;
  int debug_timeout;  // test hook: the GEMM times out on purpose (1 ms bound)
  int skip_v = 0;     // no v segment (the WANGO aggregation forms v itself)
};

cudaError_t launch_proj_tc(const ProjArgs& a, cudaStream_t s);
// h_out [M, d] = h + u [M, m] * Wo [d, m]^T
cudaError_t launch_out_tc(const void* u, const void* Wo, const void* h, void* h_out, int M, int d, int m,
                          unsigned* err, cudaStream_t s);
// C [M, N] = A [M, K] * B [N, K]^T, bf16 in and out, fp32 accumulation; K % 8 == 0,
// N % 8 == 0 and 16-byte-aligned bases (TMA).
cudaError_t launch_matmul_tc(const void* A, const void* B, void* C, int M, int N, int K, unsigned* err,
                             cudaStream_t s);
cudaError_t launch_tango_tc(const AggArgs& a, cudaStream_t s);
// Pair-weight gradients of the aggregation backward (backward_tc.cu): for every pair
// j <= i of each (batch, head), X_ij = tau w_ij (E_i . g_j - D_i) for window pairs
// (all pairs in TANGO) and E_i . g_j - D_i for older pairs (WANGO), in bf16.
struct BwdPairsArgs {
  int B, T, H, dqk, m;  // m: row width in memory (H x per-head pitch)
  int m_h;              // gates per head
  int wango, window;
  float s;
  const float* tau;
  const void* E;     // [B, T, m] bf16
  const void* g;     // [B, T, m] bf16
  const void* qhat;  // [B, T, dqk] bf16 unit
  const void* khat;
  const float* dp;   // [B * H, T_pad]
  void* X;           // [B * H, T_pad, T_pad] bf16: window pairs
  void* X_old;       // the same for older pairs (WANGO), else NULL
  unsigned* err;
};
cudaError_t launch_bwd_pairs_tc(const BwdPairsArgs& a, cudaStream_t s);
// dq and dk from X and X_old on the tensor cores (backward_tc.cu): window pairs through
// the unit vectors, older pairs through the forward's bf16 feature maps fq =
// e^-tau phi(sqrt(tau) qhat) and fk = phi(sqrt(tau) khat) and phi', then the unit
// normalisation of the raw q, k (raw == NULL: the gradient stops at the unit inputs).
struct BwdQKTcArgs {
  int B, T, H, dqk;
  int wango, window, phi_mode;
  float s;
  const float* tau;
  const void* X;
  const void* X_old;
  const void* qhat;
  const void* khat;
  const void* fq;     // WANGO only, [B, T, dqk] bf16
  const void* fk;
  const void* raw_q;
  const void* raw_k;
  void* dq;
  void* dk;
  unsigned* err;
};
cudaError_t launch_bwd_qk_tc(const BwdQKTcArgs& a, cudaStream_t s);
// Destination rows padded to whole 128-row blocks.
int bwd_tpad(int T);
// Address of the per-row WANGO denominators [B * H, T_pad] inside the scratch of the
// tensor-core path, as the last launch_wango_tc with this scratch left them.
const float* wango_den_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W);
// The forward's bf16 feature maps e^-tau phi(sqrt(tau) qhat) and phi(sqrt(tau) khat),
// [B, T, dqk], in the same scratch.
const void* wango_fq_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W);
const void* wango_fk_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W);
// The WANGO feature-map pre-pass alone (fq, fk and the block sums of fk into a.aux).
cudaError_t launch_wango_prepass(const AggArgs& a, cudaStream_t s);
cudaError_t launch_wango_tc(const AggArgs& a, cudaStream_t s);
// Scratch bytes the tensor-core WANGO path needs in AggArgs::aux (256-byte aligned):
// e^-tau phi(q~) and phi(k~) in bf16, per-block sums of phi(k~), the older-prefix
// denominator of every destination, and, when strips are split into segments, the
// states handed from one segment to the next with their flags.
size_t wango_aux_bytes(int B, int T, int H, int dqk, int m, int W);

}  // namespace tg
