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
  int band = -1;     // WANGO with the far older pairs left to the scans: only source blocks
                     // jb >= ib - band of destination block ib (band = ceil((W - 1) / 128))
  unsigned* err;
  int debug_timeout = 0;  // test hook: the MMA issuer waits on a barrier nothing signals (1 ms)
};
cudaError_t launch_bwd_pairs_tc(const BwdPairsArgs& a, cudaStream_t s);
// WANGO: the far older pairs' feature-map gradients through running sums (backward_tc.cu).
// The scans write per-strip sums (strips of 256-512 gate columns) into part[0] [strips, B*T,
// H, d_h] for dFq (sum_far (E_i . g_j) Fk_j) and part[1] for dFk (sum_far (E_i . g_j)
// Fq_i); a reduction then leaves in strip 0 of each, for every row of a far block, the
// whole far term: sum_far (E_i . g_j - D_i) Fk_j (part[0]) and sum_far (E_i . g_j - D_i)
// Fq_i (part[1]).  rb [B, H, nblk, d_h] holds the block sums of D_i Fq_i and fb [2, B,
// H, nblk, d_h] the plain far sums of Fk (per destination block) and of D_i Fq_i (per
// source block).
struct BwdScanArgs {
  int B, T, H, dqk, m, m_h, window;
  const void* E;
  const void* g;
  const void* fq;
  const void* fk;
  const float* zb;  // [B, H, nblk, d_h] block sums of Fk (the forward's)
  const float* dp;  // [B * H, T_pad]
  float* part[2];
  float* rb;
  float* fb;
  unsigned* err;
  int debug_timeout = 0;  // test hook: the MMA issuer waits on a barrier nothing signals (1 ms)
};
// Strips of the scans (of bwd_scan_ns columns each) for B * H sequence-heads of m_h gates.
int bwd_scan_strips(int B, int H, int m_h);
int bwd_scan_ns(int B, int H, int m_h);
int bwd_band(int window);
// Whether the scans are estimated to beat forming the far older pairs one by one.
bool bwd_scan_pays(int B, int T, int H, int dqk, int m_h, int window);
cudaError_t launch_bwd_scan(const BwdScanArgs& a, cudaStream_t s);
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
  // far older pairs from the scans (band >= 0): partner blocks beyond the band are skipped
  // and far[side] [B*T, H, d_h] (f32, rows of far blocks only) is added instead
  int band = -1;
  const float* far[2] = {nullptr, nullptr};
  unsigned* err;
  int debug_timeout = 0;  // test hook: the MMA issuer waits on a barrier nothing signals (1 ms)
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
const float* wango_zb_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W);
// The WANGO feature-map pre-pass alone (fq, fk and the block sums of fk into a.aux).
cudaError_t launch_wango_prepass(const AggArgs& a, cudaStream_t s);
cudaError_t launch_wango_tc(const AggArgs& a, cudaStream_t s);
// Scratch bytes the tensor-core WANGO path needs in AggArgs::aux (256-byte aligned):
// e^-tau phi(q~) and phi(k~) in bf16, per-block sums of phi(k~), the older-prefix
// denominator of every destination, and, when strips are split into segments, the
// states handed from one segment to the next with their flags.
size_t wango_aux_bytes(int B, int T, int H, int dqk, int m, int W);

}  // namespace tg
