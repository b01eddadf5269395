// WANGO windowed gate aggregation on the tensor cores (tcgen05), "TANGO:
// Token-Aggregated Nonlinear Gating Operators ...", sec. 2.2 eqs. 7-10 in sec. 2.1
// eq. 5.  For destination i and head a (all weights carry the common factor e^-tau,
// which cancels in the ratio):
//   window  i-W < j <= i :  w_ij = exp(tau (qhat_i.khat_j - 1))                 (eq. 6)
//   older   j <= i-W     :  w_ij = e^-tau phi(sqrt(tau) qhat_i).phi(sqrt(tau) khat_j)  (eq. 9)
//   u_i = [sum_j w_ij g_j] / [sum_j w_ij + (i+1) e^{b-tau}] * v_i
// The older sources enter through the running sums of eq. 10,
//   S = sum phi(k~_j) g_j^T (d_h x gate columns),   z = sum phi(k~_j),
// read out as  e^-tau phi(q~_i)^T S  and  e^-tau phi(q~_i)^T z.
//
// Destination blocks ib (128 rows) take per-pair weights from the source blocks
//     jb = jlo(ib) .. ib,   jlo(ib) = floor(max(0, 128 ib - W + 1) / 128);
// the state holds every source j < 128 jlo(ib), older than the window for every
// destination of the block.  A source block is "mixed" when it also holds older pairs
// (128 jb <= 128 ib + 127 - W): its weights need the feature-map score too.  It
// "leaves" when jb < jlo(ib + 1): after its P.G the same G tile updates the state.
//
// The weights depend on q and k only, not on the gate column, so they are computed
// once per destination block and shared by every gate column:
//  1. Pre-pass (CUDA cores): Fq = e^-tau phi(sqrt(tau) qhat), Fk = phi(sqrt(tau) khat)
//     in bf16, and the column sums of Fk per source block.
//  2. wango_p_kernel (tcgen05): per (batch, head, destination block) the scores
//     Qhat Khat^T (and Fq Fk^T for mixed blocks) in TMEM, the weights in bf16 written
//     to global memory as P [destination, (ib - jb) * 128 + source], and the full
//     denominator (the row sums of the bf16 weights as applied, the older prefix
//     Fq_i . z with z the column sums of Fk below the window, and the null term).  P is
//     a band of T x (W + 128) per head: linear in T.
//  3. wango_g_kernel (tcgen05): per (batch, head, 128-column gate strip) the
//     destination blocks in order: O = sum_jb P_jb G_jb with both operands loaded by
//     TMA, the state update S^T += G^T Fk for leaving blocks, the read-out
//     O += Fq S_bf16 of the state before the block, and u = O / den * v.  Persistent
//     CTAs take strips (or segments of strips) round-robin; O is double-buffered in
//     TMEM so one block's epilogue overlaps the next block's MMAs.
#include <algorithm>

#include "tg_common.cuh"
#include "tg_ptx.cuh"
#include "tg_tc.h"
#include "tg_tma.h"

namespace tg {
namespace {

using namespace ptx;

constexpr int kBlk = 128;
constexpr int kNg = 128;                    // gate columns per strip
constexpr uint32_t kTile = kBlk * 64 * 2;   // 16 KB: a 128 x d_h bf16 tile at d_h = 64
constexpr uint32_t kGBox = 64 * 64 * 2;     // 8 KB: 64 rows x 64 columns
constexpr uint32_t kGStage = 4 * kGBox;     // 32 KB: 128 rows x 128 columns

__host__ __device__ __forceinline__ int jlo_of(int ib, int W) {
  const int lo = ib * kBlk - W + 1;
  return lo > 0 ? lo / kBlk : 0;
}
__device__ __forceinline__ bool is_mixed(int jb, int ib, int W) { return jb * kBlk <= ib * kBlk + kBlk - 1 - W; }
// The memory row of block blk's first row.  Mirrored, the kernels solve the time-reversed
// problem on the tensors as they lie: block blk of the reversed sequence is memory block
// n_iblk - 1 - blk, whose rows come in reverse order (row r is position kBlk - 1 - r of
// the block); rows past T read as zero and are not written.
__host__ __device__ __forceinline__ int mem_row(int blk, int n_iblk, int mirror) {
  return (mirror ? n_iblk - 1 - blk : blk) * kBlk;
}

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++stage == n) { stage = 0; phase ^= 1; }
  }
};

// Bounded waits: on expiry the kernel records a timeout and sets its abort flag, after
// which every role leaves its loops.  Bars needs `abort`, Args `err` and `timeout_ns`.
template <typename Bars, typename Args>
__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernWango);
  return false;
}
template <typename Bars, typename Args>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (mbar_try_wait_nc(smem_u32(bar), parity)) return true;
  return wait_slow(bar, parity, b, a);
}

// Byte offset of element column c (16-bit elements) of row r in a tile whose rows
// are RB bytes wide, stored with the matching TMA/UMMA swizzle (RB = 32, 64, 128).
template <int RB>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  const uint32_t off = (uint32_t)(r * RB + c * 2);
  constexpr uint32_t mask = RB == 128 ? 7u : RB == 64 ? 3u : 1u;
  return off ^ (((off >> 7) & mask) << 4);
}

// Weights of 32 sources of one row, written as 16 packed bf16 pairs.
//   kMode 0: every source is in the window: exp2(c (s - 1)).
//   kMode 2: general: 0 after i, exp2(c (s - 1)) in the window (j >= jw), else the
//            feature-map score f (older source).
// Source e sits at position j0 + e (kRev: j0 - e, a mirrored block).  dsum2 accumulates
// the row sum of the weights as rounded to bf16 (the denominator as applied), two f32
// lanes per packed instruction.
template <int kMode, bool kRev = false>
__device__ __forceinline__ void weights32(const uint32_t* r, const uint32_t* f, float c, int j0, int i, int jw,
                                          uint32_t (&p)[16], uint64_t (&dsum2)[2]) {
  const uint64_t cc = f32x2_pack(c, c), nc = f32x2_pack(-c, -c);
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float x0, x1;  // c (s - 1) for two sources in one packed f32x2 instruction
    f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), cc, nc), x0, x1);
    float w0 = ex2_approx(x0);
    float w1 = ex2_approx(x1);
    if (kMode == 2) {
      const int ja = kRev ? j0 - e : j0 + e, jn = kRev ? j0 - e - 1 : j0 + e + 1;
      if (ja < jw) w0 = __uint_as_float(f[e]);
      if (jn < jw) w1 = __uint_as_float(f[e + 1]);
      if (ja > i) w0 = 0.f;
      if (jn > i) w1 = 0.f;
    }
    const uint32_t pk = pack_bf16x2(w0, w1);
    dsum2[(e >> 1) & 1] = add_f32x2(dsum2[(e >> 1) & 1], bf16x2_widen(pk));
    p[e / 2] = pk;
  }
}

// ================================================================= weights (P) kernel

constexpr int kPThreads = 384;  // warp 0 TMA, warp 1 scores (and TMEM), warps 4-11 weights
constexpr int kPWeightWarp0 = 4;
constexpr int kPSlots = 2;      // 128-column score slots in TMEM

struct __align__(8) PBars {
  uint64_t qh_full, fq_full;       // qhat and Fq of the destination block
  uint64_t k_full[2], k_empty[2];  // khat ring
  uint64_t fk_full, fk_empty;      // Fk of a mixed block
  uint64_t s_full[kPSlots], slot_free[kPSlots];
  uint64_t rs_full;                // both warpgroups' row sums are in shared memory
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float rowsum[2][kBlk];           // per warpgroup, per destination row
  float z[64];                     // sum of Fk over the sources below the block's window
};
// smem: Qhat | Fq | K x 2 | Fk | Bars
constexpr size_t kPSmemBytes = 1024 + kTile * 5 + sizeof(PBars);

struct PArgs {
  int B, T, T_pad, H, dqk, d_h, W, n_iblk, ldp;
  int mirror;                      // the time-reversed problem (mem_row)
  float s;
  const float* tau;
  const float* null_bias;
  const float* zb;                 // [B, H, n_iblk, d_h] per-block column sums of Fk
  const __nv_bfloat16* fq;         // [B, T, dqk] Fq
  __nv_bfloat16* P;      // [B * H, T_pad, ldp]
  float* den;            // [B * H, T_pad]
  unsigned* err;
  uint64_t timeout_ns;
};

// One CTA per (destination block ib, head, batch).  Work units, newest source block
// first: a whole block (cos scores, 128 columns of a slot), or one 64-source half of a
// mixed block (cos scores in columns [0, 64) of the slot, feature-map scores in
// [64, 128)).  The weight warps turn a unit's scores into bf16 weights and write them
// to P; warpgroup w takes sources [64 w, 64 w + 64) of a block or [32 w, 32 w + 32) of
// a half.
template <int DH>
__global__ void __launch_bounds__(kPThreads, 1)
    wango_p_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmFQ, const __grid_constant__ CUtensorMap tmFK,
                   const PArgs a) {
  constexpr int RB = DH * 2;  // bytes per row of the q/k/feature tiles
  constexpr uint32_t lay = DH == 64 ? kSwizzle128B : DH == 32 ? kSwizzle64B : kSwizzle32B;
  constexpr uint32_t sbo = 8u * RB;
  constexpr uint32_t tile_bytes = kBlk * RB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sFQ = sQ + kTile;
  uint8_t* sK = sFQ + kTile;  // 2 tiles
  uint8_t* sFK = sK + 2 * kTile;
  PBars& b = *reinterpret_cast<PBars*>(sFK + kTile);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ib = blockIdx.x, head = blockIdx.y, bb = blockIdx.z;
  const int W = a.W, jlo = jlo_of(ib, W);
  const bool any_mixed = is_mixed(jlo, ib, W);  // the oldest source block is mixed if any is

  if (threadIdx.x == 0) {
    mbar_init(&b.qh_full, 1);
    mbar_init(&b.fq_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&b.k_full[s], 1);
      mbar_init(&b.k_empty[s], 1);
    }
    mbar_init(&b.fk_full, 1);
    mbar_init(&b.fk_empty, 1);
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(&b.s_full[s], 1);
      mbar_init(&b.slot_free[s], 8);
    }
    mbar_init(&b.rs_full, 8);
    mbar_init(&b.drain, 1);
    b.abort = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(&b.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    bool ok = true;
    const int irow = mem_row(ib, a.n_iblk, a.mirror);
    mbar_arrive_expect_tx(&b.qh_full, tile_bytes);
    tma_load_3d(sQ, &tmQ, &b.qh_full, head * DH, irow, bb);
    if (any_mixed) {
      mbar_arrive_expect_tx(&b.fq_full, tile_bytes);
      tma_load_3d(sFQ, &tmFQ, &b.fq_full, head * DH, irow, bb);
    }
    Ring kr;
    uint32_t kmask = 0, kph[2] = {}, fkph = 0, fk_n = 0;
    for (int jb = ib; ok && jb >= jlo; --jb) {
      if (!(ok = wait_bar(&b.k_empty[kr.stage], kr.phase ^ 1, b, a))) break;
      mbar_arrive_expect_tx(&b.k_full[kr.stage], tile_bytes);
      tma_load_3d(sK + kr.stage * kTile, &tmK, &b.k_full[kr.stage], head * DH, mem_row(jb, a.n_iblk, a.mirror), bb);
      kmask |= 1u << kr.stage;
      kph[kr.stage] = kr.phase;
      kr.next(2);
      if (is_mixed(jb, ib, W)) {
        if (!(ok = wait_bar(&b.fk_empty, fkph ^ 1, b, a))) break;
        mbar_arrive_expect_tx(&b.fk_full, tile_bytes);
        tma_load_3d(sFK, &tmFK, &b.fk_full, head * DH, mem_row(jb, a.n_iblk, a.mirror), bb);
        fkph ^= 1;
        ++fk_n;
      }
    }
    // no copy may be in flight when the CTA exits
    mbar_wait(&b.qh_full, 0, a.timeout_ns);
    if (any_mixed) mbar_wait(&b.fq_full, 0, a.timeout_ns);
    if (fk_n) mbar_wait(&b.fk_full, (fk_n - 1) & 1, a.timeout_ns);
    for (int s = 0; s < 2; ++s)
      if (kmask & (1u << s)) mbar_wait(&b.k_full[s], kph[s], a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue: scores
    constexpr uint32_t idesc_s = idesc_bf16_f32(kBlk, kBlk, false, false);  // 128 sources
    constexpr uint32_t idesc_h = idesc_bf16_f32(kBlk, 64, false, false);    // 64 sources
    const uint64_t qd = smem_desc(smem_u32(sQ), 16, sbo, lay);
    const uint64_t fqd = smem_desc(smem_u32(sFQ), 16, sbo, lay);
    const uint64_t kd0 = smem_desc(smem_u32(sK), 16, sbo, lay);
    const uint64_t fkd = smem_desc(smem_u32(sFK), 16, sbo, lay);
    bool ok = wait_bar(&b.qh_full, 0, b, a);
    if (ok && any_mixed) ok = wait_bar(&b.fq_full, 0, b, a);
    Ring ks;
    uint32_t u = 0, fkph = 0;
    for (int jb = ib; ok && jb >= jlo; --jb) {
      const bool mixed = is_mixed(jb, ib, W);
      for (int h = mixed ? 0 : -1; h <= (mixed ? 1 : -1); ++h) {
        const int slot = u & 1;
        if (u >= 2 && !(ok = wait_bar(&b.slot_free[slot], ((u - 2) >> 1) & 1, b, a))) break;
        if (!(ok = wait_bar(&b.k_full[ks.stage], ks.phase, b, a))) break;
        if (h >= 0 && !(ok = wait_bar(&b.fk_full, fkph, b, a))) break;
        tc_fence_after_nc();
        const uint64_t kd = kd0 + (uint64_t)((ks.stage * kTile) >> 4);
        const uint32_t sc = tmem + (uint32_t)(slot * 128);
        if (h < 0) {
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk)
            mma_bf16_ss_nc(sc, qd + (uint64_t)(kk * 2), kd + (uint64_t)(kk * 2), idesc_s, kk != 0);
        } else {
          const uint64_t hoff = (uint64_t)((h * 64 * RB) >> 4);
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk)
            mma_bf16_ss_nc(sc, qd + (uint64_t)(kk * 2), kd + hoff + (uint64_t)(kk * 2), idesc_h, kk != 0);
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk)
            mma_bf16_ss_nc(sc + 64, fqd + (uint64_t)(kk * 2), fkd + hoff + (uint64_t)(kk * 2), idesc_h, kk != 0);
        }
        mma_commit_nc(&b.s_full[slot]);
        ++u;
        if (h != 0) {  // the block's last unit releases its khat
          mma_commit_nc(&b.k_empty[ks.stage]);
          ks.next(2);
        }
        if (h == 1) {
          mma_commit_nc(&b.fk_empty);
          fkph ^= 1;
        }
      }
    }
    mma_commit(&b.drain);
    mbar_wait(&b.drain, 0, a.timeout_ns);
  } else if (warp >= kPWeightWarp0 && warp < kPWeightWarp0 + 8) {
    // ------------------------------------------------------------ weights -> P, row sums
    const int wg = (warp - kPWeightWarp0) / 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int pi = ib * kBlk + row;                                 // this row of P and den
    const int i = ib * kBlk + (a.mirror ? kBlk - 1 - row : row);    // its position
    const int mi = mem_row(ib, a.n_iblk, a.mirror) + row;           // its row in memory
    const int i0 = ib * kBlk + (a.mirror ? kBlk - 32 - quarter * 32 : quarter * 32);  // the warp's first position
    const float tau = head_tau(a.tau, a.s, head, a.err, kKernWango);
    const float c = tau * kLog2e;
    __nv_bfloat16* prow = a.P + ((size_t)(bb * a.H + head) * a.T_pad + pi) * a.ldp;
    uint64_t dsum2[2] = {0, 0};
    // z = the column sums of Fk over the blocks below the window (jb < jlo), for the
    // older-prefix denominator Fq_i . z
    {
      const int t = threadIdx.x - kPWeightWarp0 * 32;
      if (t < a.d_h) {
        const float* zr = a.zb + ((size_t)bb * a.H + head) * a.n_iblk * a.d_h + t;
        float zs = 0.f;
        for (int j = 0; j < jlo; ++j) zs += zr[(size_t)j * a.d_h];
        b.z[t] = zs;
      }
      named_bar_sync(1, 256);
    }
    bool ok = true;
    uint32_t u = 0;
    for (int jb = ib; ok && jb >= jlo; --jb) {
      const bool mixed = is_mixed(jb, ib, W);
      for (int h = mixed ? 0 : -1; h <= (mixed ? 1 : -1); ++h, ++u) {
        const int slot = u & 1;
        const uint32_t sl = tmem + (uint32_t)(slot * 128) + lane_off;
        if (!(ok = wait_bar(&b.s_full[slot], (u >> 1) & 1, b, a))) break;
        tc_fence_after();
        // One 32-source chunk at a time: two per warpgroup for a whole block, one for a
        // half, whose feature-map scores sit 64 columns after its cos scores.  Each
        // chunk is classified for this warp's 32 rows: after every row (zero weights),
        // inside every row's window (exp only) or general.
        const int nq = h < 0 ? 2 : 1;
#pragma unroll 1
        for (int q = 0; q < nq; ++q) {
          const int off = h < 0 ? wg * 64 + q * 32 : h * 64 + wg * 32;  // first source in the block
          const uint32_t cs = sl + (uint32_t)(h < 0 ? off : wg * 32);     // its cos score column
          // the chunk's positions: j0 that of its first column, js the lowest
          const int j0 = jb * kBlk + (a.mirror ? kBlk - 1 - off : off);
          const int js = a.mirror ? j0 - 31 : j0;
          uint32_t p[16];
          if (js > i0 + 31) {
#pragma unroll
            for (int e = 0; e < 16; ++e) p[e] = 0u;
          } else if (js + 31 <= i0 && js >= i0 + 32 - W) {
            uint32_t rq[32];
            tmem_ld32(cs, rq);
            tmem_ld_wait();
            weights32<0>(rq, rq, c, js, i, 0, p, dsum2);
          } else {  // a whole block has no older sources: its cos scores stand in for f
            uint32_t r[2][32];
            tmem_ld32(cs, r[0]);
            tmem_ld32(h < 0 ? cs : cs + 64, r[1]);
            tmem_ld_wait();
            const int jw = h < 0 ? -0x7fffffff - 1 : i - W + 1;
            if (a.mirror) weights32<2, true>(r[0], r[1], c, j0, i, jw, p, dsum2);
            else weights32<2>(r[0], r[1], c, j0, i, jw, p, dsum2);
          }
          __nv_bfloat16* dst = prow + (ib - jb) * kBlk + off;
#pragma unroll
          for (int e = 0; e < 16; e += 4) st_global_v4(dst + 2 * e, p[e], p[e + 1], p[e + 2], p[e + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.slot_free[slot]);
      }
    }
    // den = row sums of the weights as applied + older prefix + null term
    float d0, d1, d2, d3;
    f32x2_unpack(dsum2[0], d0, d1);
    f32x2_unpack(dsum2[1], d2, d3);
    b.rowsum[wg][row] = (d0 + d1) + (d2 + d3);
    __syncwarp();
    if (lane == 0) mbar_arrive(&b.rs_full);
    if (ok && wg == 0 && (ok = wait_bar(&b.rs_full, 0, b, a))) {
      float den = 1.f;  // rows past T: any finite value
      if (mi < a.T) {
        const float null_w = a.null_bias ? exp2f((a.null_bias[head] - tau) * kLog2e) : 0.f;
        const __nv_bfloat16* f = a.fq + ((size_t)bb * a.T + mi) * a.dqk + (size_t)head * a.d_h;
        float older = 0.f;
        for (int c = 0; c < a.d_h; c += 8) {
          const uint4 w = *reinterpret_cast<const uint4*>(f + c);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            older = fmaf(bf16lo(ww[e]), b.z[c + 2 * e], older);
            older = fmaf(bf16hi(ww[e]), b.z[c + 2 * e + 1], older);
          }
        }
        den = b.rowsum[0][row] + b.rowsum[1][row] + older + (float)(i + 1) * null_w;
      }
      a.den[(size_t)(bb * a.H + head) * a.T_pad + pi] = den;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ================================================================= gate-strip kernel

constexpr int kGThreads = 256;  // warp 0 TMA, warp 1 MMA (and TMEM), warps 4-7 epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kPStages = 3;                 // P ring: 128 destinations x 64 sources per stage
constexpr uint32_t kPBox = kBlk * 64 * 2;   // 16 KB
constexpr int kGSlots = 3;                  // G tiles (128 sources x 128 columns) kept in place
constexpr int kGSlotsMax = kGSlots + 1;     // with v fused: the v staging tile is a fourth slot
constexpr uint32_t kColO = 0, kColSt = 256; // O double buffer [0, 256); S^T
constexpr uint32_t kColV = 384;             // fused v: the v tile x W_v^T, [384, 512)

struct __align__(8) GBars {
  uint64_t pfull[kPStages], pempty[kPStages];
  uint64_t gfull[kGSlotsMax], gempty[kGSlotsMax];
  uint64_t fk_full, fk_empty;  // Fk of the block's leaving source block
  uint64_t fq_full, fq_empty;  // Fq of the destination block (the read-out)
  uint64_t o_full[2], o_empty[2];
  uint64_t st_full;            // the block's read-out and state update are complete
  uint64_t sb_full;            // bf16 state copy in place for the next read-out
  uint64_t v_full;             // the destination block's v in the staging tile
  uint64_t vacc_full, vacc_empty;  // fused v: the v tile in TMEM / read out of it
  uint64_t drain, never;
  uint32_t tmem_base;
  int abort;
};
// smem: P stages | G slots | Fk | Fq | S_bf16 | U staging | Bars
constexpr size_t kGSmemBytes =
    1024 + kPStages * kPBox + kGSlots * kGStage + 3 * kTile + kGStage + sizeof(GBars);
static_assert(kGSmemBytes <= 232448, "shared memory budget");

struct GArgs {
  int B, T, T_pad, H, dqk, m, d_h, m_h, W;  // m: row width in memory, m_h: gates per head
  int m_hp;                                 // per-head pitch (m / H)
  int n_iblk, n_ntile, n_strips;
  int nseg, seg_len, n_items;  // each strip's destination blocks in nseg segments
  int reuse;                   // every destination block has at most kGSlots source blocks
  float* seg_state;            // [n_strips, nseg - 1, kNg, d_h] f32 state at segment ends
  int* seg_flag;               // [n_strips, nseg - 1], 0 until that state is written
  const float* den;            // [B * H, T_pad]
  const __nv_bfloat16* v;      // may be NULL (then u = gbar)
  __nv_bfloat16* out;
  unsigned* err;
  uint64_t timeout_ns;
  int debug_timeout;
  int no_norm;                 // the numerator alone: no division by the denominator
  int mirror;                  // the time-reversed problem (mem_row)
  int fuse;                    // v = x W_v^T computed here (v == NULL, reuse == 0)
  __nv_bfloat16* gbar_out;     // if set: gbar (bf16), laid out as out
  int nkc;                     // fused v: 64-column chunks of the residual width d
};

struct Strip {
  int b, head, n0;
};
// A work item: destination blocks [ib0, ib1) of one strip, segment `seg` of nseg.
// Items are numbered segment-major, so every strip's segment k comes before any
// segment k + 1.  A segment that ends with a non-empty state hands it (f32) to the
// next segment through global memory and a per-strip flag.
struct Item {
  int st, seg, ib0, ib1;
};
template <bool kSeg>
__device__ __forceinline__ Item item_of(const GArgs& a, int w) {
  Item it;
  if (kSeg) {
    it.seg = w / a.n_strips;
    it.st = w % a.n_strips;
    it.ib0 = it.seg * a.seg_len;
    it.ib1 = min(a.n_iblk, it.ib0 + a.seg_len);
  } else {  // one segment per strip
    it.seg = 0;
    it.st = w;
    it.ib0 = 0;
    it.ib1 = a.n_iblk;
  }
  return it;
}
__device__ __forceinline__ Strip strip_of(const GArgs& a, int s) {
  Strip r;
  r.n0 = (s % a.n_ntile) * kNg;
  r.head = (s / a.n_ntile) % a.H;
  r.b = s / (a.n_ntile * a.H);
  return r;
}

// Waits, bounded, until another CTA of this launch sets *flag (acquire).
__device__ __forceinline__ bool wait_flag(const int* flag, const GArgs& a) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(flag) == 0) {
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      record_error(a.err, kErrTimeout | kKernWango);
      return false;
    }
  }
  return true;
}

// Segment handoff, run once per work item (kept out of line: the hot loops stay small).
// The previous segment's state, one thread's gate column of d_h f32 at src, into TMEM
// at t_st (for the updates) and as bf16 into shared memory at s_sb (for the read-out).
// Called by all four epilogue warps; returns false (for all of them) if the wait for
// the previous segment timed out.
template <int DH>
__device__ __noinline__ bool import_state(const GArgs& a, size_t slot, uint32_t t_st, uint32_t s_sb, int row,
                                          uint64_t* sb_full, int lane, bool issuer) {
  constexpr int RB = DH * 2;
  bool ok = true;
  if (issuer) ok = wait_flag(&a.seg_flag[slot], a);
  if (!named_bar_and(2, 128, ok)) return false;
  const float* src = a.seg_state + (slot * kNg + row) * DH;
#pragma unroll 1
  for (int c0 = 0; c0 < DH; c0 += 16) {
    uint32_t t16[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 x = ld_global_cg_v4(src + c0 + 4 * q);
      t16[4 * q] = x.x; t16[4 * q + 1] = x.y; t16[4 * q + 2] = x.z; t16[4 * q + 3] = x.w;
    }
    tmem_st16(t_st + c0, t16);
#pragma unroll
    for (int c = 0; c < 16; c += 8) {
      const uint4 o = make_uint4(pack_bf16x2(__uint_as_float(t16[c]), __uint_as_float(t16[c + 1])),
                                 pack_bf16x2(__uint_as_float(t16[c + 2]), __uint_as_float(t16[c + 3])),
                                 pack_bf16x2(__uint_as_float(t16[c + 4]), __uint_as_float(t16[c + 5])),
                                 pack_bf16x2(__uint_as_float(t16[c + 6]), __uint_as_float(t16[c + 7])));
      st_shared_v4(s_sb + swz<RB>(row, c0 + c), o);
    }
  }
  tmem_st_wait();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(sb_full);
  return true;
}
// This segment's final state (one thread's gate column, TMEM at t_st) to global
// memory, then the flag for the next segment.  Called by all four epilogue warps.
template <int DH>
__device__ __noinline__ void export_state(const GArgs& a, size_t slot, uint32_t t_st, int row, bool issuer) {
  float* dst = a.seg_state + (slot * kNg + row) * DH;
  tc_fence_after();
#pragma unroll 1
  for (int c0 = 0; c0 < DH; c0 += 16) {
    uint32_t t16[16];
    tmem_ld16(t_st + c0, t16);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_global_v4(dst + c0 + 4 * q, t16[4 * q], t16[4 * q + 1], t16[4 * q + 2], t16[4 * q + 3]);
  }
  __threadfence();
  named_bar_sync(2, 128);  // every epilogue thread has written and fenced its part
  if (issuer) st_release_gpu(&a.seg_flag[slot], 1);
}

// Schedule of one destination block ib in the gate-strip kernel, followed identically
// by the TMA and MMA threads:
//  - at its start, the read-out O = Fq S_bf16 of the state before the block (the first
//    MMA into O), then the update S^T += G^T Fk of its leaving source block jlo (if
//    jlo(ib + 1) > jlo), then P.G over the source blocks oldest first, jlo .. ib;
//  - G tiles stay in kGSlots slots (tile jb in slot jb % kGSlots) for as long as later
//    blocks of the same work item need them, when every block has at most kGSlots
//    source blocks ("reuse"); a block then loads only its newest tile, prefetched
//    during the previous block.  Otherwise every use loads its tile into the next slot.
//  - the next block's Fq and Fk are prefetched after the P stages of this block's
//    source block prefetch_pos, and (reuse) its newest G tile after this block's last
//    P stages.
__device__ __forceinline__ int prefetch_pos(int ib, int W) { return ib - jlo_of(ib, W) >= 1 ? 1 : 0; }
__device__ __forceinline__ bool has_leaving(int ib, int W) { return jlo_of(ib + 1, W) > jlo_of(ib, W); }

// Roles: warp 0 TMA; warp 1 one thread issuing the MMAs; warps 4-7 the epilogue (one
// destination row per thread).
template <int DH, bool kSeg>
__global__ void __launch_bounds__(kGThreads, 1)
    wango_g_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmG,
                   const __grid_constant__ CUtensorMap tmFQ, const __grid_constant__ CUtensorMap tmFK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmU,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWv, const GArgs a) {
  constexpr int RB = DH * 2;
  constexpr uint32_t lay = DH == 64 ? kSwizzle128B : DH == 32 ? kSwizzle64B : kSwizzle32B;
  constexpr uint32_t sbo = 8u * RB;
  constexpr uint32_t tile_bytes = kBlk * RB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sP = base;                          // P stages
  uint8_t* sG = sP + kPStages * kPBox;         // G slots
  uint8_t* sFK = sG + kGSlots * kGStage;
  uint8_t* sFQ = sFK + kTile;
  uint8_t* sSB = sFQ + kTile;                  // bf16 state, [128 gate rows x d_h]
  uint8_t* sU = sSB + kTile;                   // v of the destination block, overwritten by u
  GBars& b = *reinterpret_cast<GBars*>(sU + kGStage);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int W = a.W;
  const bool reuse = a.reuse != 0;
  const bool fuse = a.fuse != 0;
  // G slots: three in place; with v fused, the v staging tile (unused then) is a fourth
  const int nslots = fuse ? kGSlotsMax : kGSlots;
  auto slot_ptr = [&](int s) -> uint8_t* { return s < kGSlots ? sG + s * kGStage : sU; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&b.pfull[s], 1);
      mbar_init(&b.pempty[s], 1);
    }
    for (int s = 0; s < kGSlotsMax; ++s) {
      mbar_init(&b.gfull[s], 1);
      mbar_init(&b.gempty[s], 1);
    }
    mbar_init(&b.vacc_full, 1);
    mbar_init(&b.vacc_empty, 4);
    mbar_init(&b.fk_full, 1);
    mbar_init(&b.fk_empty, 1);
    mbar_init(&b.fq_full, 1);
    mbar_init(&b.fq_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&b.o_full[s], 1);
      mbar_init(&b.o_empty[s], 4);
    }
    mbar_init(&b.st_full, 1);
    mbar_init(&b.sb_full, 4);
    mbar_init(&b.v_full, 1);
    mbar_init(&b.drain, 1);
    mbar_init(&b.never, 1);
    b.abort = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(&b.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    Ring pr;
    bool ok = true;
    uint32_t gload[kGSlotsMax] = {}, fq_n = 0, fk_n = 0;  // loads issued (slot phases)
    uint32_t pmask = 0, pph[kPStages] = {};
    int gseq = 0;  // slot counter when tiles are not kept
    Strip sp = {};
    int gx = 0, pz = 0;
    auto load_g = [&](int jb) -> bool {
      const int s = reuse ? jb % kGSlots : (gseq++ % nslots);
      if (!wait_bar(&b.gempty[s], (gload[s] & 1) ^ 1, b, a)) return false;
      ++gload[s];
      uint8_t* dst = slot_ptr(s);
      mbar_arrive_expect_tx(&b.gfull[s], kGStage);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_3d(dst + h * 2 * kGBox + c * kGBox, &tmG, &b.gfull[s], gx + 64 * c,
                      mem_row(jb, a.n_iblk, a.mirror) + 64 * h, sp.b);
      return true;
    };
    // fused v: chunk kc of the block's x rows (128 x 64) and of the strip's W_v rows
    // (128 gate columns x 64), together in the next slot
    auto load_xw = [&](int ib, int kc) -> bool {
      const int s = gseq++ % nslots;
      if (!wait_bar(&b.gempty[s], (gload[s] & 1) ^ 1, b, a)) return false;
      ++gload[s];
      uint8_t* dst = slot_ptr(s);
      mbar_arrive_expect_tx(&b.gfull[s], kGStage);
      tma_load_3d(dst, &tmX, &b.gfull[s], kc * 64, mem_row(ib, a.n_iblk, a.mirror), sp.b);
      tma_load_2d(dst + 2 * kGBox, &tmWv, &b.gfull[s], kc * 64, gx);
      return true;
    };
    auto load_fq = [&](int ib) -> bool {
      if (!wait_bar(&b.fq_empty, (fq_n & 1) ^ 1, b, a)) return false;
      ++fq_n;
      mbar_arrive_expect_tx(&b.fq_full, tile_bytes);
      tma_load_3d(sFQ, &tmFQ, &b.fq_full, sp.head * DH, mem_row(ib, a.n_iblk, a.mirror), sp.b);
      return true;
    };
    auto load_fk = [&](int jb) -> bool {
      if (!wait_bar(&b.fk_empty, (fk_n & 1) ^ 1, b, a)) return false;
      ++fk_n;
      mbar_arrive_expect_tx(&b.fk_full, tile_bytes);
      tma_load_3d(sFK, &tmFK, &b.fk_full, sp.head * DH, mem_row(jb, a.n_iblk, a.mirror), sp.b);
      return true;
    };
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      if (it.ib0 >= it.ib1) continue;
      sp = strip_of(a, it.st);
      gx = sp.head * a.m_hp + sp.n0;
      pz = sp.b * a.H + sp.head;
      // the first block's read-out and update operands
      if (!(ok = load_fq(it.ib0))) break;
      if (has_leaving(it.ib0, W) && !(ok = load_fk(jlo_of(it.ib0, W)))) break;
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib) {
        const int jlo = jlo_of(ib, W), ppos = prefetch_pos(ib, W);
        // the next block's v into L2 ahead of its load: the epilogue loads it only once
        // this block's u has left the staging tile, and would otherwise wait out the HBM
        // latency there.  (The same prefetch of the G tile two blocks ahead was slower:
        // that tile's load already overlaps two blocks of MMAs.)
        if (a.v && ib + 1 < it.ib1) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_prefetch_l2_3d(&tmV, gx + 64 * c, mem_row(ib + 1, a.n_iblk, a.mirror) + 64 * h, sp.b);
        }
        for (int jb = jlo; ok && jb <= ib; ++jb) {
          if ((!reuse || ib == it.ib0) && !(ok = load_g(jb))) break;
          for (int hh = 0; hh < 2; ++hh) {
            if (!(ok = wait_bar(&b.pempty[pr.stage], pr.phase ^ 1, b, a))) break;
            mbar_arrive_expect_tx(&b.pfull[pr.stage], kPBox);
            tma_load_3d(sP + pr.stage * kPBox, &tmP, &b.pfull[pr.stage], (ib - jb) * kBlk + 64 * hh, ib * kBlk,
                        pz);
            pmask |= 1u << pr.stage;
            pph[pr.stage] = pr.phase;
            pr.next(kPStages);
          }
          if (ok && jb - jlo == ppos && ib + 1 < it.ib1) {  // the next block's read-out and update
            if (!(ok = load_fq(ib + 1))) break;
            if (has_leaving(ib + 1, W) && !(ok = load_fk(jlo_of(ib + 1, W)))) break;
          }
          // the next block's newest G tile, behind this block's P loads (a tile from HBM
          // would hold up the P loads queued after it)
          if (ok && jb == ib && reuse && ib + 1 < it.ib1 && !(ok = load_g(ib + 1))) break;
        }
        for (int kc = 0; ok && fuse && kc < a.nkc; ++kc) ok = load_xw(ib, kc);
      }
    }
    // no copy may be in flight when the CTA exits
    if (fq_n) mbar_wait(&b.fq_full, (fq_n - 1) & 1, a.timeout_ns);
    if (fk_n) mbar_wait(&b.fk_full, (fk_n - 1) & 1, a.timeout_ns);
    for (int s = 0; s < nslots; ++s)
      if (gload[s]) mbar_wait(&b.gfull[s], (gload[s] - 1) & 1, a.timeout_ns);
    for (int s = 0; s < kPStages; ++s)
      if (pmask & (1u << s)) mbar_wait(&b.pfull[s], pph[s], a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idesc_o = idesc_bf16_f32(kBlk, kNg, false, true);   // O += P G
    constexpr uint32_t idesc_r = idesc_bf16_f32(kBlk, kNg, false, false);  // O += Fq S
    constexpr uint32_t idesc_u = idesc_bf16_f32(kBlk, DH, true, true);     // S^T += G^T Fk
    const uint64_t fqd = smem_desc(smem_u32(sFQ), 16, sbo, lay);
    const uint64_t fkmn = smem_desc(smem_u32(sFK), tile_bytes, sbo, lay);  // Fk as MN-major B
    const uint64_t sbd = smem_desc(smem_u32(sSB), 16, sbo, lay);
    bool ok = true;
    if (a.debug_timeout) ok = wait_bar(&b.never, 0, b, a);  // nothing ever arrives here
    Ring pr;
    constexpr uint32_t idesc_v = idesc_bf16_f32(kBlk, kNg, false, false);  // V = X W_v^T
    uint32_t guse[kGSlotsMax] = {}, sbph = 0, fkph = 0, fqph = 0;
    int gseq = 0, dc = 0;
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      // a later segment starts from the state its predecessor handed over
      bool first_update = !(kSeg && it.seg > 0 && jlo_of(it.ib0, W) > 0);
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++dc) {
        const int ob = dc & 1;
        const int jlo = jlo_of(ib, W);
        const bool leave = has_leaving(ib, W);
        if (!(ok = wait_bar(&b.o_empty[ob], ((dc >> 1) & 1) ^ 1, b, a))) break;
        // read-out of the state before this block: O = Fq S_bf16
        if (!(ok = wait_bar(&b.sb_full, sbph, b, a))) break;
        sbph ^= 1;
        if (!(ok = wait_bar(&b.fq_full, fqph, b, a))) break;
        fqph ^= 1;
        tc_fence_after_nc();
        const uint32_t od = tmem + kColO + (uint32_t)(ob * kNg);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk)
          mma_bf16_ss_nc(od, fqd + (uint64_t)(kk * 2), sbd + (uint64_t)(kk * 2), idesc_r, kk != 0 ? 1u : 0u);
        mma_commit_nc(&b.fq_empty);
        // G tile of source block jb: its slot, waiting for the load when this is the use
        // it was loaded for
        int cur_slot = -1, cur_jb = -1;
        auto tile = [&](int jb) -> int {
          if (jb == cur_jb) return cur_slot;
          const bool loaded_now = !reuse || ib == it.ib0 || jb == ib;
          const int s = reuse ? jb % kGSlots : (gseq++ % nslots);
          if (loaded_now) {
            if (!(ok = wait_bar(&b.gfull[s], guse[s] & 1, b, a))) return -1;
            ++guse[s];
            tc_fence_after_nc();
          }
          cur_jb = jb;
          cur_slot = s;
          return s;
        };
        // the leaving block enters the state: S^T += G^T Fk (after the read-out copy)
        if (leave) {
          const int s = tile(jlo);
          if (s < 0) break;
          if (!(ok = wait_bar(&b.fk_full, fkph, b, a))) break;
          fkph ^= 1;
          tc_fence_after_nc();
          const uint32_t gaddr = smem_u32(slot_ptr(s));
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint64_t gd = smem_desc(gaddr + hh * 2 * kGBox, kGBox, 1024, kSwizzle128B);
            const uint64_t fh = fkmn + (uint64_t)((64 * hh * RB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss_nc(tmem + kColSt, gd + (uint64_t)(kk * 128), fh + (uint64_t)((kk * 16 * RB) >> 4),
                             idesc_u, (first_update && hh == 0 && kk == 0) ? 0u : 1u);
          }
          first_update = false;
          mma_commit_nc(&b.fk_empty);
        }
        mma_commit_nc(&b.st_full);
        // O += P G over the source blocks, oldest first
        for (int jb = jlo; ok && jb <= ib; ++jb) {
          const int s = tile(jb);
          if (s < 0) break;
          const uint32_t gaddr = smem_u32(slot_ptr(s));
          for (int hh = 0; hh < 2; ++hh) {
            if (!(ok = wait_bar(&b.pfull[pr.stage], pr.phase, b, a))) break;
            tc_fence_after_nc();
            const uint64_t pd = smem_desc(smem_u32(sP + pr.stage * kPBox), 16, 1024, kSwizzle128B);   // K-major
            const uint64_t gd = smem_desc(gaddr + hh * 2 * kGBox, kGBox, 1024, kSwizzle128B);         // MN-major
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss_nc(od, pd + (uint64_t)(kk * 2), gd + (uint64_t)(kk * 128), idesc_o, 1u);
            mma_commit_nc(&b.pempty[pr.stage]);
            pr.next(kPStages);
          }
          if (!ok) break;
          // release the tile after its last use in this work item
          if (!reuse || ib + 1 == it.ib1 || jb < jlo_of(ib + 1, W)) mma_commit_nc(&b.gempty[s]);
        }
        if (!ok) break;
        // fused v: V = X W_v^T over the residual width (after this block's P G, so that
        // the wait for the epilogue to read the previous block's V overlaps those MMAs)
        if (ok && fuse) {
          if (!(ok = wait_bar(&b.vacc_empty, (dc & 1) ^ 1, b, a))) break;
          for (int kc = 0; ok && kc < a.nkc; ++kc) {
            const int s = gseq++ % nslots;
            if (!(ok = wait_bar(&b.gfull[s], guse[s] & 1, b, a))) break;
            ++guse[s];
            tc_fence_after_nc();
            const uint32_t xa = smem_u32(slot_ptr(s)), wa = xa + 2 * kGBox;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss_nc(tmem + kColV, smem_desc(xa + kk * 32, 16, 1024, kSwizzle128B),
                             smem_desc(wa + kk * 32, 16, 1024, kSwizzle128B), idesc_v, (kc | kk) != 0 ? 1u : 0u);
            mma_commit_nc(&b.gempty[s]);
          }
          if (!ok) break;
          mma_commit_nc(&b.vacc_full);
        }
        mma_commit_nc(&b.o_full[ob]);
      }
    }
    mma_commit(&b.drain);
    mbar_wait(&b.drain, 0, a.timeout_ns);
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------ epilogue + state copy
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // destination row; also the gate column of S^T
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool issuer = (warp == kEpiWarp0 && lane == 0);
    bool ok = true;
    int gib = 0;
    // bf16 copy of the state for a destination block's read-out (zero while no source
    // has left the window)
    auto copy_state = [&](bool empty) {
#pragma unroll
      for (int c0 = 0; c0 < DH; c0 += 16) {
        uint32_t t16[16];
        if (!empty) {
          tmem_ld16(tmem + kColSt + lane_off + c0, t16);
          tmem_ld_wait();
        }
#pragma unroll
        for (int c = 0; c < 16; c += 8) {
          uint4 o = make_uint4(0, 0, 0, 0);
          if (!empty) {
            o.x = pack_bf16x2(__uint_as_float(t16[c]), __uint_as_float(t16[c + 1]));
            o.y = pack_bf16x2(__uint_as_float(t16[c + 2]), __uint_as_float(t16[c + 3]));
            o.z = pack_bf16x2(__uint_as_float(t16[c + 4]), __uint_as_float(t16[c + 5]));
            o.w = pack_bf16x2(__uint_as_float(t16[c + 6]), __uint_as_float(t16[c + 7]));
          }
          st_shared_v4(smem_u32(sSB) + swz<RB>(row, c0 + c), o);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.sb_full);
    };
    // the destination block's v (128 rows x 128 columns) into the staging tile, once
    // the previous u store has read it; issued by one thread
    uint32_t v_n = 0;
    auto load_v = [&](const Strip& sp, int ib) {
      bulk_wait_group_read0();
      mbar_arrive_expect_tx(&b.v_full, kGStage);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sU + h * 2 * kGBox + c * kGBox, &tmV, &b.v_full, sp.head * a.m_hp + sp.n0 + 64 * c,
                      mem_row(ib, a.n_iblk, a.mirror) + 64 * h, sp.b);
    };
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      if (it.ib0 >= it.ib1) continue;
      const Strip sp = strip_of(a, it.st);
      if (issuer && a.v && !fuse) load_v(sp, it.ib0);
      // the state before the first destination block: empty, or the previous
      // segment's (into TMEM for the updates, bf16 into shared memory for the read-out)
      if (kSeg && it.seg > 0 && jlo_of(it.ib0, W) > 0) {
        if (!import_state<DH>(a, (size_t)it.st * (a.nseg - 1) + (it.seg - 1), tmem + kColSt + lane_off,
                              smem_u32(sSB), row, &b.sb_full, lane, issuer))
          break;
      } else {
        copy_state(true);
      }
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++gib) {
        const int ob = gib & 1;
        const int i = ib * kBlk + row;                          // this row of den
        const int mi = mem_row(ib, a.n_iblk, a.mirror) + row;   // its row in memory
        const bool row_ok = mi < a.T;
        const float den = a.den[(size_t)(sp.b * a.H + sp.head) * a.T_pad + i];
        const size_t grow = ((size_t)sp.b * a.T + (row_ok ? mi : 0)) * a.m + (size_t)sp.head * a.m_hp;
        // the state after this block's update, for the next block's read-out (this
        // block's read-out and update are complete; the next block changes it only after
        // its own read-out)
        if (ok) ok = wait_bar(&b.st_full, gib & 1, b, a);
        ok = named_bar_and(2, 128, ok);
        if (!ok) break;
        tc_fence_after();
        if (ib + 1 < it.ib1) copy_state(jlo_of(ib + 1, W) == 0);
        if (ok) ok = wait_bar(&b.o_full[ob], (gib >> 1) & 1, b, a);
        if (ok && a.v) ok = wait_bar(&b.v_full, v_n & 1, b, a);
        if (ok && fuse) ok = wait_bar(&b.vacc_full, gib & 1, b, a);
        ok = named_bar_and(2, 128, ok);
        if (!ok) break;
        if (a.v) ++v_n;
        tc_fence_after();
        const float inv = a.no_norm ? 1.f : 1.f / den;
        // gbar = O / den, rounded to bf16, in registers; the accumulator is released as
        // soon as it has been read
        uint32_t gb[kNg / 2];
#pragma unroll
        for (int c0 = 0; c0 < kNg; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + kColO + (uint32_t)(ob * kNg) + lane_off + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            gb[(c0 + e) / 2] = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.o_empty[ob]);
        if (a.gbar_out && row_ok) {
#pragma unroll
          for (int k = 0; k < kNg / 8; ++k)
            if (sp.n0 + 8 * k < a.m_h)
              st_global_v4(a.gbar_out + grow + sp.n0 + 8 * k, gb[4 * k], gb[4 * k + 1], gb[4 * k + 2], gb[4 * k + 3]);
        }
        if (fuse) {
          // v of this row in bf16 (as a separate projection would have stored it), u = gbar
          // * v, and the row written straight from registers (the staging tile is a G slot)
#pragma unroll
          for (int c0 = 0; c0 < kNg; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + kColV + lane_off + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              gb[(c0 + e) / 2] = mul_bf16x2(gb[(c0 + e) / 2],
                                            pack_bf16x2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&b.vacc_empty);
          if (row_ok) {
#pragma unroll
            for (int k = 0; k < kNg / 8; ++k) {
              const int col = sp.n0 + 8 * k;
              if (col < a.m_h)
                st_global_v4(a.out + grow + col, gb[4 * k], gb[4 * k + 1], gb[4 * k + 2], gb[4 * k + 3]);
            }
          }
          continue;
        }
        if (!a.v) {  // without v the tile is written from scratch: the previous store must have read it
          if (issuer) bulk_wait_group_read0();
          named_bar_sync(2, 128);
        }
        // u = gbar * v, written over v in the staging tile (each thread its own row)
        const int rh = row >> 6, rr = row & 63;
#pragma unroll
        for (int cq = 0; cq < 2; ++cq) {
          const int col0 = sp.n0 + cq * 64;
          const bool straddle = col0 < a.m_h && col0 + 64 > a.m_h;
          const uint32_t box = smem_u32(sU) + rh * 2 * kGBox + cq * kGBox + rr * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t addr = box + (uint32_t)((k ^ (rr & 7)) << 4);
            const uint32_t* g4 = &gb[cq * 32 + k * 4];
            uint32_t u[4];
            if (a.v) {
              const uint4 vv = ld_shared_v4(addr);
              u[0] = mul_bf16x2(g4[0], vv.x);
              u[1] = mul_bf16x2(g4[1], vv.y);
              u[2] = mul_bf16x2(g4[2], vv.z);
              u[3] = mul_bf16x2(g4[3], vv.w);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) u[e] = g4[e];
            }
            if (!straddle) st_shared_v4(addr, make_uint4(u[0], u[1], u[2], u[3]));
            else if (row_ok && col0 + 8 * k < a.m_h) st_global_v4(a.out + grow + col0 + 8 * k, u[0], u[1], u[2], u[3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (issuer) {
          for (int h = 0; h < 2; ++h) {
            const int y = mem_row(ib, a.n_iblk, a.mirror) + 64 * h;
            if (y >= a.T) continue;
            for (int cq = 0; cq < 2; ++cq) {
              const int c = sp.n0 + cq * 64;
              if (c + 64 > a.m_h) continue;
              tma_store_3d(&tmU, sU + h * 2 * kGBox + cq * kGBox, sp.head * a.m_hp + c, y, sp.b);
            }
          }
          bulk_commit_group();
          if (a.v && ib + 1 < it.ib1) load_v(sp, ib + 1);  // the next block's v, once the store has read u
        }
      }
      // hand this segment's final state to the next segment of the strip (the last
      // block's update is complete: its st_full was waited for above)
      if (kSeg && ok && it.seg + 1 < a.nseg && jlo_of(it.ib1, W) > 0)
        export_state<DH>(a, (size_t)it.st * (a.nseg - 1) + it.seg, tmem + kColSt + lane_off, row, issuer);
    }
    if (issuer) bulk_wait_group0();  // every store has completed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
// ---------------------------------------------------------------- pre-pass

// Feature map of eq. 8 (mode 0) or plain ELU + 1 (mode 1).  For u <= 0,
// ELU(u) + 1 = e^u exactly, so only the exponential is evaluated.
__device__ __forceinline__ float phi_fast(float u, float inv_sqrt_dh, int mode) {
  const float e1 = u > 0.f ? u + 1.f : ex2_approx(u * kLog2e);
  if (mode == 1) return e1;
  return fmaxf(e1 + 1e-4f, 1e-4f) * inv_sqrt_dh;
}

// Per (source block jb, head a, batch b), one thread per row of the block:
// Fq = e^-tau phi(sqrt(tau) qhat) and Fk = phi(sqrt(tau) khat) in bf16, and
// zb[b, a, jb, c] = the sum over the block's valid rows of Fk[., a d_h + c] as rounded to
// bf16 (the values the state update multiplies).
__global__ void __launch_bounds__(kBlk) wango_phi_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                                        __nv_bfloat16* fq, __nv_bfloat16* fk, float* zb, int T,
                                                        int H, int dqk, int n_iblk, float s, const float* tau,
                                                        int phi_mode, unsigned* err, int mirror) {
  __shared__ float part[kBlk / 32][64];
  const int jb = blockIdx.x, a = blockIdx.y, bb = blockIdx.z;
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  const int d_h = dqk / H, i = jb * kBlk + t;
  const float tt = head_tau(tau, s, a, err, kKernWango);
  const float sq = sqrtf(tt), shift = exp2f(-tt * kLog2e), inv_sqrt_dh = rsqrtf((float)d_h);
  float fkv[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) fkv[c] = 0.f;
  if (i < T) {
    const size_t off = ((size_t)bb * T + i) * dqk + (size_t)a * d_h;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 8) {
      if (c0 >= d_h) break;
      const uint4 qv = *reinterpret_cast<const uint4*>(q + off + c0);
      const uint4 kv = *reinterpret_cast<const uint4*>(k + off + c0);
      const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
      uint32_t fo[4], ko[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        fo[e] = pack_bf16x2(shift * phi_fast(sq * bf16lo(qw[e]), inv_sqrt_dh, phi_mode),
                            shift * phi_fast(sq * bf16hi(qw[e]), inv_sqrt_dh, phi_mode));
        ko[e] = pack_bf16x2(phi_fast(sq * bf16lo(kw[e]), inv_sqrt_dh, phi_mode),
                            phi_fast(sq * bf16hi(kw[e]), inv_sqrt_dh, phi_mode));
        fkv[c0 + 2 * e] = bf16lo(ko[e]);
        fkv[c0 + 2 * e + 1] = bf16hi(ko[e]);
      }
      *reinterpret_cast<uint4*>(fq + off + c0) = make_uint4(fo[0], fo[1], fo[2], fo[3]);
      *reinterpret_cast<uint4*>(fk + off + c0) = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    }
  }
  // column sums over the block's rows: across each warp, then across the four warps
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    if (c >= d_h) break;
    float v = fkv[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) part[wp][c] = v;
  }
  __syncthreads();
  if (t < d_h)
    zb[(((size_t)bb * H + a) * n_iblk + (mirror ? n_iblk - 1 - jb : jb)) * d_h + t] =
        (part[0][t] + part[1][t]) + (part[2][t] + part[3][t]);
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// Segments per strip: the count that minimises the estimated makespan on `sms`
// persistent CTAs, a destination block costing 1.  Segment k + 1 of a strip waits for
// segment k to finish; items run segment-major, so with more than one round the
// wait is normally over before it starts.
int choose_nseg(long long strips, int n_iblk, int W, int sms) {
  (void)W;
  int best = 1;
  double best_cost = 0.0;
  for (int nseg = 1; nseg <= 4 && nseg <= n_iblk; ++nseg) {
    const int len = (n_iblk + nseg - 1) / nseg;
    const long long items = strips * nseg;
    const long long rounds = (items + sms - 1) / sms;
    // a segment cannot start before its predecessor ends: at least nseg rounds
    const double cost = (double)(rounds > nseg ? rounds : nseg) * len;
    if (nseg == 1 || cost < 0.95 * best_cost) {  // more segments only for a clear gain
      best = nseg;
      best_cost = cost;
    }
  }
  return best;
}

// Source blocks per destination block at most: the width of P in 128-source blocks.
int max_sources(int n_iblk, int W) {
  int n = 1;
  for (int ib = 0; ib < n_iblk; ++ib) n = std::max(n, ib - jlo_of(ib, W) + 1);
  return n;
}

struct AuxLayout {
  size_t fq, fk, zb, P, den, seg, flag, total;
  int nseg, T_pad, ldp;
};
AuxLayout aux_layout(int B, int T, int H, int dqk, int m, int W) {
  const size_t BT = (size_t)B * T;
  const int nI = (T + kBlk - 1) / kBlk;
  const int d_h = dqk / H;
  const long long strips = (long long)B * H * ((m / H + kNg - 1) / kNg);
  AuxLayout L;
  L.T_pad = nI * kBlk;
  L.ldp = max_sources(nI, W) * kBlk;
  L.nseg = choose_nseg(strips, nI, W, num_sms());
  const size_t handoffs = (size_t)strips * (L.nseg - 1);
  L.fq = 0;
  L.fk = L.fq + a256(BT * dqk * 2);
  L.zb = L.fk + a256(BT * dqk * 2);
  L.P = L.zb + a256((size_t)B * H * nI * d_h * 4);
  L.den = L.P + a256((size_t)B * H * L.T_pad * L.ldp * 2);
  L.seg = L.den + a256((size_t)B * H * L.T_pad * 4);
  L.flag = L.seg + a256(handoffs * kNg * d_h * 4);
  L.total = L.flag + a256(handoffs * 4);
  return L;
}

template <int DH>
cudaError_t launch_p(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mfq, const CUtensorMap& mfk,
                     const PArgs& a, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(wango_p_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kPSmemBytes);
  if (e != cudaSuccess) return e;
  wango_p_kernel<DH><<<dim3(a.n_iblk, a.H, a.B), kPThreads, kPSmemBytes, s>>>(mq, mk, mfq, mfk, a);
  return cudaGetLastError();
}

// The segmented kernel waits (bounded) for states that other CTAs of the same launch
// hand over, so all its CTAs must be resident at once: it is launched cooperatively,
// which the driver either schedules with every CTA resident or refuses.  When it is
// refused (fewer SMs available than the grid, e.g. under SM partitioning), the strips
// run unsegmented, which has no waits between CTAs.
template <int DH>
cudaError_t launch_g(const CUtensorMap& mp, const CUtensorMap& mg, const CUtensorMap& mfq, const CUtensorMap& mfk,
                     const CUtensorMap& mv, const CUtensorMap& mu, const CUtensorMap& mx, const CUtensorMap& mw, GArgs a,
                     cudaStream_t s) {
  if (a.nseg > 1) {
    auto kern = wango_g_kernel<DH, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.n_items < num_sms() ? a.n_items : num_sms()));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kGSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mp, mg, mfq, mfk, mv, mu, mx, mw, a);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();  // not sticky: clear it and run the strips whole
    a.nseg = 1;
    a.seg_len = a.n_iblk;
    a.n_items = a.n_strips;
  }
  auto kern = wango_g_kernel<DH, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = a.n_items < num_sms() ? a.n_items : num_sms();
  kern<<<grid, kGThreads, kGSmemBytes, s>>>(mp, mg, mfq, mfk, mv, mu, mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

size_t wango_aux_bytes(int B, int T, int H, int dqk, int m, int W) { return aux_layout(B, T, H, dqk, m, W).total; }

const float* wango_den_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W) {
  return reinterpret_cast<const float*>(static_cast<const char*>(aux) + aux_layout(B, T, H, dqk, m, W).den);
}
const void* wango_fq_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W) {
  return static_cast<const char*>(aux) + aux_layout(B, T, H, dqk, m, W).fq;
}
const void* wango_fk_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W) {
  return static_cast<const char*>(aux) + aux_layout(B, T, H, dqk, m, W).fk;
}
const float* wango_zb_in_aux(const void* aux, int B, int T, int H, int dqk, int m, int W) {
  return reinterpret_cast<const float*>(static_cast<const char*>(aux) + aux_layout(B, T, H, dqk, m, W).zb);
}

cudaError_t launch_wango_prepass(const AggArgs& p, cudaStream_t s) {
  const int m_h = p.m_h ? p.m_h : p.m / p.H;
  const int n_iblk = ceil_div(p.T, kBlk);
  const AuxLayout L = aux_layout(p.B, p.T, p.H, p.dqk, p.H * m_h, p.window);
  char* aux = static_cast<char*>(p.aux);
  wango_phi_kernel<<<dim3(n_iblk, p.H, p.B), kBlk, 0, s>>>(
      static_cast<const __nv_bfloat16*>(p.q), static_cast<const __nv_bfloat16*>(p.k),
      reinterpret_cast<__nv_bfloat16*>(aux + L.fq), reinterpret_cast<__nv_bfloat16*>(aux + L.fk),
      reinterpret_cast<float*>(aux + L.zb), p.T, p.H, p.dqk, n_iblk, p.s, p.tau, p.phi_mode, p.err, 0);
  return cudaGetLastError();
}

cudaError_t launch_wango_tc(const AggArgs& p, cudaStream_t s) {
  const int d_h = p.dqk / p.H, m_hp = p.m / p.H, m_h = p.m_h ? p.m_h : m_hp;
  const int n_iblk = ceil_div(p.T, kBlk);
  // the scratch is laid out for the logical gate width (as wango_aux_bytes is asked)
  const AuxLayout L = aux_layout(p.B, p.T, p.H, p.dqk, p.H * m_h, p.window);
  const bool debug = (p.flags & TG_FLAG_DEBUG_TIMEOUT) != 0;
  const uint64_t timeout_ns = debug ? 1000000ull : 2000000000ull;
  char* aux = static_cast<char*>(p.aux);
  __nv_bfloat16* fq = reinterpret_cast<__nv_bfloat16*>(aux + L.fq);
  __nv_bfloat16* fk = reinterpret_cast<__nv_bfloat16*>(aux + L.fk);
  float* zb = reinterpret_cast<float*>(aux + L.zb);
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(aux + L.P);
  float* den = reinterpret_cast<float*>(aux + L.den);
  // mirrored (the time-reversed problem, for the backward's gate gradient): the numerator
  // alone, whose positions past T (the reversed sequence's leading padding) have zero
  // g rows and so add nothing; the denominator terms that count positions are not formed
  if (p.mirror && (!p.no_norm || p.v || p.null_bias || p.fuse_x)) return cudaErrorInvalidValue;

  // pre-pass: feature maps and their per-block column sums
  wango_phi_kernel<<<dim3(n_iblk, p.H, p.B), kBlk, 0, s>>>(
      static_cast<const __nv_bfloat16*>(p.q), static_cast<const __nv_bfloat16*>(p.k), fq, fk, zb, p.T, p.H, p.dqk,
      n_iblk, p.s, p.tau, p.phi_mode, p.err, p.mirror);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap mq, mk, mfq, mfk, mp, mg, mv, mu, mx, mw;
  e = make_tmap_3d(&mq, p.q, p.B, p.T, p.dqk, kBlk, d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mk, p.k, p.B, p.T, p.dqk, kBlk, d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mfq, fq, p.B, p.T, p.dqk, kBlk, d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mfk, fk, p.B, p.T, p.dqk, kBlk, d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mp, P, (uint64_t)p.B * p.H, L.T_pad, L.ldp, kBlk, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mg, p.g, p.B, p.T, p.m, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mv, p.v ? p.v : p.g, p.B, p.T, p.m, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mu, p.out, p.B, p.T, p.m, 64, 64);
  // fused v: x [B, T, d] and W_v [m, d] in 128-row x 64-column boxes
  const bool fuse = p.fuse_x != nullptr;
  if (e == cudaSuccess) e = fuse ? make_tmap_3d(&mx, p.fuse_x, p.B, p.T, p.fuse_d, kBlk, 64) : make_tmap_3d(&mx, p.g, p.B, p.T, p.m, 64, 64);
  if (e == cudaSuccess) e = fuse ? make_tmap_2d(&mw, p.fuse_wv, p.m, p.fuse_d, p.fuse_d, kBlk, 64) : make_tmap_3d(&mw, p.g, p.B, p.T, p.m, 64, 64);
  if (e != cudaSuccess) return e;

  // weights P and the denominators, once per destination block
  PArgs pa = {};
  pa.B = p.B; pa.T = p.T; pa.T_pad = L.T_pad; pa.H = p.H; pa.dqk = p.dqk; pa.d_h = d_h; pa.W = p.window;
  pa.n_iblk = n_iblk; pa.ldp = L.ldp; pa.mirror = p.mirror;
  pa.s = p.s; pa.tau = p.tau; pa.null_bias = p.null_bias; pa.zb = zb; pa.fq = fq;
  pa.P = P; pa.den = den; pa.err = p.err; pa.timeout_ns = timeout_ns;
  e = d_h == 64 ? launch_p<64>(mq, mk, mfq, mfk, pa, s)
                : d_h == 32 ? launch_p<32>(mq, mk, mfq, mfk, pa, s) : launch_p<16>(mq, mk, mfq, mfk, pa, s);
  if (e != cudaSuccess) return e;

  // the gate strips
  GArgs a = {};
  a.B = p.B; a.T = p.T; a.T_pad = L.T_pad; a.H = p.H; a.dqk = p.dqk; a.m = p.m;
  a.d_h = d_h; a.m_h = m_h; a.m_hp = m_hp; a.W = p.window;
  a.n_iblk = n_iblk;
  a.n_ntile = ceil_div(m_h, kNg);
  const long long strips = (long long)p.B * p.H * a.n_ntile;
  if (strips * L.nseg > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_strips = (int)strips;
  a.nseg = L.nseg;
  a.seg_len = ceil_div(n_iblk, a.nseg);
  a.n_items = a.n_strips * a.nseg;
  a.reuse = (L.ldp / kBlk <= kGSlots && !fuse) ? 1 : 0;
  a.fuse = fuse ? 1 : 0;
  a.nkc = fuse ? p.fuse_d / 64 : 0;
  a.seg_state = reinterpret_cast<float*>(aux + L.seg);
  a.seg_flag = reinterpret_cast<int*>(aux + L.flag);
  a.den = den;
  a.v = static_cast<const __nv_bfloat16*>(p.v);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.err = p.err;
  a.debug_timeout = debug ? 1 : 0;
  a.timeout_ns = timeout_ns;
  a.no_norm = p.no_norm;
  a.mirror = p.mirror;
  a.gbar_out = static_cast<__nv_bfloat16*>(p.gbar_out);
  if (a.nseg > 1) {  // no segment's state is ready yet
    e = cudaMemsetAsync(a.seg_flag, 0, (size_t)a.n_strips * (a.nseg - 1) * sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  return d_h == 64 ? launch_g<64>(mp, mg, mfq, mfk, mv, mu, mx, mw, a, s)
                   : d_h == 32 ? launch_g<32>(mp, mg, mfq, mfk, mv, mu, mx, mw, a, s)
                               : launch_g<16>(mp, mg, mfq, mfk, mv, mu, mx, mw, a, s);
}

}  // namespace tg
