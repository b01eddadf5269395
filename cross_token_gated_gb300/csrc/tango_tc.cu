// TANGO full-prefix gate aggregation on the tensor cores (tcgen05), "TANGO:
// Token-Aggregated Nonlinear Gating Operators ...", sec. 2.1 eq. 5 with the
// weights of sec. 2.2 eq. 6:
//   u_i = [ sum_{j<=i} e^{tau (qhat_i.khat_j - 1)} g_j ] / [ sum_{j<=i} e^{...} + (i+1) e^{b-tau} ] * v_i
// per head.  The shift by e^-tau cancels in the ratio; since |cos| <= 1 and
// tau <= 20 every weight lies in [e^-40, 1], so no running maximum is kept.
//
// A tile is 128 destinations x 256 gate columns of one (batch, head); it walks the
// 128-source blocks j = 0..ib (ib = its destination block).  Persistent CTAs, one
// per SM, take "units" round-robin: a unit is the pair of tiles (nI-1-p, p) of one
// (batch, head, gate tile), so every unit costs nI+1 source blocks and the units
// of one gate tile, which share G and khat, run side by side out of L2.
//
//   warp 0       TMA: one ring of 32 KB stages (5 of them) that carries, per tile, G in
//                half blocks of 64 sources x 256 columns and then the tile's v (2 stages).
//   warp 3       TMA: qhat tiles (2 buffers) and khat blocks (2-stage ring), in a thread of
//                their own so that score loads never wait behind the G ring.
//   warps 1, 2   MMA issue, one thread each on two SM sub-partitions (J counts source
//                blocks over all tiles of the CTA):
//                  warp 2: S_J = Qhat Khat_J^T (M=128, N=128, K=d_h) -> the TMEM score
//                          slot, once the softmax warps have read S_{J-1} out of it;
//                  warp 1: O += P_J G_J (M=128, N=256, K=64 x 2), A = P_J from TMEM P
//                          slot J % 2; warp 1 also allocates TMEM.
//                Both keep descriptors in registers and avoid compiler memory barriers.
//   warps 4-11   softmax: warpgroup w takes columns [64w, 64w+64) of every score block;
//                one row per thread from TMEM, exp2(tau log2e (s - 1)) with the causal
//                mask on the diagonal block, rounded to bf16; the ROUNDED weights are
//                summed into the row's denominator.  Once both warpgroups have read
//                S_J the score slot is released for S_{J+1}, and P_J (bf16) goes to P
//                slot J % 2 once the P.G of block J - 2 has completed.  Scores and P
//                thus have slots of their own, so S_{J+1} enters the tensor pipe ahead
//                of P.G(J) instead of behind P.G(J+1).
//   warps 12-15  epilogue: O / den from TMEM in bf16 pairs, times v from shared memory
//                (a bf16x2 product); u is written over v in shared memory, 64 columns at
//                a time, and each row half (two warps) stores its box by TMA as soon as
//                the chunk is done, so the stores overlap the next chunks and each ring
//                stage is freed by its own half.  The softmax warps meanwhile work on the
//                next tile.  (A 64-column box that straddles the end of a head's gate
//                columns is written directly instead.)
// TMEM: O in columns [0, 256), the score slot in [256, 384), P slots (bf16 pairs, 64
// columns each) in [384, 448) and [448, 512).
#include "tg_common.cuh"
#include "tg_ptx.cuh"
#include "tg_tc.h"
#include "tg_tma.h"

namespace tg {
namespace {

using namespace ptx;

constexpr int kBlk = 128;      // destinations per tile; sources per score block
constexpr int kHalf = 64;      // rows per ring stage
constexpr int kNg = 256;       // gate columns per tile
constexpr int kQBufs = 2;
constexpr int kKStages = 2;
constexpr int kGStages = 5;
constexpr int kThreads = 512;  // 16 warps
constexpr int kSoftWarp0 = 4, kEpiWarp0 = 12;
constexpr uint32_t kQKMax = kBlk * 64 * 2;     // 16 KB at d_h = 64
constexpr uint32_t kGBox = kHalf * 64 * 2;     // 8 KB: 64 rows x 64 columns
constexpr uint32_t kGStage = 4 * kGBox;        // 32 KB
constexpr uint32_t kColO = 0, kColS0 = 256, kColP0 = 384;

struct __align__(8) Bars {
  uint64_t q_full[kQBufs], q_empty[kQBufs];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t g_full[kGStages], g_empty[kGStages];
  uint64_t s_full, s_free, p_full[2];
  uint64_t o_full, o_empty, den_full, den_empty;
  uint64_t p_free[2];                            // the P.G of a P slot's block has completed
  uint64_t drain[2], never;
  uint32_t tmem_base;
  int abort;
  float rowsum[2][kBlk];
};

constexpr size_t kSmemBytes = 1024 + kQKMax * (kQBufs + kKStages) + kGStage * kGStages + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
  int B, T, H, dqk, m, d_h, m_h, m_hp;  // m: row width in memory, m_hp: per-head pitch
  int n_iblk, n_ntile, n_pair, n_units;
  float s;
  const float* tau;
  const float* null_bias;
  int has_v;
  int rev;       // sources after the destination (j >= i) instead of before it
  int no_norm;   // the numerator alone: no division by the denominator
  int T_pad;
  float* den_out;  // if set: every row's denominator, [B * H, den_pitch]
  int den_pitch;
  __nv_bfloat16* gbar_out;  // if set: gbar (bf16), laid out as out
  __nv_bfloat16* out;
  unsigned* err;
  uint64_t timeout_ns;
  int debug_timeout;
};

struct Tile {
  int b, head, ib, n0;
};

// Source blocks of a tile, and the index of its jj-th one: blocks 0 .. ib (sources up
// to the destination), or ib .. n_iblk - 1 in reverse mode (sources from it on).
__device__ __forceinline__ int n_src(const Args& a, int ib) { return a.rev ? a.n_iblk - ib : ib + 1; }
__device__ __forceinline__ int src_blk(const Args& a, int ib, int jj) { return a.rev ? ib + jj : jj; }

// Walks this CTA's tiles: units u = blockIdx.x, blockIdx.x + gridDim.x, ...; a unit
// is the pair of destination blocks (nI-1-p, p) of one (batch, head, gate tile), the
// long one first, so every unit costs nI+1 source blocks.
struct TileSeq {
  int u, k;
  Tile t;
  __device__ __forceinline__ bool load(const Args& a) {
    for (; u < a.n_units; u += gridDim.x, k = 0) {
      const int g = u / a.n_pair, p = u % a.n_pair;
      const int lo = p, hi = a.n_iblk - 1 - p;
      if (k == 1 && lo == hi) continue;
      t.ib = k == 0 ? hi : lo;
      t.n0 = (g % a.n_ntile) * kNg;
      t.head = (g / a.n_ntile) % a.H;
      t.b = g / (a.n_ntile * a.H);
      return true;
    }
    return false;
  }
  __device__ __forceinline__ bool first(const Args& a) {
    u = blockIdx.x;
    k = 0;
    return load(a);
  }
  __device__ __forceinline__ bool next(const Args& a) {
    if (++k == 2) {
      k = 0;
      u += gridDim.x;
    }
    return load(a);
  }
};

// Bounded wait with a cheap fast path: one try_wait; only when that fails, the
// abort flag and the wall-clock limit are consulted.
__device__ __forceinline__ bool wait_slow(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernTango);
  return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (mbar_try_wait_nc(smem_u32(bar), parity)) return true;
  return wait_slow(bar, parity, b, a);
}

__device__ __forceinline__ uint32_t qk_layout(int d_h) {
  return d_h == 64 ? kSwizzle128B : d_h == 32 ? kSwizzle64B : kSwizzle32B;
}

// 64 scores of one row (columns [64w, 64w+64) of a block): weights exp2(c (s - 1)),
// with sources after the destination zeroed on the diagonal block, rounded to bf16
// and written as P at TMEM columns [32w, 32w+32) of the block's P slot; the rounded
// weights are added to two partial denominators, each a pair of f32.  The exponent
// argument and the sums use packed f32x2 arithmetic (two values per instruction).
template <int kDiag>  // 0: no mask; 1: sources after the row masked; 2: sources before it
__device__ __forceinline__ void softmax64(const uint32_t (&r)[2][32], uint32_t p_tm, float c, int row,
                                          int src0, uint64_t (&dsum2)[2]) {
  const uint64_t cc = f32x2_pack(c, c), nc = f32x2_pack(-c, -c);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t p[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0, x1;
      f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(r[q][e]), __uint_as_float(r[q][e + 1])), cc, nc), x0, x1);
      float w0 = ex2_approx(x0);
      float w1 = ex2_approx(x1);
      if (kDiag == 1) {
        if (src0 + q * 32 + e > row) w0 = 0.f;
        if (src0 + q * 32 + e + 1 > row) w1 = 0.f;
      } else if (kDiag == 2) {
        if (src0 + q * 32 + e < row) w0 = 0.f;
        if (src0 + q * 32 + e + 1 < row) w1 = 0.f;
      }
      const uint32_t pk = pack_bf16x2(w0, w1);
      dsum2[(e >> 1) & 1] = add_f32x2(dsum2[(e >> 1) & 1], bf16x2_widen(pk));
      p[e / 2] = pk;
    }
    tmem_st16(p_tm + q * 16, p);
  }
}

// Ring position: stage index and the parity of its current phase.
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++stage == n) { stage = 0; phase ^= 1; }
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    tango_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmU, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = sQ + kQBufs * kQKMax;
  uint8_t* sG = sK + kKStages * kQKMax;
  Bars& b = *reinterpret_cast<Bars*>(sG + kGStages * kGStage);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t qk_bytes = kBlk * a.d_h * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQBufs; ++s) {
      mbar_init(&b.q_full[s], 1);
      mbar_init(&b.q_empty[s], 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&b.k_full[s], 1);
      mbar_init(&b.k_empty[s], 1);
    }
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&b.g_full[s], 1);
      mbar_init(&b.g_empty[s], 1);
    }
    mbar_init(&b.s_full, 1);
    mbar_init(&b.s_free, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&b.p_full[i], 8);
    mbar_init(&b.o_full, 1);
    mbar_init(&b.o_empty, 4);
    mbar_init(&b.den_full, 8);
    mbar_init(&b.den_empty, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.p_free[i], 1);
      mbar_init(&b.drain[i], 1);
    }
    mbar_init(&b.never, 1);
    b.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&b.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA: G and v
    Ring gr;
    bool ok = true;
    uint32_t gmask = 0, gph[kGStages] = {};
    TileSeq seq;
    auto ring_load = [&](const CUtensorMap* map, int x, int y, int bb) -> bool {
      if (!wait_bar(&b.g_empty[gr.stage], gr.phase ^ 1, b, a)) return false;
      uint8_t* dst = sG + gr.stage * kGStage;
      if (map) {
        mbar_arrive_expect_tx(&b.g_full[gr.stage], kGStage);
#pragma unroll
        for (int c = 0; c < 4; ++c) tma_load_3d(dst + c * kGBox, map, &b.g_full[gr.stage], x + 64 * c, y, bb);
        gmask |= 1u << gr.stage;
        gph[gr.stage] = gr.phase;
      } else {
        // no copy: the stage's phase completes here, and a final wait on the parity of an
        // earlier copy into it would no longer see that copy's phase
        mbar_arrive(&b.g_full[gr.stage]);
        gmask &= ~(1u << gr.stage);
      }
      gr.next(kGStages);
      return true;
    };
    for (bool have = seq.first(a); ok && have; have = seq.next(a)) {
      const Tile& t = seq.t;
      const int i0 = t.ib * kBlk;
      const int gx = t.head * a.m_hp + t.n0;
      const int nj = n_src(a, t.ib);
      for (int jj = 0; ok && jj < nj; ++jj)
        for (int h = 0; ok && h < 2; ++h) ok = ring_load(&tmG, gx, src_blk(a, t.ib, jj) * kBlk + h * kHalf, t.b);
      // the tile's v, rows [i0, i0+64) and [i0+64, i0+128), for the epilogue
      for (int h = 0; ok && h < 2; ++h) ok = ring_load(a.has_v ? &tmV : nullptr, gx, i0 + h * kHalf, t.b);
    }
    // Copies still in flight land before the CTA exits.
    for (int s = 0; s < kGStages; ++s)
      if (gmask & (1u << s)) mbar_wait(&b.g_full[s], gph[s], a.timeout_ns);
  } else if (warp == 3 && lane == 0) {
    // ------------------------------------------------------------ TMA: qhat and khat
    // (a thread of its own, so that score loads never queue behind the G ring)
    Ring kr;
    bool ok = true;
    uint32_t qmask = 0, kmask = 0, qph[kQBufs] = {}, kph[kKStages] = {};
    TileSeq seq;
    int tc = 0;
    for (bool have = seq.first(a); ok && have; have = seq.next(a), ++tc) {
      const Tile& t = seq.t;
      const int i0 = t.ib * kBlk, qb = tc & 1;
      const uint32_t qp = (tc >> 1) & 1;
      if (!(ok = wait_bar(&b.q_empty[qb], qp ^ 1, b, a))) break;
      mbar_arrive_expect_tx(&b.q_full[qb], qk_bytes);
      tma_load_3d(sQ + qb * kQKMax, &tmQ, &b.q_full[qb], t.head * a.d_h, i0, t.b);
      qmask |= 1u << qb;
      qph[qb] = qp;
      const int nj = n_src(a, t.ib);
      for (int jj = 0; ok && jj < nj; ++jj) {
        if (!(ok = wait_bar(&b.k_empty[kr.stage], kr.phase ^ 1, b, a))) break;
        mbar_arrive_expect_tx(&b.k_full[kr.stage], qk_bytes);
        tma_load_3d(sK + kr.stage * kQKMax, &tmK, &b.k_full[kr.stage], t.head * a.d_h,
                    src_blk(a, t.ib, jj) * kBlk, t.b);
        kmask |= 1u << kr.stage;
        kph[kr.stage] = kr.phase;
        kr.next(kKStages);
      }
    }
    for (int s = 0; s < kQBufs; ++s)
      if (qmask & (1u << s)) mbar_wait(&b.q_full[s], qph[s], a.timeout_ns);
    for (int s = 0; s < kKStages; ++s)
      if (kmask & (1u << s)) mbar_wait(&b.k_full[s], kph[s], a.timeout_ns);
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------------------ MMA issue: scores
    // S_J = Qhat Khat_J^T into the score slot once the softmax warps have read S_{J-1}.
    const uint32_t idesc_s = idesc_bf16_f32(kBlk, kBlk, false, false);
    const uint32_t lay = qk_layout(a.d_h);
    const uint32_t sbo = 8u * a.d_h * 2u;
    const int ksteps = a.d_h / 16;
    // Descriptors of stage 0; other stages differ only in the start-address field
    // ((byte offset) >> 4 added to the low bits, which never carry: smem < 256 KB).
    const uint64_t qdesc0 = smem_desc(smem_u32(sQ), 16, sbo, lay);
    const uint64_t kdesc0 = smem_desc(smem_u32(sK), 16, sbo, lay);
    bool ok = true;
    Ring kr;
    uint32_t J = 0;  // source blocks of this CTA
    TileSeq seq;
    int tc = 0;
    for (bool have = seq.first(a); ok && have; have = seq.next(a), ++tc) {
      const int qb = tc & 1;
      if (!(ok = wait_bar(&b.q_full[qb], (tc >> 1) & 1, b, a))) break;
      const uint64_t qd = qdesc0 + (uint64_t)((qb * kQKMax) >> 4);
      const int nj = n_src(a, seq.t.ib);
      for (int j = 0; j < nj; ++j, ++J) {
        if (J >= 1 && !(ok = wait_bar(&b.s_free, (J - 1) & 1, b, a))) break;
        if (!(ok = wait_bar(&b.k_full[kr.stage], kr.phase, b, a))) break;
        tc_fence_after_nc();
        const uint64_t kd = kdesc0 + (uint64_t)((kr.stage * kQKMax) >> 4);
        const uint32_t stm = tmem + kColS0;
        for (int kk = 0; kk < ksteps; ++kk)
          mma_bf16_ss_nc(stm, qd + (uint64_t)(kk * 2), kd + (uint64_t)(kk * 2), idesc_s, kk != 0);
        mma_commit_nc(&b.k_empty[kr.stage]);
        mma_commit_nc(&b.s_full);
        kr.next(kKStages);
        if (j == nj - 1) mma_commit_nc(&b.q_empty[qb]);
      }
    }
    mma_commit(&b.drain[0]);
    mbar_wait(&b.drain[0], 0, a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue: P.G
    const uint32_t idesc_o = idesc_bf16_f32(kBlk, kNg, false, true);
    const uint64_t gdesc0 = smem_desc(smem_u32(sG), kGBox, 1024, kSwizzle128B);
    bool ok = true;
    if (a.debug_timeout) ok = wait_bar(&b.never, 0, b, a);  // nothing ever arrives here
    Ring gr;
    uint32_t ophase = 0;
    uint32_t J = 0;  // source blocks of this CTA
    TileSeq seq;
    for (bool have = ok && seq.first(a); ok && have; have = seq.next(a)) {
      const int nj = n_src(a, seq.t.ib);
      for (int j = 0; j < nj; ++j, ++J) {
        // O += P_J G_J (two half blocks); the tile's first block overwrites O once the
        // epilogue has read the previous tile's accumulator out of TMEM.
        const uint32_t buf = J & 1;
        if (!(ok = wait_bar(&b.p_full[buf], (J >> 1) & 1, b, a))) break;
        if (j == 0) {
          if (!(ok = wait_bar(&b.o_empty, ophase ^ 1, b, a))) break;
          ophase ^= 1;
        }
        const uint32_t ptm = tmem + kColP0 + buf * 64;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!(ok = wait_bar(&b.g_full[gr.stage], gr.phase, b, a))) break;
          tc_fence_after_nc();
          const uint64_t gd = gdesc0 + (uint64_t)((gr.stage * kGStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            mma_bf16_ts_nc(tmem + kColO, ptm + h * 32 + kk * 8, gd + (uint64_t)(kk * (2048 >> 4)), idesc_o,
                           (j == 0 && h == 0 && kk == 0) ? 0u : 1u);
          mma_commit_nc(&b.g_empty[gr.stage]);
          gr.next(kGStages);
        }
        if (!ok) break;
        mma_commit_nc(&b.p_free[buf]);
      }
      if (!ok) break;
      mma_commit_nc(&b.o_full);
      gr.next(kGStages);  // the tile's two v stages belong to the epilogue
      gr.next(kGStages);
    }
    mma_commit(&b.drain[1]);
    mbar_wait(&b.drain[1], 0, a.timeout_ns);
  } else if (warp >= kSoftWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------ softmax
    const int wg = (warp - kSoftWarp0) / 4;  // columns [64 wg, 64 wg + 64) of every block
    const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    uint32_t J = 0;
    int tc = 0;
    TileSeq seq;
    for (bool have = seq.first(a); ok && have; have = seq.next(a), ++tc) {
      const Tile t = seq.t;
      const float tau = head_tau(a.tau, a.s, t.head, a.err, kKernTango);
      const float c = tau * kLog2e;
      uint64_t dsum2[2] = {0, 0};  // independent partial sums, pairs of f32
      const int nj = n_src(a, t.ib);
      for (int j = 0; j < nj; ++j, ++J) {
        const uint32_t buf = J & 1;
        const uint32_t stm = tmem + kColS0 + lane_off;
        const uint32_t pw = tmem + kColP0 + buf * 64 + lane_off;
        uint32_t r[2][32];
        if (ok) ok = wait_bar(&b.s_full, J & 1, b, a);
        if (ok) {
          tc_fence_after();
          tmem_ld32(stm + wg * 64, r[0]);
          tmem_ld32(stm + wg * 64 + 32, r[1]);
          tmem_ld_wait();
        }
        // this block's P slot is free once the P.G of block J - 2 has completed
        if (ok && J >= 2) ok = wait_bar(&b.p_free[buf], ((J - 2) >> 1) & 1, b, a);
        tc_fence_before();
        // both warpgroups have read their scores: the S slot takes the next block's.
        // The barrier also ANDs their status.
        ok = named_bar_and(1, 256, ok);
        if (!ok) break;
        if (warp == kSoftWarp0 && lane == 0) mbar_arrive(&b.s_free);
        tc_fence_after();
        // sources relative to the destination block; the diagonal block is masked
        const int sb = src_blk(a, t.ib, j);
        const int src0 = (sb - t.ib) * kBlk + wg * 64;
        if (sb != t.ib) softmax64<0>(r, pw + wg * 32, c, row, src0, dsum2);
        else if (a.rev) softmax64<2>(r, pw + wg * 32, c, row, src0, dsum2);
        else softmax64<1>(r, pw + wg * 32, c, row, src0, dsum2);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.p_full[buf]);
      }
      if (!ok) break;
      // Hand this warpgroup's half of the row denominators to the epilogue.  Both
      // warpgroups agree on the status before either goes on.
      if (ok) ok = wait_bar(&b.den_empty, ((tc & 1) ^ 1), b, a);
      ok = named_bar_and(1, 256, ok);
      if (!ok) break;
      float d0, d1, d2, d3;
      f32x2_unpack(dsum2[0], d0, d1);
      f32x2_unpack(dsum2[1], d2, d3);
      b.rowsum[wg][row] = (d0 + d1) + (d2 + d3);
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.den_full);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t otm = tmem + kColO + ((uint32_t)(quarter * 32) << 16);
    const int hh = quarter >> 1;  // row half: rows [64 hh, 64 hh + 64), ring stage sa or sb
    const bool hissuer = lane == 0 && (warp & 1) == 0;
    bool ok = true;
    uint32_t ophase = 0;
    int gpos = 0;  // ring stages consumed so far (G and v)
    int tc = 0;
    TileSeq seq;
    for (bool have = seq.first(a); ok && have; have = seq.next(a), ++tc) {
      const Tile t = seq.t;
      const int i = t.ib * kBlk + row;
      gpos += 2 * n_src(a, t.ib);
      const int sa = gpos % kGStages, sb = (gpos + 1) % kGStages;
      const uint32_t pa = (gpos / kGStages) & 1, pb = ((gpos + 1) / kGStages) & 1;
      gpos += 2;
      float den = 0.f;
      if (ok) ok = wait_bar(&b.den_full, tc & 1, b, a);
      if (ok) {
        den = b.rowsum[0][row] + b.rowsum[1][row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.den_empty);
      }
      if (ok) ok = wait_bar(&b.o_full, ophase, b, a);
      if (ok) ok = wait_bar(&b.g_full[sa], pa, b, a);
      if (ok) ok = wait_bar(&b.g_full[sb], pb, b, a);
      ok = named_bar_and(2, 128, ok);
      if (!ok) break;
      ophase ^= 1;
      const float tau = head_tau(a.tau, a.s, t.head, a.err, kKernTango);
      if (a.null_bias) den += (float)(i + 1) * exp2f((a.null_bias[t.head] - tau) * kLog2e);
      const bool row_ok = i < a.T;
      if (a.den_out && t.n0 == 0 && row_ok) a.den_out[(size_t)(t.b * a.H + t.head) * a.den_pitch + i] = den;
      const float inv = a.no_norm ? 1.f : 1.f / den;
      const uint64_t inv2 = f32x2_pack(inv, inv), zero2 = f32x2_pack(0.f, 0.f);
      tc_fence_after();
      const int rr = row & 63;
      const uint32_t vrow = smem_u32(sG + (row < 64 ? sa : sb) * kGStage) + rr * 128;
      const size_t grow = ((size_t)t.b * a.T + (row_ok ? i : 0)) * a.m + (size_t)t.head * a.m_hp;
#pragma unroll 1
      for (int cq = 0; cq < 4; ++cq) {
        uint32_t o[2][32];
        tmem_ld32(otm + cq * 64, o[0]);
        tmem_ld32(otm + cq * 64 + 32, o[1]);
        tmem_ld_wait();
        if (cq == 3) {  // the accumulator is free for the next tile
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&b.o_empty);
        }
        const int col0 = t.n0 + cq * 64;
        const bool straddle = col0 < a.m_h && col0 + 64 > a.m_h;
        const uint32_t box = vrow + cq * kGBox;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t addr = box + (uint32_t)((k ^ (rr & 7)) << 4);
          const uint4 vv = a.has_v ? ld_shared_v4(addr) : make_uint4(0, 0, 0, 0);
          const uint32_t* ok8 = &o[k >> 2][(k & 3) * 8];
          // gbar = O / den in bf16 pairs (a packed f32x2 scale), then one bf16x2 product
          // with v
          uint32_t gq[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float y0, y1;
            f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(ok8[2 * e]), __uint_as_float(ok8[2 * e + 1])), inv2,
                                   zero2),
                         y0, y1);
            gq[e] = pack_bf16x2(y0, y1);
          }
          if (a.gbar_out && row_ok && col0 + 8 * k < a.m_h)
            st_global_v4(a.gbar_out + grow + col0 + 8 * k, gq[0], gq[1], gq[2], gq[3]);
          uint4 uu;
          uu.x = a.has_v ? ptx::mul_bf16x2(gq[0], vv.x) : gq[0];
          uu.y = a.has_v ? ptx::mul_bf16x2(gq[1], vv.y) : gq[1];
          uu.z = a.has_v ? ptx::mul_bf16x2(gq[2], vv.z) : gq[2];
          uu.w = a.has_v ? ptx::mul_bf16x2(gq[3], vv.w) : gq[3];
          if (!straddle) {
            st_shared_v4(addr, uu);
          } else if (row_ok && col0 + 8 * k < a.m_h) {
            st_global_v4(a.out + grow + col0 + 8 * k, uu.x, uu.y, uu.z, uu.w);
          }
        }
        // this chunk of u is in shared memory: each row half stores its box now, so the
        // stores overlap the next chunks
        fence_proxy_async_smem();
        named_bar_sync(3 + hh, 64);
        if (hissuer) {
          const int y = t.ib * kBlk + hh * kHalf;
          if (y < a.T && !straddle && col0 + 64 <= a.m_h)
            tma_store_3d(&tmU, sG + (hh == 0 ? sa : sb) * kGStage + cq * kGBox, t.head * a.m_hp + col0, y, t.b);
          bulk_commit_group();
        }
      }
      // the row half's stage is free once its stores have read it
      if (hissuer) {
        bulk_wait_group_read0();
        mbar_arrive(&b.g_empty[hh == 0 ? sa : sb]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_tango_tc(const AggArgs& p, cudaStream_t s) {
  Args a = {};
  a.B = p.B; a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.m = p.m;
  a.d_h = p.dqk / p.H; a.m_hp = p.m / p.H; a.m_h = p.m_h ? p.m_h : a.m_hp;
  a.n_iblk = ceil_div(p.T, kBlk);
  a.n_ntile = ceil_div(a.m_h, kNg);
  a.n_pair = (a.n_iblk + 1) / 2;
  const long long units = (long long)p.B * p.H * a.n_ntile * a.n_pair;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_units = (int)units;
  a.s = p.s; a.tau = p.tau; a.null_bias = p.null_bias;
  a.has_v = p.v != nullptr;
  a.rev = p.rev;
  a.no_norm = p.no_norm;
  a.T_pad = a.n_iblk * kBlk;
  a.den_out = p.den_out;
  a.den_pitch = p.den_pitch ? p.den_pitch : a.T_pad;
  a.gbar_out = static_cast<__nv_bfloat16*>(p.gbar_out);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.err = p.err;
  a.debug_timeout = (p.flags & TG_FLAG_DEBUG_TIMEOUT) ? 1 : 0;
  a.timeout_ns = a.debug_timeout ? 1000000ull : 2000000000ull;
  CUtensorMap mq, mk, mg, mv, mu;
  cudaError_t e = make_tmap_3d(&mq, p.q, p.B, p.T, p.dqk, kBlk, a.d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mk, p.k, p.B, p.T, p.dqk, kBlk, a.d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mg, p.g, p.B, p.T, p.m, kHalf, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mv, p.v ? p.v : p.g, p.B, p.T, p.m, kHalf, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mu, p.out, p.B, p.T, p.m, kHalf, 64);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tango_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = a.n_units < num_sms() ? a.n_units : num_sms();
  tango_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mg, mv, mu, a);
  return cudaGetLastError();
}

}  // namespace tg
