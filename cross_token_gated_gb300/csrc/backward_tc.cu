// Backward of the gate aggregation, "TANGO: Token-Aggregated Nonlinear Gating
// Operators ...", sec. 2.1 eq. 5 with the weights of sec. 2.2 eqs. 6-9: the gradient
// of every pair weight, on the tensor cores (tcgen05).
//
// With u_i = gbar_i * v_i, gbar_i = sum_j w_ij g_j / den_i and an upstream gradient
// dU, let E_i = dU_i * v_i / den_i and D_i = E_i . gbar_i (both from the prep
// kernel).  The loss gradient with respect to a pair weight w_ij is
//     dL/dw_ij = E_i . g_j - D_i                      (the null term carries no value)
// and the contraction E_i . g_j runs over all m_h gate columns of the head, so per
// (batch, head) it is the causal half of the T x T product E G^T.  This kernel forms
// that product in 128 x 256 tiles (destinations x sources) and writes, per pair,
//     window pair (eq. 6):  X_ij = tau w_ij (E_i . g_j - D_i),  w_ij = e^{tau (qhat_i.khat_j - 1)}
//     older pair (eq. 9):   X_ij = E_i . g_j - D_i        (WANGO; the feature maps enter later)
//     j > i:                X_ij = 0
// in bf16: window pairs to X, older pairs to X_old, both [B*H, T_pad, T_pad] (each
// 128 x 128 block is written to the matrices whose pairs it holds; the other entries of
// a written block are zero).  agg_bwd_qk_kernel then forms dqhat = X Khat and
// dkhat = X^T Qhat, and the feature-map gradients X_old Phi(k~) and X_old^T Phi(q~).  The weights use the
// same static shift e^-tau as the forward kernels; E carries the matching shifted
// denominator, so X is the gradient of the shifted weight.
//
// Persistent CTAs, one per SM, take tiles round-robin:
//   warp 0      TMA: a 3-stage ring of E (128 x 64) and G (256 x 64) boxes over the
//               head's m_h columns (a 4-D map: columns past the head read as zero),
//               then the tile's 256 unit keys for the epilogue
//   warp 1      TMEM allocation and MMA issue: 128 x 256 x 16 tcgen05.mma into one of
//               two 256-column accumulators, so a tile's epilogue overlaps the next
//               tile's products
//   warps 2-9   epilogue, two warps per TMEM lane quarter (columns [0, 128) and
//               [128, 256)): the score qhat_i . khat_j on the CUDA cores from the keys in
//               shared memory, the weight, and X in bf16, each thread storing 64-byte
//               pieces of its own row (no staging: the shared memory goes to a fourth
//               operand stage)
// Every wait is bounded; on expiry the kernel records a timeout and all roles leave.
#include "tg_common.cuh"
#include "tg_ptx.cuh"
#include "tg_tc.h"
#include "tg_tma.h"

namespace tg {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = BM * BK * 2;      // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;      // 32 KB
constexpr uint32_t kKeyBytes = BN * 64 * 2;    // 32 KB: 256 unit keys at d_h <= 64
constexpr int kThreads = 320;
constexpr int kEpiWarp0 = 2;

struct __align__(8) Bars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
  uint64_t key_full, key_empty, drain, never;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + kStages * (kABytes + kBBytes) + kKeyBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
  int B, T, H, d_h, T_pad;
  int tiles_per_bh, n_tiles, nkb;
  int wango, window;
  float s;
  const float* tau;
  const __nv_bfloat16* qhat;  // [B, T, H * d_h], unit per head
  int dqk;
  const float* dp;            // D_i: [B * H, T_pad]
  __nv_bfloat16* X;           // [B * H, T_pad, T_pad]: window pairs
  __nv_bfloat16* X_old;       // the same for older pairs (WANGO), else NULL
  int band;                   // >= 0: only source blocks jb >= ib - band
  unsigned* err;
  uint64_t timeout_ns;
  int debug_timeout;          // test hook: the MMA issuer first waits on a barrier nothing signals
};

struct Tile {
  int b, head, ib, jt;
};

// The 256-source tiles of destination block ib: jt_lo .. ib / 2, every tile holding a
// pair j <= i (with a band, only those holding a source block jb >= ib - band).
__host__ __device__ __forceinline__ int jt_lo_of(int ib, int band) {
  return band < 0 ? 0 : (ib - band > 0 ? ib - band : 0) / 2;
}
__device__ __forceinline__ Tile tile_of(const Args& a, int t) {
  Tile r;
  const int bh = t / a.tiles_per_bh;
  int rem = t % a.tiles_per_bh, ib = 0;
  while (rem >= ib / 2 - jt_lo_of(ib, a.band) + 1) {
    rem -= ib / 2 - jt_lo_of(ib, a.band) + 1;
    ++ib;
  }
  r.b = bh / a.H;
  r.head = bh % a.H;
  r.ib = ib;
  r.jt = jt_lo_of(ib, a.band) + rem;
  return r;
}

__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernBackward);
  return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (mbar_try_wait_nc(smem_u32(bar), parity)) return true;
  return wait_slow(bar, parity, b, a);
}

// Byte offset of a logical offset inside a TMA box written with the swizzle that the
// tensor maps pick for rows of `row_bytes` (128: 128B, 64: 64B, 32: 32B): the 16-byte
// chunk index is XORed with address bits 7.. (as many bits as the chunk index has).
__device__ __forceinline__ uint32_t swz(uint32_t off, uint32_t row_bytes) {
  const uint32_t mask = row_bytes == 128 ? 0x70u : row_bytes == 64 ? 0x30u : 0x10u;
  return off ^ ((off >> 3) & mask);
}

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    agg_bwd_pairs_kernel(const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmG,
                         const __grid_constant__ CUtensorMap tmK, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = sA + kStages * kABytes;
  uint8_t* sKey = sB + kStages * kBBytes;
  Bars& b = *reinterpret_cast<Bars*>(sKey + kKeyBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr uint32_t kRowBytes = DH * 2;
  constexpr uint32_t kKeyHalf = 128 * kRowBytes;  // one TMA box of 128 keys

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b.full[s], 1);
      mbar_init(&b.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.acc_full[i], 1);
      mbar_init(&b.acc_empty[i], 8);
    }
    mbar_init(&b.key_full, 1);
    mbar_init(&b.key_empty, 8);
    mbar_init(&b.drain, 1);
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
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    int mask = 0, kmask = 0;
    uint32_t sph[kStages] = {}, kph = 0;
    int tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < a.n_tiles; t += gridDim.x, ++tc) {
      const Tile tl = tile_of(a, t);
      const int i0 = tl.ib * BM, j0 = tl.jt * BN;
      for (int kb = 0; kb < a.nkb; ++kb) {
        if (!(ok = wait_bar(&b.empty[stage], phase ^ 1, b, a))) break;
        mbar_arrive_expect_tx(&b.full[stage], kABytes + kBBytes);
        tma_load_4d(sA + stage * kABytes, &tmE, &b.full[stage], kb * BK, tl.head, i0, tl.b);
        tma_load_4d(sB + stage * kBBytes, &tmG, &b.full[stage], kb * BK, tl.head, j0, tl.b);
        mask |= 1 << stage;
        sph[stage] = phase;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      // the tile's keys, once the previous tile's epilogue is done with them
      if (!(ok = wait_bar(&b.key_empty, (tc & 1) ^ 1, b, a))) break;
      mbar_arrive_expect_tx(&b.key_full, 2 * kKeyHalf);
      tma_load_3d(sKey, &tmK, &b.key_full, tl.head * DH, j0, tl.b);
      tma_load_3d(sKey + kKeyHalf, &tmK, &b.key_full, tl.head * DH, j0 + 128, tl.b);
      kmask = 1;
      kph = tc & 1;
    }
    for (int s = 0; s < kStages; ++s)
      if (mask & (1 << s)) mbar_wait(&b.full[s], sph[s], a.timeout_ns);
    if (kmask) mbar_wait(&b.key_full, kph, a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    const uint32_t idesc = idesc_bf16_f32(BM, BN, false, false);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = !a.debug_timeout || wait_bar(&b.never, 0, b, a);  // nothing ever arrives there
    for (int t = blockIdx.x; ok && t < a.n_tiles; t += gridDim.x) {
      if (!(ok = wait_bar(&b.acc_empty[acc], acc_phase ^ 1, b, a))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      for (int kb = 0; kb < a.nkb; ++kb) {
        if (!(ok = wait_bar(&b.full[stage], phase, b, a))) break;
        tc_fence_after_nc();
        const uint32_t aaddr = smem_u32(sA + stage * kABytes), baddr = smem_u32(sB + stage * kBBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16_ss_nc(d_tmem, smem_desc(aaddr + kk * 32, 16, 1024, kSwizzle128B),
                         smem_desc(baddr + kk * 32, 16, 1024, kSwizzle128B), idesc, (kb | kk) != 0);
        mma_commit_nc(&b.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit_nc(&b.acc_full[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    mma_commit(&b.drain);
    mbar_wait(&b.drain, 0, a.timeout_ns);
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                // TMEM lanes 32 quarter .. + 31
    const int half = (warp - kEpiWarp0) >> 2;    // columns [128 half, 128 half + 128)
    const int lrow = quarter * 32 + lane;
    const uint32_t key = smem_u32(sKey);
    int acc = 0, tc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < a.n_tiles; t += gridDim.x, ++tc) {
      const Tile tl = tile_of(a, t);
      const int i = tl.ib * BM + lrow;
      if (ok) ok = wait_bar(&b.acc_full[acc], acc_phase, b, a);
      if (ok) ok = wait_bar(&b.key_full, tc & 1, b, a);
      ok = named_bar_and(1, 256, ok);
      if (!ok) break;
      tc_fence_after();
      const bool row_ok = i < a.T;
      const float tau = head_tau(a.tau, a.s, tl.head, a.err, kKernBackward);
      const float c = tau * kLog2e;
      const float dp = row_ok ? a.dp[(size_t)(tl.b * a.H + tl.head) * a.T_pad + i] : 0.f;
      // qhat_i as packed f32 pairs
      uint64_t qv[DH / 2];
      {
        const __nv_bfloat16* qrow = a.qhat + ((size_t)tl.b * a.T + (row_ok ? i : 0)) * a.dqk + tl.head * DH;
#pragma unroll
        for (int c8 = 0; c8 < DH / 8; ++c8) {
          const uint4 x = row_ok ? ld_global_v4(qrow + 8 * c8) : make_uint4(0, 0, 0, 0);
          qv[4 * c8 + 0] = bf16x2_widen(x.x);
          qv[4 * c8 + 1] = bf16x2_widen(x.y);
          qv[4 * c8 + 2] = bf16x2_widen(x.z);
          qv[4 * c8 + 3] = bf16x2_widen(x.w);
        }
      }
      const uint32_t trow = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16) + half * 128;
      const int jbase = tl.jt * BN + half * 128;
      const size_t xoff = ((size_t)(tl.b * a.H + tl.head) * a.T_pad + i) * a.T_pad;
      {
#pragma unroll 1
        for (int cbase = 0; cbase < 128; cbase += 16) {
          uint32_t r[16];
          tmem_ld16(trow + cbase, r);
          tmem_ld_wait();
          if (cbase == 112) {  // the accumulator is free for the tile after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.acc_empty[acc]);
          }
          uint32_t pk[8], po[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float x2[2], o2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int jl = half * 128 + cbase + e + h;  // source within the tile
              const int j = jbase + cbase + e + h;
              float x = 0.f, xo = 0.f;
              if (row_ok && j <= i) {
                const float dl = __uint_as_float(r[e + h]) - dp;
                const bool window = !a.wango || i - j < a.window;
                if (window) {
                  // score qhat_i . khat_j from the keys in shared memory
                  uint64_t s2a = 0, s2b = 0;
#pragma unroll
                  for (int c8 = 0; c8 < DH / 8; ++c8) {
                    const uint4 kv = ld_shared_v4(key + ((uint32_t)(jl >> 7) * kKeyHalf) +
                                                  swz((uint32_t)(jl & 127) * kRowBytes + c8 * 16, kRowBytes));
                    s2a = fma_f32x2(qv[4 * c8 + 0], bf16x2_widen(kv.x), s2a);
                    s2b = fma_f32x2(qv[4 * c8 + 1], bf16x2_widen(kv.y), s2b);
                    s2a = fma_f32x2(qv[4 * c8 + 2], bf16x2_widen(kv.z), s2a);
                    s2b = fma_f32x2(qv[4 * c8 + 3], bf16x2_widen(kv.w), s2b);
                  }
                  float s0, s1, s2, s3;
                  f32x2_unpack(s2a, s0, s1);
                  f32x2_unpack(s2b, s2, s3);
                  const float sc = (s0 + s1) + (s2 + s3);
                  const float w = ex2_approx(fmaf(c, sc, -c));
                  x = tau * w * dl;
                } else {
                  xo = dl;
                }
              }
              x2[h] = x;
              o2[h] = xo;
            }
            pk[e / 2] = pack_bf16x2(x2[0], x2[1]);
            po[e / 2] = pack_bf16x2(o2[0], o2[1]);
          }
          if (jbase + cbase < a.T_pad) {  // 16 whole columns inside the padded matrix
            // the 128 x 128 block of these columns: does it hold window / older pairs?
            const int dblk = tl.ib - (jbase + cbase) / 128;
            const bool has_win = !a.wango || dblk * 128 - 127 < a.window;
            const bool has_old = a.wango && dblk * 128 + 127 >= a.window;
            if (has_win) {
#pragma unroll
              for (int k = 0; k < 2; ++k)
                st_global_v4(a.X + xoff + jbase + cbase + 8 * k, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                             pk[4 * k + 3]);
            }
            if (has_old) {
#pragma unroll
              for (int k = 0; k < 2; ++k)
                st_global_v4(a.X_old + xoff + jbase + cbase + 8 * k, po[4 * k], po[4 * k + 1], po[4 * k + 2],
                             po[4 * k + 3]);
            }
          }
        }
      }
      // both halves have read the keys
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.key_empty);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dq / dk
// agg_bwd_qk_kernel: one CTA per (side, batch-head, own 128-row block).  Side 0 sums over
// the sources j <= i of its destinations i:
//     win_i = sum_j X_ij khat_j,      old_i = sum_j X_old_ij Phi(k~_j)
// side 1 over the destinations i >= j of its sources j:
//     win_j = sum_i X_ij qhat_i,      old_j = sum_i X_old_ij e^-tau Phi(q~_i)
// with Phi(k~) = phi(sqrt(tau) khat) and e^-tau Phi(q~) the bf16 feature maps of the
// forward pass.  Both sums are tcgen05 MMAs (M = 128 own rows, N = 64 vector columns,
// K = 128 partner rows per step): side 0 reads the X tile K-major, side 1 reads the same
// tile as its transpose (MN-major); the partner vectors are MN-major.  The epilogue,
// one thread per own row, takes the older part through the feature map's derivative,
//     dqhat = win + sqrt(tau) e^-tau phi'(sqrt(tau) qhat) * old,
//     dkhat = win + sqrt(tau) phi'(sqrt(tau) khat) * old,
// and then the unit normalisation: dq = (dqhat - qhat (qhat . dqhat)) / max(|q|, 1e-12).
// The vector boxes are always 64 columns wide (128-byte swizzle) from the head's first
// column; at d_h < 64 the extra accumulator columns hold other heads' sums and are
// not read.
namespace qkk {
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA and TMEM, warps 2-5 epilogue
constexpr int kStages = 2;
constexpr uint32_t kXBox = 128 * 64 * 2;       // 16 KB: 128 rows x 64 columns of X
constexpr uint32_t kXBytes = 2 * kXBox;        // 32 KB: a 128 x 128 block
constexpr uint32_t kVBytes = 128 * 64 * 2;     // 16 KB: 128 vectors, 64 columns
constexpr uint32_t kStageBytes = 2 * kXBytes + 2 * kVBytes;  // X, X_old, unit vectors, feature maps
struct __align__(8) Bars {
  uint64_t full[kStages], empty[kStages], acc_full, drain, never;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
  int B, T, H, dqk, d_h, T_pad, nblk, n_bh;
  int wango, window, phi_mode;
  float s;
  const float* tau;
  const __nv_bfloat16 *qhat, *khat, *raw_q, *raw_k;
  __nv_bfloat16 *dq, *dk;
  int band;                   // band >= 0: partners beyond it come from the scans' sums
  const float* far[2];
  unsigned* err;
  uint64_t timeout_ns;
  int debug_timeout;          // test hook: the MMA issuer first waits on a barrier nothing signals
};

__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernBackward);
  return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (mbar_try_wait_nc(smem_u32(bar), parity)) return true;
  return wait_slow(bar, parity, b, a);
}

struct Item {
  int side, bh, b, head, ob, p_lo, n_steps;
};
// Items with the most partner steps first (rank 0: side 0's last block, side 1's first).
__device__ __forceinline__ Item item_of(const Args& a) {
  Item it;
  const int idx = blockIdx.x;
  it.side = idx & 1;
  const int r = idx >> 1;
  const int rank = r / a.n_bh;
  it.bh = r % a.n_bh;
  it.b = it.bh / a.H;
  it.head = it.bh % a.H;
  it.ob = it.side == 0 ? a.nblk - 1 - rank : rank;
  if (a.band < 0) {
    it.p_lo = it.side == 0 ? 0 : it.ob;
    it.n_steps = it.side == 0 ? it.ob + 1 : a.nblk - it.ob;
  } else {  // the band's partner blocks only
    it.p_lo = it.side == 0 ? max(0, it.ob - a.band) : it.ob;
    it.n_steps = it.side == 0 ? it.ob - it.p_lo + 1 : min(a.nblk - 1, it.ob + a.band) - it.ob + 1;
  }
  return it;
}
// Destination and source blocks of step p, and which pair kinds the block holds.
__device__ __forceinline__ void step_blocks(const Args& a, const Item& it, int p, int& iblk, int& jblk, bool& hw,
                                            bool& ho) {
  const int pb = it.p_lo + p;
  iblk = it.side == 0 ? it.ob : pb;
  jblk = it.side == 0 ? pb : it.ob;
  const int d = iblk - jblk;
  hw = !a.wango || d * 128 - 127 < a.window;
  ho = a.wango && d * 128 + 127 >= a.window;
}

__device__ __forceinline__ float dphi(float u, int mode, float inv_sqrt_dh) {
  const float d = u > 0.f ? 1.f : expf(u);
  return mode == 0 ? d * inv_sqrt_dh : d;
}

__global__ void __launch_bounds__(kThreads, 1)
    agg_bwd_qk_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXo,
                      const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmFq, const __grid_constant__ CUtensorMap tmFk,
                      const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& b = *reinterpret_cast<Bars*>(base + kStages * kStageBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Item it = item_of(a);
  bool any_old = false;
  for (int p = 0; p < it.n_steps; ++p) {
    int ib, jb;
    bool hw, ho;
    step_blocks(a, it, p, ib, jb, hw, ho);
    any_old |= ho;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b.full[s], 1);
      mbar_init(&b.empty[s], 1);
    }
    mbar_init(&b.acc_full, 1);
    mbar_init(&b.drain, 1);
    mbar_init(&b.never, 1);
    b.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&b.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    int mask = 0;
    uint32_t sph[kStages] = {0, 0};
    const CUtensorMap* vmap = it.side == 0 ? &tmK : &tmQ;   // partner unit vectors
    const CUtensorMap* fmap = it.side == 0 ? &tmFk : &tmFq; // partner feature maps
    for (int p = 0; p < it.n_steps; ++p) {
      int ib, jb;
      bool hw, ho;
      step_blocks(a, it, p, ib, jb, hw, ho);
      if (!wait_bar(&b.empty[stage], phase ^ 1, b, a)) break;
      uint8_t* st = base + stage * kStageBytes;
      mbar_arrive_expect_tx(&b.full[stage], (hw ? kXBytes + kVBytes : 0u) + (ho ? kXBytes + kVBytes : 0u));
      const int prow = (it.side == 0 ? jb : ib) * 128;  // partner rows
      if (hw) {
        tma_load_3d(st, &tmX, &b.full[stage], jb * 128, ib * 128, it.bh);
        tma_load_3d(st + kXBox, &tmX, &b.full[stage], jb * 128 + 64, ib * 128, it.bh);
        tma_load_3d(st + 2 * kXBytes, vmap, &b.full[stage], it.head * a.d_h, prow, it.b);
      }
      if (ho) {
        tma_load_3d(st + kXBytes, &tmXo, &b.full[stage], jb * 128, ib * 128, it.bh);
        tma_load_3d(st + kXBytes + kXBox, &tmXo, &b.full[stage], jb * 128 + 64, ib * 128, it.bh);
        tma_load_3d(st + 2 * kXBytes + kVBytes, fmap, &b.full[stage], it.head * a.d_h, prow, it.b);
      }
      mask |= 1 << stage;
      sph[stage] = phase;
      if (++stage == kStages) { stage = 0; phase ^= 1; }
    }
    for (int s = 0; s < kStages; ++s)
      if (mask & (1 << s)) mbar_wait(&b.full[s], sph[s], a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    const bool tr = it.side == 1;  // X read as its transpose
    const uint32_t idesc = idesc_bf16_f32(128, 64, tr, true);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = !a.debug_timeout || wait_bar(&b.never, 0, b, a), first_w = true, first_o = true;
    for (int p = 0; ok && p < it.n_steps; ++p) {
      int ib, jb;
      bool hw, ho;
      step_blocks(a, it, p, ib, jb, hw, ho);
      if (!(ok = wait_bar(&b.full[stage], phase, b, a))) break;
      tc_fence_after_nc();
      const uint32_t st = smem_u32(base + stage * kStageBytes);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        if (part == 0 ? !hw : !ho) continue;
        const uint32_t xa = st + part * kXBytes, va = st + 2 * kXBytes + part * kVBytes;
        const uint32_t d_tmem = tmem + part * 64;
        bool& first = part == 0 ? first_w : first_o;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // A: X K-major (columns = partner rows, two 64-column boxes) or, transposed,
          // MN-major (rows = partner rows, M across the two boxes)
          const uint64_t ad = tr ? smem_desc(xa + kk * 2048, kXBox, 1024, kSwizzle128B)
                                 : smem_desc(xa + (kk >> 2) * kXBox + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(va + kk * 2048, kVBytes, 1024, kSwizzle128B);
          mma_bf16_ss_nc(d_tmem, ad, bd, idesc, (first && kk == 0) ? 0u : 1u);
        }
        first = false;
      }
      mma_commit_nc(&b.empty[stage]);
      if (++stage == kStages) { stage = 0; phase ^= 1; }
    }
    if (ok) mma_commit_nc(&b.acc_full);
    mma_commit(&b.drain);
    mbar_wait(&b.drain, 0, a.timeout_ns);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // One row per thread; the head's d_h <= 64 columns in two halves of 32 (unrolled, so
    // that every array stays in registers).
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;
    const int t = it.ob * 128 + lrow;
    const bool row_ok = t < a.T;
    // far older partners: the reduced scan term of the row (rows of far blocks only)
    const bool far = a.band >= 0 && (it.side == 0 ? it.ob >= a.band + 1 : it.ob <= a.nblk - a.band - 2);
    const size_t roff = ((size_t)it.b * a.T + (row_ok ? t : 0)) * a.dqk + (size_t)it.head * a.d_h;
    const __nv_bfloat16* raw = it.side == 0 ? a.raw_q : a.raw_k;
    const __nv_bfloat16* unit = it.side == 0 ? a.qhat : a.khat;
    const __nv_bfloat16* src = raw ? raw : unit;
    // the input row, as bf16 pairs, and its norm
    uint32_t up[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint4 x = make_uint4(0, 0, 0, 0);
      if (row_ok && 8 * k < a.d_h) x = *reinterpret_cast<const uint4*>(src + roff + 8 * k);
      up[4 * k] = x.x;
      up[4 * k + 1] = x.y;
      up[4 * k + 2] = x.z;
      up[4 * k + 3] = x.w;
    }
    float n2 = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float lo = bf16lo(up[k]), hi = bf16hi(up[k]);
      n2 = fmaf(lo, lo, fmaf(hi, hi, n2));
    }
    const float nrm = sqrtf(n2), inv_n = 1.f / fmaxf(nrm, 1e-12f);
    const float tau = head_tau(a.tau, a.s, it.head, a.err, kKernBackward);
    const float st = sqrtf(tau), inv_sqrt_dh = rsqrtf((float)a.d_h);
    const float fac = it.side == 0 ? st * expf(-tau) : st;
    const float* farp = far && row_ok ? a.far[it.side] + (((size_t)it.b * a.T + t) * a.H + it.head) * a.d_h : nullptr;
    bool ok = wait_bar(&b.acc_full, 0, b, a);
    if (ok) {
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
      float gv[64];
      float pr = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32], o[32];
        tmem_ld32(trow + 32 * h, w);
        if (any_old) tmem_ld32(trow + 64 + 32 * h, o);
        tmem_ld_wait();
        if (!any_old) {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        if (farp && 32 * h < a.d_h) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (32 * h + 4 * k < a.d_h) {
              const float4 f = *reinterpret_cast<const float4*>(farp + 32 * h + 4 * k);
              o[4 * k] = __float_as_uint(__uint_as_float(o[4 * k]) + f.x);
              o[4 * k + 1] = __float_as_uint(__uint_as_float(o[4 * k + 1]) + f.y);
              o[4 * k + 2] = __float_as_uint(__uint_as_float(o[4 * k + 2]) + f.z);
              o[4 * k + 3] = __float_as_uint(__uint_as_float(o[4 * k + 3]) + f.w);
            }
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int cc = 32 * h + c;
          const float u = (cc & 1) ? bf16hi(up[cc >> 1]) : bf16lo(up[cc >> 1]);
          const float uh = raw ? u * inv_n : u;
          float gg = __uint_as_float(w[c]);
          if (any_old || far) gg = fmaf(fac * dphi(st * uh, a.phi_mode, inv_sqrt_dh), __uint_as_float(o[c]), gg);
          gv[cc] = cc < a.d_h ? gg : 0.f;
          pr = fmaf(uh, gv[cc], pr);
        }
      }
      if (row_ok) {
        __nv_bfloat16* out = (it.side == 0 ? a.dq : a.dk) + roff;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (8 * k < a.d_h) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float y0 = gv[8 * k + 2 * e], y1 = gv[8 * k + 2 * e + 1];
              if (raw) {
                const float u0 = bf16lo(up[4 * k + e]), u1 = bf16hi(up[4 * k + e]);
                y0 = nrm < 1e-12f ? y0 * 1e12f : (y0 - u0 * inv_n * pr) * inv_n;
                y1 = nrm < 1e-12f ? y1 * 1e12f : (y1 - u1 * inv_n * pr) * inv_n;
              }
              pk[e] = pack_bf16x2(y0, y1);
            }
            *reinterpret_cast<uint4*>(out + 8 * k) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}
}  // namespace qkk

// ---------------------------------------------------------------- far older pairs (WANGO)
// agg_bwd_scan_kernel: the feature-map gradients of the older pairs that lie wholly
// outside the band of blocks that hold window pairs, through running sums (eq. 10 taken
// backwards) instead of pair by pair.  With d_max = ceil((W - 1) / 128), destination block
// ib sees source blocks jb <= ib - d_max - 1 only as older pairs ("far"):
//   forward  (dir 0):  S = sum_{far j} Fk_j g_j^T,   Y_i = E_i S   (d_h per row: sum_c)
//   reverse  (dir 1):  R = sum_{far i} Fq_i E_i^T,   Y_j = g_j R
// so that dFq_i (far) = Y_i - D_i z and dFk_j (far) = Y_j - rho (z, rho: plain sums over
// the far blocks).  One CTA per (dir, batch, head, strip of 256, 384 or 512 columns): the
// state's transpose (strip x 64, f32) lives in TMEM as up to four 128-row chunks; each
// active step adds one block to it (M = 128 strip columns per chunk, N = 64, K = 128 rows,
// both operands MN-major), copies it as bf16 to shared memory, and contracts one block
// with it (M = 128 rows, N = 64, K = the strip: the block's E or G rows K-major, the state
// MN-major).  Y goes to a per-strip partial buffer [strips, B * T, H, d_h]; a reduction
// kernel sums the strips and takes off the plain sums, and the dq/dk kernel adds the
// result.
// Vectors are read as 64-column boxes from the head's first column (at d_h < 64 the extra
// columns are other heads' and land in unread columns).
namespace scan {
constexpr int kThreads = 192;          // warp 0 TMA, warp 1 MMA and TMEM, warps 2-5 epilogue
constexpr int kNS = 512;               // the widest strip (columns); launches pick 512, 384 or 256
constexpr int kStages = 4;
constexpr uint32_t kBox = 128 * 64 * 2;       // 16 KB: 128 rows x 64 columns
constexpr uint32_t kStage = 2 * kBox;         // 32 KB
constexpr uint32_t kSB = kNS * 64 * 2;        // 64 KB: the state in bf16, [512 c][64 d]
struct __align__(8) Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t vec_full, vec_empty;           // the update's 128 x 64 vector tile
  uint64_t st_full;                        // the update's MMAs are done
  uint64_t sb_full, sb_empty;              // the bf16 state copy / its last reader is done
  uint64_t y_full, y_empty;
  uint64_t drain, never;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = 1024 + kStages * kStage + kBox + kSB + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
  int B, T, H, dqk, d_h, m_h, nblk, d_max, n_strips, n_act;
  int ns;           // strip columns, a multiple of 128 <= kNS
  float* part[2];   // [n_strips, B * T, H, d_h] per direction
  unsigned* err;
  uint64_t timeout_ns;
  int debug_timeout;  // test hook: the MMA issuer first waits on a barrier nothing signals
};

__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernBackward);
  return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (mbar_try_wait_nc(smem_u32(bar), parity)) return true;
  return wait_slow(bar, parity, b, a);
}

// Blocks of active step s: the one added to the state and the one contracted with it.
__device__ __forceinline__ void step_blocks(const Args& a, int dir, int s, int& ub, int& cb) {
  if (dir == 0) {
    ub = s;
    cb = a.d_max + 1 + s;
  } else {
    ub = a.nblk - 1 - s;
    cb = a.nblk - a.d_max - 2 - s;
  }
}

// tmE, tmG: 4-D maps over E and g (box 64 columns x 128 rows); tmFq, tmFk: 3-D maps over
// the forward's feature maps (box 64 x 128).
__global__ void __launch_bounds__(kThreads, 1)
    agg_bwd_scan_kernel(const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmG,
                        const __grid_constant__ CUtensorMap tmFq, const __grid_constant__ CUtensorMap tmFk,
                        const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sRing = base;
  uint8_t* sVec = sRing + kStages * kStage;
  uint8_t* sSB = sVec + kBox;
  Bars& b = *reinterpret_cast<Bars*>(sSB + kSB);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // item: (dir, batch-head, strip)
  const int dir = blockIdx.x & 1;
  const int r = blockIdx.x >> 1;
  const int strip = r % a.n_strips, bh = r / a.n_strips;
  const int bb = bh / a.H, head = bh % a.H;
  const int c0 = strip * a.ns;
  const int nchunk = min(a.ns / 128, (a.m_h - c0 + 127) / 128);  // 128-column chunks of the strip

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b.full[s], 1);
      mbar_init(&b.empty[s], 1);
    }
    mbar_init(&b.vec_full, 1);
    mbar_init(&b.vec_empty, 1);
    mbar_init(&b.st_full, 1);
    mbar_init(&b.sb_full, 4);
    mbar_init(&b.sb_empty, 1);
    mbar_init(&b.y_full, 1);
    mbar_init(&b.y_empty, 4);
    mbar_init(&b.drain, 1);
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
  const uint32_t tmem = b.tmem_base;  // state chunks at columns [64 q, 64 q + 64), Y at 256
  const CUtensorMap* upd_map = dir == 0 ? &tmG : &tmE;   // the state's gate-side operand
  const CUtensorMap* vec_map = dir == 0 ? &tmFk : &tmFq;
  const CUtensorMap* con_map = dir == 0 ? &tmE : &tmG;   // the contracted block's rows

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    int mask = 0;
    uint32_t sph[kStages] = {0, 0, 0, 0};
    int vlast = -1;  // the step of the last vector tile issued
    bool ok = true;
    for (int s = 0; ok && s < a.n_act; ++s) {
      int ub, cb;
      step_blocks(a, dir, s, ub, cb);
      // the update: the vector tile, then the strip's chunks of the added block's rows
      if (!(ok = wait_bar(&b.vec_empty, (s & 1) ^ 1, b, a))) break;
      mbar_arrive_expect_tx(&b.vec_full, kBox);
      tma_load_3d(sVec, vec_map, &b.vec_full, head * a.d_h, ub * 128, bb);
      vlast = s;
      for (int q = 0; ok && q < nchunk; ++q) {
        if (!(ok = wait_bar(&b.empty[stage], phase ^ 1, b, a))) break;
        mbar_arrive_expect_tx(&b.full[stage], kStage);
        uint8_t* dst = sRing + stage * kStage;
        tma_load_4d(dst, upd_map, &b.full[stage], c0 + 128 * q, head, ub * 128, bb);
        tma_load_4d(dst + kBox, upd_map, &b.full[stage], c0 + 128 * q + 64, head, ub * 128, bb);
        mask |= 1 << stage;
        sph[stage] = phase;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      // the contraction: the contracted block's rows, 128 strip columns a stage
      for (int q = 0; ok && q < nchunk; ++q) {
        if (!(ok = wait_bar(&b.empty[stage], phase ^ 1, b, a))) break;
        mbar_arrive_expect_tx(&b.full[stage], kStage);
        uint8_t* dst = sRing + stage * kStage;
        tma_load_4d(dst, con_map, &b.full[stage], c0 + 128 * q, head, cb * 128, bb);
        tma_load_4d(dst + kBox, con_map, &b.full[stage], c0 + 128 * q + 64, head, cb * 128, bb);
        mask |= 1 << stage;
        sph[stage] = phase;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    // copies still in flight land before the CTA exits (also when the loop was cut short)
    for (int s = 0; s < kStages; ++s)
      if (mask & (1 << s)) mbar_wait(&b.full[s], sph[s], a.timeout_ns);
    if (vlast >= 0) mbar_wait(&b.vec_full, vlast & 1, a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    const uint32_t idesc_u = idesc_bf16_f32(128, 64, true, true);    // S^T (+)= A^T V
    const uint32_t idesc_c = idesc_bf16_f32(128, 64, false, true);   // Y = A S
    int stage = 0;
    uint32_t phase = 0;
    bool ok = !a.debug_timeout || wait_bar(&b.never, 0, b, a);  // nothing ever arrives there
    for (int s = 0; ok && s < a.n_act; ++s) {
      // the update: S^T[c, d] += sum_t A[t, c] V[t, d], chunk q of 128 columns; the previous
      // state copy has been read out (sb_full of step s - 1 was waited for below)
      if (!(ok = wait_bar(&b.vec_full, s & 1, b, a))) break;
      tc_fence_after_nc();
      const uint32_t va = smem_u32(sVec);
      for (int q = 0; ok && q < nchunk; ++q) {
        if (!(ok = wait_bar(&b.full[stage], phase, b, a))) break;
        tc_fence_after_nc();
        const uint32_t xa = smem_u32(sRing + stage * kStage);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ss_nc(tmem + 64 * q, smem_desc(xa + kk * 2048, kBox, 1024, kSwizzle128B),
                         smem_desc(va + kk * 2048, kBox, 1024, kSwizzle128B), idesc_u, (s | kk) != 0 ? 1u : 0u);
        mma_commit_nc(&b.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit_nc(&b.vec_empty);
      mma_commit_nc(&b.st_full);
      // the contraction, once the state is in shared memory and Y has been read out
      if (!(ok = wait_bar(&b.sb_full, s & 1, b, a))) break;
      if (s >= 1 && !(ok = wait_bar(&b.y_empty, (s - 1) & 1, b, a))) break;
      tc_fence_after_nc();
      const uint32_t sb = smem_u32(sSB);
      for (int q = 0; ok && q < nchunk; ++q) {
        if (!(ok = wait_bar(&b.full[stage], phase, b, a))) break;
        tc_fence_after_nc();
        const uint32_t xa = smem_u32(sRing + stage * kStage);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // K: the chunk's 128 columns, 16 at a time
          mma_bf16_ss_nc(tmem + 256, smem_desc(xa + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024, kSwizzle128B),
                         smem_desc(sb + (128 * q + 16 * kk) * 128, kSB, 1024, kSwizzle128B), idesc_c,
                         (q | kk) != 0 ? 1u : 0u);
        mma_commit_nc(&b.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit_nc(&b.sb_empty);
      mma_commit_nc(&b.y_full);
    }
    mma_commit(&b.drain);
    mbar_wait(&b.drain, 0, a.timeout_ns);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ state copy and output
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // a state row (strip column) per chunk; a Y row
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float* part = a.part[dir] + (size_t)strip * a.B * a.T * a.H * a.d_h;
    bool ok = true;
    for (int s = 0; ok && s < a.n_act; ++s) {
      int ub, cb;
      step_blocks(a, dir, s, ub, cb);
      // the state, as bf16 [c][d] in shared memory (128-byte swizzle), once the update is
      // done and the previous contraction has read the previous copy
      if (ok) ok = wait_bar(&b.st_full, s & 1, b, a);
      if (ok && s >= 1) ok = wait_bar(&b.sb_empty, (s - 1) & 1, b, a);
      if (!ok) break;
      tc_fence_after();
      for (int q = 0; q < 4; ++q) {
        uint32_t v[64];
        if (q < nchunk) {
          tmem_ld32(tmem + 64 * q + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(tmem + 64 * q + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_ld_wait();
        }
        const int c = 128 * q + row;
        const uint32_t rowaddr = smem_u32(sSB) + (uint32_t)c * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint4 o = make_uint4(0, 0, 0, 0);
          if (q < nchunk) {
            o.x = pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1]));
            o.y = pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3]));
            o.z = pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5]));
            o.w = pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7]));
          }
          st_shared_v4(rowaddr + (uint32_t)((k ^ (c & 7)) << 4), o);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.sb_full);
      // Y of the contracted block's rows to the strip's partial buffer
      if (ok) ok = wait_bar(&b.y_full, s & 1, b, a);
      if (!ok) break;
      tc_fence_after();
      uint32_t y[64];
      tmem_ld32(tmem + 256 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&y[0]));
      tmem_ld32(tmem + 256 + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&y[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.y_empty);
      const int t = cb * 128 + row;
      if (t < a.T) {
        float* dst = part + (((size_t)bb * a.T + t) * a.H + head) * a.d_h;
#pragma unroll
        for (int c = 0; c < 64; c += 4)
          if (c < a.d_h)
            *reinterpret_cast<float4*>(dst + c) = make_float4(__uint_as_float(y[c]), __uint_as_float(y[c + 1]),
                                                             __uint_as_float(y[c + 2]), __uint_as_float(y[c + 3]));
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
}  // namespace scan

// Per 128-row block, sum_i D_i Fq_i (Fq: the forward's bf16 feature map of q, e^-tau
// included), [B, H, nblk, d_h]: the reverse scan's rho in block sums.  grid (nblk, H, B),
// 128 threads, one row each.
__global__ void __launch_bounds__(128) bwd_rho_kernel(const __nv_bfloat16* __restrict__ fq,
                                                      const float* __restrict__ dp, float* __restrict__ rb, int T,
                                                      int T_pad, int H, int dqk, int nblk) {
  __shared__ float part[4][64];
  const int blk = blockIdx.x, head = blockIdx.y, bb = blockIdx.z, t = threadIdx.x;
  const int d_h = dqk / H, i = blk * 128 + t, lane = t & 31, wp = t >> 5;
  const float dpi = i < T ? dp[(size_t)(bb * H + head) * T_pad + i] : 0.f;
  for (int c = 0; c < d_h; ++c) {
    float v = i < T ? dpi * __bfloat162float(fq[((size_t)bb * T + i) * dqk + head * d_h + c]) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) part[wp][c] = v;
  }
  __syncthreads();
  if (t < d_h) rb[(((size_t)bb * H + head) * nblk + blk) * d_h + t] = (part[0][t] + part[1][t]) + (part[2][t] + part[3][t]);
}

// The plain far sums: fb[0] per destination block ob, sum of zb over source blocks
// < ob - band; fb[1] per source block ob, sum of rb over destination blocks > ob + band.
// grid (B * H, 2 sides), one thread per column (d_h <= 64); the block sums are read 8 at
// a time ahead of the running sum.
__global__ void __launch_bounds__(64) bwd_far_base_kernel(const float* __restrict__ zb, const float* __restrict__ rb,
                                                          float* __restrict__ fb, int n_bh, int nblk, int d_h,
                                                          int band) {
  const int bh = blockIdx.x, side = blockIdx.y, c = threadIdx.x;
  if (c >= d_h) return;
  const size_t o = (size_t)bh * nblk * d_h + c;
  const float* src = (side == 0 ? zb : rb) + o;
  float* dst = fb + (size_t)side * n_bh * nblk * d_h + o;
  float run = 0.f;
  for (int s0 = 0; s0 < nblk; s0 += 8) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int blk = side == 0 ? s0 + u : nblk - 1 - (s0 + u);   // the block whose sum is written
      const int from = side == 0 ? blk - band - 1 : blk + band + 1;  // the block it newly takes in
      x[u] = (s0 + u < nblk && from >= 0 && from < nblk) ? src[(size_t)from * d_h] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (s0 + u < nblk) {
        run += x[u];
        dst[(size_t)(side == 0 ? s0 + u : nblk - 1 - (s0 + u)) * d_h] = run;
      }
    }
  }
}

// far[side] (strip 0 of part[side], in place) = sum over strips - the plain far sum
// (times D_i on the dq side), for rows of far blocks; 4 columns a thread, grid (n4 / 256,
// 2 sides).
__global__ void __launch_bounds__(256) bwd_far_sum_kernel(float* part0, float* part1, const float* __restrict__ fb,
                                                          const float* __restrict__ dp, long long n4, int T,
                                                          int T_pad, int H, int n_bh, int d_h, int nblk, int band,
                                                          int n_strips, long long stride) {
  const int side = blockIdx.y;
  float* part = side == 0 ? part0 : part1;
  const int hd4 = H * d_h / 4, d4 = d_h / 4;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n4; e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / hd4;
    const int rem = (int)(e - row * hd4), head = rem / d4, c = 4 * (rem - head * d4);
    const int bb = (int)(row / T), t = (int)(row - (long long)bb * T), ob = t >> 7;
    if (side == 0 ? ob < band + 1 : ob > nblk - band - 2) continue;
    const float* src = part + 4 * e;
    float4 acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    int sp = 0;
    for (; sp + 4 <= n_strips; sp += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 x = *reinterpret_cast<const float4*>(src + (sp + u) * stride);
        acc[u].x += x.x; acc[u].y += x.y; acc[u].z += x.z; acc[u].w += x.w;
      }
    }
    for (; sp < n_strips; ++sp) {
      const float4 x = *reinterpret_cast<const float4*>(src + sp * stride);
      acc[0].x += x.x; acc[0].y += x.y; acc[0].z += x.z; acc[0].w += x.w;
    }
    const int bh = bb * H + head;
    const float4 f = *reinterpret_cast<const float4*>(fb + (((size_t)side * n_bh + bh) * nblk + ob) * d_h + c);
    const float sc = side == 0 ? dp[(size_t)bh * T_pad + t] : 1.f;
    float4 r;
    r.x = (acc[0].x + acc[1].x) + (acc[2].x + acc[3].x) - sc * f.x;
    r.y = (acc[0].y + acc[1].y) + (acc[2].y + acc[3].y) - sc * f.y;
    r.z = (acc[0].z + acc[1].z) + (acc[2].z + acc[3].z) - sc * f.z;
    r.w = (acc[0].w + acc[1].w) + (acc[2].w + acc[3].w) - sc * f.w;
    *reinterpret_cast<float4*>(part + 4 * e) = r;
  }
}

// The current device's SM count; without a device (a size query on a host with no GPU)
// the GB300's 152.
int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  return n > 0 ? n : 152;
}

template <int DH>
cudaError_t launch_dh(const CUtensorMap& mE, const CUtensorMap& mG, const CUtensorMap& mK, const Args& a,
                      cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(agg_bwd_pairs_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = a.n_tiles < num_sms() ? a.n_tiles : num_sms();
  agg_bwd_pairs_kernel<DH><<<grid, kThreads, kSmemBytes, s>>>(mE, mG, mK, a);
  return cudaGetLastError();
}

}  // namespace

int bwd_tpad(int T) { return ceil_div(T, 128) * 128; }
// Strip width: the one of 512, 384, 256 columns with the fewest chunk-steps per SM
// (waves of one-CTA-per-SM items times chunks per strip); the widest on a tie (fewer
// partial sums).
int bwd_scan_ns(int B, int H, int m_h) {
  int best = scan::kNS;
  long long best_cost = -1;
  for (int ns = scan::kNS; ns >= 256; ns -= 128) {
    const long long items = 2LL * B * H * ceil_div(m_h, ns);
    const long long cost = (items + num_sms() - 1) / num_sms() * (ns / 128);
    if (best_cost < 0 || cost < best_cost) {
      best = ns;
      best_cost = cost;
    }
  }
  return best;
}
int bwd_scan_strips(int B, int H, int m_h) { return ceil_div(m_h, bwd_scan_ns(B, H, m_h)); }
int bwd_band(int window) { return (window + 126) / 128; }

// Estimated costs: the far older pairs as 128 x 256 pair tiles of K = m_h at the pair
// kernel's measured ~1.1 PFLOP/s, against the scans' serial chain of n_act steps (about
// 2.25 us per 128-column chunk of a strip, one CTA per SM) plus the strip reduction.
bool bwd_scan_pays(int B, int T, int H, int dqk, int m_h, int window) {
  const int nblk = bwd_tpad(T) / 128, band = bwd_band(window), n_act = nblk - band - 1;
  if (n_act <= 0) return false;
  long long old_tiles = 0;
  for (int ib = 0; ib < nblk; ++ib) old_tiles += jt_lo_of(ib, band);
  const double pairs_s = (double)B * H * old_tiles * 2.0 * 128 * 256 * m_h / 1.1e15;
  const int ns = bwd_scan_ns(B, H, m_h), strips = ceil_div(m_h, ns);
  const double items = 2.0 * B * H * strips, sms = num_sms();
  const double chunks = ceil_div(m_h < ns ? m_h : ns, 128);
  const double scan_s = ceil(items / sms) * n_act * chunks * 2.25e-6 + 2.0 * 2.0 * strips * B * T * dqk * 4 / 6e12;
  return scan_s < pairs_s;
}

cudaError_t launch_bwd_scan(const BwdScanArgs& p, cudaStream_t s) {
  scan::Args a = {};
  a.B = p.B; a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.d_h = p.dqk / p.H; a.m_h = p.m_h;
  a.nblk = bwd_tpad(p.T) / 128;
  a.d_max = bwd_band(p.window);
  a.ns = bwd_scan_ns(p.B, p.H, p.m_h);
  a.n_strips = ceil_div(p.m_h, a.ns);
  a.n_act = a.nblk - a.d_max - 1;
  a.part[0] = p.part[0];
  a.part[1] = p.part[1];
  a.err = p.err;
  a.debug_timeout = p.debug_timeout;
  a.timeout_ns = p.debug_timeout ? 1000000ull : 2000000000ull;
  if (a.n_act <= 0) return cudaSuccess;  // no block is wholly beyond the band
  // the block sums of D_i Fq_i for rho
  bwd_rho_kernel<<<dim3(a.nblk, p.H, p.B), 128, 0, s>>>(static_cast<const __nv_bfloat16*>(p.fq), p.dp, p.rb, p.T,
                                                        bwd_tpad(p.T), p.H, p.dqk, a.nblk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int m_hp = p.m / p.H;
  CUtensorMap mE, mG, mFq, mFk;
  e = make_tmap_4d_heads(&mE, p.E, p.B, p.T, p.H, p.m_h, m_hp, 128, 64);
  if (e == cudaSuccess) e = make_tmap_4d_heads(&mG, p.g, p.B, p.T, p.H, p.m_h, m_hp, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mFq, p.fq, p.B, p.T, p.dqk, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mFk, p.fk, p.B, p.T, p.dqk, 128, 64);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(scan::agg_bwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)scan::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long items = 2LL * p.B * p.H * a.n_strips;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  scan::agg_bwd_scan_kernel<<<(unsigned)items, scan::kThreads, scan::kSmemBytes, s>>>(mE, mG, mFq, mFk, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the plain far sums, then the strips summed into strip 0 less them
  const int n_bh = p.B * p.H;
  bwd_far_base_kernel<<<dim3(n_bh, 2), 64, 0, s>>>(p.zb, p.rb, p.fb, n_bh, a.nblk, a.d_h, a.d_max);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n4 = (long long)p.B * p.T * p.dqk / 4;
  const long long want = (n4 + 255) / 256, cap = 16LL * num_sms();
  bwd_far_sum_kernel<<<dim3((unsigned)(want < cap ? want : cap), 2), 256, 0, s>>>(
      p.part[0], p.part[1], p.fb, p.dp, n4, p.T, bwd_tpad(p.T), p.H, n_bh, a.d_h, a.nblk, a.d_max, a.n_strips,
      (long long)p.B * p.T * p.dqk);
  return cudaGetLastError();
}

cudaError_t launch_bwd_qk_tc(const BwdQKTcArgs& p, cudaStream_t s) {
  qkk::Args a = {};
  a.B = p.B; a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.d_h = p.dqk / p.H;
  a.T_pad = bwd_tpad(p.T);
  a.nblk = a.T_pad / 128;
  a.n_bh = p.B * p.H;
  a.wango = p.wango; a.window = p.window; a.phi_mode = p.phi_mode;
  a.s = p.s; a.tau = p.tau;
  a.qhat = static_cast<const __nv_bfloat16*>(p.qhat);
  a.khat = static_cast<const __nv_bfloat16*>(p.khat);
  a.raw_q = static_cast<const __nv_bfloat16*>(p.raw_q);
  a.raw_k = static_cast<const __nv_bfloat16*>(p.raw_k);
  a.dq = static_cast<__nv_bfloat16*>(p.dq);
  a.dk = static_cast<__nv_bfloat16*>(p.dk);
  a.band = p.band;
  a.far[0] = p.far[0];
  a.far[1] = p.far[1];
  a.err = p.err;
  a.debug_timeout = p.debug_timeout;
  a.timeout_ns = p.debug_timeout ? 1000000ull : 2000000000ull;
  const long long items = 2LL * a.n_bh * a.nblk;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap mX, mXo, mQ, mK, mFq, mFk;
  const uint64_t BH = (uint64_t)p.B * p.H;
  cudaError_t e = make_tmap_3d(&mX, p.X, BH, a.T_pad, a.T_pad, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mXo, p.X_old ? p.X_old : p.X, BH, a.T_pad, a.T_pad, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mQ, p.qhat, p.B, p.T, p.dqk, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mK, p.khat, p.B, p.T, p.dqk, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mFq, p.fq ? p.fq : p.qhat, p.B, p.T, p.dqk, 128, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mFk, p.fk ? p.fk : p.khat, p.B, p.T, p.dqk, 128, 64);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qkk::agg_bwd_qk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)qkk::kSmemBytes);
  if (e != cudaSuccess) return e;
  qkk::agg_bwd_qk_kernel<<<(unsigned)items, qkk::kThreads, qkk::kSmemBytes, s>>>(mX, mXo, mQ, mK, mFq, mFk, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pairs_tc(const BwdPairsArgs& p, cudaStream_t s) {
  Args a = {};
  a.B = p.B; a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.d_h = p.dqk / p.H;
  a.T_pad = bwd_tpad(p.T);
  const int m_hp = p.m / p.H, m_h = p.m_h ? p.m_h : m_hp;
  const int n_iblk = a.T_pad / BM;
  a.band = p.band;
  int per = 0;
  for (int ib = 0; ib < n_iblk; ++ib) per += ib / 2 - jt_lo_of(ib, p.band) + 1;
  a.tiles_per_bh = per;
  const long long nt = (long long)p.B * p.H * per;
  if (nt > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_tiles = (int)nt;
  a.nkb = ceil_div(m_h, BK);
  a.wango = p.wango;
  a.window = p.window;
  a.s = p.s;
  a.tau = p.tau;
  a.qhat = static_cast<const __nv_bfloat16*>(p.qhat);
  a.dp = p.dp;
  a.X = static_cast<__nv_bfloat16*>(p.X);
  a.X_old = static_cast<__nv_bfloat16*>(p.X_old);
  a.err = p.err;
  a.debug_timeout = p.debug_timeout;
  a.timeout_ns = p.debug_timeout ? 1000000ull : 2000000000ull;
  CUtensorMap mE, mG, mK;
  cudaError_t e = make_tmap_4d_heads(&mE, p.E, p.B, p.T, p.H, m_h, m_hp, BM, BK);
  if (e == cudaSuccess) e = make_tmap_4d_heads(&mG, p.g, p.B, p.T, p.H, m_h, m_hp, BN, BK);
  if (e == cudaSuccess) e = make_tmap_3d(&mK, p.khat, p.B, p.T, p.dqk, 128, a.d_h);
  if (e != cudaSuccess) return e;
  if (a.d_h == 64) return launch_dh<64>(mE, mG, mK, a, s);
  if (a.d_h == 32) return launch_dh<32>(mE, mG, mK, a, s);
  if (a.d_h == 16) return launch_dh<16>(mE, mG, mK, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace tg
