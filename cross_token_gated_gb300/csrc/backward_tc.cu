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
  uint64_t key_full, key_empty, drain;
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
  unsigned* err;
  uint64_t timeout_ns;
};

struct Tile {
  int b, head, ib, jt;
};

// Tiles of one (batch, head): destination blocks ib in order, and for each the
// 256-source tiles jt = 0 .. ib / 2 (every tile holding a pair j <= i).
__device__ __forceinline__ Tile tile_of(const Args& a, int t) {
  Tile r;
  const int bh = t / a.tiles_per_bh;
  int rem = t % a.tiles_per_bh, ib = 0;
  while (rem >= ib / 2 + 1) {
    rem -= ib / 2 + 1;
    ++ib;
  }
  r.b = bh / a.H;
  r.head = bh % a.H;
  r.ib = ib;
  r.jt = rem;
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
    bool ok = true;
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
  uint64_t full[kStages], empty[kStages], acc_full, drain;
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
  unsigned* err;
  uint64_t timeout_ns;
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
  it.p_lo = it.side == 0 ? 0 : it.ob;
  it.n_steps = it.side == 0 ? it.ob + 1 : a.nblk - it.ob;
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
    bool ok = true, first_w = true, first_o = true;
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
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;
    const int t = it.ob * 128 + lrow;
    const bool row_ok = t < a.T;
    bool ok = wait_bar(&b.acc_full, 0, b, a);
    if (ok) {
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
      uint32_t w[64], o[64];
      tmem_ld32(trow, *reinterpret_cast<uint32_t(*)[32]>(&w[0]));
      tmem_ld32(trow + 32, *reinterpret_cast<uint32_t(*)[32]>(&w[32]));
      if (any_old) {
        tmem_ld32(trow + 64, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_ld32(trow + 96, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
      }
      tmem_ld_wait();
      if (row_ok) {
        const float tau = head_tau(a.tau, a.s, it.head, a.err, kKernBackward);
        const float st = sqrtf(tau), inv_sqrt_dh = rsqrtf((float)a.d_h);
        const float fac = it.side == 0 ? st * expf(-tau) : st;
        const size_t roff = ((size_t)it.b * a.T + t) * a.dqk + (size_t)it.head * a.d_h;
        const __nv_bfloat16* raw = it.side == 0 ? a.raw_q : a.raw_k;
        const __nv_bfloat16* unit = it.side == 0 ? a.qhat : a.khat;
        const __nv_bfloat16* src = raw ? raw : unit;
        float u[64], g[64];
        float n2 = 0.f;
        for (int c = 0; c < a.d_h; ++c) {
          u[c] = __bfloat162float(src[roff + c]);
          n2 = fmaf(u[c], u[c], n2);
        }
        const float nrm = sqrtf(n2), inv_n = 1.f / fmaxf(nrm, 1e-12f);
        float pr = 0.f;
        for (int c = 0; c < a.d_h; ++c) {
          const float uh = raw ? u[c] * inv_n : u[c];
          float gg = __uint_as_float(w[c]);
          if (any_old) gg = fmaf(fac * dphi(st * uh, a.phi_mode, inv_sqrt_dh), __uint_as_float(o[c]), gg);
          g[c] = gg;
          u[c] = uh;
          pr = fmaf(uh, gg, pr);
        }
        __nv_bfloat16* out = (it.side == 0 ? a.dq : a.dk) + roff;
        for (int c = 0; c < a.d_h; ++c) {
          float y = g[c];
          if (raw) y = nrm < 1e-12f ? y * 1e12f : (y - u[c] * pr) * inv_n;
          out[c] = __float2bfloat16_rn(y);
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

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
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
  a.err = p.err;
  a.timeout_ns = 2000000000ull;
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
  int per = 0;
  for (int ib = 0; ib < n_iblk; ++ib) per += ib / 2 + 1;
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
  a.timeout_ns = 2000000000ull;
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
