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
// in bf16 to X [B*H, T_pad, T_pad].  X then gives dqhat = X Khat and dkhat = X^T Qhat
// (window pairs) and the feature-map gradients (older pairs).  The weights use the
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
  __nv_bfloat16* X;           // [B * H, T_pad, T_pad]
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
      __nv_bfloat16* xrow = a.X + ((size_t)(tl.b * a.H + tl.head) * a.T_pad + i) * a.T_pad;
      {
#pragma unroll 1
        for (int cbase = 0; cbase < 128; cbase += 32) {
          uint32_t r[32];
          tmem_ld32(trow + cbase, r);
          tmem_ld_wait();
          if (cbase == 96) {  // the accumulator is free for the tile after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.acc_empty[acc]);
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int jl = half * 128 + cbase + e + h;  // source within the tile
              const int j = jbase + cbase + e + h;
              float x = 0.f;
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
                  x = dl;
                }
              }
              x2[h] = x;
            }
            pk[e / 2] = pack_bf16x2(x2[0], x2[1]);
          }
          if (jbase + cbase < a.T_pad) {  // 32 whole columns inside the padded matrix
#pragma unroll
            for (int k = 0; k < 4; ++k)
              st_global_v4(xrow + jbase + cbase + 8 * k, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
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

cudaError_t launch_bwd_pairs_tc(const BwdPairsArgs& p, cudaStream_t s) {
  Args a = {};
  a.B = p.B; a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.d_h = p.dqk / p.H;
  a.T_pad = bwd_tpad(p.T);
  const int m_h = p.m / p.H;
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
  a.err = p.err;
  a.timeout_ns = 2000000000ull;
  CUtensorMap mE, mG, mK;
  cudaError_t e = make_tmap_4d_heads(&mE, p.E, p.B, p.T, p.H, m_h, BM, BK);
  if (e == cudaSuccess) e = make_tmap_4d_heads(&mG, p.g, p.B, p.T, p.H, m_h, BN, BK);
  if (e == cudaSuccess) e = make_tmap_3d(&mK, p.khat, p.B, p.T, p.dqk, 128, a.d_h);
  if (e != cudaSuccess) return e;
  if (a.d_h == 64) return launch_dh<64>(mE, mG, mK, a, s);
  if (a.d_h == 32) return launch_dh<32>(mE, mG, mK, a, s);
  if (a.d_h == 16) return launch_dh<16>(mE, mG, mK, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace tg
