// Tensor-core (tcgen05) GEMMs of one block, "TANGO: Token-Aggregated Nonlinear
// Gating Operators ...", sec. 2.1:
//   projection  [q | k | g | v] = x [W_q | W_k | W_g | W_v]^T      (eq. 2)
//               epilogues: RoPE then unit norm per head (q, k), SiLU (g), none (v)
//   output      h_out = h + u W_o^T                                 (eq. 3)
//   plain       C = A B^T, bf16 out (the tied-embedding logits of sec. 2.3)
//
// C[M, N] = A[M, K] * B[N, K]^T with both operands K-major bf16, fp32 accumulation
// in tensor memory.  Persistent kernel, one CTA per SM, warp-specialised:
//   warp 0      TMA producer (4-stage ring of 128x64 A and 256x64 B tiles, 128B swizzle);
//               in the output GEMM it also asks u's box 8 k-blocks ahead into L2
//   warp 1      TMEM allocator and MMA issuer (128x256x16 tcgen05.mma, one thread)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, fused elementwise, bf16 out:
//               g and v through shared memory and TMA stores (64-column chunks,
//               L2 evict-first),
//               q/k (RoPE angles in fp32 with an exact turn reduction) and the
//               residual output by direct stores
// The two 256-column accumulators in TMEM let the epilogue of one tile overlap the
// main loop of the next.  Every wait is bounded; on expiry the kernel records a
// timeout in the error word and all roles leave their loops.  A test hook
// (debug_timeout) makes the MMA issuer wait first on a barrier that nothing signals,
// with a 1 ms bound, to exercise that path.
#include <math.h>

#include "tg_common.cuh"
#include "tg_ptx.cuh"
#include "tg_tc.h"
#include "tg_tma.h"

namespace tg {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;  // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kOutBytes = BM * 64 * 2;  // 16 KB: one 128 x 64 bf16 output chunk (staging for TMA)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kPrefetch = 8;  // output GEMM: u boxes asked into L2 this many k-blocks ahead

enum Seg : int { kSegQK = 0, kSegG = 1, kSegV = 2, kSegOut = 3 };

struct GemmArgs {
  int M, K;
  int n_mblk;         // ceil(M / 128)
  int nb_qk, nb_g, nb_v, nb_out;  // n-blocks per segment (projection: 1, g, g, 0; output: 0, 0, 0, n)
  int m_major;        // tile order: 1 = m-block outer (output GEMM), 0 = n-block outer
  int T, H, dqk, m, d;
  // RoPE frequencies over pi, base^(-2c/d_h) / pi, as float pairs hi + lo
  float rope_hi[32], rope_lo[32];
  int rope;
  __nv_bfloat16 *q, *k, *g, *v;
  const __nv_bfloat16* h;
  __nv_bfloat16* h_out;
  unsigned* err;
  uint64_t timeout_ns;  // bound of every wait
  int debug_timeout;    // test hook: the MMA issuer first waits on a barrier nothing signals
};

struct __align__(8) Bars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain, never;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + kStages * (kABytes + kBBytes) + 2 * kOutBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Tile {
  int seg, nb, mb;
};

__device__ __forceinline__ Tile tile_of(const GemmArgs& a, int t) {
  const int nb_total = a.nb_qk + a.nb_g + a.nb_v + a.nb_out;
  int nb, mb;
  if (a.m_major) {
    mb = t / nb_total;
    nb = t % nb_total;
  } else {
    nb = t / a.n_mblk;
    mb = t % a.n_mblk;
  }
  Tile r;
  r.mb = mb;
  if (nb < a.nb_qk) {
    r.seg = kSegQK; r.nb = nb;
  } else if ((nb -= a.nb_qk) < a.nb_g) {
    r.seg = kSegG; r.nb = nb;
  } else if ((nb -= a.nb_g) < a.nb_v) {
    r.seg = kSegV; r.nb = nb;
  } else {
    r.seg = kSegOut; r.nb = nb - a.nb_v;
  }
  return r;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const GemmArgs& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernGemm);
  return false;
}

// SiLU(x) = x * sigmoid(x) = 0.5 x (1 + tanh(x / 2))
__device__ __forceinline__ float silu(float x) { return 0.5f * x * (1.f + tanh_approx(0.5f * x)); }

// One head of the q/k epilogue: RoPE at position t (rotate-half pairs), then unit
// normalisation, for a row held by one thread.
// The TMEM loads are warp-collective, so every lane runs them; only lanes with
// `valid` rows store.
template <int DH>
__device__ __forceinline__ void rope_norm_store(uint32_t taddr, __nv_bfloat16* dst, int t, bool valid,
                                                const GemmArgs& a) {
  float x[DH];
#pragma unroll
  for (int c0 = 0; c0 < DH; c0 += 16) {
    uint32_t r[16];
    tmem_ld16(taddr + c0, r);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 16; ++c) x[c0 + c] = __uint_as_float(r[c]);
  }
  if (a.rope) {
#pragma unroll
    for (int c = 0; c < DH / 2; ++c) {
      // angle / pi = t (hi + lo).  t * hi is kept exactly as its rounded product p plus
      // the product's error pe; whole turns (even multiples) leave p exactly; sincospi
      // then sees the angle to fp32 precision at any position t < 2^24
      const float tf = (float)t, p = tf * a.rope_hi[c];
      const float pe = fmaf(tf, a.rope_hi[c], -p);
      const float turn = (p - 2.f * rintf(0.5f * p)) + (pe + tf * a.rope_lo[c]);
      float sn, cs;
      sincospif(turn, &sn, &cs);
      const float x1 = x[c], x2 = x[c + DH / 2];
      x[c] = x1 * cs - x2 * sn;
      x[c + DH / 2] = x1 * sn + x2 * cs;
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < DH; ++c) ss = fmaf(x[c], x[c], ss);
  const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
  if (!valid) return;
#pragma unroll
  for (int c = 0; c < DH; c += 8)
    st_global_v4(dst + c, pack_bf16x2(x[c] * inv, x[c + 1] * inv), pack_bf16x2(x[c + 2] * inv, x[c + 3] * inv),
                 pack_bf16x2(x[c + 4] * inv, x[c + 5] * inv), pack_bf16x2(x[c + 6] * inv, x[c + 7] * inv));
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmOG,
                   const __grid_constant__ CUtensorMap tmOV, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kStages * kABytes;
  uint8_t* sOut = sB + kStages * kBBytes;  // two output chunks staged for TMA stores
  Bars& b = *reinterpret_cast<Bars*>(sOut + 2 * kOutBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ntiles = a.n_mblk * (a.nb_qk + a.nb_g + a.nb_v + a.nb_out);
  const int nkb = (a.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b.full[s], 1);
      mbar_init(&b.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.acc_full[i], 1);
      mbar_init(&b.acc_empty[i], 4);
    }
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
    tma_prefetch_desc(&tmA);
    int stage = 0;
    uint32_t phase = 0;
    int issued_mask = 0;
    uint32_t issued_phase[kStages] = {};
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = tile_of(a, t);
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_bar(&b.empty[stage], phase ^ 1, b, a)) goto producer_done;
        uint8_t* dA = sA + stage * kABytes;
        uint8_t* dB = sB + stage * kBBytes;
        const int k0 = kb * BK;
        if (tl.seg == kSegQK && a.nb_qk == 1) {  // q and k rows in one tile (2 d_qk <= 256)
          mbar_arrive_expect_tx(&b.full[stage], kABytes + 2u * a.dqk * 128u);
          tma_load_2d(dB, &tmB0, &b.full[stage], k0, 0);
          tma_load_2d(dB + a.dqk * 128, &tmB1, &b.full[stage], k0, 0);
        } else if (tl.seg == kSegQK) {  // 256 rows of W_q (first half of the n-blocks) or W_k
          const int nq = a.nb_qk / 2;
          mbar_arrive_expect_tx(&b.full[stage], kABytes + kBBytes);
          tma_load_2d(dB, tl.nb < nq ? &tmB0 : &tmB1, &b.full[stage], k0, (tl.nb % nq) * BN);
        } else {
          mbar_arrive_expect_tx(&b.full[stage], kABytes + kBBytes);
          const CUtensorMap* mb = tl.seg == kSegG ? &tmB2 : tl.seg == kSegV ? &tmB3 : &tmB0;
          tma_load_2d(dB, mb, &b.full[stage], k0, tl.nb * BN);
        }
        tma_load_2d(dA, &tmA, &b.full[stage], k0, tl.mb * BM);
        // u comes from HBM, further ahead than the 4 stages reach: ask for it into L2 early
        if (tl.seg == kSegOut && kb + kPrefetch < nkb) tma_prefetch_l2_2d(&tmA, k0 + kPrefetch * BK, tl.mb * BM);
        issued_mask |= 1 << stage;
        issued_phase[stage] = phase;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
  producer_done:
    // Copies still in flight must land before the CTA exits.
    for (int s = 0; s < kStages; ++s)
      if (issued_mask & (1 << s)) mbar_wait(&b.full[s], issued_phase[s], kTimeoutNs);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    const bool hooked = a.debug_timeout && !wait_bar(&b.never, 0, b, a);  // nothing ever arrives there
    for (int t = blockIdx.x; !hooked && t < ntiles; t += gridDim.x) {
      const Tile tl = tile_of(a, t);
      const int N = (tl.seg == kSegQK && a.nb_qk == 1) ? 2 * a.dqk : BN;
      const uint32_t idesc = idesc_bf16_f32(BM, N, false, false);
      if (!wait_bar(&b.acc_empty[acc], acc_phase ^ 1, b, a)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_bar(&b.full[stage], phase, b, a)) { ok = false; break; }
        tc_fence_after();
        const uint32_t aaddr = smem_u32(sA + stage * kABytes), baddr = smem_u32(sB + stage * kBBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = smem_desc(aaddr + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(baddr + kk * 32, 16, 1024, kSwizzle128B);
          mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0);
        }
        mma_commit(&b.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit(&b.acc_full[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    mma_commit(&b.drain);
    mbar_wait(&b.drain, 0, kTimeoutNs);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. 32*quarter+31
    const int lrow = quarter * 32 + lane;  // row of the tile
    const bool issuer = warp == 2 && lane == 0;
    int acc = 0, ob = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = tile_of(a, t);
      bool ok = wait_bar(&b.acc_full[acc], acc_phase, b, a);
      // the four epilogue warps agree (they meet at named barriers below)
      if (!named_bar_and(1, 128, ok)) break;
      tc_fence_after();
      const int row = tl.mb * BM + quarter * 32 + lane;
      const uint32_t trow = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
      if (tl.seg == kSegQK) {
        const bool valid = row < a.M;
        const int d_h = a.dqk / a.H, t_pos = valid ? row % a.T : 0;
        // the tile's heads: all q then all k heads (one tile), or 256 / d_h heads of q or k
        const int nheads = a.nb_qk == 1 ? 2 * a.H : BN / d_h;
        const int nq = a.nb_qk / 2;
        for (int hh = 0; hh < nheads; ++hh) {
          const bool is_q = a.nb_qk == 1 ? hh < a.H : tl.nb < nq;
          const int head = a.nb_qk == 1 ? hh % a.H : (tl.nb % nq) * (BN / d_h) + hh;
          __nv_bfloat16* dst = (is_q ? a.q : a.k) + (size_t)(valid ? row : 0) * a.dqk + head * d_h;
          const uint32_t col = (uint32_t)(a.nb_qk == 1 ? (is_q ? 0 : a.dqk) + head * d_h : hh * d_h);
          if (d_h == 64) rope_norm_store<64>(trow + col, dst, t_pos, valid, a);
          else if (d_h == 32) rope_norm_store<32>(trow + col, dst, t_pos, valid, a);
          else rope_norm_store<16>(trow + col, dst, t_pos, valid, a);
        }
      } else if (tl.seg != kSegOut) {
        // g = SiLU(x W_g^T) or v = x W_v^T: 64-column chunks in bf16, staged in shared
        // memory (128-byte swizzle) and written by TMA stores, two buffers in turn
        const CUtensorMap* om = tl.seg == kSegG ? &tmOG : &tmOV;
        const int n0 = tl.nb * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 64) {
          uint32_t r[2][32];
          tmem_ld32(trow + c0, r[0]);
          tmem_ld32(trow + c0 + 32, r[1]);
          tmem_ld_wait();
          if (n0 + c0 >= a.m) continue;  // the same for every thread of the CTA
          if (issuer) bulk_wait_group_read1();  // this buffer's previous store has read it
          named_bar_sync(1, 128);
          const uint32_t sb = smem_u32(sOut + ob * kOutBytes) + (uint32_t)lrow * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t* x = &r[k >> 2][(k & 3) * 8];
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = tl.seg == kSegG ? silu(__uint_as_float(x[e])) : __uint_as_float(x[e]);
            st_shared_v4(sb + (uint32_t)((k ^ (lrow & 7)) << 4),
                         make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                    pack_bf16x2(y[6], y[7])));
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (issuer) {
            // rows past M are clipped; g and v stream out evict-first, so x and the
            // weights stay in L2 for the other tiles
            tma_store_2d_hint(om, sOut + ob * kOutBytes, n0 + c0, tl.mb * BM, l2_evict_first());
            bulk_commit_group();
          }
          ob ^= 1;
        }
      } else {
        const int N = a.d;
        const int n0 = tl.nb * BN;
        __nv_bfloat16* dst = a.h_out;
        const size_t rowoff = (size_t)row * N;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(trow + c0, r);
          tmem_ld_wait();
          if (row >= a.M || n0 + c0 >= N) continue;  // after the collective load
          float y[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) y[c] = __uint_as_float(r[c]);
          {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (n0 + c0 + 8 * u >= N) break;
              const uint4 hv = ld_global_v4(a.h + rowoff + n0 + c0 + 8 * u);
              y[8 * u + 0] += bf16lo(hv.x); y[8 * u + 1] += bf16hi(hv.x);
              y[8 * u + 2] += bf16lo(hv.y); y[8 * u + 3] += bf16hi(hv.y);
              y[8 * u + 4] += bf16lo(hv.z); y[8 * u + 5] += bf16hi(hv.z);
              y[8 * u + 6] += bf16lo(hv.w); y[8 * u + 7] += bf16hi(hv.w);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (n0 + c0 + 8 * u >= N) break;
            st_global_v4(dst + rowoff + n0 + c0 + 8 * u, pack_bf16x2(y[8 * u], y[8 * u + 1]),
                         pack_bf16x2(y[8 * u + 2], y[8 * u + 3]), pack_bf16x2(y[8 * u + 4], y[8 * u + 5]),
                         pack_bf16x2(y[8 * u + 6], y[8 * u + 7]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.acc_empty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }
  if (warp == 2 && lane == 0) bulk_wait_group0();  // every TMA store has completed
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

cudaError_t launch(const CUtensorMap& mA, const CUtensorMap& m0, const CUtensorMap& m1, const CUtensorMap& m2,
                   const CUtensorMap& m3, const CUtensorMap& mog, const CUtensorMap& mov, const GemmArgs& a,
                   cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int ntiles = a.n_mblk * (a.nb_qk + a.nb_g + a.nb_v + a.nb_out);
  const int grid = ntiles < num_sms() ? ntiles : num_sms();
  gemm_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(mA, m0, m1, m2, m3, mog, mov, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_proj_tc(const ProjArgs& p, cudaStream_t s) {
  CUtensorMap mA, mq, mk, mg, mv, mog, mov;
  cudaError_t e = make_tmap_2d(&mA, p.x, p.M, p.d, p.d, BM, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mog, p.g, p.M, p.m, p.m, BM, 64);
  if (e == cudaSuccess) e = make_tmap_2d(&mov, p.v, p.M, p.m, p.m, BM, 64);
  // q/k: one tile of 2 d_qk <= 256 rows, or 256-row tiles of W_q then W_k (d_qk % 256 == 0)
  const uint32_t qk_box = 2 * p.dqk <= BN ? (uint32_t)p.dqk : (uint32_t)BN;
  if (e == cudaSuccess) e = make_tmap_2d(&mq, p.Wq, p.dqk, p.d, p.d, qk_box, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mk, p.Wk, p.dqk, p.d, p.d, qk_box, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mg, p.Wg, p.m, p.d, p.d, BN, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mv, p.Wv, p.m, p.d, p.d, BN, BK);
  if (e != cudaSuccess) return e;
  GemmArgs a = {};
  a.M = p.M; a.K = p.d;
  a.n_mblk = ceil_div(p.M, BM);
  a.nb_qk = 2 * p.dqk <= BN ? 1 : 2 * p.dqk / BN;
  a.nb_g = ceil_div(p.m, BN); a.nb_v = p.skip_v ? 0 : a.nb_g; a.nb_out = 0;
  a.m_major = 0;
  a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.m = p.m; a.d = p.d;
  const int d_h = p.dqk / p.H;
  a.rope = p.rope_base > 0.f;
  for (int c = 0; c < 32; ++c) {
    const double g = c < d_h / 2 ? pow((double)p.rope_base, -2.0 * c / d_h) / 3.141592653589793 : 0.0;
    a.rope_hi[c] = (float)g;
    a.rope_lo[c] = (float)(g - (double)a.rope_hi[c]);
  }
  a.q = static_cast<__nv_bfloat16*>(p.q);
  a.k = static_cast<__nv_bfloat16*>(p.k);
  a.g = static_cast<__nv_bfloat16*>(p.g);
  a.v = static_cast<__nv_bfloat16*>(p.v);
  a.err = p.err;
  a.debug_timeout = p.debug_timeout;
  a.timeout_ns = p.debug_timeout ? 1000000ull : kTimeoutNs;
  return launch(mA, mq, mk, mg, mv, mog, mov, a, s);
}

cudaError_t launch_matmul_tc(const void* A, const void* B, void* C, int M, int N, int K, unsigned* err,
                             cudaStream_t s) {
  // the identity-epilogue segment alone: 128 x 256 tiles, bf16 out through TMA stores
  CUtensorMap mA, mB, mC;
  cudaError_t e = make_tmap_2d(&mA, A, M, K, K, BM, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mB, B, N, K, K, BN, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mC, C, M, N, N, BM, 64);
  if (e != cudaSuccess) return e;
  GemmArgs a = {};
  a.M = M; a.K = K;
  a.n_mblk = ceil_div(M, BM);
  a.nb_v = ceil_div(N, BN);
  a.m_major = 0;
  a.T = 1; a.H = 1; a.m = N; a.d = 0;
  a.v = static_cast<__nv_bfloat16*>(C);
  a.err = err;
  a.timeout_ns = kTimeoutNs;
  return launch(mA, mB, mB, mB, mB, mC, mC, a, s);
}

cudaError_t launch_out_tc(const void* u, const void* Wo, const void* h, void* h_out, int M, int d, int m,
                          unsigned* err, cudaStream_t s) {
  CUtensorMap mA, mo;
  cudaError_t e = make_tmap_2d(&mA, u, M, m, m, BM, BK);
  if (e == cudaSuccess) e = make_tmap_2d(&mo, Wo, d, m, m, BN, BK);
  if (e != cudaSuccess) return e;
  GemmArgs a = {};
  a.M = M; a.K = m;
  a.n_mblk = ceil_div(M, BM);
  a.nb_out = ceil_div(d, BN);
  a.m_major = 1;
  a.T = 1; a.H = 1; a.dqk = 0; a.m = m; a.d = d;
  a.h = static_cast<const __nv_bfloat16*>(h);
  a.h_out = static_cast<__nv_bfloat16*>(h_out);
  a.err = err;
  a.timeout_ns = kTimeoutNs;
  return launch(mA, mo, mo, mo, mo, mo, mo, a, s);
}

}  // namespace tg
