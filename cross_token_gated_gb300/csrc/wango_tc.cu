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
// Two stages:
//  1. wango_prep (CUDA cores): Fq = e^-tau phi(sqrt(tau) qhat), Fk = phi(sqrt(tau) khat)
//     in bf16; per 128-source block the column sums of Fk; and per destination the
//     older-prefix denominator Fq_i . z, z summed over the blocks older than the
//     destination block's window (the same blocks the state holds below).
//  2. wango_tc_kernel: one CTA walks, in order, the 128-row destination blocks ib of one
//     (batch, head, 128-column gate tile) -- a "strip"; persistent CTAs take strips
//     round-robin.  For destination block ib the per-pair sources are the blocks
//        jb = jlo(ib) .. ib,   jlo(ib) = floor(max(0, 128 ib - W + 1) / 128),
//     and the state holds every source j < 128 jlo(ib), older than the window for every
//     destination of the block.  A block is "mixed" when it also holds older pairs
//     (128 jb <= 128 ib + 127 - W): its weights need both scores.  A block "leaves" when
//     jb < jlo(ib + 1): after its P.G MMA the same G tile updates the state.
//
// Roles of the main kernel (16 warps; warp 3 idle):
//   warp 0       TMA: qhat and Fq of the destination block (one buffer each), khat
//                (2-stage ring), Fk of mixed blocks (one buffer), G blocks (128 sources
//                x 128 columns, 2-stage ring of 32 KB) and the destination block's v
//                tile (two 32 KB buffers, which also stage u for its TMA store).
//   warps 1, 2   MMA issue, one thread each, on two SM sub-partitions.  Per destination
//                block the source blocks go newest first (jb = ib .. jlo), so the
//                mixed / leaving blocks come last; a unit is a whole block, or one
//                64-source half of a mixed block.
//                warp 1: a unit's scores into an f32 TMEM slot (ring of 2): Sc = Qhat
//                Khat^T (128 columns), or for a half Sc (64 columns) beside Sf = Fq Fk^T
//                (64 columns); it runs ahead as far as the slots allow.
//                warp 2: O (+)= P G from the unit's slot; for a leaving block
//                S^T += G^T Fk (M=128, N=d_h) in TMEM; last, the read-out O += Fq S_bf16
//                (the state before the block).
//   warps 4-11   weights: warpgroup w takes sources [64w, 64w+64) of a block (or
//                [32w, 32w+32) of a half): exp (window), the feature-map score (older) or
//                0 (after i), rounded to bf16 and written as P over its own cos columns;
//                the row sums of the bf16 weights (the denominator as applied) go to
//                the epilogue through shared memory.
//   warps 12-15  epilogue: gbar = O / den read out of TMEM into registers (rounded to
//                bf16; O is released right after), u = gbar * v over v in shared memory,
//                the copy S^T (TMEM, f32) -> S (shared memory, bf16) for the next
//                destination block's read-out, then u stored by TMA.
// TMEM: O [0,128), S^T [128, 128+d_h), score slots [256,384) and
// [384,512).
#include "tg_common.cuh"
#include "tg_ptx.cuh"
#include "tg_tc.h"
#include "tg_tma.h"

namespace tg {
namespace {

using namespace ptx;

constexpr int kBlk = 128;
constexpr int kNg = 128;       // gate columns per strip
constexpr int kKStages = 2;
constexpr int kGStages = 2;
constexpr int kThreads = 512;
constexpr int kSoftWarp0 = 4, kEpiWarp0 = 12;
constexpr uint32_t kTile = kBlk * 64 * 2;   // 16 KB: a 128 x d_h bf16 tile at d_h = 64
constexpr uint32_t kGBox = 64 * 64 * 2;     // 8 KB: 64 rows x 64 columns
constexpr uint32_t kGStage = 4 * kGBox;     // 32 KB: 128 rows x 128 columns
// TMEM columns: O, the state S^T, the row sums of P, two score slots (P, in bf16 pairs,
// is written over each warpgroup's own cos columns)
constexpr uint32_t kColO = 0, kColSt = 128, kColSlot0 = 256;

struct __align__(8) Bars {
  uint64_t qh_full, qh_empty;                   // qhat of a destination block
  uint64_t fq_full, fq_empty;                   // Fq of a destination block
  uint64_t k_full[kKStages], k_empty[kKStages]; // khat of a source block
  uint64_t fk_full, fk_empty;                   // Fk of a mixed block
  uint64_t g_full[kGStages], g_empty[kGStages]; // G of a source block
  uint64_t v_full[2], v_empty[2];               // v of a destination block, then its u
  uint64_t s_full[2], p_full[2];                // score slots; P in them
  uint64_t slot_free[2];                        // P.G and row sums have read a slot
  uint64_t o_full, o_empty;
  uint64_t st_full;                             // a destination block's MMAs are done
  uint64_t sb_full;                             // bf16 state copy in place
  uint64_t den_full, den_empty;                 // the weights' row sums -> epilogue
  uint64_t drain[2], never;
  uint32_t tmem_base;
  int abort;
  float rowsum[2][kBlk];                        // per warpgroup, per destination row
};

// smem: Qhat | Fq | K x kKStages | Fk | S_bf16 | G x kGStages | V x 2 | ones | Bars
constexpr size_t kSmemBytes = 1024 + kTile * (4 + kKStages) + kGStage * (kGStages + 2) + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
  int B, T, H, dqk, m, d_h, m_h, W;
  int n_iblk, n_ntile, n_strips;
  int nseg, seg_len, n_items;  // each strip's destination blocks in nseg segments
  float* seg_state;            // [n_strips, nseg - 1, kNg, d_h] f32 state at segment ends
  int* seg_flag;               // [n_strips, nseg - 1], 0 until that state is written
  float s;
  const float* tau;
  const float* null_bias;
  const float* den_old;  // [B, H, T]
  int has_v;
  __nv_bfloat16* out;
  unsigned* err;
  uint64_t timeout_ns;
  int debug_timeout;
};

__host__ __device__ __forceinline__ int jlo_of(int ib, int W) {
  const int lo = ib * kBlk - W + 1;
  return lo > 0 ? lo / kBlk : 0;
}
__device__ __forceinline__ bool is_mixed(int jb, int ib, int W) { return jb * kBlk <= ib * kBlk + kBlk - 1 - W; }
__device__ __forceinline__ bool is_leaving(int jb, int ib, int W) { return jb < jlo_of(ib + 1, W); }
// Slot column of P for 16-source step kk of a unit: warpgroup w writes the P of its
// sources over its own cos columns, at 64 w for a whole block (h < 0, 4 steps each) and
// at 32 w for a half (2 steps each).
__device__ __forceinline__ uint32_t p_col(int kk, int h) {
  return h < 0 ? (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8) : (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8);
}

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
__device__ __forceinline__ Item item_of(const Args& a, int w) {
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
__device__ __forceinline__ Strip strip_of(const Args& a, int s) {
  Strip r;
  r.n0 = (s % a.n_ntile) * kNg;
  r.head = (s / a.n_ntile) % a.H;
  r.b = s / (a.n_ntile * a.H);
  return r;
}

__device__ __forceinline__ bool wait_slow(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (*(volatile int*)&b.abort) return false;
  if (mbar_wait(bar, parity, a.timeout_ns)) return true;
  *(volatile int*)&b.abort = 1;
  record_error(a.err, kErrTimeout | kKernWango);
  return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars& b, const Args& a) {
  if (mbar_try_wait_nc(smem_u32(bar), parity)) return true;
  return wait_slow(bar, parity, b, a);
}

// Waits, bounded, until another CTA of this launch sets *flag (acquire).
__device__ __forceinline__ bool wait_flag(const int* flag, const Args& a) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(flag) == 0) {
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      record_error(a.err, kErrTimeout | kKernWango);
      return false;
    }
  }
  return true;
}

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++stage == n) { stage = 0; phase ^= 1; }
  }
};

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
template <int kMode>
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
      if (j0 + e < jw) w0 = __uint_as_float(f[e]);
      if (j0 + e + 1 < jw) w1 = __uint_as_float(f[e + 1]);
      if (j0 + e > i) w0 = 0.f;
      if (j0 + e + 1 > i) w1 = 0.f;
    }
    const uint32_t pk = pack_bf16x2(w0, w1);
    // the row sum of the weights as applied (bf16), two f32 lanes per instruction
    dsum2[(e >> 1) & 1] = add_f32x2(dsum2[(e >> 1) & 1], bf16x2_widen(pk));
    p[e / 2] = pk;
  }
}

// Segment handoff, run once per work item (kept out of line: the hot loops stay small).
// The previous segment's state, one thread's gate column of d_h f32 at src, into TMEM
// at t_st (for the updates) and as bf16 into shared memory at s_sb (for the read-out).
// Called by all four epilogue warps; returns false (for all of them) if the wait for
// the previous segment timed out.
template <int DH>
__device__ __noinline__ bool import_state(const Args& a, size_t slot, uint32_t t_st, uint32_t s_sb, int row,
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
__device__ __noinline__ void export_state(const Args& a, size_t slot, uint32_t t_st, int row, bool issuer) {
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

template <int DH, bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
    wango_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmFQ, const __grid_constant__ CUtensorMap tmFK,
                    const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmU, const Args a) {
  constexpr int RB = DH * 2;  // bytes per row of the q/k/feature tiles
  constexpr uint32_t lay = DH == 64 ? kSwizzle128B : DH == 32 ? kSwizzle64B : kSwizzle32B;
  constexpr uint32_t sbo = 8u * RB;
  constexpr uint32_t tile_bytes = kBlk * RB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                  // qhat
  uint8_t* sFQ = sQ + kTile;           // Fq
  uint8_t* sK = sFQ + kTile;           // khat ring, kKStages tiles
  uint8_t* sFK = sK + kKStages * kTile;
  uint8_t* sSB = sFK + kTile;          // bf16 state, [128 gate rows x d_h]
  uint8_t* sG = sSB + kTile;           // G ring
  uint8_t* sV = sG + kGStages * kGStage;  // two v / u tiles
  Bars& b = *reinterpret_cast<Bars*>(sV + 2 * kGStage);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&b.qh_full, 1);
    mbar_init(&b.qh_empty, 1);
    mbar_init(&b.fq_full, 1);
    mbar_init(&b.fq_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&b.s_full[s], 1);
      mbar_init(&b.p_full[s], 8);
      mbar_init(&b.slot_free[s], 1);
      mbar_init(&b.v_full[s], 1);
      mbar_init(&b.v_empty[s], 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&b.k_full[s], 1);
      mbar_init(&b.k_empty[s], 1);
    }
    mbar_init(&b.fk_full, 1);
    mbar_init(&b.fk_empty, 1);
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&b.g_full[s], 1);
      mbar_init(&b.g_empty[s], 1);
    }
    mbar_init(&b.o_full, 1);
    mbar_init(&b.o_empty, 4);
    mbar_init(&b.st_full, 1);
    mbar_init(&b.sb_full, 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&b.drain[s], 1);
    }
    mbar_init(&b.den_full, 8);
    mbar_init(&b.den_empty, 4);
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
  const int W = a.W;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    // Order per destination block: qhat; then, newest source block first, khat, Fq
    // (before the first mixed block, else after the sources), Fk (mixed blocks), G;
    // then the block's v.
    Ring kr, gr;
    bool ok = true;
    uint32_t kmask = 0, gmask = 0, kph[kKStages] = {}, gph[kGStages] = {}, vmask = 0, vph[2] = {};
    uint32_t fkph = 0;                               // phase of the Fk buffer
    uint32_t qh_n = 0, fq_n = 0, fk_n = 0;             // loads issued
    int dc = 0;  // destination blocks begun
    auto tile128 = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int bb) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 2; ++c) tma_load_3d(dst + h * 2 * kGBox + c * kGBox, map, bar, x + 64 * c, y + 64 * h, bb);
    };
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      const Strip sp = strip_of(a, it.st);
      const int gx = sp.head * a.m_h + sp.n0;
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++dc) {
        const uint32_t dp = dc & 1;
        if (!(ok = wait_bar(&b.qh_empty, dp ^ 1, b, a))) break;
        mbar_arrive_expect_tx(&b.qh_full, tile_bytes);
        tma_load_3d(sQ, &tmQ, &b.qh_full, sp.head * DH, ib * kBlk, sp.b);
        ++qh_n;
        bool fq_loaded = false;
        auto load_fq = [&]() -> bool {
          if (!wait_bar(&b.fq_empty, dp ^ 1, b, a)) return false;
          mbar_arrive_expect_tx(&b.fq_full, tile_bytes);
          tma_load_3d(sFQ, &tmFQ, &b.fq_full, sp.head * DH, ib * kBlk, sp.b);
          ++fq_n;
          fq_loaded = true;
          return true;
        };
        for (int jb = ib; ok && jb >= jlo_of(ib, W); --jb) {
          if (!(ok = wait_bar(&b.k_empty[kr.stage], kr.phase ^ 1, b, a))) break;
          mbar_arrive_expect_tx(&b.k_full[kr.stage], tile_bytes);
          tma_load_3d(sK + kr.stage * kTile, &tmK, &b.k_full[kr.stage], sp.head * DH, jb * kBlk, sp.b);
          kmask |= 1u << kr.stage;
          kph[kr.stage] = kr.phase;
          kr.next(kKStages);
          if (is_mixed(jb, ib, W)) {
            if (!fq_loaded && !(ok = load_fq())) break;
            if (!(ok = wait_bar(&b.fk_empty, fkph ^ 1, b, a))) break;
            mbar_arrive_expect_tx(&b.fk_full, tile_bytes);
            tma_load_3d(sFK, &tmFK, &b.fk_full, sp.head * DH, jb * kBlk, sp.b);
            ++fk_n;
            fkph ^= 1;
          }
          if (!(ok = wait_bar(&b.g_empty[gr.stage], gr.phase ^ 1, b, a))) break;
          mbar_arrive_expect_tx(&b.g_full[gr.stage], kGStage);
          tile128(sG + gr.stage * kGStage, &tmG, &b.g_full[gr.stage], gx, jb * kBlk, sp.b);
          gmask |= 1u << gr.stage;
          gph[gr.stage] = gr.phase;
          gr.next(kGStages);
        }
        if (!ok) break;
        if (!fq_loaded && !(ok = load_fq())) break;
        const int vb = dc & 1;
        const uint32_t vp = (dc >> 1) & 1;
        if (!(ok = wait_bar(&b.v_empty[vb], vp ^ 1, b, a))) break;
        if (a.has_v) {
          mbar_arrive_expect_tx(&b.v_full[vb], kGStage);
          tile128(sV + vb * kGStage, &tmV, &b.v_full[vb], gx, ib * kBlk, sp.b);
          vmask |= 1u << vb;
          vph[vb] = vp;
        } else {
          mbar_arrive(&b.v_full[vb]);
        }
      }
    }
    // no copy may be in flight when the CTA exits
    if (qh_n) mbar_wait(&b.qh_full, (qh_n - 1) & 1, a.timeout_ns);
    if (fq_n) mbar_wait(&b.fq_full, (fq_n - 1) & 1, a.timeout_ns);
    if (fk_n) mbar_wait(&b.fk_full, (fk_n - 1) & 1, a.timeout_ns);
    for (int s = 0; s < kKStages; ++s)
      if (kmask & (1u << s)) mbar_wait(&b.k_full[s], kph[s], a.timeout_ns);
    for (int s = 0; s < kGStages; ++s)
      if (gmask & (1u << s)) mbar_wait(&b.g_full[s], gph[s], a.timeout_ns);
    for (int s = 0; s < 2; ++s)
      if (vmask & (1u << s)) mbar_wait(&b.v_full[s], vph[s], a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue: scores
    // Units in order; unit u's scores go into slot u & 1 once the P.G and row sums of
    // unit u - 2 (the slot's previous user) have completed.
    constexpr uint32_t idesc_s = idesc_bf16_f32(kBlk, kBlk, false, false);  // 128 sources
    constexpr uint32_t idesc_h = idesc_bf16_f32(kBlk, 64, false, false);    // 64 sources
    const uint64_t qd = smem_desc(smem_u32(sQ), 16, sbo, lay);
    const uint64_t fqd = smem_desc(smem_u32(sFQ), 16, sbo, lay);
    const uint64_t kd0 = smem_desc(smem_u32(sK), 16, sbo, lay);
    const uint64_t fkd = smem_desc(smem_u32(sFK), 16, sbo, lay);
    bool ok = true;
    Ring ks;
    uint32_t u = 0, fkph = 0;
    int dc = 0;
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++dc) {
        const int jlo = jlo_of(ib, W);
        for (int jb = ib; ok && jb >= jlo; --jb) {
          const bool mixed = is_mixed(jb, ib, W);
          for (int h = mixed ? 0 : -1; h <= (mixed ? 1 : -1); ++h) {
            if (u >= 2 && !(ok = wait_bar(&b.slot_free[u & 1], ((u - 2) >> 1) & 1, b, a))) break;
            if (!(ok = wait_bar(&b.qh_full, dc & 1, b, a))) break;
            if (!(ok = wait_bar(&b.k_full[ks.stage], ks.phase, b, a))) break;
            if (h >= 0 && !(ok = wait_bar(&b.fq_full, dc & 1, b, a))) break;
            if (h >= 0 && !(ok = wait_bar(&b.fk_full, fkph, b, a))) break;
            tc_fence_after_nc();
            const uint64_t kd = kd0 + (uint64_t)((ks.stage * kTile) >> 4);
            const uint32_t sc = tmem + kColSlot0 + (u & 1) * 128;
            if (h < 0) {
#pragma unroll
              for (int kk = 0; kk < DH / 16; ++kk)
                mma_bf16_ss_nc(sc, qd + (uint64_t)(kk * 2), kd + (uint64_t)(kk * 2), idesc_s, kk != 0);
            } else {
              // cos scores of the half's 64 sources in columns [0, 64), feature-map
              // scores in [64, 128)
              const uint64_t hoff = (uint64_t)((h * 64 * RB) >> 4);
#pragma unroll
              for (int kk = 0; kk < DH / 16; ++kk)
                mma_bf16_ss_nc(sc, qd + (uint64_t)(kk * 2), kd + hoff + (uint64_t)(kk * 2), idesc_h, kk != 0);
#pragma unroll
              for (int kk = 0; kk < DH / 16; ++kk)
                mma_bf16_ss_nc(sc + 64, fqd + (uint64_t)(kk * 2), fkd + hoff + (uint64_t)(kk * 2), idesc_h, kk != 0);
            }
            mma_commit_nc(&b.s_full[u & 1]);
            ++u;
            if (h != 0) {  // the block's last unit releases its khat
              mma_commit_nc(&b.k_empty[ks.stage]);
              ks.next(kKStages);
            }
            if (h == 1) fkph ^= 1;
          }
        }
        if (ok) mma_commit_nc(&b.qh_empty);
      }
    }
    mma_commit(&b.drain[0]);
    mbar_wait(&b.drain[0], 0, a.timeout_ns);
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------------------ MMA issue: P.G, state
    constexpr uint32_t idesc_o = idesc_bf16_f32(kBlk, kNg, false, true);   // O += P G
    constexpr uint32_t idesc_r = idesc_bf16_f32(kBlk, kNg, false, false);  // O += Fq S
    constexpr uint32_t idesc_u = idesc_bf16_f32(kBlk, DH, true, true);     // S^T += G^T Fk
    const uint64_t fqd = smem_desc(smem_u32(sFQ), 16, sbo, lay);
    const uint64_t fkmn = smem_desc(smem_u32(sFK), tile_bytes, sbo, lay);  // Fk as MN-major B
    const uint64_t sbd = smem_desc(smem_u32(sSB), 16, sbo, lay);
    const uint64_t gd0 = smem_desc(smem_u32(sG), kGBox, 1024, kSwizzle128B);
    bool ok = true;
    if (a.debug_timeout) ok = wait_bar(&b.never, 0, b, a);  // nothing ever arrives here
    Ring gr;
    uint32_t u = 0, oph = 0, sbph = 0;
    int dc = 0;
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      // a later segment starts from the state its predecessor handed over
      bool first_update = !(kSeg && it.seg > 0 && jlo_of(it.ib0, W) > 0);
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++dc) {
        const int jlo = jlo_of(ib, W);
        bool copy_ready = false;
        for (int jb = ib; ok && jb >= jlo; --jb) {
          const bool mixed = is_mixed(jb, ib, W), leaving = is_leaving(jb, ib, W);
          for (int h = mixed ? 0 : -1; h <= (mixed ? 1 : -1); ++h) {
            // O (+)= P G; the first unit overwrites O once the epilogue has read the
            // previous destination block's accumulator.
            if (!(ok = wait_bar(&b.p_full[u & 1], (u >> 1) & 1, b, a))) break;
            const bool first = jb == ib && h <= 0;
            if (first) {
              if (!(ok = wait_bar(&b.o_empty, oph ^ 1, b, a))) break;
              oph ^= 1;
            }
            if (!(ok = wait_bar(&b.g_full[gr.stage], gr.phase, b, a))) break;
            tc_fence_after_nc();
            const uint32_t ptm = tmem + kColSlot0 + (u & 1) * 128;
            const uint64_t gd = gd0 + (uint64_t)((gr.stage * kGStage) >> 4);
            // 16-source steps of the block: all 8, or the 4 of half h
            if (h < 0) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t goff = (uint32_t)((kk >> 2) * 2 * kGBox + (kk & 3) * 2048);
                mma_bf16_ts_nc(tmem + kColO, ptm + p_col(kk, h), gd + (uint64_t)(goff >> 4), idesc_o,
                               (first && kk == 0) ? 0u : 1u);
              }
            } else {
              const uint64_t gh = gd + (uint64_t)((h * 2 * kGBox) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ts_nc(tmem + kColO, ptm + p_col(kk, h), gh + (uint64_t)((kk * 2048) >> 4), idesc_o,
                               (first && kk == 0) ? 0u : 1u);
            }
            if (leaving) {
              // S^T += G^T Fk over this unit's sources, once the read-out copy of the
              // previous state is taken (a leaving block is always mixed: h >= 0)
              if (!copy_ready) {
                if (!(ok = wait_bar(&b.sb_full, sbph, b, a))) break;
                sbph ^= 1;
                copy_ready = true;
                tc_fence_after_nc();
              }
              const uint64_t gh = gd + (uint64_t)((h * 2 * kGBox) >> 4);
              const uint64_t fh = fkmn + (uint64_t)((h * 64 * RB) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss_nc(tmem + kColSt, gh + (uint64_t)((kk * 2048) >> 4), fh + (uint64_t)((kk * 16 * RB) >> 4),
                               idesc_u, (first_update && kk == 0) ? 0u : 1u);
              first_update = false;
            }
            mma_commit_nc(&b.slot_free[u & 1]);
            ++u;
            if (h != 0) {  // the block's last unit releases its G and Fk
              mma_commit_nc(&b.g_empty[gr.stage]);
              gr.next(kGStages);
              if (h == 1) mma_commit_nc(&b.fk_empty);
            }
          }
        }
        if (!ok) break;
        // read-out of the state before this block: O += Fq S_bf16
        if (!copy_ready) {
          if (!(ok = wait_bar(&b.sb_full, sbph, b, a))) break;
          sbph ^= 1;
        }
        if (!(ok = wait_bar(&b.fq_full, dc & 1, b, a))) break;
        tc_fence_after_nc();
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk)
          mma_bf16_ss_nc(tmem + kColO, fqd + (uint64_t)(kk * 2), sbd + (uint64_t)(kk * 2), idesc_r, 1u);
        mma_commit_nc(&b.fq_empty);
        mma_commit_nc(&b.st_full);
        mma_commit_nc(&b.o_full);
      }
    }
    mma_commit(&b.drain[1]);
    mbar_wait(&b.drain[1], 0, a.timeout_ns);
  } else if (warp >= kSoftWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------ weights
    const int wg = (warp - kSoftWarp0) / 4;  // sources [64 wg, 64 wg + 64) of each block
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    uint32_t unit = 0;  // units processed
    int gib = 0;        // destination blocks processed
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      const Strip sp = strip_of(a, it.st);
      const float tau = head_tau(a.tau, a.s, sp.head, a.err, kKernWango);
      const float c = tau * kLog2e;
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++gib) {
        const int i = ib * kBlk + row;
        uint64_t dsum2[2] = {0, 0};  // this row's sum of the weights over this warpgroup's sources
        for (int jb = ib; ok && jb >= jlo_of(ib, W); --jb) {
          const bool mixed = is_mixed(jb, ib, W);
          for (int h = mixed ? 0 : -1; h <= (mixed ? 1 : -1); ++h) {
            const uint32_t n = unit++;
            const uint32_t sl = tmem + kColSlot0 + (n & 1) * 128 + lane_off;
            if (!(ok = wait_bar(&b.s_full[n & 1], (n >> 1) & 1, b, a))) break;
            tc_fence_after();
            // P (bf16 pairs) over this warpgroup's own cos columns, so the two
            // warpgroups need not wait for each other.  One 32-source chunk at a time (a
            // rolled loop with one copy of each weight form keeps the code small): two per
            // warpgroup for a whole block, one for a half of a mixed block, whose
            // feature-map scores sit 64 columns after the cos scores.  Each chunk is
            // classified for this warp's 32 rows: after every row (zero weights), inside
            // every row's window (exp only) or general.
            const int nq = h < 0 ? 2 : 1;
            const int i0 = ib * kBlk + quarter * 32;
#pragma unroll 1
            for (int q = 0; q < nq; ++q) {
              const int off = h < 0 ? wg * 64 + q * 32 : h * 64 + wg * 32;  // first source in the block
              const uint32_t cs = sl + (uint32_t)(h < 0 ? off : wg * 32);     // its cos score column
              const uint32_t pc = sl + (uint32_t)(h < 0 ? wg * 64 + q * 16 : wg * 32);
              const int js = jb * kBlk + off;
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
                weights32<2>(r[0], r[1], c, js, i, h < 0 ? -0x7fffffff - 1 : i - W + 1, p, dsum2);
              }
              tmem_st16(pc, p);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.p_full[n & 1]);
          }
        }
        if (!ok) break;
        // the row sums of this destination block -> epilogue
        if (!(ok = wait_bar(&b.den_empty, (gib & 1) ^ 1, b, a))) break;
        float d0, d1, d2, d3;
        f32x2_unpack(dsum2[0], d0, d1);
        f32x2_unpack(dsum2[1], d2, d3);
        b.rowsum[wg][row] = (d0 + d1) + (d2 + d3);
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.den_full);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue + state copy
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // destination row; also the gate column of S^T
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool issuer = (warp == kEpiWarp0 && lane == 0);
    bool ok = true;
    uint32_t oph = 0, stph = 0;
    int gib = 0;
    // bf16 copy of the state for a destination block's read-out (zero while no source
    // has left the window)
    auto copy_state = [&](bool empty) {
      if (!empty) tc_fence_after();
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
    for (int w = blockIdx.x; ok && w < a.n_items; w += gridDim.x) {
      const Item it = item_of<kSeg>(a, w);
      if (it.ib0 >= it.ib1) continue;
      const Strip sp = strip_of(a, it.st);

      const float tau = head_tau(a.tau, a.s, sp.head, a.err, kKernWango);
      // the state before the first destination block: empty, or the previous
      // segment's (into TMEM for the updates, bf16 into shared memory for the read-out)
      if (kSeg && it.seg > 0 && jlo_of(it.ib0, W) > 0) {
        if (!import_state<DH>(a, (size_t)it.st * (a.nseg - 1) + (it.seg - 1), tmem + kColSt + lane_off,
                              smem_u32(sSB), row, &b.sb_full, lane, issuer))
          break;
      } else {
        copy_state(true);
      }
      const float null_w = a.null_bias ? exp2f((a.null_bias[sp.head] - tau) * kLog2e) : 0.f;
      for (int ib = it.ib0; ok && ib < it.ib1; ++ib, ++gib) {
        const int i = ib * kBlk + row;
        const bool row_ok = i < a.T;
        const int sv = gib & 1;  // v tile buffer
        const uint32_t pv = (gib >> 1) & 1;
        // older-prefix denominator, fetched before the waits
        float den = row_ok ? a.den_old[((size_t)sp.b * a.H + sp.head) * a.T + i] : 0.f;
        den += (float)(i + 1) * null_w;
        if (ok) ok = wait_bar(&b.den_full, gib & 1, b, a);
        if (ok) {
          den += b.rowsum[0][row] + b.rowsum[1][row];  // this block's per-pair weights, as applied
          __syncwarp();
          if (lane == 0) mbar_arrive(&b.den_empty);
        }
        if (ok) ok = wait_bar(&b.o_full, oph, b, a);
        ok = named_bar_and(2, 128, ok);
        if (!ok) break;
        oph ^= 1;
        tc_fence_after();
        const float inv = 1.f / den;
        // gbar = O / den, rounded to bf16, in registers; the accumulator is released as
        // soon as it has been read
        uint32_t gb[kNg / 2];
#pragma unroll
        for (int c0 = 0; c0 < kNg; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + kColO + lane_off + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            gb[(c0 + e) / 2] = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.o_empty);
        if (ok) ok = wait_bar(&b.st_full, stph, b, a);
        if (ok) ok = wait_bar(&b.v_full[sv], pv, b, a);
        ok = named_bar_and(2, 128, ok);
        if (!ok) break;
        stph ^= 1;
        // u = gbar * v, written over v in shared memory (the TMA store's source)
        const uint32_t vst = smem_u32(sV + sv * kGStage);
        const int rh = row >> 6, rr = row & 63;
        const size_t grow = ((size_t)sp.b * a.T + (row_ok ? i : 0)) * a.m + (size_t)sp.head * a.m_h;
#pragma unroll
        for (int cq = 0; cq < 2; ++cq) {
          const int col0 = sp.n0 + cq * 64;
          const bool straddle = col0 < a.m_h && col0 + 64 > a.m_h;
          const uint32_t box = vst + rh * 2 * kGBox + cq * kGBox + rr * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t addr = box + (uint32_t)((k ^ (rr & 7)) << 4);
            const uint32_t* g4 = &gb[cq * 32 + k * 4];
            uint32_t u[4];
            if (a.has_v) {
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
        // the state copy for the next destination block (this block's updates and
        // read-out are complete; the next block updates the state only after it)
        if (ib + 1 < it.ib1) copy_state(jlo_of(ib + 1, W) == 0);
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (issuer) {
          for (int h = 0; h < 2; ++h) {
            const int y = ib * kBlk + 64 * h;
            if (y >= a.T) continue;
            for (int cq = 0; cq < 2; ++cq) {
              const int col0 = sp.n0 + cq * 64;
              if (col0 + 64 > a.m_h) continue;
              tma_store_3d(&tmU, sV + sv * kGStage + h * 2 * kGBox + cq * kGBox, sp.head * a.m_h + col0, y, sp.b);
            }
          }
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&b.v_empty[sv]);
        }
      }
      // hand this segment's final state to the next segment of the strip (the last
      // block's updates are complete: its st_full was waited for above)
      if (kSeg && ok && it.seg + 1 < a.nseg && jlo_of(it.ib1, W) > 0)
        export_state<DH>(a, (size_t)it.st * (a.nseg - 1) + it.seg, tmem + kColSt + lane_off, row, issuer);
    }
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

// Fq = e^-tau phi(sqrt(tau) qhat), Fk = phi(sqrt(tau) khat); one thread per (row, 8
// consecutive features of one head).
__global__ void wango_phi_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k, __nv_bfloat16* fq,
                                 __nv_bfloat16* fk, long long rows, int H, int dqk, float s, const float* tau,
                                 int phi_mode, unsigned* err) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int groups = dqk / 8;
  if (idx >= rows * groups) return;
  const long long r = idx / groups;
  const int c0 = (int)(idx % groups) * 8;
  const int d_h = dqk / H, a = c0 / d_h;
  const float t = head_tau(tau, s, a, err, kKernWango);
  const float sq = sqrtf(t), shift = exp2f(-t * kLog2e), inv_sqrt_dh = rsqrtf((float)d_h);
  const uint4 qv = *reinterpret_cast<const uint4*>(q + r * dqk + c0);
  const uint4 kv = *reinterpret_cast<const uint4*>(k + r * dqk + c0);
  const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
  uint32_t fo[4], ko[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    fo[e] = pack_bf16x2(shift * phi_fast(sq * bf16lo(qw[e]), inv_sqrt_dh, phi_mode),
                        shift * phi_fast(sq * bf16hi(qw[e]), inv_sqrt_dh, phi_mode));
    ko[e] = pack_bf16x2(phi_fast(sq * bf16lo(kw[e]), inv_sqrt_dh, phi_mode),
                        phi_fast(sq * bf16hi(kw[e]), inv_sqrt_dh, phi_mode));
  }
  *reinterpret_cast<uint4*>(fq + r * dqk + c0) = make_uint4(fo[0], fo[1], fo[2], fo[3]);
  *reinterpret_cast<uint4*>(fk + r * dqk + c0) = make_uint4(ko[0], ko[1], ko[2], ko[3]);
}

// zb[b, a, jb, c] = sum over the valid sources of block jb of Fk[., a*d_h + c] (the bf16
// values the state update multiplies).  grid
// (n_iblk, H, B), 256 threads: thread (g, p) sums column pair p over rows g, g + 8, ...
// (bf16x2 loads, one head row per warp), then the eight row groups are added.
__global__ void __launch_bounds__(256) wango_blocksum_kernel(const __nv_bfloat16* fk, float* zb, int T, int H,
                                                             int dqk, int n_iblk) {
  __shared__ float part[8][64];
  const int jb = blockIdx.x, a = blockIdx.y, bb = blockIdx.z;
  const int d_h = dqk / H, npair = d_h / 2;
  const int p = threadIdx.x % 32, g = threadIdx.x / 32;
  const int j0 = jb * kBlk, j1 = min(T, j0 + kBlk);
  float s0 = 0.f, s1 = 0.f;
  if (p < npair) {
    for (int j = j0 + g; j < j1; j += 8) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(fk + ((size_t)bb * T + j) * dqk + a * d_h + 2 * p);
      s0 += bf16lo(w);
      s1 += bf16hi(w);
    }
    part[g][2 * p] = s0;
    part[g][2 * p + 1] = s1;
  }
  __syncthreads();
  if (threadIdx.x < d_h) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) t += part[q][threadIdx.x];
    zb[(((size_t)bb * H + a) * n_iblk + jb) * d_h + threadIdx.x] = t;
  }
}
// den_old[b, a, i] = Fq_i . z with z the sum of zb over the blocks older than the window of
// i's destination block ib (jb < jlo(ib)).  grid (n_iblk, H, B), 128 threads, one row
// each; Fq is read 16 bytes at a time.
__global__ void __launch_bounds__(128) wango_denold_kernel(const __nv_bfloat16* fq, const float* zb, float* den_old,
                                                           int T, int H, int dqk, int n_iblk, int W) {
  __shared__ float z[64];
  const int ib = blockIdx.x, a = blockIdx.y, bb = blockIdx.z, t = threadIdx.x;
  const int d_h = dqk / H, jlo = jlo_of(ib, W);
  if (t < d_h) {
    float s = 0.f;
    for (int jb = 0; jb < jlo; ++jb) s += zb[(((size_t)bb * H + a) * n_iblk + jb) * d_h + t];
    z[t] = s;
  }
  __syncthreads();
  const int i = ib * kBlk + t;
  if (i >= T) return;
  const __nv_bfloat16* f = fq + ((size_t)bb * T + i) * dqk + a * d_h;
  float dot = 0.f;
  for (int c = 0; c < d_h; c += 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(f + c);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      dot = fmaf(bf16lo(ww[e]), z[c + 2 * e], dot);
      dot = fmaf(bf16hi(ww[e]), z[c + 2 * e + 1], dot);
    }
  }
  den_old[((size_t)bb * H + a) * T + i] = dot;
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

struct AuxLayout {
  size_t fq, fk, zb, den, seg, flag, total;
  int nseg;
};
AuxLayout aux_layout(int B, int T, int H, int dqk, int m, int W) {
  const size_t BT = (size_t)B * T, nI = (size_t)(T + kBlk - 1) / kBlk;
  const int d_h = dqk / H;
  const long long strips = (long long)B * H * ((m / H + kNg - 1) / kNg);
  AuxLayout L;
  L.nseg = choose_nseg(strips, (int)nI, W, num_sms());
  const size_t handoffs = (size_t)strips * (L.nseg - 1);
  L.fq = 0;
  L.fk = L.fq + a256(BT * dqk * 2);
  L.zb = L.fk + a256(BT * dqk * 2);
  L.den = L.zb + a256((size_t)B * H * nI * d_h * 4);
  L.seg = L.den + a256((size_t)B * H * T * 4);
  L.flag = L.seg + a256(handoffs * kNg * d_h * 4);
  L.total = L.flag + a256(handoffs * 4);
  return L;
}

}  // namespace

size_t wango_aux_bytes(int B, int T, int H, int dqk, int m, int W) { return aux_layout(B, T, H, dqk, m, W).total; }

cudaError_t launch_wango_tc(const AggArgs& p, cudaStream_t s) {
  Args a = {};
  a.B = p.B; a.T = p.T; a.H = p.H; a.dqk = p.dqk; a.m = p.m;
  a.d_h = p.dqk / p.H; a.m_h = p.m / p.H;
  a.W = p.window;
  a.n_iblk = ceil_div(p.T, kBlk);
  a.n_ntile = ceil_div(a.m_h, kNg);
  const long long strips = (long long)p.B * p.H * a.n_ntile;
  if (strips > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_strips = (int)strips;
  const AuxLayout L = aux_layout(p.B, p.T, p.H, p.dqk, p.m, p.window);
  a.nseg = L.nseg;
  a.seg_len = ceil_div(a.n_iblk, a.nseg);
  if (strips * a.nseg > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_items = a.n_strips * a.nseg;
  a.s = p.s; a.tau = p.tau; a.null_bias = p.null_bias;
  a.has_v = p.v != nullptr;
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.err = p.err;
  a.debug_timeout = (p.flags & TG_FLAG_DEBUG_TIMEOUT) ? 1 : 0;
  a.timeout_ns = a.debug_timeout ? 1000000ull : 2000000000ull;

  // pre-pass: feature maps, block sums, older-prefix denominators
  char* aux = static_cast<char*>(p.aux);
  a.seg_state = reinterpret_cast<float*>(aux + L.seg);
  a.seg_flag = reinterpret_cast<int*>(aux + L.flag);
  if (a.nseg > 1) {  // no segment's state is ready yet
    const cudaError_t me = cudaMemsetAsync(a.seg_flag, 0, (size_t)a.n_strips * (a.nseg - 1) * sizeof(int), s);
    if (me != cudaSuccess) return me;
  }
  __nv_bfloat16* fq = reinterpret_cast<__nv_bfloat16*>(aux + L.fq);
  __nv_bfloat16* fk = reinterpret_cast<__nv_bfloat16*>(aux + L.fk);
  float* zb = reinterpret_cast<float*>(aux + L.zb);
  float* den = reinterpret_cast<float*>(aux + L.den);
  const long long rows = (long long)p.B * p.T;
  const long long work = rows * (p.dqk / 8);
  wango_phi_kernel<<<(unsigned)((work + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(p.q), static_cast<const __nv_bfloat16*>(p.k), fq, fk, rows, p.H, p.dqk,
      p.s, p.tau, p.phi_mode, p.err);
  dim3 g3(a.n_iblk, p.H, p.B);
  wango_blocksum_kernel<<<g3, 256, 0, s>>>(fk, zb, p.T, p.H, p.dqk, a.n_iblk);
  wango_denold_kernel<<<g3, kBlk, 0, s>>>(fq, zb, den, p.T, p.H, p.dqk, a.n_iblk, p.window);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  a.den_old = den;

  CUtensorMap mq, mk, mfq, mfk, mg, mv, mu;
  e = make_tmap_3d(&mq, p.q, p.B, p.T, p.dqk, kBlk, a.d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mk, p.k, p.B, p.T, p.dqk, kBlk, a.d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mfq, fq, p.B, p.T, p.dqk, kBlk, a.d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mfk, fk, p.B, p.T, p.dqk, kBlk, a.d_h);
  if (e == cudaSuccess) e = make_tmap_3d(&mg, p.g, p.B, p.T, p.m, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mv, p.v ? p.v : p.g, p.B, p.T, p.m, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d(&mu, p.out, p.B, p.T, p.m, 64, 64);
  if (e != cudaSuccess) return e;
  auto kern = a.nseg > 1 ? (a.d_h == 64 ? wango_tc_kernel<64, true> : a.d_h == 32 ? wango_tc_kernel<32, true>
                                                                                  : wango_tc_kernel<16, true>)
                         : (a.d_h == 64 ? wango_tc_kernel<64, false> : a.d_h == 32 ? wango_tc_kernel<32, false>
                                                                                   : wango_tc_kernel<16, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = a.n_items < num_sms() ? a.n_items : num_sms();
  kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mfq, mfk, mg, mv, mu, a);
  return cudaGetLastError();
}

}  // namespace tg
