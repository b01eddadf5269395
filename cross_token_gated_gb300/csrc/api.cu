// C ABI of the gate-aggregation library: argument validation, workspace layout,
// dispatch to the kernels, and the per-device error word.  See include/tango.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "tango.h"
#include "tg_kernels.h"
#include "tg_common.cuh"
#include "tg_tc.h"

namespace tg {

__device__ unsigned g_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned* g_err_ptr[kMaxDevices] = {};

// Device address of this device's error word (looked up once per device).
cudaError_t error_word(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_ptr[dev];
  return cudaSuccess;
}

size_t elem_size(tg_dtype dt) { return dt == TG_F32 ? 4 : 2; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tg_status validate_agg(const tg_agg_params* p, bool wango) {
  if (!p) return TG_ERR_INVALID_ARG;
  if (p->B < 1 || p->T < 1 || p->H < 1 || p->H > TG_MAX_HEADS || p->d_qk < 1 || p->m < 1)
    return TG_ERR_INVALID_ARG;
  if (p->d_qk % p->H != 0 || p->m % p->H != 0) return TG_ERR_INVALID_ARG;
  if (p->dtype != TG_F32 && p->dtype != TG_BF16) return TG_ERR_INVALID_ARG;
  if (!p->tau && !(p->s >= 0.f && p->s <= 20.f)) return TG_ERR_INVALID_ARG;
  if (wango && p->window < 1) return TG_ERR_INVALID_ARG;
  if (wango && p->phi_mode != 0 && p->phi_mode != 1) return TG_ERR_INVALID_ARG;
  if (p->flags & ~(TG_FLAG_QK_NORMALIZED | TG_FLAG_DEBUG_TIMEOUT)) return TG_ERR_INVALID_ARG;
  if (p->m_pitch != 0 && p->m_pitch < p->m / p->H) return TG_ERR_INVALID_ARG;
  const int d_h = p->d_qk / p->H;
  if (d_h > 128) return TG_ERR_UNSUPPORTED;
  if ((long long)p->B * p->T > (1LL << 31) - 1) return TG_ERR_UNSUPPORTED;
  if ((long long)p->H * (p->m_pitch ? p->m_pitch : p->m / p->H) > (1LL << 30)) return TG_ERR_UNSUPPORTED;
  if (p->dtype == TG_BF16) {
    if (d_h != 16 && d_h != 32 && d_h != 64) return TG_ERR_UNSUPPORTED;
    if ((p->m_pitch ? p->m_pitch : p->m / p->H) % 8 != 0) return TG_ERR_UNSUPPORTED;
  }
  return TG_OK;
}

// Gate columns of a row in memory: H times the per-head pitch.
int mem_width(const tg_agg_params* p) { return p->H * (p->m_pitch ? p->m_pitch : p->m / p->H); }

// Normalised q/k copies (unless the caller passes unit vectors).
size_t agg_qk_bytes(const tg_agg_params* p) {
  if (p->flags & TG_FLAG_QK_NORMALIZED) return 0;
  const size_t qk = (size_t)p->B * p->T * p->d_qk * elem_size(p->dtype);
  return 2 * align256(qk);
}
// Feature-map scratch of the tensor-core WANGO path.
size_t agg_aux_bytes(const tg_agg_params* p, bool wango) {
  return (wango && p->dtype == TG_BF16) ? wango_aux_bytes(p->B, p->T, p->H, p->d_qk, p->m, p->window) : 0;
}
size_t agg_ws_bytes(const tg_agg_params* p, bool wango) { return agg_qk_bytes(p) + agg_aux_bytes(p, wango); }

// Per-head gate pitch of a block's internal g, u and gate-indexed weights: on the
// tensor-core path m_h rounded up to a multiple of 8 (TMA wants 16-byte pitches and
// head offsets), else m_h.  The padded entries are zero in W_g, W_v and W_o, so g, v
// and u are zero there and add nothing to h_out.
int gate_pitch(const tg_agg_params& a) {
  const int m_h = a.m / a.H;
  return a.dtype == TG_BF16 ? (m_h + 7) / 8 * 8 : m_h;
}
// The aggregation as the block runs it: gate width H * gate_pitch.
tg_agg_params block_agg(const tg_block_params* p) {
  tg_agg_params a = p->agg;
  a.m = a.H * gate_pitch(p->agg);
  return a;
}

struct BlockWs {
  size_t x, q, k, g, v, aux, wg, wv, wo, total;
  bool padded;
};

BlockWs block_ws_layout(const tg_block_params* p) {
  const tg_agg_params a = block_agg(p);
  const size_t es = elem_size(a.dtype), BT = (size_t)a.B * a.T;
  BlockWs w;
  w.padded = a.m != p->agg.m;
  w.x = 0;
  w.q = w.x + align256(BT * p->d * es);
  w.k = w.q + align256(BT * a.d_qk * es);
  w.g = w.k + align256(BT * a.d_qk * es);
  w.v = w.g + align256(BT * a.m * es);
  w.aux = w.v + align256(BT * a.m * es);
  w.wg = w.aux + agg_aux_bytes(&a, p->mode == TG_MODE_WANGO);
  const size_t wbytes = w.padded ? align256((size_t)a.m * p->d * es) : 0;
  w.wv = w.wg + wbytes;
  w.wo = w.wv + wbytes;
  w.total = w.wo + wbytes;
  return w;
}

tg_status validate_block(const tg_block_params* p) {
  if (!p) return TG_ERR_INVALID_ARG;
  if (p->agg.H < 1 || p->agg.m < 1 || p->agg.m % p->agg.H != 0) return TG_ERR_INVALID_ARG;
  tg_agg_params a = block_agg(p);
  a.flags &= ~TG_FLAG_FUSED_V;  // a block flag, checked below
  tg_status st = validate_agg(&a, p->mode == TG_MODE_WANGO);
  if (st != TG_OK) return st;
  if (p->agg.flags & ~(TG_FLAG_DEBUG_TIMEOUT | TG_FLAG_FUSED_V)) return TG_ERR_INVALID_ARG;
  if (p->agg.m_pitch != 0) return TG_ERR_INVALID_ARG;  // the block lays out its own gates
  if (p->d < 1 || !(p->rms_eps > 0.f) || !(p->rope_base >= 0.f)) return TG_ERR_INVALID_ARG;
  if (p->mode != TG_MODE_TANGO && p->mode != TG_MODE_WANGO) return TG_ERR_INVALID_ARG;
  if (p->rope_base > 0.f && (p->agg.d_qk / p->agg.H) % 2 != 0) return TG_ERR_INVALID_ARG;
  if (p->agg.dtype == TG_BF16 && p->d % 64 != 0) return TG_ERR_UNSUPPORTED;
  // the projection GEMM takes q and k in one 256-column tile, or in 256-column tiles
  if (p->agg.dtype == TG_BF16 && 2 * p->agg.d_qk > 256 && p->agg.d_qk % 256 != 0) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

// ---- model forward (sec. 2.3 eq. 11; the revision's gated-projection sets)
constexpr int kMaxApps = 64, kMaxSets = 16;

tg_status validate_model(const tg_model_params* p) {
  if (!p) return TG_ERR_INVALID_ARG;
  tg_status st = validate_block(&p->block);
  if (st != TG_OK) return st;
  if (p->vocab < 1 || p->n_apps < 1 || p->n_apps > kMaxApps || p->n_sets < 1 || p->n_sets > kMaxSets)
    return TG_ERR_INVALID_ARG;
  if (!(p->final_rms_eps > 0.f)) return TG_ERR_INVALID_ARG;
  if (p->set_of_app) {
    for (int r = 0; r < p->n_apps; ++r)
      if (p->set_of_app[r] < 0 || p->set_of_app[r] >= p->n_sets) return TG_ERR_INVALID_ARG;
  } else if (p->n_sets != 1 && p->n_sets != 3) {
    return TG_ERR_INVALID_ARG;  // no default assignment for this many sets
  }
  if (p->block.agg.dtype == TG_BF16 && p->vocab % 8 != 0) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

// The set used by application r: the caller's table, else all set 0 (one set) or the
// first / middle / last assignment of three sets.
int set_of(const tg_model_params* p, int r) {
  if (p->set_of_app) return p->set_of_app[r];
  if (p->n_sets == 1) return 0;
  return r == 0 ? 0 : (r == p->n_apps - 1 ? 2 : 1);
}

struct ModelWs {
  size_t h, x, block, total;
};

ModelWs model_ws_layout(const tg_model_params* p) {
  const tg_agg_params& a = p->block.agg;
  const size_t hb = align256((size_t)a.B * a.T * p->block.d * elem_size(a.dtype));
  ModelWs w;
  w.h = 0;
  w.x = hb;
  w.block = 2 * hb;
  w.total = w.block + block_ws_layout(&p->block).total;
  return w;
}

// ---- WANGO decode step
tg_status validate_decode(const tg_agg_params* p) {
  if (!p) return TG_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->H > TG_MAX_HEADS || p->d_qk < 1 || p->m < 1) return TG_ERR_INVALID_ARG;
  if (p->d_qk % p->H != 0 || p->m % p->H != 0) return TG_ERR_INVALID_ARG;
  if (p->dtype != TG_F32 && p->dtype != TG_BF16) return TG_ERR_INVALID_ARG;
  if (!p->tau && !(p->s >= 0.f && p->s <= 20.f)) return TG_ERR_INVALID_ARG;
  if (p->window < 1 || (p->phi_mode != 0 && p->phi_mode != 1)) return TG_ERR_INVALID_ARG;
  if (p->window > (1 << 30)) return TG_ERR_UNSUPPORTED;  // the ring's slot count stays an int
  if (p->flags & ~TG_FLAG_QK_NORMALIZED) return TG_ERR_INVALID_ARG;
  if (p->m_pitch != 0 && p->m_pitch != p->m / p->H) return TG_ERR_UNSUPPORTED;  // dense tensors only
  if (p->d_qk / p->H > 128) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

struct DecodeWs {
  size_t S, z, ring_k, ring_g, w, fq, fk, wpart, older, total;
};
DecodeWs decode_ws_layout(const tg_agg_params* p) {
  const size_t B = p->B, H = p->H, R = (size_t)p->window + kDecodeFold, d_h = p->d_qk / p->H;
  DecodeWs L;
  L.S = 0;
  L.z = L.S + align256(B * d_h * p->m * 4);
  L.ring_k = L.z + align256(2 * B * H * d_h * 4);
  L.ring_g = L.ring_k + align256(B * H * R * d_h * elem_size(p->dtype));
  L.w = L.ring_g + align256(B * R * p->m * elem_size(p->dtype));
  L.fq = L.w + align256(B * H * R * 4);
  L.fk = L.fq + align256(B * H * d_h * 4);
  L.wpart = L.fk + align256(B * H * kDecodeFold * d_h * 4);
  L.older = L.wpart + align256(B * H * 8 * 4);
  L.total = L.older + align256(B * H * 4);
  return L;
}

tg_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return TG_OK;
  if (!ws || ws_bytes < need) return TG_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return TG_ERR_WORKSPACE;
  return TG_OK;
}

tg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TG_OK : TG_ERR_CUDA; }

// Shared body of tango_aggregate / wango_aggregate (and, with gbar and den, of the
// _save variants).
tg_status aggregate(bool wango, const tg_agg_params* p, const void* q, const void* k, const void* g,
                    const void* v, void* out, void* ws, size_t ws_bytes, cudaStream_t stream, void* gbar = nullptr,
                    float* den = nullptr) {
  tg_status st = validate_agg(p, wango);
  if (st != TG_OK) return st;
  if (!q || !k || !g || !out) return TG_ERR_INVALID_ARG;
  if (gbar || den) {
    if (!gbar || !den) return TG_ERR_INVALID_ARG;
    if (p->dtype != TG_BF16) return TG_ERR_UNSUPPORTED;
    if (!aligned16(gbar) || !aligned16(den)) return TG_ERR_UNSUPPORTED;
  }
  if (p->dtype == TG_BF16 && !(aligned16(q) && aligned16(k) && aligned16(g) && aligned16(out) &&
                               (!v || aligned16(v))))
    return TG_ERR_UNSUPPORTED;
  const size_t need = agg_ws_bytes(p, wango), qk_bytes = agg_qk_bytes(p);
  st = check_ws(ws, ws_bytes, need);
  if (st != TG_OK) return st;

  AggArgs a;
  a.B = p->B; a.T = p->T; a.H = p->H; a.dqk = p->d_qk; a.m = mem_width(p); a.m_h = p->m / p->H;
  a.s = p->s; a.tau = p->tau; a.null_bias = p->null_bias;
  a.window = p->window; a.phi_mode = p->phi_mode; a.flags = p->flags; a.dtype = p->dtype;
  a.g = g; a.v = v; a.out = out;
  a.aux = static_cast<char*>(ws) + qk_bytes;
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return TG_ERR_CUDA;
  if (p->flags & TG_FLAG_QK_NORMALIZED) {
    a.q = q;
    a.k = k;
  } else {
    const long long rows = (long long)p->B * p->T;
    char* base = static_cast<char*>(ws);
    void* qn = base;
    void* kn = base + qk_bytes / 2;
    e = launch_qk_prep(p->dtype, q, qn, rows, p->T, p->H, p->d_qk, 0.f, true, stream);
    if (e == cudaSuccess) e = launch_qk_prep(p->dtype, k, kn, rows, p->T, p->H, p->d_qk, 0.f, true, stream);
    if (e != cudaSuccess) return TG_ERR_CUDA;
    a.q = qn;
    a.k = kn;
  }
  if (p->dtype == TG_F32) return cuda_status(wango ? launch_wango_simt(a, stream) : launch_tango_simt(a, stream));
  a.gbar_out = gbar;
  if (!wango) {
    a.den_out = den;
    a.den_pitch = p->T;
    return cuda_status(launch_tango_tc(a, stream));
  }
  e = launch_wango_tc(a, stream);
  if (e == cudaSuccess && den)  // the denominators as the weights kernel left them, at a pitch of T
    e = cudaMemcpy2DAsync(den, (size_t)p->T * 4, wango_den_in_aux(a.aux, p->B, p->T, p->H, p->d_qk, p->m, p->window),
                          (size_t)bwd_tpad(p->T) * 4, (size_t)p->T * 4, (size_t)p->B * p->H, cudaMemcpyDeviceToDevice,
                          stream);
  return cuda_status(e);
}

// ---- aggregation backward (bf16, tensor cores)
tg_status validate_bwd(const tg_agg_params* p, bool wango) {
  const unsigned far_flags = TG_FLAG_BWD_FAR_SCAN | TG_FLAG_BWD_FAR_PAIRS;
  if (p->flags & ~(TG_FLAG_QK_NORMALIZED | TG_FLAG_DEBUG_TIMEOUT | (wango ? far_flags : 0u)))
    return TG_ERR_INVALID_ARG;
  tg_agg_params shape = *p;  // the forward's checks, without the backward-only flags
  shape.flags &= ~far_flags;
  tg_status st = validate_agg(&shape, wango);
  if (st != TG_OK) return st;
  if ((p->flags & far_flags) == far_flags) return TG_ERR_INVALID_ARG;
  if (p->dtype != TG_BF16) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

struct BwdWs {
  size_t qn, kn, gbar, den, dp, E, X, Xo, aux, part, rb, total;
  int T_pad;
  bool scan;  // WANGO: far older pairs through the running sums
};
BwdWs bwd_ws_layout(const tg_agg_params* p, bool wango) {
  const size_t B = p->B, T = p->T, H = p->H, m = mem_width(p), dqk = p->d_qk;
  BwdWs L;
  L.T_pad = bwd_tpad(p->T);
  const size_t Tp = L.T_pad;
  const bool norm = !(p->flags & TG_FLAG_QK_NORMALIZED);
  L.qn = 0;
  L.kn = L.qn + (norm ? align256(B * T * dqk * 2) : 0);
  L.gbar = L.kn + (norm ? align256(B * T * dqk * 2) : 0);
  L.den = L.gbar + align256(B * T * m * 2);
  L.dp = L.den + (wango ? 0 : align256(B * H * Tp * 4));
  L.E = L.dp + align256(B * H * Tp * 4);
  L.X = L.E + align256(B * T * m * 2);
  L.Xo = L.X + align256(B * H * Tp * Tp * 2);
  L.aux = L.Xo + (wango ? align256(B * H * Tp * Tp * 2) : 0);
  const size_t aux = wango ? wango_aux_bytes(p->B, p->T, p->H, p->d_qk, p->m, p->window) : 0;
  L.part = L.aux + align256(aux);
  // WANGO with blocks wholly beyond the window's band: the scans' per-strip sums (two
  // directions) and the block sums for rho
  const int band = bwd_band(p->window), nblk = L.T_pad / 128;
  L.scan = wango && nblk - band - 1 > 0 && !(p->flags & TG_FLAG_BWD_FAR_PAIRS) &&
           ((p->flags & TG_FLAG_BWD_FAR_SCAN) || bwd_scan_pays(p->B, p->T, p->H, p->d_qk, p->m / p->H, p->window));
  const size_t strips = L.scan ? (size_t)bwd_scan_strips(p->B, p->H, p->m / p->H) : 0;
  L.rb = L.part + (L.scan ? align256(2 * strips * B * T * dqk * 4) : 0);
  // rb, then the two plain far sums
  L.total = L.rb + (L.scan ? align256(3 * B * H * nblk * (dqk / H) * 4) : 0);
  return L;
}

// Gradients of L = sum(dout * u) for u = aggregate(q, k, g, v), as laid out in
// tango.h.  The forward is recomputed (gbar and the denominators) unless the caller
// kept them from a _save call, then:
//   E = dout * v / den, D = E . gbar, dv = dout * gbar                       (prep)
//   WANGO, when it pays: the older pairs beyond the window's band of blocks through
//     running-sum scans, reduced over the gate strips (linear in T)
//   X, X_old = pair-weight gradients of window and older pairs (with the scans, the band
//     only), then dq, dk from them (tensor cores; WANGO's older pairs through the
//     forward's feature maps, which are still in the scratch at that point)
//   dg_j = sum_{i >= j} w_ij E_i: the forward numerator with the roles of destinations
//     and sources exchanged (TANGO: the tensor-core kernel in reverse mode; WANGO: the
//     windowed kernels on the time-reversed sequence, read and written mirrored in place,
//     whose older-pair weights e^-tau phi(k~_j) . phi(q~_i) are the same products).
tg_status aggregate_backward(bool wango, const tg_agg_params* p, const void* q, const void* k, const void* g,
                             const void* v, const void* dout, const void* saved_gbar, const float* saved_den,
                             void* dq, void* dk, void* dg, void* dv, void* ws, size_t ws_bytes, cudaStream_t stream) {
  tg_status st = validate_bwd(p, wango);
  if (st != TG_OK) return st;
  if (!q || !k || !g || !dout || !dq || !dk || !dg || (dv && !v)) return TG_ERR_INVALID_ARG;
  if (!saved_gbar != !saved_den) return TG_ERR_INVALID_ARG;
  if (saved_gbar && !(aligned16(saved_gbar) && aligned16(saved_den))) return TG_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, g, dout, dq, dk, dg};
  for (const void* x : ptrs)
    if (!aligned16(x)) return TG_ERR_UNSUPPORTED;
  if ((v && !aligned16(v)) || (dv && !aligned16(dv))) return TG_ERR_UNSUPPORTED;
  const BwdWs L = bwd_ws_layout(p, wango);
  st = check_ws(ws, ws_bytes, L.total);
  if (st != TG_OK) return st;
  char* base = static_cast<char*>(ws);
  unsigned* err = nullptr;
  if (error_word(&err) != cudaSuccess) return TG_ERR_CUDA;
  const long long rows = (long long)p->B * p->T;
  const bool norm = !(p->flags & TG_FLAG_QK_NORMALIZED);
  const void* qh = q;
  const void* kh = k;
  cudaError_t e = cudaSuccess;
  if (norm) {
    e = launch_qk_prep(p->dtype, q, base + L.qn, rows, p->T, p->H, p->d_qk, 0.f, true, stream);
    if (e == cudaSuccess) e = launch_qk_prep(p->dtype, k, base + L.kn, rows, p->T, p->H, p->d_qk, 0.f, true, stream);
    if (e != cudaSuccess) return TG_ERR_CUDA;
    qh = base + L.qn;
    kh = base + L.kn;
  }
  void* gbar = base + L.gbar;
  float* dp = reinterpret_cast<float*>(base + L.dp);
  void* E = base + L.E;
  void* aux = base + L.aux;

  // the forward again for gbar and every row's denominator, unless the caller kept them
  // from the forward (the _save calls)
  AggArgs a;
  a.B = p->B; a.T = p->T; a.H = p->H; a.dqk = p->d_qk; a.m = mem_width(p); a.m_h = p->m / p->H;
  a.s = p->s; a.tau = p->tau; a.null_bias = p->null_bias;
  a.window = p->window; a.phi_mode = p->phi_mode; a.flags = 0; a.dtype = p->dtype;
  a.q = qh; a.k = kh; a.g = g; a.v = nullptr; a.out = gbar; a.err = err; a.aux = aux;
  const float* den = nullptr;
  int den_pitch = L.T_pad;
  const void* gb = gbar;
  if (saved_gbar) {
    den = saved_den;
    den_pitch = p->T;
    gb = saved_gbar;
    if (wango) e = launch_wango_prepass(a, stream);  // the feature maps for dq and dk
  } else if (wango) {
    e = launch_wango_tc(a, stream);
    den = wango_den_in_aux(aux, p->B, p->T, p->H, p->d_qk, p->m, p->window);
  } else {
    a.den_out = reinterpret_cast<float*>(base + L.den);
    e = launch_tango_tc(a, stream);
    den = a.den_out;
  }
  if (e != cudaSuccess) return TG_ERR_CUDA;
  e = launch_bwd_prep(dout, v, gb, den, den_pitch, E, dv, dp, p->B, p->T, L.T_pad, p->H, mem_width(p), p->m / p->H,
                      stream);
  if (e != cudaSuccess) return TG_ERR_CUDA;

  // pair-weight gradients, then dq and dk
  BwdPairsArgs pa;
  pa.B = p->B; pa.T = p->T; pa.H = p->H; pa.dqk = p->d_qk; pa.m = mem_width(p); pa.m_h = p->m / p->H;
  pa.wango = wango ? 1 : 0; pa.window = p->window;
  pa.s = p->s; pa.tau = p->tau;
  pa.E = E; pa.g = g; pa.qhat = qh; pa.khat = kh; pa.dp = dp;
  pa.X = base + L.X;
  pa.X_old = wango ? base + L.Xo : nullptr;
  pa.err = err;
  // TG_FLAG_DEBUG_TIMEOUT arms the test hook of the backward's own tensor-core kernels
  // (pairs, scans, dq/dk) only; the forward kernels it also runs get no flags
  const int hook = (p->flags & TG_FLAG_DEBUG_TIMEOUT) ? 1 : 0;
  pa.debug_timeout = hook;
  const size_t part_half = L.scan ? (size_t)bwd_scan_strips(p->B, p->H, p->m / p->H) * p->B * p->T * p->d_qk : 0;
  float* part = reinterpret_cast<float*>(base + L.part);
  if (L.scan) {  // the far older pairs through the running sums; the pair kernel keeps the band
    pa.band = bwd_band(p->window);
    BwdScanArgs sa;
    sa.B = p->B; sa.T = p->T; sa.H = p->H; sa.dqk = p->d_qk; sa.m = mem_width(p); sa.m_h = p->m / p->H;
    sa.window = p->window;
    sa.E = E; sa.g = g;
    sa.fq = wango_fq_in_aux(aux, p->B, p->T, p->H, p->d_qk, p->m, p->window);
    sa.fk = wango_fk_in_aux(aux, p->B, p->T, p->H, p->d_qk, p->m, p->window);
    sa.zb = wango_zb_in_aux(aux, p->B, p->T, p->H, p->d_qk, p->m, p->window);
    sa.dp = dp;
    sa.part[0] = part;
    sa.part[1] = part + part_half;
    sa.rb = reinterpret_cast<float*>(base + L.rb);
    sa.fb = sa.rb + (size_t)p->B * p->H * (L.T_pad / 128) * (p->d_qk / p->H);
    sa.err = err;
    sa.debug_timeout = hook;
    e = launch_bwd_scan(sa, stream);
    if (e != cudaSuccess) return TG_ERR_CUDA;
  }
  e = launch_bwd_pairs_tc(pa, stream);
  if (e != cudaSuccess) return TG_ERR_CUDA;
  BwdQKTcArgs qa;
  qa.B = p->B; qa.T = p->T; qa.H = p->H; qa.dqk = p->d_qk;
  qa.wango = wango ? 1 : 0; qa.window = p->window; qa.phi_mode = p->phi_mode;
  qa.s = p->s; qa.tau = p->tau;
  qa.X = pa.X; qa.X_old = pa.X_old; qa.qhat = qh; qa.khat = kh;
  qa.fq = wango ? wango_fq_in_aux(aux, p->B, p->T, p->H, p->d_qk, p->m, p->window) : nullptr;
  qa.fk = wango ? wango_fk_in_aux(aux, p->B, p->T, p->H, p->d_qk, p->m, p->window) : nullptr;
  qa.raw_q = norm ? q : nullptr;
  qa.raw_k = norm ? k : nullptr;
  qa.dq = dq; qa.dk = dk; qa.err = err;
  qa.debug_timeout = hook;
  if (L.scan) {
    qa.band = bwd_band(p->window);
    qa.far[0] = part;
    qa.far[1] = part + part_half;
  }
  e = launch_bwd_qk_tc(qa, stream);
  if (e != cudaSuccess) return TG_ERR_CUDA;

  // dg: the numerator of the aggregation with destinations and sources exchanged
  AggArgs r = a;
  r.null_bias = nullptr;
  r.no_norm = 1;
  r.den_out = nullptr;
  if (wango) {
    // the windowed kernels on the time-reversed sequence, read and written in place
    // (mirrored: blocks in reverse order, rows reversed within each)
    r.mirror = 1;
    r.q = kh;
    r.k = qh;
    r.g = E;
    r.out = dg;
    e = launch_wango_tc(r, stream);
  } else {
    r.rev = 1;
    r.q = kh;
    r.k = qh;
    r.g = E;
    r.out = dg;
    e = launch_tango_tc(r, stream);
  }
  if (e != cudaSuccess) return TG_ERR_CUDA;

  return TG_OK;
}

}  // namespace
}  // namespace tg

using namespace tg;

extern "C" {

tg_status tango_aggregate(const tg_agg_params* p, const void* q, const void* k, const void* g, const void* v,
                          void* out, void* ws, size_t ws_bytes, tg_stream_t stream) {
  return aggregate(false, p, q, k, g, v, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

tg_status wango_aggregate(const tg_agg_params* p, const void* q, const void* k, const void* g, const void* v,
                          void* out, void* ws, size_t ws_bytes, tg_stream_t stream) {
  return aggregate(true, p, q, k, g, v, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

tg_status tango_aggregate_save(const tg_agg_params* p, const void* q, const void* k, const void* g, const void* v,
                               void* out, void* gbar, float* den, void* ws, size_t ws_bytes, tg_stream_t stream) {
  if (!gbar || !den) return TG_ERR_INVALID_ARG;
  return aggregate(false, p, q, k, g, v, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), gbar, den);
}

tg_status wango_aggregate_save(const tg_agg_params* p, const void* q, const void* k, const void* g, const void* v,
                               void* out, void* gbar, float* den, void* ws, size_t ws_bytes, tg_stream_t stream) {
  if (!gbar || !den) return TG_ERR_INVALID_ARG;
  return aggregate(true, p, q, k, g, v, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), gbar, den);
}

tg_status tango_aggregate_backward(const tg_agg_params* p, const void* q, const void* k, const void* g,
                                   const void* v, const void* dout, const void* gbar, const float* den, void* dq,
                                   void* dk, void* dg, void* dv, void* ws, size_t ws_bytes, tg_stream_t stream) {
  return aggregate_backward(false, p, q, k, g, v, dout, gbar, den, dq, dk, dg, dv, ws, ws_bytes,
                            reinterpret_cast<cudaStream_t>(stream));
}

tg_status wango_aggregate_backward(const tg_agg_params* p, const void* q, const void* k, const void* g,
                                   const void* v, const void* dout, const void* gbar, const float* den, void* dq,
                                   void* dk, void* dg, void* dv, void* ws, size_t ws_bytes, tg_stream_t stream) {
  return aggregate_backward(true, p, q, k, g, v, dout, gbar, den, dq, dk, dg, dv, ws, ws_bytes,
                            reinterpret_cast<cudaStream_t>(stream));
}

// The block forward; with pad_weights false the workspace already holds this weight
// set's per-head padded W_g, W_v, W_o (the model forward's consecutive applications of
// one set).
static tg_status block_forward(const tg_block_params* p, const tg_block_weights* w, const void* h, void* h_out,
                               void* ws, size_t ws_bytes, cudaStream_t stream, bool pad_weights) {
  tg_status st = validate_block(p);
  if (st != TG_OK) return st;
  if (!w || !w->rms_gamma || !w->Wq || !w->Wk || !w->Wg || !w->Wv || !w->Wo || !h || !h_out)
    return TG_ERR_INVALID_ARG;
  const tg_agg_params ap = block_agg(p);  // gate width padded per head where needed
  if (ap.dtype == TG_BF16) {
    const void* ptrs[] = {w->rms_gamma, w->Wq, w->Wk, w->Wg, w->Wv, w->Wo, h, h_out};
    for (const void* x : ptrs)
      if (!aligned16(x)) return TG_ERR_UNSUPPORTED;
  }
  const BlockWs L = block_ws_layout(p);
  st = check_ws(ws, ws_bytes, L.total);
  if (st != TG_OK) return st;
  char* base = static_cast<char*>(ws);
  void *x = base + L.x, *qb = base + L.q, *kb = base + L.k, *gb = base + L.g, *vb = base + L.v;
  const long long BT = (long long)ap.B * ap.T;
  const int M = (int)BT, d = p->d;

  AggArgs a;
  a.B = ap.B; a.T = ap.T; a.H = ap.H; a.dqk = ap.d_qk; a.m = ap.m;
  a.s = ap.s; a.tau = ap.tau; a.null_bias = ap.null_bias;
  a.window = ap.window; a.phi_mode = ap.phi_mode; a.flags = 0; a.dtype = ap.dtype;
  a.q = qb; a.k = kb; a.g = gb; a.v = vb; a.out = vb;  // gbar * v overwrites v in place
  a.aux = base + L.aux;
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return TG_ERR_CUDA;

  // eq. 2 and sec. 2.1: x = RMSNorm(h); q, k, g = SiLU(.), v.
  e = launch_rmsnorm(ap.dtype, h, w->rms_gamma, x, BT, d, p->rms_eps, stream);
  if (e != cudaSuccess) return TG_ERR_CUDA;
  if (ap.dtype == TG_F32) {
    e = launch_gemm_simt(ap.dtype, x, w->Wq, qb, nullptr, M, ap.d_qk, d, ap.d_qk, kEpiStore, stream);
    if (e == cudaSuccess)
      e = launch_gemm_simt(ap.dtype, x, w->Wk, kb, nullptr, M, ap.d_qk, d, ap.d_qk, kEpiStore, stream);
    if (e == cudaSuccess)
      e = launch_qk_prep(ap.dtype, qb, qb, BT, ap.T, ap.H, ap.d_qk, p->rope_base, true, stream);
    if (e == cudaSuccess)
      e = launch_qk_prep(ap.dtype, kb, kb, BT, ap.T, ap.H, ap.d_qk, p->rope_base, true, stream);
    if (e == cudaSuccess)
      e = launch_gemm_simt(ap.dtype, x, w->Wg, gb, nullptr, M, ap.m, d, ap.m, kEpiSilu, stream);
    if (e == cudaSuccess)
      e = launch_gemm_simt(ap.dtype, x, w->Wv, vb, nullptr, M, ap.m, d, ap.m, kEpiStore, stream);
    if (e != cudaSuccess) return TG_ERR_CUDA;
    // eqs. 5-10
    e = p->mode == TG_MODE_WANGO ? launch_wango_simt(a, stream) : launch_tango_simt(a, stream);
    if (e != cudaSuccess) return TG_ERR_CUDA;
    // eq. 3: h_out = h + W_o u
    e = launch_gemm_simt(ap.dtype, vb, w->Wo, h_out, h, M, d, ap.m, d, kEpiResidual, stream);
    return cuda_status(e);
  }
  const void *Wg = w->Wg, *Wv = w->Wv, *Wo = w->Wo;
  if (L.padded) {  // each head's gate rows (W_g, W_v) and columns (W_o) at the padded pitch
    const int m_h = p->agg.m / ap.H, m_hp = ap.m / ap.H;
    if (pad_weights) {
      e = launch_pad_gate(ap.dtype, w->Wg, base + L.wg, ap.m, d, 0, ap.H, m_h, m_hp, stream);
      if (e == cudaSuccess) e = launch_pad_gate(ap.dtype, w->Wv, base + L.wv, ap.m, d, 0, ap.H, m_h, m_hp, stream);
      if (e == cudaSuccess) e = launch_pad_gate(ap.dtype, w->Wo, base + L.wo, d, ap.m, 1, ap.H, m_h, m_hp, stream);
      if (e != cudaSuccess) return TG_ERR_CUDA;
    }
    Wg = base + L.wg;
    Wv = base + L.wv;
    Wo = base + L.wo;
  }
  // on request, WANGO forms v = x W_v^T inside the aggregation (no v tensor in memory)
  const bool fuse_v = p->mode == TG_MODE_WANGO && (p->agg.flags & TG_FLAG_FUSED_V);
  if (fuse_v) {
    a.v = nullptr;  // u goes to the v buffer; v itself is never stored
    a.fuse_x = x;
    a.fuse_wv = Wv;
    a.fuse_d = d;
  }
  ProjArgs pa;
  pa.x = x; pa.Wq = w->Wq; pa.Wk = w->Wk; pa.Wg = Wg; pa.Wv = Wv;
  pa.skip_v = fuse_v ? 1 : 0;
  pa.q = qb; pa.k = kb; pa.g = gb; pa.v = vb;
  pa.M = M; pa.d = d; pa.T = ap.T; pa.H = ap.H; pa.dqk = ap.d_qk; pa.m = ap.m;
  pa.rope_base = p->rope_base; pa.err = a.err;
  pa.debug_timeout = (p->agg.flags & TG_FLAG_DEBUG_TIMEOUT) ? 1 : 0;
  e = launch_proj_tc(pa, stream);
  if (e != cudaSuccess) return TG_ERR_CUDA;
  e = p->mode == TG_MODE_WANGO ? launch_wango_tc(a, stream) : launch_tango_tc(a, stream);
  if (e != cudaSuccess) return TG_ERR_CUDA;
  e = launch_out_tc(vb, Wo, h, h_out, M, d, ap.m, a.err, stream);
  return cuda_status(e);
}

tg_status tango_block_forward(const tg_block_params* p, const tg_block_weights* w, const void* h, void* h_out,
                              void* ws, size_t ws_bytes, tg_stream_t stream) {
  return block_forward(p, w, h, h_out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), true);
}

tg_status tango_model_forward(const tg_model_params* p, const tg_model_weights* w, const int* ids, void* logits,
                              void* ws, size_t ws_bytes, tg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  tg_status st = validate_model(p);
  if (st != TG_OK) return st;
  if (!w || !w->embedding || !w->final_gamma || !w->sets || !ids || !logits) return TG_ERR_INVALID_ARG;
  const tg_agg_params& ap = p->block.agg;
  if (ap.dtype == TG_BF16 && !(aligned16(w->embedding) && aligned16(w->final_gamma) && aligned16(logits)))
    return TG_ERR_UNSUPPORTED;
  const ModelWs L = model_ws_layout(p);
  st = check_ws(ws, ws_bytes, L.total);
  if (st != TG_OK) return st;
  char* base = static_cast<char*>(ws);
  void *h = base + L.h, *x = base + L.x, *bws = base + L.block;
  const long long BT = (long long)ap.B * ap.T;
  const int d = p->block.d;
  unsigned* err = nullptr;
  if (error_word(&err) != cudaSuccess) return TG_ERR_CUDA;

  // h^(0): token embeddings (the tied matrix)
  if (launch_embed(ap.dtype, ids, w->embedding, h, BT, d, p->vocab, err, stream) != cudaSuccess) return TG_ERR_CUDA;
  // eq. 11: h^(r+1) = Block(h^(r)), in place
  // (a set's padded gate weights stay in the block workspace while the next application
  // uses the same set)
  for (int r = 0; r < p->n_apps; ++r) {
    const bool new_set = r == 0 || set_of(p, r) != set_of(p, r - 1);
    st = block_forward(&p->block, &w->sets[set_of(p, r)], h, h, bws, L.total - L.block, stream, new_set);
    if (st != TG_OK) return st;
  }
  // final RMSNorm, then logits against the tied embedding: x E^T
  if (launch_rmsnorm(ap.dtype, h, w->final_gamma, x, BT, d, p->final_rms_eps, stream) != cudaSuccess)
    return TG_ERR_CUDA;
  cudaError_t e = ap.dtype == TG_BF16
                      ? launch_matmul_tc(x, w->embedding, logits, (int)BT, p->vocab, d, err, stream)
                      : launch_gemm_simt(ap.dtype, x, w->embedding, logits, nullptr, (int)BT, p->vocab, d, p->vocab,
                                         kEpiStore, stream);
  return cuda_status(e);
}

tg_status wango_decode_step(const tg_agg_params* p, long long pos, const void* q, const void* k, const void* g,
                            const void* v, void* out, void* state, size_t state_bytes, tg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  tg_status st = validate_decode(p);
  if (st != TG_OK) return st;
  if (pos < 0 || !q || !k || !g || !out) return TG_ERR_INVALID_ARG;
  const DecodeWs L = decode_ws_layout(p);
  st = check_ws(state, state_bytes, L.total);
  if (st != TG_OK) return st;
  char* base = static_cast<char*>(state);
  if (pos == 0 && cudaMemsetAsync(state, 0, L.total, stream) != cudaSuccess) return TG_ERR_CUDA;
  DecodeState ds;
  ds.S = reinterpret_cast<float*>(base + L.S);
  ds.z = reinterpret_cast<float*>(base + L.z);
  ds.ring_k = base + L.ring_k;
  ds.ring_g = base + L.ring_g;
  ds.w = reinterpret_cast<float*>(base + L.w);
  ds.fq = reinterpret_cast<float*>(base + L.fq);
  ds.fk_fold = reinterpret_cast<float*>(base + L.fk);
  ds.wpart = reinterpret_cast<float*>(base + L.wpart);
  ds.older = reinterpret_cast<float*>(base + L.older);
  unsigned* err = nullptr;
  if (error_word(&err) != cudaSuccess) return TG_ERR_CUDA;
  return cuda_status(launch_wango_decode(p->dtype, p->B, p->H, p->d_qk, p->m, p->window, pos, p->s, p->tau,
                                         p->null_bias, p->phi_mode, (p->flags & TG_FLAG_QK_NORMALIZED) ? 1 : 0, q,
                                         k, g, v, out, ds, err, stream));
}

size_t tg_workspace_size(int which, const void* params) {
  if (!params) return 0;
  if (which == TG_WS_TANGO || which == TG_WS_WANGO) {
    const tg_agg_params* p = static_cast<const tg_agg_params*>(params);
    if (validate_agg(p, which == TG_WS_WANGO) != TG_OK) return 0;
    return agg_ws_bytes(p, which == TG_WS_WANGO);
  }
  if (which == TG_WS_BLOCK) {
    const tg_block_params* p = static_cast<const tg_block_params*>(params);
    if (validate_block(p) != TG_OK) return 0;
    return block_ws_layout(p).total;
  }
  if (which == TG_WS_DECODE) {
    const tg_agg_params* p = static_cast<const tg_agg_params*>(params);
    if (validate_decode(p) != TG_OK) return 0;
    return decode_ws_layout(p).total;
  }
  if (which == TG_WS_TANGO_BWD || which == TG_WS_WANGO_BWD) {
    const tg_agg_params* p = static_cast<const tg_agg_params*>(params);
    const bool wango = which == TG_WS_WANGO_BWD;
    if (validate_bwd(p, wango) != TG_OK) return 0;
    return bwd_ws_layout(p, wango).total;
  }
  if (which == TG_WS_MODEL) {
    const tg_model_params* p = static_cast<const tg_model_params*>(params);
    if (validate_model(p) != TG_OK) return 0;
    return model_ws_layout(p).total;
  }
  return 0;
}

const char* tg_status_string(tg_status s) {
  switch (s) {
    case TG_OK: return "ok";
    case TG_ERR_INVALID_ARG: return "invalid argument";
    case TG_ERR_UNSUPPORTED: return "unsupported shape, alignment or dtype";
    case TG_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case TG_ERR_CUDA: return "CUDA call failed";
    case TG_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case TG_ERR_DEVICE: return "out-of-range value in device memory";
  }
  return "unknown status";
}

tg_status tg_check_device_error(tg_stream_t stream, unsigned* detail) {
  if (detail) *detail = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return TG_ERR_CUDA;
  unsigned* dev = nullptr;
  if (error_word(&dev) != cudaSuccess) return TG_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dev, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return TG_ERR_CUDA;
  if (word != 0 && cudaMemset(dev, 0, sizeof word) != cudaSuccess) return TG_ERR_CUDA;
  if (detail) *detail = word;
  if (word & kErrTimeout) return TG_ERR_TIMEOUT;
  if (word & kErrValue) return TG_ERR_DEVICE;
  return TG_OK;
}

int tg_version(void) { return 100; }

}  // extern "C"
