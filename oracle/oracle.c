/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the cross-token gate aggregation
 * of "TANGO: Token-Aggregated Nonlinear Gating Operators for Natural and Formal
 * Language Modeling" (arXiv 2608.22117).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  It shares no
 * code, header, table or constant with the CUDA path, and the CUDA path never
 * calls it.
 *
 * Every function evaluates the paper's definitions directly, in double
 * precision, in the order the paper states them:
 *   - pre-RMSNorm, SwiGLU gate and projected features     (sec. 2.1, eq. 2)
 *   - RoPE, then unit-normalised per-head queries/keys    (sec. 2.1)
 *   - logit  l_ij = tau_a q_i . k_j                        (sec. 2.1, eq. 4)
 *   - null-gate weight n_i exp(b_a) in the denominator     (sec. 2.1, eq. 5)
 *   - TANGO weights exp(l_ij) on every visible source      (sec. 2.2, eq. 6)
 *   - WANGO window / older-prefix partition                (sec. 2.2, eq. 7)
 *   - feature map phi and older-source weight              (sec. 2.2, eqs. 8-9)
 *   - running sums S, z                                    (sec. 2.2, eq. 10)
 *   - residual update h+ = h + W_o(gbar * v)               (sec. 2.1, eq. 3)
 *   - gradients of eq. 5 with respect to q, k, g and v     (derivative of eqs. 4-9)
 *
 * Inputs may be fp64, fp32 or bf16 (raw 16-bit patterns); they are widened
 * exactly to fp64 before any arithmetic, so input quantisation is never an
 * oracle error.  No softmax shift is used: logits are bounded by tau <= 20,
 * so exp() cannot overflow in fp64.
 *
 * Readings of points the paper leaves open (each is also listed in the design
 * notes): heads are given by the caller (H), RoPE uses base `rope_base`
 * (0 = off) with rotate-half pairing (c, c + d_h/2) and positions 0..T-1,
 * unit normalisation divides by max(|q|, 1e-12), n_i = i + 1 for both TANGO
 * and WANGO, the window includes the destination itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F64 = 0, OR_F32 = 1, OR_BF16 = 2 };

#define OR_OK 0
#define OR_EINVAL -1
#define OR_ENOMEM -2

/* ---------------------------------------------------------------- access */

static double widen_bf16(uint16_t bits16) {
    uint32_t bits = (uint32_t)bits16 << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double ld(const void *p, int dt, size_t idx) {
    if (dt == OR_F64) return ((const double *)p)[idx];
    if (dt == OR_F32) return (double)((const float *)p)[idx];
    return widen_bf16(((const uint16_t *)p)[idx]);
}

/* acc[n] += w * src[off + n], n < len */
static void axpy_from(double *acc, double w, const void *src, int dt, size_t off, int len) {
    if (dt == OR_F64) {
        const double *s = (const double *)src + off;
        for (int n = 0; n < len; ++n) acc[n] += w * s[n];
    } else if (dt == OR_F32) {
        const float *s = (const float *)src + off;
        for (int n = 0; n < len; ++n) acc[n] += w * (double)s[n];
    } else {
        const uint16_t *s = (const uint16_t *)src + off;
        for (int n = 0; n < len; ++n) acc[n] += w * widen_bf16(s[n]);
    }
}

/* copy len elements of src starting at off into dst as fp64 */
static void widen_row(double *dst, const void *src, int dt, size_t off, int len) {
    for (int n = 0; n < len; ++n) dst[n] = ld(src, dt, off + (size_t)n);
}

static double dot(const double *a, const double *b, int n) {
    double s = 0.0;
    for (int c = 0; c < n; ++c) s += a[c] * b[c];
    return s;
}

/* ---------------------------------------------------------- definitions */

/* Unit-normalise one head vector (sec. 2.1: "normalize each query and key
 * to unit length"). */
static void unit_normalize(double *x, int n) {
    double s = sqrt(dot(x, x, n));
    if (s < 1e-12) s = 1e-12;
    for (int c = 0; c < n; ++c) x[c] /= s;
}

/* Feature map of eq. 8 (mode 0): max(ELU(u) + 1 + eps, eps) / sqrt(d_h),
 * eps = 1e-4.  Mode 1 is the literal ELU(u) + 1 without eps or scaling. */
static double phi(double u, int d_h, int mode) {
    double elu = u > 0.0 ? u : expm1(u);
    if (mode == 1) return elu + 1.0;
    const double eps = 1e-4;
    double t = elu + 1.0 + eps;
    if (t < eps) t = eps;
    return t / sqrt((double)d_h);
}

/* SiLU(u) = u * sigmoid(u) (eq. 2 gate nonlinearity). */
static double silu(double u) { return u / (1.0 + exp(-u)); }

/* Rotary embedding at position t on one head vector of width d_h,
 * rotate-half pairing (c, c + d_h/2), frequency base^(-2c/d_h). */
static void rope(double *x, int d_h, int t, double base) {
    int half = d_h / 2;
    for (int c = 0; c < half; ++c) {
        double theta = (double)t * pow(base, -2.0 * (double)c / (double)d_h);
        double cs = cos(theta), sn = sin(theta);
        double x1 = x[c], x2 = x[c + half];
        x[c] = x1 * cs - x2 * sn;
        x[c + half] = x1 * sn + x2 * cs;
    }
}

/* Normalised per-head copies of q/k (B*T*dqk doubles). */
static double *prep_unit(const void *x, int dt, long long BT, int H, int dqk, int already_unit) {
    int d_h = dqk / H;
    double *out = (double *)malloc(sizeof(double) * (size_t)BT * (size_t)dqk);
    if (!out) return NULL;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < BT; ++r) {
        double *o = out + (size_t)r * dqk;
        widen_row(o, x, dt, (size_t)r * dqk, dqk);
        if (!already_unit)
            for (int a = 0; a < H; ++a) unit_normalize(o + (size_t)a * d_h, d_h);
    }
    return out;
}

/* phi(sqrt(tau_a) * unit) features (eq. 9), same layout as the unit array. */
static double *prep_phi(const double *unit, long long BT, int H, int dqk, const double *tau, int mode) {
    int d_h = dqk / H;
    double *out = (double *)malloc(sizeof(double) * (size_t)BT * (size_t)dqk);
    if (!out) return NULL;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < BT; ++r)
        for (int a = 0; a < H; ++a) {
            double st = sqrt(tau[a]);
            for (int c = 0; c < d_h; ++c) {
                size_t idx = (size_t)r * dqk + (size_t)a * d_h + c;
                out[idx] = phi(st * unit[idx], d_h, mode);
            }
        }
    return out;
}

static int check_dims(int B, int T, int H, int dqk, int m) {
    if (B < 1 || T < 1 || H < 1 || dqk < 1 || m < 1) return 0;
    if (dqk % H != 0 || m % H != 0) return 0;
    return 1;
}

/*
 * One destination row of eq. 5 for every head.  mode 0 = TANGO (eq. 6 on all
 * j <= i); mode 1 = WANGO (eq. 6 inside the window of eq. 7, eq. 9 on the
 * older prefix), evaluated pair by pair.
 *   qn/kn: unit q/k for this sequence ([T, dqk]); fq/fk: phi features (WANGO)
 *   g/v: this sequence's rows start at row0 (element offset row0*m)
 *   out: m doubles (gbar * v, or gbar when v == NULL)
 */
static void aggregate_row(int mode, int i, int T, int H, int dqk, int m, int W,
                          const double *qn, const double *kn, const double *fq, const double *fk,
                          const void *g, int gdt, const void *v, int vdt, size_t row0,
                          const double *tau, const double *null_b, double *out) {
    int d_h = dqk / H, m_h = m / H;
    (void)T;
    for (int a = 0; a < H; ++a) {
        double *num = out + (size_t)a * m_h;
        for (int n = 0; n < m_h; ++n) num[n] = 0.0;
        double den = 0.0;
        const double *qi = qn + (size_t)i * dqk + (size_t)a * d_h;
        for (int j = 0; j <= i; ++j) {
            double w;
            if (mode == 0 || j >= i - W + 1) {
                const double *kj = kn + (size_t)j * dqk + (size_t)a * d_h;
                w = exp(tau[a] * dot(qi, kj, d_h));                         /* eq. 6 */
            } else {
                w = dot(fq + (size_t)i * dqk + (size_t)a * d_h,
                        fk + (size_t)j * dqk + (size_t)a * d_h, d_h);       /* eq. 9 */
            }
            den += w;
            axpy_from(num, w, g, gdt, (row0 + (size_t)j) * (size_t)m + (size_t)a * m_h, m_h);
        }
        if (null_b) den += (double)(i + 1) * exp(null_b[a]);               /* eq. 5 */
        for (int n = 0; n < m_h; ++n) {
            double gbar = num[n] / den;
            num[n] = v ? gbar * ld(v, vdt, (row0 + (size_t)i) * (size_t)m + (size_t)a * m_h + n) : gbar;
        }
    }
}

static int aggregate_rows(int mode, int B, int T, int H, int dqk, int m, int W, int phi_mode,
                          const void *q, int qdt, const void *k, int kdt,
                          const void *g, int gdt, const void *v, int vdt,
                          const double *tau, const double *null_b, int qk_normalized,
                          const long long *rows, long long nrows, double *out) {
    if (!check_dims(B, T, H, dqk, m) || (mode == 1 && W < 1)) return OR_EINVAL;
    long long BT = (long long)B * T;
    double *qn = prep_unit(q, qdt, BT, H, dqk, qk_normalized);
    double *kn = prep_unit(k, kdt, BT, H, dqk, qk_normalized);
    double *fq = NULL, *fk = NULL;
    if (mode == 1 && qn && kn) {
        fq = prep_phi(qn, BT, H, dqk, tau, phi_mode);
        fk = prep_phi(kn, BT, H, dqk, tau, phi_mode);
    }
    if (!qn || !kn || (mode == 1 && (!fq || !fk))) {
        free(qn); free(kn); free(fq); free(fk);
        return OR_ENOMEM;
    }
    long long nr = rows ? nrows : BT;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long r = 0; r < nr; ++r) {
        long long flat = rows ? rows[r] : r;
        if (flat < 0 || flat >= BT) { bad = 1; continue; }
        long long b = flat / T;
        int i = (int)(flat % T);
        size_t row0 = (size_t)b * T;
        aggregate_row(mode, i, T, H, dqk, m, W,
                      qn + row0 * dqk, kn + row0 * dqk,
                      fq ? fq + row0 * dqk : NULL, fk ? fk + row0 * dqk : NULL,
                      g, gdt, v, vdt, row0, tau, null_b, out + (size_t)r * m);
    }
    free(qn); free(kn); free(fq); free(fk);
    return bad ? OR_EINVAL : OR_OK;
}

/* ------------------------------------------------------------ exports */

/* TANGO (eqs. 5-6).  rows: flat indices b*T+i to evaluate (NULL = all B*T);
 * out: [nrows or B*T, m]. */
int oracle_tango(int B, int T, int H, int dqk, int m,
                 const void *q, int qdt, const void *k, int kdt,
                 const void *g, int gdt, const void *v, int vdt,
                 const double *tau, const double *null_b, int qk_normalized,
                 const long long *rows, long long nrows, double *out) {
    return aggregate_rows(0, B, T, H, dqk, m, 1, 0, q, qdt, k, kdt, g, gdt, v, vdt,
                          tau, null_b, qk_normalized, rows, nrows, out);
}

/* WANGO evaluated pair by pair, O(T^2) (eqs. 5-9). */
int oracle_wango_direct(int B, int T, int H, int dqk, int m, int W, int phi_mode,
                        const void *q, int qdt, const void *k, int kdt,
                        const void *g, int gdt, const void *v, int vdt,
                        const double *tau, const double *null_b, int qk_normalized,
                        const long long *rows, long long nrows, double *out) {
    return aggregate_rows(1, B, T, H, dqk, m, W, phi_mode, q, qdt, k, kdt, g, gdt, v, vdt,
                          tau, null_b, qk_normalized, rows, nrows, out);
}

/*
 * WANGO with the running sums of eq. 10, walking destinations i = 0..T-1:
 * before destination i is evaluated, the source j = i - W (the token that
 * has just left the trailing window) is added to S = sum phi(k~) g^T and
 * z = sum phi(k~).  The older-prefix numerator and denominator are then
 * phi(q~_i)^T S and phi(q~_i)^T z; window sources are added pair by pair.
 * Work units are (b, head, block of gate columns); out: [B*T, m].
 */
int oracle_wango_scan(int B, int T, int H, int dqk, int m, int W, int phi_mode,
                      const void *q, int qdt, const void *k, int kdt,
                      const void *g, int gdt, const void *v, int vdt,
                      const double *tau, const double *null_b, int qk_normalized,
                      double *out) {
    if (!check_dims(B, T, H, dqk, m) || W < 1) return OR_EINVAL;
    int d_h = dqk / H, m_h = m / H;
    const int NC = 64;
    int nchunks = (m_h + NC - 1) / NC;
    long long BT = (long long)B * T;
    double *qn = prep_unit(q, qdt, BT, H, dqk, qk_normalized);
    double *kn = prep_unit(k, kdt, BT, H, dqk, qk_normalized);
    double *fq = qn ? prep_phi(qn, BT, H, dqk, tau, phi_mode) : NULL;
    double *fk = kn ? prep_phi(kn, BT, H, dqk, tau, phi_mode) : NULL;
    if (!qn || !kn || !fq || !fk) {
        free(qn); free(kn); free(fq); free(fk);
        return OR_ENOMEM;
    }
    long long units = (long long)B * H * nchunks;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long u = 0; u < units; ++u) {
        int c0 = (int)(u % nchunks) * NC;
        int a = (int)((u / nchunks) % H);
        long long b = u / ((long long)nchunks * H);
        int nc = m_h - c0 < NC ? m_h - c0 : NC;
        double *S = (double *)calloc((size_t)d_h * NC, sizeof(double));
        double *z = (double *)calloc((size_t)d_h, sizeof(double));
        double *num = (double *)malloc(sizeof(double) * NC);
        if (!S || !z || !num) { fail = 1; free(S); free(z); free(num); continue; }
        size_t row0 = (size_t)b * T;
        size_t col0 = (size_t)a * m_h + (size_t)c0;
        for (int i = 0; i < T; ++i) {
            int jn = i - W;                         /* leaves the window now */
            if (jn >= 0) {
                const double *fkj = fk + (row0 + jn) * dqk + (size_t)a * d_h;
                for (int c = 0; c < d_h; ++c) {
                    z[c] += fkj[c];
                    axpy_from(S + (size_t)c * NC, fkj[c], g, gdt, (row0 + jn) * (size_t)m + col0, nc);
                }
            }
            const double *fqi = fq + (row0 + i) * dqk + (size_t)a * d_h;
            for (int n = 0; n < nc; ++n) {
                double s = 0.0;
                for (int c = 0; c < d_h; ++c) s += fqi[c] * S[(size_t)c * NC + n];
                num[n] = s;
            }
            double den = dot(fqi, z, d_h);
            const double *qi = qn + (row0 + i) * dqk + (size_t)a * d_h;
            int jlo = i - W + 1 > 0 ? i - W + 1 : 0;
            for (int j = jlo; j <= i; ++j) {
                double w = exp(tau[a] * dot(qi, kn + (row0 + j) * dqk + (size_t)a * d_h, d_h));
                den += w;
                axpy_from(num, w, g, gdt, (row0 + j) * (size_t)m + col0, nc);
            }
            if (null_b) den += (double)(i + 1) * exp(null_b[a]);
            double *o = out + (row0 + i) * (size_t)m + col0;
            for (int n = 0; n < nc; ++n) {
                double gbar = num[n] / den;
                o[n] = v ? gbar * ld(v, vdt, (row0 + i) * (size_t)m + col0 + n) : gbar;
            }
        }
        free(S); free(z); free(num);
    }
    free(qn); free(kn); free(fq); free(fk);
    return fail ? OR_ENOMEM : OR_OK;
}

/* y[r] = sum_c W[r, c] x[c] for a row-major [rows, cols] matrix */
static void matvec(double *y, const void *Wm, int wdt, int rows, int cols, const double *x) {
    for (int r = 0; r < rows; ++r) {
        double s = 0.0;
        size_t base = (size_t)r * cols;
        if (wdt == OR_F64) {
            const double *w = (const double *)Wm + base;
            for (int c = 0; c < cols; ++c) s += w[c] * x[c];
        } else if (wdt == OR_F32) {
            const float *w = (const float *)Wm + base;
            for (int c = 0; c < cols; ++c) s += (double)w[c] * x[c];
        } else {
            const uint16_t *w = (const uint16_t *)Wm + base;
            for (int c = 0; c < cols; ++c) s += widen_bf16(w[c]) * x[c];
        }
        y[r] = s;
    }
}

/* RMSNorm with gain: gamma * h / sqrt(mean(h^2) + eps) (sec. 2.1). */
static void rmsnorm_row(double *x, const void *h, int hdt, size_t off, int d,
                        const void *gamma, int gdt, double eps) {
    double ss = 0.0;
    for (int c = 0; c < d; ++c) {
        double t = ld(h, hdt, off + c);
        x[c] = t;
        ss += t * t;
    }
    double r = 1.0 / sqrt(ss / (double)d + eps);
    for (int c = 0; c < d; ++c) x[c] = x[c] * r * ld(gamma, gdt, (size_t)c);
}

/*
 * One block application for the selected sequences (batches[0..nb)):
 *   x = RMSNorm(h); q,k = W_q x, W_k x; g = SiLU(W_g x); v = W_v x   (eq. 2)
 *   per head: RoPE (rope_base > 0), unit-normalise                    (sec. 2.1)
 *   gbar by TANGO (mode 0) or WANGO (mode 1), pair by pair            (eqs. 5-9)
 *   h+ = h + W_o (gbar * v)                                           (eq. 3)
 * Weights are row-major [out, in].  wdt is the dtype of gamma and all W;
 * hdt the dtype of h.  h_out: [nb, T, d].  Optional intermediate outputs
 * (NULL to skip), each [nb, T, .]: q_out/k_out (unit, after RoPE),
 * g_out, v_out, u_out (= gbar * v).
 */
int oracle_block_forward(int B, int T, int d, int H, int dqk, int m, int mode, int W, int phi_mode,
                         double rms_eps, double rope_base,
                         const void *gamma, const void *Wq, const void *Wk, const void *Wg,
                         const void *Wv, const void *Wo, int wdt,
                         const void *h, int hdt, const double *tau, const double *null_b,
                         const long long *batches, int nb, double *h_out,
                         double *q_out, double *k_out, double *g_out, double *v_out, double *u_out) {
    if (!check_dims(B, T, H, dqk, m) || d < 1 || nb < 1 || (mode == 1 && W < 1)) return OR_EINVAL;
    int d_h = dqk / H;
    if (rope_base > 0.0 && d_h % 2 != 0) return OR_EINVAL;
    size_t Tz = (size_t)T;
    double *qn = (double *)malloc(sizeof(double) * Tz * dqk);
    double *kn = (double *)malloc(sizeof(double) * Tz * dqk);
    double *gg = (double *)malloc(sizeof(double) * Tz * m);
    double *vv = (double *)malloc(sizeof(double) * Tz * m);
    double *uu = (double *)malloc(sizeof(double) * Tz * m);
    if (!qn || !kn || !gg || !vv || !uu) {
        free(qn); free(kn); free(gg); free(vv); free(uu);
        return OR_ENOMEM;
    }
    int status = OR_OK;
    for (int s = 0; s < nb && status == OR_OK; ++s) {
        long long b = batches[s];
        if (b < 0 || b >= B) { status = OR_EINVAL; break; }
        size_t hrow0 = (size_t)b * Tz;
#pragma omp parallel
        {
            double *x = (double *)malloc(sizeof(double) * (size_t)d);
            double *pre = (double *)malloc(sizeof(double) * (size_t)m);
#pragma omp for schedule(static)
            for (int t = 0; t < T; ++t) {
                if (!x || !pre) { status = OR_ENOMEM; continue; }
                rmsnorm_row(x, h, hdt, (hrow0 + t) * (size_t)d, d, gamma, wdt, rms_eps);
                double *qt = qn + (size_t)t * dqk, *kt = kn + (size_t)t * dqk;
                matvec(qt, Wq, wdt, dqk, d, x);
                matvec(kt, Wk, wdt, dqk, d, x);
                for (int a = 0; a < H; ++a) {
                    if (rope_base > 0.0) {
                        rope(qt + (size_t)a * d_h, d_h, t, rope_base);
                        rope(kt + (size_t)a * d_h, d_h, t, rope_base);
                    }
                    unit_normalize(qt + (size_t)a * d_h, d_h);
                    unit_normalize(kt + (size_t)a * d_h, d_h);
                }
                matvec(pre, Wg, wdt, m, d, x);
                for (int n = 0; n < m; ++n) gg[(size_t)t * m + n] = silu(pre[n]);
                matvec(vv + (size_t)t * m, Wv, wdt, m, d, x);
            }
            free(x); free(pre);
        }
        double *fq = NULL, *fk = NULL;
        if (mode == 1) {
            fq = prep_phi(qn, T, H, dqk, tau, phi_mode);
            fk = prep_phi(kn, T, H, dqk, tau, phi_mode);
            if (!fq || !fk) { free(fq); free(fk); status = OR_ENOMEM; break; }
        }
#pragma omp parallel for schedule(dynamic, 1)
        for (int i = 0; i < T; ++i)
            aggregate_row(mode, i, T, H, dqk, m, W, qn, kn, fq, fk, gg, OR_F64, vv, OR_F64, 0,
                          tau, null_b, uu + (size_t)i * m);
        free(fq); free(fk);
#pragma omp parallel
        {
            double *y = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
            for (int t = 0; t < T; ++t) {
                if (!y) { status = OR_ENOMEM; continue; }
                matvec(y, Wo, wdt, d, m, uu + (size_t)t * m);
                double *ho = h_out + ((size_t)s * Tz + t) * d;
                for (int c = 0; c < d; ++c) ho[c] = ld(h, hdt, (hrow0 + t) * (size_t)d + c) + y[c];
            }
            free(y);
        }
        size_t o = (size_t)s * Tz;
        if (q_out) memcpy(q_out + o * dqk, qn, sizeof(double) * Tz * dqk);
        if (k_out) memcpy(k_out + o * dqk, kn, sizeof(double) * Tz * dqk);
        if (g_out) memcpy(g_out + o * m, gg, sizeof(double) * Tz * m);
        if (v_out) memcpy(v_out + o * m, vv, sizeof(double) * Tz * m);
        if (u_out) memcpy(u_out + o * m, uu, sizeof(double) * Tz * m);
    }
    free(qn); free(kn); free(gg); free(vv); free(uu);
    return status;
}

/* Token-embedding lookup: out[r] = E[ids[r]] (the tied input matrix, sec. 2.3). */
int oracle_embed(long long n, const long long *ids, int d, int vocab,
                 const void *E, int edt, double *out) {
    for (long long r = 0; r < n; ++r) {
        if (ids[r] < 0 || ids[r] >= vocab) return OR_EINVAL;
        widen_row(out + (size_t)r * d, E, edt, (size_t)ids[r] * d, d);
    }
    return OR_OK;
}

/* Final RMSNorm then logits with the tied embedding matrix E [vocab, d]
 * (sec. 2.3).  h: [n, d] fp64; out: [n, vocab]. */
int oracle_final_logits(long long n, int d, int vocab, const double *h, const void *gamma, int gdt,
                        double eps, const void *E, int edt, double *out) {
    int fail = 0;
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
        for (long long r = 0; r < n; ++r) {
            if (!x) { fail = 1; continue; }
            rmsnorm_row(x, h, OR_F64, (size_t)r * d, d, gamma, gdt, eps);
            matvec(out + (size_t)r * vocab, E, edt, vocab, d, x);
        }
        free(x);
    }
    return fail ? OR_ENOMEM : OR_OK;
}

/* ------------------------------------------------------------ gradients */

/* Derivative of the feature map with respect to its argument: ELU'(u) = 1 for
 * u > 0 and e^u otherwise, divided by sqrt(d_h) for eq. 8 (mode 0).  The
 * max(., eps) of eq. 8 never binds, since ELU(u) + 1 > 0. */
static double phi_deriv(double u, int d_h, int mode) {
    double e = u > 0.0 ? 1.0 : exp(u);
    return mode == 1 ? e : e / sqrt((double)d_h);
}

/*
 * Gradients of the scalar L = sum_{i,c} dout_ic u_ic, where u = gbar * v (or
 * u = gbar when v == NULL) is the aggregation of eq. 5 with TANGO (mode 0, eq. 6)
 * or WANGO (mode 1, eqs. 7-9) weights, with respect to q, k, g and v.  Each pair
 * is taken directly from the derivative of eq. 5, per batch and head:
 *   alpha_ij = w_ij / den_i,  gbar_i = sum_{j<=i} alpha_ij g_j
 *   dgbar_i = dout_i * v_i (dout_i without v),  dv_i = dout_i * gbar_i
 *   dg_j = sum_{i>=j} alpha_ij dgbar_i
 *   dL/dw_ij = (g_j . dgbar_i - gbar_i . dgbar_i) / den_i   (the null term carries no
 *                                                            value, only weight)
 *   window pair, w = exp(tau qhat_i . khat_j):
 *       dqhat_i += tau w dL/dw khat_j,   dkhat_j += tau w dL/dw qhat_i
 *   older pair, w = phi(x_i) . phi(y_j) with x = sqrt(tau) qhat, y = sqrt(tau) khat:
 *       dqhat_i += sqrt(tau) dL/dw phi'(x_i) * phi(y_j)
 *       dkhat_j += sqrt(tau) dL/dw phi(x_i) * phi'(y_j)
 *   unit normalisation qhat = q / max(|q|, 1e-12) (sec. 2.1):
 *       dq = (dqhat - qhat (qhat . dqhat)) / |q|, or dqhat / 1e-12 where the clamp holds
 * Outputs (fp64): dq, dk [B*T, dqk]; dg [B*T, m]; dv [B*T, m] (untouched when v == NULL).
 */
static int agg_backward(int mode, int B, int T, int H, int dqk, int m, int W, int phi_mode,
                        const void *q, int qdt, const void *k, int kdt,
                        const void *g, int gdt, const void *v, int vdt, const void *dout, int odt,
                        const double *tau, const double *null_b, int qk_normalized,
                        double *dq, double *dk, double *dg, double *dv) {
    if (!check_dims(B, T, H, dqk, m) || (mode == 1 && W < 1)) return OR_EINVAL;
    int d_h = dqk / H, m_h = m / H;
    long long BT = (long long)B * T;
    double *qn = prep_unit(q, qdt, BT, H, dqk, qk_normalized);
    double *kn = prep_unit(k, kdt, BT, H, dqk, qk_normalized);
    double *fq = NULL, *fk = NULL;
    if (mode == 1 && qn && kn) {
        fq = prep_phi(qn, BT, H, dqk, tau, phi_mode);
        fk = prep_phi(kn, BT, H, dqk, tau, phi_mode);
    }
    if (!qn || !kn || (mode == 1 && (!fq || !fk))) {
        free(qn); free(kn); free(fq); free(fk);
        return OR_ENOMEM;
    }
    memset(dq, 0, sizeof(double) * (size_t)BT * dqk);
    memset(dk, 0, sizeof(double) * (size_t)BT * dqk);
    memset(dg, 0, sizeof(double) * (size_t)BT * m);
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long u = 0; u < (long long)B * H; ++u) {
        int a = (int)(u % H);
        size_t row0 = (size_t)(u / H) * T;
        double *gbar = (double *)malloc(sizeof(double) * (size_t)T * m_h);
        double *dgb = (double *)malloc(sizeof(double) * (size_t)T * m_h);
        double *den = (double *)malloc(sizeof(double) * (size_t)T);
        double *delta = (double *)malloc(sizeof(double) * (size_t)T);
        double *gj = (double *)malloc(sizeof(double) * (size_t)m_h);
        double *dqh = (double *)calloc((size_t)T * d_h, sizeof(double));
        double *dkh = (double *)calloc((size_t)T * d_h, sizeof(double));
        if (!gbar || !dgb || !den || !delta || !gj || !dqh || !dkh) {
            fail = 1;
            free(gbar); free(dgb); free(den); free(delta); free(gj); free(dqh); free(dkh);
            continue;
        }
        const double st = sqrt(tau[a]);
        /* weight of pair (i, j), j <= i: eq. 6 inside the window, eq. 9 older */
#define PAIR_W(i, j) ((mode == 0 || (j) >= (i) - W + 1)                                          \
        ? exp(tau[a] * dot(qn + (row0 + (i)) * dqk + (size_t)a * d_h,                            \
                           kn + (row0 + (j)) * dqk + (size_t)a * d_h, d_h))                      \
        : dot(fq + (row0 + (i)) * dqk + (size_t)a * d_h, fk + (row0 + (j)) * dqk + (size_t)a * d_h, d_h))
        /* the forward pass: den_i and gbar_i */
        for (int i = 0; i < T; ++i) {
            double *gb = gbar + (size_t)i * m_h;
            for (int n = 0; n < m_h; ++n) gb[n] = 0.0;
            double dsum = 0.0;
            for (int j = 0; j <= i; ++j) {
                double w = PAIR_W(i, j);
                dsum += w;
                axpy_from(gb, w, g, gdt, (row0 + j) * (size_t)m + (size_t)a * m_h, m_h);
            }
            if (null_b) dsum += (double)(i + 1) * exp(null_b[a]);
            den[i] = dsum;
            for (int n = 0; n < m_h; ++n) gb[n] /= dsum;
        }
        /* dgbar, dv and delta_i = gbar_i . dgbar_i */
        for (int i = 0; i < T; ++i) {
            size_t off = (row0 + i) * (size_t)m + (size_t)a * m_h;
            double dl = 0.0;
            for (int n = 0; n < m_h; ++n) {
                double o = ld(dout, odt, off + n);
                double x = v ? o * ld(v, vdt, off + n) : o;
                dgb[(size_t)i * m_h + n] = x;
                dl += gbar[(size_t)i * m_h + n] * x;
                if (v) dv[off + n] = o * gbar[(size_t)i * m_h + n];
            }
            delta[i] = dl;
        }
        /* every pair j <= i */
        for (int j = 0; j < T; ++j) {
            widen_row(gj, g, gdt, (row0 + j) * (size_t)m + (size_t)a * m_h, m_h);
            double *dgj = dg + (row0 + j) * (size_t)m + (size_t)a * m_h;
            for (int i = j; i < T; ++i) {
                double w = PAIR_W(i, j);
                const double *dgi = dgb + (size_t)i * m_h;
                double alpha = w / den[i];
                for (int n = 0; n < m_h; ++n) dgj[n] += alpha * dgi[n];
                double dw = (dot(gj, dgi, m_h) - delta[i]) / den[i];
                const double *qi = qn + (row0 + i) * dqk + (size_t)a * d_h;
                const double *kj = kn + (row0 + j) * dqk + (size_t)a * d_h;
                double *dqi = dqh + (size_t)i * d_h, *dkj = dkh + (size_t)j * d_h;
                if (mode == 0 || j >= i - W + 1) {
                    for (int c = 0; c < d_h; ++c) {
                        dqi[c] += tau[a] * w * dw * kj[c];
                        dkj[c] += tau[a] * w * dw * qi[c];
                    }
                } else {
                    const double *fqi = fq + (row0 + i) * dqk + (size_t)a * d_h;
                    const double *fkj = fk + (row0 + j) * dqk + (size_t)a * d_h;
                    for (int c = 0; c < d_h; ++c) {
                        dqi[c] += st * dw * phi_deriv(st * qi[c], d_h, phi_mode) * fkj[c];
                        dkj[c] += st * dw * fqi[c] * phi_deriv(st * kj[c], d_h, phi_mode);
                    }
                }
            }
        }
#undef PAIR_W
        /* through the unit normalisation */
        for (int i = 0; i < T; ++i) {
            for (int side = 0; side < 2; ++side) {
                const void *raw = side ? k : q;
                int rdt = side ? kdt : qdt;
                const double *unit = (side ? kn : qn) + (row0 + i) * dqk + (size_t)a * d_h;
                const double *dh = (side ? dkh : dqh) + (size_t)i * d_h;
                double *dst = (side ? dk : dq) + (row0 + i) * dqk + (size_t)a * d_h;
                if (qk_normalized) {
                    for (int c = 0; c < d_h; ++c) dst[c] = dh[c];
                    continue;
                }
                double nrm = 0.0;
                for (int c = 0; c < d_h; ++c) {
                    double x = ld(raw, rdt, (row0 + i) * dqk + (size_t)a * d_h + c);
                    nrm += x * x;
                }
                nrm = sqrt(nrm);
                if (nrm < 1e-12) {
                    for (int c = 0; c < d_h; ++c) dst[c] = dh[c] / 1e-12;
                } else {
                    double pr = dot(unit, dh, d_h);
                    for (int c = 0; c < d_h; ++c) dst[c] = (dh[c] - unit[c] * pr) / nrm;
                }
            }
        }
        free(gbar); free(dgb); free(den); free(delta); free(gj); free(dqh); free(dkh);
    }
    free(qn); free(kn); free(fq); free(fk);
    return fail ? OR_ENOMEM : OR_OK;
}

/* Gradients of TANGO (eqs. 5-6); see agg_backward. */
int oracle_tango_backward(int B, int T, int H, int dqk, int m,
                          const void *q, int qdt, const void *k, int kdt,
                          const void *g, int gdt, const void *v, int vdt, const void *dout, int odt,
                          const double *tau, const double *null_b, int qk_normalized,
                          double *dq, double *dk, double *dg, double *dv) {
    return agg_backward(0, B, T, H, dqk, m, 1, 0, q, qdt, k, kdt, g, gdt, v, vdt, dout, odt,
                        tau, null_b, qk_normalized, dq, dk, dg, dv);
}

/* Gradients of WANGO (eqs. 5-9), pair by pair; see agg_backward. */
int oracle_wango_backward(int B, int T, int H, int dqk, int m, int W, int phi_mode,
                          const void *q, int qdt, const void *k, int kdt,
                          const void *g, int gdt, const void *v, int vdt, const void *dout, int odt,
                          const double *tau, const double *null_b, int qk_normalized,
                          double *dq, double *dk, double *dg, double *dv) {
    return agg_backward(1, B, T, H, dqk, m, W, phi_mode, q, qdt, k, kdt, g, gdt, v, vdt, dout, odt,
                        tau, null_b, qk_normalized, dq, dk, dg, dv);
}

/*
 * The gradients of agg_backward for selected rows only, so that long sequences can be
 * checked without the full O(T^2 m) evaluation: dq and dv of the destination rows
 * rows_q[0..nq) and dk and dg of the source rows rows_k[0..nk) (a row is b*T + t).
 * The per-pair terms are those of agg_backward.  Per (batch, head) with a selected row it
 * takes every row's denominator (O(T^2 d_h)), gbar_i and delta_i = gbar_i . dgbar_i for
 * the destinations that the selected rows need (each selected destination; every
 * destination at or after a selected source, for dk), and dgbar_i = dout_i * v_i.
 * dk of an early source therefore costs about as much as the full backward.
 * Outputs (fp64): dq [nq, dqk], dv [nq, m] (untouched when v == NULL), dk [nk, dqk],
 * dg [nk, m].
 */
int oracle_agg_backward_rows(int mode, int B, int T, int H, int dqk, int m, int W, int phi_mode,
                             const void *q, int qdt, const void *k, int kdt,
                             const void *g, int gdt, const void *v, int vdt, const void *dout, int odt,
                             const double *tau, const double *null_b, int qk_normalized,
                             const long long *rows_q, int nq, const long long *rows_k, int nk,
                             double *dq, double *dv, double *dk, double *dg) {
    if (!check_dims(B, T, H, dqk, m) || (mode == 1 && W < 1) || nq < 0 || nk < 0) return OR_EINVAL;
    if (dqk / H > 128) return OR_EINVAL;
    for (int r = 0; r < nq; ++r) if (rows_q[r] < 0 || rows_q[r] >= (long long)B * T) return OR_EINVAL;
    for (int r = 0; r < nk; ++r) if (rows_k[r] < 0 || rows_k[r] >= (long long)B * T) return OR_EINVAL;
    int d_h = dqk / H, m_h = m / H;
    long long BT = (long long)B * T;
    double *qn = prep_unit(q, qdt, BT, H, dqk, qk_normalized);
    double *kn = prep_unit(k, kdt, BT, H, dqk, qk_normalized);
    double *fq = NULL, *fk = NULL;
    if (mode == 1 && qn && kn) {
        fq = prep_phi(qn, BT, H, dqk, tau, phi_mode);
        fk = prep_phi(kn, BT, H, dqk, tau, phi_mode);
    }
    if (!qn || !kn || (mode == 1 && (!fq || !fk))) {
        free(qn); free(kn); free(fq); free(fk);
        return OR_ENOMEM;
    }
    memset(dq, 0, sizeof(double) * (size_t)nq * dqk);
    memset(dk, 0, sizeof(double) * (size_t)nk * dqk);
    memset(dg, 0, sizeof(double) * (size_t)nk * m);
    int fail = 0;
    for (long long u = 0; u < (long long)B * H && !fail; ++u) {
        int b = (int)(u / H), a = (int)(u % H);
        size_t row0 = (size_t)b * T;
        /* which destinations need gbar and delta */
        int any = 0, jmin_k = T;
        for (int r = 0; r < nq; ++r) if (rows_q[r] / T == b) any = 1;
        for (int r = 0; r < nk; ++r)
            if (rows_k[r] / T == b) { any = 1; if ((int)(rows_k[r] % T) < jmin_k) jmin_k = (int)(rows_k[r] % T); }
        if (!any) continue;
        char *need = (char *)calloc((size_t)T, 1);
        double *den = (double *)malloc(sizeof(double) * (size_t)T);
        double *delta = (double *)calloc((size_t)T, sizeof(double));
        double **gbar = (double **)calloc((size_t)T, sizeof(double *));
        if (!need || !den || !delta || !gbar) { fail = 1; free(need); free(den); free(delta); free(gbar); break; }
        for (int r = 0; r < nq; ++r) if (rows_q[r] / T == b) need[rows_q[r] % T] = 1;
        for (int i = jmin_k; i < T; ++i) need[i] = 1;
        const double st = sqrt(tau[a]);
#define PW(i, j) ((mode == 0 || (j) >= (i) - W + 1)                                             \
        ? exp(tau[a] * dot(qn + (row0 + (i)) * dqk + (size_t)a * d_h,                            \
                           kn + (row0 + (j)) * dqk + (size_t)a * d_h, d_h))                      \
        : dot(fq + (row0 + (i)) * dqk + (size_t)a * d_h, fk + (row0 + (j)) * dqk + (size_t)a * d_h, d_h))
        /* every row's denominator */
#pragma omp parallel for schedule(dynamic, 16)
        for (int i = 0; i < T; ++i) {
            double s = 0.0;
            for (int j = 0; j <= i; ++j) s += PW(i, j);
            if (null_b) s += (double)(i + 1) * exp(null_b[a]);
            den[i] = s;
        }
        /* gbar_i and delta_i where needed */
        int nofail = 1;
#pragma omp parallel for schedule(dynamic, 1)
        for (int i = 0; i < T; ++i) {
            if (!need[i]) continue;
            double *gb = (double *)calloc((size_t)m_h, sizeof(double));
            if (!gb) { nofail = 0; continue; }
            for (int j = 0; j <= i; ++j)
                axpy_from(gb, PW(i, j) / den[i], g, gdt, (row0 + j) * (size_t)m + (size_t)a * m_h, m_h);
            size_t off = (row0 + i) * (size_t)m + (size_t)a * m_h;
            double dl = 0.0;
            for (int n = 0; n < m_h; ++n) {
                double o = ld(dout, odt, off + n);
                dl += gb[n] * (v ? o * ld(v, vdt, off + n) : o);
            }
            delta[i] = dl;
            gbar[i] = gb;
        }
        if (!nofail) fail = 1;
        /* destinations: dq (through the normalisation) and dv */
#pragma omp parallel for schedule(dynamic, 1)
        for (int r = 0; r < nq; ++r) {
            if (rows_q[r] / T != b || fail) continue;
            int i = (int)(rows_q[r] % T);
            size_t offi = (row0 + i) * (size_t)m + (size_t)a * m_h;
            double *dgi = (double *)malloc(sizeof(double) * (size_t)m_h);
            double *gj = (double *)malloc(sizeof(double) * (size_t)m_h);
            double dh[128];
            if (!dgi || !gj) { free(dgi); free(gj); continue; }
            for (int n = 0; n < m_h; ++n) {
                double o = ld(dout, odt, offi + n);
                dgi[n] = v ? o * ld(v, vdt, offi + n) : o;
                if (v && dv) dv[(size_t)r * m + (size_t)a * m_h + n] = o * gbar[i][n];
            }
            for (int c = 0; c < d_h; ++c) dh[c] = 0.0;
            const double *qi = qn + (row0 + i) * dqk + (size_t)a * d_h;
            for (int j = 0; j <= i; ++j) {
                widen_row(gj, g, gdt, (row0 + j) * (size_t)m + (size_t)a * m_h, m_h);
                double w = PW(i, j);
                double dw = (dot(gj, dgi, m_h) - delta[i]) / den[i];
                const double *kj = kn + (row0 + j) * dqk + (size_t)a * d_h;
                if (mode == 0 || j >= i - W + 1) {
                    for (int c = 0; c < d_h; ++c) dh[c] += tau[a] * w * dw * kj[c];
                } else {
                    const double *fkj = fk + (row0 + j) * dqk + (size_t)a * d_h;
                    for (int c = 0; c < d_h; ++c) dh[c] += st * dw * phi_deriv(st * qi[c], d_h, phi_mode) * fkj[c];
                }
            }
            double *dst = dq + (size_t)r * dqk + (size_t)a * d_h;
            if (qk_normalized) {
                for (int c = 0; c < d_h; ++c) dst[c] = dh[c];
            } else {
                double nrm = 0.0;
                for (int c = 0; c < d_h; ++c) {
                    double x = ld(q, qdt, (row0 + i) * dqk + (size_t)a * d_h + c);
                    nrm += x * x;
                }
                nrm = sqrt(nrm);
                double pr = dot(qi, dh, d_h);
                for (int c = 0; c < d_h; ++c) dst[c] = nrm < 1e-12 ? dh[c] / 1e-12 : (dh[c] - qi[c] * pr) / nrm;
            }
            free(dgi); free(gj);
        }
        /* sources: dg and dk (through the normalisation) */
#pragma omp parallel for schedule(dynamic, 1)
        for (int r = 0; r < nk; ++r) {
            if (rows_k[r] / T != b || fail) continue;
            int j = (int)(rows_k[r] % T);
            double *gj = (double *)malloc(sizeof(double) * (size_t)m_h);
            double *dgi = (double *)malloc(sizeof(double) * (size_t)m_h);
            double dh[128];
            if (!gj || !dgi) { free(gj); free(dgi); continue; }
            widen_row(gj, g, gdt, (row0 + j) * (size_t)m + (size_t)a * m_h, m_h);
            double *dgj = dg + (size_t)r * m + (size_t)a * m_h;
            for (int c = 0; c < d_h; ++c) dh[c] = 0.0;
            const double *kj = kn + (row0 + j) * dqk + (size_t)a * d_h;
            for (int i = j; i < T; ++i) {
                size_t offi = (row0 + i) * (size_t)m + (size_t)a * m_h;
                for (int n = 0; n < m_h; ++n) {
                    double o = ld(dout, odt, offi + n);
                    dgi[n] = v ? o * ld(v, vdt, offi + n) : o;
                }
                double w = PW(i, j);
                for (int n = 0; n < m_h; ++n) dgj[n] += w / den[i] * dgi[n];
                double dw = (dot(gj, dgi, m_h) - delta[i]) / den[i];
                const double *qi = qn + (row0 + i) * dqk + (size_t)a * d_h;
                if (mode == 0 || j >= i - W + 1) {
                    for (int c = 0; c < d_h; ++c) dh[c] += tau[a] * w * dw * qi[c];
                } else {
                    const double *fqi = fq + (row0 + i) * dqk + (size_t)a * d_h;
                    for (int c = 0; c < d_h; ++c) dh[c] += st * dw * fqi[c] * phi_deriv(st * kj[c], d_h, phi_mode);
                }
            }
            double *dst = dk + (size_t)r * dqk + (size_t)a * d_h;
            if (qk_normalized) {
                for (int c = 0; c < d_h; ++c) dst[c] = dh[c];
            } else {
                double nrm = 0.0;
                for (int c = 0; c < d_h; ++c) {
                    double x = ld(k, kdt, (row0 + j) * dqk + (size_t)a * d_h + c);
                    nrm += x * x;
                }
                nrm = sqrt(nrm);
                double pr = dot(kj, dh, d_h);
                for (int c = 0; c < d_h; ++c) dst[c] = nrm < 1e-12 ? dh[c] / 1e-12 : (dh[c] - kj[c] * pr) / nrm;
            }
            free(gj); free(dgi);
        }
#undef PW
        for (int i = 0; i < T; ++i) free(gbar[i]);
        free(need); free(den); free(delta); free(gbar);
    }
    free(qn); free(kn); free(fq); free(fk);
    return fail ? OR_ENOMEM : OR_OK;
}

/* Number of OpenMP threads the oracle runs on. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
