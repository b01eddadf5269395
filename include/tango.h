/*
 * tango.h -- C ABI of the GB300 (sm_103a) cross-token gate aggregation library.
 *
 * Operations defined by "TANGO: Token-Aggregated Nonlinear Gating Operators for
 * Natural and Formal Language Modeling" (arXiv 2608.22117):
 *   - tango_aggregate      sec. 2.1 eq. 5 with the full-prefix weights of sec. 2.2 eq. 6
 *   - wango_aggregate      sec. 2.1 eq. 5 with the windowed weights of sec. 2.2 eqs. 7-10
 *   - tango_block_forward  one block application, sec. 2.1 eqs. 2-3 around either of the above
 *   - wango_decode_step    one autoregressive token of the windowed aggregation (eqs. 7-10)
 *                          from a constant-size state
 *   - tango_model_forward  the language model of sec. 2.3: token embedding, the shared block
 *                          applied n times (eq. 11), final RMSNorm and tied logits; with
 *                          one weight set, or with the revision's gated-projection sets
 *   - tango_aggregate_backward, wango_aggregate_backward
 *                          gradients of the two aggregations (eq. 5 differentiated with
 *                          respect to q, k, g and v), for training (sec. 3); the
 *                          tango_aggregate_save / wango_aggregate_save forwards keep what
 *                          they need
 *
 * Conventions shared by every call:
 *   - Every pointer argument named as "device" is a CUDA device pointer owned by the
 *     caller.  The library never allocates, frees or synchronises; scratch memory is
 *     passed in as a workspace whose size tg_workspace_size() reports.
 *   - Tensors are row-major and contiguous.  q, k: [B, T, d_qk]; g, v, out: [B, T, m];
 *     h: [B, T, d]; weights are [out_features, in_features].  Head a owns columns
 *     [a*d_qk/H, (a+1)*d_qk/H) of q/k and [a*m/H, (a+1)*m/H) of g/v/out.
 *   - All tensors of one call share one storage type (tg_dtype).  Accumulation is
 *     always fp32.  TG_BF16 runs on the tensor cores (tcgen05); TG_F32 runs on the
 *     CUDA cores in full fp32 (no TF32).
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns an error status and launches nothing.  A failed launch
 *     returns TG_ERR_CUDA.  Errors found on the device (a bounded wait that ran out,
 *     a temperature outside [0, 20]) are recorded in a per-device error word that
 *     tg_check_device_error() reads and clears.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Calls are thread-safe with respect to each other; concurrent calls that share
 *     a workspace race.
 *   - The library runs in each device's primary context (the CUDA runtime's); the
 *     device address of the error word is looked up once per device and kept, so
 *     cudaDeviceReset, or a non-primary context made current through the driver API,
 *     is not supported.
 */
#ifndef TANGO_GB300_H
#define TANGO_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tg_stream_t; /* identical to cudaStream_t */

typedef enum {
    TG_OK = 0,
    TG_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, inconsistent shape */
    TG_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. bf16 head width not in {16,32,64}) */
    TG_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or smaller than required */
    TG_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
    TG_ERR_TIMEOUT = 5,     /* (device) a bounded wait inside a kernel ran out */
    TG_ERR_DEVICE = 6       /* (device) an out-of-range value was seen in device memory */
} tg_status;

typedef enum { TG_F32 = 0, TG_BF16 = 1 } tg_dtype;

/* tg_agg_params.flags */
#define TG_FLAG_QK_NORMALIZED 0x1u  /* q and k are already unit vectors per head */
#define TG_FLAG_DEBUG_TIMEOUT 0x100u /* test hook: a bf16 kernel waits on a barrier that is
                                        never signalled, with a ~1 ms limit, and returns
                                        TG_ERR_TIMEOUT through tg_check_device_error().
                                        tango_aggregate: the TANGO kernel; wango_aggregate:
                                        the gate-strip kernel; tango_block_forward: the
                                        projection GEMM; tango/wango_aggregate_backward:
                                        the pair-gradient, dq/dk and running-sum scan
                                        kernels (the outputs are then undefined) */
#define TG_FLAG_FUSED_V 0x200u       /* tango_block_forward, WANGO mode, bf16: v = W_v x is
                                        formed inside the aggregation kernel instead of by
                                        the projection GEMM (v is then never stored); see
                                        tango_block_forward */
#define TG_FLAG_BWD_FAR_SCAN 0x400u  /* wango_aggregate_backward: the older pairs beyond the
                                        window's band of 128-row blocks always go through
                                        running-sum scans (linear in T) */
#define TG_FLAG_BWD_FAR_PAIRS 0x800u /* wango_aggregate_backward: every older pair is formed
                                        pair by pair (T^2 m).  With neither flag the call
                                        picks by an estimate of the two costs (scans from
                                        about T = 4,096 at B = 8, m = 28,480); both flags:
                                        TG_ERR_INVALID_ARG */

/* tango_block_forward mode */
#define TG_MODE_TANGO 0
#define TG_MODE_WANGO 1

/* tg_workspace_size() selector */
#define TG_WS_TANGO 0 /* params: const tg_agg_params*   */
#define TG_WS_WANGO 1 /* params: const tg_agg_params*   */
#define TG_WS_BLOCK 2 /* params: const tg_block_params* */
#define TG_WS_MODEL 3 /* params: const tg_model_params* */
#define TG_WS_DECODE 4 /* params: const tg_agg_params*: bytes of the wango_decode_step state */
#define TG_WS_TANGO_BWD 5 /* params: const tg_agg_params*: tango_aggregate_backward */
#define TG_WS_WANGO_BWD 6 /* params: const tg_agg_params*: wango_aggregate_backward */

#define TG_MAX_HEADS 64

/*
 * Parameters of one aggregation (eq. 5).
 *   B, T       batch and sequence length (>= 1)
 *   H          heads (1..TG_MAX_HEADS); d_qk % H == 0 and m % H == 0
 *   d_qk       total query/key width (d_h = d_qk / H per head)
 *   m          total gate width F (m_h = m / H per head)
 *   s          temperature tau used for every head when tau == NULL; 0 <= s <= 20
 *              (eq. 4 caps tau at 20)
 *   tau        device float[H] of per-head temperatures, or NULL.  Values outside
 *              [0, 20] are clamped and flagged as TG_ERR_DEVICE.
 *   null_bias  device float[H] of null-gate biases b_a, or NULL for no null gate
 *              (eq. 5: weight n_i exp(b_a), n_i = i + 1, in the denominator only)
 *   window     WANGO window W >= 1, counting the destination itself (eq. 7);
 *              ignored by tango_aggregate
 *   phi_mode   WANGO feature map: 0 = eq. 8 (max(ELU(u)+1+1e-4, 1e-4)/sqrt(d_h)),
 *              1 = plain ELU(u) + 1
 *   flags      TG_FLAG_*
 *   dtype      storage type of q, k, g, v, out
 *   m_pitch    gate columns per head in memory: 0 means m_h = m / H (dense).  Otherwise
 *              >= m_h, and the gate-indexed tensors (g, v, out, and the backward's dout,
 *              dg, dv) are [B, T, H * m_pitch] with head a's m_h gates in columns
 *              [a*m_pitch, a*m_pitch + m_h); the other columns are not read, and in
 *              the outputs their contents are unspecified.  This lets a head width that is not a multiple of 8 (e.g. the
 *              revision's three-set width m = 9,494, m_h = 4,747) run in bf16 at a padded
 *              pitch.  wango_decode_step takes dense tensors only (0 or m_h), and a
 *              block's agg.m_pitch must be 0 (the block pads its own gates).
 * bf16 requirements: d_h in {16, 32, 64}, the per-head pitch (m_pitch, else m_h) a
 * multiple of 8, all tensor base addresses 16-byte aligned (else TG_ERR_UNSUPPORTED).
 */
typedef struct {
    int B, T, H, d_qk, m;
    float s;
    const float *tau;
    const float *null_bias;
    int window;
    int phi_mode;
    unsigned flags;
    tg_dtype dtype;
    int m_pitch;
} tg_agg_params;

/*
 * Full-prefix aggregation (sec. 2.2 eq. 6 in sec. 2.1 eq. 5):
 *   out[b,i,a-cols] = gbar_ia * v[b,i,a-cols],
 *   gbar_ia = sum_{j<=i} e^{l_ija} g_ja / (sum_{j<=i} e^{l_ija} + (i+1) e^{b_a}),
 *   l_ija = tau_a qhat_ia . khat_ja (unit-normalised unless TG_FLAG_QK_NORMALIZED).
 * q, k, g: device, read only.  v: device, or NULL (then out = gbar).  out: device,
 * written; may alias v, must not overlap q, k or g.  ws: device scratch of at least
 * tg_workspace_size(TG_WS_TANGO, p) bytes (256-byte aligned; may be NULL if 0).
 */
tg_status tango_aggregate(const tg_agg_params *p, const void *q, const void *k, const void *g,
                          const void *v, void *out, void *ws, size_t ws_bytes,
                          tg_stream_t stream);

/*
 * Windowed aggregation (sec. 2.2 eqs. 7-10): sources i-W < j <= i get e^{l_ija};
 * older sources j <= i-W get phi(sqrt(tau_a) qhat_ia) . phi(sqrt(tau_a) khat_ja),
 * evaluated through the running sums S = sum phi(k~) g^T, z = sum phi(k~); one joint
 * numerator and denominator (with the null term) per destination.  Arguments as for
 * tango_aggregate; the workspace is sized by tg_workspace_size(TG_WS_WANGO, p).
 */
tg_status wango_aggregate(const tg_agg_params *p, const void *q, const void *k, const void *g,
                          const void *v, void *out, void *ws, size_t ws_bytes,
                          tg_stream_t stream);

/*
 * tango_aggregate / wango_aggregate that also keep what their backward needs, as a
 * training forward does (bf16 only; TG_F32 returns TG_ERR_UNSUPPORTED):
 *   gbar  device, laid out as out: gbar = out / v (the aggregated gate before the
 *         product with v), in the storage type; written
 *   den   device float [B, H, T]: every row's denominator as the kernels form it
 *         (sum of the weights e^{tau (qhat.khat - 1)} as applied, plus the null term,
 *         all shifted by e^-tau); written.  An opaque statistic for the backward.
 * Passing both to the backward skips its recomputation of the forward.  Other arguments
 * as for tango_aggregate / wango_aggregate.
 */
tg_status tango_aggregate_save(const tg_agg_params *p, const void *q, const void *k, const void *g,
                               const void *v, void *out, void *gbar, float *den, void *ws,
                               size_t ws_bytes, tg_stream_t stream);
tg_status wango_aggregate_save(const tg_agg_params *p, const void *q, const void *k, const void *g,
                               const void *v, void *out, void *gbar, float *den, void *ws,
                               size_t ws_bytes, tg_stream_t stream);

/*
 * Backward of tango_aggregate (sec. 2.1 eq. 5 with the weights of sec. 2.2 eq. 6):
 * given dout = dL/d(out) for the output out = gbar * v (out = gbar when v == NULL),
 * writes the gradients of L with respect to the call's inputs:
 *   dv_i = dout_i * gbar_i,   dg_j = sum_{i>=j} alpha_ij (dout_i * v_i),
 *   dq, dk through the weights alpha_ij = w_ij / den_i: with
 *   dL/dw_ij = (dout_i * v_i) . (g_j - gbar_i) / den_i, the score gradient
 *   tau w_ij dL/dw_ij goes to qhat_i (times khat_j) and khat_j (times qhat_i), and from
 *   there through the unit normalisation qhat = q / max(|q|, 1e-12) of sec. 2.1 (with
 *   TG_FLAG_QK_NORMALIZED the gradients are those of the given unit vectors).
 * The null gate, if any, enters through the denominator; tau and null_bias receive no
 * gradient.
 *   p, q, k, g, v   as for the forward call (bf16 only: TG_F32 returns TG_ERR_UNSUPPORTED;
 *                   flags may hold TG_FLAG_QK_NORMALIZED only)
 *   dout            device [B, T, m], read only
 *   gbar, den       the forward's gbar and den from tango_aggregate_save with the same
 *                   arguments, or both NULL: the backward then recomputes them
 *   dq, dk          device [B, T, d_qk], written
 *   dg              device [B, T, m], written
 *   dv              device [B, T, m], written, or NULL (must be NULL when v is NULL)
 *   ws              device scratch of tg_workspace_size(TG_WS_TANGO_BWD, p) bytes,
 *                   256-byte aligned.  It holds the recomputed forward (gbar and the
 *                   denominators), E = dout * v / den, and the pair-weight gradients of
 *                   every causal pair in bf16, B * H * T_pad^2 * 2 bytes with
 *                   T_pad = T rounded up to a multiple of 128.
 * Outputs must not overlap inputs or each other.  Arithmetic: bf16 operands and fp32
 * accumulation on the tensor cores for the two T^2 m contractions; fp32 on the CUDA
 * cores elsewhere.
 */
tg_status tango_aggregate_backward(const tg_agg_params *p, const void *q, const void *k, const void *g,
                                   const void *v, const void *dout, const void *gbar, const float *den,
                                   void *dq, void *dk, void *dg, void *dv, void *ws, size_t ws_bytes,
                                   tg_stream_t stream);

/*
 * Backward of wango_aggregate (sec. 2.2 eqs. 7-10 in sec. 2.1 eq. 5).  Arguments,
 * outputs and requirements as for tango_aggregate_backward; the workspace is sized by
 * tg_workspace_size(TG_WS_WANGO_BWD, p); gbar and den come from wango_aggregate_save.
 * Window pairs contribute as in TANGO; an older
 * pair's weight phi(sqrt(tau) qhat_i) . phi(sqrt(tau) khat_j) passes its gradient
 * through phi' (ELU's derivative, over sqrt(d_h) for eq. 8) and sqrt(tau).  dg is the
 * forward numerator of the time-reversed sequence (linear in T).  The older pairs next
 * to the window (128-row blocks within ceil((W-1)/128) of the destination's) are formed
 * pair by pair; the rest either pair by pair too (T^2 m) or through running sums of
 * phi(k~_j) g_j^T and of phi(q~_i) E_i^T, eq. 10 taken backwards (linear in T): flags may
 * add TG_FLAG_BWD_FAR_SCAN or TG_FLAG_BWD_FAR_PAIRS to force one, else the call picks
 * by a cost estimate that depends on the current device's SM count (query the workspace
 * with the same device current).  The scans add 2 * ceil(m_h / n_s) * B * T * d_qk * 4
 * bytes of workspace (strips of n_s = 256, 384 or 512 gate columns, also picked by the SM
 * count).
 */
tg_status wango_aggregate_backward(const tg_agg_params *p, const void *q, const void *k, const void *g,
                                   const void *v, const void *dout, const void *gbar, const float *den,
                                   void *dq, void *dk, void *dg, void *dv, void *ws, size_t ws_bytes,
                                   tg_stream_t stream);

/*
 * One autoregressive step of the windowed aggregation (sec. 2.2 eqs. 7-10) for B
 * sequences that are all at position pos.  For destination i = pos the output equals row
 * i of wango_aggregate over the sequence so far: window sources i-W < j <= i get
 * e^{l_ij}, older sources enter through the running sums S = sum phi(k~_j) g_j^T and
 * z = sum phi(k~_j) (eq. 10).
 *   p         as for wango_aggregate; T is ignored; flags may hold TG_FLAG_QK_NORMALIZED
 *   q, k      device [B, d_qk]: this token's query and key (unit-normalised per head
 *             unless TG_FLAG_QK_NORMALIZED)
 *   g, v      device [B, m]: this token's gate and feature; v may be NULL (out = gbar)
 *   out       device [B, m], written
 *   state     device buffer of tg_workspace_size(TG_WS_DECODE, p) bytes, 256-byte aligned,
 *             owned by the caller and kept between steps: S and z in f32, a ring of the
 *             last W + 8 tokens' unit k and g (storage type), and per-step scratch.  The
 *             call with pos == 0 clears it; steps must then come in order pos = 0, 1, 2, ...
 * Sources enter S and z in groups of 8: one that has left the window waits in the ring,
 * weighted by e^-tau phi(q~_i) . phi(k~_j) directly, until the step that completes its
 * group adds the group to S and z (the same sums, formed later).
 * Requirements: d_h <= 128, W <= 2^30.  Arithmetic is fp32 for either storage type; the
 * weights are not rounded to bf16.  The step reads the ring (W + 8 g vectors) and S, and
 * rewrites S on one step in 8: it is bound by HBM bandwidth and, for one sequence, by
 * latency.
 */
tg_status wango_decode_step(const tg_agg_params *p, long long pos, const void *q, const void *k,
                            const void *g, const void *v, void *out, void *state,
                            size_t state_bytes, tg_stream_t stream);

/* Weights of one block, all of the block's dtype, row-major [out, in]. */
typedef struct {
    const void *rms_gamma; /* [d]      RMSNorm gain                           */
    const void *Wq;        /* [d_qk, d]                                        */
    const void *Wk;        /* [d_qk, d]                                        */
    const void *Wg;        /* [m, d]   gate projection (SiLU applied, eq. 2)   */
    const void *Wv;        /* [m, d]   feature projection (eq. 2)              */
    const void *Wo;        /* [d, m]   output projection (eq. 3)               */
} tg_block_weights;

/*
 * Block parameters: agg gives B, T, H, d_qk, m, s/tau, null_bias, window, phi_mode,
 * dtype (agg.flags: 0, TG_FLAG_DEBUG_TIMEOUT and/or TG_FLAG_FUSED_V).  d: residual width.  mode: TG_MODE_TANGO or
 * TG_MODE_WANGO.  rms_eps: RMSNorm epsilon (> 0).  rope_base: RoPE base (0 = no
 * RoPE); rotate-half pairing (c, c + d_h/2), positions 0..T-1 per sequence.
 */
typedef struct {
    tg_agg_params agg;
    int d;
    int mode;
    float rms_eps;
    float rope_base;
} tg_block_params;

/*
 * One block application (sec. 2.1 eqs. 2-3):
 *   x = RMSNorm(h); q, k = RoPE(W_q x), RoPE(W_k x), unit-normalised per head;
 *   g = SiLU(W_g x); v = W_v x; gbar by TANGO or WANGO; h_out = h + W_o (gbar * v).
 * h: device [B, T, d], read.  h_out: device [B, T, d], written; may alias h.
 * ws: device scratch of at least tg_workspace_size(TG_WS_BLOCK, p) bytes, 256-byte
 * aligned.  On return it holds, in this order, each region starting on a 256-byte
 * boundary: x [B*T, d], unit q [B*T, d_qk], unit k [B*T, d_qk], g [B*T, m'] and
 * u = gbar * v [B*T, m'] (v is overwritten in place).  With TG_FLAG_FUSED_V (bf16 WANGO
 * mode), v = W_v x is formed tile by tile inside the aggregation kernel (a 128-row x
 * 128-column tile on the tensor cores, rounded to bf16 as a stored v would be) and never
 * written to memory; the region then holds u only.  Both forms give the same v.  The
 * fused form saves the v write and read in HBM (2 m 2 bytes per token) but streams x and
 * a 128-row strip of W_v (256 KB at d = 512) through shared memory for every 128 x 128
 * output tile; on GB300 it is the slower of the two (2.31 against 1.72 ms per WANGO block
 * at B=8, T=2048, d=512, m=28,480), so it is not the default.
 * Gate width: the aggregate calls need m_h % 8 == 0 in bf16; the block does not.  In
 * bf16 it keeps each head's gates at a pitch of m_hp = m_h rounded up to a multiple
 * of 8, m' = H * m_hp: it copies W_g, W_v (rows) and W_o (columns) into the end of ws
 * at that pitch with zeros in the added entries, so g, v and u are zero there and
 * h_out is the unpadded block's.  Otherwise (fp32, or m_h % 8 == 0) m' = m and no copy
 * is made.
 */
tg_status tango_block_forward(const tg_block_params *p, const tg_block_weights *w,
                              const void *h, void *h_out, void *ws, size_t ws_bytes,
                              tg_stream_t stream);

/*
 * A language model built from one shared block (sec. 2.3): token embedding with the
 * tied matrix E, n_apps block applications h^(r+1) = Block(h^(r)) (eq. 11), a final
 * RMSNorm and logits = RMSNorm(h) E^T.  No application embedding is added and the
 * token embeddings are not re-added between applications.
 */
typedef struct {
    const void *embedding;          /* device [vocab, d]: input lookup and output matrix */
    const void *final_gamma;        /* device [d]: gain of the final RMSNorm              */
    const tg_block_weights *sets;   /* HOST array [n_sets] of weight sets (device
                                       pointers); the sets may share rms_gamma, Wq and Wk */
} tg_model_weights;

/*
 * block          every application's parameters (B, T, H, d_qk, m, s/tau, null_bias,
 *                window, phi_mode, dtype, d, mode, rms_eps, rope_base); m is the gate
 *                width of every set
 * vocab          rows of the embedding (>= 1; bf16 needs vocab % 8 == 0)
 * n_apps         block applications (1..64)
 * n_sets         weight sets (1..16)
 * set_of_app     HOST int[n_apps]: the set of each application, or NULL for the
 *                default: set 0 everywhere (n_sets == 1), or set 0 for the first
 *                application, set 2 for the last and set 1 for the others (n_sets ==
 *                3, the revision's first / middle / last assignment); NULL with any
 *                other n_sets is TG_ERR_INVALID_ARG
 * final_rms_eps  epsilon of the final RMSNorm (> 0)
 */
typedef struct {
    tg_block_params block;
    int vocab;
    int n_apps;
    int n_sets;
    const int *set_of_app;
    float final_rms_eps;
} tg_model_params;

/*
 * ids: device int32 [B, T] token ids; an id outside [0, vocab) gives a zero embedding
 * row and TG_ERR_DEVICE (kernel code 4) through tg_check_device_error().  logits:
 * device [B, T, vocab], written.  ws: device scratch of at least
 * tg_workspace_size(TG_WS_MODEL, p) bytes, 256-byte aligned: the residual stream
 * [B*T, d], the final normalised x [B*T, d], then one block's workspace.  Each
 * application is a tango_block_forward call and returns its errors.
 */
tg_status tango_model_forward(const tg_model_params *p, const tg_model_weights *w, const int *ids,
                              void *logits, void *ws, size_t ws_bytes, tg_stream_t stream);

/*
 * tango_aggregate for callers that cannot allocate device memory: runtimes that
 * forbid cudaMalloc once they are running, code confined to a memory pool it does not
 * own, or drivers that must not meet an out-of-memory failure mid-work.  The paper has
 * no counterpart; this is a deployment variant of tango_aggregate with no workspace
 * argument.
 *   - Scratch: one fixed array of TG_NOALLOC_SCRATCH_BYTES in device memory, declared
 *     by the library; every GPU that loads the library holds it until the process
 *     exits.  The call itself allocates nothing (no cudaMalloc, cudaFree or allocating
 *     library routine).
 *   - Limit: the call needs tg_workspace_size(TG_WS_TANGO, p) bytes of that array
 *     (two 256-byte-aligned copies of B*T*d_qk elements; none with
 *     TG_FLAG_QK_NORMALIZED).  Larger problems return TG_ERR_WORKSPACE and launch
 *     nothing; for bf16 that is B*T*d_qk > 4,194,304.
 *   - The first call on each device looks up the array's device address with that
 *     device current (cudaGetSymbolAddress); make that first call before any stream
 *     capture.  The address is kept for the life of the process and belongs to the
 *     device's primary context (the one the CUDA runtime uses): cudaDeviceReset, or a
 *     non-primary context made current through the driver API, is not supported.
 *   - Every call on a device shares the one array and keeps the last call's contents;
 *     each call overwrites the part it reads before reading it, so nothing has to be
 *     cleared between calls.  Calls whose kernels overlap on the GPU (different
 *     streams, or concurrent host threads) race on the array.
 * Other arguments, results and errors are those of tango_aggregate.
 */
#define TG_NOALLOC_SCRATCH_BYTES (16u << 20)
tg_status tango_aggregate_noalloc(const tg_agg_params *p, const void *q, const void *k,
                                  const void *g, const void *v, void *out, tg_stream_t stream);

/* Workspace bytes needed by the call `which` (TG_WS_*) with `params`; 0 for invalid
 * parameters (validate with the call itself to get the reason). */
size_t tg_workspace_size(int which, const void *params);

/* Static, NUL-terminated description of a status. */
const char *tg_status_string(tg_status s);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.
 * Returns TG_OK, TG_ERR_TIMEOUT or TG_ERR_DEVICE (the first kind recorded), or
 * TG_ERR_CUDA if the synchronisation itself failed.  If `detail` is not NULL it
 * receives the raw word (bit 0: timeout, bit 1: value out of range; bits 8..15:
 * the kernel that recorded it, 1 = TANGO, 2 = WANGO, 3 = GEMM, 4 = embedding lookup,
 * 5 = the aggregation backward).
 */
tg_status tg_check_device_error(tg_stream_t stream, unsigned *detail);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int tg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TANGO_GB300_H */
