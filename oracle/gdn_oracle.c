/*
 * gdn_oracle.c - plain fp64 CPU oracle for the packed variable-length
 * gated-delta layer (causal depthwise conv1d -> prepare -> gated delta rule).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: it is used by tests/, by __graft_entry__.smoke() and by
 * the cpu_baseline / reference legs of bench.py.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * Every function restates the method as the source pages define it, in the
 * pages' order, in double precision, with no blocking, fusion or reordering:
 *
 *   [paged_ssm.rs, onnxruntime-ep-mlx 0.31.1, CONV kernel]
 *       varlen causal depthwise conv with per-sequence initial state,
 *       optional bias, optional SiLU, and the emitted final conv state.
 *   [paged_ssm.rs, DELTA_PREPARE kernel]
 *       q/k L2 normalisation x*rsqrt(sum x^2 + 1e-12), decay
 *       g = exp(-exp(A_log) * softplus(a + dt_bias)), rate beta = sigmoid(b).
 *   [gated_delta_rate_activation.rs (mlx-c-rust), decay chain]
 *       softplus as logaddexp(x, 0), A_log taken in float32 before exp.
 *   [paged_ssm.rs, DELTA kernel]
 *       per (sequence, value head, state row): decay the state, retrieve
 *       with the decayed state, beta-scaled delta, rank-1 update, read out
 *       the updated state with q, multiply by scale; key head kh = h/(H/HQ).
 *   [paged_ssm.rs, GatedDeltaNet attributes update_rule, gate_activation,
 *    beta_activation, qk_l2_norm; flags DECAY, RETRIEVE, SOFTPLUS, BETA,
 *    SIGMOID, NORM]  the rule and activation variants (oracle_*_ex).
 *   [rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet]  the dense-layout call,
 *       optional per-key-channel gate (oracle_dense_delta), and the same
 *       per-channel gate on the packed layout (OPT_GATE_PER_CHANNEL).
 *   [paged_ssm.rs, CONV_CAPTURE_* and DELTA_CAPTURE_* kernels]
 *       capture of the first min(counts[b], capacity, len) tokens' updates:
 *       raw conv input rows and the (g, normalised k, beta-scaled delta)
 *       capsule from which S <- g S + delta k^T replays the prefix.
 *
 * Readings where the pages leave a step open are listed at each function.
 * Status codes: 0 ok, 2 bad shape, 4 malformed offsets.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE 2
#define ORACLE_ERR_OFFSETS 4

int oracle_version(void) { return 1; }

/* Round a double to the nearest bfloat16 value, ties to even, returned as a
 * double.  bfloat16 keeps 8 significant bits and float32's exponent range
 * (normal exponents down to 2^-126, subnormal quantum 2^-133, largest finite
 * value (2 - 2^-7) * 2^127).  The rounding mode is round-to-nearest-even
 * [rlx-cpu thunk/types.rs, CastF32ToBf16 note]. */
double oracle_round_bf16(double x) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    int e;
    (void)frexp(x, &e);              /* x = m * 2^e with 0.5 <= |m| < 1 */
    int q = e - 8;                   /* quantum of an 8-significant-bit value */
    if (q < -133) q = -133;          /* subnormal range of the float32 exponent */
    double scaled = ldexp(x, -q);    /* exact: a power-of-two scaling */
    double r = nearbyint(scaled);    /* default rounding mode: ties to even */
    double y = ldexp(r, q);
    const double max_bf16 = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(y) > max_bf16) return x > 0 ? INFINITY : -INFINITY;
    return y;
}

/* Round a double to the nearest float32 value (ties to even). */
static double round_f32(double x) { return (double)(float)x; }

static int check_offsets(const int32_t *offsets, int B, int N) {
    if (offsets[0] != 0 || offsets[B] != N) return ORACLE_ERR_OFFSETS;
    for (int b = 0; b < B; ++b)
        if (offsets[b + 1] < offsets[b]) return ORACLE_ERR_OFFSETS;
    return ORACLE_OK;
}

/*
 * Varlen causal depthwise conv1d  [paged_ssm.rs, CONV kernel].
 *
 *   x     [N, C]      packed inputs (one row per token)
 *   w     [C, Kc]     weight of shape [C, 1, Kc]; tap j multiplies the input
 *                     (Kc-1-j)*D steps back, tap Kc-1 is the current token
 *   bias  [C] or NULL
 *   init  [B, C, L]   initial conv state, L = (Kc-1)*D, index L-1 = newest
 *   y     [N, C]      output;  fin [B, C, L] final conv state
 *   out_round: 0 keep fp64, 1 round outputs to bfloat16, 2 round to float32
 *
 * For token t of sequence b (start s, end e) and channel c:
 *   y[t,c] = act(bias[c] + sum_j w[c,j] * x~(t - s - (Kc-1-j)*D)),
 * with x~(i) = x[s+i, c] for i >= 0 and init[b, c, L+i] for i < 0.
 * act is SiLU z/(1+exp(-z)) when silu != 0.
 * fin[b,c,j] = x~(e - s - L + j): the last L raw inputs of init || sequence.
 */
int oracle_conv1d_varlen(const double *x, const double *w, const double *bias,
                         const int32_t *offsets, const double *init,
                         double *y, double *fin, int B, int N, int C, int Kc,
                         int D, int silu, int out_round) {
    if (B < 1 || N < 0 || C < 1 || Kc < 1 || D < 1) return ORACLE_ERR_SHAPE;
    if (check_offsets(offsets, B, N)) return ORACLE_ERR_OFFSETS;
    const int L = (Kc - 1) * D;
    for (int b = 0; b < B; ++b) {
        const int s = offsets[b], e = offsets[b + 1];
#pragma omp parallel for schedule(static)
        for (int c = 0; c < C; ++c) {
            for (int t = s; t < e; ++t) {
                double sum = bias ? bias[c] : 0.0;
                for (int j = 0; j < Kc; ++j) {
                    int local = t - s - (Kc - 1 - j) * D;
                    double xv = local >= 0
                                    ? x[(size_t)(s + local) * C + c]
                                    : init[((size_t)b * C + c) * L + L + local];
                    sum += xv * w[(size_t)c * Kc + j];
                }
                if (silu) sum = sum / (1.0 + exp(-sum));
                if (out_round == 1) sum = oracle_round_bf16(sum);
                else if (out_round == 2) sum = round_f32(sum);
                y[(size_t)t * C + c] = sum;
            }
            for (int j = 0; j < L; ++j) {
                int local = e - s - L + j;
                fin[((size_t)b * C + c) * L + j] =
                    local >= 0 ? x[(size_t)(s + local) * C + c]
                               : init[((size_t)b * C + c) * L + L + local];
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Prepare  [paged_ssm.rs, DELTA_PREPARE kernel; gated_delta_rate_activation.rs].
 *
 *   y        [N, W]   conv output, W = 2*HQ*K + H*V: q heads in columns
 *                     [0, HQ*K), k heads in [HQ*K, 2*HQ*K), v heads after
 *   a, bl    [N, H]   decay logits and rate logits
 *   A_log, dt_bias [H]
 *   qk       [2, N, HQ, K]   plane 0 = q/|q|, plane 1 = k/|k| (unscaled)
 *   gb       [2, N, H]       plane 0 = g, plane 1 = beta
 *
 * Readings: the epsilon 1e-12 is added to the sum of squares inside the
 * root; softplus(x) = max(x,0) + log(1 + exp(-|x|)) (= logaddexp(x, 0));
 * A_log is rounded to float32 before exp (the rate-activation graph casts it).
 */
/* Rule and activation options (paged_ssm.rs, GatedDeltaNet attributes
 * update_rule, gate_activation, beta_activation, qk_l2_norm and the optional
 * decay / beta inputs); 0 is the default method (gated_delta, softplus gate,
 * sigmoid rate, L2-normalised q and k). */
#define OPT_NO_DECAY 1     /* update_rule linear or delta, or no decay input: g = 1 */
#define OPT_NO_RETRIEVE 2  /* update_rule linear or gated: delta = beta v */
#define OPT_GATE_EXP 4     /* gate_activation none: g = exp(a) */
#define OPT_NO_BETA 8      /* no beta input: beta = 1 */
#define OPT_BETA_RAW 16    /* beta_activation none: beta = b */
#define OPT_NO_QK_NORM 32  /* qk_l2_norm 0: q and k used as they are */
/* Per-key-channel gate [rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet,
 * gate_per_channel], on the packed layout: one decay logit per key channel,
 * a [N, H, K], and g [N, H, K].  The gate activation is the scalar one applied
 * to each channel's logit (A_log and dt_bias stay per head).  Storage of the
 * prepared gates: gb = g [N, H, K] followed by beta [N, H].  In the
 * recurrence, column i of every state row of head h decays by g[t, h, i]. */
#define OPT_GATE_PER_CHANNEL 64

/*
 * [paged_ssm.rs, DELTA_PREPARE with flags NORM, DECAY, SOFTPLUS, BETA, SIGMOID]
 *   q, k scaled by rsqrt(sum^2 + 1e-12) when NORM (else by 1);
 *   g = exp(x) with x = -exp(A_log) softplus(a + dt_bias) under SOFTPLUS, x = a
 *   otherwise, and g = 1 without DECAY; rate = sigmoid(b) under SIGMOID, b
 *   otherwise, and 1 without BETA.
 */
int oracle_prepare_ex(const double *y, const double *a, const double *bl,
                      const double *A_log, const double *dt_bias, double *qk,
                      double *gb, int N, int H, int HQ, int K, int V, int opts) {
    if (N < 0 || H < 1 || HQ < 1 || K < 1 || V < 1 || H % HQ) return ORACLE_ERR_SHAPE;
    const size_t W = (size_t)2 * HQ * K + (size_t)H * V;
    const int norm = !(opts & OPT_NO_QK_NORM), decay = !(opts & OPT_NO_DECAY);
    const int softplus_gate = !(opts & OPT_GATE_EXP), has_beta = !(opts & OPT_NO_BETA);
    const int sigmoid = !(opts & OPT_BETA_RAW);
    const int per_channel = (opts & OPT_GATE_PER_CHANNEL) != 0;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < N; ++t) {
        for (int kh = 0; kh < HQ; ++kh) {
            const double *q = y + (size_t)t * W + (size_t)kh * K;
            const double *k = y + (size_t)t * W + (size_t)HQ * K + (size_t)kh * K;
            double nq = 0.0, nk = 0.0;
            for (int i = 0; i < K; ++i) {
                nq += q[i] * q[i];
                nk += k[i] * k[i];
            }
            double rq = norm ? 1.0 / sqrt(nq + 1e-12) : 1.0;
            double rk = norm ? 1.0 / sqrt(nk + 1e-12) : 1.0;
            for (int i = 0; i < K; ++i) {
                qk[((size_t)t * HQ + kh) * K + i] = q[i] * rq;
                qk[(((size_t)N + t) * HQ + kh) * K + i] = k[i] * rk;
            }
        }
        for (int h = 0; h < H; ++h) {
            const int nch = per_channel ? K : 1;  /* gates of this (token, head) */
            for (int i = 0; i < nch; ++i) {
                double g = 1.0;
                if (decay) {
                    double x = a[((size_t)t * H + h) * nch + i];
                    if (softplus_gate) {
                        x += dt_bias[h];
                        double softplus = fmax(x, 0.0) + log1p(exp(-fabs(x)));
                        double alog = round_f32(A_log[h]);
                        x = -exp(alog) * softplus;
                    }
                    g = exp(x);
                }
                gb[((size_t)t * H + h) * nch + i] = g;
            }
            double beta = has_beta ? bl[(size_t)t * H + h] : 1.0;
            if (has_beta && sigmoid) beta = 1.0 / (1.0 + exp(-beta));
            gb[(size_t)N * H * nch + (size_t)t * H + h] = beta;
        }
    }
    return ORACLE_OK;
}

int oracle_prepare(const double *y, const double *a, const double *bl,
                   const double *A_log, const double *dt_bias, double *qk,
                   double *gb, int N, int H, int HQ, int K, int V) {
    return oracle_prepare_ex(y, a, bl, A_log, dt_bias, qk, gb, N, H, HQ, K, V, 0);
}

/*
 * Gated delta recurrence over packed sequences  [paged_ssm.rs, DELTA kernel].
 *
 *   y      [N, W]          conv output; v of value head h is columns
 *                          2*HQ*K + h*V + [0, V)
 *   qk     [2, N, HQ, K]   normalised q and k (from oracle_prepare)
 *   gb     [2, N, H]       g and beta
 *   init   [B, H, V, K]    initial state (row vi of head h is S[vi, :])
 *   out    [N, H, V]       o_t = scale * S_t q_t
 *   fin    [B, H, V, K]    final state
 *   scale  0 means 1/sqrt(K)
 *
 * For every state row, per token in order:  S *= g;  r = S . k;
 * delta = beta * (v - r);  S += delta * k;  o = scale * (S . q).
 * That is S_t = g_t S_{t-1} + beta_t (v_t - g_t S_{t-1} k_t) k_t^T and
 * o_t = S_t (scale q_t), with value head h reading key head h / (H/HQ).
 */
/* Number of leading tokens of sequence b whose updates are captured:
 * max(0, min(counts[b], cap, len)), or 0 when an active flag is given and is 0
 * (paged_ssm.rs, DELTA_CAPTURE_INIT / CONV_CAPTURE_INIT). */
static int captured_tokens(const int32_t *counts, const int32_t *active, int cap, int b,
                           int len) {
    if (active && active[0] == 0) return 0;
    int n = counts[b];
    if (n > cap) n = cap;
    if (n > len) n = len;
    return n > 0 ? n : 0;
}

/* The recurrence, optionally writing the compact capsule of the first
 * captured tokens (capsule == NULL: no capture). */
static int delta_recurrence(const double *y, const double *qk, const double *gb,
                            const int32_t *offsets, const double *init, double *out,
                            double *fin, int B, int N, int H, int HQ, int K, int V,
                            double scale, const int32_t *counts, const int32_t *active,
                            double *capsule, int cap, int opts) {
    const int retrieve = !(opts & OPT_NO_RETRIEVE);
    const int per_channel = (opts & OPT_GATE_PER_CHANNEL) != 0;
    if (B < 1 || N < 0 || H < 1 || HQ < 1 || K < 1 || V < 1 || H % HQ)
        return ORACLE_ERR_SHAPE;
    if (per_channel && capsule) return ORACLE_ERR_SHAPE;  /* the capsule holds one g per head */
    const size_t nch = per_channel ? (size_t)K : 1;
    if (check_offsets(offsets, B, N)) return ORACLE_ERR_OFFSETS;
    if (scale == 0.0) scale = 1.0 / sqrt((double)K);
    const size_t W = (size_t)2 * HQ * K + (size_t)H * V;
    const int G = H / HQ;
    const size_t width = (size_t)H + (size_t)HQ * K + (size_t)H * V;  /* per captured token */
    if (capsule) memset(capsule, 0, sizeof(double) * (size_t)B * cap * width);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const int kh = h / G;
            const int s = offsets[b], e = offsets[b + 1];
            const int ncap = capsule ? captured_tokens(counts, active, cap, b, e - s) : 0;
            double *cb = capsule ? capsule + (size_t)b * cap * width : NULL;
            double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
            memcpy(S, init + ((size_t)b * H + h) * V * K, sizeof(double) * (size_t)V * K);
            for (int t = s; t < e; ++t) {
                const double *q = qk + ((size_t)t * HQ + kh) * K;
                const double *k = qk + (((size_t)N + t) * HQ + kh) * K;
                const double *gt = gb + ((size_t)t * H + h) * nch;  /* g, or g per key channel */
                const double g = gt[0];
                const double beta = gb[(size_t)N * H * nch + (size_t)t * H + h];
                const int slot = t - s;
                if (slot < ncap) {  /* g of the head; k of the key head (its first value head) */
                    cb[(size_t)slot * H + h] = g;
                    if (h == kh * G)
                        for (int i = 0; i < K; ++i)
                            cb[(size_t)cap * H + ((size_t)slot * HQ + kh) * K + i] = k[i];
                }
                for (int vi = 0; vi < V; ++vi) {
                    double *row = S + (size_t)vi * K;
                    double retrieval = 0.0;
                    for (int i = 0; i < K; ++i) {
                        row[i] *= per_channel ? gt[i] : g;
                        retrieval += k[i] * row[i];
                    }
                    double delta = y[(size_t)t * W + (size_t)2 * HQ * K + (size_t)h * V + vi];
                    if (retrieve) delta -= retrieval;  /* RETRIEVE: delta rules only */
                    delta *= beta;
                    if (slot < ncap)  /* the beta-scaled delta of this state row */
                        cb[(size_t)cap * (H + (size_t)HQ * K) + ((size_t)slot * H + h) * V + vi] = delta;
                    double readout = 0.0;
                    for (int i = 0; i < K; ++i) {
                        row[i] += k[i] * delta;
                        readout += q[i] * row[i];
                    }
                    out[((size_t)t * H + h) * V + vi] = readout * scale;
                }
            }
            memcpy(fin + ((size_t)b * H + h) * V * K, S, sizeof(double) * (size_t)V * K);
            free(S);
        }
    }
    return ORACLE_OK;
}

int oracle_delta_varlen(const double *y, const double *qk, const double *gb,
                        const int32_t *offsets, const double *init, double *out,
                        double *fin, int B, int N, int H, int HQ, int K, int V,
                        double scale) {
    return delta_recurrence(y, qk, gb, offsets, init, out, fin, B, N, H, HQ, K, V, scale,
                            NULL, NULL, NULL, 0, 0);
}

/* The recurrence with rule options (only OPT_NO_RETRIEVE acts here; the
 * decay and rate options act in oracle_prepare_ex). */
int oracle_delta_varlen_ex(const double *y, const double *qk, const double *gb,
                           const int32_t *offsets, const double *init, double *out,
                           double *fin, int B, int N, int H, int HQ, int K, int V,
                           double scale, int opts) {
    return delta_recurrence(y, qk, gb, offsets, init, out, fin, B, N, H, HQ, K, V, scale,
                            NULL, NULL, NULL, 0, opts);
}

/*
 * [paged_ssm.rs, DELTA kernel with DELTA_CAPTURE_INIT / DELTA_CAPTURE_STEP;
 *  GatedDeltaNet handler, state_update_capacity in [0, 8]]
 * The recurrence of oracle_delta_varlen plus the compact transition capsule
 *   capsule [B, cap * (H + HQ*K + H*V)], per sequence b and slot i < captured:
 *     [i*H + h]                              g of token start+i, value head h
 *     [cap*H + (i*HQ + kh)*K + ki]           normalised k of key head kh
 *     [cap*(H + HQ*K) + (i*H + h)*V + vi]    beta-scaled delta of state row vi
 *   and zero in every other slot; captured = max(0, min(counts[b], cap, len)),
 *   or 0 for every sequence when active is given and active[0] == 0.
 * Replaying S <- g S + delta k^T over the captured slots from the initial
 * state gives the state after those tokens.
 */
int oracle_delta_varlen_capture(const double *y, const double *qk, const double *gb,
                                const int32_t *offsets, const double *init, double *out,
                                double *fin, const int32_t *counts, const int32_t *active,
                                double *capsule, int B, int N, int H, int HQ, int K, int V,
                                double scale, int cap) {
    if (cap < 1 || cap > 8 || !counts || !capsule) return ORACLE_ERR_SHAPE;
    return delta_recurrence(y, qk, gb, offsets, init, out, fin, B, N, H, HQ, K, V, scale,
                            counts, active, capsule, cap, 0);
}

/*
 * [paged_ssm.rs, CONV_CAPTURE_INIT / CONV_CAPTURE_STEP]
 *   updates [B, cap, C]: row i < captured of sequence b is the raw input
 *   x[start_b + i, :]; every other row is zero.  captured = max(0,
 *   min(counts[b], cap, len)); the conv operator has no active flag.
 */
int oracle_conv_capture(const double *x, const int32_t *offsets, const int32_t *counts,
                        double *updates, int B, int N, int C, int cap) {
    if (B < 1 || N < 0 || C < 1 || cap < 1 || cap > 8) return ORACLE_ERR_SHAPE;
    if (check_offsets(offsets, B, N)) return ORACLE_ERR_OFFSETS;
    for (int b = 0; b < B; ++b) {
        const int s = offsets[b];
        const int n = captured_tokens(counts, NULL, cap, b, offsets[b + 1] - s);
        for (int i = 0; i < cap; ++i)
            for (int c = 0; c < C; ++c)
                updates[((size_t)b * cap + i) * C + c] = i < n ? x[(size_t)(s + i) * C + c] : 0.0;
    }
    return ORACLE_OK;
}

/*
 * The whole layer: conv -> prepare -> recurrence, composed from the three
 * functions above exactly as the two separate operators of the pages chain
 * (VarlenCausalConvWithState feeds GatedDeltaNet).  When act_dtype is
 * bfloat16 (1) the conv output is rounded to bfloat16 before the later
 * stages, because the conv operator writes its output in the activation
 * dtype and the delta operator reads it back from there; act_dtype 2 rounds
 * to float32, 0 keeps fp64.  Outputs of the recurrence stay in fp64.
 * Readings: scale 0 means 1/sqrt(K); work buffers are owned here.
 */
int oracle_layer_varlen(const double *qkv, const double *w, const double *bias,
                        const double *a, const double *bl, const double *A_log,
                        const double *dt_bias, const int32_t *offsets,
                        const double *conv_init, double *conv_fin,
                        const double *state_init, double *out, double *state_fin,
                        int B, int N, int H, int HQ, int K, int V, int Kc, int D,
                        int silu, double scale, int act_dtype) {
    if (H < 1 || HQ < 1 || K < 1 || V < 1 || H % HQ) return ORACLE_ERR_SHAPE;
    const int C = 2 * HQ * K + H * V;
    double *y = (double *)malloc(sizeof(double) * ((size_t)N * C + 1));
    double *qk = (double *)malloc(sizeof(double) * ((size_t)2 * N * HQ * K + 1));
    double *gb = (double *)malloc(sizeof(double) * ((size_t)2 * N * H + 1));
    int rc = oracle_conv1d_varlen(qkv, w, bias, offsets, conv_init, y, conv_fin, B, N,
                                  C, Kc, D, silu, act_dtype);
    if (!rc) rc = oracle_prepare(y, a, bl, A_log, dt_bias, qk, gb, N, H, HQ, K, V);
    if (!rc) rc = oracle_delta_varlen(y, qk, gb, offsets, state_init, out, state_fin,
                                      B, N, H, HQ, K, V, scale);
    free(y);
    free(qk);
    free(gb);
    return rc;
}

/*
 * The layer with capture: conv capture of the raw qkv rows and the delta
 * capsule (both operators of paged_ssm.rs with state_update_capacity = cap),
 * composed like oracle_layer_varlen.
 */
int oracle_layer_varlen_capture(const double *qkv, const double *w, const double *bias,
                                const double *a, const double *bl, const double *A_log,
                                const double *dt_bias, const int32_t *offsets,
                                const double *conv_init, double *conv_fin,
                                const double *state_init, double *out, double *state_fin,
                                const int32_t *counts, const int32_t *active,
                                double *conv_updates, double *capsule, int B, int N, int H,
                                int HQ, int K, int V, int Kc, int D, int silu, double scale,
                                int act_dtype, int cap) {
    if (H < 1 || HQ < 1 || K < 1 || V < 1 || H % HQ) return ORACLE_ERR_SHAPE;
    const int C = 2 * HQ * K + H * V;
    double *y = (double *)malloc(sizeof(double) * ((size_t)N * C + 1));
    double *qk = (double *)malloc(sizeof(double) * ((size_t)2 * N * HQ * K + 1));
    double *gb = (double *)malloc(sizeof(double) * ((size_t)2 * N * H + 1));
    int rc = oracle_conv1d_varlen(qkv, w, bias, offsets, conv_init, y, conv_fin, B, N,
                                  C, Kc, D, silu, act_dtype);
    if (!rc) rc = oracle_conv_capture(qkv, offsets, counts, conv_updates, B, N, C, cap);
    if (!rc) rc = oracle_prepare(y, a, bl, A_log, dt_bias, qk, gb, N, H, HQ, K, V);
    if (!rc) rc = oracle_delta_varlen_capture(y, qk, gb, offsets, state_init, out, state_fin,
                                              counts, active, capsule, B, N, H, HQ, K, V,
                                              scale, cap);
    free(y);
    free(qk);
    free(gb);
    return rc;
}

/* The layer with rule / activation options (see OPT_*). */
int oracle_layer_varlen_ex(const double *qkv, const double *w, const double *bias,
                           const double *a, const double *bl, const double *A_log,
                           const double *dt_bias, const int32_t *offsets,
                           const double *conv_init, double *conv_fin,
                           const double *state_init, double *out, double *state_fin,
                           int B, int N, int H, int HQ, int K, int V, int Kc, int D,
                           int silu, double scale, int act_dtype, int opts) {
    if (H < 1 || HQ < 1 || K < 1 || V < 1 || H % HQ) return ORACLE_ERR_SHAPE;
    const int C = 2 * HQ * K + H * V;
    const size_t ngate = (opts & OPT_GATE_PER_CHANNEL) ? (size_t)K : 1;
    double *y = (double *)malloc(sizeof(double) * ((size_t)N * C + 1));
    double *qk = (double *)malloc(sizeof(double) * ((size_t)2 * N * HQ * K + 1));
    double *gb = (double *)malloc(sizeof(double) * ((size_t)N * H * (ngate + 1) + 1));
    int rc = oracle_conv1d_varlen(qkv, w, bias, offsets, conv_init, y, conv_fin, B, N,
                                  C, Kc, D, silu, act_dtype);
    if (!rc) rc = oracle_prepare_ex(y, a, bl, A_log, dt_bias, qk, gb, N, H, HQ, K, V, opts);
    if (!rc) rc = oracle_delta_varlen_ex(y, qk, gb, offsets, state_init, out, state_fin,
                                         B, N, H, HQ, K, V, scale, opts);
    free(y);
    free(qk);
    free(gb);
    return rc;
}

/*
 * [rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet (dense layout, gate_per_channel,
 *  carry_state), with the recurrence of the DELTA kernel of paged_ssm.rs]
 *   q, k, v, out [B, S, H, n]; g [B, S, H] or, per channel, [B, S, H, n];
 *   beta [B, S, H]; state [B, H, n, n] (row vi, column key ki).
 * Per (b, h, vi) and token in order: S[vi, :] *= g (per column when per
 * channel); r = S[vi, :] . k; delta = beta (v[vi] - r); S[vi, :] += delta k;
 * out[vi] = scale (S[vi, :] . q).  q, k, g, beta are used as given.  A NULL
 * state_init starts from zero; a NULL state_fin is not written.  The thunk
 * names its math without stating it; this is the DELTA kernel's order.
 */
int oracle_dense_delta(const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const double *state_init, double *out,
                       double *state_fin, int B, int S, int H, int n, int per_channel,
                       double scale) {
    if (B < 1 || S < 0 || H < 1 || n < 1) return ORACLE_ERR_SHAPE;
    if (scale == 0.0) scale = 1.0 / sqrt((double)n);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *St = (double *)malloc(sizeof(double) * (size_t)n * n);
            const size_t head = ((size_t)b * H + h) * n * n;
            for (size_t i = 0; i < (size_t)n * n; ++i) St[i] = state_init ? state_init[head + i] : 0.0;
            for (int t = 0; t < S; ++t) {
                const size_t row = ((size_t)b * S + t) * H + h;
                const double *qt = q + row * n, *kt = k + row * n, *vt = v + row * n;
                for (int vi = 0; vi < n; ++vi) {
                    double *sr = St + (size_t)vi * n;
                    double retrieval = 0.0;
                    for (int i = 0; i < n; ++i) {
                        sr[i] *= per_channel ? g[row * n + i] : g[row];
                        retrieval += kt[i] * sr[i];
                    }
                    const double delta = beta[row] * (vt[vi] - retrieval);
                    double readout = 0.0;
                    for (int i = 0; i < n; ++i) {
                        sr[i] += kt[i] * delta;
                        readout += qt[i] * sr[i];
                    }
                    out[row * n + vi] = readout * scale;
                }
            }
            if (state_fin)
                for (size_t i = 0; i < (size_t)n * n; ++i) state_fin[head + i] = St[i];
            free(St);
        }
    }
    return ORACLE_OK;
}

/* Number of OpenMP threads the oracle's parallel loops use (1 without OpenMP). */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
