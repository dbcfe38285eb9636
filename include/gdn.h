/*
 * gdn.h - C ABI of libgdn.so, a GB300 (sm_103a) implementation of the packed
 * variable-length gated-delta-rule layer:
 *
 *   causal depthwise conv1d (+bias, +SiLU) with per-sequence conv state
 *     -> prepare: L2-normalised q/k, decay g and update rate beta
 *     -> gated delta recurrence with a per-sequence fp32 state.
 *
 * The operations follow the two operators of paged_ssm.rs
 * (onnxruntime-ep-mlx 0.31.1): VarlenCausalConvWithState (CONV kernel and
 * the `conv` handler) and GatedDeltaNet (DELTA_PREPARE and DELTA kernels and
 * the `delta` handler), with the decay formula of
 * gated_delta_rate_activation.rs (mlx-c-rust).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Sizes: B sequences packed into N tokens; offsets[B+1] (int32) delimit
 *   them: sequence b is tokens [offsets[b], offsets[b+1]).  offsets[0] must
 *   be 0, offsets[B] must be N, and offsets must be nondecreasing.  Empty
 *   sequences are allowed (their states pass through unchanged).
 * - Heads: HQ key heads of width K, H value heads of width V, G = H/HQ
 *   (H % HQ == 0); value head h reads key head kh = h / G.
 * - Packed qkv / conv output rows have WIDTH = 2*HQ*K + H*V channels: q heads
 *   in [0, HQ*K), k heads in [HQ*K, 2*HQ*K), v heads in [2*HQ*K, WIDTH).
 * - dtype (gdn_dtype) is the activation type T of qkv, the conv weight, bias,
 *   conv states, conv output and layer output.  Decay/rate logits a, b,
 *   A_log, dt_bias and the recurrent state are always float32.
 * - Every tensor is dense, row-major (last index fastest).  Pointers are
 *   DEVICE pointers unless the name ends in _host.  `stream` is a
 *   cudaStream_t passed as void* (NULL = legacy default stream).
 * - Calls are asynchronous on `stream`; they validate arguments on the host
 *   and return a gdn_status.  On error nothing is launched and
 *   gdn_last_error() returns a message (thread-local, valid until the next
 *   call on the same thread).
 * - The caller owns all memory.  No call allocates device memory; the layer
 *   call takes a caller-provided workspace sized by gdn_workspace_bytes().
 * - In-place carry: a *_fin pointer may equal the matching *_init pointer
 *   (the final state overwrites the initial state).  No other output may
 *   alias any input or another output.
 * - Offsets are also checked on the device: a sequence whose bounds are
 *   malformed is skipped (its outputs are not written) and, for the layer
 *   call, GDN_ERR_OFFSETS is recorded in the workspace status word
 *   (gdn_workspace_status).  Pass offsets_host to the layer call to get the
 *   error synchronously instead.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

/* Symbols of this header are the library's only exported symbols. */
#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,       /* inconsistent or out-of-range geometry */
    GDN_ERR_OVERFLOW = 3,    /* a size or launch grid exceeds its integer range */
    GDN_ERR_OFFSETS = 4,     /* offsets[0] != 0, offsets[B] != N or decreasing */
    GDN_ERR_UNSUPPORTED = 5, /* valid request the library does not implement */
    GDN_ERR_CUDA = 6,        /* a CUDA runtime call failed (message has detail) */
    GDN_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up */
    GDN_ERR_WORKSPACE = 8    /* workspace missing, misaligned or too small */
} gdn_status;

typedef enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Conv activation: "none" or "silu" ("swish" is the same function). */
typedef enum gdn_activation { GDN_ACT_NONE = 0, GDN_ACT_SILU = 1 } gdn_activation;

/* ABI version (GDN_ABI_VERSION of the built library). */
GDN_API int gdn_version(void);

/* Message of the last failing call on this thread ("" if none). */
GDN_API const char *gdn_last_error(void);

/*
 * gdn_conv1d_varlen - varlen causal depthwise conv1d with state
 * [paged_ssm.rs, CONV kernel and `conv` handler].
 *
 *   x         [N, C] T       packed inputs
 *   w         [C, Kc] T      weight of shape [C, 1, Kc]; tap j multiplies the
 *                            input (Kc-1-j)*D tokens back (tap Kc-1 = now)
 *   bias      [C] T or NULL
 *   offsets   [B+1] int32
 *   conv_init [B, C, L] T    L = (Kc-1)*D; index L-1 is the newest token
 *   y         [N, C] T       y[t,c] = act(bias[c] + sum_j w[c,j] x~(t-s-(Kc-1-j)D)),
 *                            x~(i) = x[s+i,c] for i >= 0, conv_init[b,c,L+i] else;
 *                            accumulated in fp32 and rounded to T (nearest even)
 *   conv_fin  [B, C, L] T    last L raw inputs of (conv_init || sequence),
 *                            copied bit-exactly; may equal conv_init
 *   act       gdn_activation
 * Requires B >= 1, N >= 0, C >= 1, 1 <= Kc <= 64, D >= 1, (Kc-1)*D <= 4096.
 * When L == 0, conv_init and conv_fin may be NULL.
 */
GDN_API int gdn_conv1d_varlen(const void *x, const void *w, const void *bias,
                      const int32_t *offsets, const void *conv_init, void *y,
                      void *conv_fin, int B, int N, int C, int Kc, int D, int act,
                      int dtype, void *stream);

/*
 * gdn_prepare - per-token coefficients [paged_ssm.rs, DELTA_PREPARE kernel;
 * gated_delta_rate_activation.rs, decay chain].
 *
 *   y        [N, WIDTH] T   conv output (q and k heads are read)
 *   a, b     [N, H] f32     decay logits and rate logits
 *   A_log    [H] f32, dt_bias [H] f32
 *   qk_norm  [2, N, HQ, K] f32   plane 0: q/sqrt(|q|^2 + 1e-12),
 *                                plane 1: k/sqrt(|k|^2 + 1e-12)
 *   g_beta   [2, N, H] f32       plane 0: g = exp(-exp(A_log) softplus(a + dt_bias)),
 *                                plane 1: beta = sigmoid(b)
 * Requires N >= 0, 1 <= K <= 256, V >= 1, H % HQ == 0.
 */
GDN_API int gdn_prepare(const void *y, const float *a, const float *b, const float *A_log,
                const float *dt_bias, float *qk_norm, float *g_beta, int N, int H,
                int HQ, int K, int V, int dtype, void *stream);

/*
 * gdn_delta_varlen - the gated delta recurrence over packed sequences
 * [paged_ssm.rs, DELTA kernel and `delta` handler].
 *
 *   y          [N, WIDTH] T      v of head h is columns 2*HQ*K + h*V + [0, V)
 *   qk_norm    [2, N, HQ, K] f32 g_beta [2, N, H] f32 (from gdn_prepare)
 *   offsets    [B+1] int32
 *   state_init [B, H, V, K] f32  row vi of head h is S[vi, :]
 *   out        [N, H, V] T       o_t = scale * S_t q_t
 *   state_fin  [B, H, V, K] f32  final state; may equal state_init
 *   scale      0 means 1/sqrt(K)
 * Per token: S_t = g_t S_{t-1} + beta_t (v_t - g_t S_{t-1} k_t) k_t^T.
 * This call always runs the token-serial kernel.
 * Requires 1 <= K <= 256, 1 <= V, H % HQ == 0.
 */
GDN_API int gdn_delta_varlen(const void *y, const float *qk_norm, const float *g_beta,
                     const int32_t *offsets, const float *state_init, void *out,
                     float *state_fin, int B, int N, int H, int HQ, int K, int V,
                     float scale, int dtype, void *stream);

/*
 * gdn_layer_varlen - the whole layer, conv -> prepare -> recurrence, fused
 * where the hardware path allows; results equal the three calls above run
 * in sequence (conv output rounded to T before the later stages).
 *
 *   qkv [N, WIDTH] T; w [WIDTH, Kc] T; bias [WIDTH] T or NULL;
 *   a, b [N, H] f32; A_log, dt_bias [H] f32; offsets [B+1] int32 (device);
 *   offsets_host [B+1] int32 host copy of offsets, or NULL (then the
 *     schedule is built on the device and offsets errors are reported
 *     through gdn_workspace_status);
 *   conv_init / conv_fin [B, WIDTH, L] T; state_init / state_fin [B, H, V, K] f32;
 *   out [N, H, V] T; act, scale as above;
 *   workspace: device buffer of at least gdn_workspace_bytes(...) bytes,
 *     256-byte aligned, not shared with a concurrently running call.
 * Sequences of at least gdn_chunk_min_len() tokens run on the chunkwise
 * tensor-core kernel when the geometry allows it (bf16, K == 128,
 * V % 128 == 0); the rest run on the token-serial kernel.
 */
GDN_API int gdn_layer_varlen(const void *qkv, const void *w, const void *bias, const float *a,
                     const float *b, const float *A_log, const float *dt_bias,
                     const int32_t *offsets, const int32_t *offsets_host,
                     const void *conv_init, void *conv_fin, const float *state_init,
                     void *out, float *state_fin, int B, int N, int H, int HQ, int K,
                     int V, int Kc, int D, int act, float scale, int dtype,
                     void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes gdn_layer_varlen needs for this geometry (0 on bad input). */
GDN_API size_t gdn_workspace_bytes(int B, int N, int H, int HQ, int K, int V, int Kc, int D,
                           int dtype);

/*
 * Synchronises `stream`, then reads the status the last layer call wrote into
 * `workspace`: returns GDN_OK or GDN_ERR_OFFSETS / GDN_ERR_TIMEOUT.  When
 * `counts` is not NULL it receives {sequences on the token-serial kernel,
 * sequences on the chunked kernel, chunked work units}.
 */
GDN_API int gdn_workspace_status(const void *workspace, int *counts, void *stream);

/*
 * Length threshold (tokens) from which a sequence takes the chunked kernel.
 * gdn_set_chunk_min_len(n): n > 0 sets it, n == 0 restores the default
 * (environment variable GDN_CHUNK_MIN_LEN if set, else 8); a very large n
 * keeps every sequence on the token-serial kernel.  Process-wide setting.
 */
GDN_API int gdn_set_chunk_min_len(int n);
GDN_API int gdn_chunk_min_len(void);

/* Number of kernels this library has launched in this process. */
GDN_API uint64_t gdn_launch_count(void);

/*
 * Segment-parallel chunked path (the chunk map is linear in the start state:
 * S_end = S_start M + L).  When a layer call has offsets_host, every chunked
 * sequence has at least gdn_segment_min_len() tokens and there are at most 4
 * of them (and as many as N / gdn_segment_min_len()), sequence i may be cut
 * into P_i <= 8 segments run in parallel: each segment's M and L are computed
 * from a zero start, the start states are chained, and every segment is rerun
 * from its start state.  The counts come from gdn_segment_plan.
 * gdn_set_segment_min_len(n): n > 0 sets the length (default 16384), 0
 * restores the default.  Process-wide.  The workspace holds the segment
 * buffers when N >= that length (gdn_workspace_bytes follows the setting).
 */
GDN_API int gdn_set_segment_min_len(int n);
GDN_API int gdn_segment_min_len(void);

/*
 * The segment counts a layer call with these host offsets would use on a GPU
 * with sm_count SMs (two chunked CTAs per SM), for H value heads of V
 * channels (V a multiple of 128).  Host-only, no GPU needed.
 *   offsets_host  int32 [B+1] host, valid packing (0 = offsets[0] <= ... = N)
 *   counts        int32 [B] host, written: P_i for each chunked sequence of a
 *                 segmented call (1 for one that keeps a single segment), 1 for
 *                 every other sequence
 * Returns the number of chunked sequences the segment-parallel launches run
 * (some may keep P_i = 1; 0: the call runs unsegmented), or a negative
 * GDN_ERR_* code (negated) for NULL pointers, invalid sizes or bad offsets.
 * Capacity: the buffers of one workspace hold min(4, N / gdn_segment_min_len())
 * segmented sequences.
 */
GDN_API int gdn_segment_plan(const int32_t *offsets_host, int B, int H, int V, int sm_count,
                             int32_t *counts);

/* Kernels that gdn_set_kernel_events can bracket. */
typedef enum gdn_kernel_id {
    GDN_KERNEL_CONV = 0,    /* conv (+ fused prepare) pass */
    GDN_KERNEL_CHUNKED = 1, /* chunked tensor-core recurrence */
    GDN_KERNEL_SERIAL = 2   /* token-serial recurrence */
} gdn_kernel_id;

/*
 * Profiling aid: when `start` / `stop` are non-NULL cudaEvent_t handles, every
 * later layer call records `start` on its stream right before launching the
 * given kernel and `stop` right after it, so the caller can time that kernel
 * alone with cudaEventElapsedTime.  Passing NULL for both disables it.  The
 * records sit between dependent launches, so they also serialise the overlap
 * those launches otherwise have.  Process-wide setting; not thread-safe.
 * Returns GDN_ERR_SHAPE for an unknown kernel id.
 */
GDN_API int gdn_set_kernel_events(int kernel, void *start, void *stop);

/*
 * Self-test of the failure path: launches one warp on `stream` that waits, with
 * the same bounded wait as every mbarrier wait of the chunked kernel, for a
 * barrier phase that never completes.  After about limit_us microseconds of
 * GPU global time the wait gives up and the kernel writes GDN_ERR_TIMEOUT to
 * *status (device int32; GDN_OK would mean the wait completed, which cannot
 * happen) and returns; the context stays usable.  Asynchronous: read *status
 * after synchronising the stream.
 *   status    int32 device pointer (written)
 *   limit_us  1 .. 1000000
 * Returns GDN_ERR_NULL / GDN_ERR_SHAPE for bad arguments, GDN_ERR_CUDA if the
 * launch fails, else GDN_OK.
 */
GDN_API int gdn_selftest_wait_timeout(int32_t *status, int limit_us, void *stream);

/* Size of the static device scratch used by gdn_layer_varlen_noalloc. */
#define GDN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * gdn_layer_varlen_noalloc - gdn_layer_varlen for callers that cannot
 * allocate device memory (no counterpart on the source pages; this is an
 * interface convenience, not part of the method).
 *
 * Some callers cannot call cudaMalloc for a workspace: a plain-C host runtime
 * without a device allocator, an inference plugin whose host framework owns
 * all device memory, or a latency-critical loop that cannot accept
 * cudaMalloc's implicit device synchronisation.  This call takes the same
 * inputs and outputs as gdn_layer_varlen (the caller still provides them)
 * but uses a fixed device array of GDN_NOALLOC_SCRATCH_BYTES (16 MiB) inside
 * the library as its workspace; it allocates nothing.
 *
 * - Every GPU that loads the library holds the 16 MiB array until exit.
 * - The first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress (the device must be current); make that first call
 *   before any stream capture.
 * - Geometries whose gdn_workspace_bytes() exceeds the array are rejected
 *   with GDN_ERR_WORKSPACE and a message naming both sizes (for the
 *   HQ=16, H=32, K=V=128 bf16 geometry that is about 500 tokens per call).
 * - All calls share the array and it keeps the last call's contents; the
 *   part that must start cleared is cleared on `stream` before use.  Calls
 *   that overlap on the GPU (for example on two streams) race on the array:
 *   serialise them.
 * - Errors in the offsets are reported only when offsets_host is given
 *   (synchronously, before any launch).  Without it the device-side check
 *   still skips malformed sequences, but its status word sits in the static
 *   array, which gdn_workspace_status() cannot read: pass offsets_host when
 *   the offsets may be malformed.
 * - The device address is cached per device ordinal for the life of the
 *   process.  After cudaDeviceReset() on a device (or with a context other
 *   than the device's primary context current) that cached address is no
 *   longer valid: do not call this entry point on that device afterwards.
 */
GDN_API int gdn_layer_varlen_noalloc(const void *qkv, const void *w, const void *bias,
                                     const float *a, const float *b, const float *A_log,
                                     const float *dt_bias, const int32_t *offsets,
                                     const int32_t *offsets_host, const void *conv_init,
                                     void *conv_fin, const float *state_init, void *out,
                                     float *state_fin, int B, int N, int H, int HQ, int K,
                                     int V, int Kc, int D, int act, float scale, int dtype,
                                     void *stream);

/*
 * Rule and activation options (paged_ssm.rs, GatedDeltaNet attributes
 * update_rule, gate_activation, beta_activation, qk_l2_norm and its optional
 * decay / beta inputs; kernel flags DECAY, RETRIEVE, SOFTPLUS, BETA, SIGMOID,
 * NORM).  A bitmask; 0 is the default method of the plain calls: the
 * gated_delta rule, softplus gate g = exp(-exp(A_log) softplus(a + dt_bias)),
 * sigmoid rate and L2-normalised q and k.
 *   update_rule gated_delta: 0;   delta: GDN_OPT_NO_DECAY;
 *   gated: GDN_OPT_NO_RETRIEVE;   linear: GDN_OPT_NO_DECAY | GDN_OPT_NO_RETRIEVE.
 */
#define GDN_OPT_NO_DECAY 1     /* g = 1 (no decay input; a may be NULL) */
#define GDN_OPT_NO_RETRIEVE 2  /* delta = beta v: no retrieval S k */
#define GDN_OPT_GATE_EXP 4     /* gate_activation none: g = exp(a) (A_log, dt_bias unused) */
#define GDN_OPT_NO_BETA 8      /* no beta input: beta = 1 (b may be NULL) */
#define GDN_OPT_BETA_RAW 16    /* beta_activation none: beta = b */
#define GDN_OPT_NO_QK_NORM 32  /* qk_l2_norm 0: q and k are used as they are */
/*
 * Per-key-channel gate (rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet,
 * gate_per_channel) on the packed layout: every key channel of a (token, value
 * head) has its own decay.  With this bit:
 *   gdn_layer_varlen_ex, gdn_prepare_ex: a is [N, H, K] fp32, one decay logit
 *     per key channel; the gate activation is the scalar one applied to each
 *     logit (softplus gate with the head's A_log and dt_bias, or exp with
 *     GDN_OPT_GATE_EXP).
 *   gdn_prepare_ex writes g_beta as g [N, H, K] followed by beta [N, H]
 *     (N*H*(K+1) floats); gdn_delta_varlen_ex reads that layout.
 *   The recurrence decays column i of every state row of head h by g[t, h, i]:
 *     S_t = S_{t-1} diag(g_t) + beta_t (v_t - S_{t-1} diag(g_t) k_t) k_t^T.
 *   In gdn_layer_varlen_ex, sequences of at least gdn_chunk_min_len() tokens
 *   run on a chunked tensor-core form (16-token chunks: a prepare kernel over
 *   all chunks, then a scan kernel carrying the state) when the geometry
 *   allows it (bf16, K == 128, V % 128 == 0, a, state_init and state_fin
 *   16-byte aligned) and the workspace holds gdn_workspace_bytes_ex(...,
 *   opts) bytes; otherwise, and in gdn_delta_varlen_ex, on the token-serial
 *   kernel.  Not combinable with state-update capture (GDN_ERR_UNSUPPORTED).
 */
#define GDN_OPT_GATE_PER_CHANNEL 64
#define GDN_OPT_ALL 127

/*
 * The calls with rule / activation options (GDN_OPT_*, above); opts = 0 is
 * the plain call.  gdn_layer_varlen_ex also takes the capture arguments
 * documented below (cap = 0: no capture, the capture pointers are ignored).
 * Pointers an option makes unused may be NULL (a with GDN_OPT_NO_DECAY,
 * A_log and dt_bias without the softplus gate, b with GDN_OPT_NO_BETA).
 * Errors: GDN_ERR_UNSUPPORTED for unknown option bits, GDN_ERR_NULL for a
 * pointer the options need, then the plain call's errors.
 */
GDN_API int gdn_prepare_ex(const void *y, const float *a, const float *b, const float *A_log,
                           const float *dt_bias, float *qk_norm, float *g_beta, int N, int H,
                           int HQ, int K, int V, int opts, int dtype, void *stream);

GDN_API int gdn_delta_varlen_ex(const void *y, const float *qk_norm, const float *g_beta,
                                const int32_t *offsets, const float *state_init, void *out,
                                float *state_fin, int B, int N, int H, int HQ, int K, int V,
                                float scale, int opts, int dtype, void *stream);

/*
 * Workspace bytes gdn_layer_varlen_ex needs for this geometry and these
 * options (0 on bad input).  Equal to gdn_workspace_bytes() unless opts has
 * GDN_OPT_GATE_PER_CHANNEL and the geometry has the per-channel chunked form;
 * then it adds the chunk images of that form:
 *   ((N + 15) / 16 + B) * H * 14848 bytes (rounded up to 256).
 * A smaller workspace (at least gdn_workspace_bytes()) is accepted: the
 * per-channel sequences then run on the token-serial kernel.
 */
GDN_API size_t gdn_workspace_bytes_ex(int B, int N, int H, int HQ, int K, int V, int Kc, int D,
                                      int dtype, int opts);

GDN_API int gdn_layer_varlen_ex(const void *qkv, const void *w, const void *bias, const float *a,
                                const float *b, const float *A_log, const float *dt_bias,
                                const int32_t *offsets, const int32_t *offsets_host,
                                const void *conv_init, void *conv_fin, const float *state_init,
                                void *out, float *state_fin, int opts, int cap,
                                const int32_t *counts, const int32_t *active, void *conv_updates,
                                float *capsule, int B, int N, int H, int HQ, int K, int V, int Kc,
                                int D, int act, float scale, int dtype, void *workspace,
                                size_t ws_bytes, void *stream);

/*
 * State-update capture (paged_ssm.rs, onnxruntime-ep-mlx 0.31.1: kernels
 * CONV_CAPTURE_INIT/STEP and DELTA_CAPTURE_INIT/STEP; attribute
 * state_update_capacity in [0, 8], inputs capture_count [B] int32 and the
 * optional state_update_active [1] int32).  A capture call is the plain call
 * plus these arguments:
 *
 *   cap      capacity, 1 .. GDN_CAPTURE_MAX tokens per sequence
 *   counts   device int32 [B]: tokens wanted per sequence; sequence b
 *            captures max(0, min(counts[b], cap, len_b)) tokens
 *   active   device int32 [1] or NULL; active[0] == 0 captures nothing
 *            (the capsule is all zero).  The conv capture has no such flag.
 *   updates / conv_updates
 *            device T [B, cap, C] (C = the conv's channel count, WIDTH for
 *            the layer): row i < captured of sequence b is the RAW input row
 *            x[start_b + i, :] (before the conv); other rows are zero.
 *   capsule  device fp32 [B, cap * (H + HQ*K + H*V)], per sequence:
 *              [i*H + h]                             g of token start_b + i, value head h
 *              [cap*H + (i*HQ + kh)*K + ki]          its normalised key of key head kh
 *              [cap*(H + HQ*K) + (i*H + h)*V + vi]   beta-scaled delta of state row vi
 *            for slots i < captured, zero elsewhere.  From the initial state,
 *            S <- g S + delta k^T over the captured slots gives the state
 *            after those tokens (a caller verifying several draft tokens can
 *            advance the state to any accepted prefix).
 *
 * Buffers are caller-owned and fully written (zeros included); outputs and
 * final states are the same as the plain call's.  The capsule of a sequence
 * taken by the chunked path is computed by a token-serial replay of its
 * captured prefix in fp32.  Errors: GDN_ERR_SHAPE for cap outside [1, 8],
 * GDN_ERR_NULL for a missing counts or capture buffer, GDN_ERR_OVERFLOW for
 * buffers above int32 elements, then the plain call's errors.
 */
#define GDN_CAPTURE_MAX 8

GDN_API int gdn_conv1d_varlen_capture(const void *x, const void *w, const void *bias,
                                      const int32_t *offsets, const void *conv_init, void *y,
                                      void *conv_fin, int cap, const int32_t *counts,
                                      void *updates, int B, int N, int C, int Kc, int D, int act,
                                      int dtype, void *stream);

GDN_API int gdn_delta_varlen_capture(const void *y, const float *qk_norm, const float *g_beta,
                                     const int32_t *offsets, const float *state_init, void *out,
                                     float *state_fin, int cap, const int32_t *counts,
                                     const int32_t *active, float *capsule, int B, int N, int H,
                                     int HQ, int K, int V, float scale, int dtype, void *stream);

/* conv_updates or capsule may be NULL (that capture is skipped), not both. */
GDN_API int gdn_layer_varlen_capture(const void *qkv, const void *w, const void *bias,
                                     const float *a, const float *b, const float *A_log,
                                     const float *dt_bias, const int32_t *offsets,
                                     const int32_t *offsets_host, const void *conv_init,
                                     void *conv_fin, const float *state_init, void *out,
                                     float *state_fin, int cap, const int32_t *counts,
                                     const int32_t *active, void *conv_updates, float *capsule,
                                     int B, int N, int H, int HQ, int K, int V, int Kc, int D,
                                     int act, float scale, int dtype, void *workspace,
                                     size_t ws_bytes, void *stream);

/*
 * gdn_gated_delta_dense - the recurrence on the dense layout of the
 * GatedDeltaNet CPU thunk (rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet:
 * q, k, v [b, s, h, n]; g, beta [b, s, h]; gate_per_channel makes g
 * [b, s, h, n]; state [b, h, n, n] resumed from and written back in place
 * with carry_state).  The thunk defers its math to an operator not on the
 * page; this call applies the DELTA kernel of paged_ssm.rs to the values as
 * given, per (sequence, head, state row vi) and token in order:
 *   S <- S diag(g) (scalar g: S <- g S);  r = S k;  delta = beta (v[vi] - r);
 *   S <- S + delta k^T;  out[vi] = scale (S q)[vi]
 * with no convolution and no normalisation (q, k, g, beta as passed).
 *
 *   q, k, v, out  device T [B, S, H, n]   (n <= 256; v uses n value channels)
 *   g             device fp32 [B, S, H], or [B, S, H, n] when gate_per_channel
 *   beta          device fp32 [B, S, H]
 *   state_init    device fp32 [B, H, n, n] (row vi, column key ki) or NULL for
 *                 a zero initial state (carry_state false)
 *   state_fin     device fp32 [B, H, n, n] or NULL (not written); may alias
 *                 state_init (in-place carry)
 *   scale         0 means 1/sqrt(n)
 * Errors: GDN_ERR_SHAPE, GDN_ERR_OVERFLOW, GDN_ERR_NULL, GDN_ERR_UNSUPPORTED
 * (dtype), GDN_ERR_CUDA.  Sequences run on the token-serial kernel (see
 * gdn_gated_delta_dense_ws for the chunked route).
 */
GDN_API int gdn_gated_delta_dense(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const float *state_init, void *out,
                                  float *state_fin, int B, int S, int H, int n,
                                  int gate_per_channel, float scale, int dtype, void *stream);

/*
 * gdn_gated_delta_dense_ws - gdn_gated_delta_dense with a caller workspace, so
 * that long sequences can take the chunked tensor-core kernel: for bf16, n =
 * 128, a scalar gate, S >= gdn_chunk_min_len() and 16-byte aligned q, k, v and
 * out, a packing kernel writes the rows [q | k | v] of every token and ln g
 * into the workspace and the chunked kernel runs them with the values as
 * given (exp gate of ln g, raw beta, no q/k normalisation).  Gates below
 * 1e-30 are taken as 1e-30 on that route (the chunk keeps decays in the log
 * domain).  Other calls run exactly as gdn_gated_delta_dense and need no
 * workspace.
 *   workspace  device, 256-byte aligned, gdn_dense_workspace_bytes() bytes
 *              (0 from that query: no chunked route for this geometry)
 * With gate_per_channel (g [B, S, H, n] gate factors, 16-byte aligned) the
 * chunked route is the per-key-channel one (16-token chunks: a prepare kernel
 * over all chunks, then a scan kernel carrying the state; the factors are used
 * as they are); it needs gdn_dense_workspace_bytes_ex(..., 1) bytes, and with
 * a smaller workspace the call runs on the token-serial kernel.
 * Errors: as gdn_gated_delta_dense, plus GDN_ERR_WORKSPACE when the chunked
 * route applies and the workspace is missing, misaligned or too small.
 */
GDN_API size_t gdn_dense_workspace_bytes(int B, int S, int H, int n, int dtype);
/* Workspace of gdn_gated_delta_dense_ws for this gate kind (0: no chunked
 * route): gdn_dense_workspace_bytes() plus, with gate_per_channel, the chunk
 * images ((B S + 15) / 16 + B) * H * 14848 bytes (rounded up to 256). */
GDN_API size_t gdn_dense_workspace_bytes_ex(int B, int S, int H, int n, int dtype,
                                            int gate_per_channel);
GDN_API int gdn_gated_delta_dense_ws(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *state_init, void *out,
                                     float *state_fin, int B, int S, int H, int n,
                                     int gate_per_channel, float scale, int dtype,
                                     void *workspace, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
