// api.cpp - the C ABI of libgdn.so (declared in include/gdn.h): argument
// validation, workspace carving, path selection and kernel dispatch.
//
// The checks restate the operator contracts of paged_ssm.rs
// (onnxruntime-ep-mlx 0.31.1): the `conv` / `delta` handlers (shapes,
// receptive-field and dispatch-size overflow, key width <= 256, grouped-head
// divisibility, scale 0 -> 1/sqrt(K)) and the claim predicates (dtype and
// activation rules).  Where the pages' kernels silently skip malformed
// offsets, this library reports GDN_ERR_OFFSETS.
#include "../../include/gdn.h"

#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <mutex>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "internal.h"

namespace gdn {

static std::atomic<uint64_t> g_launches{0};
void note_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static thread_local char g_err[512] = "";
static cudaEvent_t g_ev_start[3] = {nullptr, nullptr, nullptr};
static cudaEvent_t g_ev_stop[3] = {nullptr, nullptr, nullptr};

// External records, so that inside a stream capture they become real event
// record nodes of the graph (and stay ordinary records outside a capture).
// Inside a stream capture the records are external, so that they become
// real event-record nodes of the graph; outside a capture they are plain.
static void record_event(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) st = cudaStreamCaptureStatusNone;
    if (st == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else cudaEventRecord(ev, s);
}
static void mark_before(int k, cudaStream_t s) {
    if (g_ev_start[k]) record_event(g_ev_start[k], s);
}
static void mark_after(int k, cudaStream_t s) {
    if (g_ev_stop[k]) record_event(g_ev_stop[k], s);
}
static std::atomic<int> g_chunk_min_len{0};

static int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

static int cuda_fail(cudaError_t e, const char *what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Sequences of at least this many tokens take the chunked kernel.  Measured
// on GB300 (decode head geometry, bf16): 64 sequences of 4 tokens take 0.100 ms
// token-serially against 0.221 ms chunked, 64 of 16 tokens 0.249 ms against
// 0.231 ms, 256 of 32 tokens 2.01 ms against 0.875 ms, and a batch of 512
// sequences of 1..63 tokens 3.87 ms with a threshold of 64 against 1.63 ms
// with 8: a token-serial CTA walks its tokens one after another, while the
// chunked kernel takes 64 of them per step.
static int default_chunk_min_len() {
    const char *env = getenv("GDN_CHUNK_MIN_LEN");
    if (env && *env) {
        long v = strtol(env, nullptr, 10);
        if (v > 0 && v <= INT_MAX) return (int)v;
    }
    return 8;
}

static int chunk_min_len() {
    int v = g_chunk_min_len.load(std::memory_order_relaxed);
    return v > 0 ? v : default_chunk_min_len();
}

// Length from which long chunked sequences may be cut into segments that run
// in parallel (segment-parallel chunked path); 0 = default.
static std::atomic<int> g_segment_min_len{0};
static int segment_min_len() {
    int v = g_segment_min_len.load(std::memory_order_relaxed);
    return v > 0 ? v : 16384;
}

// SM count of the current device (asked per call: a process may drive
// several devices).
static int sm_count_host() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 1;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Side stream on which the token-serial kernel runs beside the chunked kernel
// of the same layer call, and the two events that fork it from and join it
// to the caller's stream.  One set per device, created by the first call that
// would fork outside a stream capture (captured calls before that run the two
// kernels one after the other); calls from several host threads take turns on
// it under a mutex, so each call's dependencies stay exact (a wait on an event
// takes the record enqueued just before it).
struct ForkSet {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
static std::mutex g_fork_mu;
static ForkSet g_fork[64];

// The set of the current device (g_fork_mu held); created on first use, but
// not while `s` is being captured (then cudaErrorNotReady: no fork).
static cudaError_t fork_set(ForkSet **out, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    ForkSet &f = g_fork[dev];
    if (f.side == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return cudaErrorNotReady;
        e = cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            f = ForkSet{};
            return e;
        }
    }
    *out = &f;
    return cudaSuccess;
}

static bool dtype_ok(int dtype) { return dtype == GDN_F32 || dtype == GDN_BF16; }
static size_t dsize(int dtype) { return dtype == GDN_BF16 ? 2 : 4; }

// Geometry of the recurrence: mirrors the `delta` handler's rules.
static int check_heads(int H, int HQ, int K, int V, long *width) {
    if (H < 1 || HQ < 1 || K < 1 || V < 1)
        return fail(GDN_ERR_SHAPE, "head geometry must be positive (H=%d HQ=%d K=%d V=%d)", H, HQ, K, V);
    if (K > 256) return fail(GDN_ERR_SHAPE, "key width K=%d exceeds 256", K);
    if (H % HQ != 0) return fail(GDN_ERR_SHAPE, "value heads H=%d not a multiple of key heads HQ=%d", H, HQ);
    long w = 2L * HQ * K + (long)H * V;
    if (w > INT_MAX) return fail(GDN_ERR_OVERFLOW, "packed width 2*HQ*K+H*V exceeds int32");
    *width = w;
    return GDN_OK;
}

static int check_offsets_host(const int32_t *offsets_host, int B, int N) {
    if (offsets_host[0] != 0) return fail(GDN_ERR_OFFSETS, "offsets[0]=%d, expected 0", offsets_host[0]);
    if (offsets_host[B] != N) return fail(GDN_ERR_OFFSETS, "offsets[B]=%d, expected N=%d", offsets_host[B], N);
    for (int b = 0; b < B; ++b)
        if (offsets_host[b + 1] < offsets_host[b])
            return fail(GDN_ERR_OFFSETS, "offsets decrease at b=%d (%d > %d)", b, offsets_host[b], offsets_host[b + 1]);
    return GDN_OK;
}

// Segment plan of a call: which chunked sequences are cut into how many
// segments.  n = 0: no segmentation.
struct SegmentPlan {
    int n = 0;
    int seq[kMaxSegSeqs] = {};
    int m0[kMaxSegSeqs + 1] = {};  // prefix sums of P_i - 1
    int s0[kMaxSegSeqs + 1] = {};  // prefix sums of P_i
};

// Chunk threshold under which the segment planner looks at a batch: sequences
// shorter than one chunk do not stop a long sequence from being segmented (they
// then run on the token-serial kernel).
static int segment_plan_thr(int thr) { return thr > 64 ? thr : 64; }

// Length of the segments of len tokens cut into P (a multiple of the chunk).
static long segment_len(long len, long P) { return ((len + P - 1) / P + 63) / 64 * 64; }

// Segmentation applies when every chunked sequence (>= thr tokens) has at
// least gdn_segment_min_len() tokens and there are at most max_seqs of them.
// Counts P_i are raised one at a time on the sequence whose segments are
// longest while both chunked launches still fit in one wave of CTA slots:
// sum P_i (head, V tile) units in the rerun, sum (P_i - 1) (head, V tile +
// transition tile) units in the first pass.  The two passes take about the
// longest phase-1 segment plus the longest segment; the plan with the least
// of that is kept when it is no longer than the longest sequence (what the
// unsegmented chunked launch takes).
static SegmentPlan plan_segments(const int32_t *offsets_host, int B, int H, int V, int thr,
                                 int max_seqs, int sm_count) {
    SegmentPlan best;
    int seq[kMaxSegSeqs];
    long len[kMaxSegSeqs], P[kMaxSegSeqs];
    int n = 0;
    for (int i = 0; i < B; ++i) {
        const long l = offsets_host[i + 1] - offsets_host[i];
        if (l < thr) continue;
        if (l < segment_min_len() || n == max_seqs || n == kMaxSegSeqs) return best;
        seq[n] = i;
        len[n] = l;
        P[n] = 1;
        ++n;
    }
    if (n == 0) return best;
    const long VT = V / 128, slots = 2L * sm_count;
    long plain = 0;
    for (int i = 0; i < n; ++i) plain = len[i] > plain ? len[i] : plain;
    if ((long)n * H * VT > slots) return best;  // the rerun alone would not fit one wave
    long best_cost = plain + 1;
    while (true) {
        int arg = 0;
        for (int i = 1; i < n; ++i)
            if (segment_len(len[i], P[i]) > segment_len(len[arg], P[arg])) arg = i;
        if (P[arg] == kMaxSegments) break;
        long sumP = 0, sumP1 = 0;
        for (int i = 0; i < n; ++i) {
            sumP += P[i] + (i == arg);
            sumP1 += P[i] + (i == arg) - 1;
        }
        if (sumP * H * VT > slots || sumP1 * H * (VT + 1) > slots) break;
        ++P[arg];
        long cost1 = 0, cost2 = 0;
        for (int i = 0; i < n; ++i) {
            const long sl = segment_len(len[i], P[i]);
            if (P[i] > 1 && sl > cost1) cost1 = sl;
            if (sl > cost2) cost2 = sl;
        }
        if (cost1 + cost2 < best_cost) {
            best_cost = cost1 + cost2;
            best.n = n;
            best.m0[0] = best.s0[0] = 0;
            for (int i = 0; i < n; ++i) {
                // the segments segments_of makes: never more than P_i
                const long sl = segment_len(len[i], P[i]);
                const long cnt = (len[i] + sl - 1) / sl;
                best.seq[i] = seq[i];
                best.s0[i + 1] = best.s0[i] + (int)cnt;
                best.m0[i + 1] = best.m0[i] + (int)cnt - 1;
            }
        }
    }
    for (int i = best.n; i < kMaxSegSeqs; ++i) {  // unused entries repeat the totals
        best.s0[i + 1] = best.s0[i];
        best.m0[i + 1] = best.m0[i];
    }
    return best;
}

struct WsLayout {
    size_t header, order, y, qk, gb, seg, total;  // seg: 0 when no segment buffers fit
    int seg_seqs;                                 // sequences the segment buffers hold
};

static WsLayout ws_layout(int B, int N, int H, int HQ, int K, int V, int dtype) {
    WsLayout l;
    const size_t W = 2 * (size_t)HQ * K + (size_t)H * V;
    size_t off = 0;
    l.header = off;
    off += align256(sizeof(WsHeader));
    l.order = off;
    off += align256((size_t)B * 4);
    l.y = off;
    off += align256((size_t)N * W * dsize(dtype));
    l.qk = off;
    off += align256((size_t)2 * N * HQ * K * 4);
    l.gb = off;
    off += align256((size_t)2 * N * H * 4);
    // segment buffers when a sequence can be long enough to be segmented, for
    // as many such sequences as N tokens can hold (at most kMaxSegSeqs)
    l.seg = 0;
    l.seg_seqs = 0;
    if (N >= segment_min_len() && K == 128 && V % 128 == 0) {
        const long n = N / segment_min_len();
        l.seg_seqs = (int)(n < kMaxSegSeqs ? n : kMaxSegSeqs);
        l.seg = off;
        off += align256(segment_floats(H, V, l.seg_seqs) * 4);
    }
    l.total = off;
    return l;
}

}  // namespace gdn

using namespace gdn;

// Optional state-update capture of a call (nullptr: none).
struct Capture {
    int cap;
    const int32_t *counts;
    const int32_t *active;
    void *conv_updates;
    float *capsule;
};

// Pointers the rule options need: the decay logits a unless GDN_OPT_NO_DECAY,
// A_log and dt_bias for the softplus gate, the rate logits b unless
// GDN_OPT_NO_BETA.
static int check_opts(int opts, int N, const float *a, const float *b, const float *A_log,
                      const float *dt_bias, const char *what) {
    if (opts & ~GDN_OPT_ALL) return fail(GDN_ERR_UNSUPPORTED, "%s: unknown option bits 0x%x", what, opts);
    const bool decay = !(opts & GDN_OPT_NO_DECAY);
    if (decay && !(opts & GDN_OPT_GATE_EXP) && (!A_log || !dt_bias))
        return fail(GDN_ERR_NULL, "%s: A_log / dt_bias is NULL (softplus gate)", what);
    if (N > 0 && decay && !a) return fail(GDN_ERR_NULL, "%s: decay logits a is NULL", what);
    if (N > 0 && !(opts & GDN_OPT_NO_BETA) && !b) return fail(GDN_ERR_NULL, "%s: rate logits b is NULL", what);
    return GDN_OK;
}

static int check_capture(const Capture &c, const char *what) {
    if (c.cap < 1 || c.cap > GDN_CAPTURE_MAX)
        return fail(GDN_ERR_SHAPE, "%s: capture capacity %d outside [1, %d]", what, c.cap, GDN_CAPTURE_MAX);
    if (!c.counts) return fail(GDN_ERR_NULL, "%s: capture counts is NULL", what);
    return GDN_OK;
}

extern "C" {

int gdn_version(void) { return GDN_ABI_VERSION; }

const char *gdn_last_error(void) { return g_err; }

uint64_t gdn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int gdn_set_chunk_min_len(int n) {
    if (n < 0) return fail(GDN_ERR_SHAPE, "chunk threshold must be >= 0");
    g_chunk_min_len.store(n, std::memory_order_relaxed);
    return GDN_OK;
}

int gdn_chunk_min_len(void) { return chunk_min_len(); }

int gdn_set_segment_min_len(int n) {
    if (n < 0) return fail(GDN_ERR_SHAPE, "segment length %d < 0", n);
    g_segment_min_len.store(n, std::memory_order_relaxed);
    return GDN_OK;
}

int gdn_segment_min_len(void) { return segment_min_len(); }

int gdn_segment_plan(const int32_t *offsets_host, int B, int H, int V, int sm_count,
                     int32_t *counts) {
    // errors are returned negated: a non-negative result is a count
    if (!offsets_host || !counts) return -set_error(GDN_ERR_NULL, "offsets_host and counts are required");
    if (B < 0 || H <= 0 || V <= 0 || V % 128 != 0 || sm_count <= 0)
        return -set_error(GDN_ERR_SHAPE, "B >= 0, H > 0, V a positive multiple of 128, sm_count > 0");
    const int N = B > 0 ? offsets_host[B] : 0;
    const int rc = check_offsets_host(offsets_host, B, N);
    if (rc) return -rc;
    for (int i = 0; i < B; ++i) counts[i] = 1;
    if (N < segment_min_len()) return 0;
    const long cap = N / segment_min_len();
    const SegmentPlan p = plan_segments(offsets_host, B, H, V, segment_plan_thr(chunk_min_len()),
                                        (int)(cap < kMaxSegSeqs ? cap : kMaxSegSeqs), sm_count);
    for (int i = 0; i < p.n; ++i) counts[p.seq[i]] = p.s0[i + 1] - p.s0[i];
    return p.n;
}

int gdn_set_kernel_events(int kernel, void *start, void *stop) {
    if (kernel < 0 || kernel > 2) return fail(GDN_ERR_SHAPE, "unknown kernel id %d", kernel);
    g_ev_start[kernel] = static_cast<cudaEvent_t>(start);
    g_ev_stop[kernel] = static_cast<cudaEvent_t>(stop);
    return GDN_OK;
}

static int conv_impl(const void *x, const void *w, const void *bias, const int32_t *offsets,
                     const void *conv_init, void *y, void *conv_fin, int B, int N, int C, int Kc,
                     int D, int act, int dtype, void *stream, const Capture *cap) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
    if (act != GDN_ACT_NONE && act != GDN_ACT_SILU) return fail(GDN_ERR_UNSUPPORTED, "activation %d not supported", act);
    if (B < 1 || N < 0 || C < 1 || Kc < 1 || D < 1)
        return fail(GDN_ERR_SHAPE, "need B>=1, N>=0, C>=1, Kc>=1, D>=1 (B=%d N=%d C=%d Kc=%d D=%d)", B, N, C, Kc, D);
    const long L = (long)(Kc - 1) * D;
    if (L >= INT_MAX) return fail(GDN_ERR_OVERFLOW, "receptive field (Kc-1)*D exceeds int32");
    if (!w || !offsets || !y || (N > 0 && !x) || (L > 0 && (!conv_init || !conv_fin)))
        return fail(GDN_ERR_NULL, "conv1d: a required pointer is NULL");
    if ((long)B * C > INT_MAX) return fail(GDN_ERR_OVERFLOW, "conv dispatch B*C exceeds int32");
    if (L > 4096) return fail(GDN_ERR_UNSUPPORTED, "receptive field L=%ld above 4096", L);
    if (Kc > 64) return fail(GDN_ERR_UNSUPPORTED, "conv width Kc=%d above 64", Kc);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ConvParams p{};
    p.x = x; p.w = w; p.bias = bias; p.offsets = offsets; p.init = conv_init; p.y = y;
    p.B = B; p.N = N; p.C = C; p.Kc = Kc; p.D = D; p.L = (int)L; p.silu = act == GDN_ACT_SILU;
    p.prep = 0;
    cudaError_t e = launch_conv(p, dtype, s, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "conv kernel launch");
    e = launch_conv_final(x, offsets, conv_init, conv_fin, B, N, C, (int)L, dtype, s,
                          cap ? cap->cap : 0, cap ? cap->counts : nullptr,
                          cap ? cap->conv_updates : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "conv final-state kernel launch");
    return GDN_OK;
}

int gdn_conv1d_varlen(const void *x, const void *w, const void *bias, const int32_t *offsets,
                      const void *conv_init, void *y, void *conv_fin, int B, int N, int C, int Kc,
                      int D, int act, int dtype, void *stream) {
    g_err[0] = 0;
    return conv_impl(x, w, bias, offsets, conv_init, y, conv_fin, B, N, C, Kc, D, act, dtype,
                     stream, nullptr);
}

int gdn_conv1d_varlen_capture(const void *x, const void *w, const void *bias,
                              const int32_t *offsets, const void *conv_init, void *y,
                              void *conv_fin, int cap, const int32_t *counts, void *updates,
                              int B, int N, int C, int Kc, int D, int act, int dtype,
                              void *stream) {
    g_err[0] = 0;
    const Capture c{cap, counts, nullptr, updates, nullptr};
    int rc = check_capture(c, "conv1d capture");
    if (rc) return rc;
    if (!updates) return fail(GDN_ERR_NULL, "conv1d capture: updates is NULL");
    if ((long)B * cap * C > INT_MAX) return fail(GDN_ERR_OVERFLOW, "conv capture B*cap*C exceeds int32");
    return conv_impl(x, w, bias, offsets, conv_init, y, conv_fin, B, N, C, Kc, D, act, dtype,
                     stream, &c);
}

static int prepare_impl(const void *y, const float *a, const float *b, const float *A_log,
                        const float *dt_bias, float *qk_norm, float *g_beta, int N, int H,
                        int HQ, int K, int V, int opts, int dtype, void *stream) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
    long width;
    int rc = check_heads(H, HQ, K, V, &width);
    if (rc) return rc;
    if (N < 0) return fail(GDN_ERR_SHAPE, "N=%d < 0", N);
    if (N > 0 && (!y || !qk_norm || !g_beta)) return fail(GDN_ERR_NULL, "prepare: a required pointer is NULL");
    rc = check_opts(opts, N, a, b, A_log, dt_bias, "prepare");
    if (rc) return rc;
    if ((opts & GDN_OPT_GATE_PER_CHANNEL) && (long)N * H * (K + 1) > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "prepare: N*H*(K+1) gates exceed int32");
    if ((long)N * H > INT_MAX / 2 || (long)N * HQ * 32 > INT_MAX) return fail(GDN_ERR_OVERFLOW, "prepare dispatch exceeds int32");
    PrepParams p{};
    p.y = y; p.a = a; p.bl = b; p.A_log = A_log; p.dt_bias = dt_bias; p.qk = qk_norm; p.gb = g_beta;
    p.N = N; p.H = H; p.HQ = HQ; p.K = K; p.V = V; p.opts = opts;
    cudaError_t e = launch_prepare(p, dtype, static_cast<cudaStream_t>(stream), false);
    if (e != cudaSuccess) return cuda_fail(e, "prepare kernel launch");
    return GDN_OK;
}

int gdn_prepare(const void *y, const float *a, const float *b, const float *A_log,
                const float *dt_bias, float *qk_norm, float *g_beta, int N, int H, int HQ, int K,
                int V, int dtype, void *stream) {
    g_err[0] = 0;
    return prepare_impl(y, a, b, A_log, dt_bias, qk_norm, g_beta, N, H, HQ, K, V, 0, dtype, stream);
}

int gdn_prepare_ex(const void *y, const float *a, const float *b, const float *A_log,
                   const float *dt_bias, float *qk_norm, float *g_beta, int N, int H, int HQ,
                   int K, int V, int opts, int dtype, void *stream) {
    g_err[0] = 0;
    return prepare_impl(y, a, b, A_log, dt_bias, qk_norm, g_beta, N, H, HQ, K, V, opts, dtype,
                        stream);
}

static int delta_impl(const void *y, const float *qk_norm, const float *g_beta,
                      const int32_t *offsets, const float *state_init, void *out,
                      float *state_fin, int B, int N, int H, int HQ, int K, int V, float scale,
                      int dtype, void *stream, const Capture *cap, int opts = 0) {
    if (opts & ~GDN_OPT_ALL) return fail(GDN_ERR_UNSUPPORTED, "delta: unknown option bits 0x%x", opts);
    if (!dtype_ok(dtype)) return fail(GDN_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
    long width;
    int rc = check_heads(H, HQ, K, V, &width);
    if (rc) return rc;
    if (B < 1 || N < 0) return fail(GDN_ERR_SHAPE, "need B>=1 and N>=0 (B=%d N=%d)", B, N);
    if (!offsets || !state_init || !state_fin || (N > 0 && (!y || !qk_norm || !g_beta || !out)))
        return fail(GDN_ERR_NULL, "delta: a required pointer is NULL");
    if ((long)B * H * V * 32 > INT_MAX) return fail(GDN_ERR_OVERFLOW, "delta dispatch B*H*V*32 exceeds int32");
    if (!std::isfinite(scale)) return fail(GDN_ERR_SHAPE, "scale is not finite");
    if ((opts & GDN_OPT_GATE_PER_CHANNEL) && cap)
        return fail(GDN_ERR_UNSUPPORTED, "delta: state-update capture with the per-channel gate");
    DeltaParams p{};
    p.y = y; p.qk = qk_norm; p.gb = g_beta; p.offsets = offsets; p.state_init = state_init;
    p.out = out; p.state_fin = state_fin; p.B = B; p.N = N; p.H = H; p.HQ = HQ; p.K = K; p.V = V;
    p.scale = scale == 0.f ? 1.f / std::sqrt((float)K) : scale;
    p.serial_max_len = INT_MAX;
    p.max_len = INT_MAX;
    p.conv_fin = nullptr;
    p.opts = opts;
    if (opts & GDN_OPT_GATE_PER_CHANNEL) {  // g_beta = g [N, H, K] then beta [N, H]
        if ((long)N * H * K > INT_MAX) return fail(GDN_ERR_OVERFLOW, "delta: N*H*K gates exceed int32");
        p.gpc = g_beta;
        p.gpc_logits = 0;
        p.beta_base = g_beta + (size_t)N * H * K;
    }
    if (cap) {
        p.cap = cap->cap; p.counts = cap->counts; p.active = cap->active; p.capsule = cap->capsule;
    }
    cudaError_t e = launch_delta_serial(p, dtype, static_cast<cudaStream_t>(stream), false);
    if (e != cudaSuccess) return cuda_fail(e, "delta kernel launch");
    return GDN_OK;
}

int gdn_delta_varlen(const void *y, const float *qk_norm, const float *g_beta,
                     const int32_t *offsets, const float *state_init, void *out, float *state_fin,
                     int B, int N, int H, int HQ, int K, int V, float scale, int dtype,
                     void *stream) {
    g_err[0] = 0;
    return delta_impl(y, qk_norm, g_beta, offsets, state_init, out, state_fin, B, N, H, HQ, K,
                      V, scale, dtype, stream, nullptr);
}

int gdn_delta_varlen_ex(const void *y, const float *qk_norm, const float *g_beta,
                        const int32_t *offsets, const float *state_init, void *out,
                        float *state_fin, int B, int N, int H, int HQ, int K, int V,
                        float scale, int opts, int dtype, void *stream) {
    g_err[0] = 0;
    return delta_impl(y, qk_norm, g_beta, offsets, state_init, out, state_fin, B, N, H, HQ, K,
                      V, scale, dtype, stream, nullptr, opts);
}

int gdn_delta_varlen_capture(const void *y, const float *qk_norm, const float *g_beta,
                             const int32_t *offsets, const float *state_init, void *out,
                             float *state_fin, int cap, const int32_t *counts,
                             const int32_t *active, float *capsule, int B, int N, int H, int HQ,
                             int K, int V, float scale, int dtype, void *stream) {
    g_err[0] = 0;
    const Capture c{cap, counts, active, nullptr, capsule};
    int rc = check_capture(c, "delta capture");
    if (rc) return rc;
    if (!capsule) return fail(GDN_ERR_NULL, "delta capture: capsule is NULL");
    if ((long)B * cap * ((long)H + (long)HQ * K + (long)H * V) > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "delta capsule size exceeds int32");
    return delta_impl(y, qk_norm, g_beta, offsets, state_init, out, state_fin, B, N, H, HQ, K,
                      V, scale, dtype, stream, &c);
}

size_t gdn_workspace_bytes(int B, int N, int H, int HQ, int K, int V, int Kc, int D, int dtype) {
    if (B < 1 || N < 0 || H < 1 || HQ < 1 || K < 1 || V < 1 || Kc < 1 || D < 1) return 0;
    if (!dtype_ok(dtype) || H % HQ != 0 || K > 256) return 0;
    return ws_layout(B, N, H, HQ, K, V, dtype).total;
}

size_t gdn_workspace_bytes_ex(int B, int N, int H, int HQ, int K, int V, int Kc, int D, int dtype,
                              int opts) {
    const size_t base = gdn_workspace_bytes(B, N, H, HQ, K, V, Kc, D, dtype);
    if (base == 0 || (opts & ~GDN_OPT_ALL) != 0) return 0;
    if (!(opts & GDN_OPT_GATE_PER_CHANNEL) || (opts & GDN_OPT_NO_DECAY)) return base;
    const int width = 2 * HQ * K + H * V;
    if (!chunked_supported(dtype, K, V, width)) return base;
    return base + align256(pc_slots(B, N) * H * pc_img_bytes());
}

int gdn_workspace_status(const void *workspace, int *counts, void *stream) {
    g_err[0] = 0;
    if (!workspace) return fail(GDN_ERR_NULL, "workspace is NULL");
    WsHeader h;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status");
    if (counts) {
        counts[0] = h.n_serial;
        counts[1] = h.n_chunked;
        counts[2] = h.n_units;
    }
    if (h.status == GDN_ERR_OFFSETS) return fail(GDN_ERR_OFFSETS, "device check: malformed offsets");
    if (h.status == GDN_ERR_TIMEOUT) return fail(GDN_ERR_TIMEOUT, "device check: a bounded wait gave up");
    return h.status;
}

static int layer_impl(const void *qkv, const void *w, const void *bias, const float *a,
                      const float *b, const float *A_log, const float *dt_bias,
                      const int32_t *offsets, const int32_t *offsets_host, const void *conv_init,
                      void *conv_fin, const float *state_init, void *out, float *state_fin,
                      int B, int N, int H, int HQ, int K, int V, int Kc, int D, int act,
                      float scale, int dtype, void *workspace, size_t ws_bytes, void *stream,
                      const Capture *cap, int opts = 0, bool allow_fork = true) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
    if (act != GDN_ACT_NONE && act != GDN_ACT_SILU) return fail(GDN_ERR_UNSUPPORTED, "activation %d not supported", act);
    long width;
    int rc = check_heads(H, HQ, K, V, &width);
    if (rc) return rc;
    if (B < 1 || N < 0 || Kc < 1 || D < 1)
        return fail(GDN_ERR_SHAPE, "need B>=1, N>=0, Kc>=1, D>=1 (B=%d N=%d Kc=%d D=%d)", B, N, Kc, D);
    const long L = (long)(Kc - 1) * D;
    if (L >= INT_MAX) return fail(GDN_ERR_OVERFLOW, "receptive field (Kc-1)*D exceeds int32");
    if (L > 4096) return fail(GDN_ERR_UNSUPPORTED, "receptive field L=%ld above 4096", L);
    if (Kc > 64) return fail(GDN_ERR_UNSUPPORTED, "conv width Kc=%d above 64", Kc);
    if (!w || !offsets || !state_init || !state_fin || (N > 0 && (!qkv || !out)) ||
        (L > 0 && (!conv_init || !conv_fin)))
        return fail(GDN_ERR_NULL, "layer: a required pointer is NULL");
    rc = check_opts(opts, N, a, b, A_log, dt_bias, "layer");
    if (rc) return rc;
    // without decay a per-channel gate is g = 1 in every channel: the plain rule
    if (opts & GDN_OPT_NO_DECAY) opts &= ~GDN_OPT_GATE_PER_CHANNEL;
    const bool per_channel = (opts & GDN_OPT_GATE_PER_CHANNEL) != 0;
    if (per_channel && cap)
        return fail(GDN_ERR_UNSUPPORTED, "layer: state-update capture with the per-channel gate");
    if (per_channel && (long)N * H * K > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "layer: N*H*K decay logits exceed int32");
    if ((long)B * H * V * 32 > INT_MAX || (long)B * width > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "layer dispatch size exceeds int32");
    if (!std::isfinite(scale)) return fail(GDN_ERR_SHAPE, "scale is not finite");
    const WsLayout lay = ws_layout(B, N, H, HQ, K, V, dtype);
    if (!workspace || ((uintptr_t)workspace & 255) != 0)
        return fail(GDN_ERR_WORKSPACE, "workspace must be a non-NULL 256-byte aligned device pointer");
    if (ws_bytes < lay.total)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, lay.total);
    if (offsets_host) {
        rc = check_offsets_host(offsets_host, B, N);
        if (rc) return rc;
    }
    // path choice per sequence: at least `thr` tokens -> chunked kernel
    // (the per-channel gate has its own chunked kernel; it reads a [N, H, K] as
    // 16-byte vectors)
    const size_t pc_img = per_channel ? pc_slots(B, N) * H * pc_img_bytes() : 0;
    const bool chunk_ok = chunked_supported(dtype, K, V, (int)width) &&
                          (!per_channel || (((uintptr_t)a & 15) == 0 && ((uintptr_t)state_init & 15) == 0 &&
                                            ((uintptr_t)state_fin & 15) == 0 &&
                                            ws_bytes >= lay.total + pc_img));
    int thr = chunk_min_len();
    // Long chunked sequences that leave most of the GPU idle are cut into
    // segments run in parallel (two chunked launches and a combine step).
    // Sequences shorter than one chunk beside them run token-serially then.
    const SegmentPlan seg = chunk_ok && offsets_host && lay.seg != 0
                                ? plan_segments(offsets_host, B, H, V, segment_plan_thr(thr),
                                                lay.seg_seqs, sm_count_host())
                                : SegmentPlan{};
    if (seg.n > 0) thr = segment_plan_thr(thr);
    const int serial_max = chunk_ok ? thr : INT_MAX;
    bool run_chunked = chunk_ok && N >= thr;
    long max_units = run_chunked ? (long)(B < N / thr ? B : N / thr) * H * (V / 128) : 0;
    if (run_chunked && offsets_host) {
        long n = 0;
        for (int i = 0; i < B; ++i) n += (offsets_host[i + 1] - offsets_host[i]) >= thr;
        run_chunked = n > 0;
        max_units = n * H * (V / 128);
    }
    // tokens of token-serial sequences need the prepare step; with host
    // offsets a batch of chunked sequences only skips it
    const bool capsule = cap && cap->capsule;
    bool need_prep = true;
    if (offsets_host && !capsule) {
        need_prep = false;
        for (int i = 0; i < B && !need_prep; ++i) {
            const int len = offsets_host[i + 1] - offsets_host[i];
            need_prep = len > 0 && len < serial_max;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws + lay.header);
    const float eff_scale = scale == 0.f ? 1.f / std::sqrt((float)K) : scale;
    int max_len = INT_MAX;  // unknown without host offsets
    if (offsets_host) {
        max_len = 0;
        for (int i = 0; i < B; ++i) {
            const int len = offsets_host[i + 1] - offsets_host[i];
            max_len = len > max_len ? len : max_len;
        }
    }
    void *y = ws + lay.y;
    float *qk = reinterpret_cast<float *>(ws + lay.qk);
    float *gb = reinterpret_cast<float *>(ws + lay.gb);
    int32_t *order = reinterpret_cast<int32_t *>(ws + lay.order);

    ConvParams cp{};
    cp.x = qkv; cp.w = w; cp.bias = bias; cp.offsets = offsets; cp.init = conv_init; cp.y = y;
    cp.B = B; cp.N = N; cp.C = (int)width; cp.Kc = Kc; cp.D = D; cp.L = (int)L;
    cp.silu = act == GDN_ACT_SILU;
    cp.prep = need_prep ? 1 : 0; cp.qk = qk; cp.gb = gb; cp.a = a; cp.bl = b; cp.A_log = A_log; cp.dt_bias = dt_bias;
    cp.H = H; cp.HQ = HQ; cp.K = K; cp.V = V; cp.prep_max_len = serial_max;
    cp.header = hdr; cp.chunk_min_len = serial_max;
    cp.prep_cap = capsule ? cap->cap : 0;  // the captured prefix of chunked sequences
    cp.opts = opts;
    cp.seq_order = run_chunked ? order : nullptr; cp.VT = V / 128;
    bool fused = false;
    mark_before(GDN_KERNEL_CONV, s);
    cudaError_t e = launch_conv(cp, dtype, s, &fused);
    mark_after(GDN_KERNEL_CONV, s);
    if (e != cudaSuccess) return cuda_fail(e, "conv kernel launch");
    if (need_prep && !fused && N > 0) {
        PrepParams pp{};
        pp.y = y; pp.a = a; pp.bl = b; pp.A_log = A_log; pp.dt_bias = dt_bias; pp.qk = qk; pp.gb = gb;
        pp.N = N; pp.H = H; pp.HQ = HQ; pp.K = K; pp.V = V; pp.opts = opts;
        e = launch_prepare(pp, dtype, s, true);
        if (e != cudaSuccess) return cuda_fail(e, "prepare kernel launch");
    }
    // segment-parallel buffers and plan (both chunked forms)
    ChunkLaunch segl{};
    if (seg.n > 0) {
        float *segb = reinterpret_cast<float *>(ws + lay.seg);
        segl.nseq_seg = seg.n;
        for (int i = 0; i < kMaxSegSeqs; ++i) segl.seg_seq[i] = seg.seq[i];
        for (int i = 0; i <= kMaxSegSeqs; ++i) {
            segl.seg_m0[i] = seg.m0[i];
            segl.seg_s0[i] = seg.s0[i];
        }
        segl.seg_M = segb;
        segl.seg_L = segl.seg_M + (size_t)lay.seg_seqs * segment_m_floats(H);
        segl.seg_S = segl.seg_L + (size_t)lay.seg_seqs * segment_l_floats(H, V);
        segl.offsets = offsets; segl.state_init = state_init; segl.header = hdr;
        segl.H = H; segl.V = V;
    }
    auto launch_chunked = [&]() -> int {
        if (per_channel) {  // the per-key-channel chunked kernels
            const __nv_bfloat16 *yb = static_cast<const __nv_bfloat16 *>(y);
            PcParams pp{};
            pp.qb = yb; pp.kb = yb + (size_t)HQ * K; pp.rs = width;
            pp.g = a; pp.bl = b; pp.A_log = A_log; pp.dt_bias = dt_bias;
            pp.offsets = offsets; pp.seq_order = order; pp.header = hdr;
            pp.state_init = state_init; pp.state_fin = state_fin;
            pp.out = static_cast<__nv_bfloat16 *>(out); pp.ors = (long)H * V;
            pp.B = B; pp.N = N; pp.H = H; pp.HQ = HQ; pp.V = V; pp.VT = V / 128;
            pp.scale = eff_scale; pp.opts = opts; pp.gate_factor = 0;
            pp.thr = thr;
            pp.img = reinterpret_cast<unsigned char *>(ws + lay.total);  // after the plain layout
            pp.img_bytes = (long)pc_img_bytes();
            // the v rows, read by the scan kernel in [64 x 16] boxes of the conv output
            if (!encode_operand_map(&pp.vmap, y, N, width, 16))
                return fail(GDN_ERR_CUDA, "encoding the per-channel v tensor map failed");
            pp.vcol0 = 2 * HQ * K;
            // a (chunk, sequence, head) grid unless most of its CTAs would be empty
            const long gchunks = offsets_host && B <= 65535 ? (max_len + 15) / 16 : 0;
            pp.grid_chunks = gchunks * B * 4 <= (long)pc_slots(B, N) * 5 ? (int)gchunks : 0;
            pp.uniform_len = 0;
            mark_before(GDN_KERNEL_CHUNKED, s);
            cudaError_t ce = seg.n > 0 ? launch_delta_chunked_pc_segmented(pp, segl, s)
                                       : launch_delta_chunked_pc(pp, max_units, s);
            mark_after(GDN_KERNEL_CHUNKED, s);
            if (ce != cudaSuccess) return cuda_fail(ce, "per-channel chunked kernel launch");
            return GDN_OK;
        }
        ChunkLaunch cl{};
        cl.y = y; cl.a = a; cl.bl = b; cl.A_log = A_log; cl.dt_bias = dt_bias;
        cl.offsets = offsets; cl.seq_order = order; cl.header = hdr;
        cl.state_init = state_init; cl.state_fin = state_fin; cl.out = out;
        cl.B = B; cl.N = N; cl.H = H; cl.HQ = HQ; cl.V = V; cl.W = (int)width;
        cl.scale = eff_scale; cl.max_units = max_units; cl.opts = opts;
        if (seg.n > 0) {
            cl.nseq_seg = seg.n;
            for (int i = 0; i < kMaxSegSeqs; ++i) cl.seg_seq[i] = seg.seq[i];
            for (int i = 0; i <= kMaxSegSeqs; ++i) {
                cl.seg_m0[i] = seg.m0[i];
                cl.seg_s0[i] = seg.s0[i];
            }
            cl.seg_M = segl.seg_M;
            cl.seg_L = segl.seg_L;
            cl.seg_S = segl.seg_S;
        }
        mark_before(GDN_KERNEL_CHUNKED, s);
        cudaError_t ce = seg.n > 0 ? launch_delta_chunked_segmented(cl, s) : launch_delta_chunked(cl, s);
        mark_after(GDN_KERNEL_CHUNKED, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "chunked kernel launch");
        return GDN_OK;
    };

    DeltaParams dp{};
    dp.y = y; dp.qk = qk; dp.gb = gb; dp.offsets = offsets; dp.state_init = state_init;
    dp.out = out; dp.state_fin = state_fin; dp.B = B; dp.N = N; dp.H = H; dp.HQ = HQ; dp.K = K; dp.V = V;
    dp.scale = eff_scale;
    dp.serial_max_len = serial_max;
    dp.max_len = max_len;
    // the recurrence kernel also writes the final conv state (after the conv
    // kernel has finished reading the initial one) and overlaps, through
    // programmatic dependent launch, its state loads with the conv kernel
    dp.conv_x = qkv; dp.conv_init = conv_init; dp.conv_fin = L > 0 ? conv_fin : nullptr;
    dp.conv_L = (int)L;
    dp.opts = opts;
    if (per_channel) {  // gates from the per-channel logits; beta from the prepare step
        dp.gpc = a;
        dp.gpc_logits = 1;
        dp.A_log = A_log;
        dp.dt_bias = dt_bias;
        dp.beta_base = gb + (size_t)N * H;
    }
    if (cap) {
        dp.cap = cap->cap; dp.counts = cap->counts; dp.active = cap->active;
        dp.conv_updates = cap->conv_updates; dp.capsule = cap->capsule;
    }
    // With a capsule the token-serial kernel also replays the captured prefix
    // of chunked sequences from their initial state, so it runs before the
    // chunked kernel (which may overwrite that state in place).
    const bool serial_first = capsule && run_chunked;
    // With CTA slots left free by the chunked units, the token-serial kernel
    // (short sequences, and the final conv state of all) runs beside the
    // chunked kernel on a side stream: both read only what the conv pass wrote
    // and write disjoint outputs.  Also with no short sequence at all: the
    // final conv state then leaves the chunked kernel's critical path (prefill
    // 729 -> 719 us a step).
    int n_serial_host = 0;
    if (offsets_host)
        for (int i = 0; i < B; ++i) {
            const int len = offsets_host[i + 1] - offsets_host[i];
            n_serial_host += len > 0 && len < serial_max;
        }
    // (with no short sequence the token-serial kernel still writes the final
    // conv state, which nothing else in the call reads or writes)
    const bool conv_fin_written = L > 0 && conv_fin != nullptr;
    ForkSet *f = nullptr;
    std::unique_lock<std::mutex> fork_lock(g_fork_mu, std::defer_lock);
    // (Only with slots left free: with more units than slots the token-serial
    // CTAs take the slots the last chunked units leave and share their SMs,
    // which cost the ragged batch's chunked kernel 5% of its time for a 1%
    // shorter step, and made the per-channel prepare kernel's grid 1.3% slower.)
    if (allow_fork && run_chunked && !serial_first && seg.n == 0 && (n_serial_host > 0 || conv_fin_written) &&
        max_units < 2L * sm_count_host()) {
        fork_lock.lock();
        if (fork_set(&f, s) != cudaSuccess) {  // not available: one after the other
            f = nullptr;
            fork_lock.unlock();
        }
    }
    if (f != nullptr) {
        e = cudaEventRecord(f->fork, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(f->side, f->fork, 0);
        if (e != cudaSuccess) return cuda_fail(e, "forking the token-serial kernel");
        mark_before(GDN_KERNEL_SERIAL, f->side);
        e = launch_delta_serial(dp, dtype, f->side, /*pdl=*/false);
        mark_after(GDN_KERNEL_SERIAL, f->side);
        if (e != cudaSuccess) return cuda_fail(e, "delta kernel launch");
        e = cudaEventRecord(f->join, f->side);
        if (e != cudaSuccess) return cuda_fail(e, "joining the token-serial kernel");
        rc = launch_chunked();
        e = cudaStreamWaitEvent(s, f->join, 0);  // joined even if the chunked launch failed
        if (rc) return rc;
        if (e != cudaSuccess) return cuda_fail(e, "joining the token-serial kernel");
        return GDN_OK;
    }
    if (run_chunked && !serial_first) {
        rc = launch_chunked();
        if (rc) return rc;
    }
    mark_before(GDN_KERNEL_SERIAL, s);
    e = launch_delta_serial(dp, dtype, s, /*pdl=*/true);
    mark_after(GDN_KERNEL_SERIAL, s);
    if (e != cudaSuccess) return cuda_fail(e, "delta kernel launch");
    if (serial_first) {
        rc = launch_chunked();
        if (rc) return rc;
    }
    return GDN_OK;
}

}  // extern "C"

namespace gdn {
// The layer call without the side-stream fork (creates no stream or event).
int layer_varlen_nofork(const void *qkv, const void *w, const void *bias, const float *a,
                        const float *b, const float *A_log, const float *dt_bias,
                        const int32_t *offsets, const int32_t *offsets_host,
                        const void *conv_init, void *conv_fin, const float *state_init,
                        void *out, float *state_fin, int B, int N, int H, int HQ, int K, int V,
                        int Kc, int D, int act, float scale, int dtype, void *workspace,
                        size_t ws_bytes, void *stream) {
    g_err[0] = 0;
    return layer_impl(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host, conv_init,
                      conv_fin, state_init, out, state_fin, B, N, H, HQ, K, V, Kc, D, act, scale,
                      dtype, workspace, ws_bytes, stream, nullptr, 0, /*allow_fork=*/false);
}
}  // namespace gdn

extern "C" {

int gdn_layer_varlen(const void *qkv, const void *w, const void *bias, const float *a,
                     const float *b, const float *A_log, const float *dt_bias,
                     const int32_t *offsets, const int32_t *offsets_host, const void *conv_init,
                     void *conv_fin, const float *state_init, void *out, float *state_fin, int B,
                     int N, int H, int HQ, int K, int V, int Kc, int D, int act, float scale,
                     int dtype, void *workspace, size_t ws_bytes, void *stream) {
    g_err[0] = 0;
    return layer_impl(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host, conv_init,
                      conv_fin, state_init, out, state_fin, B, N, H, HQ, K, V, Kc, D, act, scale,
                      dtype, workspace, ws_bytes, stream, nullptr);
}

int gdn_layer_varlen_capture(const void *qkv, const void *w, const void *bias, const float *a,
                             const float *b, const float *A_log, const float *dt_bias,
                             const int32_t *offsets, const int32_t *offsets_host,
                             const void *conv_init, void *conv_fin, const float *state_init,
                             void *out, float *state_fin, int cap, const int32_t *counts,
                             const int32_t *active, void *conv_updates, float *capsule, int B,
                             int N, int H, int HQ, int K, int V, int Kc, int D, int act,
                             float scale, int dtype, void *workspace, size_t ws_bytes,
                             void *stream) {
    g_err[0] = 0;
    const Capture c{cap, counts, active, conv_updates, capsule};
    int rc = check_capture(c, "layer capture");
    if (rc) return rc;
    if (!conv_updates && !capsule) return fail(GDN_ERR_NULL, "layer capture: no capture buffer given");
    if ((long)B * cap * (2L * HQ * K + (long)H * V) > INT_MAX ||
        (long)B * cap * ((long)H + (long)HQ * K + (long)H * V) > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "layer capture buffers exceed int32 elements");
    return layer_impl(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host, conv_init,
                      conv_fin, state_init, out, state_fin, B, N, H, HQ, K, V, Kc, D, act, scale,
                      dtype, workspace, ws_bytes, stream, &c);
}

static int dense_check(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, void *out, int B, int S, int H, int n,
                       int gate_per_channel, float scale, int dtype) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
    if (B < 1 || S < 0 || H < 1 || n < 1)
        return fail(GDN_ERR_SHAPE, "dense: need B>=1, S>=0, H>=1, n>=1 (B=%d S=%d H=%d n=%d)", B, S, H, n);
    if (n > 256) return fail(GDN_ERR_SHAPE, "dense: head size n=%d above 256", n);
    if (gate_per_channel != 0 && gate_per_channel != 1)
        return fail(GDN_ERR_SHAPE, "dense: gate_per_channel must be 0 or 1");
    if ((long)B * S * H * n > INT_MAX || (long)B * H * n * 32 > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "dense: tensor or dispatch size exceeds int32");
    if (S > 0 && (!q || !k || !v || !g || !beta || !out))
        return fail(GDN_ERR_NULL, "dense: a required pointer is NULL");
    if (!std::isfinite(scale)) return fail(GDN_ERR_SHAPE, "scale is not finite");
    return GDN_OK;
}

static int dense_serial(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *state_init, void *out, float *state_fin,
                        int B, int S, int H, int n, int gate_per_channel, float scale, int dtype,
                        void *stream) {
    DenseParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.state_init = state_init; p.out = out;
    p.state_fin = state_fin; p.B = B; p.S = S; p.H = H; p.n = n; p.per_channel = gate_per_channel;
    p.scale = scale == 0.f ? 1.f / std::sqrt((float)n) : scale;
    cudaError_t e = launch_delta_dense(p, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dense kernel launch");
    return GDN_OK;
}

int gdn_gated_delta_dense(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *state_init, void *out,
                          float *state_fin, int B, int S, int H, int n, int gate_per_channel,
                          float scale, int dtype, void *stream) {
    g_err[0] = 0;
    int rc = dense_check(q, k, v, g, beta, out, B, S, H, n, gate_per_channel, scale, dtype);
    if (rc) return rc;
    return dense_serial(q, k, v, g, beta, state_init, out, state_fin, B, S, H, n,
                        gate_per_channel, scale, dtype, stream);
}

// Workspace of the dense call's chunked route: header, order, offsets, the
// three operand maps (q, k, v read in place), log gates [B S, H], a zero
// initial state and a final-state scratch [B, H, n, n] (for NULL state_init /
// state_fin).
struct DenseWs {
    size_t header, order, offsets, maps, a, zero, fin, total;
};
static DenseWs dense_ws_layout(int B, int S, int H, int n) {
    DenseWs l;
    const size_t N = (size_t)B * S, st = (size_t)B * H * n * n * 4;
    size_t off = 0;
    l.header = off; off += align256(sizeof(WsHeader));
    l.order = off; off += align256((size_t)B * 4);
    l.offsets = off; off += align256((size_t)(B + 1) * 4);
    l.maps = off; off += align256(3 * sizeof(CUtensorMap));
    l.a = off; off += align256(N * H * 4);
    l.zero = off; off += align256(st);
    l.fin = off; off += align256(st);
    l.total = off;
    return l;
}

size_t gdn_dense_workspace_bytes(int B, int S, int H, int n, int dtype) {
    if (dtype != GDN_BF16 || n != 128 || B < 1 || S < 1 || H < 1) return 0;
    if ((long)B * S * H * n * 3 > INT_MAX) return 0;
    return dense_ws_layout(B, S, H, n).total;
}

size_t gdn_dense_workspace_bytes_ex(int B, int S, int H, int n, int dtype, int gate_per_channel) {
    const size_t base = gdn_dense_workspace_bytes(B, S, H, n, dtype);
    if (base == 0 || !gate_per_channel) return base;
    return base + align256(pc_slots(B, B * S) * H * pc_img_bytes());
}

// The dense call's per-key-channel route: the two-kernel chunked form on q,
// k, v read in place, the gate factors as given, raw beta, no q/k norm.
static int dense_per_channel_chunked(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *state_init, void *out,
                                     float *state_fin, int B, int S, int H, int n, float scale,
                                     char *ws, cudaStream_t st) {
    const DenseWs lay = dense_ws_layout(B, S, H, n);
    const float *s0 = state_init;
    if (!s0) {
        cudaError_t e = cudaMemsetAsync(ws + lay.zero, 0, (size_t)B * H * n * n * 4, st);
        if (e != cudaSuccess) return cuda_fail(e, "dense: zero initial state");
        s0 = reinterpret_cast<const float *>(ws + lay.zero);
    }
    float *sf = state_fin ? state_fin : reinterpret_cast<float *>(ws + lay.fin);
    DensePack pk{};  // offsets, order and header only
    pk.offsets = reinterpret_cast<int32_t *>(ws + lay.offsets);
    pk.order = reinterpret_cast<int32_t *>(ws + lay.order);
    pk.header = reinterpret_cast<WsHeader *>(ws + lay.header);
    pk.B = B; pk.S = S; pk.H = H; pk.n = n;
    cudaError_t e = launch_dense_pack(pk, st);
    if (e != cudaSuccess) return cuda_fail(e, "dense pack kernel launch");
    const long N = (long)B * S;
    PcParams pp{};
    if (!encode_operand_map(&pp.vmap, v, N, (long)H * n, 16))
        return fail(GDN_ERR_CUDA, "dense: encoding the v tensor map failed");
    pp.qb = static_cast<const __nv_bfloat16 *>(q);
    pp.kb = static_cast<const __nv_bfloat16 *>(k);
    pp.rs = (long)H * n;
    pp.g = g; pp.bl = beta; pp.A_log = nullptr; pp.dt_bias = nullptr;
    pp.offsets = pk.offsets; pp.seq_order = pk.order; pp.header = pk.header;
    pp.state_init = s0; pp.state_fin = sf;
    pp.out = static_cast<__nv_bfloat16 *>(out); pp.ors = (long)H * n;
    pp.B = B; pp.N = (int)N; pp.H = H; pp.HQ = H; pp.V = n; pp.VT = n / 128; pp.vcol0 = 0;
    pp.scale = scale == 0.f ? 1.f / std::sqrt((float)n) : scale;
    pp.opts = GDN_OPT_BETA_RAW | GDN_OPT_NO_QK_NORM;
    pp.gate_factor = 1;
    pp.thr = 1;
    pp.img = reinterpret_cast<unsigned char *>(ws + lay.total);
    pp.img_bytes = (long)pc_img_bytes();
    pp.grid_chunks = B <= 65535 ? (S + 15) / 16 : 0;
    pp.uniform_len = S;
    mark_before(GDN_KERNEL_CHUNKED, st);
    e = launch_delta_chunked_pc(pp, (long)B * H * (n / 128), st);
    mark_after(GDN_KERNEL_CHUNKED, st);
    if (e != cudaSuccess) return cuda_fail(e, "dense: per-channel chunked kernel launch");
    return GDN_OK;
}

int gdn_gated_delta_dense_ws(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *state_init, void *out,
                             float *state_fin, int B, int S, int H, int n, int gate_per_channel,
                             float scale, int dtype, void *workspace, size_t ws_bytes,
                             void *stream) {
    g_err[0] = 0;
    int rc = dense_check(q, k, v, g, beta, out, B, S, H, n, gate_per_channel, scale, dtype);
    if (rc) return rc;
    const bool aligned = ((uintptr_t)q & 15) == 0 && ((uintptr_t)k & 15) == 0 &&
                         ((uintptr_t)v & 15) == 0 && ((uintptr_t)out & 15) == 0;
    const size_t need = gdn_dense_workspace_bytes(B, S, H, n, dtype);
    if (gate_per_channel) {
        // the per-channel chunked route when the workspace holds its chunk images
        const size_t need_pc = gdn_dense_workspace_bytes_ex(B, S, H, n, dtype, 1);
        const bool pc = need > 0 && S >= chunk_min_len() && aligned &&
                        chunked_supported(dtype, n, n, 3 * H * n) && ((uintptr_t)g & 15) == 0 &&
                        ((uintptr_t)state_init & 15) == 0 && ((uintptr_t)state_fin & 15) == 0 &&
                        workspace != nullptr && ((uintptr_t)workspace & 255) == 0 && ws_bytes >= need_pc;
        if (pc)
            return dense_per_channel_chunked(q, k, v, g, beta, state_init, out, state_fin, B, S, H,
                                             n, scale, static_cast<char *>(workspace),
                                             static_cast<cudaStream_t>(stream));
    }
    const bool chunked = need > 0 && !gate_per_channel && S >= chunk_min_len() && aligned &&
                         chunked_supported(dtype, n, n, 3 * H * n);
    if (!chunked)
        return dense_serial(q, k, v, g, beta, state_init, out, state_fin, B, S, H, n,
                            gate_per_channel, scale, dtype, stream);
    if (!workspace || ((uintptr_t)workspace & 255) != 0)
        return fail(GDN_ERR_WORKSPACE, "dense: workspace must be a non-NULL 256-byte aligned device pointer");
    if (ws_bytes < need) return fail(GDN_ERR_WORKSPACE, "dense: workspace has %zu bytes, needs %zu", ws_bytes, need);
    const DenseWs lay = dense_ws_layout(B, S, H, n);
    char *ws = static_cast<char *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const float *s0 = state_init;
    if (!s0) {
        cudaError_t e = cudaMemsetAsync(ws + lay.zero, 0, (size_t)B * H * n * n * 4, st);
        if (e != cudaSuccess) return cuda_fail(e, "dense: zero initial state");
        s0 = reinterpret_cast<const float *>(ws + lay.zero);
    }
    float *sf = state_fin ? state_fin : reinterpret_cast<float *>(ws + lay.fin);
    DensePack pk{};
    pk.g = g;
    pk.a = reinterpret_cast<float *>(ws + lay.a);
    pk.offsets = reinterpret_cast<int32_t *>(ws + lay.offsets);
    pk.order = reinterpret_cast<int32_t *>(ws + lay.order);
    pk.header = reinterpret_cast<WsHeader *>(ws + lay.header);
    pk.B = B; pk.S = S; pk.H = H; pk.n = n;
    // q, k, v are read in place by the chunked kernel: one operand map each
    const long N = (long)B * S;
    if (!encode_operand_map(&pk.maps[0], q, N, (long)H * n) ||
        !encode_operand_map(&pk.maps[1], k, N, (long)H * n) ||
        !encode_operand_map(&pk.maps[2], v, N, (long)H * n))
        return fail(GDN_ERR_CUDA, "dense: encoding the q, k, v tensor maps failed");
    pk.maps_dst = ws + lay.maps;
    cudaError_t e = launch_dense_pack(pk, st);
    if (e != cudaSuccess) return cuda_fail(e, "dense pack kernel launch");
    ChunkLaunch cl{};
    cl.y = nullptr; cl.gmaps = ws + lay.maps;
    cl.a = pk.a; cl.bl = beta; cl.A_log = nullptr; cl.dt_bias = nullptr;
    cl.offsets = pk.offsets; cl.seq_order = pk.order; cl.header = pk.header;
    cl.state_init = s0; cl.state_fin = sf; cl.out = out;
    cl.B = B; cl.N = B * S; cl.H = H; cl.HQ = H; cl.V = n; cl.W = 3 * H * n;
    cl.scale = scale == 0.f ? 1.f / std::sqrt((float)n) : scale;
    cl.max_units = (long)B * H * (n / 128);
    // the dense call's values as given: exp gate of ln g, raw rate, no q/k norm
    cl.opts = GDN_OPT_GATE_EXP | GDN_OPT_BETA_RAW | GDN_OPT_NO_QK_NORM;
    mark_before(GDN_KERNEL_CHUNKED, st);
    e = launch_delta_chunked(cl, st);
    mark_after(GDN_KERNEL_CHUNKED, st);
    if (e != cudaSuccess) return cuda_fail(e, "dense: chunked kernel launch");
    return GDN_OK;
}

int gdn_layer_varlen_ex(const void *qkv, const void *w, const void *bias, const float *a,
                        const float *b, const float *A_log, const float *dt_bias,
                        const int32_t *offsets, const int32_t *offsets_host,
                        const void *conv_init, void *conv_fin, const float *state_init,
                        void *out, float *state_fin, int opts, int cap, const int32_t *counts,
                        const int32_t *active, void *conv_updates, float *capsule, int B, int N,
                        int H, int HQ, int K, int V, int Kc, int D, int act, float scale,
                        int dtype, void *workspace, size_t ws_bytes, void *stream) {
    g_err[0] = 0;
    if (cap == 0)
        return layer_impl(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host, conv_init,
                          conv_fin, state_init, out, state_fin, B, N, H, HQ, K, V, Kc, D, act,
                          scale, dtype, workspace, ws_bytes, stream, nullptr, opts);
    const Capture c{cap, counts, active, conv_updates, capsule};
    int rc = check_capture(c, "layer capture");
    if (rc) return rc;
    if (!conv_updates && !capsule) return fail(GDN_ERR_NULL, "layer capture: no capture buffer given");
    if ((long)B * cap * (2L * HQ * K + (long)H * V) > INT_MAX ||
        (long)B * cap * ((long)H + (long)HQ * K + (long)H * V) > INT_MAX)
        return fail(GDN_ERR_OVERFLOW, "layer capture buffers exceed int32 elements");
    return layer_impl(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host, conv_init,
                      conv_fin, state_init, out, state_fin, B, N, H, HQ, K, V, Kc, D, act, scale,
                      dtype, workspace, ws_bytes, stream, &c, opts);
}

}  // extern "C"
