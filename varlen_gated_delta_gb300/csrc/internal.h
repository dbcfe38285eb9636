// internal.h - host-side interface between the C ABI (api.cpp) and the
// kernel launchers (*.cu).  Not installed; the public ABI is include/gdn.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "gdn.h"  // GDN_OPT_* rule / activation options

namespace gdn {

// Workspace header written by the device (first 256 bytes of a workspace).
struct WsHeader {
    int status;          // gdn_status of the device-side checks
    int n_serial;        // sequences run by the token-serial kernel
    int n_chunked;       // sequences run by the chunked kernel
    int n_units;         // chunked work units
    unsigned int next_unit;  // work counter of the persistent chunked kernel
    unsigned int seg_next[2];  // work counters of the two segmented chunked launches
    int pad[57];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

// Runs set() once per device (ids below 64; others every time) and records
// success in `done`: for per-device function attributes such as a kernel's
// dynamic shared memory limit.
template <typename F>
inline cudaError_t once_per_device(std::atomic<uint64_t> &done, F set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

struct ConvParams {
    const void *x, *w, *bias;
    const int32_t *offsets;
    const void *init;
    void *y;
    int B, N, C, Kc, D, L, silu;
    // fused prepare (prep != 0): q/k norms and g/beta for tokens of sequences
    // shorter than prep_max_len.
    int prep;
    float *qk, *gb;
    const float *a, *bl, *A_log, *dt_bias;
    int H, HQ, K, V, prep_max_len;
    int prep_cap;  // also prepare the first prep_cap tokens of every sequence
    int opts;      // GDN_OPT_* rule / activation options
    // block 0 validates offsets and writes counts when header != nullptr;
    // with seq_order != nullptr it also lists the sequences of at least
    // chunk_min_len tokens, longest first, and sets n_units = count * H * VT
    WsHeader *header;
    int chunk_min_len;
    int32_t *seq_order;
    int VT;
};

struct PrepParams {
    const void *y;
    const float *a, *bl, *A_log, *dt_bias;
    float *qk, *gb;
    int N, H, HQ, K, V;
    int opts;  // GDN_OPT_*
};

struct DeltaParams {
    const void *y;
    const float *qk, *gb;
    const int32_t *offsets;
    const float *state_init;
    void *out;
    float *state_fin;
    int B, N, H, HQ, K, V;
    float scale;
    int serial_max_len;  // sequences with len >= this are skipped (chunked path)
    int max_len;         // upper bound on sequence length (<= 1 selects the decode variant)
    // optional fused conv final-state copy (layer path): conv_fin[b,c,:] =
    // last L raw inputs of (conv_init || sequence) for every sequence
    const void *conv_x;
    const void *conv_init;
    void *conv_fin;
    int conv_L;
    // optional state-update capture (cap > 0): conv_updates [B, cap, W] T (raw
    // input rows, written with the final conv state) and capsule
    // [B, cap * (H + HQ*K + H*V)] fp32; captured tokens of sequence b:
    // max(0, min(counts[b], cap, len)), none when active && active[0] == 0.
    // Chunked sequences get their capsule from a capture-only pass here.
    int cap;
    const int32_t *counts;
    const int32_t *active;
    void *conv_updates;
    float *capsule;
    int opts;  // GDN_OPT_* (GDN_OPT_NO_RETRIEVE and GDN_OPT_GATE_PER_CHANNEL act here)
    // per-key-channel gate (GDN_OPT_GATE_PER_CHANNEL): gpc [N, H, K] holds the
    // gates (gpc_logits == 0) or the decay logits, activated here with the
    // head's A_log / dt_bias (gpc_logits != 0: the layer); beta of token t,
    // head h is beta_base[t * H + h]
    const float *gpc;
    int gpc_logits;
    const float *A_log, *dt_bias;
    const float *beta_base;
};

// Launch `kernel` on `s`; with pdl the launch may overlap the previous kernel
// on the stream (the kernel must call pdl_wait_primary() before consuming it).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel launchers (return the launch error, counted in gdn_launch_count()).
cudaError_t launch_conv(const ConvParams &p, int dtype, cudaStream_t s, bool *fused_prep);
cudaError_t launch_conv_final(const void *x, const int32_t *offsets, const void *init,
                              void *fin, int B, int N, int C, int L, int dtype,
                              cudaStream_t s, int cap = 0, const int32_t *counts = nullptr,
                              void *updates = nullptr);
cudaError_t launch_prepare(const PrepParams &p, int dtype, cudaStream_t s, bool pdl);
cudaError_t launch_delta_serial(const DeltaParams &p, int dtype, cudaStream_t s, bool pdl);

// Segment-parallel chunked path: at most kMaxSegments segments per sequence,
// at most kMaxSegSeqs segmented sequences per call.
constexpr int kMaxSegments = 8;
constexpr int kMaxSegSeqs = 4;

// Chunked (tensor-core) recurrence for sequences listed in seq_order.
struct ChunkLaunch {
    const void *y;  // conv output [N, W] bf16
    const float *a, *bl, *A_log, *dt_bias;
    const int32_t *offsets, *seq_order;
    WsHeader *header;
    const float *state_init;
    float *state_fin;
    void *out;
    int B, N, H, HQ, V, W;
    float scale;
    long max_units;  // upper bound on work units (grid sizing)
    int opts;        // GDN_OPT_*
    // segment-parallel mode (nseq_seg > 0): sequences seg_seq[i], i < nseq_seg,
    // sequence i in P_i = seg_s0[i+1] - seg_s0[i] segments, seg_m0[i] =
    // sum over j < i of (P_j - 1); see launch_delta_chunked_segmented.
    // seg_M [seg_m0[n]][H][128][128], seg_L [seg_m0[n]][H][V][128],
    // seg_S [seg_s0[n]][H][V][128]
    int nseq_seg;
    int seg_seq[kMaxSegSeqs], seg_m0[kMaxSegSeqs + 1], seg_s0[kMaxSegSeqs + 1];
    float *seg_M, *seg_L, *seg_S;
    // dense layout: three CUtensorMaps (q, k, v [N, H V], bf16, see
    // encode_operand_map) in global memory, 64-byte aligned; y is unused then
    const void *gmaps = nullptr;
};
// Tensor map of a bf16 row-major [rows, cols] operand in the chunked kernel's
// tile format (64 x 64 boxes, 128-byte swizzle); false if encoding fails.
bool encode_operand_map(CUtensorMap *map, const void *base, long rows, long cols,
                        int box_rows = 64);
// Segments of a segmented sequence of `len` tokens cut into at most `nseg`:
// seg_len tokens each (a multiple of 64, so also of every chunk length),
// `count` segments in all.
__host__ __device__ inline void segment_split(int len, int nseg, int &seg_len, int &count) {
    seg_len = ((len + nseg - 1) / nseg + 63) / 64 * 64;
    count = seg_len > 0 ? (len + seg_len - 1) / seg_len : 0;
}
// Start states of the segments of c's segmented sequences from the phase-1
// transitions and local states (S_0 = state_init, S_{j+1} = S_j M_j + L_j),
// written to c.seg_S; launched with programmatic dependent launch.
cudaError_t launch_segment_combine(const ChunkLaunch &c, cudaStream_t s);
// Segment buffers: up to kMaxSegments segments of up to kMaxSegSeqs sequences.
inline size_t segment_m_floats(int H) { return (size_t)(kMaxSegments - 1) * H * 128 * 128; }
inline size_t segment_l_floats(int H, int V) { return (size_t)(kMaxSegments - 1) * H * V * 128; }
inline size_t segment_floats(int H, int V, int nseq) {  // M, L of P-1 segments; starts of P
    return (size_t)nseq * (segment_m_floats(H) + segment_l_floats(H, V) +
                           (size_t)kMaxSegments * H * V * 128);
}
// Dense-layout recurrence (q, k, v, out [B, S, H, n] T; g [B, S, H] or, with
// per_channel, [B, S, H, n] f32; beta [B, S, H] f32; state [B, H, n, n] f32,
// state_init NULL = zero, state_fin NULL = not written).
struct DenseParams {
    const void *q, *k, *v;
    const float *g, *beta;
    const float *state_init;
    void *out;
    float *state_fin;
    int B, S, H, n, per_channel;
    float scale;
};
cudaError_t launch_delta_dense(const DenseParams &p, int dtype, cudaStream_t s);

// Dense layout -> the chunked kernel's inputs (bf16, scalar gate, n = 128): the
// kernel reads q, k and v in place through three tensor maps that this step
// copies to global memory; it also writes a = ln(max(g, 1e-30)) [B S, H] (the
// kernel's exp gate), offsets i S, the sequence order and the workspace header
// for B H (n / 128) units.
struct DensePack {
    const float *g;
    float *a;
    int32_t *offsets, *order;
    WsHeader *header;
    int B, S, H, n;
    // the q, k, v operand maps, copied to maps_dst (global, 64-byte aligned)
    CUtensorMap maps[3];
    void *maps_dst;
};
cudaError_t launch_dense_pack(const DensePack &p, cudaStream_t s);

// Chunked recurrence with a per-key-channel gate (bf16, K = 128, V a multiple
// of 128), in two launches:
//  - a prepare kernel, one CTA per (16-token chunk, value head), parallel over
//    every chunk: it writes the chunk's state-independent operands (the chunk
//    image below) to the workspace;
//  - a scan kernel, persistent over (sequence, value head, V tile) units, that
//    carries the fp32 state in tensor memory and streams the images in.
// q, k rows of token t at qb / kb + t * rs (bf16, the first key head's
// columns; key head kh adds kh * 128), v rows through vmap (below);
// g [N, H, 128] holds the decay logits, or the gate
// factors when gate_factor; out [N, ors] (head h at column h * V).  Only
// sequences of at least `thr` tokens are processed.  Units and their order
// come from the workspace header and seq_order.
//
// Chunk n of sequence i (start s_i) has image slot (s_i >> 4) + i + n; slots
// of a valid offsets array never collide and number below pc_slots(B, N).
// The image of (slot, value head h) sits at img + (slot * H + h) * img_bytes:
//   [0, 8192)       [-W ; Qt], bf16 [32][128] as two SW128 blocks of [32][64]:
//                   rows 0..15 -W = -T diag(beta) Kt, rows 16..31 Qt = scale q e^{b_t}
//   [8192, 12288)   Kp = k e^{b_C - b_t}, bf16 [16 t][128 c], two SW128 blocks
//   [12288, 14336)  an SW128 [16][64] bf16 tile: columns 0..15 hold
//                   P = scale tril(QK) [t][i], columns 16..31 T diag(beta) [t][s]
//   [14336, 14848)  e^{b_C}, fp32 [128]
// The scan kernel reads the chunk's v rows itself, through vmap (a [64 x 16]
// box map of the matrix whose row t holds token t's v; value head h, V tile
// vt at column vcol0 + h * V + vt * 128).
constexpr uint32_t kPcImgHead = 14848;
inline size_t pc_img_bytes() { return kPcImgHead; }
inline size_t pc_slots(int B, int N) { return ((size_t)N + 15) / 16 + (size_t)B; }
struct PcParams {
    CUtensorMap vmap;  // (first: the map type carries its own alignment)
    const __nv_bfloat16 *qb, *kb;
    long rs;
    const float *g, *bl, *A_log, *dt_bias;
    const int32_t *offsets, *seq_order;
    WsHeader *header;
    const float *state_init;
    float *state_fin;
    __nv_bfloat16 *out;
    long ors;
    int B, N, H, HQ, V, VT;
    int vcol0;
    float scale;
    int opts;         // GDN_OPT_* (rule and activation options)
    int gate_factor;  // g holds gate factors, not logits
    int thr;          // chunked sequences have at least thr tokens
    unsigned char *img;  // chunk images, pc_slots(B, N) * H * pc_img_bytes() bytes
    long img_bytes;      // pc_img_bytes()
    // prepare grid: grid_chunks > 0 (at least the chunks of the longest
    // sequence; B <= 65535) runs a (chunk, sequence, head) grid, 0 a (slot,
    // head) grid; uniform_len > 0: sequence i is [i L, i L + L) (offsets are
    // then read by the scan kernel only)
    int grid_chunks;
    int uniform_len;
    // segment-parallel scan (seg_mode 1 / 2, as in ChunkLaunch; 0: one pass)
    int seg_mode, nseq_seg, seg_units;
    int seg_seq[kMaxSegSeqs], seg_m0[kMaxSegSeqs + 1], seg_s0[kMaxSegSeqs + 1];
    unsigned int *counter;  // work counter of a segment pass
    float *seg_M, *seg_L;
    const float *seg_S;
};
cudaError_t launch_delta_chunked_pc(const PcParams &p, long max_units, cudaStream_t s);
// The same with the scan segment-parallel for the sequences of `seg` (its
// nseq_seg, seg_seq, seg_m0, seg_s0 and seg buffers; p's seg fields are set here):
// prepare kernel, scan pass 1 (transitions M and local states L), segment
// combine, scan pass 2 (outputs and final states).
cudaError_t launch_delta_chunked_pc_segmented(const PcParams &p, const ChunkLaunch &seg,
                                              cudaStream_t s);

bool chunked_supported(int dtype, int K, int V, int W);
cudaError_t launch_delta_chunked(const ChunkLaunch &c, cudaStream_t s);
cudaError_t launch_delta_chunked_segmented(const ChunkLaunch &c, cudaStream_t s);

// Whether launch_conv can fuse the prepare step for this geometry.
bool conv_can_fuse_prepare(int dtype, int C, int K, const void *const *ptrs, int nptrs);

void note_launch(unsigned n = 1);

// gdn_layer_varlen without running the token-serial kernel on a side stream
// (so it creates no stream or event); same arguments and errors.
int layer_varlen_nofork(const void *qkv, const void *w, const void *bias, const float *a,
                        const float *b, const float *A_log, const float *dt_bias,
                        const int32_t *offsets, const int32_t *offsets_host,
                        const void *conv_init, void *conv_fin, const float *state_init,
                        void *out, float *state_fin, int B, int N, int H, int HQ, int K, int V,
                        int Kc, int D, int act, float scale, int dtype, void *workspace,
                        size_t ws_bytes, void *stream);

// Record a message for gdn_last_error() on this thread and return `code`.
int set_error(int code, const char *fmt, ...);

}  // namespace gdn
