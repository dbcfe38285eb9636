// delta_chunked.cu - chunkwise-parallel gated delta rule for prefill, on
// tcgen05 tensor cores with TMA-fed operands and the recurrent state held in
// tensor memory across chunks.
//
// The recurrence is the DELTA kernel of paged_ssm.rs (onnxruntime-ep-mlx
// 0.31.1): S_t = g_t S_{t-1} + beta_t (v_t - g_t S_{t-1} k_t) k_t^T,
// o_t = scale S_t q_t.  The pages print no chunked form; this kernel uses the
// WY/UT form derived from it.  Within a chunk of C = 64 tokens, with
// b_t = sum_{s<=t} log g_s, gamma_t = exp(b_t) and Gamma[t,i] = exp(b_t - b_i):
//   delta_t = beta_t (v_t - g_t S_{t-1} k_t) satisfies (I + A) Delta = diag(beta) V
//             - diag(beta gamma) K S_0^T,  A[t,i] = beta_t Gamma[t,i] k_t.k_i (i < t),
//   so with T = (I + A)^-1:  Delta = T diag(beta) V - (T diag(beta gamma) K) S_0^T,
//   O = scale (diag(gamma) Q S_0^T + (tril(Q K^T) o Gamma) Delta),
//   S_C = gamma_C S_0 + Delta^T diag(Gamma[C, .]) K.
// q and k enter unnormalised (the bf16 conv outputs, straight from TMA); the
// L2 norms r = 1/sqrt(|x|^2 + 1e-12) are applied as row/column scales.
//
// Per chunk and (sequence, value head, 128-row V tile) unit, every dense
// product is one tcgen05 MMA group with M = 128 (operands in SMEM, fp32
// accumulators in TMEM):
//   D1 = [Kr; Qr] Kr^T            (K K^T and Q K^T in one M=128 product)
//   D2 = Kr^T Tw^T   = W^T        (Tw = T diag(r_k beta gamma))
//   D3 = V^T Tb^T - S0 W^T = Delta^T  (Tb = T diag(beta); S0 = bf16 copy of the state)
//   D4 = S0 Qr^T                  (inter-chunk part of the output)
//   D5 = Delta^T P^T              (P = tril(Q K^T) o Gamma with the norms folded in)
//   S += Delta'^T Kr              (Delta' = Delta diag(Gamma[C,.] r_k)), S pre-scaled by gamma_C
// The 64x64 triangular inverse runs on CUDA cores in fp32 (two 32x32 diagonal
// blocks by forward substitution, one column per lane, then the off-diagonal
// block as two 32x32 products).  Tokens past the end of a sequence are
// neutralised with beta = 0 and log g = 0 (they leave the state unchanged).
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace gdn {

namespace {

using namespace sm100;

constexpr int kC = 64;            // chunk length
constexpr int kThreads = 256;     // 8 warps; thread 0 issues TMA and MMA
constexpr int kCtasPerSm = 2;
constexpr int kAtStride = 72;     // fp32 row stride of A^T (row = column token i)
constexpr int kTStride = 68;      // fp32 row stride of T
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s

// Shared memory layout (offsets from a 1024-aligned base), sized so that two
// CTAs fit on one SM.  Buffers whose live ranges do not overlap share space:
//   scratch: A^T, T (fp32, triangular inverse) -> S0 (bf16 state copy, E2..D4)
//            -> Delta^T, Delta'^T (E3..D5/S) -> output tile (E4)
//   Tw, Tb (until D2/D3 complete) -> W^T (E2..D3b)
constexpr uint32_t kStageBytes = 49152;  // [Kr|Qr] x 2 K-blocks (32 KB) + V 2 blocks (16 KB)
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffScratch = kStageBytes;                      // 34 KB
constexpr uint32_t kScratchBytes = 64 * (kAtStride + kTStride) * 4;
constexpr uint32_t kOffS0 = kOffScratch;                           // 32 KB [128 vi][128 kk] K-major
constexpr uint32_t kOffDt = kOffScratch;                           // 16 KB [128 vi][64 t] K-major
constexpr uint32_t kOffDt2 = kOffScratch + 16384;                  // 16 KB
constexpr uint32_t kOffOut = kOffScratch;                          // 16 KB [64 t][128 vi] bf16
constexpr uint32_t kOffTw = kOffScratch + ((kScratchBytes + 1023) & ~1023u);  // 8 KB [64 t][64 t']
constexpr uint32_t kOffTb = kOffTw + 8192;                         // 8 KB
constexpr uint32_t kOffWt = kOffTw;                                // 16 KB [128 kk][64 t] MN-major
constexpr uint32_t kOffP = kOffTw + 16384;                         // 8 KB  [64 t][64 i] K-major
constexpr uint32_t kOffVec = kOffP + 8192;                         // per-token vectors
constexpr uint32_t kVecFloats = 11 * 64;
constexpr uint32_t kOffBar = kOffVec + kVecFloats * 4;
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;   // + alignment slack
static_assert(kScratchBytes >= 32768, "the A/T scratch must hold S0 and the Delta buffers");
static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");

// TMEM: 256 columns per CTA (two CTAs per SM).  Accumulators share the two
// 64-column slots X and Y by live range:  D1 (N = 128: K K^T | Q K^T and
// Q Q^T) uses X and Y; then D2 = W^T -> Y, D3 = Delta^T -> X, D4 -> Y,
// D5 -> X; the state S keeps columns [128, 256).
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColX = 0, kColY = 64;
constexpr uint32_t kColD1 = kColX, kColD2 = kColY, kColD3 = kColX, kColD4 = kColY, kColD5 = kColX,
                   kColS = 128;

struct ChunkParams {
    const float *a, *bl, *A_log, *dt_bias;
    const int32_t *offsets;
    const int32_t *seq_order;  // chunked sequences, longest first
    WsHeader *header;          // n_units, work counter, status
    const float *state_init;
    float *state_fin;
    __nv_bfloat16 *out;
    int B, N, H, HQ, V, VT;
    float scale;
    int tma_store;  // full output tiles leave through omap
    int opts;       // GDN_OPT_* rule / activation options
    // Segment-parallel mode for nseq_seg long sequences seg_seq[i], sequence i
    // cut into up to P_i = seg_s0[i+1] - seg_s0[i] segments (segments_of).
    // seg_mode 1: every segment but the last of each sequence from a zero
    // state, plus a 128-row tile starting from the identity with v = 0 whose
    // final state is the segment's transition M (S_end = S_start M + L);
    // writes M and the local final state L, no outputs.  seg_mode 2: every
    // segment from its true start state (seg_S), writing outputs; the last
    // segment writes state_fin.  A sequence's first start state is a copy of
    // its initial state, so state_fin may alias state_init.
    int seg_mode, nseq_seg, seg_units;
    int seg_seq[kMaxSegSeqs];
    int seg_m0[kMaxSegSeqs + 1];  // first phase-1 segment of each sequence (P_i - 1 each)
    int seg_s0[kMaxSegSeqs + 1];  // first segment of each sequence (P_i each)
    unsigned int *counter;        // work counter of this launch
    float *seg_M, *seg_L;  // [phase-1 segment][H][128][128], [phase-1 segment][H][V][128]
    const float *seg_S;    // [segment][H][V][128]: start states of the segments
    // Dense layout (DENSE3 kernels): three tensor maps in global memory over
    // q, k and v [B S, H n] (written by the packing kernel); key head = value head.
    const CUtensorMap *gmaps;
};

// Segment length of a sequence of len tokens cut into at most nseg segments
// (a multiple of the chunk) and the number of non-empty segments.
__device__ __forceinline__ void segments_of(int len, int nseg, int &seg_len, int &count) {
    static_assert(kC == 64, "segment_split rounds segments to the 64-token chunk");
    segment_split(len, nseg, seg_len, count);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Store 8 consecutive values (cols c8*8 .. c8*8+7 of `row`) as bf16 into a
// SW128 tile.
__device__ __forceinline__ void st_sw128_8(unsigned char *tile, int row, int c8, const float *v) {
    uint4 q;
    q.x = pack_bf16(v[0], v[1]);
    q.y = pack_bf16(v[2], v[3]);
    q.z = pack_bf16(v[4], v[5]);
    q.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, c8 * 8)) = q;
}

// TF32 operand of mma.sync: the fp32 bits as they are (the tensor core reads
// the top 19 bits, i.e. rounds toward zero; the explicit round-to-nearest
// conversion cost a dependent instruction per operand on the merge chain).
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x); }

// 2^x and log2(x) on the special-function unit.
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2f(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Plain non-coherent load issued where it stands (the value is consumed much later).
__device__ __forceinline__ float ld_nc_f32(const float *ptr) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

// 4-byte asynchronous global -> shared copy (this thread's group)
__device__ __forceinline__ void cp_async_4(float *smem_dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// log2 g_t and beta_t of one token from its logits (zero for padded tokens):
// log2 g = -exp(A_log) softplus(a + dt_bias) log2(e), beta = sigmoid(b), with
// the special-function-unit exponential and logarithm (this path computes in
// bf16 operands; their few-ulp error is far below that rounding).
// neg_ea_log2e = -exp(A_log) log2(e) of the head.  The rule options
// (GDN_OPT_*) give log2 g = 0 without decay, a log2(e) for the exp gate,
// beta = 1 without a rate input and beta = b for the raw rate.
__device__ __forceinline__ void chunk_gates(float a, float b, bool valid, float dt_bias,
                                            float neg_ea_log2e, int opts, float *lg,
                                            float *beta) {
    float l = 0.f, r = 1.f;
    if (!(opts & GDN_OPT_NO_DECAY)) {
        if (opts & GDN_OPT_GATE_EXP) {
            l = a * 1.4426950408889634f;
        } else {
            const float x = a + dt_bias;
            const float softplus = fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)));
            l = neg_ea_log2e * softplus;
        }
    }
    if (!(opts & GDN_OPT_NO_BETA)) r = (opts & GDN_OPT_BETA_RAW) ? b : __fdividef(1.f, 1.f + __expf(-b));
    *lg = valid ? l : 0.f;
    *beta = valid ? r : 0.f;
}

// f[lane] for a register array (a tree of selects on the lane bits, so the
// array is never indexed dynamically).
__device__ __forceinline__ float lane_pick(const float (&f)[32], int lane) {
    float a16[16], a8[8], a4[4], a2[2];
#pragma unroll
    for (int m = 0; m < 16; ++m) a16[m] = (lane & 1) ? f[2 * m + 1] : f[2 * m];
#pragma unroll
    for (int m = 0; m < 8; ++m) a8[m] = (lane & 2) ? a16[2 * m + 1] : a16[2 * m];
#pragma unroll
    for (int m = 0; m < 4; ++m) a4[m] = (lane & 4) ? a8[2 * m + 1] : a8[2 * m];
#pragma unroll
    for (int m = 0; m < 2; ++m) a2[m] = (lane & 8) ? a4[2 * m + 1] : a4[2 * m];
    return (lane & 16) ? a2[1] : a2[0];
}

__device__ __forceinline__ float warp_scan_incl(float v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
    }
    return v;
}

// c += a * b on a warp-level m16n8k8 TF32 tensor-core tile: a is the 16x8
// block with element (r, k) at ap[r * ARS + k * ACS], b the 8x8 block with
// element (k, n) at bp[k * BRS + n] (fp32 in shared memory).
template <int ARS, int ACS, int BRS>
__device__ __forceinline__ void mma_tf32_16x8x8(float (&c)[4], const float *ap, const float *bp,
                                                int g, int tg) {
    const uint32_t a0 = to_tf32(ap[g * ARS + tg * ACS]);
    const uint32_t a1 = to_tf32(ap[(g + 8) * ARS + tg * ACS]);
    const uint32_t a2 = to_tf32(ap[g * ARS + (tg + 4) * ACS]);
    const uint32_t a3 = to_tf32(ap[(g + 8) * ARS + (tg + 4) * ACS]);
    const uint32_t b0 = to_tf32(bp[tg * BRS + g]);
    const uint32_t b1 = to_tf32(bp[(tg + 4) * BRS + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Write rows (r0, r0 + 8), columns (c, c + 1) of Tw = T diag(ws) and
// Tb = T diag(beta) (bf16, 128-byte swizzled, K-major) from an MMA tile.
__device__ __forceinline__ void store_tw_tb(unsigned char *tw, unsigned char *tb, int r0, int c,
                                            const float (&d)[4], float2 ws, float2 be) {
    *reinterpret_cast<uint32_t *>(tw + sw128_offset(r0, c)) = pack_bf16(d[0] * ws.x, d[1] * ws.y);
    *reinterpret_cast<uint32_t *>(tw + sw128_offset(r0 + 8, c)) = pack_bf16(d[2] * ws.x, d[3] * ws.y);
    *reinterpret_cast<uint32_t *>(tb + sw128_offset(r0, c)) = pack_bf16(d[0] * be.x, d[1] * be.y);
    *reinterpret_cast<uint32_t *>(tb + sw128_offset(r0 + 8, c)) = pack_bf16(d[2] * be.x, d[3] * be.y);
}

// DENSE3: the q, k, v tiles come from three tensor maps in global memory
// (p.gmaps) over the dense layout's separate q, k, v tensors instead of the
// packed conv output (ymap).
template <bool DENSE3>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    chunked_delta_kernel(const __grid_constant__ CUtensorMap ymap,
                         const __grid_constant__ CUtensorMap omap, const ChunkParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // per-token vectors of the current chunk (log2 units for the decays):
    //   lg: log2 g_t, beta: beta_t, lb: sum_{s<=t} log2 g_s, ck: log2 r_k(t) - lb_t,
    //   fa: beta_t r_k(t), fp: scale r_q(t), ws: beta_t r_k(t) gamma_t,
    //   c: Gamma[C, t] r_k(t), s: scale r_q(t) gamma_t
    float *vec = reinterpret_cast<float *>(sm + kOffVec);
    float *v_lg = vec, *v_beta = vec + 64, *v_lb = vec + 128, *v_ck = vec + 192;
    float *v_fa = vec + 256, *v_fp = vec + 320, *v_ws = vec + 384, *v_c = vec + 448;
    float *v_s = vec + 512;
    float *v_na = vec + 576, *v_nb = vec + 640;  // gate logits of the next chunk (cp.async)
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(sm + kOffBar);  // [2]
    uint64_t *bar_mma = bar_full + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar_full + 3);
    int *s_unit = reinterpret_cast<int *>(bar_full + 4);
    int *s_abort = s_unit + 1;
    float *sAt = reinterpret_cast<float *>(sm + kOffScratch);         // A^T [64 i][kAtStride]
    float *sT = sAt + 64 * kAtStride;                                  // T [64 t][kTStride]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // TMEM access: warp w reads lane quadrant (w & 3); warps w and w + 4 split
    // the columns of an accumulator into halves hc = w >> 2.
    const int quad = warp & 3, hc = warp >> 2;
    const int row = quad * 32 + lane;  // this thread's TMEM lane (accumulator row)

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&ymap);
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);

    // everything below reads what the conv kernel wrote
    pdl_wait_primary();
    if constexpr (DENSE3) {
        if (tid == 0)
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                tensormap_acquire(p.gmaps + m);
                tma_prefetch_desc(p.gmaps + m);
            }
    }

    const int H = p.H, HQ = p.HQ, V = p.V;
    const int G = H / HQ;
    const int n_units = p.seg_mode ? p.seg_units : p.header->n_units;
    uint32_t gchunk = 0;      // chunks loaded by this CTA (parity of the stage barrier)
    uint32_t mma_phase = 0;   // completed MMA commits

    // D1 rows: lanes 0..63 hold k_t, lanes 64..127 hold q_t (t = token in chunk)
    const bool krow = row < 64;
    const int t_row = krow ? row : row - 64;
    // the warp whose 32 columns contain the diagonal of its 32 rows
    const bool diag_warp = (t_row >> 5) == hc;
    // the warp whose columns lie right of its rows' diagonal block (A: unused, P: zero)
    const bool upper_warp = hc == 1 && t_row < 32;

    auto wait_mma = [&]() {
        const bool ok = mbar_wait(bar_mma, mma_phase & 1, kWaitLimitNs);
        ++mma_phase;
        if (!ok) atomicExch(s_abort, 1);
        tc_fence_after();
    };
    auto sync_all = [&]() {  // thread barrier that orders TMEM/SMEM accesses with the MMA issuer
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    auto ld32f = [&](uint32_t col, float (&f)[32]) {
        uint32_t r[32];
        tmem_ld32(lane_base + col, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
    };

    while (true) {
        if (tid == 0) *s_unit = (int)atomicAdd(p.counter, 1u);
        __syncthreads();
        const int u = *s_unit;
        if (u >= n_units || *s_abort) break;
        int seq, h, vt, q = 0, seg = 0, nseg_here = 1;
        bool mtile = false;  // the transition tile of a segment (seg_mode 1)
        if (p.seg_mode == 0) {
            seq = p.seq_order[u / (H * p.VT)];
            h = (u / p.VT) % H;
            vt = u % p.VT;
        } else {
            // q: the segment's index among this launch's segments, numbering
            // the M / L (seg_mode 1) or start-state (seg_mode 2) buffers.
            // Constant indices only: a dynamic index into the parameter
            // arrays would copy them to local memory.
            const int tiles = p.VT + (p.seg_mode == 1);
            q = u / (H * tiles);
            h = (u / tiles) % H;
            const int tile = u % tiles;
            mtile = tile == p.VT;
            vt = mtile ? 0 : tile;
            seq = p.seg_seq[0];
            seg = q;
            nseg_here = p.seg_s0[1];
#pragma unroll
            for (int i = 1; i < kMaxSegSeqs; ++i) {
                const int f = p.seg_mode == 1 ? p.seg_m0[i] : p.seg_s0[i];
                if (i < p.nseq_seg && q >= f) {
                    seq = p.seg_seq[i];
                    seg = q - f;
                    nseg_here = p.seg_s0[i + 1] - p.seg_s0[i];
                }
            }
        }
        int s = p.offsets[seq], e = p.offsets[seq + 1];
        if (s < 0 || e < s || e > p.N) {
            // malformed offsets (the schedule lists no unit then; this guard
            // keeps every load and store inside [0, N) regardless)
            __syncthreads();  // every thread has read s_unit before thread 0 rewrites it
            continue;
        }
        if (p.seg_mode) {  // this segment's tokens (units past the sequence's last segment are empty)
            int seg_len;
            segments_of(e - s, nseg_here, seg_len, nseg_here);
            if (seg >= (p.seg_mode == 1 ? nseg_here - 1 : nseg_here)) {
                __syncthreads();  // every thread has read s_unit before thread 0 rewrites it
                continue;
            }
            s += seg * seg_len;
            e = min(e, s + seg_len);
        }
        const bool write_out = p.seg_mode != 1;
        const int nchunks = (e - s + kC - 1) / kC;
        const int kh = h / G;
        const int qcol = kh * 128, kcol = HQ * 128 + kh * 128;
        const int vcol = 2 * HQ * 128 + h * V + vt * 128;
        const size_t state_row = ((size_t)seq * H + h) * V + vt * 128 + row;
        const int opts = p.opts;
        const bool need_a = !(opts & GDN_OPT_NO_DECAY), need_b = !(opts & GDN_OPT_NO_BETA);
        const bool softplus_gate = need_a && !(opts & GDN_OPT_GATE_EXP);
        const float dtb = softplus_gate ? __ldg(p.dt_bias + h) : 0.f;
        const float neg_ea = softplus_gate ? -expf(__ldg(p.A_log + h)) * 1.4426950408889634f : 0.f;

        // state row `row`, columns [64 hc, 64 hc + 64) -> TMEM
        {
            const float *src = p.state_init + state_row * 128 + hc * 64;
            if (p.seg_mode == 2)
                src = p.seg_S + ((((size_t)q * H + h) * V + vt * 128 + row) * 128 + hc * 64);
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                if (p.seg_mode == 1) {  // zero, or the identity for the transition tile
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = __float_as_uint(mtile && row == hc * 64 + c0 + j ? 1.f : 0.f);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 f = *reinterpret_cast<const float4 *>(src + c0 + j);
                        r[j] = __float_as_uint(f.x);
                        r[j + 1] = __float_as_uint(f.y);
                        r[j + 2] = __float_as_uint(f.z);
                        r[j + 3] = __float_as_uint(f.w);
                    }
                }
                tmem_st32(lane_base + kColS + hc * 64 + c0, r);
            }
            tmem_wait_st();
        }

        auto issue_tma = [&](int n) {
            unsigned char *base = sm + kOffStage;
            const int t0 = s + n * kC;
            mbar_arrive_expect_tx(&bar_full[0], kStageBytes);
            if constexpr (DENSE3) {  // q, k, v [B S, H n] with n = 128: head h at column 128 h
                const CUtensorMap *qm = p.gmaps, *km = p.gmaps + 1, *vm = p.gmaps + 2;
                const int c = h * 128;
                tma_load_2d(base + 0, km, &bar_full[0], c, t0);
                tma_load_2d(base + 8192, qm, &bar_full[0], c, t0);
                tma_load_2d(base + 16384, km, &bar_full[0], c + 64, t0);
                tma_load_2d(base + 24576, qm, &bar_full[0], c + 64, t0);
                tma_load_2d(base + 32768, vm, &bar_full[0], c, t0);
                tma_load_2d(base + 40960, vm, &bar_full[0], c + 64, t0);
            } else {
                tma_load_2d(base + 0, &ymap, &bar_full[0], kcol, t0);
                tma_load_2d(base + 8192, &ymap, &bar_full[0], qcol, t0);
                tma_load_2d(base + 16384, &ymap, &bar_full[0], kcol + 64, t0);
                tma_load_2d(base + 24576, &ymap, &bar_full[0], qcol + 64, t0);
                tma_load_2d(base + 32768, &ymap, &bar_full[0], vcol, t0);
                tma_load_2d(base + 40960, &ymap, &bar_full[0], vcol + 64, t0);
            }
        };
        if (tid == 0) issue_tma(0);
        // gates of chunk 0 (threads 0..63); later chunks' gates are computed
        // during the previous chunk's state update
        float ga = 0.f, gbl = 0.f;
        if (tid < 64) {
            if (tid < e - s) {
                if (need_a) ga = ld_nc_f32(p.a + (size_t)(s + tid) * H + h);
                if (need_b) gbl = ld_nc_f32(p.bl + (size_t)(s + tid) * H + h);
            }
            chunk_gates(ga, gbl, tid < e - s, dtb, neg_ea, opts, v_lg + tid, v_beta + tid);
        }

#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const uint32_t full_parity = (gchunk + n) & 1;
            unsigned char *stage = sm + kOffStage;
            const uint32_t kq = smem_u32(stage), vb = kq + 32768;
            const int t0 = s + n * kC;
            const int Cn = min(kC, e - t0);

            if (!mbar_wait(&bar_full[0], full_parity, kWaitLimitNs)) atomicExch(s_abort, 1);
            __syncthreads();
            if (*s_abort) break;
            // the next chunk's gate logits -> shared memory, consumed by chunk_gates below
            if (tid < 64 && t0 + kC + tid < e) {
                if (need_a) cp_async_4(v_na + tid, p.a + (size_t)(t0 + kC + tid) * H + h);
                if (need_b) cp_async_4(v_nb + tid, p.bl + (size_t)(t0 + kC + tid) * H + h);
                cp_async_commit();
            }

            // ---- D1 = [K; Q] [K; Q]^T  (K K^T | K Q^T over Q K^T | Q Q^T)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(128, 128, false, false);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + kColD1, sdesc_sw128(kq + off, 16, 1024),
                             sdesc_sw128(kq + off, 16, 1024), idesc, ks > 0);
                }
                mma_commit(bar_mma);
            }
            wait_mma();

            // ---- E1a: norms from the diagonals, cumulative log2 decay, and the
            // per-token vectors built from them (four diagonal warps)
            float rq = 0.f;
            if (diag_warp && !krow) {
                float dq[32];
                ld32f(kColD1 + 64 + hc * 32, dq);
                rq = (opts & GDN_OPT_NO_QK_NORM) ? 1.f : rsqrtf(lane_pick(dq, lane) + 1e-12f);
            }
            float d1[32];  // columns [32 hc, 32 hc + 32) of K K^T (k rows) or Q K^T (q rows)
            if (!upper_warp) ld32f(kColD1 + hc * 32, d1);
            if (diag_warp) {
                const float lo = warp_scan_incl(v_lg[lane], lane);
                const float hi = warp_scan_incl(v_lg[32 + lane], lane) + __shfl_sync(0xffffffffu, lo, 31);
                const float lbC = __shfl_sync(0xffffffffu, hi, 31);
                const float lb = hc == 0 ? lo : hi;  // t_row = 32 hc + lane
                if (krow) {
                    const float rk = (opts & GDN_OPT_NO_QK_NORM) ? 1.f : rsqrtf(lane_pick(d1, lane) + 1e-12f);
                    const float ck = lg2f(rk) - lb;
                    const float be = v_beta[t_row];
                    // without retrieval A = 0 (T = I) and W = 0: Delta = diag(beta) V
                    const float fr = (opts & GDN_OPT_NO_RETRIEVE) ? 0.f : 1.f;
                    v_lb[t_row] = lb;
                    v_ck[t_row] = ck;
                    v_fa[t_row] = fr * be * rk;
                    v_ws[t_row] = fr * be * rk * ex2f(lb);
                    v_c[t_row] = ex2f(lbC + ck);
                } else {
                    v_fp[t_row] = p.scale * rq;
                    v_s[t_row] = p.scale * rq * ex2f(lb);
                }
            }
            if (tid == 0) bulk_wait_read();  // the output tile (scratch) is rewritten below
            __syncthreads();

            // ---- E1b: A[t,i] = beta_t r_k(t) r_k(i) Gamma[t,i] k_t.k_i (i < t), fp32, stored transposed;
            //           P[t,i] = scale r_q(t) r_k(i) Gamma[t,i] q_t.k_i (i <= t), bf16;
            // with r_k(i) Gamma[t,i] = 2^(lb_t + ck_i)
            if (!upper_warp) {
                const float ft = krow ? v_fa[t_row] : v_fp[t_row];
                const float lbt = v_lb[t_row];
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float ck8[8], o[8];
                    *reinterpret_cast<float4 *>(ck8) = *reinterpret_cast<const float4 *>(v_ck + hc * 32 + c8 * 8);
                    *reinterpret_cast<float4 *>(ck8 + 4) = *reinterpret_cast<const float4 *>(v_ck + hc * 32 + c8 * 8 + 4);
#pragma unroll
                    for (int u2 = 0; u2 < 8; ++u2) {
                        const int j = c8 * 8 + u2;  // column token 32 hc + j; the row's is 32 hc + lane
                        o[u2] = ft * ex2f(lbt + ck8[u2]) * d1[j];
                        if (diag_warp) o[u2] = (krow ? j < lane : j <= lane) ? o[u2] : 0.f;
                    }
                    if (krow) {  // A^T[i][t]: the 32 lanes write 32 consecutive words
                        float *acol = sAt + (hc * 32 + c8 * 8) * kAtStride + t_row;
#pragma unroll
                        for (int u2 = 0; u2 < 8; ++u2) acol[u2 * kAtStride] = o[u2];
                    } else {
                        st_sw128_8(sm + kOffP, t_row, hc * 4 + c8, o);
                    }
                }
            } else if (!krow) {  // P[t, i] = 0 for t < 32 <= i
                const float z8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_sw128_8(sm + kOffP, t_row, 4 + c8, z8);
            }
            __syncthreads();

            // ---- T = (I + A)^-1 (lower unit-triangular) from 16x16 blocks T_ij:
            // step 1: diagonal blocks by right-looking forward substitution, one
            //   column per lane (warps 0, 1); warps 6, 7 zero the upper blocks of Tw, Tb;
            // step 2: T_10 = -T_11 (A_10 T_00) and T_32 = -T_33 (A_32 T_22) on TF32
            //   tensor-core tiles (warps 0..3); warps 4..7 write Tw, Tb of the diagonal blocks;
            // step 3: T[32:64, 0:32] = -T2 (A[32:64, 0:32] T1) with T1, T2 the two 32x32
            //   diagonal blocks (all warps).
            // Tw = T diag(beta r_k gamma) and Tb = T diag(beta) are the bf16 MMA operands.
            unsigned char *twp = sm + kOffTw, *tbp = sm + kOffTb;
            const int g = lane >> 2, tg = lane & 3;
            if (warp < 2) {
                const int blk = warp * 2 + (lane >> 4), c = lane & 15, base = blk * 16;
                // column i of the block (A[base + r][base + i], r > i) is row i of A^T
                // (loaded right before its use: prefetching one step ahead costs
                // registers that the rest of the loop spills for)
                auto load_col = [&](int i, float (&av)[16]) {
                    const float *acol = sAt + (base + i) * kAtStride + base;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        if (4 * q4 + 3 > i) {
                            const float4 x4 = *reinterpret_cast<const float4 *>(acol + 4 * q4);
                            av[4 * q4] = x4.x;
                            av[4 * q4 + 1] = x4.y;
                            av[4 * q4 + 2] = x4.z;
                            av[4 * q4 + 3] = x4.w;
                        }
                    }
                };
                float pr[16], tc[16], av0[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) pr[r] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (i < 15) load_col(i, av0);
                    tc[i] = (i == c) ? 1.f : (i > c ? -pr[i] : 0.f);
#pragma unroll
                    for (int r = i + 1; r < 16; ++r) pr[r] = fmaf(av0[r], tc[i], pr[r]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) sT[(base + r) * kTStride + base + c] = tc[r];
            } else if (warp >= 6) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int q = tid - 192; q < 2 * 192; q += 64) {
                    const int r = q % 192;
                    int rr, c8;
                    if (r < 96) {
                        rr = r / 6;
                        c8 = 2 + r % 6;
                    } else if (r < 160) {
                        rr = 16 + (r - 96) / 4;
                        c8 = 4 + (r - 96) % 4;
                    } else {
                        rr = 32 + (r - 160) / 2;
                        c8 = 6 + (r - 160) % 2;
                    }
                    *reinterpret_cast<uint4 *>((q < 192 ? twp : tbp) + sw128_offset(rr, c8 * 8)) = z;
                }
            }
            __syncthreads();
            if (warp < 4) {
                const int lo = (warp >> 1) * 32, hi = lo + 16, n0 = lo + (warp & 1) * 8;
                float *xs = sT + (warp >> 1) * 16 * kTStride + 32 + (warp & 1) * 8;  // unused upper block
                float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k0 = 0; k0 < 16; k0 += 8)  // X = A[hi, lo] T[lo, lo]
                    mma_tf32_16x8x8<1, kAtStride, kTStride>(x, sAt + (lo + k0) * kAtStride + hi,
                                                            sT + (lo + k0) * kTStride + n0, g, tg);
                *reinterpret_cast<float2 *>(xs + g * kTStride + 2 * tg) = make_float2(x[0], x[1]);
                *reinterpret_cast<float2 *>(xs + (g + 8) * kTStride + 2 * tg) = make_float2(x[2], x[3]);
                __syncwarp();
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k0 = 0; k0 < 16; k0 += 8)  // T[hi, lo] = -T[hi, hi] X
                    mma_tf32_16x8x8<kTStride, 1, kTStride>(d, sT + hi * kTStride + hi + k0,
                                                           xs + k0 * kTStride, g, tg);
#pragma unroll
                for (int u2 = 0; u2 < 4; ++u2) d[u2] = -d[u2];
                const int r0 = hi + g, cc = n0 + 2 * tg;
                *reinterpret_cast<float2 *>(sT + r0 * kTStride + cc) = make_float2(d[0], d[1]);
                *reinterpret_cast<float2 *>(sT + (r0 + 8) * kTStride + cc) = make_float2(d[2], d[3]);
                store_tw_tb(twp, tbp, r0, cc, d, *reinterpret_cast<const float2 *>(v_ws + cc),
                            *reinterpret_cast<const float2 *>(v_beta + cc));
            } else {  // diagonal blocks: 4 blocks x 16 rows x 2 column halves, one per thread
                const int q = tid - 128;
                const int blk = q >> 5, rr = blk * 16 + ((q >> 1) & 15), c0 = blk * 16 + (q & 1) * 8;
                float t8[8], ws8[8], be8[8], w8[8], b8[8];
                *reinterpret_cast<float4 *>(t8) = *reinterpret_cast<const float4 *>(sT + rr * kTStride + c0);
                *reinterpret_cast<float4 *>(t8 + 4) = *reinterpret_cast<const float4 *>(sT + rr * kTStride + c0 + 4);
                *reinterpret_cast<float4 *>(ws8) = *reinterpret_cast<const float4 *>(v_ws + c0);
                *reinterpret_cast<float4 *>(ws8 + 4) = *reinterpret_cast<const float4 *>(v_ws + c0 + 4);
                *reinterpret_cast<float4 *>(be8) = *reinterpret_cast<const float4 *>(v_beta + c0);
                *reinterpret_cast<float4 *>(be8 + 4) = *reinterpret_cast<const float4 *>(v_beta + c0 + 4);
#pragma unroll
                for (int u2 = 0; u2 < 8; ++u2) {
                    w8[u2] = t8[u2] * ws8[u2];
                    b8[u2] = t8[u2] * be8[u2];
                }
                st_sw128_8(twp, rr, c0 >> 3, w8);
                st_sw128_8(tbp, rr, c0 >> 3, b8);
            }
            __syncthreads();
            {
                const int ni = warp & 3, mi = warp >> 2, c0 = ni * 8;
                // X2 = A[32:64, 0:32] T1 (columns c0..c0+7; T1[k][c] = 0 for k < c0),
                // rows 0 .. 16 mi + 15, into a scratch block T does not need any more
                float *xs = mi ? sT + 32 + c0 : sT + 32 * kTStride + c0;
#pragma unroll
                for (int m2 = 0; m2 < 2; ++m2) {
                    if (m2 > mi) break;
                    float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k0 = 0; k0 < 32; k0 += 8)
                        if (k0 >= c0)
                            mma_tf32_16x8x8<1, kAtStride, kTStride>(x, sAt + k0 * kAtStride + 32 + 16 * m2,
                                                                    sT + k0 * kTStride + c0, g, tg);
                    float *xr = xs + 16 * m2 * kTStride;
                    *reinterpret_cast<float2 *>(xr + g * kTStride + 2 * tg) = make_float2(x[0], x[1]);
                    *reinterpret_cast<float2 *>(xr + (g + 8) * kTStride + 2 * tg) = make_float2(x[2], x[3]);
                }
                __syncwarp();
                // T[32 + 16 mi + r][c0 + n] = -sum_k T2[16 mi + r][k] X2[k][n], k < 16 mi + 16
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                const float *t2 = sT + (32 + 16 * mi) * kTStride + 32;
#pragma unroll
                for (int k0 = 0; k0 < 32; k0 += 8)
                    if (k0 < 16 * mi + 16)
                        mma_tf32_16x8x8<kTStride, 1, kTStride>(d, t2 + k0, xs + k0 * kTStride, g, tg);
#pragma unroll
                for (int u2 = 0; u2 < 4; ++u2) d[u2] = -d[u2];
                const int cc = c0 + 2 * tg;
                store_tw_tb(twp, tbp, 32 + 16 * mi + g, cc, d, *reinterpret_cast<const float2 *>(v_ws + cc),
                            *reinterpret_cast<const float2 *>(v_beta + cc));
            }
            fence_async_smem();
            sync_all();

            // ---- D2 = K^T Tw^T (= W^T), D3 = V^T Tb^T
            if (tid == 0) {
                const uint32_t id = idesc_bf16(128, 64, true, false);
                const uint32_t tw = smem_u32(sm + kOffTw), tb = smem_u32(sm + kOffTb);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColD2, sdesc_sw128(kq + ks * 2048, 16384, 1024),
                             sdesc_sw128(tw + ks * 32, 16, 1024), id, ks > 0);
                if (!mtile)  // the transition tile has v = 0: Delta = -W S0^T only
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem + kColD3, sdesc_sw128(vb + ks * 2048, 8192, 1024),
                                 sdesc_sw128(tb + ks * 32, 16, 1024), id, ks > 0);
                mma_commit(bar_mma);
            }
            wait_mma();

            // ---- E2: W^T -> bf16 (MN-major B operand); S -> bf16 S0; S *= gamma_C
            {
                float f[32];
                ld32f(kColD2 + hc * 32, f);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_sw128_8(sm + kOffWt, row, hc * 4 + c8, f + c8 * 8);
                const float gC = ex2f(v_lb[63]);
                unsigned char *s0 = sm + kOffS0 + hc * 16384;  // this half is one K-block
                // (rolled loops here and in E4 keep the kernel under 128 registers
                // with fewer spills)
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + kColS + hc * 64 + c0, r);
                    tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) st_sw128_8(s0, row, (c0 >> 3) + c8, v + c8 * 8);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j] * gC);
                    tmem_st32(lane_base + kColS + hc * 64 + c0, r);
                }
                tmem_wait_st();
            }
            fence_async_smem();
            sync_all();

            // ---- D3 -= S0 W^T ;  D4 = S0 Q^T
            if (tid == 0) {
                const uint32_t s0 = smem_u32(sm + kOffS0), wt = smem_u32(sm + kOffWt);
                const uint32_t idn = idesc_bf16(128, 64, false, true, true);
                const uint32_t idq = idesc_bf16(128, 64, false, false);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + kColD3, sdesc_sw128(s0 + aoff, 16, 1024),
                             sdesc_sw128(wt + ks * 2048, 8192, 1024), idn, !(mtile && ks == 0));
                }
                if (write_out)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16(tmem + kColD4, sdesc_sw128(s0 + aoff, 16, 1024),
                                 sdesc_sw128(kq + 8192 + aoff, 16, 1024), idq, ks > 0);
                    }
                mma_commit(bar_mma);
            }
            // gates of the next chunk while the MMAs run (this chunk is done with them)
            if (tid < 64 && n + 1 < nchunks) {
                const bool valid = t0 + kC + tid < e;
                cp_async_wait_all();
                chunk_gates(valid && need_a ? v_na[tid] : 0.f, valid && need_b ? v_nb[tid] : 0.f,
                            valid, dtb, neg_ea, opts, v_lg + tid, v_beta + tid);
            }
            wait_mma();

            // ---- E3: Delta^T and Delta'^T = Delta^T diag(c) -> bf16 (K-major A operands)
            {
                float f[32];
                ld32f(kColD3 + hc * 32, f);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float w8[8];
#pragma unroll
                    for (int u2 = 0; u2 < 8; ++u2) w8[u2] = f[c8 * 8 + u2] * v_c[hc * 32 + c8 * 8 + u2];
                    st_sw128_8(sm + kOffDt, row, hc * 4 + c8, f + c8 * 8);
                    st_sw128_8(sm + kOffDt2, row, hc * 4 + c8, w8);
                }
            }
            fence_async_smem();
            sync_all();

            // ---- D5 = Delta^T P^T ;  S += Delta'^T K
            if (tid == 0) {
                const uint32_t dt = smem_u32(sm + kOffDt), dt2 = smem_u32(sm + kOffDt2);
                const uint32_t pp = smem_u32(sm + kOffP);
                const uint32_t id5 = idesc_bf16(128, 64, false, false);
                const uint32_t id6 = idesc_bf16(128, 128, false, true);
                if (write_out)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem + kColD5, sdesc_sw128(dt + ks * 32, 16, 1024),
                                 sdesc_sw128(pp + ks * 32, 16, 1024), id5, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColS, sdesc_sw128(dt2 + ks * 32, 16, 1024),
                             sdesc_sw128(kq + ks * 2048, 16384, 1024), id6, 1);
                mma_commit(bar_mma);
            }
            wait_mma();
            // the stage is free: load the next chunk while the outputs are written
            if (tid == 0 && n + 1 < nchunks) issue_tma(n + 1);

            // ---- E4: o[vi, t] = s_t (S0 Q^T)[vi, t] + (Delta^T P^T)[vi, t], staged as a
            // [64 t][128 vi] bf16 tile in the (now free) Delta buffers, then written
            // as 16-byte rows
            if (write_out)
            {
                __nv_bfloat16 *otile = reinterpret_cast<__nv_bfloat16 *>(sm + kOffOut);
#pragma unroll 1
                for (int c16 = 0; c16 < 2; ++c16) {
                    uint32_t r4[16], r5[16];
                    tmem_ld16(lane_base + kColD4 + hc * 32 + c16 * 16, r4);
                    tmem_ld16(lane_base + kColD5 + hc * 32 + c16 * 16, r5);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const int tt = hc * 32 + c16 * 16 + j;
                        const float4 s4 = *reinterpret_cast<const float4 *>(v_s + tt);
                        const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                        for (int u2 = 0; u2 < 4; ++u2)
                            otile[(tt + u2) * 128 + row] = __float2bfloat16_rn(
                                fmaf(sv[u2], __uint_as_float(r4[j + u2]), __uint_as_float(r5[j + u2])));
                    }
                }
                if (p.tma_store && Cn == kC) {  // a full tile: one bulk store
                    fence_async_smem();
                    __syncthreads();
                    if (tid == 0) {
                        tma_store_2d(&omap, otile, h * V + vt * 128, t0);
                        bulk_commit();
                    }
                } else {  // the last, ragged tile of a sequence: rows t < Cn only
                    __syncthreads();
                    __nv_bfloat16 *obase = p.out + (size_t)t0 * H * V + (size_t)h * V + vt * 128;
                    for (int q = tid; q < Cn * 16; q += kThreads) {
                        const int t = q >> 4, c16 = q & 15;
                        *reinterpret_cast<uint4 *>(obase + (size_t)t * H * V + c16 * 8) =
                            *reinterpret_cast<const uint4 *>(otile + t * 128 + c16 * 8);
                    }
                }
            }
            sync_all();
        }
        gchunk += nchunks;
        if (*s_abort) break;

        // final state row `row`, columns [64 hc, 64 hc + 64) -> global
        if (p.seg_mode != 2 || seg == nseg_here - 1) {
            float *dst = p.state_fin + state_row * 128 + hc * 64;
            if (p.seg_mode == 1)
                dst = mtile ? p.seg_M + ((((size_t)q * H + h) * 128 + row) * 128 + hc * 64)
                            : p.seg_L + ((((size_t)q * H + h) * V + vt * 128 + row) * 128 + hc * 64);
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_base + kColS + hc * 64 + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + c0 + j) =
                        make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                    __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
            }
        }
        sync_all();
    }

    if (*s_abort) {
        // a bounded wait gave up: record it and give in-flight copies time to
        // land before the shared memory is released
        if (tid == 0) {
            atomicExch(&p.header->status, 7 /* GDN_ERR_TIMEOUT */);
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 10000000ull) {  // 10 ms
            }
        }
    }
    if (tid == 0) bulk_wait_all();
    sync_all();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

bool chunked_supported(int dtype, int K, int V, int W) {
    return dtype == 1 && K == 128 && V % 128 == 0 && W % 8 == 0;
}

namespace {

}  // namespace

// Operand map of a bf16 row-major matrix [rows, cols] read in [64 x box_rows]
// tiles with the 128-byte swizzle the chunked kernel's MMA descriptors expect.
// (box_rows: rows of the box, 64 by default.)
bool encode_operand_map(CUtensorMap *map, const void *base, long rows, long cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Tensor maps and kernel parameters of a chunked launch.
cudaError_t chunk_setup(const ChunkLaunch &c, CUtensorMap &map, CUtensorMap &omap, ChunkParams &p) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint32_t es[2] = {1, 1};
    // the packed conv output [N, W]; with the dense layout (c.gmaps) the kernel
    // reads its three maps from global memory and this parameter is unused
    if (c.gmaps == nullptr ? !encode_operand_map(&map, c.y, c.N, c.W)
                           : !encode_operand_map(&map, c.out, c.N, (long)c.H * c.V))
        return cudaErrorInvalidValue;
    // output tiles [64 t][128 vi] of out viewed as [N, H V] (no swizzle)
    int tma_store = 0;
    if ((reinterpret_cast<uintptr_t>(c.out) & 15) == 0 && c.N > 0) {
        const cuuint64_t odims[2] = {(cuuint64_t)c.H * c.V, (cuuint64_t)c.N};
        const cuuint64_t ostrides[1] = {(cuuint64_t)c.H * c.V * 2};
        const cuuint32_t obox[2] = {128, 64};
        tma_store = enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.out, odims, ostrides, obox, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if (!tma_store) omap = map;  // unused
    p = ChunkParams{};
    p.a = c.a; p.bl = c.bl; p.A_log = c.A_log; p.dt_bias = c.dt_bias;
    p.offsets = c.offsets; p.seq_order = c.seq_order; p.header = c.header;
    p.state_init = c.state_init; p.state_fin = c.state_fin;
    p.out = static_cast<__nv_bfloat16 *>(c.out);
    p.B = c.B; p.N = c.N; p.H = c.H; p.HQ = c.HQ; p.V = c.V; p.VT = c.V / 128;
    p.scale = c.scale;
    p.tma_store = tma_store;
    p.opts = c.opts;
    p.counter = &c.header->next_unit;
    p.gmaps = static_cast<const CUtensorMap *>(c.gmaps);
    static std::atomic<uint64_t> attr_set{0};
    return once_per_device(attr_set, [] {
        cudaError_t e = cudaFuncSetAttribute(chunked_delta_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(chunked_delta_kernel<true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    });
}

cudaError_t chunk_launch(const CUtensorMap &map, const CUtensorMap &omap, const ChunkParams &p,
                         long units, cudaStream_t s) {
    const long slots = (long)sm_count() * kCtasPerSm;
    const int grid = (int)(units < slots ? units : slots);
    if (grid <= 0) return cudaSuccess;
    cudaError_t e = p.gmaps != nullptr
                        ? launch_kernel(chunked_delta_kernel<true>, dim3(grid), dim3(kThreads),
                                        kSmemBytes, s, true, map, omap, p)
                        : launch_kernel(chunked_delta_kernel<false>, dim3(grid), dim3(kThreads),
                                        kSmemBytes, s, true, map, omap, p);
    note_launch();
    return e;
}

// Start states of the segments of each segmented sequence i (seg_seq[i]):
// S_0 = state_init, S_{j+1} = S_j M_j + L_j (rows of S independent), written
// to seg_S.  One block per (sequence, value head, 32 state rows), one thread
// per state column.
__global__ void __launch_bounds__(128) segment_combine_kernel(const ChunkParams p) {
    pdl_wait_primary();  // M and L come from the previous (phase 1) launch
    __shared__ float srow[32][128];
    const int V = p.V, H = p.H, nrb = V / 32;
    const int sidx = blockIdx.x / (H * nrb);
    const int h = (blockIdx.x / nrb) % H, r0 = (blockIdx.x % nrb) * 32, j = threadIdx.x;
    const int seq = p.seg_seq[sidx];
    int seg_len, count;
    segments_of(p.offsets[seq + 1] - p.offsets[seq], p.seg_s0[sidx + 1] - p.seg_s0[sidx], seg_len,
                count);
    float *S = const_cast<float *>(p.seg_S) + (size_t)p.seg_s0[sidx] * H * V * 128;
    for (int r = 0; r < 32; ++r) {
        const float x = p.state_init[(((size_t)seq * H + h) * V + r0 + r) * 128 + j];
        srow[r][j] = x;
        S[(((size_t)h) * V + r0 + r) * 128 + j] = x;
    }
    __syncthreads();
    for (int q = 0; q + 1 < count; ++q) {
        const size_t sq = (size_t)p.seg_m0[sidx] + q;
        float acc[32];
        const float *L = p.seg_L + ((sq * H + h) * V + r0) * 128 + j;
#pragma unroll
        for (int r = 0; r < 32; ++r) acc[r] = L[(size_t)r * 128];
        const float *M = p.seg_M + (sq * H + h) * 128 * 128 + j;
#pragma unroll 4
        for (int k = 0; k < 128; ++k) {
            const float m = M[(size_t)k * 128];
#pragma unroll
            for (int r = 0; r < 32; ++r) acc[r] = fmaf(srow[r][k], m, acc[r]);
        }
        __syncthreads();
        float *dst = S + (((size_t)(q + 1) * H + h) * V + r0) * 128 + j;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            srow[r][j] = acc[r];
            dst[(size_t)r * 128] = acc[r];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_delta_chunked(const ChunkLaunch &c, cudaStream_t s) {
    CUtensorMap map, omap;
    ChunkParams p;
    cudaError_t e = chunk_setup(c, map, omap, p);
    if (e != cudaSuccess) return e;
    return chunk_launch(map, omap, p, c.max_units, s);
}

cudaError_t launch_segment_combine(const ChunkLaunch &c, cudaStream_t s) {
    if (c.nseq_seg < 1 || c.nseq_seg > kMaxSegSeqs) return cudaErrorInvalidValue;
    ChunkParams p{};
    p.offsets = c.offsets;
    p.state_init = c.state_init;
    p.H = c.H;
    p.V = c.V;
    p.nseq_seg = c.nseq_seg;
    for (int i = 0; i < kMaxSegSeqs; ++i) p.seg_seq[i] = c.seg_seq[i];
    for (int i = 0; i <= kMaxSegSeqs; ++i) {
        p.seg_m0[i] = c.seg_m0[i];
        p.seg_s0[i] = c.seg_s0[i];
    }
    p.seg_M = c.seg_M;
    p.seg_L = c.seg_L;
    p.seg_S = c.seg_S;
    cudaError_t e = launch_kernel(segment_combine_kernel, dim3((unsigned)(c.nseq_seg * c.H * (c.V / 32))),
                                  dim3(128), 0, s, true, p);
    note_launch();
    return e;
}

// c.nseq_seg long chunked sequences (c.seg_seq), sequence i cut into up to
// c.seg_s0[i+1] - c.seg_s0[i] segments: phase 1 computes each segment's
// transition M and local final state L from a zero start (all but the last
// segment of every sequence, in parallel), the combine kernel chains the start
// states S_{j+1} = S_j M_j + L_j, and phase 2 reruns every segment from its
// start state (in parallel), writing the outputs.
cudaError_t launch_delta_chunked_segmented(const ChunkLaunch &c, cudaStream_t s) {
    CUtensorMap map, omap;
    ChunkParams p;
    cudaError_t e = chunk_setup(c, map, omap, p);
    if (e != cudaSuccess) return e;
    if (c.nseq_seg < 1 || c.nseq_seg > kMaxSegSeqs) return cudaErrorInvalidValue;
    const int VT = c.V / 128;
    p.nseq_seg = c.nseq_seg;
    for (int i = 0; i < kMaxSegSeqs; ++i) p.seg_seq[i] = c.seg_seq[i];
    for (int i = 0; i <= kMaxSegSeqs; ++i) {
        p.seg_m0[i] = c.seg_m0[i];
        p.seg_s0[i] = c.seg_s0[i];
    }
    p.seg_M = c.seg_M;
    p.seg_L = c.seg_L;
    p.seg_S = c.seg_S;
    p.seg_mode = 1;
    p.seg_units = c.seg_m0[c.nseq_seg] * c.H * (VT + 1);
    p.counter = &c.header->seg_next[0];
    e = chunk_launch(map, omap, p, p.seg_units, s);
    if (e != cudaSuccess) return e;
    e = launch_kernel(segment_combine_kernel, dim3((unsigned)(c.nseq_seg * c.H * (c.V / 32))),
                      dim3(128), 0, s, true, p);
    note_launch();
    if (e != cudaSuccess) return e;
    p.seg_mode = 2;
    p.seg_units = c.seg_s0[c.nseq_seg] * c.H * VT;
    p.counter = &c.header->seg_next[1];
    return chunk_launch(map, omap, p, p.seg_units, s);
}

}  // namespace gdn
