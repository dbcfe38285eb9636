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
constexpr int kAStride = 68;      // fp32 row stride of the A / T scratch (bank-conflict free)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s

// Shared memory layout (offsets from a 1024-aligned base), sized so that two
// CTAs fit on one SM.  Buffers whose live ranges do not overlap share space:
//   scratch: A, T (fp32, triangular inverse) -> S0 (bf16 state copy, E2..D4)
//            -> Delta^T, Delta'^T (E3..D5/S) -> output tile (E4)
//   Tw, Tb (until D2/D3 complete) -> W^T (E2..D3b)
constexpr uint32_t kStageBytes = 49152;  // [Kr|Qr] x 2 K-blocks (32 KB) + V 2 blocks (16 KB)
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffScratch = kStageBytes;                      // 34 KB
constexpr uint32_t kScratchBytes = 2 * 64 * kAStride * 4;
constexpr uint32_t kOffS0 = kOffScratch;                           // 32 KB [128 vi][128 kk] K-major
constexpr uint32_t kOffDt = kOffScratch;                           // 16 KB [128 vi][64 t] K-major
constexpr uint32_t kOffDt2 = kOffScratch + 16384;                  // 16 KB
constexpr uint32_t kOffOut = kOffScratch;                          // 16 KB [64 t][128 vi] bf16
constexpr uint32_t kOffTw = kOffScratch + ((kScratchBytes + 1023) & ~1023u);  // 8 KB [64 t][64 t']
constexpr uint32_t kOffTb = kOffTw + 8192;                         // 8 KB
constexpr uint32_t kOffWt = kOffTw;                                // 16 KB [128 kk][64 t] MN-major
constexpr uint32_t kOffP = kOffTw + 16384;                         // 8 KB  [64 t][64 i] K-major
constexpr uint32_t kOffVec = kOffP + 8192;                         // per-token vectors
constexpr uint32_t kVecFloats = 7 * 64;
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
};

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

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// One warp: C[16 x 8] tile at (m0, n0) of sgn * (a[:, 0:kd] * b[0:kd, :]) with
// warp-level m16n8k8 TF32 tensor-core MMAs; a, b, dst are fp32 row-major
// with row stride kAStride.  Used for the merges of the triangular inverse.
__device__ __forceinline__ void warp_tile_product(const float *a, const float *b, float *dst,
                                                  int m0, int n0, int kd, float sgn, int lane) {
    const int g = lane >> 2, tg = lane & 3;
    float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
    for (int k0 = 0; k0 < kd; k0 += 8) {
        const uint32_t a0 = to_tf32(a[(m0 + g) * kAStride + k0 + tg]);
        const uint32_t a1 = to_tf32(a[(m0 + g + 8) * kAStride + k0 + tg]);
        const uint32_t a2 = to_tf32(a[(m0 + g) * kAStride + k0 + tg + 4]);
        const uint32_t a3 = to_tf32(a[(m0 + g + 8) * kAStride + k0 + tg + 4]);
        const uint32_t b0 = to_tf32(b[(k0 + tg) * kAStride + n0 + g]);
        const uint32_t b1 = to_tf32(b[(k0 + tg + 4) * kAStride + n0 + g]);
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    *reinterpret_cast<float2 *>(dst + (m0 + g) * kAStride + n0 + 2 * tg) = make_float2(sgn * c0, sgn * c1);
    *reinterpret_cast<float2 *>(dst + (m0 + g + 8) * kAStride + n0 + 2 * tg) =
        make_float2(sgn * c2, sgn * c3);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    chunked_delta_kernel(const __grid_constant__ CUtensorMap ymap, const ChunkParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *vec = reinterpret_cast<float *>(sm + kOffVec);
    float *v_rq = vec, *v_rk = vec + 64, *v_beta = vec + 128, *v_lg = vec + 192;
    float *v_b = vec + 256, *v_gam = vec + 320, *v_c = vec + 384;
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(sm + kOffBar);  // [2]
    uint64_t *bar_mma = bar_full + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar_full + 3);
    int *s_unit = reinterpret_cast<int *>(bar_full + 4);
    int *s_abort = s_unit + 1;
    float *sA = reinterpret_cast<float *>(sm + kOffScratch);          // [64][kAStride]
    float *sT = sA + 64 * kAStride;                                    // [64][kAStride]

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

    const int H = p.H, HQ = p.HQ, V = p.V;
    const int G = H / HQ;
    const int n_units = p.header->n_units;
    uint32_t gchunk = 0;      // chunks loaded by this CTA (parity of the stage barrier)
    uint32_t mma_phase = 0;   // completed MMA commits

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
        if (tid == 0) *s_unit = (int)atomicAdd(&p.header->next_unit, 1u);
        __syncthreads();
        const int u = *s_unit;
        if (u >= n_units || *s_abort) break;
        const int seq = p.seq_order[u / (H * p.VT)];
        const int h = (u / p.VT) % H;
        const int vt = u % p.VT;
        const int s = p.offsets[seq], e = p.offsets[seq + 1];
        const int nchunks = (e - s + kC - 1) / kC;
        const int kh = h / G;
        const int qcol = kh * 128, kcol = HQ * 128 + kh * 128;
        const int vcol = 2 * HQ * 128 + h * V + vt * 128;
        const float A_log = __ldg(p.A_log + h), dtb = __ldg(p.dt_bias + h);
        const size_t state_row = ((size_t)seq * H + h) * V + vt * 128 + row;

        // state row `row`, columns [64 hc, 64 hc + 64) -> TMEM
        {
            const float *src = p.state_init + state_row * 128 + hc * 64;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 f = *reinterpret_cast<const float4 *>(src + c0 + j);
                    r[j] = __float_as_uint(f.x);
                    r[j + 1] = __float_as_uint(f.y);
                    r[j + 2] = __float_as_uint(f.z);
                    r[j + 3] = __float_as_uint(f.w);
                }
                tmem_st32(lane_base + kColS + hc * 64 + c0, r);
            }
            tmem_wait_st();
        }

        auto issue_tma = [&](int n) {
            unsigned char *base = sm + kOffStage;
            const int t0 = s + n * kC;
            mbar_arrive_expect_tx(&bar_full[0], kStageBytes);
            tma_load_2d(base + 0, &ymap, &bar_full[0], kcol, t0);
            tma_load_2d(base + 8192, &ymap, &bar_full[0], qcol, t0);
            tma_load_2d(base + 16384, &ymap, &bar_full[0], kcol + 64, t0);
            tma_load_2d(base + 24576, &ymap, &bar_full[0], qcol + 64, t0);
            tma_load_2d(base + 32768, &ymap, &bar_full[0], vcol, t0);
            tma_load_2d(base + 40960, &ymap, &bar_full[0], vcol + 64, t0);
        };
        if (tid == 0) issue_tma(0);
        // gate logits of the current chunk, loaded one chunk ahead
        float ga = 0.f, gbl = 0.f;
        if (tid < 64 && tid < e - s) {
            ga = __ldg(p.a + (size_t)(s + tid) * H + h);
            gbl = __ldg(p.bl + (size_t)(s + tid) * H + h);
        }

#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const uint32_t full_parity = (gchunk + n) & 1;
            unsigned char *stage = sm + kOffStage;
            const uint32_t kq = smem_u32(stage), vb = kq + 32768;
            const int t0 = s + n * kC;
            const int Cn = min(kC, e - t0);

            // per-token gates (threads 0..63) while the tiles land
            if (tid < 64) {
                float lg = 0.f, beta = 0.f;
                if (tid < Cn) {
                    lg = log_decay(ga, dtb, A_log);
                    beta = 1.f / (1.f + expf(-gbl));
                }
                v_lg[tid] = lg;
                v_beta[tid] = beta;
                ga = gbl = 0.f;
                if (t0 + kC + tid < e) {
                    ga = __ldg(p.a + (size_t)(t0 + kC + tid) * H + h);
                    gbl = __ldg(p.bl + (size_t)(t0 + kC + tid) * H + h);
                }
            }
            if (!mbar_wait(&bar_full[0], full_parity, kWaitLimitNs)) atomicExch(s_abort, 1);
            __syncthreads();
            if (*s_abort) break;

            // ---- D1 = [Kr; Qr] [Kr; Qr]^T  (K K^T | Q K^T, Q Q^T)
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
            // cumulative log decay b_t (warp 1)
            if (warp == 1) {
                const float x0 = v_lg[2 * lane], x1 = v_lg[2 * lane + 1];
                float sum = x0 + x1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, sum, off);
                    if (lane >= off) sum += y;
                }
                const float b1 = sum, b0 = sum - x1;
                v_b[2 * lane] = b0;
                v_b[2 * lane + 1] = b1;
                v_gam[2 * lane] = __expf(b0);
                v_gam[2 * lane + 1] = __expf(b1);
            }
            wait_mma();

            // ---- E1: norms (diagonals), A (rows 0..63), P (rows 64..127)
            float d1[32];
            ld32f(kColD1 + hc * 32, d1);  // columns [32 hc, 32 hc + 32) of K K^T / Q K^T
            auto pick = [&](const float (&f)[32]) {  // f[lane] without dynamic indexing
                float d = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) d = (j == lane) ? f[j] : d;
                return d;
            };
            if (row < 64) {
                if ((row >> 5) == hc) v_rk[row] = rsqrtf(pick(d1) + 1e-12f);
            } else {
                float dq[32];  // Q Q^T columns; the warp's load stays convergent
                ld32f(kColD1 + 64 + hc * 32, dq);
                if (((row - 64) >> 5) == hc) v_rq[row - 64] = rsqrtf(pick(dq) + 1e-12f);
            }
            __syncthreads();
            const float bC = v_b[63];
            if (row < 64) {
                const int t = row;
                float *arow = sA + t * kAStride + hc * 32;
                if (hc == 1 && t < 32) {  // A is strictly lower triangular: this half is zero
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(arow + j) = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    const float bt = v_b[t], f = v_beta[t] * v_rk[t];
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const int i0 = hc * 32 + j;
                        const float4 rk4 = *reinterpret_cast<const float4 *>(v_rk + i0);
                        const float4 b4 = *reinterpret_cast<const float4 *>(v_b + i0);
                        float4 o;
                        o.x = (i0 + 0 < t) ? f * rk4.x * __expf(bt - b4.x) * d1[j + 0] : 0.f;
                        o.y = (i0 + 1 < t) ? f * rk4.y * __expf(bt - b4.y) * d1[j + 1] : 0.f;
                        o.z = (i0 + 2 < t) ? f * rk4.z * __expf(bt - b4.z) * d1[j + 2] : 0.f;
                        o.w = (i0 + 3 < t) ? f * rk4.w * __expf(bt - b4.w) * d1[j + 3] : 0.f;
                        *reinterpret_cast<float4 *>(arow + j) = o;
                    }
                }
                if (hc == 0) v_c[t] = __expf(bC - v_b[t]) * v_rk[t];
            } else {
                // P = scale * tril(Q K^T) o Gamma with the norms folded in
                const int t = row - 64;
                if (hc == 1 && t < 32) {
                    const float z8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) st_sw128_8(sm + kOffP, t, 4 + c8, z8);
                } else {
                    const float bt = v_b[t], f = p.scale * v_rq[t];
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const int i0 = hc * 32 + c8 * 8;
                        float rk8[8], b8[8], v8[8];
                        *reinterpret_cast<float4 *>(rk8) = *reinterpret_cast<const float4 *>(v_rk + i0);
                        *reinterpret_cast<float4 *>(rk8 + 4) = *reinterpret_cast<const float4 *>(v_rk + i0 + 4);
                        *reinterpret_cast<float4 *>(b8) = *reinterpret_cast<const float4 *>(v_b + i0);
                        *reinterpret_cast<float4 *>(b8 + 4) = *reinterpret_cast<const float4 *>(v_b + i0 + 4);
#pragma unroll
                        for (int u2 = 0; u2 < 8; ++u2)
                            v8[u2] = (i0 + u2 <= t) ? f * rk8[u2] * __expf(bt - b8[u2]) * d1[c8 * 8 + u2] : 0.f;
                        st_sw128_8(sm + kOffP, t, hc * 4 + c8, v8);
                    }
                }
            }
            __syncthreads();

            // ---- T = (I + A)^-1, lower unit-triangular, built from the bottom up:
            // 8x8 diagonal blocks by forward substitution (one column per lane),
            // then merges of neighbouring diagonal blocks lo, hi of growing size,
            //   T[hi, lo] = -T[hi, hi] (A[hi, lo] T[lo, lo]),
            // at size 8 on CUDA cores and at sizes 16 and 32 with warp-level
            // TF32 tensor-core tiles.  The product A[hi, lo] T[lo, lo] is kept in
            // A's (unused) upper triangle.
            if (warp < 2) {
                const int blk = warp * 4 + (lane >> 3), j = lane & 7, base = blk * 8;
                float tc[8];
#pragma unroll
                for (int r2 = 0; r2 < 8; ++r2) {
                    const float *arow = sA + (base + r2) * kAStride + base;
                    const float4 lo4 = *reinterpret_cast<const float4 *>(arow);
                    const float4 hi4 = *reinterpret_cast<const float4 *>(arow + 4);
                    const float av[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
                    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                    for (int i = 0; i < r2; ++i) {
                        if (i & 1) acc1 = fmaf(av[i], tc[i], acc1);
                        else acc0 = fmaf(av[i], tc[i], acc0);
                    }
                    tc[r2] = (r2 == j) ? 1.f : (r2 > j ? -(acc0 + acc1) : 0.f);
                }
#pragma unroll
                for (int r2 = 0; r2 < 8; ++r2) sT[(base + r2) * kAStride + base + j] = tc[r2];
            } else {
                const int q0 = tid - 64, nq = kThreads - 64;
                // the merges read the upper-right zero blocks of the diagonal
                // blocks they combine: T[lo:lo+8, lo+8:lo+16] (size 8) and
                // T[lo:lo+16, lo+16:lo+32] (size 16)
                for (int q = q0; q < 4 * 64 + 2 * 256; q += nq) {
                    if (q < 256) {
                        const int lo = (q >> 6) * 16, r2 = (q >> 3) & 7, c = q & 7;
                        sT[(lo + r2) * kAStride + lo + 8 + c] = 0.f;
                    } else {
                        const int q2 = q - 256, lo = (q2 >> 8) * 32, r2 = (q2 >> 4) & 15, c = q2 & 15;
                        sT[(lo + r2) * kAStride + lo + 16 + c] = 0.f;
                    }
                }
                // Q tile rows t scaled by scale * r_q(t) * gamma_t (MMA1 is done
                // with it), so that S0 Q^T and Delta^T P^T share one accumulator
                unsigned char *qt = stage + 8192;
                for (int q = q0; q < 64 * 16; q += nq) {
                    const int t = q >> 4, kb = (q >> 3) & 1, c8 = q & 7;
                    uint4 *ptr = reinterpret_cast<uint4 *>(qt + kb * 16384 + sw128_offset(t, c8 * 8));
                    const float f = p.scale * v_rq[t] * v_gam[t];
                    uint4 w = *ptr;
                    __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
                    for (int u2 = 0; u2 < 4; ++u2) {
                        const float2 v2 = __bfloat1622float2(h2[u2]);
                        h2[u2] = __floats2bfloat162_rn(v2.x * f, v2.y * f);
                    }
                    *ptr = w;
                }
            }
            __syncthreads();
            {   // size 8: 4 pairs, X = A[hi, lo] T[lo, lo] (8x8x8), one output per thread
                const int pr = tid >> 6, r2 = (tid >> 3) & 7, c = tid & 7;
                const int lo = pr * 16, hi = lo + 8;
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    acc = fmaf(sA[(hi + r2) * kAStride + lo + k], sT[(lo + k) * kAStride + lo + c], acc);
                sA[(lo + r2) * kAStride + hi + c] = acc;
            }
            __syncthreads();
            {   // T[hi, lo] = -T[hi, hi] X
                const int pr = tid >> 6, r2 = (tid >> 3) & 7, c = tid & 7;
                const int lo = pr * 16, hi = lo + 8;
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    acc = fmaf(sT[(hi + r2) * kAStride + hi + k], sA[(lo + k) * kAStride + hi + c], acc);
                sT[(hi + r2) * kAStride + lo + c] = -acc;
            }
            __syncthreads();
            // size 16: 2 pairs x (16 x 16) outputs = 4 warps x two 16x8 tiles... one tile per warp
            if (warp < 4) {
                const int lo = (warp >> 1) * 32, hi = lo + 16, n0 = (warp & 1) * 8;
                warp_tile_product(sA + hi * kAStride + lo, sT + lo * kAStride + lo,
                                  sA + lo * kAStride + hi, 0, n0, 16, 1.f, lane);
            }
            __syncthreads();
            if (warp < 4) {
                const int lo = (warp >> 1) * 32, hi = lo + 16, n0 = (warp & 1) * 8;
                warp_tile_product(sT + hi * kAStride + hi, sA + lo * kAStride + hi,
                                  sT + hi * kAStride + lo, 0, n0, 16, -1.f, lane);
            }
            __syncthreads();
            // size 32: X2 = A[32:64, 0:32] T[0:32, 0:32] (32 x 32: 8 warps x one 16x8 tile)
            {
                const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
                warp_tile_product(sA + 32 * kAStride, sT, sA + 32, m0, n0, 32, 1.f, lane);
            }
            __syncthreads();
            {   // T[32:64, 0:32] = -T[32:64, 32:64] X2
                const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
                warp_tile_product(sT + 32 * kAStride + 32, sA + 32, sT + 32 * kAStride, m0, n0, 32,
                                  -1.f, lane);
            }
            __syncthreads();
            // Tw = T diag(r_k beta gamma), Tb = T diag(beta), bf16 (T is lower triangular)
#pragma unroll
            for (int q = tid; q < 64 * 8; q += kThreads) {
                const int t = q >> 3, c8 = q & 7, i0 = c8 * 8;
                float t8[8], be8[8], ga8[8], rk8[8], w8[8], b8[8];
                *reinterpret_cast<float4 *>(t8) = *reinterpret_cast<const float4 *>(sT + t * kAStride + i0);
                *reinterpret_cast<float4 *>(t8 + 4) = *reinterpret_cast<const float4 *>(sT + t * kAStride + i0 + 4);
                *reinterpret_cast<float4 *>(be8) = *reinterpret_cast<const float4 *>(v_beta + i0);
                *reinterpret_cast<float4 *>(be8 + 4) = *reinterpret_cast<const float4 *>(v_beta + i0 + 4);
                *reinterpret_cast<float4 *>(ga8) = *reinterpret_cast<const float4 *>(v_gam + i0);
                *reinterpret_cast<float4 *>(ga8 + 4) = *reinterpret_cast<const float4 *>(v_gam + i0 + 4);
                *reinterpret_cast<float4 *>(rk8) = *reinterpret_cast<const float4 *>(v_rk + i0);
                *reinterpret_cast<float4 *>(rk8 + 4) = *reinterpret_cast<const float4 *>(v_rk + i0 + 4);
#pragma unroll
                for (int u2 = 0; u2 < 8; ++u2) {
                    const float tv = (i0 + u2 <= t) ? t8[u2] : 0.f;
                    b8[u2] = tv * be8[u2];
                    w8[u2] = b8[u2] * ga8[u2] * rk8[u2];
                }
                st_sw128_8(sm + kOffTw, t, c8, w8);
                st_sw128_8(sm + kOffTb, t, c8, b8);
            }
            fence_async_smem();
            sync_all();

            // ---- D2 = Kr^T Tw^T (= W^T), D3 = V^T Tb^T
            if (tid == 0) {
                const uint32_t id = idesc_bf16(128, 64, true, false);
                const uint32_t tw = smem_u32(sm + kOffTw), tb = smem_u32(sm + kOffTb);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColD2, sdesc_sw128(kq + ks * 2048, 16384, 1024),
                             sdesc_sw128(tw + ks * 32, 16, 1024), id, ks > 0);
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
                const float gC = __expf(bC);
                unsigned char *s0 = sm + kOffS0 + hc * 16384;  // this half is one K-block
#pragma unroll
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

            // ---- D3 -= S0 W^T ;  D4 = S0 Qr^T
            if (tid == 0) {
                const uint32_t s0 = smem_u32(sm + kOffS0), wt = smem_u32(sm + kOffWt);
                const uint32_t idn = idesc_bf16(128, 64, false, true, true);
                const uint32_t idq = idesc_bf16(128, 64, false, false);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + kColD3, sdesc_sw128(s0 + aoff, 16, 1024),
                             sdesc_sw128(wt + ks * 2048, 8192, 1024), idn, 1);
                }
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + kColD4, sdesc_sw128(s0 + aoff, 16, 1024),
                             sdesc_sw128(kq + 8192 + aoff, 16, 1024), idq, ks > 0);
                }
                mma_commit(bar_mma);
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

            // ---- D5 = Delta^T P^T ;  S += Delta'^T Kr
            if (tid == 0) {
                const uint32_t dt = smem_u32(sm + kOffDt), dt2 = smem_u32(sm + kOffDt2);
                const uint32_t pp = smem_u32(sm + kOffP);
                const uint32_t id5 = idesc_bf16(128, 64, false, false);
                const uint32_t id6 = idesc_bf16(128, 128, false, true);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // accumulate onto S0 Q~^T
                    mma_bf16(tmem + kColD4, sdesc_sw128(dt + ks * 32, 16, 1024),
                             sdesc_sw128(pp + ks * 32, 16, 1024), id5, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColS, sdesc_sw128(dt2 + ks * 32, 16, 1024),
                             sdesc_sw128(kq + ks * 2048, 16384, 1024), id6, 1);
                mma_commit(bar_mma);
            }
            wait_mma();
            // the stage is free: load the next chunk while the outputs are written
            if (tid == 0 && n + 1 < nchunks) issue_tma(n + 1);

            // ---- E4: o = D4 (= scale (r_q gamma S0 Q^T + P Delta), the scalings
            // being folded into Q~ and P), staged as a [64 t][128 vi] bf16 tile
            // in the (now free) Delta buffers, then written as 16-byte rows
            {
                float f4[32];
                ld32f(kColD4 + hc * 32, f4);
                __nv_bfloat16 *otile = reinterpret_cast<__nv_bfloat16 *>(sm + kOffOut);
#pragma unroll
                for (int j = 0; j < 32; ++j) otile[(hc * 32 + j) * 128 + row] = __float2bfloat16_rn(f4[j]);
                __syncthreads();
                __nv_bfloat16 *obase = p.out + (size_t)t0 * H * V + (size_t)h * V + vt * 128;
                for (int q = tid; q < Cn * 16; q += kThreads) {
                    const int t = q >> 4, c16 = q & 15;
                    *reinterpret_cast<uint4 *>(obase + (size_t)t * H * V + c16 * 8) =
                        *reinterpret_cast<const uint4 *>(otile + t * 128 + c16 * 8);
                }
            }
            sync_all();
        }
        gchunk += nchunks;
        if (*s_abort) break;

        // final state row `row`, columns [64 hc, 64 hc + 64) -> global
        {
            float *dst = p.state_fin + state_row * 128 + hc * 64;
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

cudaError_t launch_delta_chunked(const ChunkLaunch &c, cudaStream_t s) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)c.W, (cuuint64_t)(c.N > 0 ? c.N : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)c.W * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(c.y), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    ChunkParams p{};
    p.a = c.a; p.bl = c.bl; p.A_log = c.A_log; p.dt_bias = c.dt_bias;
    p.offsets = c.offsets; p.seq_order = c.seq_order; p.header = c.header;
    p.state_init = c.state_init; p.state_fin = c.state_fin;
    p.out = static_cast<__nv_bfloat16 *>(c.out);
    p.B = c.B; p.N = c.N; p.H = c.H; p.HQ = c.HQ; p.V = c.V; p.VT = c.V / 128;
    p.scale = c.scale;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunked_delta_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const long max_units = c.max_units;
    const long slots = (long)sm_count() * kCtasPerSm;
    const int grid = (int)(max_units < slots ? max_units : slots);
    if (grid <= 0) return cudaSuccess;
    cudaError_t e = launch_kernel(chunked_delta_kernel, dim3(grid), dim3(kThreads), kSmemBytes, s,
                                  true, map, p);
    note_launch();
    return e;
}

}  // namespace gdn
