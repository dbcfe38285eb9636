// delta_chunked_pc.cu - chunkwise gated delta rule with a per-key-channel gate
// (GDN_OPT_GATE_PER_CHANNEL; rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet,
// gate_per_channel) on tcgen05 tensor cores, the fp32 state held in tensor
// memory across chunks.
//
// The recurrence (the DELTA kernel of paged_ssm.rs with a diagonal decay) is
//   S_t = S_{t-1} diag(g_t) + beta_t (v_t - S_{t-1} diag(g_t) k_t) k_t^T,
//   o_t = scale S_t q_t,
// with normalised q, k.  Within a chunk of C = 16 tokens, with the per-channel
// cumulative log decay b_t[c] = sum_{s<=t} log g_s[c] (so every factor
// e^{b_t - b_i}, e^{b_t}, e^{b_C - b_t} with i <= t is at most 1):
//   KK[t,i] = sum_c k_t[c] k_i[c] e^{b_t[c] - b_i[c]},  QK[t,i] likewise with q_t,
//   A[t,i] = beta_t KK[t,i] (i < t),  T = (I + A)^-1,
//   W = T diag(beta) Kt,  Kt[s,c] = k_s[c] e^{b_s[c]},   U = T diag(beta) V,
//   Delta = U - W S_0^T,
//   O = scale (Qt S_0^T + tril(QK) Delta),  Qt[t,c] = q_t[c] e^{b_t[c]},
//   S_C = S_0 diag(e^{b_C}) + Delta^T Kp,  Kp[t,c] = k_t[c] e^{b_C[c] - b_t[c]}.
// The exponentials of KK and QK are formed in 4-token blocks: for tokens t in
// a later block than i, e^{b_t - b_i} = e^{b_t - b_r} e^{b_r - b_i} with b_r the
// last token of i's block, two factors of at most 1 each; inside a block they
// are taken pair by pair.  No factor can overflow, whatever the gates.
//
// Everything but Delta, O and S_C is independent of the state, so it is
// computed for all chunks at once by pc_prep_kernel (CUDA cores; one CTA per
// chunk and value head) and written out as a chunk image laid out exactly as
// the scan kernel's shared-memory operands.  pc_scan_kernel then walks each
// (sequence, value head, V tile) unit's chunks in order, copying each image in
// with a bulk copy and the chunk's v rows with a tensor copy (two chunks
// ahead), and runs on tcgen05 (M = 128 state rows, bf16 operands, fp32
// accumulators in tensor memory):
//   [Delta^T | Do] = S0 [-W ; Qt]^T + [V^T (T diag(beta))^T | 0]
//                                 (S0 = bf16 copy of the state, N = 32 and 16)
//   Do += Delta^T P^T             (P = scale tril(QK), K = 16)
//   S  += Delta^T Kp              (S first scaled by e^{b_C} per column, N = 128)
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace gdn {

namespace {

using namespace sm100;

constexpr int kPc = 16;                        // chunk length
constexpr uint64_t kPcWaitNs = 2000000000ull;  // bounded waits: 2 s

// chunk image offsets (bytes); P and T diag(beta) share one SW128 tile
// [-W ; Qt] is one [32][128] operand: two SW128 blocks of [32][64], 4096 bytes
// apart, rows 0..15 = -W and 16..31 = Qt
constexpr uint32_t kImWQ = 0, kImKp = 8192, kImPT = 12288, kImCs = 14336;
static_assert(kImCs + 512 == kPcImgHead, "image head layout");

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint4 pack8(const float *v) {
    return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}
// byte offset of element (row, col) of a [rows][128] bf16 operand kept as two
// SW128 blocks of [rows][64], 2048 bytes apart (rows < 16)
__device__ __forceinline__ uint32_t op_offset(int row, int col) {
    return (uint32_t)(col >> 6) * 2048u + sw128_offset(row, col & 63);
}
// the same for the [32][128] operand [-W ; Qt] (blocks 4096 bytes apart)
__device__ __forceinline__ uint32_t wq_offset(int row, int col) {
    return (uint32_t)(col >> 6) * 4096u + sw128_offset(row, col & 63);
}
__device__ __forceinline__ void st_bf16(unsigned char *p, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}
// Packed fp32 (two lanes of one instruction; each component rounds exactly as
// the scalar multiply / fused multiply-add).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }
// dot4 of a and of b with the same f, two chains side by side: (a.f + acc.x, b.f + acc.y)
__device__ __forceinline__ float2 dot4x2(float4 a, float4 b, float4 f, float2 acc) {
    acc = __ffma2_rn(make_float2(a.x, b.x), splat2(f.x), acc);
    acc = __ffma2_rn(make_float2(a.y, b.y), splat2(f.y), acc);
    acc = __ffma2_rn(make_float2(a.z, b.z), splat2(f.z), acc);
    return __ffma2_rn(make_float2(a.w, b.w), splat2(f.w), acc);
}

// ------------------------------------------------------------------ prepare
// One CTA per (image slot, value head): finds the slot's sequence and chunk,
// and writes the chunk image (the P / T diag(beta) tile is built in shared
// memory, an operand of the W MMA, and copied out at the end).  Slots with no chunk (short sequences, the end of a sequence's slot range)
// return at once.
//
// Every decay factor is a product of per-token gates g_j = e^{log g_j} (each
// at most 1): with P_t = prod_{j<=t} g_j, Kt = k P_t, Qt = q P_t and
// Kp = k prod_{j>t} g_j.  For KK / QK the 16 tokens form four blocks of 4;
// for t in block TB and i in an earlier block, with r = 4 TB - 1,
//   e^{b_t - b_i} = X_TB[t] Z_TB[i],  X_TB[t] = prod_{r<j<=t} g_j,
//   Z_TB[i] = prod_{i<j<=r} g_j,
// so those entries are dot products of the rows k_t X_TB[t] (or q_t X_TB[t])
// and k_i Z_TB[i]: one tcgen05 MMA of the 24 Z rows (M, padded to 128: the
// rows past 24 are whatever shared memory follows them, and their results are
// never read) with the 24 X rows (N = 32).  Inside a block the factor of
// (t, i) is formed from the gates between them, on CUDA cores.  q/k norms
// are applied to the finished dot products.  W^T = Kt^T (T diag(beta rk))^T
// is a second MMA (M = 128 channels, N = 16, K = 16).
constexpr int kPrepThreads = 256;

// shared memory of the prepare kernel (bytes from a 1024-aligned base)
constexpr uint32_t kPZ0 = 0;          // Z rows, channels 0..63: SW128 rows 0..23 of a [128][64] span
constexpr uint32_t kPK = 3072;        // raw k, fp32 [16][128]
constexpr uint32_t kPAm = 11264;      // A[t][i] = fr beta_t rk_t rk_i KK, fp32 [16][16]
constexpr uint32_t kPVec = 12288;     // beta[16], rk[16], rq[16]; barrier, TMEM address, flag
constexpr uint32_t kPZ1 = 16384;      // Z rows, channels 64..127 (second half of the span)
constexpr uint32_t kPQ = 19456;       // raw q, fp32 [16][128]
constexpr uint32_t kPL = 28672;       // X rows (k X: 0..11, q X: 12..23): two SW128 blocks [32][64]
constexpr uint32_t kPG = 36864;       // gate inputs, then gate factors, fp32 [16][128]
constexpr uint32_t kPKt = 45056;      // Kt = k P_t, bf16: two SW128 blocks [16][64]
constexpr uint32_t kPPT = 49152;      // the image's P / T diag(beta) tile (SW128 [16][64])
constexpr uint32_t kPrepSmem = kPPT + 2048 + 1024;  // + alignment slack: four CTAs per SM
static_assert(kPK >= 24 * 128 && kPQ >= kPZ1 + 24 * 128 && kPL >= kPQ + 8192, "prepare layout");
static_assert(kPVec + 256 <= kPZ1 && kPPT % 1024 == 0, "prepare layout");
constexpr uint32_t kPrepTmemCols = 64;  // KK / QK products in [0, 32), W^T in [32, 48)

// gate factor of one key channel from its input under the options
__device__ __forceinline__ float gate_factor_of(float x, float dtb, float neg_a, int opts, int factor) {
    if (opts & GDN_OPT_NO_DECAY) return 1.f;
    if (factor) return fmaxf(x, 0.f);
    if (opts & GDN_OPT_GATE_EXP) return __expf(x);
    x += dtb;
    const float softplus = fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)));
    return __expf(neg_a * softplus);
}

__global__ void __launch_bounds__(kPrepThreads, 4) pc_prep_kernel(const __grid_constant__ PcParams p) {
    // Every CTA waits for the conv kernel before it exits, slots without a
    // chunk included: the scan kernel's wait on this grid then also covers
    // the conv kernel's output (the schedule in the workspace header).
    pdl_wait_primary();

    // the CTA's sequence lo, chunk n and value head h: from a (chunk, sequence,
    // head) grid, or from the image slot q (a (slot, head) grid): the last
    // sequence with (offsets[i] >> 4) + i <= q
    int lo, n, h, s, e;
    if (p.grid_chunks > 0) {
        n = blockIdx.x;
        lo = blockIdx.y;
        h = blockIdx.z;
        if (p.uniform_len > 0) {
            s = lo * p.uniform_len;
            e = s + p.uniform_len;
        } else {
            s = __ldg(p.offsets + lo);
            e = __ldg(p.offsets + lo + 1);
        }
    } else {
        const int slot = blockIdx.x;
        h = blockIdx.y;
        lo = 0;
        int hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((__ldg(p.offsets + mid) >> 4) + mid <= slot) lo = mid;
            else hi = mid - 1;
        }
        s = __ldg(p.offsets + lo);
        e = __ldg(p.offsets + lo + 1);
        n = slot - ((s >> 4) + lo);
    }
    if (s < 0 || e < s || e > p.N || e - s < p.thr) return;
    if (n < 0 || n >= (e - s + kPc - 1) / kPc) return;
    const int q = (s >> 4) + lo + n;  // the image slot
    const int t0 = s + n * kPc, Cn = min(kPc, e - t0);

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sK = reinterpret_cast<float *>(sm + kPK), *sQ = reinterpret_cast<float *>(sm + kPQ);
    float *sG = reinterpret_cast<float *>(sm + kPG), *sAm = reinterpret_cast<float *>(sm + kPAm);
    float *v_beta = reinterpret_cast<float *>(sm + kPVec), *v_rk = v_beta + 16, *v_rq = v_rk + 16;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kPVec + 192);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar + 1);
    int *s_bad = reinterpret_cast<int *>(s_tmem + 1);
    unsigned char *pt = sm + kPPT;  // the P / T diag(beta) tile
    unsigned char *img = p.img + ((size_t)q * p.H + h) * (size_t)p.img_bytes;  // global

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, opts = p.opts;
    const int kh = h / (H / p.HQ);
    const __nv_bfloat16 *qsrc = p.qb + (size_t)kh * 128;
    const __nv_bfloat16 *ksrc = p.kb + (size_t)kh * 128;
    const bool soft = !(opts & (GDN_OPT_NO_DECAY | GDN_OPT_GATE_EXP)) && !p.gate_factor;
    const float dtb = soft ? __ldg(p.dt_bias + h) : 0.f;
    const float neg_a = soft ? -expf(__ldg(p.A_log + h)) : 0.f;
    const float fr = (opts & GDN_OPT_NO_RETRIEVE) ? 0.f : 1.f;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *s_bad = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kPrepTmemCols);
        tmem_relinquish();
    }

    // ---- L: raw k, q rows as fp32 (rows past the sequence are 0), the gate
    // inputs and beta; every load is issued before the first is used
    {
        const bool decay = !(opts & GDN_OPT_NO_DECAY);
        uint4 kq[2];
        float4 lg[2];
        float be = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = tid + j * kPrepThreads;
            const int tile = i >> 8, r = (i >> 4) & 15, c8 = (i & 15) * 8;
            kq[j] = make_uint4(0u, 0u, 0u, 0u);
            if (r < Cn)
                kq[j] = __ldg(reinterpret_cast<const uint4 *>((tile == 0 ? ksrc : qsrc) + (size_t)(t0 + r) * p.rs + c8));
            const int r2 = i >> 5, c4 = i & 31;
            lg[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r2 < Cn && decay)
                lg[j] = __ldg(reinterpret_cast<const float4 *>(p.g + ((size_t)(t0 + r2) * H + h) * 128) + c4);
        }
        if (tid < Cn) {
            be = 1.f;
            if (!(opts & GDN_OPT_NO_BETA)) be = __ldg(p.bl + (size_t)(t0 + tid) * H + h);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = tid + j * kPrepThreads;
            const int tile = i >> 8, r = (i >> 4) & 15, c8 = (i & 15) * 8;
            const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(&kq[j]);
            float *dst = (tile == 0 ? sK : sQ) + r * 128 + c8;
            *reinterpret_cast<float4 *>(dst) = make_float4(__bfloat162float(x[0]), __bfloat162float(x[1]),
                                                           __bfloat162float(x[2]), __bfloat162float(x[3]));
            *reinterpret_cast<float4 *>(dst + 4) = make_float4(__bfloat162float(x[4]), __bfloat162float(x[5]),
                                                               __bfloat162float(x[6]), __bfloat162float(x[7]));
            reinterpret_cast<float4 *>(sG)[i] = lg[j];
        }
        if (tid < kPc) {
            if (tid < Cn && !(opts & (GDN_OPT_NO_BETA | GDN_OPT_BETA_RAW))) be = 1.f / (1.f + expf(-be));
            v_beta[tid] = be;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // ---- G: gate factors (1 past the sequence); q/k norms, 8 threads per
    // (token, q|k)
    for (int i = tid; i < kPc * 128; i += kPrepThreads)
        sG[i] = (i >> 7) < Cn ? gate_factor_of(sG[i], dtb, neg_a, opts, p.gate_factor) : 1.f;
    {
        const int red = tid >> 3, part = tid & 7;
        const int t = red & 15;
        const float *src = ((red >> 4) ? sQ : sK) + t * 128 + part * 16;
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + j);
            ss = dot4(x, x, ss);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        if (part == 0) {
            const float rn = (opts & GDN_OPT_NO_QK_NORM) ? 1.f : rsqrtf(ss + 1e-12f);
            ((red >> 4) ? v_rq : v_rk)[t] = rn;
        }
    }
    __syncthreads();

    // ---- R: per pair of key channels (c, c + 1), the decay products and the
    // bf16 operands, written two channels at a time; four roles of 64 threads:
    //   0: P_t, Kt = rk k P_t (MMA operand), Qt (image), e^{b_C} (image);
    //   1: the X rows k X, q X (MMA operand);
    //   2: the suffix products and Kp (image);
    //   3: the Z rows (MMA operand).
    {
        const int role = tid >> 6, c = (tid & 63) * 2;
        const uint32_t cb = (uint32_t)(c & 63);
        auto ld2 = [&](const float *base, int t) {
            return *reinterpret_cast<const float2 *>(base + t * 128 + c);
        };
        auto st2 = [&](unsigned char *dst, float x, float y) {
            *reinterpret_cast<uint32_t *>(dst) = pack2(x, y);
        };
        if (role == 0) {
            float2 P = make_float2(1.f, 1.f);
            const float qs = p.scale;
#pragma unroll
            for (int t = 0; t < kPc; ++t) {
                const float2 g = ld2(sG, t), k = ld2(sK, t), qv = ld2(sQ, t);
                P = mul2(P, g);
                const float fk = v_rk[t], fq = v_rq[t] * qs;
                const float2 kt = mul2(mul2(k, splat2(fk)), P), qt = mul2(mul2(qv, splat2(fq)), P);
                st2(sm + kPKt + op_offset(t, c), kt.x, kt.y);
                st2(img + kImWQ + wq_offset(16 + t, c), qt.x, qt.y);
            }
            *reinterpret_cast<float2 *>(img + kImCs + c * 4) = P;
        } else if (role == 1) {
            unsigned char *L = sm + kPL + (c >> 6) * 4096;
#pragma unroll
            for (int TB = 1; TB < 4; ++TB) {
                float2 X = make_float2(1.f, 1.f);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const int t = 4 * TB + a, row = 4 * (TB - 1) + a;
                    const float2 g = ld2(sG, t), k = ld2(sK, t), qv = ld2(sQ, t);
                    X = mul2(X, g);
                    const float2 kx = mul2(k, X), qx = mul2(qv, X);
                    st2(L + sw128_offset(row, cb), kx.x, kx.y);
                    st2(L + sw128_offset(12 + row, cb), qx.x, qx.y);
                }
            }
        } else if (role == 2) {
            float2 Qs = make_float2(1.f, 1.f);
#pragma unroll
            for (int t = kPc - 1; t >= 0; --t) {
                const float2 g = ld2(sG, t), k = ld2(sK, t);
                const float fk = v_rk[t];
                const float2 kp = mul2(mul2(k, splat2(fk)), Qs);
                st2(img + kImKp + op_offset(t, c), kp.x, kp.y);
                Qs = mul2(Qs, g);
            }
        } else {
            unsigned char *Zt = sm + ((c >> 6) ? kPZ1 : kPZ0);
#pragma unroll
            for (int TB = 1; TB < 4; ++TB) {
                const int base = TB == 1 ? 0 : TB == 2 ? 4 : 12;
                float2 Z = make_float2(1.f, 1.f);
#pragma unroll
                for (int i = 4 * TB - 1; i >= 0; --i) {
                    const float2 g = ld2(sG, i), k = ld2(sK, i);
                    const float2 kz = mul2(k, Z);
                    st2(Zt + sw128_offset(base + i, cb), kz.x, kz.y);
                    Z = mul2(Z, g);
                }
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- D: KK and QK.  Later-block entries: one MMA, D[m][j] = Z_m . X_j
    // (TMEM columns 0..31), issued by thread 0 and read by warp 0.  A block
    // with itself: a half-warp per block (warps 4, 5), a lane per 8 channels,
    // summed over the half-warp.  KK lands as A[t,i] = fr beta_t rk_t rk_i KK
    // (i < t), QK as P[t,i] = scale rq_t rk_i QK (i <= t) in the image.
    if (tid == 0) {
        const uint32_t za = smem_u32(sm + kPZ0), xb = smem_u32(sm + kPL);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
            const uint32_t bo = (ks >> 2) * 4096 + (ks & 3) * 32;
            mma_bf16(tmem, sdesc_sw128(za + ao, 16, 1024), sdesc_sw128(xb + bo, 16, 1024),
                     idesc_bf16(128, 32, false, false), ks > 0);
        }
        mma_commit(bar);
    }
    if (warp == 4 || warp == 5) {
        const int TB = (tid - 128) >> 4, cg = tid & 15;
        const int t0b = 4 * TB;
        float kk[4][4], qk[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) kk[a][b] = qk[a][b] = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = cg * 4 + j * 64;
            float4 kr[4], qr[4], gr[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                kr[a] = *reinterpret_cast<const float4 *>(sK + (t0b + a) * 128 + c);
                qr[a] = *reinterpret_cast<const float4 *>(sQ + (t0b + a) * 128 + c);
                gr[a] = *reinterpret_cast<const float4 *>(sG + (t0b + a) * 128 + c);
            }
            // column b: f = k_b times the gates of tokens b+1 .. a of the block
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                float4 f = kr[b];
                qk[b][b] = dot4(qr[b], f, qk[b][b]);
#pragma unroll
                for (int a = b + 1; a < 4; ++a) {
                    const float2 fxy = mul2(make_float2(f.x, f.y), make_float2(gr[a].x, gr[a].y));
                    const float2 fzw = mul2(make_float2(f.z, f.w), make_float2(gr[a].z, gr[a].w));
                    f = make_float4(fxy.x, fxy.y, fzw.x, fzw.y);
                    // the KK and QK chains of (a, b) side by side
                    const float2 kq = dot4x2(kr[a], qr[a], f, make_float2(kk[a][b], qk[a][b]));
                    kk[a][b] = kq.x;
                    qk[a][b] = kq.y;
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b <= a; ++b)
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    if (b < a) kk[a][b] += __shfl_xor_sync(0xffffffffu, kk[a][b], o);
                    qk[a][b] += __shfl_xor_sync(0xffffffffu, qk[a][b], o);
                }
        if (cg == 0) {
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b <= a; ++b) {
                    const int t = t0b + a, i = t0b + b;
                    if (b < a) sAm[t * 16 + i] = fr * v_beta[t] * v_rk[t] * v_rk[i] * kk[a][b];
                    st_bf16(pt + sw128_offset(t, i), p.scale * v_rq[t] * v_rk[i] * qk[a][b]);
                }
        }
    }
    {  // the zero upper triangle of P (i > t)
        const int t = tid >> 4, i = tid & 15;
        if (i > t) st_bf16(pt + sw128_offset(t, i), 0.f);
    }
    if (warp == 0) {
        if (!mbar_wait(bar, 0, kPcWaitNs)) atomicExch(s_bad, 1);
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(tmem, r);  // lanes 0..31 = Z rows
        tmem_wait_ld();
        if (lane < 24) {
            const int TB = lane < 4 ? 1 : lane < 12 ? 2 : 3;
            const int i = lane - (TB == 1 ? 0 : TB == 2 ? 4 : 12);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const uint32_t kx = TB == 1 ? r[a] : TB == 2 ? r[4 + a] : r[8 + a];
                const uint32_t qx = TB == 1 ? r[12 + a] : TB == 2 ? r[16 + a] : r[20 + a];
                const int t = 4 * TB + a;
                sAm[t * 16 + i] = fr * v_beta[t] * v_rk[t] * v_rk[i] * __uint_as_float(kx);
                st_bf16(pt + sw128_offset(t, i), p.scale * v_rq[t] * v_rk[i] * __uint_as_float(qx));
            }
        }
    }
    __syncthreads();

    // ---- T = (I + A)^-1 (A strictly lower): forward substitution, one column
    // per lane of warp 0, stored as T diag(beta) (image columns 16..31 of the
    // P tile: the B operand of the scan's V^T MMA and of the W MMA below)
    if (warp == 0 && lane < 16) {
        const int c = lane;
        float pr[16], tc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) pr[r] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            tc[i] = (i == c) ? 1.f : (i > c ? -pr[i] : 0.f);
#pragma unroll
            for (int r = i + 1; r < 16; ++r) pr[r] = fmaf(sAm[r * 16 + i], tc[i], pr[r]);
        }
        const float bc = v_beta[c];
#pragma unroll
        for (int r = 0; r < 16; ++r) st_bf16(pt + sw128_offset(r, 16 + c), tc[r] * bc);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- W^T[c][t] = sum_s Kt[s][c] (T diag(beta))[t][s] (M = 128 channels,
    // N = 16, K = 16; A is Kt, MN-major); warps 0..3 write W (times fr)
    if (tid == 0) {
        mma_bf16(tmem + 32, sdesc_sw128(smem_u32(sm + kPKt), 2048, 1024),
                 sdesc_sw128(smem_u32(pt) + 32, 16, 1024), idesc_bf16(128, 16, true, false), 0);
        mma_commit(bar);
    }
    if (warp < 4) {
        if (!mbar_wait(bar, 1, kPcWaitNs)) atomicExch(s_bad, 1);
        tc_fence_after();
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 32, r);
        tmem_wait_ld();
        const int c = warp * 32 + lane;
#pragma unroll
        for (int t = 0; t < kPc; ++t) st_bf16(img + kImWQ + wq_offset(t, c), -fr * __uint_as_float(r[t]));
    } else {  // warps 4..7: the P / T diag(beta) tile to the image
        const int i = tid - 128;
        reinterpret_cast<uint4 *>(img + kImPT)[i] = reinterpret_cast<const uint4 *>(pt)[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0 && *s_bad) {
        atomicExch(&p.header->status, 7 /* GDN_ERR_TIMEOUT */);
        const uint64_t ts = global_timer_ns();  // let a late MMA land before the
        while (global_timer_ns() - ts < 10000000ull) {  // tensor memory is released
        }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// --------------------------------------------------------------------- scan
constexpr int kScanThreads = 256;   // 8 warps; thread 0 issues copies and MMAs
constexpr int kStages = 3;          // chunk images in flight (two ahead)
// stage: the chunk's v rows of one V tile (two SW128 blocks [16 t][64 vi],
// loaded through vmap), then the image head
constexpr uint32_t kStV = 0, kStImg = 4096;
constexpr uint32_t kStageBytes = 19456;  // rounded to 1 KB
static_assert(kStImg + kPcImgHead <= kStageBytes, "stage size");

// Shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kOS0 = 0;          // S0 bf16 [128 vi][128 kk]: two SW128 blocks of 16 KB
constexpr uint32_t kODt = 32768;      // Delta^T bf16 [128 vi][16 t] in an SW128 [128][64] tile
constexpr uint32_t kOStage = 49152;   // kStages chunk images
constexpr uint32_t kOBar = kOStage + kStages * kStageBytes;
constexpr uint32_t kScanSmem = kOBar + 64 + 1024;  // + alignment slack
static_assert(kScanSmem <= 112 * 1024, "two CTAs per SM");

// TMEM: the state in columns [0, 128); then per chunk parity a 32-column
// block [Dd | Do] at 128 (even chunks) or 160 (odd chunks).
constexpr uint32_t kScanTmemCols = 256;
constexpr uint32_t kColS = 0, kColD = 128;

__device__ __forceinline__ void st8(unsigned char *tile, int row, int c8, const float *v) {
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, c8 * 8)) = pack8(v);
}

// SEG: the segment passes (p.seg_mode 1 or 2); the one-pass instance carries
// none of their code.
template <bool SEG>
__global__ void __launch_bounds__(kScanThreads, 2) pc_scan_kernel(const __grid_constant__ PcParams p) {
    const int seg_mode = SEG ? p.seg_mode : 0;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(sm + kOBar);  // [kStages]
    uint64_t *bar_mma = bar_full + kStages;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar_mma + 1);
    int *s_unit = reinterpret_cast<int *>(s_tmem + 1);
    int *s_abort = s_unit + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hc = warp >> 2;
    const int row = quad * 32 + lane;  // this thread's TMEM lane (state row)

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(bar_full + i, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kScanTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);

    pdl_wait_primary();  // the chunk images are the prepare kernel's output

    const int H = p.H, V = p.V, VT = p.VT;
    const int n_units = seg_mode ? p.seg_units : p.header->n_units;
    unsigned int *counter = seg_mode ? p.counter : &p.header->next_unit;
    uint32_t mma_phase = 0;
    uint32_t gc = 0;  // chunks this CTA has consumed: the stage ring position

    auto wait_mma = [&]() {
        const bool ok = mbar_wait(bar_mma, mma_phase & 1, kPcWaitNs);
        ++mma_phase;
        if (!ok) atomicExch(s_abort, 1);
        tc_fence_after();
    };
    auto sync_all = [&]() {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    // output rows t < rows of the chunk starting at token t0, from Do buffer `buf`
    auto store_out = [&](int buf, int t0, int rows, int h, int vt) {
        uint32_t r[16];
        tmem_ld16(lane_base + kColD + 32 * buf + 16, r);
        tmem_wait_ld();
        __nv_bfloat16 *o = p.out + (size_t)t0 * p.ors + (size_t)h * V + (size_t)vt * 128 + row;
#pragma unroll
        for (int t = 0; t < kPc; ++t)
            if (t < rows) o[(size_t)t * p.ors] = __float2bfloat16_rn(__uint_as_float(r[t]));
    };

    while (true) {
        if (tid == 0) *s_unit = (int)atomicAdd(counter, 1u);
        __syncthreads();
        const int u = *s_unit;
        if (u >= n_units || *s_abort) break;
        int seq, h, vt, q = 0, seg = 0, nseg_here = 1;
        bool mtile = false;  // the transition tile of a segment (seg_mode 1)
        if (seg_mode == 0) {
            seq = p.seq_order[u / (H * VT)];
            h = (u / VT) % H;
            vt = u % VT;
        } else {
            // q: the segment's index among this pass's segments (numbering the M /
            // L or start-state buffers); constant indices into the tables only
            const int tiles = VT + (seg_mode == 1);
            q = u / (H * tiles);
            h = (u / tiles) % H;
            const int tile = u % tiles;
            mtile = tile == VT;
            vt = mtile ? 0 : tile;
            seq = p.seg_seq[0];
            seg = q;
            nseg_here = p.seg_s0[1];
#pragma unroll
            for (int i = 1; i < kMaxSegSeqs; ++i) {
                const int f = seg_mode == 1 ? p.seg_m0[i] : p.seg_s0[i];
                if (i < p.nseq_seg && q >= f) {
                    seq = p.seg_seq[i];
                    seg = q - f;
                    nseg_here = p.seg_s0[i + 1] - p.seg_s0[i];
                }
            }
        }
        const int s_seq = p.offsets[seq];
        int s = s_seq, e = p.offsets[seq + 1];
        if (s < 0 || e < s || e > p.N) {  // malformed offsets: nothing is read or written
            __syncthreads();
            continue;
        }
        if (seg_mode) {  // this segment's tokens (a multiple of 64 from the sequence start)
            int seg_len;
            segment_split(e - s, nseg_here, seg_len, nseg_here);
            if (seg >= (seg_mode == 1 ? nseg_here - 1 : nseg_here)) {
                __syncthreads();
                continue;
            }
            s += seg * seg_len;
            e = min(e, s + seg_len);
        }
        const bool write_out = seg_mode != 1;
        const int nch = (e - s + kPc - 1) / kPc;
        const size_t chunk_stride = (size_t)H * p.img_bytes;
        // the image of the unit's first chunk: chunk (s - s_seq) / 16 of its sequence
        const unsigned char *img0 =
            p.img + ((size_t)((s_seq >> 4) + seq + (s - s_seq) / kPc) * H + h) * p.img_bytes;
        const int vcol = p.vcol0 + h * V + vt * 128;
        auto issue = [&](int n) {  // thread 0: chunk n's image head and v rows
            const uint32_t st = (gc + n) % kStages;
            unsigned char *dst = sm + kOStage + st * kStageBytes;
            uint64_t *bar = bar_full + st;
            mbar_arrive_expect_tx(bar, kPcImgHead + 4096);
            bulk_load(dst + kStImg, img0 + (size_t)n * chunk_stride, kPcImgHead, bar);
            tma_load_2d(dst + kStV, &p.vmap, bar, vcol, s + n * kPc);
            tma_load_2d(dst + kStV + 2048, &p.vmap, bar, vcol + 64, s + n * kPc);
        };
        if (tid == 0) {
            if (nch > 0) issue(0);
            if (nch > 1) issue(1);
        }
        const size_t state_row = ((size_t)seq * H + h) * V + (size_t)vt * 128 + row;

        // state row `row`, columns [64 hc, 64 hc + 64) -> TMEM: the initial
        // state, a segment's start state, zero, or the identity (transition tile)
        {
            const float *src = p.state_init + state_row * 128 + hc * 64;
            if (seg_mode == 2)
                src = p.seg_S + ((((size_t)q * H + h) * V + vt * 128 + row) * 128 + hc * 64);
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                if (seg_mode == 1) {
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

#pragma unroll 1
        for (int n = 0; n < nch; ++n) {
            const uint32_t st = (gc + n) % kStages;
            unsigned char *stage = sm + kOStage + st * kStageBytes;
            if (!mbar_wait(bar_full + st, ((gc + n) / kStages) & 1, kPcWaitNs)) atomicExch(s_abort, 1);

            // ---- E1: the previous chunk's output rows (warps 0..3); the state's
            // bf16 copy S0 and its column decay S *= e^{b_C} (all warps)
            if (hc == 0 && n > 0 && write_out) store_out((n - 1) & 1, s + (n - 1) * kPc, kPc, h, vt);
            {
                const float *cs = reinterpret_cast<const float *>(stage + kStImg + kImCs);
                unsigned char *s0 = sm + kOS0 + hc * 16384;  // this half is one K-block
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + kColS + hc * 64 + c0, r);
                    tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) st8(s0, row, (c0 >> 3) + c8, v + c8 * 8);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 f = *reinterpret_cast<const float4 *>(cs + hc * 64 + c0 + j);
                        r[j] = __float_as_uint(v[j] * f.x);
                        r[j + 1] = __float_as_uint(v[j + 1] * f.y);
                        r[j + 2] = __float_as_uint(v[j + 2] * f.z);
                        r[j + 3] = __float_as_uint(v[j + 3] * f.w);
                    }
                    tmem_st32(lane_base + kColS + hc * 64 + c0, r);
                }
                tmem_wait_st();
            }
            fence_async_smem();
            sync_all();

            // ---- [Dd | Do] = S0 [-W ; Qt]^T (M = 128, N = 32, K = 128), then
            // Dd += V^T (T diag(beta))^T (N = 16, K = 16): Dd = Delta^T, Do = S0 Qt^T.
            // The image two chunks ahead goes into the stage chunk n - 1 used.
            const uint32_t dbuf = kColD + 32 * (n & 1);  // [Dd | Do] of this chunk
            if (tid == 0) {
                if (n + 2 < nch) issue(n + 2);
                const uint32_t s0 = smem_u32(sm + kOS0), wq = smem_u32(stage + kStImg + kImWQ);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
                    const uint32_t bo = (ks >> 2) * 4096 + (ks & 3) * 32;
                    mma_bf16(tmem + dbuf, sdesc_sw128(s0 + ao, 16, 1024), sdesc_sw128(wq + bo, 16, 1024),
                             idesc_bf16(128, 32, false, false), ks > 0);
                }
                // V^T: MN-major A (two 64-row blocks 2048 bytes apart); T diag(beta):
                // columns 16..31 of the P tile (v = 0 for a transition tile)
                if (!mtile)
                    mma_bf16(tmem + dbuf, sdesc_sw128(smem_u32(stage + kStV), 2048, 1024),
                             sdesc_sw128(smem_u32(stage + kStImg + kImPT) + 32, 16, 1024),
                             idesc_bf16(128, 16, true, false), 1);
                mma_commit(bar_mma);
            }
            wait_mma();

            // ---- Delta^T -> bf16 A operand (warps 0..3)
            if (hc == 0) {
                uint32_t r[16];
                tmem_ld16(lane_base + dbuf, r);
                tmem_wait_ld();
                float d[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) d[t] = __uint_as_float(r[t]);
                st8(sm + kODt, row, 0, d);
                st8(sm + kODt, row, 1, d + 8);
            }
            fence_async_smem();
            sync_all();

            // ---- Do += Delta^T P^T (K = 16);  S += Delta^T Kp (N = 128, K = 16)
            if (tid == 0) {
                const uint32_t dt = smem_u32(sm + kODt), pp = smem_u32(stage + kStImg + kImPT);
                const uint32_t kp = smem_u32(stage + kStImg + kImKp);
                mma_bf16(tmem + dbuf + 16, sdesc_sw128(dt, 16, 1024), sdesc_sw128(pp, 16, 1024),
                         idesc_bf16(128, 16, false, false), 1);
                mma_bf16(tmem + kColS, sdesc_sw128(dt, 16, 1024), sdesc_sw128(kp, 2048, 1024),
                         idesc_bf16(128, 128, false, true), 1);
                mma_commit(bar_mma);
            }
            wait_mma();
            if (*s_abort) break;
        }
        gc += nch;
        if (*s_abort) break;

        // the last chunk's output rows; the final state row `row`, columns
        // [64 hc, 64 hc + 64) -> global
        if (hc == 0 && nch > 0 && write_out)
            store_out((nch - 1) & 1, s + (nch - 1) * kPc, e - s - (nch - 1) * kPc, h, vt);
        if (seg_mode != 2 || seg == nseg_here - 1) {
            float *dst = p.state_fin + state_row * 128 + hc * 64;
            if (seg_mode == 1)
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

    if (*s_abort && tid == 0) {
        // a bounded wait gave up: record it and give copies and MMAs still in
        // flight time to land before the shared and tensor memory are released
        atomicExch(&p.header->status, 7 /* GDN_ERR_TIMEOUT */);
        const uint64_t ts = global_timer_ns();
        while (global_timer_ns() - ts < 10000000ull) {  // 10 ms
        }
    }
    sync_all();
    if (warp == 0) tmem_dealloc(tmem, kScanTmemCols);
}

int pc_sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_delta_chunked_pc(const PcParams &p, long max_units, cudaStream_t s) {
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [] {
        cudaError_t e2 = cudaFuncSetAttribute(pc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)kPrepSmem);
        if (e2 == cudaSuccess)
            e2 = cudaFuncSetAttribute(pc_scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kScanSmem);
        if (e2 != cudaSuccess) return e2;
        return cudaFuncSetAttribute(pc_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kScanSmem);
    });
    if (e != cudaSuccess) return e;
    const size_t slots = pc_slots(p.B, p.N);
    if (slots > 0x7fffffffull || p.H > 65535) return cudaErrorInvalidValue;
    // a (chunk, sequence, head) grid when the longest sequence is known, else
    // one CTA per (image slot, head) that searches the offsets for its sequence
    const dim3 pgrid = p.grid_chunks > 0 ? dim3((unsigned)p.grid_chunks, (unsigned)p.B, (unsigned)p.H)
                                         : dim3((unsigned)slots, (unsigned)p.H);
    e = launch_kernel(pc_prep_kernel, pgrid, dim3(kPrepThreads), kPrepSmem, s, true, p);
    note_launch();
    if (e != cudaSuccess) return e;
    const long ctas = (long)pc_sm_count() * 2;
    const int grid = (int)(max_units < ctas ? max_units : ctas);
    if (grid <= 0) return cudaSuccess;  // (the prepare kernel ran: a segment pass may follow)
    e = p.seg_mode ? launch_kernel(pc_scan_kernel<true>, dim3(grid), dim3(kScanThreads), kScanSmem, s, true, p)
                   : launch_kernel(pc_scan_kernel<false>, dim3(grid), dim3(kScanThreads), kScanSmem, s, true, p);
    note_launch();
    return e;
}

cudaError_t launch_delta_chunked_pc_segmented(const PcParams &p0, const ChunkLaunch &c, cudaStream_t s) {
    if (c.nseq_seg < 1 || c.nseq_seg > kMaxSegSeqs) return cudaErrorInvalidValue;
    PcParams p = p0;
    p.nseq_seg = c.nseq_seg;
    for (int i = 0; i < kMaxSegSeqs; ++i) p.seg_seq[i] = c.seg_seq[i];
    for (int i = 0; i <= kMaxSegSeqs; ++i) {
        p.seg_m0[i] = c.seg_m0[i];
        p.seg_s0[i] = c.seg_s0[i];
    }
    p.seg_M = c.seg_M;
    p.seg_L = c.seg_L;
    p.seg_S = c.seg_S;
    // the prepare kernel (images of every chunk) and pass 1 (transitions and
    // local states of every segment but the last, from zero)
    p.seg_mode = 1;
    p.seg_units = c.seg_m0[c.nseq_seg] * p.H * (p.VT + 1);
    p.counter = &c.header->seg_next[0];
    cudaError_t e = launch_delta_chunked_pc(p, p.seg_units, s);
    if (e != cudaSuccess) return e;
    e = launch_segment_combine(c, s);
    if (e != cudaSuccess) return e;
    // pass 2: every segment from its start state, outputs and final states
    p.seg_mode = 2;
    p.seg_units = c.seg_s0[c.nseq_seg] * p.H * p.VT;
    p.counter = &c.header->seg_next[1];
    const long ctas = (long)pc_sm_count() * 2;
    const int grid = (int)(p.seg_units < ctas ? p.seg_units : ctas);
    if (grid <= 0) return cudaSuccess;
    e = launch_kernel(pc_scan_kernel<true>, dim3(grid), dim3(kScanThreads), kScanSmem, s, true, p);
    note_launch();
    return e;
}

}  // namespace gdn
