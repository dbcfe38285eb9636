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
// Per chunk and (sequence, value head, 128-row V tile) unit, on CUDA cores:
// the gates, norms, KK / QK, T, W, U and the scaled operands; on tcgen05
// (M = 128 state rows, bf16 operands, fp32 accumulators in tensor memory):
//   Dd = S0 W^T,  Do = S0 Qt^T   (S0 = bf16 copy of the state, N = 16)
//   Do += Delta^T P^T             (P = scale tril(QK), K = 16)
//   S  += Delta^T Kp              (S first scaled by e^{b_C} per column, N = 128)
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace gdn {

namespace {

using namespace sm100;

constexpr int kPc = 16;            // chunk length
constexpr int kPcThreads = 256;    // 8 warps; thread 0 issues the MMAs
constexpr uint64_t kPcWaitNs = 2000000000ull;  // bounded waits: 2 s

// Shared memory (offsets from a 1024-aligned base).  SW128 = rows of 128 bytes
// in the 128-byte swizzle the MMA descriptors read.
constexpr uint32_t kOS0 = 0;              // S0 bf16 [128 vi][128 kk]: two SW128 blocks of 16 KB
constexpr uint32_t kODt = 32768;          // Delta^T bf16 [128 vi][16 t] in an SW128 [128][64] tile
constexpr uint32_t kOW = 49152;           // W bf16 [16 t][128 kk]: two SW128 blocks of 2 KB
constexpr uint32_t kOQt = kOW + 4096;     // Qt bf16 [16 t][128 kk], same layout
constexpr uint32_t kOKp = kOQt + 4096;    // Kp bf16 [16 t][128 kk], same layout (MN-major B)
constexpr uint32_t kOP = kOKp + 4096;     // P bf16 [16 t][16 i] in an SW128 [16][64] tile
constexpr uint32_t kORawK = kOP + 2048;   // raw k rows bf16 [16][128]
constexpr uint32_t kORawQ = kORawK + 4096;
constexpr uint32_t kORawV = kORawQ + 4096;
constexpr uint32_t kOB = kORawV + 4096;   // logits, then cumulative log decays, fp32 [16][128]
constexpr uint32_t kOKt = kOB + 8192;     // Kt fp32 [16][128] (norm folded in)
constexpr uint32_t kOU = kOKt + 8192;     // U fp32 [16][128]
constexpr uint32_t kOKK = kOU + 8192;     // KK fp32 [16][16]
constexpr uint32_t kOQK = kOKK + 1024;    // QK fp32 [16][16]
constexpr uint32_t kOT = kOQK + 1024;     // T fp32 [16][16]
constexpr uint32_t kOVec = kOT + 1024;    // beta[16], rk[16], rq[16], colscale[128]
constexpr uint32_t kVecN = 16 * 3 + 128;
constexpr uint32_t kOBar = kOVec + kVecN * 4;
constexpr uint32_t kPcSmem = kOBar + 64 + 1024;  // + alignment slack
static_assert(kOBar % 8 == 0, "mbarrier alignment");
static_assert(kPcSmem <= 113 * 1024, "two CTAs per SM");

// TMEM: the state in columns [0, 128); Dd in [128, 144), Do in [144, 160).
constexpr uint32_t kPcTmemCols = 256;
constexpr uint32_t kColS = 0, kColDd = 128, kColDo = 144;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void st8(unsigned char *tile, int row, int c8, const float *v) {
    uint4 q;
    q.x = pack2(v[0], v[1]);
    q.y = pack2(v[2], v[3]);
    q.z = pack2(v[4], v[5]);
    q.w = pack2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, c8 * 8)) = q;
}
// element (row, col) of a [rows][128] bf16 operand kept as two SW128 blocks
// of [rows][64] that are `block` bytes apart
__device__ __forceinline__ void st_el(unsigned char *tile, uint32_t block, int row, int col, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(tile + (col >> 6) * block + sw128_offset(row, col & 63)) =
        __float2bfloat16_rn(v);
}

// Natural-log gate of one key channel from its input under the options:
// logits through the softplus gate (-exp(A_log) softplus(x + dt_bias)), the
// exp gate (x), or (gate_factor) the gate factor itself, log(max(x, 1e-30)).
__device__ __forceinline__ float log_gate(float x, float dtb, float alog, int opts, int gate_factor) {
    if (opts & GDN_OPT_NO_DECAY) return 0.f;
    if (gate_factor) return logf(fmaxf(x, 1e-30f));
    if (opts & GDN_OPT_GATE_EXP) return x;
    x += dtb;
    const float softplus = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
    return -expf(alog) * softplus;
}

__global__ void __launch_bounds__(kPcThreads, 2) chunked_pc_kernel(const PcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *v_beta = reinterpret_cast<float *>(sm + kOVec);
    float *v_rk = v_beta + 16, *v_rq = v_rk + 16, *v_cs = v_rq + 16;
    uint64_t *bar_mma = reinterpret_cast<uint64_t *>(sm + kOBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar_mma + 1);
    int *s_unit = reinterpret_cast<int *>(bar_mma + 2);
    int *s_abort = s_unit + 1;
    float *sB = reinterpret_cast<float *>(sm + kOB);
    float *sKt = reinterpret_cast<float *>(sm + kOKt);
    float *sU = reinterpret_cast<float *>(sm + kOU);
    float *sKK = reinterpret_cast<float *>(sm + kOKK);
    float *sQK = reinterpret_cast<float *>(sm + kOQK);
    float *sT = reinterpret_cast<float *>(sm + kOT);
    __nv_bfloat16 *rawK = reinterpret_cast<__nv_bfloat16 *>(sm + kORawK);
    __nv_bfloat16 *rawQ = reinterpret_cast<__nv_bfloat16 *>(sm + kORawQ);
    __nv_bfloat16 *rawV = reinterpret_cast<__nv_bfloat16 *>(sm + kORawV);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hc = warp >> 2;
    const int row = quad * 32 + lane;  // this thread's TMEM lane (state row)

    if (tid == 0) {
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kPcTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);

    pdl_wait_primary();  // everything below reads what the conv kernel wrote

    const int H = p.H, HQ = p.HQ, V = p.V, VT = p.VT;
    const int G = H / HQ;
    const int n_units = p.header->n_units;
    const int opts = p.opts;
    const float fr = (opts & GDN_OPT_NO_RETRIEVE) ? 0.f : 1.f;
    uint32_t mma_phase = 0;

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

    while (true) {
        if (tid == 0) *s_unit = (int)atomicAdd(&p.header->next_unit, 1u);
        __syncthreads();
        const int u = *s_unit;
        if (u >= n_units || *s_abort) break;
        const int seq = p.seq_order[u / (H * VT)];
        const int h = (u / VT) % H, vt = u % VT;
        const int s = p.offsets[seq], e = p.offsets[seq + 1];
        if (s < 0 || e < s || e > p.N) {  // malformed offsets: nothing is read or written
            __syncthreads();
            continue;
        }
        const int kh = h / G;
        const __nv_bfloat16 *qsrc = p.qb + (size_t)kh * 128;
        const __nv_bfloat16 *ksrc = p.kb + (size_t)kh * 128;
        const __nv_bfloat16 *vsrc = p.vb + (size_t)h * V + (size_t)vt * 128;
        const bool soft = !(opts & (GDN_OPT_NO_DECAY | GDN_OPT_GATE_EXP)) && !p.gate_factor;
        const float dtb = soft ? __ldg(p.dt_bias + h) : 0.f;
        const float alog = soft ? __ldg(p.A_log + h) : 0.f;
        const size_t state_row = ((size_t)seq * H + h) * V + (size_t)vt * 128 + row;

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

        const int nchunks = (e - s + kPc - 1) / kPc;
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int t0 = s + n * kPc;
            const int Cn = min(kPc, e - t0);

            // ---- L: raw k, q, v rows (16-byte vectors) and the gate inputs
            for (int i = tid; i < 3 * kPc * 16; i += kPcThreads) {
                const int tile = i >> 8, r = (i >> 4) & 15, c16 = i & 15;
                const __nv_bfloat16 *src = tile == 0 ? ksrc : tile == 1 ? qsrc : vsrc;
                __nv_bfloat16 *dst = tile == 0 ? rawK : tile == 1 ? rawQ : rawV;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < Cn) v = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)(t0 + r) * p.rs) + c16);
                *reinterpret_cast<uint4 *>(dst + r * 128 + c16 * 8) = v;
            }
            const bool decay = !(opts & GDN_OPT_NO_DECAY);
            for (int i = tid; i < kPc * 32; i += kPcThreads) {
                const int r = i >> 5, c4 = i & 31;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < Cn && decay)
                    v = __ldg(reinterpret_cast<const float4 *>(p.g + ((size_t)(t0 + r) * H + h) * 128) + c4);
                *reinterpret_cast<float4 *>(sB + r * 128 + c4 * 4) = v;
            }
            if (tid < kPc) {
                float be = 0.f;
                if (tid < Cn) {
                    be = 1.f;
                    if (!(opts & GDN_OPT_NO_BETA)) {
                        be = __ldg(p.bl + (size_t)(t0 + tid) * H + h);
                        if (!(opts & GDN_OPT_BETA_RAW)) be = 1.f / (1.f + expf(-be));
                    }
                }
                v_beta[tid] = be;
            }
            __syncthreads();

            // ---- G: cumulative log decays per channel (threads 0..127) and the
            // q/k norms (threads 128..255: 4 threads per (token, q|k))
            if (tid < 128) {
                float acc = 0.f;
#pragma unroll 4
                for (int t = 0; t < kPc; ++t) {
                    const float lg = t < Cn ? log_gate(sB[t * 128 + tid], dtb, alog, opts, p.gate_factor) : 0.f;
                    acc += lg;
                    sB[t * 128 + tid] = acc;
                }
                v_cs[tid] = expf(acc);  // e^{b_C}: the state's column decay over the chunk
            } else {
                const int idx = tid - 128, red = idx >> 2, part = idx & 3;
                const int t = red & 15;
                const __nv_bfloat16 *src = (red >> 4) ? rawQ : rawK;
                float ss = 0.f;
#pragma unroll 8
                for (int c = part * 32; c < part * 32 + 32; ++c) {
                    const float x = __bfloat162float(src[t * 128 + c]);
                    ss = fmaf(x, x, ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                if (part == 0) {
                    const float rn = (opts & GDN_OPT_NO_QK_NORM) ? 1.f : rsqrtf(ss + 1e-12f);
                    ((red >> 4) ? v_rq : v_rk)[t] = rn;
                }
            }
            __syncthreads();

            // ---- AP: KK and QK in 4x4-token blocks (threads 0..159: a half-warp
            // per block pair, a lane per 8 channels); the scaled operands
            // Kt, Qt, Kp (threads 160..255)
            if (tid < 160) {
                const int bp = tid >> 4, cg = tid & 15;
                // block pairs (T, I), I <= T
                const int TB = bp < 1 ? 0 : bp < 3 ? 1 : bp < 6 ? 2 : 3;
                const int IB = bp - (TB * (TB + 1)) / 2;
                float kk[4][4], qk[4][4];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) kk[a][b] = qk[a][b] = 0.f;
#pragma unroll 2
                for (int j = 0; j < 8; ++j) {
                    const int c = cg * 8 + j;
                    float kt[4], qt[4], ki[4], bt[4], bi[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        kt[a] = __bfloat162float(rawK[(4 * TB + a) * 128 + c]);
                        qt[a] = __bfloat162float(rawQ[(4 * TB + a) * 128 + c]);
                        ki[a] = __bfloat162float(rawK[(4 * IB + a) * 128 + c]);
                        bt[a] = sB[(4 * TB + a) * 128 + c];
                        bi[a] = sB[(4 * IB + a) * 128 + c];
                    }
                    if (TB > IB) {
                        const float ref = bi[3];
                        float xk[4], xq[4], y[4];
#pragma unroll
                        for (int a = 0; a < 4; ++a) {
                            const float ft = __expf(bt[a] - ref);
                            xk[a] = kt[a] * ft;
                            xq[a] = qt[a] * ft;
                            y[a] = ki[a] * __expf(ref - bi[a]);
                        }
#pragma unroll
                        for (int a = 0; a < 4; ++a)
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                kk[a][b] = fmaf(xk[a], y[b], kk[a][b]);
                                qk[a][b] = fmaf(xq[a], y[b], qk[a][b]);
                            }
                    } else {
#pragma unroll
                        for (int a = 0; a < 4; ++a)
#pragma unroll
                            for (int b = 0; b <= a; ++b) {
                                const float y = ki[b] * __expf(bt[a] - bi[b]);
                                if (b < a) kk[a][b] = fmaf(kt[a], y, kk[a][b]);
                                qk[a][b] = fmaf(qt[a], y, qk[a][b]);
                            }
                    }
                }
                // sum over the 16 channel groups of the half-warp
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b)
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1) {
                            kk[a][b] += __shfl_xor_sync(0xffffffffu, kk[a][b], o);
                            qk[a][b] += __shfl_xor_sync(0xffffffffu, qk[a][b], o);
                        }
                if (cg == 0) {
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const int t = 4 * TB + a, i = 4 * IB + b;
                            sKK[t * 16 + i] = kk[a][b];
                            sQK[t * 16 + i] = qk[a][b];
                        }
                }
            } else {
                for (int idx = tid - 160; idx < kPc * 128; idx += kPcThreads - 160) {
                    const int t = idx >> 7, c = idx & 127;
                    const float bt = sB[t * 128 + c], bC = sB[(kPc - 1) * 128 + c];
                    const float kr = __bfloat162float(rawK[t * 128 + c]) * v_rk[t];
                    const float qr = __bfloat162float(rawQ[t * 128 + c]) * v_rq[t] * p.scale;
                    const float et = __expf(bt);
                    sKt[t * 128 + c] = kr * et;
                    st_el(sm + kOQt, 2048, t, c, qr * et);
                    st_el(sm + kOKp, 2048, t, c, kr * __expf(bC - bt));
                }
            }
            __syncthreads();

            // ---- T = (I + A)^-1 with A[t,i] = beta_t rk_t rk_i KK[t,i] (i < t):
            // forward substitution, one column per lane (warp 0); the other
            // warps write P[t,i] = scale rq_t rk_i QK[t,i] (i <= t) as bf16
            if (warp == 0) {
                if (lane < 16) {
                    const int c = lane;
                    float pr[16], tc[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) pr[r] = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        tc[i] = (i == c) ? 1.f : (i > c ? -pr[i] : 0.f);
#pragma unroll
                        for (int r = i + 1; r < 16; ++r)
                            pr[r] = fmaf(fr * v_beta[r] * v_rk[r] * v_rk[i] * sKK[r * 16 + i], tc[i], pr[r]);
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) sT[r * 16 + c] = tc[r];
                }
            } else if (tid < 32 + kPc * 2) {
                // row t = (tid - 32) >> 1, eight columns per thread
                const int q = tid - 32, t = q >> 1, c8 = q & 1;
                float v8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = c8 * 8 + j;
                    v8[j] = i <= t ? p.scale * v_rq[t] * v_rk[i] * sQK[t * 16 + i] : 0.f;
                }
                st8(sm + kOP, t, c8, v8);
            }
            __syncthreads();

            // ---- W = T diag(beta) Kt (bf16 operand), U = T diag(beta) V (fp32);
            // then the state's bf16 copy S0 and its column decay S *= e^{b_C}
            for (int idx = tid; idx < 2 * kPc * 128; idx += kPcThreads) {
                const int which = idx >> 11, t = (idx >> 7) & 15, c = idx & 127;
                float acc = 0.f;
                if (which == 0) {
#pragma unroll
                    for (int s2 = 0; s2 < kPc; ++s2)
                        acc = fmaf(sT[t * 16 + s2] * v_beta[s2], sKt[s2 * 128 + c], acc);
                    st_el(sm + kOW, 2048, t, c, fr * acc);
                } else {
#pragma unroll
                    for (int s2 = 0; s2 < kPc; ++s2)
                        acc = fmaf(sT[t * 16 + s2] * v_beta[s2], __bfloat162float(rawV[s2 * 128 + c]), acc);
                    sU[t * 128 + c] = acc;
                }
            }
            {
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
                    for (int j = 0; j < 32; ++j)
                        r[j] = __float_as_uint(v[j] * v_cs[hc * 64 + c0 + j]);
                    tmem_st32(lane_base + kColS + hc * 64 + c0, r);
                }
                tmem_wait_st();
            }
            fence_async_smem();
            sync_all();

            // ---- Dd = S0 W^T, Do = S0 Qt^T (M = 128, N = 16, K = 128)
            if (tid == 0) {
                const uint32_t s0 = smem_u32(sm + kOS0), w = smem_u32(sm + kOW);
                const uint32_t qt = smem_u32(sm + kOQt);
                const uint32_t id = idesc_bf16(128, 16, false, false);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
                    const uint32_t bo = (ks >> 2) * 2048 + (ks & 3) * 32;
                    mma_bf16(tmem + kColDd, sdesc_sw128(s0 + ao, 16, 1024), sdesc_sw128(w + bo, 16, 1024),
                             id, ks > 0);
                    mma_bf16(tmem + kColDo, sdesc_sw128(s0 + ao, 16, 1024), sdesc_sw128(qt + bo, 16, 1024),
                             id, ks > 0);
                }
                mma_commit(bar_mma);
            }
            wait_mma();

            // ---- Delta^T[vi, t] = U[t, vi] - Dd[vi, t] -> bf16 A operand (warps 0..3)
            if (hc == 0) {
                uint32_t r[16];
                tmem_ld16(lane_base + kColDd, r);
                tmem_wait_ld();
                float d[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) d[t] = sU[t * 128 + row] - __uint_as_float(r[t]);
                st8(sm + kODt, row, 0, d);
                st8(sm + kODt, row, 1, d + 8);
            }
            fence_async_smem();
            sync_all();

            // ---- Do += Delta^T P^T (K = 16);  S += Delta^T Kp (N = 128, K = 16)
            if (tid == 0) {
                const uint32_t dt = smem_u32(sm + kODt), pp = smem_u32(sm + kOP);
                const uint32_t kp = smem_u32(sm + kOKp);
                mma_bf16(tmem + kColDo, sdesc_sw128(dt, 16, 1024), sdesc_sw128(pp, 16, 1024),
                         idesc_bf16(128, 16, false, false), 1);
                mma_bf16(tmem + kColS, sdesc_sw128(dt, 16, 1024), sdesc_sw128(kp, 2048, 1024),
                         idesc_bf16(128, 128, false, true), 1);
                mma_commit(bar_mma);
            }
            wait_mma();

            // ---- output rows t < Cn (warps 0..3; a warp writes 32 consecutive values of a row)
            if (hc == 0) {
                uint32_t r[16];
                tmem_ld16(lane_base + kColDo, r);
                tmem_wait_ld();
                __nv_bfloat16 *obase = p.out + (size_t)t0 * p.ors + (size_t)h * V + (size_t)vt * 128 + row;
                for (int t = 0; t < Cn; ++t)
                    obase[(size_t)t * p.ors] = __float2bfloat16_rn(__uint_as_float(r[t]));
            }
            sync_all();
            if (*s_abort) break;
        }
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

    if (*s_abort && tid == 0) {
        // a bounded wait gave up: record it and give MMAs still in flight time
        // to land before the tensor memory is released
        atomicExch(&p.header->status, 7 /* GDN_ERR_TIMEOUT */);
        const uint64_t ts = global_timer_ns();
        while (global_timer_ns() - ts < 10000000ull) {  // 10 ms
        }
    }
    sync_all();
    if (warp == 0) tmem_dealloc(tmem, kPcTmemCols);
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
        return cudaFuncSetAttribute(chunked_pc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kPcSmem);
    });
    if (e != cudaSuccess) return e;
    const long slots = (long)pc_sm_count() * 2;
    const int grid = (int)(max_units < slots ? max_units : slots);
    if (grid <= 0) return cudaSuccess;
    e = launch_kernel(chunked_pc_kernel, dim3(grid), dim3(kPcThreads), kPcSmem, s, true, p);
    note_launch();
    return e;
}

}  // namespace gdn
