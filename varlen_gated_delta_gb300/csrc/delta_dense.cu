// delta_dense.cu - the gated delta rule on the dense layout of the
// GatedDeltaNet CPU thunk (rlx-cpu thunk/types.rs): q, k, v [b, s, h, n],
// g [b, s, h] or, with gate_per_channel, [b, s, h, n] (per key channel), beta
// [b, s, h], state [b, h, n, n] resumed from and written back when carried.
//
// The thunk defers its math to an operator that is not on the page; this
// kernel applies the DELTA kernel of paged_ssm.rs (onnxruntime-ep-mlx 0.31.1)
// to the given values: per state row S[vi, :] and token in order,
//   S <- S diag(g) (a scalar g decays the whole row);  r = S.k;
//   delta = beta (v[vi] - r);  S <- S + delta k;  o[vi] = scale S.q
// with q, k, g and beta used as given (no convolution, no normalisation).
//
// GB300 design: as the token-serial varlen kernel, a warp owns 8 state rows
// in registers for the whole sequence (16 fp32 per lane, n/16 lanes a row);
// the two dot products of a token are reduced by one xor-shuffle tree.
#include "common.cuh"
#include "sm100.cuh"

namespace gdn {

namespace {

constexpr int kDenseThreads = 128;

// VEC4: n % 4 == 0 and 16-byte aligned states (state rows move as float4).
// The scalar-gate instance with n = 128 is held to six CTAs per SM (80
// registers; it took 96 and ran five): dense decode 49.4 -> 47.2 us a step.
// The per-channel instance takes 80 registers unbounded; bounded it spilled
// and ran 47.2 -> 50.4 us.  (A minimum of 0 CTAs leaves the bound unset.)
template <typename T, int KP, int RG, bool PERCH, bool VEC4>
__global__ void __launch_bounds__(kDenseThreads, (KP == 128 && !PERCH) ? 6 : 0)
    delta_dense_kernel(const DenseParams p) {
    constexpr int EPL = 16;           // state values per lane per row
    constexpr int LPR = KP / EPL;     // lanes per row
    constexpr int RPI = 32 / LPR;     // rows per warp per row group
    constexpr int ROWS_W = RPI * RG;  // rows per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPR, rlane = lane / LPR;
    const int n = p.n, H = p.H, S = p.S;
    const int rows_cta = (blockDim.x >> 5) * ROWS_W;
    const int nrb = (n + rows_cta - 1) / rows_cta;
    long blk = blockIdx.x;
    const int rb = (int)(blk % nrb);
    blk /= nrb;
    const int h = (int)(blk % H);
    const int b = (int)(blk / H);

    int kidx[4];  // this lane's key columns: 4-float blocks (sub + LPR m)
#pragma unroll
    for (int m = 0; m < 4; ++m) kidx[m] = 4 * (sub + LPR * m);
    int vi[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) vi[r] = rb * rows_cta + warp * ROWS_W + r * RPI + rlane;

    float st[RG][EPL];
    const size_t head = ((size_t)b * H + h) * n;  // state rows of (b, h)
#pragma unroll
    for (int r = 0; r < RG; ++r)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const bool in = p.state_init != nullptr && vi[r] < n;
            if constexpr (VEC4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (in && kidx[m] < n)
                    x = *reinterpret_cast<const float4 *>(p.state_init + (head + vi[r]) * n + kidx[m]);
                st[r][4 * m] = x.x; st[r][4 * m + 1] = x.y; st[r][4 * m + 2] = x.z; st[r][4 * m + 3] = x.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int kk = kidx[m] + u;
                    st[r][4 * m + u] = (in && kk < n) ? p.state_init[(head + vi[r]) * n + kk] : 0.f;
                }
            }
        }

    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    T *out = static_cast<T *>(p.out);
    for (int t = 0; t < S; ++t) {
        const size_t row = ((size_t)b * S + t) * H + h;  // token-head row of [b, s, h, .]
        float qc[EPL], kc[EPL], gc[PERCH ? EPL : 1];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int kk = kidx[m] + u;
                qc[4 * m + u] = kk < n ? to_f32(q[row * n + kk]) : 0.f;
                kc[4 * m + u] = kk < n ? to_f32(k[row * n + kk]) : 0.f;
                if constexpr (PERCH) gc[4 * m + u] = kk < n ? __ldg(p.g + row * n + kk) : 1.f;
            }
        if constexpr (!PERCH) gc[0] = __ldg(p.g + row);
        const float bt = __ldg(p.beta + row);
        float kq = 0.f;
#pragma unroll
        for (int u = 0; u < EPL; ++u) kq = fmaf(kc[u], qc[u], kq);
        kq = group_sum<LPR>(kq);

        float sk[RG], sq[RG];
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int u = 0; u < EPL; ++u) {
                st[r][u] *= gc[PERCH ? u : 0];  // decay first: retrieval reads the decayed state
                a0 = fmaf(st[r][u], kc[u], a0);
                a1 = fmaf(st[r][u], qc[u], a1);
            }
            sk[r] = a0;
            sq[r] = a1;
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) {
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                sk[r] += __shfl_xor_sync(0xffffffffu, sk[r], off);
                sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], off);
            }
        }
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const float vv = vi[r] < n ? to_f32(v[row * n + vi[r]]) : 0.f;
            const float delta = bt * (vv - sk[r]);
            // read-out of the updated row: (S + delta k).q = S.q + delta (k.q)
            const float o = sq[r] + delta * kq;
#pragma unroll
            for (int u = 0; u < EPL; ++u) st[r][u] = fmaf(delta, kc[u], st[r][u]);
            if (sub == 0 && vi[r] < n) out[row * n + vi[r]] = from_f32<T>(o * p.scale);
        }
    }
    if (p.state_fin == nullptr) return;
#pragma unroll
    for (int r = 0; r < RG; ++r)
        if (vi[r] < n)
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float *dst = p.state_fin + (head + vi[r]) * n + kidx[m];
                if constexpr (VEC4) {
                    if (kidx[m] < n)  // streaming store: not read again by this call
                        __stcs(reinterpret_cast<float4 *>(dst),
                               make_float4(st[r][4 * m], st[r][4 * m + 1], st[r][4 * m + 2], st[r][4 * m + 3]));
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (kidx[m] + u < n) dst[u] = st[r][4 * m + u];
                }
            }
}

template <typename T, int KP, int RG>
cudaError_t launch_dense_kp(const DenseParams &p, cudaStream_t s) {
    constexpr int ROWS_W = (32 / (KP / 16)) * RG;
    const int rows_cta = (kDenseThreads / 32) * ROWS_W;
    const long nrb = (p.n + rows_cta - 1) / rows_cta;
    const long blocks = (long)p.B * p.H * nrb;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks), block(kDenseThreads);
    const bool vec4 = p.n % 4 == 0 && ((uintptr_t)p.state_init % 16 == 0) &&
                      ((uintptr_t)p.state_fin % 16 == 0);
    cudaError_t e;
    if (vec4)
        e = p.per_channel ? launch_kernel(delta_dense_kernel<T, KP, RG, true, true>, grid, block, 0, s, false, p)
                          : launch_kernel(delta_dense_kernel<T, KP, RG, false, true>, grid, block, 0, s, false, p);
    else
        e = p.per_channel ? launch_kernel(delta_dense_kernel<T, KP, RG, true, false>, grid, block, 0, s, false, p)
                          : launch_kernel(delta_dense_kernel<T, KP, RG, false, false>, grid, block, 0, s, false, p);
    note_launch();
    return e;
}

template <typename T>
cudaError_t launch_dense_t(const DenseParams &p, cudaStream_t s) {
    if (p.n <= 16) return launch_dense_kp<T, 16, 1>(p, s);
    if (p.n <= 32) return launch_dense_kp<T, 32, 1>(p, s);
    if (p.n <= 64) return launch_dense_kp<T, 64, 1>(p, s);
    if (p.n <= 128) return launch_dense_kp<T, 128, 2>(p, s);
    return launch_dense_kp<T, 256, 4>(p, s);
}

// Prepares the dense layout for the chunked kernel (see DensePack): the log
// gates, and block 0 copies the three operand maps to global memory and writes
// the schedule.
__global__ void __launch_bounds__(256) dense_pack_kernel(const __grid_constant__ DensePack p) {
    const long N = (long)p.B * p.S;
    const long stride = (long)gridDim.x * blockDim.x;
    const long i0 = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (p.a != nullptr)  // (the per-channel route reads the gate factors itself)
        for (long i = i0; i < N * p.H; i += stride) p.a[i] = logf(fmaxf(__ldg(p.g + i), 1e-30f));
    if (blockIdx.x == 0) {
        if (p.maps_dst != nullptr) {
            // 3 maps x 128 bytes as 8-byte words
            const uint64_t *src = reinterpret_cast<const uint64_t *>(p.maps);
            uint64_t *dst = static_cast<uint64_t *>(p.maps_dst);
            if (threadIdx.x < 3 * sizeof(CUtensorMap) / 8) dst[threadIdx.x] = src[threadIdx.x];
            sm100::tensormap_release();
        }
        for (int i = threadIdx.x; i <= p.B; i += blockDim.x) p.offsets[i] = i * p.S;
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) p.order[i] = i;
        if (threadIdx.x == 0) {
            p.header->status = 0;
            p.header->n_serial = 0;
            p.header->n_chunked = p.B;
            p.header->n_units = p.B * p.H * (p.n / 128);
            p.header->next_unit = 0;
            p.header->seg_next[0] = p.header->seg_next[1] = 0;
        }
    }
}

}  // namespace

cudaError_t launch_dense_pack(const DensePack &p, cudaStream_t s) {
    const long work = p.a != nullptr ? (long)p.B * p.S * p.H : 1;
    long blocks = (work + 255) / 256;
    blocks = blocks < 1 ? 1 : (blocks > 4L * 152 * 8 ? 4L * 152 * 8 : blocks);
    dense_pack_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_delta_dense(const DenseParams &p, int dtype, cudaStream_t s) {
    if (dtype == 1) return launch_dense_t<__nv_bfloat16>(p, s);
    return launch_dense_t<float>(p, s);
}

}  // namespace gdn
