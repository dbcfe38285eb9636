// delta_serial.cu - token-serial gated delta recurrence (decode and short
// sequences).
//
// Operation: paged_ssm.rs (onnxruntime-ep-mlx 0.31.1), DELTA kernel: per state
// row S[vi,:] of (sequence b, value head h) and per token t in order,
//   S <- g S;  r = S.k;  delta = beta (v - r);  S <- S + delta k;  o = scale S.q
// with k, q the normalised key/query of key head kh = h / (H/HQ).
//
// GB300 design.  The state is streamed through HBM exactly once per call: a
// warp owns a set of state rows and keeps them in registers for the whole
// sequence.  Each row is split over LPR = KP/16 lanes holding 16 fp32 values
// (four 16-byte loads), so the two dot products a row needs per token,
// S_old.k and S_old.q, are reduced with log2(LPR) xor-shuffles for LPR rows at
// once.  Using S_old.q instead of S_new.q, the read-out is
//   o = scale (g (S_old.q) + delta (k.q)),
// which is the same quantity (S_new = g S_old + delta k^T) with one shuffle
// tree per token instead of two dependent ones; k.q is shared by all rows.
// The next token's q/k/g/beta/v are prefetched while the current one is
// applied.
#include "common.cuh"

namespace gdn {

namespace {

constexpr int kSerialThreads = 128;

// Final conv state of sequence b for the channel slice `slice` of `nslices`:
// fin[b,c,j] = x~(len - L + j), and the conv capture rows when asked for.  One thread per channel walks j upward and
// reads index len + j >= j of its own row before writing index j, so the
// final state may alias the initial one.
// BATCH: read all L values of a channel before writing any (L <= 8), so the
// loads overlap (the per-channel and capture decode instances: 9% and 6%
// faster; the plain decode instance, held to 80 registers, ran 3% slower
// with it and keeps one value at a time).
template <typename T, bool BATCH>
__device__ void conv_final_slice(const DeltaParams &p, int b, int s, int e, int slice,
                                 int nslices, size_t C) {
    const int L = p.conv_L;
    const int len = e - s;
    const size_t cs = (C + nslices - 1) / nslices;
    const size_t c0 = (size_t)slice * cs;
    const size_t c1 = c0 + cs < C ? c0 + cs : C;
    const T *x = static_cast<const T *>(p.conv_x);
    const T *init = static_cast<const T *>(p.conv_init);
    T *fin = static_cast<T *>(p.conv_fin);
    for (size_t c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
        if (fin != nullptr) {
            const T *irow = init + ((size_t)b * C + c) * L;
            T *frow = fin + ((size_t)b * C + c) * L;
            if (BATCH && L <= 8) {  // all reads before the first write: the loads overlap
                T v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int local = len - L + j;
                    if (j < L) v[j] = local >= 0 ? x[(size_t)(s + local) * C + c] : irow[L + local];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < L) frow[j] = v[j];
            } else {
                for (int j = 0; j < L; ++j) {
                    const int local = len - L + j;
                    const T v = local >= 0 ? x[(size_t)(s + local) * C + c] : irow[L + local];
                    frow[j] = v;
                }
            }
        }
        if (p.conv_updates != nullptr) {  // CONV_CAPTURE: first raw input rows, zero beyond
            const int n = captured_tokens(p.counts, nullptr, p.cap, b, len);
            T *upd = static_cast<T *>(p.conv_updates) + (size_t)b * p.cap * C + c;
            for (int i = 0; i < p.cap; ++i)
                upd[(size_t)i * C] = i < n ? x[(size_t)(s + i) * C + c] : from_f32<T>(0.f);
        }
    }
}

// PF: prefetch the next token's operands while applying the current one
// (sequences of several tokens); without it (one token per sequence, decode)
// the kernel needs fewer registers and more CTAs keep state loads in flight.
// CAPT: write the compact capsule of the first captured tokens (and run the
// captured prefix of sequences owned by the chunked kernel, outputs untouched).
// PC: per-key-channel gate (GDN_OPT_GATE_PER_CHANNEL): each lane decays its 16
// key columns by their own gates, S <- S diag(g); with the decayed directions
// g.k and g.q the retrieval and read-out are S_old.(g.k) and S_old.(g.q).
// The plain one-token (decode) variant with K = 128 is held to 80 registers so
// that six CTAs share an SM: more state loads in flight per SM (measured on the
// decode batch: 51.2 us a step against 52.8 us at five CTAs and 53.7 us at
// seven, where spills grow); its per-channel-gate and capture twins are held to
// five (96 registers; the capture twin unbounded took 144 registers, three
// CTAs per SM, and ran the capture-8 decode batch at 84 us against 63.5 us).
// The prefetching variants take the registers they want: held to three or four
// CTAs per SM they ran 6-19% slower.
template <typename T, int KP, int RG, bool VEC4, bool PF, bool CAPT, bool PC = false>
__global__ void __launch_bounds__(kSerialThreads, (!PF && KP == 128) ? (CAPT ? 5 : (PC ? 5 : 6)) : 1)
    delta_serial_kernel(const DeltaParams p) {
    // the next kernel of the stream (the following call's conv pass, which
    // waits for this grid before it reads anything) may be placed while this
    // grid's last CTAs run
    pdl_launch_dependents();
    constexpr int EPL = 16;          // state values per lane per row
    constexpr int LPR = KP / EPL;    // lanes per row
    constexpr int RPI = 32 / LPR;    // rows per warp per row group
    constexpr int ROWS_W = RPI * RG; // rows per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPR, rlane = lane / LPR;
    const int rows_cta = (blockDim.x >> 5) * ROWS_W;
    const int nrb = (p.V + rows_cta - 1) / rows_cta;
    const int K = p.K, V = p.V, H = p.H, HQ = p.HQ, N = p.N;

    long blk = blockIdx.x;
    const int rb = (int)(blk % nrb);
    blk /= nrb;
    const int h = (int)(blk % H);
    const int b = (int)(blk / H);
    int s, e;
    if (!seq_bounds(p.offsets, p.B, N, b, s, e)) return;
    const bool own = e - s < p.serial_max_len;  // else owned by the chunked kernel
    const int kh = h / (H / HQ);
    const size_t W = (size_t)2 * HQ * K + (size_t)H * V;

    // this lane's K columns: float4 blocks (sub + LPR*m), m = 0..3
    int kidx[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) kidx[m] = 4 * (sub + LPR * m);

    int vi[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) vi[r] = rb * rows_cta + warp * ROWS_W + r * RPI + rlane;

    auto load4 = [&](const float *base, int k0, float *dst) {
        if constexpr (VEC4) {
            if (k0 < K) {
                const float4 v = *reinterpret_cast<const float4 *>(base + k0);
                dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
            } else {
                dst[0] = dst[1] = dst[2] = dst[3] = 0.f;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) dst[u] = (k0 + u < K) ? base[k0 + u] : 0.f;
        }
    };
    auto store4 = [&](float *base, int k0, const float *src) {
        if constexpr (VEC4) {
            if (k0 < K)  // streaming store: the state is not read again by this call
                __stcs(reinterpret_cast<float4 *>(base + k0), make_float4(src[0], src[1], src[2], src[3]));
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (k0 + u < K) base[k0 + u] = src[u];
        }
    };

    // captured tokens (CAPT; counts and active are inputs of the call, not of
    // the previous kernel, so they are read before the dependency wait)
    const int ncap = CAPT ? captured_tokens(p.counts, p.active, p.cap, b, e - s) : 0;
    float S[RG][EPL];
    const size_t head_base = ((size_t)b * H + h) * V;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        if ((own || ncap > 0) && vi[r] < V) {
            const float *row = p.state_init + (head_base + vi[r]) * K;
#pragma unroll
            for (int m = 0; m < 4; ++m) load4(row, kidx[m], &S[r][4 * m]);
        } else {
#pragma unroll
            for (int u = 0; u < EPL; ++u) S[r][u] = 0.f;
        }
    }

    // The state loads above are in flight; everything below reads what the
    // conv/prepare kernel wrote (when launched as its PDL dependent).
    pdl_wait_primary();
    if (p.conv_fin != nullptr || p.conv_updates != nullptr)
        conv_final_slice<T, PC || CAPT>(p, b, s, e, h * nrb + rb, H * nrb, W);

    // capsule blocks of this sequence (CAPT): g [cap][H], k [cap][HQ][K], delta [cap][H][V]
    float *cap_g = nullptr, *cap_k = nullptr, *cap_d = nullptr;
    const bool key_owner = rb == 0 && warp == 0 && rlane == 0 && h == kh * (H / HQ);
    if constexpr (CAPT) {
        const int cap = p.cap;
        float *base = p.capsule + (size_t)b * cap * ((size_t)H + (size_t)HQ * K + (size_t)H * V);
        cap_g = base;
        cap_k = base + (size_t)cap * H;
        cap_d = base + (size_t)cap * (H + (size_t)HQ * K);
        // slots past the captured prefix are zero (the whole block writes them,
        // consecutive threads on consecutive floats)
        const int nz = cap - ncap, tid = threadIdx.x, nt = blockDim.x;
        for (int q = tid; q < nz * rows_cta; q += nt) {
            const int i = ncap + q / rows_cta, row = rb * rows_cta + q % rows_cta;
            if (row < V) cap_d[((size_t)i * H + h) * V + row] = 0.f;
        }
        if (rb == 0) {
            for (int q = tid; q < nz; q += nt) cap_g[(size_t)(ncap + q) * H + h] = 0.f;
            if (h == kh * (H / HQ))
                for (int q = tid; q < nz * K; q += nt)
                    cap_k[((size_t)(ncap + q / K) * HQ + kh) * K + q % K] = 0.f;
        }
    }
    if (!own && ncap == 0) return;
    // the chunked kernel owns the outputs and final state of long sequences:
    // only their captured prefix runs here
    const int t_end = own ? e : s + ncap;

    const T *y = static_cast<const T *>(p.y);
    T *out = static_cast<T *>(p.out);
    const float scale = p.scale;
    const bool retrieve = !(p.opts & GDN_OPT_NO_RETRIEVE);

    float qc[EPL], kc[EPL], vc[RG], gc = 1.f, bc = 0.f;
    float gcv[EPL];  // per-channel gates of the lane's columns (PC)
    const float pc_dtb = PC && p.gpc_logits && p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    const float pc_alog = PC && p.gpc_logits && p.A_log ? __ldg(p.A_log + h) : 0.f;
    // PC with decay logits: the CTA activates each key column's gate once per
    // token into shared memory (double-buffered by token parity) instead of
    // every lane that holds the column doing it; every thread of the CTA walks
    // the same tokens, so the barrier is uniform.
    __shared__ __align__(16) float s_gate[PC ? 2 * KP : 4];
    auto fetch = [&](int t, float *q, float *k, float *v, float &g, float &beta, float *gv) {
        const float *qrow = p.qk + ((size_t)t * HQ + kh) * K;
        const float *krow = p.qk + (((size_t)N + t) * HQ + kh) * K;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            load4(qrow, kidx[m], &q[4 * m]);
            load4(krow, kidx[m], &k[4 * m]);
        }
        if constexpr (PC) {
            const float *grow = p.gpc + ((size_t)t * H + h) * K;
            if (p.gpc_logits) {
                float *sg = s_gate + (t & 1) * KP;
                for (int i = threadIdx.x; i < KP; i += blockDim.x)
                    sg[i] = i < K ? gate_of_logit(__ldg(grow + i), pc_dtb, pc_alog, p.opts) : 0.f;
                __syncthreads();
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(sg + kidx[m]);
                    gv[4 * m] = g4.x;
                    gv[4 * m + 1] = g4.y;
                    gv[4 * m + 2] = g4.z;
                    gv[4 * m + 3] = g4.w;
                }
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) load4(grow, kidx[m], &gv[4 * m]);
            }
            g = 1.f;
            beta = __ldg(p.beta_base + (size_t)t * H + h);
        } else {
            g = __ldg(p.gb + (size_t)t * H + h);
            beta = __ldg(p.gb + ((size_t)N + t) * H + h);
        }
        const T *vrow = y + (size_t)t * W + (size_t)2 * HQ * K + (size_t)h * V;
#pragma unroll
        for (int r = 0; r < RG; ++r) v[r] = vi[r] < V ? to_f32(vrow[vi[r]]) : 0.f;
    };
    if (s < t_end) fetch(s, qc, kc, vc, gc, bc, gcv);

    for (int t = s; t < t_end; ++t) {
        float qn[PF ? EPL : 1], kn[PF ? EPL : 1], vn[RG], gn = 1.f, bn = 0.f;
        float gvn[EPL];
        if constexpr (PF) {
            if (t + 1 < t_end) fetch(t + 1, qn, kn, vn, gn, bn, gvn);
        }
        // per-channel gate: the state's key columns are decayed first, each by
        // its own gate; retrieval and read-out then use the decayed state
        // With PF (runs of tokens) the column pairs below take the packed fp32
        // pipe (each component rounds exactly as the scalar multiply / fused
        // multiply-add): measured 10% faster there, and 4% slower on the
        // one-token decode instances, which keep the scalar form.
        if constexpr (PC) {
#pragma unroll
            for (int r = 0; r < RG; ++r)
#pragma unroll
                for (int u = 0; u < EPL; u += 2) {
                    if constexpr (PF) {
                        const float2 d2 = __fmul2_rn(make_float2(S[r][u], S[r][u + 1]),
                                                     make_float2(gcv[u], gcv[u + 1]));
                        S[r][u] = d2.x;
                        S[r][u + 1] = d2.y;
                    } else {
                        S[r][u] *= gcv[u];
                        S[r][u + 1] *= gcv[u + 1];
                    }
                }
        }

        float kq = 0.f;
#pragma unroll
        for (int u = 0; u < EPL; ++u) kq = fmaf(kc[u], qc[u], kq);
        kq = group_sum<LPR>(kq);

        float sk[RG], sq[RG];
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            if constexpr (PF) {
                float2 a = make_float2(0.f, 0.f);  // the S k and S q chains side by side
#pragma unroll
                for (int u = 0; u < EPL; ++u)
                    a = __ffma2_rn(make_float2(S[r][u], S[r][u]), make_float2(kc[u], qc[u]), a);
                sk[r] = a.x;
                sq[r] = a.y;
            } else {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int u = 0; u < EPL; ++u) {
                    a0 = fmaf(S[r][u], kc[u], a0);
                    a1 = fmaf(S[r][u], qc[u], a1);
                }
                sk[r] = a0;
                sq[r] = a1;
            }
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) {
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                sk[r] += __shfl_xor_sync(0xffffffffu, sk[r], off);
                sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], off);
            }
        }
        const int slot = t - s;
        if constexpr (CAPT) {
            if (slot < ncap) {  // DELTA_CAPTURE_STEP: g and the normalised k of this token
                if (rb == 0 && warp == 0 && lane == 0) cap_g[(size_t)slot * H + h] = gc;
                if (key_owner)
#pragma unroll
                    for (int m = 0; m < 4; ++m)
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (kidx[m] + u < K)
                                cap_k[((size_t)slot * HQ + kh) * K + kidx[m] + u] = kc[4 * m + u];
            }
        }
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            // RETRIEVE (delta rules): subtract the decayed state's retrieval S k
            // (with the per-channel gate gc = 1: S is already decayed)
            const float delta = bc * (retrieve ? vc[r] - gc * sk[r] : vc[r]);
            const float o = gc * sq[r] + delta * kq;
            if constexpr (PF) {
#pragma unroll
                for (int u = 0; u < EPL; u += 2) {
                    const float2 s2 = make_float2(S[r][u], S[r][u + 1]), k2 = make_float2(kc[u], kc[u + 1]);
                    const float2 d2 = make_float2(delta, delta);
                    const float2 n2 = PC ? __ffma2_rn(d2, k2, s2)
                                         : __ffma2_rn(make_float2(gc, gc), s2, __fmul2_rn(d2, k2));
                    S[r][u] = n2.x;
                    S[r][u + 1] = n2.y;
                }
            } else {
#pragma unroll
                for (int u = 0; u < EPL; ++u)
                    S[r][u] = PC ? S[r][u] + delta * kc[u] : fmaf(gc, S[r][u], delta * kc[u]);
            }
            if (sub == 0 && vi[r] < V) {
                if (own) out[((size_t)t * H + h) * V + vi[r]] = from_f32<T>(o * scale);
                if constexpr (CAPT) {
                    if (slot < ncap) cap_d[((size_t)slot * H + h) * V + vi[r]] = delta;
                }
            }
        }
        if (t + 1 < t_end) {
            if constexpr (PF) {
#pragma unroll
                for (int u = 0; u < EPL; ++u) {
                    qc[u] = qn[u];
                    kc[u] = kn[u];
                }
#pragma unroll
                for (int r = 0; r < RG; ++r) vc[r] = vn[r];
                gc = gn;
                bc = bn;
                if constexpr (PC) {
#pragma unroll
                    for (int u = 0; u < EPL; ++u) gcv[u] = gvn[u];
                }
            } else {
                fetch(t + 1, qc, kc, vc, gc, bc, gcv);
            }
        }
    }

    if (!own) return;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        if (vi[r] < V) {
            float *row = p.state_fin + (head_base + vi[r]) * K;
#pragma unroll
            for (int m = 0; m < 4; ++m) store4(row, kidx[m], &S[r][4 * m]);
        }
    }
}

template <typename T, int KP, int RG>
cudaError_t launch_serial_kp(const DeltaParams &p, bool vec4, cudaStream_t s, bool pdl) {
    constexpr int ROWS_W = (32 / (KP / 16)) * RG;
    const int rows_cta = (kSerialThreads / 32) * ROWS_W;
    const long nrb = (p.V + rows_cta - 1) / rows_cta;
    const long blocks = (long)p.B * p.H * nrb;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    const bool pf = p.max_len > 1;
    const dim3 grid((unsigned)blocks), block(kSerialThreads);
    if (p.opts & GDN_OPT_GATE_PER_CHANNEL) {  // no capture with the per-channel gate
        if (vec4 && !pf)
            e = launch_kernel(delta_serial_kernel<T, KP, RG, true, false, false, true>, grid, block, 0, s, pdl, p);
        else if (vec4)
            e = launch_kernel(delta_serial_kernel<T, KP, RG, true, true, false, true>, grid, block, 0, s, pdl, p);
        else
            e = launch_kernel(delta_serial_kernel<T, KP, RG, false, true, false, true>, grid, block, 0, s, pdl, p);
        note_launch();
        return e;
    }
    if (p.capsule != nullptr && vec4 && !pf)
        e = launch_kernel(delta_serial_kernel<T, KP, RG, true, false, true>, grid, block, 0, s, pdl, p);
    else if (p.capsule != nullptr)
        e = vec4 ? launch_kernel(delta_serial_kernel<T, KP, RG, true, true, true>, grid, block, 0, s, pdl, p)
                 : launch_kernel(delta_serial_kernel<T, KP, RG, false, true, true>, grid, block, 0, s, pdl, p);
    else if (vec4 && pf)
        e = launch_kernel(delta_serial_kernel<T, KP, RG, true, true, false>, grid, block, 0, s, pdl, p);
    else if (vec4)
        e = launch_kernel(delta_serial_kernel<T, KP, RG, true, false, false>, grid, block, 0, s, pdl, p);
    else
        e = launch_kernel(delta_serial_kernel<T, KP, RG, false, true, false>, grid, block, 0, s, pdl, p);
    note_launch();
    return e;
}

template <typename T>
cudaError_t launch_serial_t(const DeltaParams &p, cudaStream_t s, bool pdl) {
    const bool vec4 = (p.K % 4 == 0) && ((uintptr_t)p.qk % 16 == 0) &&
                      ((uintptr_t)p.state_init % 16 == 0) && ((uintptr_t)p.state_fin % 16 == 0) &&
                      ((uintptr_t)p.gpc % 16 == 0);
    if (p.K <= 16) return launch_serial_kp<T, 16, 1>(p, vec4, s, pdl);
    if (p.K <= 32) return launch_serial_kp<T, 32, 1>(p, vec4, s, pdl);
    if (p.K <= 64) return launch_serial_kp<T, 64, 1>(p, vec4, s, pdl);
    if (p.K <= 128) return launch_serial_kp<T, 128, 2>(p, vec4, s, pdl);
    return launch_serial_kp<T, 256, 4>(p, vec4, s, pdl);
}

}  // namespace

cudaError_t launch_delta_serial(const DeltaParams &p, int dtype, cudaStream_t s, bool pdl) {
    if (dtype == 1) return launch_serial_t<__nv_bfloat16>(p, s, pdl);
    return launch_serial_t<float>(p, s, pdl);
}

}  // namespace gdn
