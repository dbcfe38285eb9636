// conv_prepare.cu - varlen causal depthwise conv1d with state, fused with the
// prepare step (q/k L2 norms, decay g, rate beta).
//
// Operations: paged_ssm.rs (onnxruntime-ep-mlx 0.31.1), CONV kernel (conv,
// SiLU, final conv state) and DELTA_PREPARE kernel (norms, g, beta);
// gated_delta_rate_activation.rs (mlx-c-rust), decay chain.
//
// GB300 design: one CTA owns a tile of TT tokens x CT channels, CT = 32 lanes
// x one 16-byte vector per lane (256 bf16 / 128 fp32 channels).  The tile's
// input rows plus the L-row causal halo are staged once in shared memory with
// 128-bit loads, so every x element is read from HBM once; weights are
// transposed to [Kc][CT] fp32 in shared memory.  Each warp then produces
// whole token rows, so a head's K channels sit in K/VEC consecutive lanes and
// its sum of squares is a segmented xor-shuffle: the prepare step is fused
// into the conv pass without another read of the conv output.
#include <math.h>

#include <type_traits>
#include <utility>

#include "common.cuh"

namespace gdn {

namespace {

constexpr int kConvThreads = 256;
constexpr int kOffsetsCache = 4096;  // offsets entries cached in shared memory

template <typename T, int VEC>
__device__ __forceinline__ void load_f(const T *p, float (&f)[VEC]) {
    if constexpr (sizeof(T) * VEC == 16) {
        Vec16<T> v;
        v.u = *reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = to_f32(v.v[e]);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = to_f32(p[e]);
    }
}

template <typename T, int VEC>
__device__ __forceinline__ void store_f(T *p, const float (&f)[VEC]) {
    if constexpr (sizeof(T) * VEC == 16) {
        Vec16<T> v;
#pragma unroll
        for (int e = 0; e < VEC; ++e) v.v[e] = from_f32<T>(f[e]);
        *reinterpret_cast<uint4 *>(p) = v.u;
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) p[e] = from_f32<T>(f[e]);
    }
}

template <typename T, int VEC>
__device__ __forceinline__ void copy_raw(T *dst, const T *src) {
    if constexpr (sizeof(T) * VEC == 16) {
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) dst[e] = src[e];
    }
}

// 16-byte global -> shared copy that bypasses registers; `valid` false fills zeros.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src, bool valid) {
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    const int bytes = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(gmem_src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <typename T, int VEC>
__device__ __forceinline__ void zero_raw(T *dst) {
    if constexpr (sizeof(T) * VEC == 16) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) dst[e] = from_f32<T>(0.f);
    }
}

// Round two fp32 values to T into elements (q, q + 1) of a 16-byte vector
// (one packed conversion for bf16).
template <typename T>
__device__ __forceinline__ void store_pair(Vec16<T> &v, int q, float a, float b) {
    if constexpr (std::is_same_v<T, __nv_bfloat16>) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
        v.v[q] = h2.x;
        v.v[q + 1] = h2.y;
    } else {
        v.v[q] = from_f32<T>(a);
        v.v[q + 1] = from_f32<T>(b);
    }
}

// silu_for on a pair of values; for bf16 the scale, add and product run as
// packed fp32 operations with the scalar roundings.
template <typename T>
__device__ __forceinline__ float2 silu2_for(float2 z) {
    if constexpr (std::is_same_v<T, __nv_bfloat16>) {
        const float2 hz = __fmul2_rn(make_float2(0.5f, 0.5f), z);
        float2 th;
        asm("tanh.approx.f32 %0, %1;" : "=f"(th.x) : "f"(hz.x));
        asm("tanh.approx.f32 %0, %1;" : "=f"(th.y) : "f"(hz.y));
        return __fmul2_rn(hz, __fadd2_rn(make_float2(1.f, 1.f), th));
    } else {
        return make_float2(silu_for<T>(z.x), silu_for<T>(z.y));
    }
}

__device__ __forceinline__ void decay_rate(const ConvParams &p, int t, int h, float &g,
                                           float &beta) {
    gates_opt(p.a, p.bl, (size_t)t * p.H + h, p.A_log, p.dt_bias, h, p.opts, g, beta);
}

// Block 0 of the conv launch checks the whole offsets array, records the
// status and the serial / chunked sequence counts in the workspace header
// and, when asked, schedules the chunked work: the sequences of at least
// chunk_min_len tokens are listed longest first (ties by index) and the work
// counter is reset.  The order comes from a bitonic sort of the keys
// (~len << 32 | index) in `keys`, the first kSortKeys * 8 bytes of the
// block's dynamic shared memory (used before the block's own conv work); with
// more chunked sequences than that they are listed in index order.
constexpr int kSortKeys = 4096;
__device__ void schedule_block(const ConvParams &p, unsigned long long *keys) {
    __shared__ int s_bad, s_serial, s_chunked, s_base;
    __shared__ int s_warp[kConvThreads / 32];
    const int B = p.B;
    if (threadIdx.x == 0) {
        s_bad = (__ldg(p.offsets) != 0 || __ldg(p.offsets + B) != p.N);
        s_serial = 0;
        s_chunked = 0;
        s_base = 0;
    }
    __syncthreads();
    int bad = 0, ns = 0, nc = 0;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int len = __ldg(p.offsets + b + 1) - __ldg(p.offsets + b);
        if (len < 0) bad = 1;
        else if (len >= p.chunk_min_len) ++nc;
        else ++ns;
    }
    if (bad) atomicOr(&s_bad, 1);
    atomicAdd(&s_serial, ns);
    atomicAdd(&s_chunked, nc);
    __syncthreads();
    const bool ok = !s_bad;
    const int nchunked = s_chunked;
    if (p.seq_order != nullptr && ok) {
        const int thr = p.chunk_min_len;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        if (nchunked <= kSortKeys) {
            // keys of the chunked sequences, padded to a power of two with the
            // largest key (they sort last and are not listed)
            int P = 1;
            while (P < nchunked) P <<= 1;
            for (int i = threadIdx.x; i < P; i += blockDim.x) keys[i] = ~0ull;
            __syncthreads();
            if (threadIdx.x == 0) s_base = 0;
            __syncthreads();
            for (int b0 = 0; b0 < B; b0 += blockDim.x) {
                const int b = b0 + threadIdx.x;
                const int len = b < B ? __ldg(p.offsets + b + 1) - __ldg(p.offsets + b) : 0;
                const bool take = b < B && len >= thr;
                const unsigned m = __ballot_sync(0xffffffffu, take);
                if (lane == 0) s_warp[warp] = __popc(m);
                __syncthreads();
                int before = s_base;
                for (int w = 0; w < warp; ++w) before += s_warp[w];
                if (take)
                    keys[before + __popc(m & ((1u << lane) - 1u))] =
                        ((unsigned long long)(~(unsigned)len) << 32) | (unsigned)b;
                __syncthreads();
                if (threadIdx.x == 0)
                    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s_base += s_warp[w];
                __syncthreads();
            }
            // bitonic sort, ascending: longest first, then lower index
            for (int k = 2; k <= P; k <<= 1) {
                for (int j = k >> 1; j > 0; j >>= 1) {
                    for (int i = threadIdx.x; i < P; i += blockDim.x) {
                        const int l = i ^ j;
                        if (l > i) {
                            const unsigned long long x = keys[i], y = keys[l];
                            if (((i & k) == 0) == (x > y)) {
                                keys[i] = y;
                                keys[l] = x;
                            }
                        }
                    }
                    __syncthreads();
                }
            }
            for (int i = threadIdx.x; i < nchunked; i += blockDim.x)
                p.seq_order[i] = (int)(keys[i] & 0xffffffffu);
        } else {
            for (int b0 = 0; b0 < B; b0 += blockDim.x) {
                const int b = b0 + threadIdx.x;
                const bool take = b < B && (__ldg(p.offsets + b + 1) - __ldg(p.offsets + b)) >= thr;
                const unsigned m = __ballot_sync(0xffffffffu, take);
                if (lane == 0) s_warp[warp] = __popc(m);
                __syncthreads();
                int before = s_base;
                for (int w = 0; w < warp; ++w) before += s_warp[w];
                if (take) p.seq_order[before + __popc(m & ((1u << lane) - 1u))] = b;
                __syncthreads();
                if (threadIdx.x == 0)
                    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s_base += s_warp[w];
                __syncthreads();
            }
        }
    }
    if (threadIdx.x == 0) {
        p.header->status = ok ? 0 : 4 /* GDN_ERR_OFFSETS */;
        p.header->n_serial = ok ? s_serial : 0;
        p.header->n_chunked = ok ? nchunked : 0;
        p.header->n_units = (ok && p.seq_order != nullptr) ? nchunked * p.H * p.VT : 0;
        p.header->next_unit = 0;
        p.header->seg_next[0] = 0;
        p.header->seg_next[1] = 0;
    }
    __syncthreads();  // the keys' shared memory is the block's conv scratch next
}

// Dynamic shared memory: [Kc][CT] f32 weights (KC == 0 only) | [TT+L][CT] T
// window (only when STAGE) | 3 x [TT] int token info | offsets cache.  With
// KC > 0 (conv width known at compile time) every lane keeps its VEC x KC
// weights in registers.  Without STAGE (very long receptive fields) the taps
// are read from global memory directly.  The window is staged with
// asynchronous 16-byte copies so all of a thread's loads are in flight at once.
template <typename T, int VEC, bool PREP, bool STAGE, int KC>
__global__ void __launch_bounds__(kConvThreads)
    conv_prepare_kernel(const ConvParams p, const int TT, const int n_ctiles) {
    constexpr int CT = 32 * VEC;
    extern __shared__ __align__(16) unsigned char smem[];
    const int tile_c = blockIdx.x % n_ctiles;
    const int tile_t = blockIdx.x / n_ctiles;
    const int c0 = tile_c * CT;
    const int t0 = tile_t * TT;
    const int L = p.L, Kc = p.Kc, D = p.D, C = p.C, N = p.N, B = p.B;

    float *sw = reinterpret_cast<float *>(smem);
    T *sx = reinterpret_cast<T *>(smem + (KC > 0 ? 0 : (((size_t)Kc * CT * 4 + 15) & ~size_t(15))));
    int *s_seq = reinterpret_cast<int *>(sx + (STAGE ? (size_t)(TT + L) * CT : 0));
    int *s_start = s_seq + TT;
    int *s_len = s_start + TT;
    int *s_offs = s_len + TT;  // offsets[0..B] when B + 1 <= kOffsetsCache
    const bool cache_offs = B + 1 <= kOffsetsCache;

    // The dependent kernel (recurrence / final state) may start streaming its
    // own inputs now; it waits for this grid before reading what it writes.
    pdl_launch_dependents();
    if (p.header != nullptr && blockIdx.x == 0)
        schedule_block(p, reinterpret_cast<unsigned long long *>(smem));

    // 1. token -> sequence (or -1 when the token's sequence is malformed); the
    //    search runs in shared memory when the offsets fit there
    if (cache_offs) {
        for (int i = threadIdx.x; i <= B; i += blockDim.x) s_offs[i] = __ldg(p.offsets + i);
        __syncthreads();
    }
    for (int i = threadIdx.x; i < TT; i += blockDim.x) {
        const int t = t0 + i;
        int b = -1, st = 0, en = 0;
        if (t < N) {
            if (cache_offs) {
                int lo = 0, hi = B - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_offs[mid] <= t) lo = mid;
                    else hi = mid - 1;
                }
                st = s_offs[lo];
                en = s_offs[lo + 1];
                if (s_offs[0] == 0 && s_offs[B] == N && st >= 0 && en >= st && en <= N && t >= st &&
                    t < en)
                    b = lo;
            } else {
                const int bb = seq_of_token(p.offsets, B, t);
                if (seq_bounds(p.offsets, B, N, bb, st, en) && t >= st && t < en) b = bb;
            }
        }
        s_seq[i] = b;
        s_start[i] = st;
        s_len[i] = en - st;
    }
    // 2. input window rows [t0 - L, t0 + TT), 16-byte asynchronous copies
    const T *x = static_cast<const T *>(p.x);
    const int rows = STAGE ? TT + L : 0;
    for (int i = threadIdx.x; i < rows * 32; i += blockDim.x) {
        const int r = i >> 5, v = i & 31;
        const long t = (long)t0 - L + r;
        const int c = c0 + v * VEC;
        T *dst = sx + (size_t)r * CT + v * VEC;
        const bool valid = t >= 0 && t < N && c < C;
        if constexpr (sizeof(T) * VEC == 16) {
            if (valid) cp_async16(dst, x + (size_t)t * C + c, true);
            else zero_raw<T, VEC>(dst);
        } else {
            if (valid) copy_raw<T, VEC>(dst, x + (size_t)t * C + c);
            else zero_raw<T, VEC>(dst);
        }
    }
    // 3. weights: in registers (KC > 0) or transposed to [Kc][CT] in shared memory
    const T *w = static_cast<const T *>(p.w);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int c = c0 + lane * VEC;
    const bool cvalid = c < C;
    float wr[KC > 0 ? KC : 1][VEC];
    if constexpr (KC > 0) {
        // the lane's VEC channels hold VEC * KC consecutive weights
        T wraw[VEC * KC];
#pragma unroll
        for (int q = 0; q < VEC * KC; ++q) wraw[q] = from_f32<T>(0.f);
        if (cvalid) {
            if constexpr ((sizeof(T) * VEC * KC) % 16 == 0) {
#pragma unroll
                for (int q = 0; q < VEC * KC; q += 16 / sizeof(T))
                    *reinterpret_cast<uint4 *>(wraw + q) =
                        *reinterpret_cast<const uint4 *>(w + (size_t)c * KC + q);
            } else {
#pragma unroll
                for (int q = 0; q < VEC * KC; ++q) wraw[q] = w[(size_t)c * KC + q];
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
            for (int j = 0; j < KC; ++j) wr[j][e] = to_f32(wraw[e * KC + j]);
    } else {
#pragma unroll 4
        for (int i = threadIdx.x; i < Kc * CT; i += blockDim.x) {
            const int j = i / CT, cc = c0 + i % CT;
            sw[i] = cc < C ? to_f32(w[(size_t)cc * Kc + j]) : 0.f;
        }
    }
    if constexpr (STAGE && sizeof(T) * VEC == 16) cp_async_wait_all();
    __syncthreads();

    float bias[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) bias[e] = 0.f;
    if (p.bias != nullptr && cvalid) load_f<T, VEC>(static_cast<const T *>(p.bias) + c, bias);
    const T *init = static_cast<const T *>(p.init);
    T *y = static_cast<T *>(p.y);
    const int qk_width = PREP ? 2 * p.HQ * p.K : 0;
    const int lanes_per_head = PREP ? p.K / VEC : 1;

    for (int i = warp; i < TT; i += nwarps) {
        const int b = s_seq[i];
        if (b < 0) continue;  // warp-uniform
        const int t = t0 + i, s = s_start[i];
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = bias[e];
        constexpr int kTaps = KC > 0 ? KC : 64;
#pragma unroll
        for (int j = 0; j < kTaps; ++j) {
            if (KC == 0 && j >= Kc) break;
            const int src = t - (Kc - 1 - j) * D;
            float xv[VEC];
            if (src >= s) {
                if constexpr (STAGE) {
                    load_f<T, VEC>(sx + (size_t)(src - t0 + L) * CT + lane * VEC, xv);
                } else if (cvalid) {
                    load_f<T, VEC>(x + (size_t)src * C + c, xv);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) xv[e] = 0.f;
                }
            } else {
                const int local = src - s;  // in [-L, -1]: read the initial conv state
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    xv[e] = cvalid ? to_f32(init[((size_t)b * C + c + e) * L + L + local]) : 0.f;
            }
            if constexpr (KC > 0) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = fmaf(xv[e], wr[j][e], acc[e]);
            } else {
                const float *wj = sw + j * CT + lane * VEC;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = fmaf(xv[e], wj[e], acc[e]);
            }
        }
        float yv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float z = acc[e];
            if (p.silu) z = silu_for<T>(z);
            yv[e] = round_through<T>(z);  // the conv output is stored in T
        }
        if (cvalid) store_f<T, VEC>(y + (size_t)t * C + c, yv);

        if constexpr (PREP) {
            if (c0 < qk_width) {  // warp-uniform
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) ss = fmaf(yv[e], yv[e], ss);
                for (int off = lanes_per_head >> 1; off > 0; off >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (cvalid && c < qk_width &&
                    (s_len[i] < p.prep_max_len || t - s_start[i] < p.prep_cap)) {
                    const float r = (p.opts & GDN_OPT_NO_QK_NORM) ? 1.f : rsqrtf(ss + 1e-12f);
                    const int plane = c >= p.HQ * p.K;
                    const int cc = c - plane * p.HQ * p.K;
                    float *dst = p.qk + (((size_t)plane * N + t) * p.HQ + cc / p.K) * p.K + cc % p.K;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) dst[e] = yv[e] * r;
                }
            }
        }
    }

    if constexpr (PREP) {
        if (tile_c == 0) {
            for (int i = threadIdx.x; i < TT * p.H; i += blockDim.x) {
                const int ti = i / p.H, h = i % p.H;
                const int t = t0 + ti;
                if (s_seq[ti] < 0 || (s_len[ti] >= p.prep_max_len && t - s_start[ti] >= p.prep_cap))
                    continue;
                float g, beta;
                decay_rate(p, t, h, g, beta);
                p.gb[(size_t)t * p.H + h] = g;
                p.gb[((size_t)N + t) * p.H + h] = beta;
            }
        }
    }
}

// Streaming variant for a compile-time conv width KC and dilation D (the
// common Kc <= 4 cases).  Each warp walks a run of R tokens of one residue
// class t = t_start + D i (for D = 1 simply R consecutive tokens) for one tile
// of CT = 32 * VEC channels, so the conv taps of a token are the KC - 1
// previous tokens of the same run.  Input rows stream through a per-warp
// ring of kRing rows in shared memory filled by 16-byte cp.async copies
// (kRing rows in flight per warp, no registers held), and the taps live in a
// register window that rotates with the KC-fold unrolled loop, so every
// input element is loaded, converted and moved once.  At each sequence start
// the window is refilled from that sequence's initial conv state.
constexpr int kRing = 8;
constexpr int kRingBytes = (kConvThreads / 32) * kRing * 512;  // 32 lanes x 16 bytes per row
static_assert(kRingBytes >= kSortKeys * (int)sizeof(unsigned long long),
              "block 0 sorts the schedule keys in the ring's shared memory");

template <typename T, int VEC, bool PREP, int KC, int D>
__global__ void __launch_bounds__(kConvThreads, 2)
    conv_stream_kernel(const ConvParams p, const int R, const int n_ctiles) {
    constexpr int L = (KC - 1) * D;
    constexpr int CT = 32 * VEC;
    static_assert(sizeof(T) * VEC == 16, "streaming conv works on 16-byte vectors");
    // dynamic shared memory: the rows ring [warps][kRing][CT], then offsets[0..B]
    // when B + 1 <= kOffsetsCache
    extern __shared__ __align__(16) unsigned char conv_dsm[];
    T *s_ring = reinterpret_cast<T *>(conv_dsm);
    int *s_offs = reinterpret_cast<int *>(conv_dsm + kRingBytes);

    // Launched as a dependent of the stream's previous kernel: nothing is read
    // before that kernel has finished.  Only then may this kernel's own
    // dependents start (the recurrence issues its state loads before it waits
    // for this kernel, and a state carried in place from the previous call
    // must be final by then).
    pdl_wait_primary();
    pdl_launch_dependents();
    if (p.header != nullptr && blockIdx.x == 0)
        schedule_block(p, reinterpret_cast<unsigned long long *>(conv_dsm));

    const int B = p.B, N = p.N, C = p.C;
    const bool cache_offs = B + 1 <= kOffsetsCache;
    if (cache_offs) {
        for (int i = threadIdx.x; i <= B; i += blockDim.x) s_offs[i] = __ldg(p.offsets + i);
    }
    __syncthreads();
    auto off = [&](int i) { return cache_offs ? s_offs[i] : __ldg(p.offsets + i); };
    if (off(0) != 0 || off(B) != N) return;  // malformed offsets: nothing is written

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile_c = blockIdx.x % n_ctiles, tile_t = blockIdx.x / n_ctiles;
    const int c0 = tile_c * CT, c = c0 + lane * VEC;
    const bool cvalid = c < C;
    // run of this warp: tokens tb + D i, i = 0 .. n - 1
    const int gw = tile_t * (kConvThreads / 32) + warp;
    const int span = gw / D, cls = gw % D;
    const long tb_l = (long)span * R * D + cls;
    if (tb_l >= N) return;
    const int tb = (int)tb_l;
    const int n = min(R, (N - 1 - tb) / D + 1);

    const T *x = static_cast<const T *>(p.x);
    const T *w = static_cast<const T *>(p.w);
    const T *init = static_cast<const T *>(p.init);
    T *y = static_cast<T *>(p.y);
    T *ring = s_ring + (size_t)warp * kRing * CT + lane * VEC;

    // the first kRing rows of the run start streaming in
#pragma unroll
    for (int q = 0; q < kRing; ++q) {
        const int t = tb + D * q;
        cp_async16(ring + q * CT, x + (size_t)(q < n ? t : tb) * C + (cvalid ? c : 0), q < n && cvalid);
        cp_async_commit();
    }

    // weights and bias of the lane's channels
    float wr[KC][VEC], bias[VEC];
    {
        T wraw[VEC * KC];
#pragma unroll
        for (int q = 0; q < VEC * KC; ++q) wraw[q] = from_f32<T>(0.f);
        if (cvalid) {
            if constexpr ((sizeof(T) * VEC * KC) % 16 == 0) {
#pragma unroll
                for (int q = 0; q < VEC * KC; q += 16 / sizeof(T))
                    *reinterpret_cast<uint4 *>(wraw + q) =
                        *reinterpret_cast<const uint4 *>(w + (size_t)c * KC + q);
            } else {
#pragma unroll
                for (int q = 0; q < VEC * KC; ++q) wraw[q] = w[(size_t)c * KC + q];
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
#pragma unroll
            for (int j = 0; j < KC; ++j) wr[j][e] = to_f32(wraw[e * KC + j]);
            bias[e] = 0.f;
        }
        if (p.bias != nullptr && cvalid) load_f<T, VEC>(static_cast<const T *>(p.bias) + c, bias);
    }

    // sequence of the first token
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off(mid) <= tb) lo = mid;
        else hi = mid - 1;
    }
    int b = lo, s = off(b), e = off(b + 1);
    bool seq_ok = e >= s && s >= 0 && e <= N && tb >= s && tb < e;

    // win[r % KC] holds run row r (as fp32); tap m of row r reads win[(r - m) % KC]
    float win[KC][VEC];
    // the KC - 1 rows before run row r (token t) from x or, before the sequence
    // start, from the sequence's initial conv state
    auto fill_window = [&](int t, auto ph_c) {
        constexpr int ph = decltype(ph_c)::value;
#pragma unroll
        for (int m = 1; m < KC; ++m) {
            float(&dst)[VEC] = win[(ph - m + KC * 4) % KC];
            const int src = t - m * D;
            if (src >= s) {
                if (cvalid) load_f<T, VEC>(x + (size_t)src * C + c, dst);
                else
#pragma unroll
                    for (int q = 0; q < VEC; ++q) dst[q] = 0.f;
            } else {
                const int local = src - s;  // in [-L, -1]
#pragma unroll
                for (int q = 0; q < VEC; ++q)
                    dst[q] = cvalid ? to_f32(init[((size_t)b * C + c + q) * L + L + local]) : 0.f;
            }
        }
    };

    const int qk_width = PREP ? 2 * p.HQ * p.K : 0;
    const int lanes_per_head = PREP ? p.K / VEC : 1;

    const size_t xstep = (size_t)D * C;
    const T *xfirst = x + (size_t)tb * C + (cvalid ? c : 0);
    const T *xnext = xfirst + kRing * xstep;
    T *yfirst = y + (size_t)tb * C + (cvalid ? c : 0);
    for (int r0 = 0; r0 < n; r0 += KC) {
        [&]<int... PH>(std::integer_sequence<int, PH...>) {
            (
                [&] {
                    constexpr int ph = PH;
                    const int r = r0 + ph;
                    if (r >= n) return;
                    const int t = tb + D * r;
                    // row r has landed (one commit group per row, in order)
                    asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
                    Vec16<T> cur;
                    cur.u = *reinterpret_cast<const uint4 *>(ring + (r & (kRing - 1)) * CT);
                    float(&xc)[VEC] = win[ph];  // lanes past C read the ring's zero fill
#pragma unroll
                    for (int q = 0; q < VEC; ++q) xc[q] = to_f32(cur.v[q]);
                    // the slot is free again: stream in row r + kRing
                    {
                        const int rn = r + kRing;
                        cp_async16(ring + (r & (kRing - 1)) * CT, rn < n ? xnext : xfirst,
                                   rn < n && cvalid);
                        xnext += xstep;
                        cp_async_commit();
                    }
                    if (r == 0 || t >= e) {  // run start or next sequence (warp-uniform)
                        if (t >= e) {
                            while (b + 1 < B && off(b + 1) <= t) ++b;
                            s = off(b);
                            e = off(b + 1);
                            seq_ok = e >= s && s >= 0 && e <= N && t >= s && t < e;
                        }
                        if (seq_ok) fill_window(t, std::integral_constant<int, ph>{});
                    }
                    T *yrow = yfirst + (size_t)r * xstep;
                    if (!seq_ok) return;
                    // channel pairs on the packed fp32 pipe: each component of
                    // __ffma2_rn / __fmul2_rn / __fadd2_rn rounds exactly as the
                    // scalar operation, so the outputs are those of scalar code
                    Vec16<T> yo;
#pragma unroll
                    for (int q = 0; q < VEC; q += 2) {
                        float2 acc = make_float2(bias[q], bias[q + 1]);
#pragma unroll
                        for (int j = 0; j < KC; ++j) {
                            const float(&xs)[VEC] = win[(ph - (KC - 1 - j) + KC * 4) % KC];
                            acc = __ffma2_rn(make_float2(xs[q], xs[q + 1]),
                                             make_float2(wr[j][q], wr[j][q + 1]), acc);
                        }
                        if (p.silu) acc = silu2_for<T>(acc);
                        store_pair<T>(yo, q, acc.x, acc.y);  // the conv output is stored in T
                    }
                    if (cvalid) *reinterpret_cast<uint4 *>(yrow) = yo.u;
                    if constexpr (PREP) {
                        // tokens of token-serial sequences, and the captured prefix
                        const bool prep_t = e - s < p.prep_max_len || t - s < p.prep_cap;
                        if (c0 < qk_width && prep_t) {  // warp-uniform
                            float yv[VEC];
#pragma unroll
                            for (int q = 0; q < VEC; ++q) yv[q] = to_f32(yo.v[q]);
                            float ss = 0.f;
#pragma unroll
                            for (int q = 0; q < VEC; ++q) ss = fmaf(yv[q], yv[q], ss);
                            for (int o = lanes_per_head >> 1; o > 0; o >>= 1)
                                ss += __shfl_xor_sync(0xffffffffu, ss, o);
                            if (cvalid && c < qk_width) {
                                const float rr = (p.opts & GDN_OPT_NO_QK_NORM) ? 1.f : rsqrtf(ss + 1e-12f);
                                const int plane = c >= p.HQ * p.K;
                                const int cc = c - plane * p.HQ * p.K;
                                float *dst = p.qk + (((size_t)plane * N + t) * p.HQ + cc / p.K) * p.K + cc % p.K;
#pragma unroll
                                for (int q = 0; q < VEC; ++q) dst[q] = yv[q] * rr;
                            }
                        }
                        if (tile_c == 0 && prep_t) {
                            for (int h = lane; h < p.H; h += 32) {
                                float g, beta;
                                decay_rate(p, t, h, g, beta);
                                p.gb[(size_t)t * p.H + h] = g;
                                p.gb[((size_t)N + t) * p.H + h] = beta;
                            }
                        }
                    }
                }(),
                ...);
        }(std::make_integer_sequence<int, KC>{});
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename T, int VEC, bool PREP, int KC, int D>
cudaError_t launch_conv_stream(const ConvParams &p, cudaStream_t s) {
    constexpr int CT = 32 * VEC;
    const int n_ctiles = (p.C + CT - 1) / CT;
    // run length: enough warps for several waves, at most 64 tokens per warp
    const long target_warps = 148L * 64;
    long R = ((long)p.N * n_ctiles) / target_warps;
    R = R < 1 ? 1 : (R > 64 ? 64 : R);
    const long spans = p.N > 0 ? (p.N + R * D - 1) / (R * D) : 1;
    const long warps = spans * D;
    const long ttiles = (warps + (kConvThreads / 32) - 1) / (kConvThreads / 32);
    const long blocks = ttiles * n_ctiles;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    const size_t smem = kRingBytes + (p.B + 1 <= kOffsetsCache ? sizeof(int) * (p.B + 1) : 0);
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(conv_stream_kernel<T, VEC, PREP, KC, D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(kRingBytes + sizeof(int) * kOffsetsCache));
    });
    if (e != cudaSuccess) return e;
    e = launch_kernel(conv_stream_kernel<T, VEC, PREP, KC, D>, dim3((unsigned)blocks), dim3(kConvThreads), smem, s,
                      /*pdl=*/true, p, (int)R, n_ctiles);
    note_launch();
    return e;
}

// Final conv state: fin[b,c,j] = x~(len - L + j).  One thread per (b, c) walks
// j upward; it reads init index len + j >= j before writing index j, so
// fin may alias init.
template <typename T>
__global__ void __launch_bounds__(256)
    conv_final_kernel(const T *__restrict__ x, const int32_t *__restrict__ offsets,
                      const T *init, T *fin, int B, int N, int C, int L, int cap,
                      const int32_t *counts, T *updates) {
    pdl_wait_primary();  // the conv kernel reads init before fin may overwrite it
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)B * C) return;
    const int b = (int)(i / C), c = (int)(i % C);
    int s, e;
    if (!seq_bounds(offsets, B, N, b, s, e)) return;
    const int len = e - s;
    const T *irow = init + ((size_t)b * C + c) * L;
    T *frow = fin + ((size_t)b * C + c) * L;
    for (int j = 0; j < L; ++j) {
        const int local = len - L + j;
        const T v = local >= 0 ? x[(size_t)(s + local) * C + c] : irow[L + local];
        frow[j] = v;
    }
    if (updates != nullptr) {  // CONV_CAPTURE: first raw input rows, zero beyond
        const int n = captured_tokens(counts, nullptr, cap, b, len);
        T *upd = updates + (size_t)b * cap * C + c;
        for (int k = 0; k < cap; ++k) upd[(size_t)k * C] = k < n ? x[(size_t)(s + k) * C + c] : from_f32<T>(0.f);
    }
}

// Standalone prepare: one warp per (token, key head) for the norms, then one
// thread per (token, value head) for g and beta.  With VEC > 1 lane l holds
// the VEC consecutive channels [l*VEC, (l+1)*VEC) of the head and the sum of
// squares is reduced over K/VEC lanes in the same order as the fused conv
// kernel, so both routes give identical bits.  VEC == 1 covers any K <= 256
// with a strided layout.
template <typename T, int VEC>
__global__ void __launch_bounds__(256) prepare_kernel(const PrepParams p, const int nb_norm) {
    pdl_launch_dependents();
    pdl_wait_primary();  // reads the conv output when launched as a PDL dependent
    const int W = 2 * p.HQ * p.K + p.H * p.V;
    if ((int)blockIdx.x < nb_norm) {
        const int lane = threadIdx.x & 31;
        const long pair = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
        if (pair >= (long)p.N * p.HQ) return;  // warp-uniform
        const int t = (int)(pair / p.HQ), kh = (int)(pair % p.HQ);
        const T *y = static_cast<const T *>(p.y) + (size_t)t * W;
        float *qdst = p.qk + ((size_t)t * p.HQ + kh) * p.K;
        float *kdst = p.qk + (((size_t)p.N + t) * p.HQ + kh) * p.K;
        if constexpr (VEC > 1) {
            const int lph = p.K / VEC;
            const bool act = lane < lph;
            float q[VEC], k[VEC], nq = 0.f, nk = 0.f;
            if (act) {
                load_f<T, VEC>(y + kh * p.K + lane * VEC, q);
                load_f<T, VEC>(y + p.HQ * p.K + kh * p.K + lane * VEC, k);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) q[e] = k[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                nq = fmaf(q[e], q[e], nq);
                nk = fmaf(k[e], k[e], nk);
            }
            for (int off = lph >> 1; off > 0; off >>= 1) {
                nq += __shfl_xor_sync(0xffffffffu, nq, off);
                nk += __shfl_xor_sync(0xffffffffu, nk, off);
            }
            if (act) {
                const bool nn = p.opts & GDN_OPT_NO_QK_NORM;
                const float rq = nn ? 1.f : rsqrtf(nq + 1e-12f), rk = nn ? 1.f : rsqrtf(nk + 1e-12f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    qdst[lane * VEC + e] = q[e] * rq;
                    kdst[lane * VEC + e] = k[e] * rk;
                }
            }
        } else {
            float q[8], k[8], nq = 0.f, nk = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = lane + 32 * j;
                q[j] = i < p.K ? to_f32(y[kh * p.K + i]) : 0.f;
                k[j] = i < p.K ? to_f32(y[p.HQ * p.K + kh * p.K + i]) : 0.f;
                nq = fmaf(q[j], q[j], nq);
                nk = fmaf(k[j], k[j], nk);
            }
            nq = group_sum<32>(nq);
            nk = group_sum<32>(nk);
            const bool nn = p.opts & GDN_OPT_NO_QK_NORM;
                const float rq = nn ? 1.f : rsqrtf(nq + 1e-12f), rk = nn ? 1.f : rsqrtf(nk + 1e-12f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = lane + 32 * j;
                if (i < p.K) {
                    qdst[i] = q[j] * rq;
                    kdst[i] = k[j] * rk;
                }
            }
        }
    } else {
        const long i = (long)(blockIdx.x - nb_norm) * blockDim.x + threadIdx.x;
        if (i >= (long)p.N * p.H) return;
        const int h = (int)(i % p.H);
        float g, beta;
        gates_opt(p.a, p.bl, (size_t)i, p.A_log, p.dt_bias, h, p.opts, g, beta);
        if (p.opts & GDN_OPT_GATE_PER_CHANNEL) {  // g [N, H, K], then beta [N, H]
            const bool soft = !(p.opts & (GDN_OPT_NO_DECAY | GDN_OPT_GATE_EXP));
            const float dtb = soft ? __ldg(p.dt_bias + h) : 0.f;
            const float alog = soft ? __ldg(p.A_log + h) : 0.f;
            const bool decay = !(p.opts & GDN_OPT_NO_DECAY);
            for (int c = 0; c < p.K; ++c)
                p.gb[(size_t)i * p.K + c] =
                    gate_of_logit(decay ? __ldg(p.a + (size_t)i * p.K + c) : 0.f, dtb, alog, p.opts);
            p.gb[(size_t)p.N * p.H * p.K + i] = beta;
        } else {
            p.gb[i] = g;
            p.gb[(size_t)p.N * p.H + i] = beta;
        }
    }
}

template <typename T, int VEC, bool PREP, int KC>
cudaError_t launch_conv_kc(const ConvParams &p, cudaStream_t s) {
    constexpr int CT = 32 * VEC;
    const int n_ctiles = (p.C + CT - 1) / CT;
    // tokens per CTA: small batches (decode) use short tiles for parallelism
    int TT = p.N >= 4096 ? 64 : (p.N >= 512 ? 32 : 8);
    const long n_ttiles = p.N > 0 ? (p.N + TT - 1) / TT : 1;  // >= 1 block for block 0 duties
    const long blocks = n_ttiles * n_ctiles;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    const size_t wbytes = KC > 0 ? 0 : ((size_t)p.Kc * CT * 4 + 15) & ~size_t(15);
    const size_t window = (size_t)(TT + p.L) * CT * sizeof(T);
    const bool stage = window <= 64 * 1024;
    const size_t offs_bytes = p.B + 1 <= kOffsetsCache ? sizeof(int) * (p.B + 1) : 0;
    size_t smem = wbytes + (stage ? window : 0) + 3 * sizeof(int) * TT + offs_bytes;
    // block 0 sorts the chunked sequences in the same shared memory first
    if (p.header != nullptr && p.seq_order != nullptr && smem < kSortKeys * sizeof(unsigned long long))
        smem = kSortKeys * sizeof(unsigned long long);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    auto kern = stage ? conv_prepare_kernel<T, VEC, PREP, true, KC>
                      : conv_prepare_kernel<T, VEC, PREP, false, KC>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<(unsigned)blocks, kConvThreads, smem, s>>>(p, TT, n_ctiles);
    note_launch();
    return cudaGetLastError();
}

template <typename T, int VEC, bool PREP>
cudaError_t launch_conv_t(const ConvParams &p, cudaStream_t s) {
    if constexpr (VEC > 1) {
        if (p.Kc == 4 && p.D == 1) return launch_conv_stream<T, VEC, PREP, 4, 1>(p, s);
        if (p.Kc == 4 && p.D == 2) return launch_conv_stream<T, VEC, PREP, 4, 2>(p, s);
        if (p.Kc == 3 && p.D == 1) return launch_conv_stream<T, VEC, PREP, 3, 1>(p, s);
        if (p.Kc == 2 && p.D == 1) return launch_conv_stream<T, VEC, PREP, 2, 1>(p, s);
    }
    if (VEC > 1 && p.Kc == 4) return launch_conv_kc<T, VEC, PREP, 4>(p, s);
    if (VEC > 1 && p.Kc == 3) return launch_conv_kc<T, VEC, PREP, 3>(p, s);
    if (VEC > 1 && p.Kc == 2) return launch_conv_kc<T, VEC, PREP, 2>(p, s);
    return launch_conv_kc<T, VEC, PREP, 0>(p, s);
}

bool aligned16(const void *ptr) { return ptr == nullptr || (((uintptr_t)ptr) & 15) == 0; }

}  // namespace

bool conv_can_fuse_prepare(int dtype, int C, int K, const void *const *ptrs, int nptrs) {
    const int vec = dtype == 1 ? 8 : 4;
    for (int i = 0; i < nptrs; ++i)
        if (!aligned16(ptrs[i])) return false;
    if (C % vec != 0) return false;
    if (K % vec != 0) return false;
    const int lph = K / vec;
    return lph >= 1 && lph <= 32 && (lph & (lph - 1)) == 0;
}

cudaError_t launch_conv(const ConvParams &p, int dtype, cudaStream_t s, bool *fused_prep) {
    const void *ptrs[] = {p.x, p.y, p.bias};
    const bool vec_ok = dtype == 1 ? (p.C % 8 == 0) : (p.C % 4 == 0);
    const bool aligned = vec_ok && aligned16(p.x) && aligned16(p.y) && aligned16(p.bias);
    const bool fuse = p.prep && conv_can_fuse_prepare(dtype, p.C, p.K, ptrs, 3);
    if (fused_prep) *fused_prep = fuse;
    ConvParams q = p;
    q.prep = fuse;
    if (dtype == 1) {
        using T = __nv_bfloat16;
        if (aligned) return fuse ? launch_conv_t<T, 8, true>(q, s) : launch_conv_t<T, 8, false>(q, s);
        return launch_conv_t<T, 1, false>(q, s);
    }
    if (aligned) return fuse ? launch_conv_t<float, 4, true>(q, s) : launch_conv_t<float, 4, false>(q, s);
    return launch_conv_t<float, 1, false>(q, s);
}

cudaError_t launch_conv_final(const void *x, const int32_t *offsets, const void *init,
                              void *fin, int B, int N, int C, int L, int dtype,
                              cudaStream_t s, int cap, const int32_t *counts, void *updates) {
    if (L == 0 && updates == nullptr) return cudaSuccess;
    const long total = (long)B * C;
    const long blocks = (total + 255) / 256;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    if (dtype == 1) {
        using T = __nv_bfloat16;
        e = launch_kernel(conv_final_kernel<T>, dim3((unsigned)blocks), dim3(256), 0, s, true,
                          static_cast<const T *>(x), offsets, static_cast<const T *>(init),
                          static_cast<T *>(fin), B, N, C, L, cap, counts, static_cast<T *>(updates));
    } else {
        e = launch_kernel(conv_final_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s, true,
                          static_cast<const float *>(x), offsets,
                          static_cast<const float *>(init), static_cast<float *>(fin), B, N, C,
                          L, cap, counts, static_cast<float *>(updates));
    }
    note_launch();
    return e;
}

cudaError_t launch_prepare(const PrepParams &p, int dtype, cudaStream_t s, bool pdl) {
    const long nb_norm = ((long)p.N * p.HQ + 7) / 8;
    const long nb_gb = ((long)p.N * p.H + 255) / 256;
    const long blocks = nb_norm + nb_gb;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    const int W = 2 * p.HQ * p.K + p.H * p.V;
    const void *ptrs[] = {p.y};
    const bool chunked = conv_can_fuse_prepare(dtype, W, p.K, ptrs, 1);
    const dim3 grid((unsigned)blocks), block(256);
    const int nb = (int)nb_norm;
    cudaError_t e;
    if (dtype == 1) {
        using T = __nv_bfloat16;
        e = chunked ? launch_kernel(prepare_kernel<T, 8>, grid, block, 0, s, pdl, p, nb)
                    : launch_kernel(prepare_kernel<T, 1>, grid, block, 0, s, pdl, p, nb);
    } else {
        e = chunked ? launch_kernel(prepare_kernel<float, 4>, grid, block, 0, s, pdl, p, nb)
                    : launch_kernel(prepare_kernel<float, 1>, grid, block, 0, s, pdl, p, nb);
    }
    note_launch();
    return e;
}

}  // namespace gdn
