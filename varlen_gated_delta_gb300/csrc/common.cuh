// common.cuh - small device helpers shared by the libgdn kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"

namespace gdn {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);  // round to nearest even
}

// Round an fp32 value to T and back (what a store of T followed by a load sees).
template <typename T>
__device__ __forceinline__ float round_through(float x) { return to_f32(from_f32<T>(x)); }

// 16-byte vector of T: 8 bf16 or 4 fp32 values.
template <typename T>
struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    union {
        uint4 u;
        T v[N];
    };
};

// Programmatic dependent launch: a primary grid lets its dependent grid start
// early; the dependent waits for the primary's completion (and memory) only
// where it consumes the primary's outputs.  Both are no-ops without PDL.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// SiLU z sigmoid(z) = z (1 + tanh(z/2)) / 2 of a conv output stored in T: for
// bf16 with the special-function unit's tanh (relative error about 2^-11,
// below the output's rounding step), for fp32 with the fast exponential and
// division (a few fp32 ulp).
template <typename T>
__device__ __forceinline__ float silu_for(float z) {
    if constexpr (std::is_same_v<T, __nv_bfloat16>) {
        float h;
        asm("tanh.approx.f32 %0, %1;" : "=f"(h) : "f"(0.5f * z));
        return 0.5f * z * (1.f + h);
    } else {
        return __fdividef(z, 1.f + __expf(-z));
    }
}

// Full-warp xor reduction over groups of `W` consecutive lanes (W a power of 2).
template <int W>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// True when offsets are globally consistent and sequence b is well formed
// (offsets[0] == 0, offsets[B] == N, 0 <= start <= end <= N).
__device__ __forceinline__ bool seq_bounds(const int32_t *offsets, int B, int N, int b,
                                           int &start, int &end) {
    start = __ldg(offsets + b);
    end = __ldg(offsets + b + 1);
    return __ldg(offsets) == 0 && __ldg(offsets + B) == N && start >= 0 && end >= start &&
           end <= N;
}

// Tokens of a sequence of `len` whose state updates are captured
// (paged_ssm.rs, *_CAPTURE_INIT): max(0, min(counts[b], cap, len)), or 0 when
// an active flag is given and is 0.
__device__ __forceinline__ int captured_tokens(const int32_t *counts, const int32_t *active,
                                               int cap, int b, int len) {
    if (active != nullptr && __ldg(active) == 0) return 0;
    int n = __ldg(counts + b);
    n = n < cap ? n : cap;
    n = n < len ? n : len;
    return n > 0 ? n : 0;
}

// Index of the sequence holding token t (0 <= t < offsets[B]): the largest b
// in [0, B) with offsets[b] <= t.  For nondecreasing offsets that sequence is
// not empty and offsets[b] <= t < offsets[b+1].
__device__ __forceinline__ int seq_of_token(const int32_t *offsets, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(offsets + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Decay and update rate of one (token, value head) [paged_ssm.rs,
// DELTA_PREPARE; gated_delta_rate_activation.rs, decay chain]:
//   g = exp(-exp(A_log) * softplus(a + dt_bias)),  beta = sigmoid(b),
// softplus(x) = max(x, 0) + log1p(exp(-|x|)).  Shared by every kernel that
// computes them so the fused and standalone routes give identical bits.
__device__ __forceinline__ void decay_and_rate(float a, float dt_bias, float A_log, float b,
                                               float &g, float &beta) {
    const float x = a + dt_bias;
    const float softplus = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
    g = expf(-expf(A_log) * softplus);
    beta = 1.f / (1.f + expf(-b));
}

// g and beta of token-head element i (head h) under the rule options
// (GDN_OPT_*): g = 1 without decay, exp(a) for the exp gate, else the softplus
// gate above; beta = 1 without a rate input, b raw, or sigmoid(b).
__device__ __forceinline__ void gates_opt(const float *a, const float *b, size_t i,
                                          const float *A_log, const float *dt_bias, int h,
                                          int opts, float &g, float &beta) {
    if (opts == 0) {
        decay_and_rate(__ldg(a + i), __ldg(dt_bias + h), __ldg(A_log + h), __ldg(b + i), g, beta);
        return;
    }
    g = 1.f;  // (with the per-channel gate the gates come from gate_of_logit)
    if (!(opts & (GDN_OPT_NO_DECAY | GDN_OPT_GATE_PER_CHANNEL))) {
        float x = __ldg(a + i);
        if (!(opts & GDN_OPT_GATE_EXP)) {
            x += __ldg(dt_bias + h);
            const float softplus = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
            x = -expf(__ldg(A_log + h)) * softplus;
        }
        g = expf(x);
    }
    beta = 1.f;
    if (!(opts & GDN_OPT_NO_BETA)) {
        beta = __ldg(b + i);
        if (!(opts & GDN_OPT_BETA_RAW)) beta = 1.f / (1.f + expf(-beta));
    }
}

// Gate of one key channel from its decay logit x (GDN_OPT_GATE_PER_CHANNEL):
// the scalar gate's activation applied to the channel's logit -- 1 without
// decay, exp(x) for the exp gate, else exp(-exp(A_log) softplus(x + dt_bias)).
__device__ __forceinline__ float gate_of_logit(float x, float dt_bias, float A_log, int opts) {
    if (opts & GDN_OPT_NO_DECAY) return 1.f;
    if (!(opts & GDN_OPT_GATE_EXP)) {
        x += dt_bias;
        const float softplus = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
        x = -expf(A_log) * softplus;
    }
    return expf(x);
}

// log(g) for the same (token, value head), kept in the log domain.
__device__ __forceinline__ float log_decay(float a, float dt_bias, float A_log) {
    const float x = a + dt_bias;
    const float softplus = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
    return -expf(A_log) * softplus;
}

}  // namespace gdn
