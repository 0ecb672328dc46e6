// Device helpers shared by the scan kernels: element loads/stores, the
// discretisation step, the gate and the fast base-2 exponential.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the special-function unit (approximate, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Element access for the two I/O types.
template <typename T> struct Io;

template <> struct Io<float> {
    static __device__ __forceinline__ float ld(const void *p, int64_t i) {
        return __ldg(static_cast<const float *>(p) + i);
    }
    static __device__ __forceinline__ void st(void *p, int64_t i, float v) {
        static_cast<float *>(p)[i] = v;
    }
};

template <> struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const void *p, int64_t i) {
        return __bfloat162float(__ldg(static_cast<const __nv_bfloat16 *>(p) + i));
    }
    static __device__ __forceinline__ void st(void *p, int64_t i, float v) {
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    }
};

// softplus(v) = log(1 + e^v), written max(v, 0) + log(1 + e^-|v|) so the
// exponential never overflows.  log1pf keeps full relative accuracy for the
// small arguments that large negative v produce.
__device__ __forceinline__ float softplus_f(float v) {
    return fmaxf(v, 0.0f) + log1pf(ex2(-fabsf(v) * kLog2e));
}

constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float lg2(float x) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// softplus on a pair, for the hot loops: max(v, 0) + log(1 + w), w = e^-|v|
// in (0, 1].  log(1 + w) is ln 2 * log2(1 + w) from the special-function unit
// (absolute error about 2^-22, so relative error below 1.1e-5 once
// log(1 + w) >= 0.015), and for w < 2^-6, where 1 + w loses w's low bits,
// the series w - w^2/2 + w^3/3 (truncation error below w^4/4, relative
// 1e-6).
__device__ __forceinline__ float2 softplus2(float2 v) {
    const float2 m = __fmul2_rn(make_float2(-fabsf(v.x), -fabsf(v.y)), make_float2(kLog2e, kLog2e));
    const float2 w = make_float2(ex2(m.x), ex2(m.y));
    const float2 w1 = __fadd2_rn(w, make_float2(1.0f, 1.0f));
    const float2 big = __fmul2_rn(make_float2(lg2(w1.x), lg2(w1.y)), make_float2(kLn2, kLn2));
    float2 sm = __ffma2_rn(w, make_float2(1.0f / 3.0f, 1.0f / 3.0f), make_float2(-0.5f, -0.5f));
    sm = __ffma2_rn(w, sm, make_float2(1.0f, 1.0f));
    sm = __fmul2_rn(w, sm);
    const float2 lp = make_float2(w.x < 0.015625f ? sm.x : big.x, w.y < 0.015625f ? sm.y : big.y);
    return __fadd2_rn(make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f)), lp);
}

// silu(z) = z / (1 + e^-z).  For z < -87 the exponential is +inf and the
// quotient is -0, the correctly rounded limit.
__device__ __forceinline__ float silu_f(float z) {
    return __fdividef(z, 1.0f + ex2(-z * kLog2e));
}

// Step size Delta from the raw delta, the channel bias and the flag.
__device__ __forceinline__ float step_delta(float dv, float bias, int softplus) {
    float v = dv + bias;
    return softplus ? softplus_f(v) : v;
}

}  // namespace ssm
