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
