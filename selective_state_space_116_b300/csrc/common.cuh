// Device helpers shared by the scan and state-step kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (MUFU.EX2), flush-to-zero.
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// log2(x) on the special-function unit (MUFU.LG2).
__device__ __forceinline__ float lg2(float x) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// 1/x on the special-function unit (MUFU.RCP).
__device__ __forceinline__ float rcp(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// log2(1 + e) for e = 2^x in [0, 1/32): the series of ln(1 + e) to e^4,
// times log2(e).  The truncation error is below e^4 / 5 relative, under
// 2e-7 for these e, where forming 1 + e in fp32 would lose log2(1/e) bits.
__device__ __forceinline__ float log2_1p_small(float e) {
    float t = fmaf(e, -0.25f * kLog2e, kLog2e / 3.0f);
    t = fmaf(e, t, -0.5f * kLog2e);
    t = fmaf(e, t, kLog2e);
    return e * t;
}
__device__ __forceinline__ float2 log2_1p_small2(float2 e) {
    float2 t = __ffma2_rn(e, make_float2(-0.25f * kLog2e, -0.25f * kLog2e),
                          make_float2(kLog2e / 3.0f, kLog2e / 3.0f));
    t = __ffma2_rn(e, t, make_float2(-0.5f * kLog2e, -0.5f * kLog2e));
    t = __ffma2_rn(e, t, make_float2(kLog2e, kLog2e));
    return __fmul2_rn(e, t);
}

// log2(1 + 2^x): the special-function unit's log2 of 1 + 2^x, or the
// series above once 2^x < 1/32 (x < -5).
__device__ __forceinline__ float log2_1p_exp2(float x) {
    const float e = ex2(x);
    return x < -5.0f ? log2_1p_small(e) : lg2(1.0f + e);
}

// softplus(v) = ln(1 + e^v) = ln2 * log2(1 + 2^(v log2 e)); for v > 20 the
// correction e^-v is below half an fp32 ulp of v, so v itself is returned.
__device__ __forceinline__ float softplus(float v) {
    const float s = kLn2 * log2_1p_exp2(v * kLog2e);
    return v > 20.0f ? v : s;
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z).  For z -> -inf, e^-z -> inf and
// the reciprocal flushes to 0, giving -0.
__device__ __forceinline__ float silu(float z) {
    return z * rcp(1.0f + ex2(-z * kLog2e));
}

// I/O element conversion.
template <typename T> struct io;
template <> struct io<float> {
    static __device__ __forceinline__ float load(const float* p, int64_t i) { return p[i]; }
    static __device__ __forceinline__ float to_f32(float v) { return v; }
    static __device__ __forceinline__ float from_f32(float v) { return v; }
};
template <> struct io<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p, int64_t i) {
        return __bfloat162float(p[i]);
    }
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
    // round to nearest even
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

}  // namespace ssm
