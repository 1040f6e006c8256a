// Single-token state update (recurrent / generation mode).
//
// Mapping: kS = min(N, 4) state entries per thread, kG = N / kS threads per
// channel, so a warp reads and writes whole 16-byte pieces of consecutive
// state rows (fully coalesced).  The kG partial sums of C.h are combined with
// warp shuffles inside the group; the group's first lane writes y.  The
// kernel streams the state once in and once out: it is bound by HBM.
// VEC: the state rows are 16-byte aligned, so 4 entries move as one float4.
#pragma once

#include "common.cuh"

namespace ssm {

struct StepParams {
    float* state;
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;      // may be null
    const void* z;       // may be null
    const float* bias;   // may be null
    void* y;
    int64_t batch, dim;
};

constexpr int kStepThreads = 256;

template <int N> struct StepShape {
    static constexpr int kS = N < 4 ? N : 4;   // state entries per thread
    static constexpr int kG = N / kS;          // threads per channel
};

template <typename T, int N, bool HAS_Z, bool SOFTPLUS, bool VEC>
__global__ void __launch_bounds__(kStepThreads) state_step_kernel(StepParams p) {
    constexpr int kS = StepShape<N>::kS, kG = StepShape<N>::kG;
    const int64_t gid = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;
    const int64_t c = gid / kG;                  // flat channel b*dim + d
    const int j = (int)(gid % kG);               // which kS-slice of the state
    const int64_t nch = p.batch * p.dim;
    const bool active = c < nch;
    const int64_t cc = active ? c : 0;           // keep loads in bounds for idle lanes
    const int64_t b = cc / p.dim, d = cc % p.dim;
    const int n0 = j * kS;

    const float bias = p.bias ? p.bias[d] : 0.0f;
    const float v = io<T>::load(static_cast<const T*>(p.delta), cc) + bias;
    const float dt = SOFTPLUS ? softplus(v) : v;
    const float xv = io<T>::load(static_cast<const T*>(p.x), cc);
    const float dtx = dt * xv;
    const T* Bb = static_cast<const T*>(p.B) + b * N + n0;
    const T* Cb = static_cast<const T*>(p.C) + b * N + n0;
    const float* Ad = p.A + d * N + n0;
    float* st = p.state + cc * N + n0;

    float h[kS];
    if constexpr (kS == 4 && VEC) {
        const float4 v4 = *reinterpret_cast<const float4*>(st);
        h[0] = v4.x; h[1] = v4.y; h[2] = v4.z; h[3] = v4.w;
    } else {
#pragma unroll
        for (int k = 0; k < kS; k++) h[k] = st[k];
    }
    float part = 0.0f;
#pragma unroll
    for (int k = 0; k < kS; k++) {
        const float a = ex2(dt * (Ad[k] * kLog2e));
        h[k] = fmaf(a, h[k], dtx * io<T>::load(Bb, k));
        part = fmaf(io<T>::load(Cb, k), h[k], part);
    }
    if (active) {
        if constexpr (kS == 4 && VEC) {
            *reinterpret_cast<float4*>(st) = make_float4(h[0], h[1], h[2], h[3]);
        } else {
#pragma unroll
            for (int k = 0; k < kS; k++) st[k] = h[k];
        }
    }
    // combine the kG partial dot products of one channel (adjacent lanes)
#pragma unroll
    for (int off = kG / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (active && j == 0) {
        float yv = fmaf(p.D ? p.D[d] : 0.0f, xv, part);
        if constexpr (HAS_Z) yv *= silu(io<T>::load(static_cast<const T*>(p.z), cc));
        static_cast<T*>(p.y)[cc] = io<T>::from_f32(yv);
    }
}

}  // namespace ssm
