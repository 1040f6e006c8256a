// Single-token state update (recurrent / generation mode).
//
// The kernel streams the fp32 state once in and once out (128 of the ~136
// bytes it moves per channel at N = 16), so it is bound by HBM bandwidth, and
// what matters is how many bytes each SM keeps in flight.  Mapping: kS =
// min(N, 8) state entries per thread and kG = N / kS threads per channel; a
// thread issues all of its state loads (two 16-byte loads at N = 16) before
// any arithmetic, and the per-channel inputs (x, delta, z) and per-batch-row
// B, C rows are loaded alongside.  The kG partial sums of C.h are combined
// with warp shuffles inside the group; the group's first lane writes y.
// VEC: the state and A rows are 16-byte aligned, so 4 entries move as one
// float4.
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
    static constexpr int kS = N < 8 ? N : 8;   // state entries per thread
    static constexpr int kG = N / kS;          // threads per channel
};

// One kS-slice of one channel: load, update, store.
template <typename T, int N, bool HAS_Z, bool SOFTPLUS, bool VEC>
__device__ __forceinline__ void step_item(const StepParams& p, int64_t gid) {
    constexpr int kS = StepShape<N>::kS, kG = StepShape<N>::kG;
    const int64_t c = gid / kG;                  // flat channel b*dim + d
    const int j = (int)(gid % kG);               // which kS-slice of the state
    const int64_t nch = p.batch * p.dim;
    const bool active = c < nch;
    const int64_t cc = active ? c : 0;           // keep loads in bounds for idle lanes
    const int64_t b = cc / p.dim, d = cc % p.dim;
    const int n0 = j * kS;
    float* st = p.state + cc * N + n0;

    // the state first: the long-latency loads go out before anything else
    float h[kS];
    if constexpr (VEC && kS % 4 == 0) {
#pragma unroll
        for (int k = 0; k < kS; k += 4) {
            const float4 v4 = __ldcs(reinterpret_cast<const float4*>(st + k));
            h[k] = v4.x; h[k + 1] = v4.y; h[k + 2] = v4.z; h[k + 3] = v4.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kS; k++) h[k] = __ldcs(st + k);
    }
    const float xv = io<T>::load(static_cast<const T*>(p.x), cc);
    const float dl = io<T>::load(static_cast<const T*>(p.delta), cc);
    const float zv = HAS_Z ? io<T>::load(static_cast<const T*>(p.z), cc) : 0.0f;
    const float bias = p.bias ? p.bias[d] : 0.0f;
    const float Dv = p.D ? p.D[d] : 0.0f;
    const T* Bb = static_cast<const T*>(p.B) + b * N + n0;
    const T* Cb = static_cast<const T*>(p.C) + b * N + n0;
    const float* Ad = p.A + d * N + n0;
    // B and C rows: scalar loads (a warp's lanes read two rows, so each load
    // is one broadcast); A rows differ per channel: 16-byte loads where the
    // rows are aligned (a warp-wide scalar load of A touches 16 channels' rows)
    float Bv[kS], Cv[kS], Av[kS];
    if constexpr (VEC && kS == 8 && sizeof(T) == 2) {   // one 16-byte load per row
        const uint4 b4 = __ldg(reinterpret_cast<const uint4*>(Bb));
        const uint4 c4 = __ldg(reinterpret_cast<const uint4*>(Cb));
        const unsigned bw[4] = {b4.x, b4.y, b4.z, b4.w}, cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            Bv[2 * k] = __uint_as_float(bw[k] << 16); Bv[2 * k + 1] = __uint_as_float(bw[k] & 0xffff0000u);
            Cv[2 * k] = __uint_as_float(cw[k] << 16); Cv[2 * k + 1] = __uint_as_float(cw[k] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int k = 0; k < kS; k++) {
            Bv[k] = io<T>::load(Bb, k);
            Cv[k] = io<T>::load(Cb, k);
        }
    }
    if constexpr (VEC && kS % 4 == 0) {
#pragma unroll
        for (int k = 0; k < kS; k += 4) {
            const float4 a4 = __ldg(reinterpret_cast<const float4*>(Ad + k));
            Av[k] = a4.x; Av[k + 1] = a4.y; Av[k + 2] = a4.z; Av[k + 3] = a4.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kS; k++) Av[k] = Ad[k];
    }

    const float v = dl + bias;
    const float dt = SOFTPLUS ? softplus(v) : v;
    const float dtx = dt * xv;
    float part = 0.0f;
#pragma unroll
    for (int k = 0; k < kS; k++) {
        const float a = ex2(dt * (Av[k] * kLog2e));
        h[k] = fmaf(a, h[k], dtx * Bv[k]);
        part = fmaf(Cv[k], h[k], part);
    }
    if (active) {
        if constexpr (VEC && kS % 4 == 0) {
#pragma unroll
            for (int k = 0; k < kS; k += 4)
                __stcs(reinterpret_cast<float4*>(st + k), make_float4(h[k], h[k + 1], h[k + 2], h[k + 3]));
        } else {
#pragma unroll
            for (int k = 0; k < kS; k++) __stcs(st + k, h[k]);
        }
    }
    // combine the kG partial dot products of one channel (adjacent lanes)
#pragma unroll
    for (int off = kG / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (active && j == 0) {
        float yv = fmaf(Dv, xv, part);
        if constexpr (HAS_Z) yv *= silu(zv);
        static_cast<T*>(p.y)[cc] = io<T>::from_f32(yv);
    }
}

// One (channel, slice) item per thread.  (A persistent grid-stride variant
// measured slower: it serialises each thread's items.)
//
// Launched with programmatic dependent launch: a token's step is scheduled
// while the previous kernel on the stream (typically the previous token's
// step) drains, and waits at griddepcontrol.wait until that kernel has
// completed and its writes are visible, so the state it reads is the state
// the previous step wrote.  Each CTA signals its own dependents once its
// stores are issued.  Without a programmatic predecessor the wait returns at
// once.
template <typename T, int N, bool HAS_Z, bool SOFTPLUS, bool VEC>
__global__ void __launch_bounds__(kStepThreads) state_step_kernel(StepParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    step_item<T, N, HAS_Z, SOFTPLUS, VEC>(p, (int64_t)blockIdx.x * kStepThreads + threadIdx.x);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ssm
