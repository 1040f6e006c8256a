// Throughput probe for the special-function unit's 2^x (MUFU.EX2).
//
// Each thread runs kChains independent dependency chains x <- 2^-x, so the
// unit sees kChains outstanding requests per thread; with enough resident
// warps the launch is limited only by the unit's issue rate.  The caller
// times the launch; the ex2 count is blocks * threads * iters * kChains.
#pragma once

#include "common.cuh"

namespace ssm {

constexpr int kProbeChains = 8;

__global__ void probe_ex2_kernel(int iters, float* sink) {
    float x[kProbeChains];
#pragma unroll
    for (int i = 0; i < kProbeChains; i++) x[i] = 1e-3f * (float)(threadIdx.x + i);
    for (int it = 0; it < iters; it++) {
#pragma unroll
        for (int i = 0; i < kProbeChains; i++) x[i] = ex2(-x[i]);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kProbeChains; i++) s += x[i];
    // never true for these inputs (values stay in (0.5, 1]); keeps the chains alive
    if (s < 0.0f) sink[threadIdx.x] = s;
}

}  // namespace ssm
