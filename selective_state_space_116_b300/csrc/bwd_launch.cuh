// Backward-scan launch and dispatch over the compile-time variants (state
// size, gate, softplus, vector staging, input term, gradient type GT of du,
// ddelta, dz); instantiated by bwd.cu and bwd_zoh.cu (first-order and exact
// zero-order-hold input terms, fp32 gradients) and bwd_gio.cu and
// bwd_zoh_gio.cu (the same with bf16 gradients for bf16 I/O).
#pragma once
#include "host_plan.h"

namespace ssm_host {
namespace bwd_detail {

// With more than one chunk: the chunks' maps (one thread per channel and
// min(N, 4) states), their composition (one thread per channel and state),
// then every chunk at once (grid z).
template <typename T, int N, bool Z, bool SP, bool VEC, bool ZOH, typename GT, int K>
int launch_bwd(const ssm::bwd::BwdParams& p, cudaStream_t st) {
    using Sh = ssm::bwd::BwdShape<T, N, K>;
    static_assert(Sh::CH == ssm::bwd::channels_per_cta(N, K), "channels per CTA");
    if (p.nchunks > 1) {
        constexpr int S = N < 4 ? N : 4;
        const int64_t threads = p.batch * p.dim * (N / S), cells = p.batch * p.dim * N;
        const dim3 ga((unsigned)((threads + ssm::bwd::kAggThreads - 1) / ssm::bwd::kAggThreads),
                      (unsigned)p.nchunks);
        ssm::bwd::scan_bwd_chunk_agg_kernel<T, N, Z, SP, ZOH, GT><<<ga, ssm::bwd::kAggThreads, 0, st>>>(p);
        ssm::bwd::scan_bwd_chunk_carry_kernel<N><<<(unsigned)((cells + ssm::bwd::kAggThreads - 1) /
                                                              ssm::bwd::kAggThreads),
                                                   ssm::bwd::kAggThreads, 0, st>>>(p);
        if (cudaPeekAtLastError() != cudaSuccess) return SSM_ERR_CUDA;
    }
    auto kern = ssm::bwd::scan_bwd_kernel<T, N, K, Z, SP, VEC, ZOH, GT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return SSM_ERR_CUDA;
    const dim3 grid((unsigned)((p.dim + Sh::CH - 1) / Sh::CH), (unsigned)p.batch, (unsigned)p.nchunks);
    kern<<<grid, ssm::bwd::kThreads, Sh::SMEM, st>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N, bool VEC, bool ZOH, typename GT, int K>
int dispatch_bwd_zs(const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    if (z && sp) return launch_bwd<T, N, true, true, VEC, ZOH, GT, K>(p, st);
    if (z) return launch_bwd<T, N, true, false, VEC, ZOH, GT, K>(p, st);
    if (sp) return launch_bwd<T, N, false, true, VEC, ZOH, GT, K>(p, st);
    return launch_bwd<T, N, false, false, VEC, ZOH, GT, K>(p, st);
}

// two channels per thread only at N = 16 on a wide enough grid
template <typename T, int N, bool VEC, bool ZOH, typename GT>
int dispatch_bwd_k(const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    if constexpr (N == 16) {
        if (ssm::bwd::channels_per_thread(N, p.batch, p.dim, p.L) == 2)
            return dispatch_bwd_zs<T, N, VEC, ZOH, GT, 2>(p, z, sp, st);
    }
    return dispatch_bwd_zs<T, N, VEC, ZOH, GT, 1>(p, z, sp, st);
}

inline bool bwd_aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

// The vector path (asynchronous staging, 16-byte stores) needs whole tiles
// and 16-byte aligned sequence tensors.
template <typename T, int N, bool ZOH, typename GT>
int dispatch_bwd_n(const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    const bool vec = p.L % ssm::bwd::kTT == 0 && bwd_aligned16(p.u) && bwd_aligned16(p.delta) &&
                     bwd_aligned16(p.B) && bwd_aligned16(p.C) && bwd_aligned16(p.dy) &&
                     bwd_aligned16(p.du) && bwd_aligned16(p.ddelta) &&
                     (!z || (bwd_aligned16(p.z) && bwd_aligned16(p.dz)));
    return vec ? dispatch_bwd_k<T, N, true, ZOH, GT>(p, z, sp, st)
               : dispatch_bwd_k<T, N, false, ZOH, GT>(p, z, sp, st);
}

template <typename T, bool ZOH, typename GT = float>
int dispatch_bwd(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    switch (n) {
        case 1: return dispatch_bwd_n<T, 1, ZOH, GT>(p, z, sp, st);
        case 2: return dispatch_bwd_n<T, 2, ZOH, GT>(p, z, sp, st);
        case 4: return dispatch_bwd_n<T, 4, ZOH, GT>(p, z, sp, st);
        case 8: return dispatch_bwd_n<T, 8, ZOH, GT>(p, z, sp, st);
        case 16: return dispatch_bwd_n<T, 16, ZOH, GT>(p, z, sp, st);
    }
    return SSM_ERR_UNSUPPORTED_N;
}

}  // namespace bwd_detail
}  // namespace ssm_host
