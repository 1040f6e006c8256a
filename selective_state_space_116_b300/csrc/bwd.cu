// Backward-scan instances (fp32 and bf16 I/O, every supported N).
#include "host_plan.h"

namespace ssm_host {
namespace {

// Channels per thread: two at N = 16 (their dB, dC products summed in
// registers before the shared-memory reduction), one for smaller states.
template <int N> constexpr int bwd_channels_per_thread() { return N == 16 ? 2 : 1; }

template <typename T, int N, bool Z, bool SP, bool VEC>
int launch_bwd(const ssm::bwd::BwdParams& p, cudaStream_t st) {
    constexpr int K = bwd_channels_per_thread<N>();
    using Sh = ssm::bwd::BwdShape<T, N, K>;
    auto kern = ssm::bwd::scan_bwd_kernel<T, N, K, Z, SP, VEC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return SSM_ERR_CUDA;
    const dim3 grid((unsigned)((p.dim + Sh::CH - 1) / Sh::CH), (unsigned)p.batch);
    kern<<<grid, ssm::bwd::kThreads, Sh::SMEM, st>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N, bool VEC>
int dispatch_bwd_zs(const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    if (z && sp) return launch_bwd<T, N, true, true, VEC>(p, st);
    if (z) return launch_bwd<T, N, true, false, VEC>(p, st);
    if (sp) return launch_bwd<T, N, false, true, VEC>(p, st);
    return launch_bwd<T, N, false, false, VEC>(p, st);
}

inline bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

// The vector path (asynchronous staging, 16-byte stores) needs whole tiles
// and 16-byte aligned sequence tensors.
template <typename T, int N>
int dispatch_bwd_n(const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    const bool vec = p.L % ssm::bwd::kTT == 0 && aligned16(p.u) && aligned16(p.delta) &&
                     aligned16(p.B) && aligned16(p.C) && aligned16(p.dy) && aligned16(p.du) &&
                     aligned16(p.ddelta) && (!z || (aligned16(p.z) && aligned16(p.dz)));
    return vec ? dispatch_bwd_zs<T, N, true>(p, z, sp, st) : dispatch_bwd_zs<T, N, false>(p, z, sp, st);
}

template <typename T>
int dispatch_bwd(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    switch (n) {
        case 1: return dispatch_bwd_n<T, 1>(p, z, sp, st);
        case 2: return dispatch_bwd_n<T, 2>(p, z, sp, st);
        case 4: return dispatch_bwd_n<T, 4>(p, z, sp, st);
        case 8: return dispatch_bwd_n<T, 8>(p, z, sp, st);
        case 16: return dispatch_bwd_n<T, 16>(p, z, sp, st);
    }
    return SSM_ERR_UNSUPPORTED_N;
}

}  // namespace

int bwd_f32(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    return dispatch_bwd<float>(n, p, z, sp, st);
}
int bwd_bf16(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    return dispatch_bwd<__nv_bfloat16>(n, p, z, sp, st);
}

}  // namespace ssm_host
