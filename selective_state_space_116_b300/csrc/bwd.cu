// Backward-scan instances (fp32 and bf16 I/O, every supported N).
#include "host_plan.h"

namespace ssm_host {
namespace {

template <typename T, int N, bool Z, bool SP>
int launch_bwd(const ssm::bwd::BwdParams& p, cudaStream_t st) {
    using Sh = ssm::bwd::BwdShape<N>;
    auto kern = ssm::bwd::scan_bwd_kernel<T, N, Z, SP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess)
        return SSM_ERR_CUDA;
    const dim3 grid((unsigned)((p.dim + Sh::CH - 1) / Sh::CH), (unsigned)p.batch);
    kern<<<grid, ssm::bwd::kThreads, Sh::SMEM, st>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N>
int dispatch_bwd_n(const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    if (z && sp) return launch_bwd<T, N, true, true>(p, st);
    if (z) return launch_bwd<T, N, true, false>(p, st);
    if (sp) return launch_bwd<T, N, false, true>(p, st);
    return launch_bwd<T, N, false, false>(p, st);
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
