// Single-token state-step instances (fp32 and bf16 I/O, every supported N).
#include "host_plan.h"

namespace ssm_host {
namespace {

template <typename T, int N, bool Z, bool SP, bool VEC>
int launch_step(const ssm::StepParams& p, cudaStream_t stream) {
    constexpr int kG = ssm::StepShape<N>::kG;
    const int64_t threads = p.batch * p.dim * kG;
    const int64_t blocks = (threads + ssm::kStepThreads - 1) / ssm::kStepThreads;
    if (blocks > INT32_MAX) return SSM_ERR_BAD_DIMS;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(ssm::kStepThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see state_step_kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, ssm::state_step_kernel<T, N, Z, SP, VEC>, p) != cudaSuccess)
        return SSM_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N>
int dispatch_step_n(const ssm::StepParams& p, bool z, bool sp, bool vec, cudaStream_t s) {
#define SSM_STEP_CASE(Z, SP, V) \
    if (z == Z && sp == SP && vec == V) return launch_step<T, N, Z, SP, V>(p, s);
    SSM_STEP_CASE(false, false, false)
    SSM_STEP_CASE(false, false, true)
    SSM_STEP_CASE(false, true, false)
    SSM_STEP_CASE(false, true, true)
    SSM_STEP_CASE(true, false, false)
    SSM_STEP_CASE(true, false, true)
    SSM_STEP_CASE(true, true, false)
    SSM_STEP_CASE(true, true, true)
#undef SSM_STEP_CASE
    return SSM_ERR_BAD_DIMS;
}

template <typename T>
int dispatch_step(int n, const ssm::StepParams& p, bool z, bool sp, bool vec, cudaStream_t s) {
    switch (n) {
        case 1: return dispatch_step_n<T, 1>(p, z, sp, vec, s);
        case 2: return dispatch_step_n<T, 2>(p, z, sp, vec, s);
        case 4: return dispatch_step_n<T, 4>(p, z, sp, vec, s);
        case 8: return dispatch_step_n<T, 8>(p, z, sp, vec, s);
        case 16: return dispatch_step_n<T, 16>(p, z, sp, vec, s);
    }
    return SSM_ERR_UNSUPPORTED_N;
}

}  // namespace

int step_f32(int n, const ssm::StepParams& p, bool z, bool sp, bool vec, cudaStream_t st) {
    return dispatch_step<float>(n, p, z, sp, vec, st);
}
int step_bf16(int n, const ssm::StepParams& p, bool z, bool sp, bool vec, cudaStream_t st) {
    return dispatch_step<__nv_bfloat16>(n, p, z, sp, vec, st);
}

}  // namespace ssm_host
