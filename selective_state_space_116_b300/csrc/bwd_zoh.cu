// Backward-scan instances with the exact zero-order-hold input term (fp32
// and bf16 I/O, every supported N).
#include "bwd_launch.cuh"

namespace ssm_host {

int bwd_zoh_f32(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    return bwd_detail::dispatch_bwd<float, true>(n, p, z, sp, st);
}
int bwd_zoh_bf16(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    return bwd_detail::dispatch_bwd<__nv_bfloat16, true>(n, p, z, sp, st);
}

}  // namespace ssm_host
