// Backward-scan instances with the first-order input term, bf16 I/O and
// bf16 du, ddelta, dz (every supported N).
#include "bwd_launch.cuh"

namespace ssm_host {

int bwd_bf16_gio(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st) {
    return bwd_detail::dispatch_bwd<__nv_bfloat16, false, __nv_bfloat16>(n, p, z, sp, st);
}

}  // namespace ssm_host
