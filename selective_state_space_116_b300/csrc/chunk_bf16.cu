// Chunked (L-parallel) schedule instances: bf16 I/O, every supported N.
#include "fwd_launch.cuh"

namespace ssm_host {

int fwd_chunked_bf16(int n, const ssm::ScanParams& p, const ChunkPlan& c, bool zoh, bool conv, bool vec,
                    unsigned char* ws, int sms, cudaStream_t st) {
    using T = __nv_bfloat16;
    switch (n) {
        case 1: return dispatch_chunked_n<T, 1, 1>(p, c, zoh, conv, vec, ws, sms, st);
        case 2: return dispatch_chunked_n<T, 2, 2>(p, c, zoh, conv, vec, ws, sms, st);
        case 4: return dispatch_chunked_n<T, 4, 4>(p, c, zoh, conv, vec, ws, sms, st);
        case 8: return dispatch_chunked_n<T, 8, 8>(p, c, zoh, conv, vec, ws, sms, st);
        case 16: return dispatch_chunked_n<T, 16, 8>(p, c, zoh, conv, vec, ws, sms, st);
    }
    return SSM_ERR_UNSUPPORTED_N;
}

}  // namespace ssm_host
