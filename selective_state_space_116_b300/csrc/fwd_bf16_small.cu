// Forward-scan instances: bf16 I/O, N in {1, 2, 4, 8}, one thread per channel state set.
#include "fwd_launch.cuh"

namespace ssm_host {

int fwd_scan_bf16_small(int n, const ssm::ScanParams& p, int64_t chunk, bool zoh,
                 bool conv, bool vec, unsigned char* ws, int sms, cudaStream_t st) {
    using T = __nv_bfloat16;
    switch (n) {
        case 1: return dispatch_scan_n<T, 1, 1>(p, chunk, zoh, conv, vec, ws, sms, st);
        case 2: return dispatch_scan_n<T, 2, 2>(p, chunk, zoh, conv, vec, ws, sms, st);
        case 4: return dispatch_scan_n<T, 4, 4>(p, chunk, zoh, conv, vec, ws, sms, st);
        case 8: return dispatch_scan_n<T, 8, 8>(p, chunk, zoh, conv, vec, ws, sms, st);
    }
    return SSM_ERR_UNSUPPORTED_N;
}

}  // namespace ssm_host
