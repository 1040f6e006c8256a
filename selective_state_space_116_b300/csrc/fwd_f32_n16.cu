// Forward-scan instances: f32 I/O, N = 16 with 8 or 4 states per thread.
#include "fwd_launch.cuh"

namespace ssm_host {

int fwd_scan_f32_n16(int s, const ssm::ScanParams& p, int64_t chunk, bool zoh,
                 bool conv, bool vec, unsigned char* ws, int sms, cudaStream_t st) {
    using T = float;
    if (s == 8) return dispatch_scan_n<T, 16, 8>(p, chunk, zoh, conv, vec, ws, sms, st);
    if (s == 4) return dispatch_scan_n<T, 16, 4>(p, chunk, zoh, conv, vec, ws, sms, st);
    return SSM_ERR_UNSUPPORTED_N;
}

}  // namespace ssm_host
