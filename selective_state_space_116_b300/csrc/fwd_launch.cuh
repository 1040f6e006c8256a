// Launch templates of the forward scan: the state-split kernel under the
// persistent balanced schedule and the three passes of the chunked schedule.
// Included by the forward translation units, each of which instantiates one
// group of (I/O type, N, states per thread) instances, each in eight variants:
// first-order or exact zero-order-hold input term, with or without the fused
// convolution prologue, 16-byte or element-wise copies.  The gate and
// softplus are per-call flags in the parameters.
#pragma once

#include "host_plan.h"

namespace ssm_host {

// Chunked schedule: the three passes on `stream`.
template <typename T, int N, int S, bool ZOH, bool CONV, bool VEC>
int launch_chunked(ssm::ScanParams p, const ChunkPlan& c, unsigned char* ws, int sms,
                   cudaStream_t stream) {
    using namespace ssm::seq;
    constexpr int NT = kSeqThreads;
    using Sh = Shape<T, N, S, CONV, NT>;
    auto agg = scan_chunk_agg_kernel<T, N, S, NT, ZOH, CONV, VEC>;
    auto full = scan_fwd_kernel<T, N, S, NT, ZOH, CONV, VEC>;
    static std::atomic<int> occ_agg[64], occ_full[64];
    const int oa = occupancy(agg, Sh::NT, Sh::SMEM, occ_agg),
              of = occupancy(full, Sh::NT, Sh::SMEM, occ_full);
    if (oa < 1 || of < 1) return SSM_ERR_CUDA;
    p.groups_per_row = (p.dim + Sh::CH - 1) / Sh::CH;
    p.ngroups = p.batch * p.groups_per_row;
    p.ntiles = c.ntiles;
    p.nchunks = c.nchunks;
    p.tiles_per_chunk = c.tpc;
    const ScanWorkspace wl = chunk_workspace(c, N);
    p.status = reinterpret_cast<int*>(ws);
    p.dsum = reinterpret_cast<float*>(ws + wl.flags_off);
    p.agg = reinterpret_cast<float*>(ws + wl.carry_off);
    const int64_t units = p.ngroups * p.nchunks;
    if (cudaMemsetAsync(ws, 0, wl.clear_bytes, stream) != cudaSuccess) return SSM_ERR_CUDA;
    const int64_t ga = units < (int64_t)oa * sms ? units : (int64_t)oa * sms;
    agg<<<(unsigned)ga, Sh::NT, Sh::SMEM, stream>>>(p);
    const int64_t nseq = p.ngroups * Sh::CH * N;   // one CTA per (group, channel, state)
    if (nseq > INT32_MAX) return SSM_ERR_BAD_DIMS;
    scan_chunk_carry_kernel<N, Sh::CH><<<(unsigned)nseq, kCarryThreads, 0, stream>>>(p);
    const int64_t gf = units < (int64_t)of * sms ? units : (int64_t)of * sms;
    full<<<(unsigned)gf, Sh::NT, Sh::SMEM, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N, int S, bool ZOH, bool CONV, bool VEC, bool GS = false>
int launch_scan(ssm::ScanParams p, int64_t chunk, unsigned char* ws, int sms,
                cudaStream_t stream) {
    using namespace ssm::seq;
    constexpr int NT = scan_threads(N / S, ZOH);
    using Sh = Shape<T, N, S, CONV, NT>;
    auto kern = scan_fwd_kernel<T, N, S, NT, ZOH, CONV, VEC, GS>;
    // per kernel instance: raise its shared-memory limit and ask how many
    // CTAs fit on an SM, once
    static std::atomic<int> occ_cache[64];   // per device: the attribute is per context
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSM_ERR_CUDA;
    int occ = occ_cache[dev].load();
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Sh::NT, Sh::SMEM) !=
                cudaSuccess)
            return SSM_ERR_CUDA;
        if (occ < 1) return SSM_ERR_CUDA;
        occ_cache[dev].store(occ);
    }
    p.groups_per_row = (p.dim + Sh::CH - 1) / Sh::CH;
    p.ngroups = p.batch * p.groups_per_row;
    p.ntiles = (p.L + kTL - 1) / kTL;
    // One resident wave of persistent CTAs, the same number on every SM, and
    // never more CTAs than channel groups (so that no group is split twice).
    if (SSM_SCAN_CTAS_PER_SM > 0 && SSM_SCAN_CTAS_PER_SM < occ) occ = SSM_SCAN_CTAS_PER_SM;
    int64_t per_sm = p.ngroups / sms;
    if (per_sm > occ) per_sm = occ;
    int64_t ctas = per_sm >= 1 ? per_sm * sms : p.ngroups;
    if (chunk > 0 && p.ntiles > 0) {   // caller-chosen work per CTA (>= one group's tokens)
        const int64_t per = (chunk + kTL - 1) / kTL;
        const int64_t want = (p.ngroups * p.ntiles + per - 1) / per;
        if (want < ctas) ctas = want;
    }
    if (ctas < 1) ctas = 1;
    const ssm_dims own_dims = wl_dims(p, N);
    const ScanWorkspace own = scan_workspace_for(&own_dims, Sh::CH);
    if (p.ntiles > 0) {
        p.status = reinterpret_cast<int*>(ws);
        p.flags = reinterpret_cast<unsigned*>(ws + own.flags_off);
        p.carry = reinterpret_cast<float*>(ws + own.carry_off);
        if (cudaMemsetAsync(ws, 0, own.clear_bytes, stream) != cudaSuccess) return SSM_ERR_CUDA;
    }
    kern<<<(unsigned)ctas, Sh::NT, Sh::SMEM, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N, int S>
int dispatch_scan_n(const ssm::ScanParams& p, int64_t chunk, bool zoh, bool conv, bool vec,
                    unsigned char* ws, int sms, cudaStream_t s) {
    // the common layer configuration (gate and softplus, 16-byte rows) has
    // an instance of its own with both options fixed
    if (!zoh && !conv && vec && p.gate && p.softplus)
        return launch_scan<T, N, S, false, false, true, true>(p, chunk, ws, sms, s);
#define SSM_SCAN_CASE(Z, C, V) \
    if (zoh == Z && conv == C && vec == V) return launch_scan<T, N, S, Z, C, V>(p, chunk, ws, sms, s);
    SSM_SCAN_CASE(false, false, true)
    SSM_SCAN_CASE(false, false, false)
    SSM_SCAN_CASE(true, false, true)
    SSM_SCAN_CASE(true, false, false)
    SSM_SCAN_CASE(false, true, true)
    SSM_SCAN_CASE(false, true, false)
    SSM_SCAN_CASE(true, true, true)
    SSM_SCAN_CASE(true, true, false)
#undef SSM_SCAN_CASE
    return SSM_ERR_BAD_DIMS;
}

template <typename T, int N, int S>
int dispatch_chunked_n(const ssm::ScanParams& p, const ChunkPlan& c, bool zoh, bool conv, bool vec,
                       unsigned char* ws, int sms, cudaStream_t s) {
#define SSM_CHUNK_CASE(Z, C, V) \
    if (zoh == Z && conv == C && vec == V) return launch_chunked<T, N, S, Z, C, V>(p, c, ws, sms, s);
    SSM_CHUNK_CASE(false, false, true)
    SSM_CHUNK_CASE(false, false, false)
    SSM_CHUNK_CASE(true, false, true)
    SSM_CHUNK_CASE(true, false, false)
    SSM_CHUNK_CASE(false, true, true)
    SSM_CHUNK_CASE(false, true, false)
    SSM_CHUNK_CASE(true, true, true)
    SSM_CHUNK_CASE(true, true, false)
#undef SSM_CHUNK_CASE
    return SSM_ERR_BAD_DIMS;
}

}  // namespace ssm_host
