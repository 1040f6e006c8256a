// Host-side planning shared by the library's translation units: argument
// and size checks, the scan's schedule (state split, chunked schedule) and the
// layout of its workspace, and the per-unit entry points that launch the
// kernel instances.  Internal; the public contract is include/ssm_scan.h.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "ssm_scan.h"
#include "scan_fwd.cuh"
#include "scan_bwd.cuh"
#include "state_step.cuh"

namespace ssm_host {

inline bool valid_n(int64_t n) { return n == 1 || n == 2 || n == 4 || n == 8 || n == 16; }

inline size_t io_size(int io) { return io == SSM_IO_BF16 ? 2 : 4; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b with overflow check against INT64_MAX
inline bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

struct Range {
    const void* p;
    int64_t bytes;
};

inline bool overlap(Range a, Range b) {
    if (!a.p || !b.p || a.bytes <= 0 || b.bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + (uintptr_t)b.bytes && b0 < a0 + (uintptr_t)a.bytes;
}

// Sizes of the problem in elements, with overflow checks.
struct Sizes {
    int64_t chan;    // batch * dim
    int64_t seq;     // batch * dim * L        (u, delta, z, y)
    int64_t bc;      // batch * L * N          (B, C)
    int64_t state;   // batch * dim * N
    int64_t par;     // dim * N                (A)
};

inline int check_dims(const ssm_dims* dims, bool scan, Sizes* s) {
    if (!dims) return SSM_ERR_NULL_ARG;
    if (dims->io != SSM_IO_F32 && dims->io != SSM_IO_BF16) return SSM_ERR_BAD_DTYPE;
    if (dims->batch < 1 || dims->dim < 1 || dims->dstate < 1) return SSM_ERR_BAD_DIMS;
    if (scan && dims->seqlen < 0) return SSM_ERR_BAD_DIMS;
    if (!valid_n(dims->dstate)) return SSM_ERR_UNSUPPORTED_N;
    if (scan && dims->chunk < 0)
        return SSM_ERR_BAD_DIMS;
    if (scan && dims->batch > 65535) return SSM_ERR_BAD_DIMS;  // grid.y limit of the scan launch
    const int64_t L = scan ? dims->seqlen : 1;
    int64_t bytes;
    if (!mul_ok(dims->batch, dims->dim, &s->chan) || !mul_ok(s->chan, L, &s->seq) ||
        !mul_ok(dims->batch * 1, L, &s->bc) || !mul_ok(s->bc, dims->dstate, &s->bc) ||
        !mul_ok(s->chan, dims->dstate, &s->state) || !mul_ok(dims->dim, dims->dstate, &s->par) ||
        !mul_ok(s->seq, 4, &bytes) || !mul_ok(s->bc, 4, &bytes) || !mul_ok(s->state, 4, &bytes))
        return SSM_ERR_BAD_DIMS;
    return SSM_OK;
}

// Build-time tuning knob: a cap on resident scan CTAs per SM (0: as many as
// fit).
#ifndef SSM_SCAN_CTAS_PER_SM
#define SSM_SCAN_CTAS_PER_SM 0
#endif

// Workspace of the scan: a 256-byte header (status word), one flag per
// channel group, one carried state (CH x N fp32) per channel group.
struct ScanWorkspace {
    size_t flags_off, carry_off, clear_bytes, total;
};

// SM count of the current device, looked up once per device.
inline int device_sms(int* sms) {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
    if (dev >= 0 && dev < 64 && cache[dev].load() > 0) {
        *sms = cache[dev].load();
        return SSM_OK;
    }
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        *sms < 1)
        return SSM_ERR_CUDA;
    if (dev >= 0 && dev < 64) cache[dev].store(*sms);
    return SSM_OK;
}

// Channels one CTA of the state-split kernel scans with S states per thread
// and NT threads.
constexpr int seq_channels(int n, int s, int nt) { return nt / (n / s); }

// States per thread for N = 16: 8 (two thread groups per channel, less
// shared-memory traffic per element) when the problem has at least 128
// channels per SM, else 4 (twice the threads per channel).
inline int n16_split(const ssm_dims* d, int sms) {
    const int64_t groups8 = d->batch * ((d->dim + 63) / 64);
    return groups8 >= 2 * (int64_t)sms ? 8 : 4;
}

inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

inline ssm_dims wl_dims(const ssm::ScanParams& p, int n) {
    return ssm_dims{p.batch, p.dim, n, p.L, SSM_IO_F32, 0};
}

inline ScanWorkspace scan_workspace_for(const ssm_dims* d, int ch) {
    ScanWorkspace w{};
    if (d->seqlen == 0) return w;
    const int64_t groups = d->batch * ((d->dim + ch - 1) / ch);
    w.flags_off = 256;
    w.carry_off = w.flags_off + round256((size_t)groups * 4);
    w.clear_bytes = w.carry_off;
    w.total = w.carry_off + round256((size_t)groups * ch * d->dstate * 4);
    return w;
}

// The chunked (L-parallel) schedule: for problems whose channel groups of the
// state-split kernel cover fewer than 4096 channels and that have at least 64
// tiles per group, or whenever the
// caller's `chunk` is below seqlen.  The plan depends only on the sizes, so
// that the workspace size does too.  N = 16 uses 8 states per thread here
// (the chunks supply the parallelism).
struct ChunkPlan {
    bool on = false;
    int ch = 0;                     // channels per group
    int64_t groups = 0, ntiles = 0, tpc = 0, nchunks = 0;
};

inline ChunkPlan chunk_plan(const ssm_dims* d) {
    ChunkPlan c;
    if (d->seqlen <= 0) return c;
    const int n = (int)d->dstate;
    c.ch = seq_channels(n, n <= 8 ? n : 8, ssm::seq::kSeqThreads);
    c.groups = d->batch * ((d->dim + c.ch - 1) / c.ch);
    c.ntiles = (d->seqlen + ssm::seq::kTL - 1) / ssm::seq::kTL;
    if (d->chunk > 0 && d->chunk < d->seqlen) {
        c.tpc = (d->chunk + ssm::seq::kTL - 1) / ssm::seq::kTL;
    } else if (d->chunk == 0 && c.groups * c.ch < 64 * 64 && c.ntiles >= 64) {
        const int64_t want_units = 2048;
        c.tpc = (c.ntiles * c.groups + want_units - 1) / want_units;
        if (c.tpc < 8) c.tpc = 8;
    } else {
        return c;
    }
    c.nchunks = (c.ntiles + c.tpc - 1) / c.tpc;
    c.on = c.nchunks >= 2;
    return c;
}

// workspace of the chunked schedule: header, per unit the aggregate state
// (overwritten by the carry-in) and the Delta sums
inline ScanWorkspace chunk_workspace(const ChunkPlan& c, int n) {
    ScanWorkspace w{};
    if (!c.on) return w;
    const size_t units = (size_t)(c.groups * c.nchunks);
    w.flags_off = 256;                                        // (no flags: the Delta sums)
    w.carry_off = w.flags_off + round256(units * c.ch * 4);   // aggregate states
    w.clear_bytes = 256;
    w.total = w.carry_off + round256(units * c.ch * n * 4);
    return w;
}

// The workspace covers whichever kernel and split the call selects.
inline ScanWorkspace scan_workspace(const ssm_dims* d) {
    const int n = (int)d->dstate;
    const int s = n <= 8 ? n : 8;
    ScanWorkspace w = scan_workspace_for(d, seq_channels(n, s, ssm::seq::scan_threads(n / s, true)));
    const ScanWorkspace wf = scan_workspace_for(d, seq_channels(n, s, ssm::seq::scan_threads(n / s, false)));
    if (wf.total > w.total) w = wf;
    if (n == 16) {
        const ScanWorkspace w4 = scan_workspace_for(d, seq_channels(16, 4, ssm::seq::scan_threads(4, false)));
        if (w4.total > w.total) w = w4;
    }
    const ScanWorkspace cw = chunk_workspace(chunk_plan(d), n);
    if (cw.total > w.total) w = cw;
    return w;
}

// Number of CTAs of `kern` that fit on one SM (queried once per device).
template <typename K>
inline int occupancy(K kern, int threads, int smem, std::atomic<int>* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    int occ = cache[dev].load();
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem) !=
                cudaSuccess || occ < 1)
            return -1;
        cache[dev].store(occ);
    }
    return occ;
}



// ---------------------------------------------------------------------------
// Kernel launches, one translation unit per group of instances (they compile
// in parallel).  Each returns SSM_OK or a negative ssm_status.

// State-split scan, N in {1, 2, 4, 8} (S = N) or N = 16 with S in {4, 8};
// zoh: the exact zero-order-hold input term; conv: the fused convolution
// prologue; vec: the 16-byte copy paths (gate and softplus travel in the
// parameters).
int fwd_scan_f32_small(int n, const ssm::ScanParams& p, int64_t chunk, bool zoh, bool conv, bool vec,
                       unsigned char* ws, int sms, cudaStream_t st);
int fwd_scan_f32_n16(int s, const ssm::ScanParams& p, int64_t chunk, bool zoh, bool conv, bool vec,
                     unsigned char* ws, int sms, cudaStream_t st);
int fwd_scan_bf16_small(int n, const ssm::ScanParams& p, int64_t chunk, bool zoh, bool conv, bool vec,
                        unsigned char* ws, int sms, cudaStream_t st);
int fwd_scan_bf16_n16(int s, const ssm::ScanParams& p, int64_t chunk, bool zoh, bool conv, bool vec,
                      unsigned char* ws, int sms, cudaStream_t st);
// Chunked (L-parallel) schedule, any supported N.
int fwd_chunked_f32(int n, const ssm::ScanParams& p, const ChunkPlan& c, bool zoh, bool conv, bool vec,
                    unsigned char* ws, int sms, cudaStream_t st);
int fwd_chunked_bf16(int n, const ssm::ScanParams& p, const ChunkPlan& c, bool zoh, bool conv, bool vec,
                     unsigned char* ws, int sms, cudaStream_t st);
// Single-token state step.
int step_f32(int n, const ssm::StepParams& p, bool z, bool sp, bool vec, cudaStream_t st);
int step_bf16(int n, const ssm::StepParams& p, bool z, bool sp, bool vec, cudaStream_t st);
// Backward scan: first-order input term, exact zero-order hold.
int bwd_f32(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st);
int bwd_bf16(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st);
int bwd_zoh_f32(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st);
int bwd_zoh_bf16(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st);

}  // namespace ssm_host
