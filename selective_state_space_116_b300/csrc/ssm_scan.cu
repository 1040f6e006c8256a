// C ABI of the selective-scan library: argument checks on the host, then a
// launch of the kernel instance that matches (I/O type, N, gate, softplus,
// alignment) on the caller's stream.  See include/ssm_scan.h for the contract.
#include "ssm_scan.h"

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "probe.cuh"
#include "scan_fwd.cuh"
#include "scan_fwd_tc.cuh"
#include "scan_fwd_ws.cuh"
#include "scan_bwd.cuh"
#include "state_step.cuh"

namespace {

using bf16 = __nv_bfloat16;

constexpr int kVersion = 100;  // 0.1.0

bool valid_n(int64_t n) { return n == 1 || n == 2 || n == 4 || n == 8 || n == 16; }

size_t io_size(int io) { return io == SSM_IO_BF16 ? 2 : 4; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b with overflow check against INT64_MAX
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

struct Range {
    const void* p;
    int64_t bytes;
};

bool overlap(Range a, Range b) {
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

int check_dims(const ssm_dims* dims, bool scan, Sizes* s) {
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

// Build-time tuning knobs: a cap on resident scan CTAs per SM (0: as many as
// fit), and whether bf16 / N = 16 scans take the tensor-core kernel of
// scan_fwd_tc.cuh (off: its warp-specialised pipeline runs the Mamba-2.8B
// layer shape in ~605 us against ~450 us for the state-split kernel; it is
// bound by hand-off latency, not by any pipe).
#ifndef SSM_SCAN_CTAS_PER_SM
#define SSM_SCAN_CTAS_PER_SM 0
#endif
#ifndef SSM_SCAN_TC
#define SSM_SCAN_TC 0
#endif
// whether bf16 / N = 16 scans with L % 16 == 0 take the warp-specialised
// state-split kernel of scan_fwd_ws.cuh
#ifndef SSM_SCAN_WS
#define SSM_SCAN_WS 0
#endif

// Workspace of the scan: a 256-byte header (status word), one flag per
// channel group, one carried state (CH x N fp32) per channel group.
struct ScanWorkspace {
    size_t flags_off, carry_off, clear_bytes, total;
};

// SM count of the current device, looked up once per device.
int device_sms(int* sms) {
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

// Channels one CTA of the state-split kernel scans with S states per thread.
constexpr int seq_channels(int n, int s) { return ssm::seq::kThreads / (n / s); }

// States per thread for N = 16: 8 (two thread groups per channel, less
// shared-memory traffic per element) when the problem has enough 64-channel
// groups to give every SM two of them, else 4 (twice the CTAs).
int n16_split(const ssm_dims* d, int sms) {
    const int64_t groups8 = d->batch * ((d->dim + 63) / 64);
    return groups8 >= 2 * (int64_t)sms ? 8 : 4;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

ssm_dims wl_dims(const ssm::ScanParams& p, int n) {
    return ssm_dims{p.batch, p.dim, n, p.L, SSM_IO_F32, 0};
}

ScanWorkspace scan_workspace_for(const ssm_dims* d, int ch) {
    ScanWorkspace w{};
    if (d->seqlen == 0) return w;
    const int64_t groups = d->batch * ((d->dim + ch - 1) / ch);
    w.flags_off = 256;
    w.carry_off = w.flags_off + round256((size_t)groups * 4);
    w.clear_bytes = w.carry_off;
    w.total = w.carry_off + round256((size_t)groups * ch * d->dstate * 4);
    return w;
}

// The chunked (L-parallel) schedule: for problems with fewer than 64 groups
// of the state-split kernel and at least 64 tiles per group, or whenever the
// caller's `chunk` is below seqlen.  The plan depends only on the sizes, so
// that the workspace size does too.  N = 16 uses 8 states per thread here
// (the chunks supply the parallelism).
struct ChunkPlan {
    bool on = false;
    int ch = 0;                     // channels per group
    int64_t groups = 0, ntiles = 0, tpc = 0, nchunks = 0;
};

ChunkPlan chunk_plan(const ssm_dims* d) {
    ChunkPlan c;
    if (d->seqlen <= 0) return c;
    const int n = (int)d->dstate;
    c.ch = seq_channels(n, n <= 8 ? n : 8);
    c.groups = d->batch * ((d->dim + c.ch - 1) / c.ch);
    c.ntiles = (d->seqlen + ssm::seq::kTL - 1) / ssm::seq::kTL;
    if (d->chunk > 0 && d->chunk < d->seqlen) {
        c.tpc = (d->chunk + ssm::seq::kTL - 1) / ssm::seq::kTL;
    } else if (d->chunk == 0 && c.groups < 64 && c.ntiles >= 64) {
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
ScanWorkspace chunk_workspace(const ChunkPlan& c, int n) {
    ScanWorkspace w{};
    if (!c.on) return w;
    const size_t units = (size_t)(c.groups * c.nchunks);
    w.flags_off = 256;                                        // (no flags: the Delta sums)
    w.carry_off = w.flags_off + round256(units * c.ch * 4);   // aggregate states
    w.clear_bytes = 256;
    w.total = w.carry_off + round256(units * c.ch * n * 4);
    return w;
}

// The tensor-core kernel serves bf16 I/O with N = 16 when every row of the
// (batch, dim, L) tensors is 16-byte aligned and L is a whole number of its
// 8-token blocks; it groups 128 channels, the other kernel 64.
bool tc_shape(const ssm_dims* d) {
    return SSM_SCAN_TC && d->io == SSM_IO_BF16 && d->dstate == 16 && d->seqlen > 0 && d->seqlen % 8 == 0;
}

// The warp-specialised kernel serves the same shapes with L a whole number of
// its 16-token blocks, unless the chunked schedule takes the call.
bool ws_shape(const ssm_dims* d) {
    return SSM_SCAN_WS && d->io == SSM_IO_BF16 && d->dstate == 16 && d->seqlen > 0 &&
           d->seqlen % 16 == 0 && !chunk_plan(d).on;
}

// The workspace covers whichever kernel and split the call selects.
ScanWorkspace scan_workspace(const ssm_dims* d) {
    const int n = (int)d->dstate;
    ScanWorkspace w = scan_workspace_for(d, seq_channels(n, n <= 8 ? n : 8));
    if (n == 16) {
        const ScanWorkspace w4 = scan_workspace_for(d, seq_channels(16, 4));
        if (w4.total > w.total) w = w4;
    }
    if (tc_shape(d)) {
        const ScanWorkspace t = scan_workspace_for(d, ssm::tc::kCH);
        if (t.total > w.total) w = t;
    }
    if (ws_shape(d)) {
        const ScanWorkspace t = scan_workspace_for(d, ssm::ws::kCH);
        if (t.total > w.total) w = t;
    }
    const ScanWorkspace cw = chunk_workspace(chunk_plan(d), n);
    if (cw.total > w.total) w = cw;
    return w;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on the driver library)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// A (L, dim, batch) bf16 tensor as 16-token x 128-channel boxes with 32-byte
// swizzle; rows past `dim` read as zero.
bool encode_plane(CUtensorMap* m, const void* base, int64_t batch, int64_t dim, int64_t L) {
    const EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)L, (cuuint64_t)dim, (cuuint64_t)batch};
    const cuuint64_t gstride[2] = {(cuuint64_t)L * 2, (cuuint64_t)(dim * L * 2)};
    const cuuint32_t box[3] = {(cuuint32_t)ssm::tc::kTT, (cuuint32_t)ssm::tc::kCH, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool Z, bool SP>
int launch_scan_tc(ssm::ScanParams p, int64_t chunk, unsigned char* ws, cudaStream_t stream) {
    using namespace ssm::tc;
    TmaMaps maps;
    if (!encode_plane(&maps.u, p.u, p.batch, p.dim, p.L) ||
        !encode_plane(&maps.delta, p.delta, p.batch, p.dim, p.L) ||
        !encode_plane(&maps.z, Z ? p.z : p.u, p.batch, p.dim, p.L))
        return SSM_ERR_CUDA;
    auto kern = scan_fwd_tc_kernel<Z, SP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    ssm_dims d{p.batch, p.dim, 16, p.L, SSM_IO_BF16, 0};
    const ScanWorkspace wl = scan_workspace_for(&d, kCH);
    p.groups_per_row = (p.dim + kCH - 1) / kCH;
    p.ngroups = p.batch * p.groups_per_row;
    p.ntiles = p.L / kTB;   // in 8-token blocks
    int sms = 0;
    if (device_sms(&sms) != SSM_OK) return SSM_ERR_CUDA;
    int64_t ctas = sms;   // one CTA per SM: each holds all of its tensor memory
    if (ctas > p.ngroups) ctas = p.ngroups;
    if (chunk > 0) {
        const int64_t per = (chunk + kTB - 1) / kTB;
        const int64_t want = (p.ngroups * p.ntiles + per - 1) / per;
        if (want < ctas) ctas = want;
    }
    if (ctas < 1) ctas = 1;
    p.status = reinterpret_cast<int*>(ws);
    p.flags = reinterpret_cast<unsigned*>(ws + wl.flags_off);
    p.carry = reinterpret_cast<float*>(ws + wl.carry_off);
    if (cudaMemsetAsync(ws, 0, wl.clear_bytes, stream) != cudaSuccess) return SSM_ERR_CUDA;
    kern<<<(unsigned)ctas, kThreads, kSmem, stream>>>(p, maps);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <bool Z, bool SP>
int launch_scan_ws(ssm::ScanParams p, int64_t chunk, unsigned char* ws, cudaStream_t stream) {
    using namespace ssm::ws;
    TmaMaps maps;
    if (!encode_plane(&maps.u, p.u, p.batch, p.dim, p.L) ||
        !encode_plane(&maps.delta, p.delta, p.batch, p.dim, p.L) ||
        !encode_plane(&maps.z, Z ? p.z : p.u, p.batch, p.dim, p.L))
        return SSM_ERR_CUDA;
    auto kern = scan_fwd_ws_kernel<Z, SP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    ssm_dims d{p.batch, p.dim, 16, p.L, SSM_IO_BF16, 0};
    const ScanWorkspace wl = scan_workspace_for(&d, kCH);
    p.groups_per_row = (p.dim + kCH - 1) / kCH;
    p.ngroups = p.batch * p.groups_per_row;
    p.ntiles = p.L / kTB;   // in 16-token blocks
    int sms = 0;
    if (device_sms(&sms) != SSM_OK) return SSM_ERR_CUDA;
    int64_t ctas = sms;   // one CTA per SM (its shared memory)
    if (ctas > p.ngroups) ctas = p.ngroups;
    if (chunk > 0) {
        const int64_t per = (chunk + kTB - 1) / kTB;
        const int64_t want = (p.ngroups * p.ntiles + per - 1) / per;
        if (want < ctas) ctas = want;
    }
    if (ctas < 1) ctas = 1;
    p.status = reinterpret_cast<int*>(ws);
    p.flags = reinterpret_cast<unsigned*>(ws + wl.flags_off);
    p.carry = reinterpret_cast<float*>(ws + wl.carry_off);
    if (cudaMemsetAsync(ws, 0, wl.clear_bytes, stream) != cudaSuccess) return SSM_ERR_CUDA;
    kern<<<(unsigned)ctas, kThreads, kSmem, stream>>>(p, maps);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Number of CTAs of `kern` that fit on one SM (queried once per device).
template <typename K>
int occupancy(K kern, int smem, std::atomic<int>* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    int occ = cache[dev].load();
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, ssm::seq::kThreads, smem) !=
                cudaSuccess || occ < 1)
            return -1;
        cache[dev].store(occ);
    }
    return occ;
}

// Chunked schedule: the three passes on `stream`.
template <typename T, int N, int S, bool Z, bool SP, bool VEC>
int launch_chunked(ssm::ScanParams p, const ChunkPlan& c, unsigned char* ws, int sms,
                   cudaStream_t stream) {
    using namespace ssm::seq;
    using Sh = Shape<T, N, S, Z>;
    using ShA = Shape<T, N, S, false>;
    static_assert(Sh::CH == ShA::CH, "same channel groups in both passes");
    auto agg = scan_chunk_agg_kernel<T, N, S, SP, VEC>;
    auto full = scan_fwd_kernel<T, N, S, Z, SP, VEC>;
    static std::atomic<int> occ_agg[64], occ_full[64];
    const int oa = occupancy(agg, ShA::SMEM, occ_agg), of = occupancy(full, Sh::SMEM, occ_full);
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
    agg<<<(unsigned)ga, kThreads, ShA::SMEM, stream>>>(p);
    const int64_t nthr = p.ngroups * Sh::CH * N;
    scan_chunk_carry_kernel<N, Sh::CH><<<(unsigned)((nthr + 255) / 256), 256, 0, stream>>>(p);
    const int64_t gf = units < (int64_t)of * sms ? units : (int64_t)of * sms;
    full<<<(unsigned)gf, kThreads, Sh::SMEM, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N, int S, bool Z, bool SP, bool VEC>
int launch_scan(ssm::ScanParams p, int64_t chunk, unsigned char* ws, int sms,
                cudaStream_t stream) {
    using namespace ssm::seq;
    using Sh = Shape<T, N, S, Z>;
    auto kern = scan_fwd_kernel<T, N, S, Z, SP, VEC>;
    // per kernel instance: raise its shared-memory limit and ask how many
    // CTAs fit on an SM, once
    static std::atomic<int> occ_cache[64];   // per device: the attribute is per context
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSM_ERR_CUDA;
    int occ = occ_cache[dev].load();
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, Sh::SMEM) !=
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
    kern<<<(unsigned)ctas, kThreads, Sh::SMEM, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int N, int S>
int dispatch_scan_n(const ssm::ScanParams& p, int64_t chunk, bool z, bool sp, bool vec,
                    unsigned char* ws, int sms, cudaStream_t s) {
#define SSM_SCAN_CASE(Z, SP, V) \
    if (z == Z && sp == SP && vec == V) return launch_scan<T, N, S, Z, SP, V>(p, chunk, ws, sms, s);
    SSM_SCAN_CASE(false, false, false)
    SSM_SCAN_CASE(false, false, true)
    SSM_SCAN_CASE(false, true, false)
    SSM_SCAN_CASE(false, true, true)
    SSM_SCAN_CASE(true, false, false)
    SSM_SCAN_CASE(true, false, true)
    SSM_SCAN_CASE(true, true, false)
    SSM_SCAN_CASE(true, true, true)
#undef SSM_SCAN_CASE
    return SSM_ERR_BAD_DIMS;
}

template <typename T, int N, int S>
int dispatch_chunked_n(const ssm::ScanParams& p, const ChunkPlan& c, bool z, bool sp, bool vec,
                       unsigned char* ws, int sms, cudaStream_t s) {
#define SSM_CHUNK_CASE(Z, SP, V) \
    if (z == Z && sp == SP && vec == V) return launch_chunked<T, N, S, Z, SP, V>(p, c, ws, sms, s);
    SSM_CHUNK_CASE(false, false, false)
    SSM_CHUNK_CASE(false, false, true)
    SSM_CHUNK_CASE(false, true, false)
    SSM_CHUNK_CASE(false, true, true)
    SSM_CHUNK_CASE(true, false, false)
    SSM_CHUNK_CASE(true, false, true)
    SSM_CHUNK_CASE(true, true, false)
    SSM_CHUNK_CASE(true, true, true)
#undef SSM_CHUNK_CASE
    return SSM_ERR_BAD_DIMS;
}

template <typename T>
int dispatch_scan(const ssm_dims* d, const ssm::ScanParams& p, bool z, bool sp, bool vec,
                  unsigned char* ws, int sms, cudaStream_t s, int split) {
    const int64_t chunk = d->chunk;
    const ChunkPlan cp = chunk_plan(d);
    if (cp.on) {
        switch (d->dstate) {
            case 1: return dispatch_chunked_n<T, 1, 1>(p, cp, z, sp, vec, ws, sms, s);
            case 2: return dispatch_chunked_n<T, 2, 2>(p, cp, z, sp, vec, ws, sms, s);
            case 4: return dispatch_chunked_n<T, 4, 4>(p, cp, z, sp, vec, ws, sms, s);
            case 8: return dispatch_chunked_n<T, 8, 8>(p, cp, z, sp, vec, ws, sms, s);
            case 16: return dispatch_chunked_n<T, 16, 8>(p, cp, z, sp, vec, ws, sms, s);
        }
        return SSM_ERR_UNSUPPORTED_N;
    }
    switch (d->dstate) {
        case 1: return dispatch_scan_n<T, 1, 1>(p, chunk, z, sp, vec, ws, sms, s);
        case 2: return dispatch_scan_n<T, 2, 2>(p, chunk, z, sp, vec, ws, sms, s);
        case 4: return dispatch_scan_n<T, 4, 4>(p, chunk, z, sp, vec, ws, sms, s);
        case 8: return dispatch_scan_n<T, 8, 8>(p, chunk, z, sp, vec, ws, sms, s);
        case 16:
            if ((split ? split : n16_split(d, sms)) == 8)
                return dispatch_scan_n<T, 16, 8>(p, chunk, z, sp, vec, ws, sms, s);
            return dispatch_scan_n<T, 16, 4>(p, chunk, z, sp, vec, ws, sms, s);
    }
    return SSM_ERR_UNSUPPORTED_N;
}

template <typename T, int N, bool Z, bool SP, bool VEC>
int launch_step(const ssm::StepParams& p, cudaStream_t stream) {
    constexpr int kG = ssm::StepShape<N>::kG;
    const int64_t threads = p.batch * p.dim * kG;
    const int64_t blocks = (threads + ssm::kStepThreads - 1) / ssm::kStepThreads;
    if (blocks > INT32_MAX) return SSM_ERR_BAD_DIMS;
    ssm::state_step_kernel<T, N, Z, SP, VEC><<<(unsigned)blocks, ssm::kStepThreads, 0, stream>>>(p);
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
int dispatch_step(const ssm::StepParams& p, int64_t n, bool z, bool sp, bool vec, cudaStream_t s) {
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

namespace {

// The scan; split (N = 16 only): 0 picks the state split from the sizes, 4 or
// 8 forces it (the host entry point keeps its slices on the full problem's
// choice).
int scan_fwd_impl(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                  const void* B, const void* C, const float* D, const void* z,
                  const float* delta_bias, int delta_softplus, void* y, float* last_state,
                  void* workspace, size_t workspace_bytes, void* stream, int split) {
    Sizes s;
    int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    // With L = 0 the (batch, dim, L) and (batch, L, N) tensors are empty and
    // may be NULL; only last_state is written (zeros).
    const bool empty = dims->seqlen == 0;
    if (!A || (!empty && (!u || !delta || !B || !C || !y))) return SSM_ERR_NULL_ARG;
    const size_t es = io_size(dims->io);
    for (const void* q : {u, delta, B, C, z, static_cast<const void*>(y)})
        if (q && !aligned(q, es)) return SSM_ERR_MISALIGNED;
    for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D),
                          static_cast<const void*>(delta_bias),
                          static_cast<const void*>(last_state)})
        if (q && !aligned(q, 4)) return SSM_ERR_MISALIGNED;
    const Range in[] = {{u, s.seq * (int64_t)es}, {delta, s.seq * (int64_t)es},
                        {z, s.seq * (int64_t)es}, {B, s.bc * (int64_t)es},
                        {C, s.bc * (int64_t)es},  {A, s.par * 4},
                        {D, dims->dim * 4},       {delta_bias, dims->dim * 4}};
    const Range out_y{y, s.seq * (int64_t)es}, out_h{last_state, s.state * 4};
    for (const Range& r : in)
        if (overlap(r, out_y) || overlap(r, out_h)) return SSM_ERR_ALIAS;
    if (overlap(out_y, out_h)) return SSM_ERR_ALIAS;

    const ScanWorkspace wl = scan_workspace(dims);
    if (wl.total > 0) {
        if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256))
            return SSM_ERR_WORKSPACE;
        const Range ws{workspace, (int64_t)wl.total};
        for (const Range& r : in)
            if (overlap(r, ws)) return SSM_ERR_ALIAS;
        if (overlap(out_y, ws) || overlap(out_h, ws)) return SSM_ERR_ALIAS;
    }
    ssm::ScanParams p{};
    p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.bias = delta_bias; p.y = y; p.last_state = last_state;
    p.batch = dims->batch; p.dim = dims->dim; p.L = dims->seqlen;
    // 16-byte vector path: every row of u/delta/z/y starts on a 16-byte boundary
    const bool vec = (dims->seqlen * (int64_t)es) % 16 == 0 && aligned(u, 16) &&
                     aligned(delta, 16) && aligned(y, 16) && (!z || aligned(z, 16)) &&
                     aligned(B, 16) && aligned(C, 16);
    const bool sp = delta_softplus != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int sms = 0;
    if (device_sms(&sms) != SSM_OK) return SSM_ERR_CUDA;
    if (vec && ws_shape(dims)) {
        const bool zz = z != nullptr;
        if (zz && sp) return launch_scan_ws<true, true>(p, dims->chunk, ws, st);
        if (zz) return launch_scan_ws<true, false>(p, dims->chunk, ws, st);
        if (sp) return launch_scan_ws<false, true>(p, dims->chunk, ws, st);
        return launch_scan_ws<false, false>(p, dims->chunk, ws, st);
    }
    if (vec && tc_shape(dims)) {
        const bool zz = z != nullptr;
        if (zz && sp) return launch_scan_tc<true, true>(p, dims->chunk, ws, st);
        if (zz) return launch_scan_tc<true, false>(p, dims->chunk, ws, st);
        if (sp) return launch_scan_tc<false, true>(p, dims->chunk, ws, st);
        return launch_scan_tc<false, false>(p, dims->chunk, ws, st);
    }
    if (dims->io == SSM_IO_BF16)
        return dispatch_scan<bf16>(dims, p, z != nullptr, sp, vec, ws, sms, st, split);
    return dispatch_scan<float>(dims, p, z != nullptr, sp, vec, ws, sms, st, split);
}

}  // namespace

extern "C" {

int ssm_version(void) { return kVersion; }

const char* ssm_status_string(int status) {
    switch (status) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL_ARG: return "a required pointer is NULL";
        case SSM_ERR_BAD_DIMS: return "a size is out of range or overflows";
        case SSM_ERR_UNSUPPORTED_N: return "dstate must be 1, 2, 4, 8 or 16";
        case SSM_ERR_BAD_DTYPE: return "unknown I/O element type";
        case SSM_ERR_MISALIGNED: return "a pointer is not aligned to its element size";
        case SSM_ERR_CUDA: return "the CUDA runtime refused the launch";
        case SSM_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case SSM_ERR_ALIAS: return "an output buffer overlaps an input buffer";
        case SSM_ERR_TIMEOUT: return "a bounded on-device wait gave up";
        case SSM_ERR_TOO_LARGE:
            return "the problem needs more scratch than the library's built-in buffer holds";
    }
    return "unknown status";
}

int ssm_probe_ex2(int32_t blocks, int32_t threads, int32_t iters, float* sink, void* stream) {
    if (!sink) return SSM_ERR_NULL_ARG;
    if (blocks < 1 || iters < 1 || threads < 32 || threads > 1024 || threads % 32 != 0)
        return SSM_ERR_BAD_DIMS;
    ssm::probe_ex2_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(iters, sink);
    return cudaPeekAtLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_scan_fwd_workspace_size(const ssm_dims* dims, size_t* bytes) {
    Sizes s;
    const int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    if (!bytes) return SSM_ERR_NULL_ARG;
    *bytes = scan_workspace(dims).total;
    return SSM_OK;
}

int ssm_scan_fwd(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus, void* y, float* last_state,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return scan_fwd_impl(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                         workspace, workspace_bytes, stream, 0);
}

int ssm_state_step(const ssm_dims* dims, float* state, const void* x, const void* delta,
                   const float* A, const void* B, const void* C, const float* D, const void* z,
                   const float* delta_bias, int delta_softplus, void* y, void* stream) {
    Sizes s;
    int rc = check_dims(dims, false, &s);
    if (rc != SSM_OK) return rc;
    if (!state || !x || !delta || !A || !B || !C || !y) return SSM_ERR_NULL_ARG;
    const size_t es = io_size(dims->io);
    for (const void* q : {x, delta, B, C, z, static_cast<const void*>(y)})
        if (q && !aligned(q, es)) return SSM_ERR_MISALIGNED;
    for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D),
                          static_cast<const void*>(delta_bias), static_cast<const void*>(state)})
        if (q && !aligned(q, 4)) return SSM_ERR_MISALIGNED;
    const Range in[] = {{x, s.chan * (int64_t)es}, {delta, s.chan * (int64_t)es},
                        {z, s.chan * (int64_t)es}, {B, dims->batch * dims->dstate * (int64_t)es},
                        {C, dims->batch * dims->dstate * (int64_t)es}, {A, s.par * 4},
                        {D, dims->dim * 4}, {delta_bias, dims->dim * 4}};
    const Range out_y{y, s.chan * (int64_t)es}, io_h{state, s.state * 4};
    for (const Range& r : in)
        if (overlap(r, out_y) || overlap(r, io_h)) return SSM_ERR_ALIAS;
    if (overlap(out_y, io_h)) return SSM_ERR_ALIAS;

    ssm::StepParams p{state, x, delta, A, B, C, D, z, delta_bias, y, dims->batch, dims->dim};
    const bool vec = aligned(state, 16);
    const bool sp = delta_softplus != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->io == SSM_IO_BF16) return dispatch_step<bf16>(p, dims->dstate, z != nullptr, sp, vec, st);
    return dispatch_step<float>(p, dims->dstate, z != nullptr, sp, vec, st);
}

// ---------------------------------------------------------------------------
// Backward scan.

}  // extern "C"

namespace {

size_t bwd_workspace(const ssm_dims* d) {
    const int64_t ntiles = (d->seqlen + ssm::bwd::kTT - 1) / ssm::bwd::kTT;
    return (size_t)d->batch * d->dim * ntiles * d->dstate * sizeof(float);
}

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
int dispatch_bwd(const ssm::bwd::BwdParams& p, int64_t n, bool z, bool sp, cudaStream_t st) {
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

extern "C" {

int ssm_scan_bwd_workspace_size(const ssm_dims* dims, size_t* bytes) {
    if (!bytes) return SSM_ERR_NULL_ARG;
    Sizes s;
    const int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    *bytes = bwd_workspace(dims);
    return SSM_OK;
}

int ssm_scan_bwd(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus, const float* dy,
                 const float* dlast_state, float* du, float* ddelta, float* dz, float* dA,
                 float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                 void* workspace, size_t workspace_bytes, void* stream) {
    Sizes s;
    int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    const bool empty = dims->seqlen == 0;
    if (!A || !dA || (!empty && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)))
        return SSM_ERR_NULL_ARG;
    if (z && !empty && !dz) return SSM_ERR_NULL_ARG;
    const size_t es = io_size(dims->io);
    for (const void* q : {u, delta, B, C, z})
        if (!aligned(q, es)) return SSM_ERR_MISALIGNED;
    for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D),
                          static_cast<const void*>(delta_bias), static_cast<const void*>(dy),
                          static_cast<const void*>(dlast_state), static_cast<const void*>(du),
                          static_cast<const void*>(ddelta), static_cast<const void*>(dz),
                          static_cast<const void*>(dA), static_cast<const void*>(dB),
                          static_cast<const void*>(dC), static_cast<const void*>(dD),
                          static_cast<const void*>(ddelta_bias), static_cast<const void*>(dh0)})
        if (!aligned(q, 4)) return SSM_ERR_MISALIGNED;
    const size_t need = bwd_workspace(dims);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the accumulated gradients start from zero
    const int64_t N = dims->dstate;
    if (cudaMemsetAsync(dA, 0, (size_t)dims->dim * N * 4, st) != cudaSuccess) return SSM_ERR_CUDA;
    if (!empty) {
        if (cudaMemsetAsync(dB, 0, (size_t)s.bc * 4, st) != cudaSuccess ||
            cudaMemsetAsync(dC, 0, (size_t)s.bc * 4, st) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    if (dD && cudaMemsetAsync(dD, 0, (size_t)dims->dim * 4, st) != cudaSuccess) return SSM_ERR_CUDA;
    if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)dims->dim * 4, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    ssm::bwd::BwdParams p{u, delta, A, B, C, D, z && !empty ? z : nullptr, delta_bias, dy,
                          dlast_state, du, ddelta, z ? dz : nullptr, dA, dB, dC,
                          D ? dD : nullptr, delta_bias ? ddelta_bias : nullptr, dh0,
                          static_cast<float*>(workspace), dims->batch, dims->dim, dims->seqlen,
                          (dims->seqlen + ssm::bwd::kTT - 1) / ssm::bwd::kTT};
    if (empty) p.z = nullptr;
    const bool zz = p.z != nullptr, sp = delta_softplus != 0;
    if (dims->io == SSM_IO_BF16) return dispatch_bwd<bf16>(p, N, zz, sp, st);
    return dispatch_bwd<float>(p, N, zz, sp, st);
}

// ---------------------------------------------------------------------------
// Forward scan from host buffers.
//
// Batch rows, and channel ranges within a row, are independent scans, so the
// problem is cut into slices (one batch row, or a range of its channels,
// each) that pass through three streams: copy in (H2D) on one, the scan on
// the caller's stream, copy out (D2H) on a third, with two sets of device
// buffers.  Slice k's copy in overlaps slice k-1's scan and slice k-2's copy
// out; with pinned host memory the time approaches that of the copies in.

}  // extern "C"

namespace {

struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
};
std::mutex g_host_mu;
HostStreams g_host_streams[64];

int host_streams(HostStreams* hs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostStreams& h = g_host_streams[dev];
    if (!h.in) {
        if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess) return SSM_ERR_CUDA;
        if (cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(h.in);
            h.in = nullptr;
            return SSM_ERR_CUDA;
        }
    }
    *hs = h;
    return SSM_OK;
}

// Events of one call: the copies in of a buffer set done, its scan done, its
// copies out done; plus the start fence.
struct HostEvents {
    cudaEvent_t ev[7] = {};
    int n = 0;
    ~HostEvents() {
        for (int i = 0; i < n; i++) cudaEventDestroy(ev[i]);
    }
    bool make() {
        for (n = 0; n < 7; n++)
            if (cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming) != cudaSuccess) return false;
        return true;
    }
};

}  // namespace

extern "C" {

int ssm_scan_fwd_host(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                      const void* B, const void* C, const float* D, const void* z,
                      const float* delta_bias, int delta_softplus, void* y, float* last_state,
                      void* stream) {
    Sizes s;
    int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    const bool empty = dims->seqlen == 0;
    if (!A || (!empty && (!u || !delta || !B || !C || !y))) return SSM_ERR_NULL_ARG;
    const size_t es = io_size(dims->io);
    const int64_t batch = dims->batch, dim = dims->dim, N = dims->dstate, L = dims->seqlen;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // slices: every batch row cut into `parts` channel ranges, at least 16
    // slices in all when the rows allow it (the pipeline's fill and drain
    // cost about one slice's copies and scan)
    int64_t parts = (16 + batch - 1) / batch;
    if (parts > dim) parts = dim;
    const int64_t cw = (dim + parts - 1) / parts;   // channels per slice (the last may be fewer)
    parts = (dim + cw - 1) / cw;
    const int64_t nslices = batch * parts;

    // the slices take the kernel the whole problem would: its state split and
    // its chunk boundaries (or no chunking), so the outputs are the same
    int sms = 0;
    if (device_sms(&sms) != SSM_OK) return SSM_ERR_CUDA;
    const ChunkPlan full = chunk_plan(dims);
    int64_t sc = dims->chunk;
    if (full.on) sc = full.tpc * ssm::seq::kTL;
    else if (sc == 0) sc = L;
    const int32_t slice_chunk = (int32_t)(sc > INT32_MAX ? INT32_MAX : sc);
    const int split = (N == 16 && !full.on) ? n16_split(dims, sms) : 0;

    ssm_dims sd{1, cw, N, L, dims->io, slice_chunk};
    size_t ws_bytes = 0;
    if ((rc = ssm_scan_fwd_workspace_size(&sd, &ws_bytes)) != SSM_OK) return rc;

    // device layout: parameters, workspace, then two buffer sets
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t seq_b = (size_t)cw * L * es, bc_b = (size_t)L * N * es, st_b = (size_t)cw * N * 4;
    const size_t off_A = 0, off_D = up(off_A + (size_t)dim * N * 4), off_bias = up(off_D + (size_t)dim * 4);
    const size_t off_ws = up(off_bias + (size_t)dim * 4);
    const size_t off_set = up(off_ws + ws_bytes);
    const size_t o_u = 0, o_dl = up(seq_b), o_z = o_dl + up(seq_b), o_B = o_z + up(seq_b),
                 o_C = o_B + up(bc_b), o_y = o_C + up(bc_b), o_h = o_y + up(seq_b);
    const size_t set_b = o_h + up(st_b);
    const size_t total = off_set + 2 * set_b;

    HostStreams hs;
    if ((rc = host_streams(&hs)) != SSM_OK) return rc;
    HostEvents he;
    if (!he.make()) return SSM_ERR_CUDA;
    cudaEvent_t ev_in[2] = {he.ev[0], he.ev[1]}, ev_scan[2] = {he.ev[2], he.ev[3]},
                ev_out[2] = {he.ev[4], he.ev[5]}, ev_start = he.ev[6];

    unsigned char* dev = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void**>(&dev), total, st) != cudaSuccess) return SSM_ERR_CUDA;
    bool ok = cudaEventRecord(ev_start, st) == cudaSuccess &&
              cudaStreamWaitEvent(hs.in, ev_start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hs.out, ev_start, 0) == cudaSuccess;
    float* dA = reinterpret_cast<float*>(dev + off_A);
    float* dD = D ? reinterpret_cast<float*>(dev + off_D) : nullptr;
    float* dbias = delta_bias ? reinterpret_cast<float*>(dev + off_bias) : nullptr;
    ok = ok && cudaMemcpyAsync(dA, A, (size_t)dim * N * 4, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
    if (D) ok = ok && cudaMemcpyAsync(dD, D, (size_t)dim * 4, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
    if (delta_bias)
        ok = ok && cudaMemcpyAsync(dbias, delta_bias, (size_t)dim * 4, cudaMemcpyHostToDevice, hs.in) ==
                       cudaSuccess;

    const unsigned char* hu = static_cast<const unsigned char*>(u);
    const unsigned char* hdl = static_cast<const unsigned char*>(delta);
    const unsigned char* hz = static_cast<const unsigned char*>(z);
    const unsigned char* hB = static_cast<const unsigned char*>(B);
    const unsigned char* hC = static_cast<const unsigned char*>(C);
    unsigned char* hy = static_cast<unsigned char*>(y);
    for (int64_t k = 0; ok && k < nslices; k++) {
        const int set = (int)(k & 1);
        const int64_t b = k / parts, d0 = (k % parts) * cw;
        const int64_t w = dim - d0 < cw ? dim - d0 : cw;   // channels of this slice
        unsigned char* sb = dev + off_set + set * set_b;
        const size_t row = (size_t)(b * dim + d0);         // first flat (b, d) row
        const size_t nseq = (size_t)w * L * es;
        // copy in, once the set's previous slice has been copied out
        if (k >= 2) ok = ok && cudaStreamWaitEvent(hs.in, ev_out[set], 0) == cudaSuccess;
        if (nseq > 0) {
            ok = ok && cudaMemcpyAsync(sb + o_u, hu + row * L * es, nseq, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(sb + o_dl, hdl + row * L * es, nseq, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
            if (z) ok = ok && cudaMemcpyAsync(sb + o_z, hz + row * L * es, nseq, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(sb + o_B, hB + (size_t)b * L * N * es, bc_b, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(sb + o_C, hC + (size_t)b * L * N * es, bc_b, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
        }
        ok = ok && cudaEventRecord(ev_in[set], hs.in) == cudaSuccess;
        // the scan of the slice
        ok = ok && cudaStreamWaitEvent(st, ev_in[set], 0) == cudaSuccess;
        if (ok) {
            ssm_dims d1{1, w, N, L, dims->io, slice_chunk};
            rc = scan_fwd_impl(&d1, sb + o_u, sb + o_dl, dA + d0 * N, sb + o_B, sb + o_C,
                              dD ? dD + d0 : nullptr, z ? sb + o_z : nullptr, dbias ? dbias + d0 : nullptr,
                              delta_softplus, sb + o_y, last_state ? reinterpret_cast<float*>(sb + o_h) : nullptr,
                              ws_bytes ? dev + off_ws : nullptr, ws_bytes, st, split);
            ok = rc == SSM_OK;
        }
        ok = ok && cudaEventRecord(ev_scan[set], st) == cudaSuccess;
        // copy out
        ok = ok && cudaStreamWaitEvent(hs.out, ev_scan[set], 0) == cudaSuccess;
        if (nseq > 0)
            ok = ok && cudaMemcpyAsync(hy + row * L * es, sb + o_y, nseq, cudaMemcpyDeviceToHost, hs.out) == cudaSuccess;
        if (last_state)
            ok = ok && cudaMemcpyAsync(last_state + row * N, sb + o_h, (size_t)w * N * 4, cudaMemcpyDeviceToHost, hs.out) ==
                           cudaSuccess;
        ok = ok && cudaEventRecord(ev_out[set], hs.out) == cudaSuccess;
    }
    // join: the caller's stream waits for the last copies out, then frees
    if (ok) ok = cudaStreamWaitEvent(st, ev_out[0], 0) == cudaSuccess;
    if (ok && nslices > 1) ok = cudaStreamWaitEvent(st, ev_out[1], 0) == cudaSuccess;
    if (ok) ok = cudaStreamWaitEvent(st, ev_in[0], 0) == cudaSuccess;   // (covers the parameter copies)
    if (!ok) {
        // an enqueue failed: wait for what was enqueued before freeing
        cudaStreamSynchronize(hs.in);
        cudaStreamSynchronize(hs.out);
        cudaStreamSynchronize(st);
        cudaFree(dev);
        return rc != SSM_OK ? rc : SSM_ERR_CUDA;
    }
    return cudaFreeAsync(dev, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free forward scan.
//
// Some callers cannot allocate device memory when they call the scan: an
// inference engine's plugin that must live inside a memory plan fixed before
// it runs, or code on a real-time or safety-critical path where allocation is
// forbidden.  For them the scan's scratch (the status word, hand-over flags
// and carried states) lives in this fixed device buffer instead of a
// caller-supplied workspace.  Every device that loads the library holds the
// buffer until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;   // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];   // device address of g_noalloc_scratch, per device

// The buffer's device address on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSM_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SSM_OK;
}

}  // namespace

int ssm_scan_fwd_noalloc(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                         const void* B, const void* C, const float* D, const void* z,
                         const float* delta_bias, int delta_softplus, void* y,
                         float* last_state, void* stream) {
    size_t need = 0;
    const int rc = ssm_scan_fwd_workspace_size(dims, &need);
    if (rc != SSM_OK) return rc;
    if (need > kNoAllocScratchBytes) return SSM_ERR_TOO_LARGE;
    void* scratch = nullptr;
    if (need > 0) {
        const int rs = noalloc_scratch(&scratch);
        if (rs != SSM_OK) return rs;
    }
    return ssm_scan_fwd(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                        scratch, need > 0 ? kNoAllocScratchBytes : 0, stream);
}

size_t ssm_scan_fwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

}  // extern "C"
