// C ABI of the selective-scan library: argument checks on the host, then a
// launch of the kernel instance that matches (I/O type, N, gate, softplus,
// alignment) on the caller's stream.  See include/ssm_scan.h for the contract.
#include "ssm_scan.h"

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "host_plan.h"
#include "probe.cuh"


using namespace ssm_host;

static_assert(ssm::kStatusTimeout == SSM_ERR_TIMEOUT, "device and host timeout codes agree");
static_assert(ssm::kStatusDevice == SSM_ERR_DEVICE, "device and host debug codes agree");

namespace {

using bf16 = __nv_bfloat16;

constexpr int kVersion = 100;  // 0.1.0

// The kernel instance for these sizes and options.  split (N = 16 only): 0
// picks the state split from the sizes, 4 or 8 forces it.
int dispatch_scan(const ssm_dims* d, const ssm::ScanParams& p, bool zoh, bool conv, bool vec,
                  unsigned char* ws, int sms, cudaStream_t s, int split) {
    const bool bf = d->io == SSM_IO_BF16;
    const int n = (int)d->dstate;
    const ChunkPlan cp = chunk_plan(d);
    if (cp.on)
        return bf ? fwd_chunked_bf16(n, p, cp, zoh, conv, vec, ws, sms, s)
                  : fwd_chunked_f32(n, p, cp, zoh, conv, vec, ws, sms, s);
    if (n == 16) {
        const int sp16 = split ? split : n16_split(d, sms);
        return bf ? fwd_scan_bf16_n16(sp16, p, d->chunk, zoh, conv, vec, ws, sms, s)
                  : fwd_scan_f32_n16(sp16, p, d->chunk, zoh, conv, vec, ws, sms, s);
    }
    return bf ? fwd_scan_bf16_small(n, p, d->chunk, zoh, conv, vec, ws, sms, s)
              : fwd_scan_f32_small(n, p, d->chunk, zoh, conv, vec, ws, sms, s);
}

}  // namespace


namespace {

// The scan; split (N = 16 only): 0 picks the state split from the sizes, 4 or
// 8 forces it (the host entry point keeps its slices on the full problem's
// choice).
int scan_fwd_impl(const ssm_dims* dims, const ssm_scan_opts* opts, const void* u,
                  const void* delta, const float* A, const void* B, const void* C,
                  const float* D, const void* z, const float* delta_bias, int delta_softplus,
                  void* y, float* last_state, void* workspace, size_t workspace_bytes,
                  void* stream, int split) {
    Sizes s;
    int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    const ssm_scan_opts none{};
    const ssm_scan_opts& o = opts ? *opts : none;
    if (o.input_term != SSM_INPUT_DELTA_B && o.input_term != SSM_INPUT_ZOH) return SSM_ERR_BAD_OPTION;
    if (o.conv_width < 0 || o.conv_width > 4 || o.wait_limit < 0) return SSM_ERR_BAD_OPTION;
    const bool conv = o.conv_width > 0;
    if (conv && !o.conv_weight) return SSM_ERR_NULL_ARG;
    // With L = 0 the (batch, dim, L) and (batch, L, N) tensors are empty and
    // may be NULL; only last_state is written (the initial state).
    const bool empty = dims->seqlen == 0;
    if (!A || (!empty && (!u || !delta || !B || !C || !y))) return SSM_ERR_NULL_ARG;
    const size_t es = io_size(dims->io);
    const void* u_out = conv ? o.u_out : nullptr;
    const void* cstate = conv ? o.conv_state : nullptr;
    for (const void* q : {u, delta, B, C, z, static_cast<const void*>(y), u_out, cstate})
        if (q && !aligned(q, es)) return SSM_ERR_MISALIGNED;
    for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D),
                          static_cast<const void*>(delta_bias),
                          static_cast<const void*>(last_state), static_cast<const void*>(o.h0),
                          static_cast<const void*>(conv ? o.conv_weight : nullptr),
                          static_cast<const void*>(conv ? o.conv_bias : nullptr)})
        if (q && !aligned(q, 4)) return SSM_ERR_MISALIGNED;
    const int64_t K = o.conv_width;
    const Range in[] = {{u, s.seq * (int64_t)es}, {delta, s.seq * (int64_t)es},
                        {z, s.seq * (int64_t)es}, {B, s.bc * (int64_t)es},
                        {C, s.bc * (int64_t)es},  {A, s.par * 4},
                        {D, dims->dim * 4},       {delta_bias, dims->dim * 4},
                        {conv ? o.conv_weight : nullptr, dims->dim * K * 4},
                        {conv ? o.conv_bias : nullptr, dims->dim * 4},
                        {cstate, s.chan * (K > 0 ? K - 1 : 0) * (int64_t)es}};
    const Range out_y{y, s.seq * (int64_t)es}, out_h{last_state, s.state * 4},
        out_u{u_out, s.seq * (int64_t)es}, in_h0{o.h0, s.state * 4};
    for (const Range& r : in)
        if (overlap(r, out_y) || overlap(r, out_h) || overlap(r, out_u)) return SSM_ERR_ALIAS;
    if (overlap(out_y, out_h) || overlap(out_y, out_u) || overlap(out_h, out_u))
        return SSM_ERR_ALIAS;
    // the initial state may be last_state itself (a state continued in place),
    // but no other output
    if (overlap(in_h0, out_y) || overlap(in_h0, out_u)) return SSM_ERR_ALIAS;
    if (overlap(in_h0, out_h) && o.h0 != last_state) return SSM_ERR_ALIAS;

    const ScanWorkspace wl = scan_workspace(dims);
    if (wl.total > 0) {
        if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256))
            return SSM_ERR_WORKSPACE;
        const Range ws{workspace, (int64_t)wl.total};
        for (const Range& r : in)
            if (overlap(r, ws)) return SSM_ERR_ALIAS;
        if (overlap(out_y, ws) || overlap(out_h, ws) || overlap(out_u, ws) || overlap(in_h0, ws))
            return SSM_ERR_ALIAS;
    }
    ssm::ScanParams p{};
    p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.bias = delta_bias; p.y = y; p.last_state = last_state;
    p.batch = dims->batch; p.dim = dims->dim; p.L = dims->seqlen;
    // 16-byte vector path: every row of u/delta/z/y (and u_out) starts on a
    // 16-byte boundary
    const bool vec = (dims->seqlen * (int64_t)es) % 16 == 0 && aligned(u, 16) &&
                     aligned(delta, 16) && aligned(y, 16) && (!z || aligned(z, 16)) &&
                     aligned(B, 16) && aligned(C, 16) && (!u_out || aligned(u_out, 16));
    p.gate = z != nullptr;
    p.softplus = delta_softplus != 0;
    p.h0 = o.h0;
    p.wait_limit = o.wait_limit > 0 ? o.wait_limit : (1l << 22);
    p.skip_handoff = o.test_skip_handoff != 0;
    if (conv) {
        p.conv_w = o.conv_weight;
        p.conv_b = o.conv_bias;
        p.conv_state = cstate;
        p.u_out = const_cast<void*>(u_out);
        p.conv_k = (int)K;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int sms = 0;
    if (device_sms(&sms) != SSM_OK) return SSM_ERR_CUDA;
    return dispatch_scan(dims, p, o.input_term == SSM_INPUT_ZOH, conv, vec, ws, sms, st, split);
}

}  // namespace

extern "C" {

int ssm_version(void) { return kVersion; }

#ifndef SSM_BUILD_ID
#define SSM_BUILD_ID "unknown"
#endif
const char* ssm_build_id(void) { return SSM_BUILD_ID; }

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
        case SSM_ERR_BAD_OPTION: return "an option of ssm_scan_opts is out of range";
        case SSM_ERR_DEVICE: return "a bounds check of the debug build failed on the device";
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
    return scan_fwd_impl(dims, nullptr, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y,
                         last_state, workspace, workspace_bytes, stream, 0);
}

}  // extern "C"

namespace {

// The outcome the scan left in a workspace header (see ssm_scan_fwd_status).
int read_status(const void* header, cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSM_ERR_CUDA;
    int32_t w[4] = {0, 0, 0, 0};
    if (cudaMemcpy(w, header, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return SSM_ERR_CUDA;
    if (w[ssm::kHdrDebug] != 0) return SSM_ERR_DEVICE;
    return w[ssm::kHdrStatus] == ssm::kStatusTimeout ? SSM_ERR_TIMEOUT : SSM_OK;
}

}  // namespace

extern "C" {

int ssm_scan_fwd_status(const void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace) return SSM_OK;
    if (workspace_bytes < 16 || !aligned(workspace, 256)) return SSM_ERR_WORKSPACE;
    return read_status(workspace, static_cast<cudaStream_t>(stream));
}

int ssm_scan_fwd_ex(const ssm_dims* dims, const ssm_scan_opts* opts, const void* u,
                    const void* delta, const float* A, const void* B, const void* C,
                    const float* D, const void* z, const float* delta_bias, int delta_softplus,
                    void* y, float* last_state, void* workspace, size_t workspace_bytes,
                    void* stream) {
    return scan_fwd_impl(dims, opts, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y,
                         last_state, workspace, workspace_bytes, stream, 0);
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
    const bool vec = aligned(state, 16) && aligned(A, 16) && aligned(B, 16) && aligned(C, 16);
    const bool sp = delta_softplus != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int n = (int)dims->dstate;
    if (dims->io == SSM_IO_BF16) return step_bf16(n, p, z != nullptr, sp, vec, st);
    return step_f32(n, p, z != nullptr, sp, vec, st);
}

// ---------------------------------------------------------------------------
// Backward scan.

}  // extern "C"

namespace {

}  // namespace

namespace ssm_host {
// bf16 I/O with du, ddelta, dz written in bf16 (bwd_gio.cu, bwd_zoh_gio.cu).
int bwd_bf16_gio(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st);
int bwd_zoh_bf16_gio(int n, const ssm::bwd::BwdParams& p, bool z, bool sp, cudaStream_t st);
}  // namespace ssm_host

namespace {

// Chunk plan and workspace of the backward scan.  dims->chunk > 0: chunks
// of that many tokens (rounded up to a multiple of 32), one chunk when it is
// >= seqlen.  0: a sequence of at least 8192 tokens is chunked by itself when
// its grid would hold fewer than 640 one-warp CTAs (about half of what 148
// SMs hold), into about 4608 CTAs' worth of chunks of at least 2048 tokens:
// several waves, so that the last one's share is small (at the DNA-like
// shape 1 x 1024 x 2^20 with two channels per thread: 18 chunks, one wave,
// 35.2 ms; 20 chunks, a second wave of 96 CTAs, 48.3 ms; 72 chunks 34.0 ms).
// Chunks never exceed the 65535 of grid z.
// Workspace: the checkpoints (batch, dim, ceil(L / 8), N), then with more
// than one chunk six (nchunks, batch, dim, N) arrays: the states before the
// chunks, the adjoints into them, and the maps F, PF, Q, PQ.
struct BwdPlan {
    int64_t chunk_len;
    int nchunks;
    size_t ckpt_bytes, arr_bytes, total;
};

size_t round16(int64_t v) { return (size_t)((v + 15) / 16 * 16); }

BwdPlan bwd_plan(const ssm_dims* d) {
    const int64_t L = d->seqlen, N = d->dstate, rows = d->batch * d->dim;
    const int64_t al = ssm::bwd::kChunkAlign;
    int64_t len = L;
    if (d->chunk > 0 && d->chunk < L) {
        len = ((int64_t)d->chunk + al - 1) / al * al;
    } else if (d->chunk == 0 && L >= ssm::bwd::kChunkedSeq) {
        const int64_t cpc = ssm::bwd::channels_per_cta(
            (int)N, ssm::bwd::channels_per_thread((int)N, d->batch, d->dim, L));
        const int64_t ctas = d->batch * ((d->dim + cpc - 1) / cpc);
        if (ctas < 640) {
            const int64_t want = (4608 + ctas - 1) / ctas;
            len = ((L + want - 1) / want + al - 1) / al * al;
            if (len < 2048) len = 2048;
        }
    }
    const int64_t cap = ((L + 65534) / 65535 + al - 1) / al * al;
    if (len < cap) len = cap;
    BwdPlan pl;
    pl.nchunks = len >= L ? 1 : (int)((L + len - 1) / len);
    pl.chunk_len = pl.nchunks == 1 ? (L > 1 ? L : 1) : len;
    const int64_t ntiles = (L + ssm::bwd::kTT - 1) / ssm::bwd::kTT;
    pl.ckpt_bytes = round16(rows * ntiles * N * 4);
    pl.arr_bytes = pl.nchunks > 1 ? round16((int64_t)pl.nchunks * rows * N * 4) : 0;
    pl.total = pl.ckpt_bytes + 6 * pl.arr_bytes;
    return pl;
}

size_t bwd_workspace(const ssm_dims* d) { return bwd_plan(d).total; }

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

int ssm_scan_bwd_ex(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                    const void* B, const void* C, const float* D, const void* z,
                    const float* delta_bias, int delta_softplus, const void* dy,
                    const float* dlast_state, const float* h0, int input_term, int grad_io,
                    void* du, void* ddelta, void* dz, float* dA, float* dB, float* dC, float* dD,
                    float* ddelta_bias, float* dh0, void* workspace, size_t workspace_bytes,
                    void* stream) {
    Sizes s;
    int rc = check_dims(dims, true, &s);
    if (rc != SSM_OK) return rc;
    if (input_term != SSM_INPUT_DELTA_B && input_term != SSM_INPUT_ZOH) return SSM_ERR_BAD_OPTION;
    if (grad_io != SSM_IO_F32 && grad_io != dims->io) return SSM_ERR_BAD_DTYPE;
    const bool gio = grad_io == SSM_IO_BF16;   // du, ddelta, dz in bf16
    const bool empty = dims->seqlen == 0;
    if (!A || !dA || (!empty && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)))
        return SSM_ERR_NULL_ARG;
    if (z && !empty && !dz) return SSM_ERR_NULL_ARG;
    const size_t es = io_size(dims->io);
    for (const void* q : {u, delta, B, C, z})
        if (!aligned(q, es)) return SSM_ERR_MISALIGNED;
    for (const void* q : {dy, static_cast<const void*>(du), static_cast<const void*>(ddelta),
                          static_cast<const void*>(dz)})
        if (!aligned(q, io_size(grad_io))) return SSM_ERR_MISALIGNED;
    for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D),
                          static_cast<const void*>(delta_bias),
                          static_cast<const void*>(dlast_state), static_cast<const void*>(h0),
                          static_cast<const void*>(dA), static_cast<const void*>(dB),
                          static_cast<const void*>(dC), static_cast<const void*>(dD),
                          static_cast<const void*>(ddelta_bias), static_cast<const void*>(dh0)})
        if (!aligned(q, 4)) return SSM_ERR_MISALIGNED;
    const BwdPlan pl = bwd_plan(dims);
    const size_t need = pl.total;
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
                          dlast_state, h0, du, ddelta, z ? dz : nullptr, dA, dB, dC,
                          D ? dD : nullptr, delta_bias ? ddelta_bias : nullptr, dh0,
                          static_cast<float*>(workspace), nullptr, nullptr, nullptr,
                          dims->batch, dims->dim, dims->seqlen,
                          (dims->seqlen + ssm::bwd::kTT - 1) / ssm::bwd::kTT, pl.chunk_len,
                          pl.nchunks};
    if (pl.nchunks > 1) {
        unsigned char* ws = static_cast<unsigned char*>(workspace) + pl.ckpt_bytes;
        p.hc = reinterpret_cast<float*>(ws);
        p.xc = reinterpret_cast<float*>(ws + pl.arr_bytes);
        p.agg = reinterpret_cast<float*>(ws + 2 * pl.arr_bytes);
    }
    if (empty) p.z = nullptr;
    const bool zz = p.z != nullptr, sp = delta_softplus != 0;
    if (input_term == SSM_INPUT_ZOH) {
        if (dims->io == SSM_IO_BF16)
            return gio ? bwd_zoh_bf16_gio((int)N, p, zz, sp, st) : bwd_zoh_bf16((int)N, p, zz, sp, st);
        return bwd_zoh_f32((int)N, p, zz, sp, st);
    }
    if (dims->io == SSM_IO_BF16)
        return gio ? bwd_bf16_gio((int)N, p, zz, sp, st) : bwd_bf16((int)N, p, zz, sp, st);
    return bwd_f32((int)N, p, zz, sp, st);
}

int ssm_scan_bwd(const ssm_dims* dims, const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus, const float* dy,
                 const float* dlast_state, float* du, float* ddelta, float* dz, float* dA,
                 float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return ssm_scan_bwd_ex(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, dy,
                           dlast_state, nullptr, SSM_INPUT_DELTA_B, SSM_IO_F32, du, ddelta, dz, dA,
                           dB, dC, dD, ddelta_bias, dh0, workspace, workspace_bytes, stream);
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
            rc = scan_fwd_impl(&d1, nullptr, sb + o_u, sb + o_dl, dA + d0 * N, sb + o_B, sb + o_C,
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

int ssm_scan_fwd_noalloc_status(void* stream) {
    void* scratch = nullptr;
    const int rs = noalloc_scratch(&scratch);
    if (rs != SSM_OK) return rs;
    return read_status(scratch, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
