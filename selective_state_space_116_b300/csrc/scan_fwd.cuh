// Forward selective scan: state-split sequential kernel.
//
// The recurrence h_t = exp(Delta_t A) h_{t-1} + Bbar_t u_t is diagonal, so the
// N state entries of a channel are N independent scalar recurrences that
// only meet in the output sum y_t = sum_n C_{t,n} h_{t,n}.  This kernel
// therefore walks each channel's sequence in order, exactly once, with its
// state held in registers: S state entries per thread and G = N / S threads
// per channel.  Per element-state that is the minimum work of the method (one
// 2^x on the special-function unit, a multiply for Delta*A, a multiply for
// the input term, one FMA for the state and one for the output); no second
// pass and no scan of affine pairs is needed, and the B x D x L x N expanded
// state never leaves the register file.
//
// The G threads of a channel sit in different warps (the group index is
// warp-uniform), so every warp reads the same B/C row of shared memory
// (a broadcast) and the G partial output sums meet in shared memory, not
// through shuffles.
//
// A CTA owns CH = 128 / G channels of one batch row and a contiguous range of
// that row's tokens, walked in tiles of kTL tokens.  Per tile:
//   load      u (or x), delta, z rows and the B, C tile -> shared memory
//             (16-byte cp.async, double-buffered, zero-filled past the edges)
//   prologue  [CONV: u = silu(causal depthwise conv(x) + bias)]
//             Delta = softplus(delta + bias), Delta*u  -> fp32 pairs; B, C ->
//             fp32, grouped by thread group
//   recur     every thread advances its S states over the tile's tokens and
//             writes its partial output sums
//   epilogue  y = (sum of partials + D u) * silu(z) -> global, 16-byte stores
//
// Compile-time variants: ZOH, the exact zero-order-hold input term
// Bbar u = (exp(Delta A) - 1) / A * B u in place of Delta B u; CONV, the
// block's short convolution fused into the prologue, so that u never goes
// through memory; VEC, the 16-byte copy and store paths, for calls whose rows
// all start on 16-byte boundaries.  The gate and softplus are per-call flags.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace ssm {

struct ScanParams {
    const void* u;        // the scan input u; CONV: the convolution's input x
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;       // may be null
    const void* z;        // may be null
    const float* bias;    // may be null
    void* y;
    float* last_state;    // may be null
    int64_t batch, dim, L;
    // per-call options
    int gate;             // z is given: y *= silu(z)
    int softplus;         // Delta = softplus(delta + bias)
    const float* h0;      // (batch, dim, N) initial state, or null for zero
    // convolution prologue (CONV instances)
    const float* conv_w;      // (dim, conv_k) taps, oldest input first
    const float* conv_b;      // (dim), or null
    const void* conv_state;   // (batch, dim, conv_k - 1) inputs before token 0, or null
    void* u_out;              // (batch, dim, L): the convolution's output, or null
    int conv_k;               // 1 .. 4
    // schedule (see scan_fwd_kernel)
    int64_t groups_per_row;   // ceil(dim / channels per CTA)
    int64_t ngroups;          // batch * groups_per_row
    int64_t ntiles;           // ceil(L / tile)
    // workspace: a header of int32 words (kHdr*), one flag per group, one
    // carried state per group
    int* status;
    long wait_limit;          // spin iterations of a bounded wait (~256 ns each)
    int skip_handoff;         // test hook: no CTA publishes its hand-over
    unsigned* flags;
    float* carry;
    // chunked (L-parallel) schedule: chunks of tiles_per_chunk tiles; per
    // (group, chunk) unit the aggregate state / carry-in [CH][N] and the sum
    // of Delta per channel [CH]
    int64_t nchunks, tiles_per_chunk;
    float* agg;
    float* dsum;
};

// How one part of a channel group starts and ends.
struct PartIO {
    int init;            // 0: zero state, 1: handed over (flag + carry),
                         // 2: from h0 below, 3: from the caller's initial state
    const float* h0;     // [CH][N] initial state when init == 2
    float* hout;         // [CH][N] final state (chunk aggregate), or null
    float* dsum;         // [CH] sum of Delta over the part, or null
    bool handoff;        // a part ending inside its group hands the state on (flag + carry)
};

// The workspace header (int32 words): the status a bounded wait that gave up
// leaves (kStatusTimeout, the ABI's SSM_ERR_TIMEOUT), the ticket counter that
// orders the persistent CTAs, and, in -DSSM_DEBUG builds, the first failed
// bounds check (kStatusDevice, the ABI's SSM_ERR_DEVICE) and its site.
constexpr int kHdrStatus = 0, kHdrTicket = 1, kHdrDebug = 2, kHdrDebugSite = 3;
constexpr int kStatusTimeout = -9;
constexpr int kStatusDevice = -12;

// Bounds checks of the -DSSM_DEBUG build: a failed check records the site in
// the workspace header and skips the access (no trap, no abort); release
// builds compile them away.
#ifdef SSM_DEBUG
__device__ __forceinline__ bool debug_ok(bool ok, int* hdr, int site) {
    if (!ok && hdr) {
        if (atomicCAS(hdr + kHdrDebug, 0, kStatusDevice) == 0) atomicExch(hdr + kHdrDebugSite, site);
    }
    return ok;
}
#define SSM_INBOUNDS(cond, hdr, site) ::ssm::debug_ok((cond), (hdr), (site))
#else
#define SSM_INBOUNDS(cond, hdr, site) true
#endif

namespace seq {

// Threads per CTA.  The single-pass scan with the first-order input term and
// the state split over G = 2 lanes uses 2-warp CTAs of 32 channels: more,
// smaller CTAs share an SM, so one CTA's tile prologue overlaps another's
// recurrence.  Everything else (other splits, the exact-ZOH term, the
// chunked schedule) uses 4-warp CTAs: there the larger shared memory and
// register footprint would leave fewer 2-warp CTAs resident than warps lost.
constexpr int kSeqThreads = 128;
constexpr int scan_threads(int g, bool zoh) { return (g == 2 && !zoh) ? 64 : kSeqThreads; }
constexpr int kTL = 32;         // tokens per tile

// Shared-memory layout.  Row paddings of 16 bytes make every access pattern
// below free of bank conflicts (each quarter-warp touches 8 distinct 16-byte
// bank groups).
template <typename T, int N, int S, bool CONV, int NT_>
struct Shape {
    static constexpr int G = N / S;                    // thread groups per channel
    static constexpr int NT = NT_;                     // threads per CTA
    static constexpr int CH = NT / G;                  // channels per CTA
    static constexpr int ES = (int)sizeof(T);
    static constexpr int EPC = 16 / ES;                // elements per 16-byte chunk
    static constexpr int RAW_ROW = kTL * ES + 16;      // one channel's tokens, raw
    static constexpr int RAW_PLANE = CH * RAW_ROW;
    static constexpr int BC_RAW = kTL * N * ES;        // one raw B (or C) tile
    static constexpr int NPLANES = 3;                  // u (or x), delta, z
    static constexpr int RAW_BUF = NPLANES * RAW_PLANE + 2 * BC_RAW;
    static constexpr int W_ROW = kTL * 8 + 16;         // (Delta, Delta u) per token
    static constexpr int Y_ROW = kTL * 4 + 16;         // partial output per token
    static constexpr int OFF_W = 2 * RAW_BUF;
    static constexpr int OFF_BC = OFF_W + CH * W_ROW;
    static constexpr int OFF_Y = OFF_BC + kTL * N * 2 * 4;
    static constexpr int END_Y = OFF_Y + G * CH * Y_ROW;
    // CONV: the convolution's output u per token (fp32, for D u) and the last
    // three inputs of the previous tile per channel (two slots)
    static constexpr int U_ROW = kTL * 4 + 16;
    static constexpr int OFF_U = END_Y;
    static constexpr int OFF_HALO = OFF_U + CH * U_ROW;
    static constexpr int SMEM = CONV ? OFF_HALO + 2 * CH * 16 : END_Y;
    // (row, 8-token chunk) work items of the prologue / epilogue per thread
    static constexpr int CHUNKS = CH * kTL / 8;
    static constexpr int CHUNK_ITERS = CHUNKS / NT;
    static_assert(N % S == 0 && CH % 32 == 0, "bad state split");
    static_assert(CHUNKS % NT == 0 && kTL % 32 == 0, "bad tile");
    static_assert(RAW_BUF % 16 == 0 && OFF_BC % 16 == 0 && OFF_Y % 16 == 0 && OFF_U % 16 == 0,
                  "alignment");
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// The (row, chunk) item a thread handles in prologue / epilogue iteration `it`:
// a warp covers 8 rows x 4 consecutive 8-token chunks, lanes 0..7 on rows 0..7.
template <int CH, int NT>
__device__ __forceinline__ void chunk_of(int it, int& r, int& q) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = it * (NT / 32) + warp;
    constexpr int RB = CH / 8;
    r = (blk % RB) * 8 + (lane & 7);
    q = (blk / RB) * 4 + (lane >> 3);
}

// 8 consecutive elements of a raw shared-memory row -> fp32
template <typename T> __device__ __forceinline__ void unpack8(const unsigned char* p, float (&v)[8]);
template <> __device__ __forceinline__ void unpack8<float>(const unsigned char* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <> __device__ __forceinline__ void unpack8<__nv_bfloat16>(const unsigned char* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const unsigned w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 8 consecutive fp32 values -> global row (16-byte stores; dst 16-byte aligned)
template <typename T> __device__ __forceinline__ void store8(T* dst, const float (&v)[8]);
template <> __device__ __forceinline__ void store8<float>(float* dst, const float (&v)[8]) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[8]) {
    uint4 q;
    unsigned* w = reinterpret_cast<unsigned*>(&q);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);  // RNE
        w[i] = *reinterpret_cast<const unsigned*>(&p);
    }
    *reinterpret_cast<uint4*>(dst) = q;
}

// The first n of 8 values -> global, one element at a time (n >= 8: all).
template <typename T>
__device__ __forceinline__ void store_first(T* dst, const float (&v)[8], int n) {
#pragma unroll
    for (int e = 0; e < 8; e++)
        if (e < n) dst[e] = io<T>::from_f32(v[e]);
}

// silu on a pair.  bf16 I/O takes the one-instruction tanh form
// silu(z) = z/2 (1 + tanh(z/2)) (relative error ~2^-11, far below bf16's
// 2^-9 rounding); fp32 takes z / (1 + 2^(-z log2 e)).
template <typename T> __device__ __forceinline__ float2 silu2(float2 z);
template <> __device__ __forceinline__ float2 silu2<float>(float2 z) {
    const float2 e = __fmul2_rn(make_float2(-z.x, -z.y), make_float2(kLog2e, kLog2e));
    const float2 p = __fadd2_rn(make_float2(1.0f, 1.0f), make_float2(ex2(e.x), ex2(e.y)));
    return __fmul2_rn(z, make_float2(rcp(p.x), rcp(p.y)));
}
template <> __device__ __forceinline__ float2 silu2<__nv_bfloat16>(float2 z) {
    const float2 hz = __fmul2_rn(make_float2(0.5f, 0.5f), z);
    float tx, ty;
    asm("tanh.approx.f32 %0, %1;" : "=f"(tx) : "f"(hz.x));
    asm("tanh.approx.f32 %0, %1;" : "=f"(ty) : "f"(hz.y));
    return __ffma2_rn(hz, make_float2(tx, ty), hz);
}

// Copy tile [t0, t0 + kTL) of CH rows of a (rows, L) tensor into a raw plane.
// VEC: rows are 16-byte aligned and L is a multiple of EPC, so a 16-byte chunk
// is either wholly inside or wholly outside the tensor.
template <typename T, int CH, int NT, int RAW_ROW, bool VEC>
__device__ __forceinline__ void load_plane(unsigned char* plane, const T* g, int64_t row0,
                                           int rows, int64_t L, int64_t t0,
                                           int64_t nrows_total, int* hdr) {
    constexpr int EPC = 16 / (int)sizeof(T);
    constexpr int CPR = kTL / EPC;  // chunks per row
    static_assert((CH * CPR) % NT == 0, "plane chunks must split evenly");
#pragma unroll
    for (int k = 0; k < CH * CPR / NT; k++) {
        const int i = k * NT + threadIdx.x;
        const int r = i / CPR, c = i % CPR;
        const int64_t t = t0 + (int64_t)c * EPC;
        unsigned char* dst = plane + r * RAW_ROW + c * 16;
        if constexpr (VEC) {
            bool ok = r < rows && t < L;
            if (ok) ok = SSM_INBOUNDS(row0 + r < nrows_total && t + EPC <= L, hdr, 1);
            cp_async16(dst, ok ? static_cast<const void*>(g + (row0 + r) * L + t) : g, ok ? 16 : 0);
        } else {
            T* d = reinterpret_cast<T*>(dst);
#pragma unroll
            for (int e = 0; e < EPC; e++) {
                bool ok = r < rows && t + e < L;
                if (ok) ok = SSM_INBOUNDS(row0 + r < nrows_total, hdr, 1);
                d[e] = ok ? g[(row0 + r) * L + t + e] : io<T>::from_f32(0.0f);
            }
        }
    }
}

// Copy tokens [t0, t0 + kTL) of one batch row of B or C (contiguous kTL*N run).
template <typename T, int N, int NT, bool VEC>
__device__ __forceinline__ void load_bc(unsigned char* dst, const T* g, int64_t L, int64_t t0,
                                        int* hdr) {
    constexpr int EPC = 16 / (int)sizeof(T);
    constexpr int CHUNKS = kTL * N / EPC;
    const int64_t valid = (L - t0) * N;  // elements of this tile inside the tensor
#pragma unroll
    for (int rr = 0; rr < (CHUNKS + NT - 1) / NT; rr++) {
        const int i = threadIdx.x + rr * NT;
        if (CHUNKS % NT != 0 && i >= CHUNKS) break;
        const int64_t e0 = (int64_t)i * EPC;
        if constexpr (VEC) {
            bool ok = e0 < valid;
            if (ok) ok = SSM_INBOUNDS(e0 + EPC <= valid && t0 >= 0, hdr, 2);
            cp_async16(dst + i * 16, ok ? static_cast<const void*>(g + t0 * N + e0) : g, ok ? 16 : 0);
        } else {
            T* d = reinterpret_cast<T*>(dst + i * 16);
#pragma unroll
            for (int e = 0; e < EPC; e++)
                d[e] = (e0 + e < valid) ? g[t0 * N + e0 + e] : io<T>::from_f32(0.0f);
        }
    }
}

// bf16 pair in a 32-bit word -> two floats (low half first)
__device__ __forceinline__ float2 bf2_to_f2(unsigned w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// ---------------------------------------------------------------------------
// The input term of the state update, for a pair of states.
//
// First order (ZOH = false): Bbar u = Delta B u; xs is Delta u.
// Exact zero-order hold (ZOH = true): Bbar u = w B u with the weight
// w = (exp(Delta A) - 1) / A; xs is u, dt is Delta, ia = 1 / A (0 where
// A = 0), a = exp(Delta A) = 2^e with e = Delta A log2(e).
// w = (a - 1) ia = a ia - ia (one fused multiply-add), except for |e| < 1/8,
// where a - 1 would keep only the absolute accuracy of the 2^x unit
// (~2^-22, a relative error up to 2^-22 / |Delta A|) and w = Delta (1 +
// Delta A / 2 + (Delta A)^2 / 6 + (Delta A)^3 / 24) is used instead, in
// Horner form in e with the coefficients times Delta, formed once per token
// (truncation below 5e-7 relative; at A = 0 it is Delta, the limit of w).
constexpr float kZohSeries = 0.125f;
constexpr float kZ2 = 0.34657359027997264f;    // ln 2 / 2
constexpr float kZ3 = 0.08007550231970023f;    // (ln 2)^2 / 6
constexpr float kZ4 = 0.013876027166205394f;   // (ln 2)^3 / 24

template <bool ZOH>
__device__ __forceinline__ float2 input_term2(float2 a, float2 e, float dt, float xs, float2 Bv,
                                              float2 ia) {
    const float2 xb = __fmul2_rn(make_float2(xs, xs), Bv);
    if constexpr (!ZOH) {
        return xb;
    } else {
        float2 w = __ffma2_rn(a, ia, make_float2(-ia.x, -ia.y));
        const float d2 = dt * kZ2, d3 = dt * kZ3, d4 = dt * kZ4;
        float2 t = __ffma2_rn(e, make_float2(d4, d4), make_float2(d3, d3));
        t = __ffma2_rn(e, t, make_float2(d2, d2));
        const float2 ws = __ffma2_rn(e, t, make_float2(dt, dt));
        if (fabsf(e.x) < kZohSeries) w.x = ws.x;
        if (fabsf(e.y) < kZohSeries) w.y = ws.y;
        return __fmul2_rn(w, xb);
    }
}
template <bool ZOH>
__device__ __forceinline__ float input_term1(float a, float e, float dt, float xs, float Bv,
                                             float ia) {
    const float xb = xs * Bv;
    if constexpr (!ZOH) {
        return xb;
    } else {
        float w = fmaf(a, ia, -ia);
        if (fabsf(e) < kZohSeries) w = fmaf(e, fmaf(e, fmaf(e, dt * kZ4, dt * kZ3), dt * kZ2), dt);
        return w * xb;
    }
}

// NT consecutive tokens for one thread, software-pipelined: while the state
// update of token t runs, the 2^x of token t + 1 are issued two at a time
// between its FMAs, so that the special-function unit and the FMA pipe work
// side by side instead of in alternating bursts (the two pipes bound this
// loop together: per element-state one 2^x and four fp32 operations).  The
// B, C rows and (Delta, Delta u) of token t + 1 are loaded before token t's
// update.  Same operations per token as token_step, in the same order:
// bit-identical.
// wrow: (Delta, xs) pairs, two tokens per float4 (xs = Delta u, or u for
// ZOH); bcp: B (S floats) then C (S floats) of this thread's states, BCT
// floats per token; yrow: NT partial outputs (16-byte aligned).  ia: 1 / A
// per state (ZOH only).
// RAW: B and C are bf16 rows of the raw tile instead (bcp then points at this
// thread's B states, C follows RAW_C bytes on, BCT bytes per token; S = 4 or
// 8), unpacked exactly in registers.
template <int S, int BCT, int NT, bool ZOH, bool RAW = false, int RAW_C = 0>
__device__ __forceinline__ void scan_tokens(const float4* __restrict__ wrow, const void* __restrict__ bcp,
                                            float (&h)[S], const float (&A2)[S], const float (&ia)[S],
                                            float* __restrict__ yrow) {
    static_assert(S % 4 == 0 && NT % 4 == 0, "scan_tokens takes S and NT multiples of 4");
    static_assert(!RAW || S == 4 || S == 8, "raw B/C rows take 4 or 8 states");
    float a[S], ec[S], B_n[S], C_n[S];
    float dt_n, xs_n;
    float4 wq = wrow[0];
    auto load = [&](int t) {   // inputs of token t
        if (t % 2 == 0) {
            wq = wrow[t / 2];
            dt_n = wq.x;
            xs_n = wq.y;
        } else {
            dt_n = wq.z;
            xs_n = wq.w;
        }
        if constexpr (RAW) {
            const unsigned char* bc = static_cast<const unsigned char*>(bcp) + t * BCT;
            unsigned bw[S / 2], cw[S / 2];
            if constexpr (S == 8) {
                const uint4 b4 = *reinterpret_cast<const uint4*>(bc);
                const uint4 c4 = *reinterpret_cast<const uint4*>(bc + RAW_C);
                bw[0] = b4.x; bw[1] = b4.y; bw[2] = b4.z; bw[3] = b4.w;
                cw[0] = c4.x; cw[1] = c4.y; cw[2] = c4.z; cw[3] = c4.w;
            } else {
                const uint2 b2 = *reinterpret_cast<const uint2*>(bc);
                const uint2 c2 = *reinterpret_cast<const uint2*>(bc + RAW_C);
                bw[0] = b2.x; bw[1] = b2.y;
                cw[0] = c2.x; cw[1] = c2.y;
            }
#pragma unroll
            for (int n = 0; n < S; n += 2) {
                const float2 bf = bf2_to_f2(bw[n / 2]), cf = bf2_to_f2(cw[n / 2]);
                B_n[n] = bf.x; B_n[n + 1] = bf.y;
                C_n[n] = cf.x; C_n[n + 1] = cf.y;
            }
        } else {
            const float* bc = static_cast<const float*>(bcp) + t * BCT;
#pragma unroll
            for (int n = 0; n < S; n += 4) {
                const float4 b4 = *reinterpret_cast<const float4*>(bc + n);
                const float4 c4 = *reinterpret_cast<const float4*>(bc + S + n);
                B_n[n] = b4.x; B_n[n + 1] = b4.y; B_n[n + 2] = b4.z; B_n[n + 3] = b4.w;
                C_n[n] = c4.x; C_n[n + 1] = c4.y; C_n[n + 2] = c4.z; C_n[n + 3] = c4.w;
            }
        }
    };
    load(0);
    {
        const float2 dt2 = make_float2(dt_n, dt_n);
#pragma unroll
        for (int n = 0; n < S; n += 2) {
            const float2 e = __fmul2_rn(dt2, make_float2(A2[n], A2[n + 1]));
            a[n] = ex2(e.x);
            a[n + 1] = ex2(e.y);
            ec[n] = e.x;
            ec[n + 1] = e.y;
        }
    }
    float4 out;
#pragma unroll
    for (int t = 0; t < NT; t++) {
        float Bv[S], Cv[S];
#pragma unroll
        for (int n = 0; n < S; n++) { Bv[n] = B_n[n]; Cv[n] = C_n[n]; }
        const float dt = dt_n, xs = xs_n;
        if (t + 1 < NT) load(t + 1);
        const float2 dtn2 = make_float2(dt_n, dt_n);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int n = 0; n < S; n += 2) {
            const float2 bb = input_term2<ZOH>(make_float2(a[n], a[n + 1]), make_float2(ec[n], ec[n + 1]),
                                               dt, xs, make_float2(Bv[n], Bv[n + 1]),
                                               make_float2(ia[n], ia[n + 1]));
            const float2 hn = __ffma2_rn(make_float2(a[n], a[n + 1]), make_float2(h[n], h[n + 1]), bb);
            h[n] = hn.x;
            h[n + 1] = hn.y;
            acc = __ffma2_rn(make_float2(Cv[n], Cv[n + 1]), hn, acc);
            if (t + 1 < NT) {   // token t + 1's decays for these two states
                const float2 e = __fmul2_rn(dtn2, make_float2(A2[n], A2[n + 1]));
                a[n] = ex2(e.x);
                a[n + 1] = ex2(e.y);
                ec[n] = e.x;
                ec[n + 1] = e.y;
            }
        }
        const float yv = acc.x + acc.y;
        if (t % 4 == 0) out.x = yv;
        if (t % 4 == 1) out.y = yv;
        if (t % 4 == 2) out.z = yv;
        if (t % 4 == 3) {
            out.w = yv;
            *reinterpret_cast<float4*>(yrow + t - 3) = out;
        }
    }
}

// The aggregate pass's token loop (state only: no C, no output), pipelined
// like scan_tokens; returns the tile's sum of Delta, added pairwise in token
// order exactly as the unpipelined loop does.
template <int S, int BCT, int NT, bool ZOH>
__device__ __forceinline__ float scan_tokens_state(const float4* __restrict__ wrow,
                                                   const float* __restrict__ bcf, float (&h)[S],
                                                   const float (&A2)[S], const float (&ia)[S]) {
    static_assert(S % 4 == 0 && NT % 2 == 0, "scan_tokens_state takes S % 4 == 0, even NT");
    float a[S], ec[S], B_n[S];
    float dt_n, xs_n;
    float4 wq = wrow[0];
    float tsum = 0.0f;
    auto load = [&](int t) {
        if (t % 2 == 0) {
            wq = wrow[t / 2];
            dt_n = wq.x;
            xs_n = wq.y;
            tsum += wq.x + wq.z;
        } else {
            dt_n = wq.z;
            xs_n = wq.w;
        }
        const float* bc = bcf + t * BCT;
#pragma unroll
        for (int n = 0; n < S; n += 4) {
            const float4 b4 = *reinterpret_cast<const float4*>(bc + n);
            B_n[n] = b4.x; B_n[n + 1] = b4.y; B_n[n + 2] = b4.z; B_n[n + 3] = b4.w;
        }
    };
    load(0);
    {
        const float2 dt2 = make_float2(dt_n, dt_n);
#pragma unroll
        for (int n = 0; n < S; n += 2) {
            const float2 e = __fmul2_rn(dt2, make_float2(A2[n], A2[n + 1]));
            a[n] = ex2(e.x);
            a[n + 1] = ex2(e.y);
            ec[n] = e.x;
            ec[n + 1] = e.y;
        }
    }
#pragma unroll
    for (int t = 0; t < NT; t++) {
        float Bv[S];
#pragma unroll
        for (int n = 0; n < S; n++) Bv[n] = B_n[n];
        const float dt = dt_n, xs = xs_n;
        if (t + 1 < NT) load(t + 1);
        const float2 dtn2 = make_float2(dt_n, dt_n);
#pragma unroll
        for (int n = 0; n < S; n += 2) {
            const float2 bb = input_term2<ZOH>(make_float2(a[n], a[n + 1]), make_float2(ec[n], ec[n + 1]),
                                               dt, xs, make_float2(Bv[n], Bv[n + 1]),
                                               make_float2(ia[n], ia[n + 1]));
            const float2 hn = __ffma2_rn(make_float2(a[n], a[n + 1]), make_float2(h[n], h[n + 1]), bb);
            h[n] = hn.x;
            h[n + 1] = hn.y;
            if (t + 1 < NT) {
                const float2 e = __fmul2_rn(dtn2, make_float2(A2[n], A2[n + 1]));
                a[n] = ex2(e.x);
                a[n + 1] = ex2(e.y);
                ec[n] = e.x;
                ec[n + 1] = e.y;
            }
        }
    }
    return tsum;
}

// The aggregate pass's token loop run backwards from the end of a chunk (the
// chunk's tokens in reverse, NT at a time): the chunk's state from zero is
// sum_t (prod_(s>t) a_s) b_t, so with W the product of the decays of the
// tokens already passed, each token adds W b_t and multiplies W by its a_t.
// Returns the tile's sum of Delta.  Once every W is below 2^-40 the tokens
// further back change the chunk's state by less than 2^-40 of their own
// contributions (which the decays keep geometrically bounded), and the
// caller stops.
template <int S, int BCT, int NT, bool ZOH>
__device__ __forceinline__ float scan_tokens_tail(const float4* __restrict__ wrow,
                                                  const float* __restrict__ bcf, float (&acc)[S],
                                                  float (&W)[S], const float (&A2)[S],
                                                  const float (&ia)[S]) {
    static_assert(S % 2 == 0 && NT % 2 == 0, "scan_tokens_tail takes even S and NT");
    float tsum = 0.0f;
#pragma unroll
    for (int t = NT - 1; t >= 0; t--) {
        const float4 wq = wrow[t / 2];
        const float dt = t % 2 ? wq.z : wq.x, xs = t % 2 ? wq.w : wq.y;
        if (t % 2 == 0) tsum += wq.x + wq.z;
        const float* bc = bcf + t * BCT;
        const float2 dt2 = make_float2(dt, dt);
#pragma unroll
        for (int n = 0; n < S; n += 2) {
            const float2 e = __fmul2_rn(dt2, make_float2(A2[n], A2[n + 1]));
            const float2 a = make_float2(ex2(e.x), ex2(e.y));
            const float2 bb = input_term2<ZOH>(a, e, dt, xs, make_float2(bc[n], bc[n + 1]),
                                               make_float2(ia[n], ia[n + 1]));
            const float2 w2 = make_float2(W[n], W[n + 1]);
            const float2 s2 = __ffma2_rn(w2, bb, make_float2(acc[n], acc[n + 1]));
            const float2 wn = __fmul2_rn(w2, a);
            acc[n] = s2.x; acc[n + 1] = s2.y;
            W[n] = wn.x; W[n + 1] = wn.y;
        }
    }
    return tsum;
}
constexpr float kTailCut = 9.094947e-13f;   // 2^-40

// One token for one thread (S = 1 or 2): advance S states; with WITH_Y,
// return the partial C.h.
template <int S, bool ZOH, bool WITH_Y>
__device__ __forceinline__ float token_step(float dt, float xs, const float* __restrict__ bc,
                                            float (&h)[S], const float (&A2)[S],
                                            const float (&ia)[S]) {
    float Bv[S], Cv[S];
#pragma unroll
    for (int n = 0; n < S; n++) {
        Bv[n] = bc[n];
        Cv[n] = WITH_Y ? bc[S + n] : 0.0f;
    }
    if constexpr (S == 1) {
        const float e = dt * A2[0];
        const float a = ex2(e);
        h[0] = fmaf(a, h[0], input_term1<ZOH>(a, e, dt, xs, Bv[0], ia[0]));
        return WITH_Y ? Cv[0] * h[0] : 0.0f;
    } else {
        const float2 dt2 = make_float2(dt, dt);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int n = 0; n < S; n += 2) {
            const float2 e = __fmul2_rn(dt2, make_float2(A2[n], A2[n + 1]));
            const float2 a = make_float2(ex2(e.x), ex2(e.y));
            const float2 bb = input_term2<ZOH>(a, e, dt, xs, make_float2(Bv[n], Bv[n + 1]),
                                               make_float2(ia[n], ia[n + 1]));
            const float2 hn = __ffma2_rn(a, make_float2(h[n], h[n + 1]), bb);
            h[n] = hn.x;
            h[n + 1] = hn.y;
            if constexpr (WITH_Y) acc = __ffma2_rn(make_float2(Cv[n], Cv[n + 1]), hn, acc);
        }
        return acc.x + acc.y;
    }
}

// softplus_log2 on a pair, for the whole warp (every lane must call it).
// log2(1 + 2^x) comes from the special-function unit's log2 of 1 + 2^x,
// except below x = XS, where the series of log2_1p_small2 replaces it: with
// 2^x small, forming 1 + 2^x in fp32 and the log2 unit's absolute error
// (~2^-22) would leave a relative error of about 2^-22 / 2^x in Delta.
// XS = -5 keeps that below 1e-5 (fp32 I/O); XS = -10 below 3e-4, far inside
// the bf16 tolerance, and the series is then rarely needed.  It is evaluated
// only when some lane of the warp needs it (`series`, a warp vote taken by
// the caller), so typical step sizes never pay for it.  Returns Delta in
// natural units; for v > 20 it is v.
template <int XS>
__device__ __forceinline__ float2 softplus2_log2(float2 x, bool series) {
    constexpr float kX20 = 20.0f * kLog2e;
    const float2 e = make_float2(ex2(x.x), ex2(x.y));
    const float2 p = __fadd2_rn(make_float2(1.0f, 1.0f), e);
    float2 s = make_float2(x.x > kX20 ? x.x : lg2(p.x), x.y > kX20 ? x.y : lg2(p.y));
    if (series) {
        const float2 q = log2_1p_small2(e);
        if (x.x < (float)XS) s.x = q.x;
        if (x.y < (float)XS) s.y = q.y;
    }
    return __fmul2_rn(make_float2(kLn2, kLn2), s);
}

// Bounded wait for the carry of `group` (set by the CTA that scanned the
// group's earlier tokens): at most `limit` polls, 256 ns apart (the library
// passes 2^22, about a second).  Returns false if the wait gave up.
__device__ __forceinline__ bool wait_flag(const unsigned* flag, long limit) {
    for (long it = 0; it < limit; it++) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v) return true;
        __nanosleep(256);
    }
    return false;
}

// Tiles [tb, te) of channel group `grp`.  AGG: the aggregate pass of the
// chunked schedule (no output; the final state and the sum of Delta go to
// part.hout / part.dsum).
template <typename T, int N, int S, int NT, bool ZOH, bool CONV, bool VEC, bool GS = false,
          bool AGG = false, bool TAIL = false>
__device__ __forceinline__ void scan_part(const ScanParams& p, unsigned char* smem, int64_t grp,
                                          int64_t tb, int64_t te, int* s_ok, const PartIO& part) {
    using Sh = Shape<T, N, S, CONV, NT>;
    constexpr int G = Sh::G, CH = Sh::CH;
    constexpr int QLAST = kTL / 8 - 1;   // the last 8-token chunk of a tile
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    // bf16 B and C read by the recurrence straight from the raw tile (S = 4:
    // one 8-byte load each, no fp32 staging pass; the Mamba-130M layer shape
    // runs 168 -> 156 us.  At S = 8 the extra unpacking made the Mamba-2.8B
    // shape 5% slower, 428 -> 450 us, so S = 8 keeps the fp32 staging.)
    constexpr bool RAW_BC = BF && S == 4 && !AGG && VEC;

    const int64_t b = grp / p.groups_per_row;
    const int64_t d0 = (grp % p.groups_per_row) * CH;
    const int rows = (int)(p.dim - d0 < CH ? p.dim - d0 : CH);
    const int64_t row0 = b * p.dim + d0;   // first flat (b, d) row of the group
    const int64_t L = p.L;
    // GS: an instance for calls with both the gate and softplus, where both
    // are known at compile time (the common layer configuration)
    const bool gate = GS || p.gate != 0, softplus = GS || p.softplus != 0;

    const T* gu = static_cast<const T*>(p.u);
    const T* gdl = static_cast<const T*>(p.delta);
    const T* gz = static_cast<const T*>(p.z);
    const T* gB = static_cast<const T*>(p.B) + b * L * N;
    const T* gC = static_cast<const T*>(p.C) + b * L * N;
    T* gy = static_cast<T*>(p.y);

    // recurrence role: group g, channel ch; g is warp-uniform
    const int g = threadIdx.x / CH, ch = threadIdx.x % CH;
    const bool active = ch < rows;
    float A2[S], h[S], ia[S];
#pragma unroll
    for (int j = 0; j < S; j++) {   // exp(Delta A) = 2^(Delta A log2 e)
        const float av = active ? p.A[(d0 + ch) * N + g * S + j] : 0.0f;
        A2[j] = av * kLog2e;
        ia[j] = (ZOH && av != 0.0f) ? 1.0f / av : 0.0f;   // the ZOH weight's 1/A
    }

    // prologue / epilogue role: constants of the rows this thread touches
    float bias_r[Sh::CHUNK_ITERS], D_r[Sh::CHUNK_ITERS];
    float cw_r[CONV ? Sh::CHUNK_ITERS : 1][4], cb_r[CONV ? Sh::CHUNK_ITERS : 1];
#pragma unroll
    for (int it = 0; it < Sh::CHUNK_ITERS; it++) {
        int r, q;
        chunk_of<CH, Sh::NT>(it, r, q);
        const float bv = (p.bias && r < rows) ? p.bias[d0 + r] : 0.0f;
        bias_r[it] = softplus ? bv * kLog2e : bv;
        D_r[it] = (p.D && r < rows) ? p.D[d0 + r] : 0.0f;
        if constexpr (CONV) {   // taps aligned to the newest input (4 - K leading zeros)
            const int K = p.conv_k;
#pragma unroll
            for (int j = 0; j < 4; j++)
                cw_r[it][j] = (r < rows && j >= 4 - K) ? p.conv_w[(d0 + r) * K + j - (4 - K)] : 0.0f;
            cb_r[it] = (p.conv_b && r < rows) ? p.conv_b[d0 + r] : 0.0f;
        }
    }

    int* const hdr = p.status;             // workspace header (debug checks)
    const int64_t nrows = p.batch * p.dim;
    (void)hdr;
    (void)nrows;
    auto load_tile = [&](int64_t tile, int slot) {
        unsigned char* buf = smem + slot * Sh::RAW_BUF;
        const int64_t t0 = tile * kTL;
        load_plane<T, CH, Sh::NT, Sh::RAW_ROW, VEC>(buf, gu, row0, rows, L, t0, nrows, hdr);
        load_plane<T, CH, Sh::NT, Sh::RAW_ROW, VEC>(buf + Sh::RAW_PLANE, gdl, row0, rows, L, t0, nrows, hdr);
        if (gate && !AGG)
            load_plane<T, CH, Sh::NT, Sh::RAW_ROW, VEC>(buf + 2 * Sh::RAW_PLANE, gz, row0, rows, L, t0, nrows, hdr);
        unsigned char* bcraw = buf + Sh::NPLANES * Sh::RAW_PLANE;
        load_bc<T, N, Sh::NT, VEC>(bcraw, gB, L, t0, hdr);
        load_bc<T, N, Sh::NT, VEC>(bcraw + Sh::BC_RAW, gC, L, t0, hdr);
    };

    // the first tile's copies overlap the wait for the carry (TAIL: the
    // aggregate pass walks the part's tiles from its last one backwards)
    static_assert(!TAIL || (AGG && !CONV && S % 2 == 0), "the tail walk is an aggregate pass");
    load_tile(TAIL ? te - 1 : tb, 0);
    cp_async_commit();

    if constexpr (CONV) {   // the three inputs before the part's first token
        const int64_t t0 = tb * kTL;
        const int K = p.conv_k;
        const T* gs = static_cast<const T*>(p.conv_state);
        for (int r = threadIdx.x; r < CH; r += Sh::NT) {
            float hv[3] = {0.0f, 0.0f, 0.0f};
            if (r < rows) {
#pragma unroll
                for (int j = 0; j < 3; j++) {
                    const int64_t src = t0 - 3 + j;   // token index of halo entry j
                    if (src >= 0)
                        hv[j] = io<T>::to_f32(gu[(row0 + r) * L + src]);
                    else if (gs && src >= -(K - 1))
                        hv[j] = io<T>::to_f32(gs[(row0 + r) * (K - 1) + (K - 1) + src]);
                }
            }
            *reinterpret_cast<float4*>(smem + Sh::OFF_HALO + r * 16) = make_float4(hv[0], hv[1], hv[2], 0.0f);
        }
    }

    // initial state: zero, given, or the carry handed over by another CTA
    if (part.init == 0) {
#pragma unroll
        for (int j = 0; j < S; j++) h[j] = 0.0f;
    } else if (part.init == 2 || part.init == 3) {
        const float* src = (part.init == 2 ? part.h0 + ch * N : p.h0 + (row0 + ch) * N) + g * S;
        const bool ok = active && (part.init == 2 || SSM_INBOUNDS(row0 + ch < nrows, hdr, 3));
#pragma unroll
        for (int j = 0; j < S; j++) h[j] = ok ? __ldcg(src + j) : 0.0f;
    } else {
        if (threadIdx.x == 0) {
            const bool ok = wait_flag(p.flags + grp, p.wait_limit);
            if (!ok) atomicExch(p.status + kHdrStatus, kStatusTimeout);
            __threadfence();
            *s_ok = ok;
        }
        __syncthreads();
        const bool ok = *s_ok;
        const float* src = p.carry + (grp * CH + ch) * N + g * S;
#pragma unroll
        for (int j = 0; j < S; j++) h[j] = ok ? __ldcg(src + j) : __int_as_float(0x7fc00000);
    }

    float dsum = 0.0f, dcomp = 0.0f;   // sum of Delta over the part (compensated)
    float W[S];                        // TAIL: the decay products of the tokens passed
#pragma unroll
    for (int j = 0; j < S; j++) W[j] = 1.0f;
    for (int64_t step = 0; step < te - tb; step++) {
        const int64_t tile = TAIL ? te - 1 - step : tb + step;
        const int slot = (int)(step & 1);
        if (step + 1 < te - tb) load_tile(TAIL ? tile - 1 : tile + 1, slot ^ 1);
        cp_async_commit();
        cp_async_wait_1();
        __syncthreads();

        const unsigned char* buf = smem + slot * Sh::RAW_BUF;
        const int64_t t0 = tile * kTL;
        const int tvalid = (int)(L - t0 < kTL ? L - t0 : kTL);

        // ---- prologue: [u from the convolution], (Delta, Delta u) pairs, B/C to fp32 ----
#pragma unroll
        for (int it = 0; it < Sh::CHUNK_ITERS; it++) {
            int r, q;
            chunk_of<CH, Sh::NT>(it, r, q);
            float uv[8], dv[8];
            if constexpr (CONV) {
                // inputs t-3 .. t+7 for the chunk's tokens t = 8q .. 8q+7: the
                // previous chunk's last three, or the previous tile's (halo)
                float xx[11], xc[8];
                unpack8<T>(buf + r * Sh::RAW_ROW + q * 8 * Sh::ES, xc);
                if (q == 0) {
                    const float4 hv = *reinterpret_cast<const float4*>(smem + Sh::OFF_HALO +
                                                                       slot * CH * 16 + r * 16);
                    xx[0] = hv.x; xx[1] = hv.y; xx[2] = hv.z;
                } else {
                    float xp[8];
                    unpack8<T>(buf + r * Sh::RAW_ROW + (q - 1) * 8 * Sh::ES, xp);
                    xx[0] = xp[5]; xx[1] = xp[6]; xx[2] = xp[7];
                }
#pragma unroll
                for (int e = 0; e < 8; e++) xx[3 + e] = xc[e];
                if (q == QLAST)   // the next tile's first chunk reads these
                    *reinterpret_cast<float4*>(smem + Sh::OFF_HALO + (slot ^ 1) * CH * 16 + r * 16) =
                        make_float4(xc[5], xc[6], xc[7], 0.0f);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float2 s2 = make_float2(cb_r[it], cb_r[it]);
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        s2 = __ffma2_rn(make_float2(cw_r[it][j], cw_r[it][j]),
                                        make_float2(xx[e + j], xx[e + 1 + j]), s2);
                    const float2 sv = silu2<T>(s2);
                    uv[e] = sv.x;
                    uv[e + 1] = sv.y;
                }
                float4* us = reinterpret_cast<float4*>(smem + Sh::OFF_U + r * Sh::U_ROW + q * 32);
                us[0] = make_float4(uv[0], uv[1], uv[2], uv[3]);
                us[1] = make_float4(uv[4], uv[5], uv[6], uv[7]);
                if (!AGG && p.u_out && r < rows && q * 8 < tvalid &&
                    SSM_INBOUNDS(row0 + r < nrows && t0 + q * 8 < L, hdr, 5)) {
                    T* dst = static_cast<T*>(p.u_out) + (row0 + r) * L + t0 + q * 8;
                    if (VEC && q * 8 + 8 <= tvalid) store8<T>(dst, uv);
                    else store_first<T>(dst, uv, tvalid - q * 8);
                }
            } else {
                unpack8<T>(buf + r * Sh::RAW_ROW + q * 8 * Sh::ES, uv);
            }
            unpack8<T>(buf + Sh::RAW_PLANE + r * Sh::RAW_ROW + q * 8 * Sh::ES, dv);
            // pairs of tokens in packed fp32 arithmetic (same roundings as
            // the scalar form: fused multiply-add, add, multiply)
            float2 dt[4];
            const float2 bias2 = make_float2(bias_r[it], bias_r[it]);
            if (softplus) {
                constexpr int XS = BF ? -10 : -5;
                float2 xv[4];
                float xmin = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    xv[e / 2] = __ffma2_rn(make_float2(dv[e], dv[e + 1]), make_float2(kLog2e, kLog2e), bias2);
                    xmin = fminf(xmin, fminf(xv[e / 2].x, xv[e / 2].y));
                }
                const bool series = __any_sync(0xffffffffu, xmin < (float)XS);
#pragma unroll
                for (int e = 0; e < 8; e += 2) dt[e / 2] = softplus2_log2<XS>(xv[e / 2], series);
            } else {
#pragma unroll
                for (int e = 0; e < 8; e += 2) dt[e / 2] = __fadd2_rn(make_float2(dv[e], dv[e + 1]), bias2);
            }
            if (tvalid < kTL) {   // tokens past the end leave the state untouched
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    if (q * 8 + e >= tvalid) dt[e / 2].x = 0.0f;
                    if (q * 8 + e + 1 >= tvalid) dt[e / 2].y = 0.0f;
                }
            }
            float4* w = reinterpret_cast<float4*>(smem + Sh::OFF_W + r * Sh::W_ROW + q * 64);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                // the second entry of each token: Delta u, or u itself for the
                // exact zero-order hold (which weighs it by (2^e - 1) / A)
                const float2 xs = ZOH ? make_float2(uv[e], uv[e + 1])
                                      : __fmul2_rn(dt[e / 2], make_float2(uv[e], uv[e + 1]));
                w[e / 2] = make_float4(dt[e / 2].x, xs.x, dt[e / 2].y, xs.y);
            }
        }
        if constexpr (!RAW_BC) {
            const unsigned char* bcraw = buf + Sh::NPLANES * Sh::RAW_PLANE;
            float* bcf = reinterpret_cast<float*>(smem + Sh::OFF_BC);
            if constexpr (N % 4 == 0 && S % 4 == 0) {
                // 4 consecutive n of one token lie in one thread group: one
                // 8- or 16-byte load and one 16-byte store per group (a loop
                // of fixed trip count, so that the indices fold)
                constexpr int Q = 2 * kTL * N / 4;              // 4-element groups of B and C
#pragma unroll
                for (int r = 0; r < (Q + Sh::NT - 1) / Sh::NT; r++) {
                    const int i = threadIdx.x + r * Sh::NT;
                    if (Q % Sh::NT == 0 || i < Q) {
                        const int which = i / (kTL * N / 4);           // 0: B, 1: C
                        const int e0 = (i % (kTL * N / 4)) * 4;
                        const int t = e0 / N, n = e0 % N;
                        const unsigned char* src = bcraw + which * Sh::BC_RAW + e0 * Sh::ES;
                        float4 v;
                        if constexpr (sizeof(T) == 2) {
                            const uint2 w2 = *reinterpret_cast<const uint2*>(src);
                            const float2 lo = bf2_to_f2(w2.x), hi = bf2_to_f2(w2.y);
                            v = make_float4(lo.x, lo.y, hi.x, hi.y);
                        } else {
                            v = *reinterpret_cast<const float4*>(src);
                        }
                        *reinterpret_cast<float4*>(bcf + (t * G + n / S) * 2 * S + which * S + n % S) = v;
                    }
                }
            } else {
                const T* rb = reinterpret_cast<const T*>(bcraw);
                const T* rc = reinterpret_cast<const T*>(bcraw + Sh::BC_RAW);
                for (int i = threadIdx.x; i < kTL * N; i += Sh::NT) {
                    const int t = i / N, n = i % N;
                    float* o = bcf + (t * G + n / S) * 2 * S + n % S;
                    o[0] = io<T>::to_f32(rb[i]);
                    o[S] = io<T>::to_f32(rc[i]);
                }
            }
        }
        __syncthreads();

        // ---- recurrence over the tile ----
        {
            const float4* wrow = reinterpret_cast<const float4*>(smem + Sh::OFF_W + ch * Sh::W_ROW);
            const float* bcf = reinterpret_cast<const float*>(smem + Sh::OFF_BC) + g * 2 * S;
            float* yrow = reinterpret_cast<float*>(smem + Sh::OFF_Y + (g * CH + ch) * Sh::Y_ROW);
            if constexpr (TAIL) {
                const float tsum = scan_tokens_tail<S, G * 2 * S, kTL, ZOH>(wrow, bcf, h, W, A2, ia);
                const float yk = tsum - dcomp, tk = dsum + yk;
                dcomp = (tk - dsum) - yk;
                dsum = tk;
            } else if constexpr (AGG && S % 4 == 0) {
                const float tsum = scan_tokens_state<S, G * 2 * S, kTL, ZOH>(wrow, bcf, h, A2, ia);
                const float yk = tsum - dcomp, tk = dsum + yk;
                dcomp = (tk - dsum) - yk;
                dsum = tk;
            } else if constexpr (AGG) {
                float tsum = 0.0f;
#pragma unroll 2
                for (int t = 0; t < kTL; t += 2) {
                    const float4 w = wrow[t / 2];
                    token_step<S, ZOH, false>(w.x, w.y, bcf + (t + 0) * G * 2 * S, h, A2, ia);
                    token_step<S, ZOH, false>(w.z, w.w, bcf + (t + 1) * G * 2 * S, h, A2, ia);
                    tsum += w.x + w.z;
                }
                const float yk = tsum - dcomp, tk = dsum + yk;
                dcomp = (tk - dsum) - yk;
                dsum = tk;
            } else if constexpr (RAW_BC) {
                const unsigned char* braw = buf + Sh::NPLANES * Sh::RAW_PLANE + g * S * 2;
                scan_tokens<S, N * 2, kTL, ZOH, true, Sh::BC_RAW>(wrow, braw, h, A2, ia, yrow);
            } else if constexpr (S % 4 == 0) {
                scan_tokens<S, G * 2 * S, kTL, ZOH>(wrow, bcf, h, A2, ia, yrow);
            } else {
#pragma unroll 2
                for (int t = 0; t < kTL; t += 4) {
                    const float4 w01 = wrow[t / 2];
                    const float4 w23 = wrow[t / 2 + 1];
                    float4 out;
                    out.x = token_step<S, ZOH, true>(w01.x, w01.y, bcf + (t + 0) * G * 2 * S, h, A2, ia);
                    out.y = token_step<S, ZOH, true>(w01.z, w01.w, bcf + (t + 1) * G * 2 * S, h, A2, ia);
                    out.z = token_step<S, ZOH, true>(w23.x, w23.y, bcf + (t + 2) * G * 2 * S, h, A2, ia);
                    out.w = token_step<S, ZOH, true>(w23.z, w23.w, bcf + (t + 3) * G * 2 * S, h, A2, ia);
                    *reinterpret_cast<float4*>(yrow + t) = out;
                }
            }
        }
        __syncthreads();

        // ---- epilogue: y = (sum of partials + D u) * silu(z) ----
#pragma unroll
        for (int it = 0; it < (AGG ? 0 : Sh::CHUNK_ITERS); it++) {
            int r, q;
            chunk_of<CH, Sh::NT>(it, r, q);
            // pairs of tokens in packed fp32 arithmetic, the partial sums
            // added in group order
            float2 y2[4];
#pragma unroll
            for (int gg = 0; gg < G; gg++) {
                const float4* yp = reinterpret_cast<const float4*>(
                    smem + Sh::OFF_Y + (gg * CH + r) * Sh::Y_ROW + q * 32);
                const float4 a = yp[0], c = yp[1];
                const float2 v[4] = {make_float2(a.x, a.y), make_float2(a.z, a.w),
                                     make_float2(c.x, c.y), make_float2(c.z, c.w)};
#pragma unroll
                for (int e = 0; e < 4; e++) y2[e] = gg == 0 ? v[e] : __fadd2_rn(y2[e], v[e]);
            }
            float uv[8];
            if constexpr (CONV) {
                const float4* us = reinterpret_cast<const float4*>(smem + Sh::OFF_U + r * Sh::U_ROW + q * 32);
                const float4 u0 = us[0], u1 = us[1];
                uv[0] = u0.x; uv[1] = u0.y; uv[2] = u0.z; uv[3] = u0.w;
                uv[4] = u1.x; uv[5] = u1.y; uv[6] = u1.z; uv[7] = u1.w;
            } else {
                unpack8<T>(buf + r * Sh::RAW_ROW + q * 8 * Sh::ES, uv);
            }
            const float2 D2 = make_float2(D_r[it], D_r[it]);
#pragma unroll
            for (int e = 0; e < 4; e++)
                y2[e] = __ffma2_rn(D2, make_float2(uv[2 * e], uv[2 * e + 1]), y2[e]);
            if (gate) {
                float zv[8];
                unpack8<T>(buf + 2 * Sh::RAW_PLANE + r * Sh::RAW_ROW + q * 8 * Sh::ES, zv);
#pragma unroll
                for (int e = 0; e < 4; e++)
                    y2[e] = __fmul2_rn(y2[e], silu2<T>(make_float2(zv[2 * e], zv[2 * e + 1])));
            }
            float ys[8];
#pragma unroll
            for (int e = 0; e < 4; e++) { ys[2 * e] = y2[e].x; ys[2 * e + 1] = y2[e].y; }
            if (r < rows && q * 8 < tvalid &&
                SSM_INBOUNDS(row0 + r < nrows && t0 + q * 8 < L, hdr, 4)) {
                T* dst = gy + (row0 + r) * L + t0 + q * 8;
                if (VEC && q * 8 + 8 <= tvalid) store8<T>(dst, ys);
                else store_first<T>(dst, ys, tvalid - q * 8);
            }
        }
        __syncthreads();
        if constexpr (TAIL) {   // stop once every decay product of the CTA is below the cut
            float wmax = 0.0f;
#pragma unroll
            for (int j = 0; j < S; j++) wmax = fmaxf(wmax, W[j]);
            const bool live = active && !(wmax < kTailCut);   // NaN keeps walking
            if (!__syncthreads_or(live)) {
                cp_async_commit();
                cp_async_wait_0();   // the copy of the next tile is still in flight
                break;
            }
        }
    }

    if (part.hout) {   // chunk aggregate: final state from zero and the Delta sum
        float* dst = part.hout + ch * N + g * S;
#pragma unroll
        for (int j = 0; j < S; j++) dst[j] = h[j];
        if (g == 0) part.dsum[ch] = dsum;
    } else if (te == p.ntiles) {
        if (active && p.last_state && SSM_INBOUNDS(row0 + ch < nrows, hdr, 6)) {
            float* dst = p.last_state + (row0 + ch) * N + g * S;
#pragma unroll
            for (int j = 0; j < S; j++) dst[j] = h[j];
        }
    } else if (part.handoff) {
        // hand the state over to the CTA that scans the rest of this group
        float* dst = p.carry + (grp * CH + ch) * N + g * S;
#pragma unroll
        for (int j = 0; j < S; j++) __stcg(dst + j, h[j]);
        __threadfence();
        __syncthreads();
        // (the test hook withholds the flag: the successor's bounded wait
        // then runs out and reports SSM_ERR_TIMEOUT)
        if (threadIdx.x == 0 && !p.skip_handoff)
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + grp), "r"(1u) : "memory");
    }
}

// Persistent, balanced schedule.  The work is ngroups x ntiles tiles (a
// group is CH channels of one batch row); CTA c takes the contiguous range
// [c W / P, (c+1) W / P) of the group-major order, so every CTA gets the same
// number of tiles to within one.  A range that starts inside a group
// continues the state of the CTA before it: each CTA scans its last group's
// head first (publishing that state), then its whole groups, and the
// continuation of its first group last, so the state it needs has long been
// published when it gets there.  With P <= ngroups no group is split twice.
template <typename T, int N, int S, int NT, bool ZOH, bool CONV, bool VEC, bool GS = false>
__global__ void __launch_bounds__(NT, 256 / NT) scan_fwd_kernel(ScanParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_ok;
    using Sh = Shape<T, N, S, CONV, NT>;
    if (p.nchunks > 0) {   // pass 3 of the chunked schedule (see scan_chunk_agg_kernel)
        const int64_t units = p.ngroups * p.nchunks;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
            const int64_t grp = u / p.nchunks, ck = u % p.nchunks;
            const int64_t tb = ck * p.tiles_per_chunk;
            const int64_t te = tb + p.tiles_per_chunk < p.ntiles ? tb + p.tiles_per_chunk : p.ntiles;
            // every chunk starts from its carry-in (the first: the initial state)
            const PartIO io{2, p.agg + u * Sh::CH * N, nullptr, nullptr, false};
            scan_part<T, N, S, NT, ZOH, CONV, VEC, GS>(p, smem, grp, tb, te, &s_ok, io);
            __syncthreads();
        }
        return;
    }
    // The CTA's place in the schedule is a ticket taken on arrival, not its
    // block index: the CTA whose range precedes this one took its ticket
    // earlier, so it is running, and it publishes the state this CTA may wait
    // for without waiting itself (its first part starts at a group's first
    // tile).  Block indices carry no such guarantee of dispatch order.
    __shared__ int64_t s_ticket;
    if (threadIdx.x == 0)
        s_ticket = p.status ? (int64_t)atomicAdd(reinterpret_cast<unsigned*>(p.status + kHdrTicket), 1u)
                            : (int64_t)blockIdx.x;
    __syncthreads();
    const int64_t c = s_ticket;
    const int64_t W = p.ngroups * p.ntiles;
    const int64_t s = W * c / gridDim.x;
    const int64_t e = W * (c + 1) / gridDim.x;
    if (s >= e) {   // empty sequence (or more CTAs than tiles): only last_state remains
        if (p.ntiles == 0 && p.last_state) {
            for (int64_t grp = c; grp < p.ngroups; grp += gridDim.x) {
                const int64_t b = grp / p.groups_per_row;
                const int64_t d0 = (grp % p.groups_per_row) * Sh::CH;
                const int rows = (int)(p.dim - d0 < Sh::CH ? p.dim - d0 : Sh::CH);
                const int64_t base = (b * p.dim + d0) * N;
                for (int i = threadIdx.x; i < rows * N; i += Sh::NT)
                    p.last_state[base + i] = p.h0 ? p.h0[base + i] : 0.0f;
            }
        }
        return;
    }
    const int64_t g_first = s / p.ntiles, g_last = (e - 1) / p.ntiles;
    for (int64_t grp = g_last; grp >= g_first; grp--) {
        const int64_t lo = grp * p.ntiles;
        const int64_t tb = (s > lo ? s : lo) - lo;
        const int64_t te = (e < lo + p.ntiles ? e : lo + p.ntiles) - lo;
        const int init = tb > 0 ? 1 : (p.h0 ? 3 : 0);
        const PartIO io{init, nullptr, nullptr, nullptr, true};
        scan_part<T, N, S, NT, ZOH, CONV, VEC, GS>(p, smem, grp, tb, te, &s_ok, io);
    }
}

// Chunked (L-parallel) schedule for problems with too few channel groups to
// fill the GPU (a long sequence over few channels).  The token range of every
// group is cut into chunks, and the affine maps h -> a h + b of the steps
// compose associatively ((a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2)), so:
//   pass 1  every (group, chunk) unit finds its chunk's map: b, the state the
//           chunk reaches from zero, and a = exp(A sum Delta)
//           (scan_chunk_agg_kernel).  Without the convolution it walks the
//           chunk from its end (scan_tokens_tail) and stops once the decay
//           products are negligible, so for decaying states it reads only the
//           chunk's last tokens; with it, it scans the chunk forward.
//   pass 2  per (channel, state) an exclusive scan of the chunks' maps under
//           composition (lanes, warps, tiles of chunks) gives each chunk's
//           carry-in from the initial state (scan_chunk_carry_kernel)
//   pass 3  every unit scans its chunk again from its carry-in and writes y
//           and, for the last chunk, last_state (scan_fwd_kernel with
//           p.nchunks > 0).
// Passes 1 and 3 are independent over units: grid-stride loops of
// persistent CTAs.  The price is pass 1's reading of the chunks' tails.
template <typename T, int N, int S, int NT, bool ZOH, bool CONV, bool VEC>
__global__ void __launch_bounds__(NT, 256 / NT) scan_chunk_agg_kernel(ScanParams p) {
    using Sh = Shape<T, N, S, CONV, NT>;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_ok;
    const int64_t units = p.ngroups * p.nchunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t grp = u / p.nchunks, ck = u % p.nchunks;
        const int64_t tb = ck * p.tiles_per_chunk;
        const int64_t te = tb + p.tiles_per_chunk < p.ntiles ? tb + p.tiles_per_chunk : p.ntiles;
        const PartIO io{0, nullptr, p.agg + u * Sh::CH * N, p.dsum + u * Sh::CH, false};
        // without the convolution (whose inputs reach back across tiles) the
        // chunk is walked from its end and the walk stops when the decays
        // have made the earlier tokens negligible
        constexpr bool kTail = !CONV && S % 2 == 0;
        scan_part<T, N, S, NT, ZOH, CONV, VEC, false, true, kTail>(p, smem, grp, tb, te, &s_ok, io);
        __syncthreads();
    }
}

// Pass 2: the carry-in of every chunk, as an exclusive scan of the chunks'
// affine maps under composition.  Chunk k maps the state entering it to the
// state leaving it: h -> a_k h + b_k, with a_k = exp(A sum of Delta over the
// chunk) and b_k its state from zero (pass 1).  Composition
// (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2) is associative ("Mamba remembers
// by forgetting, read closely", interactiveml.org: the compose operator and
// its associativity; "Mamba", sghael.github.io, "Training without stepping
// token by token": updates combined in pairs, then pairs of pairs), so one
// CTA per (group, channel, state) sequence scans it in tiles of kCarryThreads
// chunks: lanes combine with __shfl_up_sync (log2 32 rounds), warps through
// shared memory, and each tile starts from the previous tiles' total.  The
// carry-in of chunk k is the composition of chunks 0 .. k-1 applied to the
// initial state; it overwrites the chunk's aggregate.
constexpr int kCarryThreads = 256;

struct Affine {
    float a, b;
};
// (later) o (earlier)
__device__ __forceinline__ Affine compose(Affine later, Affine earlier) {
    return Affine{later.a * earlier.a, fmaf(later.a, earlier.b, later.b)};
}

template <int N, int CH>
__global__ void __launch_bounds__(kCarryThreads) scan_chunk_carry_kernel(ScanParams p) {
    constexpr int kWarps = kCarryThreads / 32;
    __shared__ Affine s_warp[kWarps];
    const int64_t seq = blockIdx.x;                   // (group, channel, state)
    const int64_t grp = seq / (CH * N);
    const int rem = (int)(seq % (CH * N)), ch = rem / N, n = rem % N;
    const int64_t b = grp / p.groups_per_row;
    const int64_t d = (grp % p.groups_per_row) * CH + ch;
    const bool in = d < p.dim;
    const float A2 = in ? p.A[d * N + n] * kLog2e : 0.0f;
    const float h0 = (in && p.h0) ? p.h0[(b * p.dim + d) * N + n] : 0.0f;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    Affine carry{1.0f, 0.0f};                         // the chunks of earlier tiles
    for (int64_t base = 0; base < p.nchunks; base += kCarryThreads) {
        const int64_t ck = base + threadIdx.x;
        const bool live = ck < p.nchunks;
        const int64_t u = grp * p.nchunks + ck;
        float* st = p.agg + (u * CH + ch) * N + n;
        // this chunk's map (the identity past the last chunk)
        Affine x{1.0f, 0.0f};
        if (live) x = Affine{ex2(A2 * p.dsum[u * CH + ch]), *st};
        // inclusive scan over the warp's lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float pa = __shfl_up_sync(0xffffffffu, x.a, off);
            const float pb = __shfl_up_sync(0xffffffffu, x.b, off);
            if (lane >= off) x = compose(x, Affine{pa, pb});
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        // the warps before this one, then the earlier tiles
        Affine before = carry;
        for (int w = 0; w < warp; w++) before = compose(s_warp[w], before);
        // exclusive: the lane before's inclusive map, or the warp's prefix
        const float ea = __shfl_up_sync(0xffffffffu, x.a, 1);
        const float eb = __shfl_up_sync(0xffffffffu, x.b, 1);
        const Affine excl = lane == 0 ? before : compose(Affine{ea, eb}, before);
        if (live) *st = fmaf(excl.a, h0, excl.b);     // the state entering chunk ck
        Affine total = carry;
        for (int w = 0; w < kWarps; w++) total = compose(s_warp[w], total);
        carry = total;
        __syncthreads();                              // s_warp is reused by the next tile
    }
}

}  // namespace seq
}  // namespace ssm
