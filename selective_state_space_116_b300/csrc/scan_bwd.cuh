// Backward selective scan (gradients for training), with recomputation.
//
// The forward pass keeps no state for the backward pass; the backward pass
// recomputes the forward states on chip instead of reading an expanded state
// from memory ("State Spaces, Selectively - Mamba", papermap, "The
// hardware-aware scan").  Per channel and token t (Delta_t after bias and
// softplus, a_tn = exp(Delta_t A_n), x = u):
//
//   forward   h_tn = a_tn h_(t-1)n + Delta_t x_t B_tn,   s_t = sum_n C_tn h_tn
//             y_t = (s_t + D x_t) silu(z_t)
//   adjoint   ds_t = dy_t silu(z_t);  g_tn = ds_t C_tn + a_(t+1)n g_(t+1)n
//             (g = dLoss/dh_t, started from dLoss/dlast_state)
//   gradients dx_t = ds_t D + Delta_t q_t,          q_t = sum_n g_tn B_tn
//             dDelta_t = r_t + x_t q_t,             r_t = sum_n A_n g_tn a_tn h_(t-1)n
//             dA_n = sum_t Delta_t g_tn a_tn h_(t-1)n
//             dB_tn = sum_channels g_tn Delta_t x_t, dC_tn = sum_channels ds_t h_tn
//             dz_t = dy_t (s_t + D x_t) silu'(z_t),  dD = sum_t ds_t x_t
//
// With the exact zero-order hold (ZOH) the input term is w_tn B_tn x_t with
// w = (exp(Delta A) - 1) / A per state ("Mamba remembers by forgetting, read
// closely", interactiveml.org, the discretisation and the selective_scan
// recurrence): dw/dDelta = a, dw/dA = (Delta a - w) / A, so
//             dx_t = ds_t D + sum_n g_tn w_tn B_tn
//             dDelta_t = r_t + x_t v_t,             v_t = sum_n g_tn a_tn B_tn
//             dA_n = sum_t g_tn (Delta_t a_tn h_(t-1)n + dw/dA_tn B_tn x_t)
//             dB_tn = sum_channels g_tn w_tn x_t
//
// Work split.  A thread holds S = min(N, 4) states of K channels (the same
// batch row); the G = N / S adjacent lanes of a "slot" hold the whole state of
// those K channels.  A CTA of one warp covers SLOTS = 32 / G slots, i.e.
// CH = SLOTS K channels, through the whole sequence (or its chunk of it, see
// below) in 8-token tiles, from the initial state h0 (zero if none):
//
//   pass 1  the forward recurrence, writing the state at the start of every
//           8-token tile to the workspace (batch x dim x ceil(L/8) x N fp32);
//           it stages 32 tokens at a time in the same shared memory;
//   pass 2  the tiles in reverse: the tile's 9 states (the one before it and
//           its 8) are recomputed into registers from the checkpoint, then
//           the adjoint runs backwards through them.
//
// The sums of a token run in three places.  Over a channel's states (s, q,
// r): within the thread, then over the G lanes through per-lane partials in
// shared memory.  Over channels (dB, dC): within the thread over its K
// channels, then per tile through shared memory over the CTA's slots, then
// one 16-byte atomic add per 4 states into the batch row.  Over tokens (dA):
// in registers for the whole sequence.  Everything per element (softplus,
// the gate and its derivative, the input and output of every (channel,
// token)) is done once per element by the thread that stages it: each thread
// stages EPT consecutive tokens of one channel, copied in by cp.async while
// the tile before computes, and writes their gradients with vector stores.
//
// Long sequences over few channels (too few CTAs to fill the GPU) are cut
// into chunks that run side by side (grid z).  Both recurrences are affine
// in their carried vector ("Mamba remembers by forgetting, read closely",
// interactiveml.org: the compose operator and its associativity; "Mamba",
// sghael.github.io, "Training without stepping token by token"): per chunk
// the state at its end from a zero start is F plus PF times the state at
// its start, and the adjoint it hands to the state before it is Q plus PQ
// times the adjoint it receives, PF = PQ = the product of its decays.
// scan_bwd_chunk_agg_kernel finds F and Q by walks that stop where the
// decay product passed falls below 2^-40 (forward: back from the chunk's
// end; adjoint: on from its start), scan_bwd_chunk_carry_kernel composes
// them across the chunks into each chunk's starting state and incoming
// adjoint, and scan_bwd_kernel then runs every chunk from those.
#pragma once

#include "common.cuh"

namespace ssm {
namespace bwd {

constexpr int kThreads = 32;    // threads per CTA (one warp: the finest split of the channels)
constexpr int kTT = 8;          // tokens per tile
constexpr int kChunkAlign = 32; // chunk boundaries of the chunked backward: multiples of pass 1's staging

// Channels per thread: two at N = 16 (their dB, dC products summed in
// registers before the shared-memory reduction) when the grid of such CTAs
// holds at least kWideGrid of them, or when the sequence is long enough to
// be cut into chunks (8192 tokens) that make up the CTAs; one otherwise,
// and for smaller states, so that a small problem gets twice the CTAs
// (which also need less shared memory: 12 fit on an SM instead of 9; the
// Mamba-130M layer shape 1.06 -> 0.93 ms; at the DNA-like shape, chunked,
// two channels per thread stay faster, 32.7 against 35.9 ms).  Channels per
// CTA follow (32 / (N / min(N, 4)) slots, times the channels per thread).
constexpr int64_t kWideGrid = 1024;
constexpr int64_t kChunkedSeq = 8192;
constexpr int channels_per_thread(int n, int64_t batch, int64_t dim, int64_t L) {
    return n == 16 && (batch * ((dim + 15) / 16) >= kWideGrid || L >= kChunkedSeq) ? 2 : 1;
}
constexpr int channels_per_cta(int n, int k) { return kThreads / (n / (n < 4 ? n : 4)) * k; }

struct BwdParams {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;      // may be null
    const void* z;       // may be null
    const float* bias;   // may be null
    const void* dy;      // (batch, dim, L) of the gradient type GT
    const float* dlast;  // (batch, dim, N) fp32, may be null
    const float* h0;     // (batch, dim, N) fp32 initial state of the forward, may be null
    void* du;            // (batch, dim, L) of the gradient type GT: fp32 or the I/O type
    void* ddelta;        // (batch, dim, L) GT
    void* dz;            // (batch, dim, L) GT, null when z is null
    float* dA;           // (dim, N), accumulated: zeroed by the host
    float* dB;           // (batch, L, N), accumulated
    float* dC;           // (batch, L, N), accumulated
    float* dD;           // (dim), accumulated, may be null when D is null
    float* dbias;        // (dim), accumulated, may be null
    float* dh0;          // (batch, dim, N), may be null
    float* ckpt;         // workspace: (batch, dim, ntiles, N)
    // Chunked backward (nchunks > 1): CTA z takes tokens [z chunk_len,
    // (z + 1) chunk_len), starting from the state hc[z] (z > 0; h0 for z = 0)
    // with the adjoint xc[z] flowing in from the later chunks (z < nchunks - 1;
    // dlast for the last chunk); only chunk 0 writes dh0.  Both are
    // (nchunks, batch, dim, N) in the workspace.
    float* hc;
    float* xc;
    float* agg;          // the chunks' maps: F, PF, Q, PQ, each (nchunks, batch, dim, N)
    int64_t batch, dim, L, ntiles;
    int64_t chunk_len;   // a multiple of kChunkAlign, or >= L with one chunk
    int nchunks;
};


// K: channels per thread (2 at N = 16, 1 otherwise).
template <typename T, int N, int K> struct BwdShape {
    static constexpr int S = N < 4 ? N : 4;     // states per thread and channel
    static constexpr int G = N / S;             // lanes per slot
    static constexpr int SLOTS = kThreads / G;  // slots per CTA
    static constexpr int CH = SLOTS * K;        // channels per CTA
    static constexpr int ES = (int)sizeof(T);
    // staging: thread tid takes tokens [(tid % TPR) EPT, +EPT) of channel tid / TPR
    static constexpr int EPT = CH * kTT / kThreads;
    static constexpr int TPR = kTT / EPT;
    // (Delta, Delta x, ds, 0) per (channel, token); rows padded by 16 bytes so
    // that the 32 / G channels a warp reads at once fall in distinct banks
    static constexpr int REC_ROW = kTT * 16 + 16;
    static constexpr int OFF_W = 0;
    // per (channel, lane, token) the lane's partial (s, q, r, 0), at 16-byte
    // unit c R_ROW/16 + lane (kTT + 8 / G) + token with R_ROW/16 = 1 mod 8:
    // the lanes storing one token (2 or more channels x G lanes) and the
    // threads reading one lane's partials (4 channels x 2 token halves) each
    // hit 8 distinct 16-byte bank groups per quarter-warp
    static constexpr int LANE_U = kTT + 8 / G;
    static constexpr int R_ROW = (G * LANE_U + 1) * 16;
    static constexpr int OFF_R = OFF_W + CH * REC_ROW;
    static constexpr int OFF_BC = OFF_R + CH * R_ROW;     // fp32 B[kTT][N], C[kTT][N]
    // per slot and token the K-channel sums of g Delta x (dB) and ds h (dC);
    // rows padded to 16 words mod 32 (conflict-free 16-byte stores)
    static constexpr int P_ROW = kTT * 2 * N + 16;        // floats
    static constexpr int OFF_P = OFF_BC + 2 * kTT * N * 4;
    // the next tile's raw inputs: u, delta, z as [CH][kTT] of T, dy as
    // [CH][kTT] of fp32 or T (room for fp32), B and C as [kTT][N] of T
    static constexpr int RAW_PLANE = CH * kTT * ES;
    static constexpr int OFF_RAW = OFF_P + SLOTS * P_ROW * 4;
    static constexpr int OFF_DY = OFF_RAW + 3 * RAW_PLANE;
    static constexpr int OFF_RB = OFF_DY + CH * kTT * 4;
    static constexpr int OFF_RC = OFF_RB + kTT * N * ES;
    static constexpr int SMEM2 = OFF_RC + kTT * N * ES;
    static_assert(EPT * kThreads == CH * kTT && kTT % EPT == 0, "staging split");
    // Pass 1 stages T1 = 4 kTT tokens at a time in its own layout over the
    // same shared memory (it ends before pass 2 starts): (Delta, Delta x) per
    // (channel, token), fp32 B rows, and the raw u, delta and B of the next
    // tile.  Thread tid stages tokens [(tid % TPR1) EPT1, +EPT1) of channel
    // tid / TPR1.
    static constexpr int T1 = 4 * kTT;
    static constexpr int EPT1 = CH * T1 / kThreads;
    static constexpr int TPR1 = T1 / EPT1;
    static constexpr int W1_ROW = T1 * 8 + 8;
    static constexpr int OFF1_W = 0;
    static constexpr int OFF1_B = (CH * W1_ROW + 15) / 16 * 16;     // fp32 B[T1][N]
    static constexpr int OFF1_RAW = OFF1_B + T1 * N * 4;            // u, delta: [CH][T1] of T
    static constexpr int RAW1_PLANE = CH * T1 * ES;
    static constexpr int OFF1_RB = OFF1_RAW + 2 * RAW1_PLANE;       // B: [T1][N] of T
    static constexpr int SMEM1 = OFF1_RB + (T1 * N * ES + 15) / 16 * 16;
    static constexpr int SMEM = SMEM1 > SMEM2 ? SMEM1 : SMEM2;
    static_assert(EPT1 * kThreads == CH * T1 && T1 % EPT1 == 0 && EPT1 % 8 == 0, "pass-1 staging split");
    static_assert(OFF1_RAW % 16 == 0 && OFF1_RB % 16 == 0 && RAW1_PLANE % 16 == 0, "pass-1 alignment");
    static_assert(N % S == 0 && 32 % G == 0 && R_ROW / 16 % 8 == 1, "state split");
    static_assert(OFF_R % 16 == 0 && OFF_P % 16 == 0 && OFF_RAW % 16 == 0 && OFF_DY % 16 == 0 &&
                  OFF_RB % 16 == 0 && OFF_RC % 16 == 0, "alignment");
};

__device__ __forceinline__ float sigmoid(float v) { return rcp(1.0f + ex2(-v * kLog2e)); }

// The S states a thread holds for one channel, as (S + 1) / 2 pairs for the
// paired fp32 instructions; with S = 1 the pair's second lane is padding,
// loaded as 0 and never stored.  Rows are aligned to 4 S bytes.
template <int S>
__device__ __forceinline__ void ld_pairs(const float* p, float2* v) {
    if constexpr (S == 4) {
        const float4 q = *reinterpret_cast<const float4*>(p);
        v[0] = make_float2(q.x, q.y);
        v[1] = make_float2(q.z, q.w);
    } else if constexpr (S == 2) {
        v[0] = *reinterpret_cast<const float2*>(p);
    } else {
        v[0] = make_float2(p[0], 0.0f);
    }
}
template <int S>
__device__ __forceinline__ void st_pairs(float* p, const float2* v) {
    if constexpr (S == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    } else if constexpr (S == 2) {
        *reinterpret_cast<float2*>(p) = v[0];
    } else {
        p[0] = v[0].x;
    }
}
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }
// 2^x of both lanes on the special-function unit
__device__ __forceinline__ float2 ex2x2(float2 x) { return make_float2(ex2(x.x), ex2(x.y)); }

// Exact zero-order hold, for a pair of states: e = Delta A log2(e), a = 2^e,
// ia = 1 / A (0 where A = 0).
// The weight w = (exp(Delta A) - 1) / A = (a - 1) ia, except for |e| < 1/8,
// where a - 1 keeps only the absolute accuracy of 2^x; there the series
// Delta (1 + x / 2 + x^2 / 6 + x^3 / 24) in x = Delta A (Delta at A = 0)
// is used, as in the forward scan.
constexpr float kZohW = 0.125f;
constexpr float kW1 = 0.34657359027997264f;    // ln 2 / 2
constexpr float kW2 = 0.08007550231970023f;    // (ln 2)^2 / 6
constexpr float kW3 = 0.013876027166205394f;   // (ln 2)^3 / 24
__device__ __forceinline__ float2 zoh_weight(float2 a, float2 e, float2 dt, float2 ia) {
    float2 w = __fmul2_rn(__fadd2_rn(a, f2(-1.0f)), ia);
    float2 t = __ffma2_rn(e, f2(kW3), f2(kW2));
    t = __ffma2_rn(e, t, f2(kW1));
    t = __ffma2_rn(e, t, f2(1.0f));
    const float2 ws = __fmul2_rn(dt, t);
    if (fabsf(e.x) < kZohW) w.x = ws.x;
    if (fabsf(e.y) < kZohW) w.y = ws.y;
    return w;
}
// dw/dA = (Delta a - w) / A = Delta^2 psi(x), psi(x) = (x e^x - e^x + 1) / x^2
// = sum_k (k + 1) x^k / (k + 2)!.  Where |x| < 1/2 the difference Delta a - w
// cancels, and psi is summed to k = 7 instead (the first term left out is
// below 3e-8 of psi there); the coefficients are in powers of e = x log2(e).
constexpr float kZohWA = 0.72134752044448170f;   // |x| < 1/2
__device__ __forceinline__ float2 zoh_weight_da(float2 a, float2 e, float2 dt, float2 ia, float2 w) {
    float2 wa = __fmul2_rn(__ffma2_rn(dt, a, make_float2(-w.x, -w.y)), ia);
    // (k + 1) (ln 2)^k / (k + 2)!, k = 7 down to 0
    float2 t = __ffma2_rn(e, f2(1.694748200451093e-06f), f2(1.925441299172701e-05f));
    t = __ffma2_rn(e, t, f2(0.0001904794020918349f));
    t = __ffma2_rn(e, t, f2(0.0016030215179380792f));
    t = __ffma2_rn(e, t, f2(0.011100821732964315f));
    t = __ffma2_rn(e, t, f2(0.060056626739775174f));
    t = __ffma2_rn(e, t, f2(0.23104906018664842f));
    t = __ffma2_rn(e, t, f2(0.5f));
    const float2 ws = __fmul2_rn(__fmul2_rn(dt, dt), t);
    if (fabsf(e.x) < kZohWA) wa.x = ws.x;
    if (fabsf(e.y) < kZohWA) wa.y = ws.y;
    return wa;
}

// cp.async of `bytes` (4, 8, 16 or 32) from global to shared memory, both
// aligned to min(bytes, 16); src_ok false fills zeros
template <int BYTES>
__device__ __forceinline__ void cp_async_bytes(void* smem, const void* gmem, bool src_ok) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    if constexpr (BYTES == 32) {
        cp_async_bytes<16>(smem, gmem, src_ok);
        cp_async_bytes<16>(static_cast<char*>(smem) + 16, static_cast<const char*>(gmem) + 16, src_ok);
    } else if constexpr (BYTES == 16) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                     "r"(src_ok ? 16 : 0) : "memory");
    } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;\n" ::"r"(s), "l"(gmem),
                     "n"(BYTES), "r"(src_ok ? BYTES : 0) : "memory");
    }
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// E consecutive elements of type T in shared memory -> fp32 (16-byte aligned
// when E * sizeof(T) >= 16, else E * sizeof(T)-aligned)
template <typename T, int E>
__device__ __forceinline__ void lds_row(const unsigned char* p, float* v) {
    if constexpr (sizeof(T) == 2 && E % 4 == 0) {
#pragma unroll
        for (int q = 0; q < E / 4; q++) {
            const uint2 w = reinterpret_cast<const uint2*>(p)[q];
            v[4 * q] = __uint_as_float(w.x << 16);
            v[4 * q + 1] = __uint_as_float(w.x & 0xffff0000u);
            v[4 * q + 2] = __uint_as_float(w.y << 16);
            v[4 * q + 3] = __uint_as_float(w.y & 0xffff0000u);
        }
    } else if constexpr (sizeof(T) == 4 && E % 4 == 0) {
#pragma unroll
        for (int q = 0; q < E / 4; q++) {
            const float4 w = reinterpret_cast<const float4*>(p)[q];
            v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; e++) v[e] = io<T>::to_f32(reinterpret_cast<const T*>(p)[e]);
    }
}

// E consecutive fp32 values to global memory as GT (fp32, or bf16 rounded to
// nearest even): 16-byte (fp32) or 8-byte (bf16) stores of 4 values when VEC
// (dst 16-byte aligned at the row, 4-element aligned here)
template <typename GT, int E, bool VEC>
__device__ __forceinline__ void stg_row(GT* dst, const float* v, int valid) {
    if constexpr (VEC && E % 4 == 0) {
#pragma unroll
        for (int q = 0; q < E / 4; q++) {
            if constexpr (sizeof(GT) == 4) {
                reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(v[4 * q], v[4 * q + 1]);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(v[4 * q + 2], v[4 * q + 3]);
                reinterpret_cast<uint2*>(dst)[q] = make_uint2(*reinterpret_cast<const unsigned*>(&lo),
                                                              *reinterpret_cast<const unsigned*>(&hi));
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; e++)
            if (e < valid) dst[e] = io<GT>::from_f32(v[e]);
    }
}

// VEC: L % 8 == 0 and every tensor 16-byte aligned (cp.async staging, vector
// stores); otherwise bounds-checked scalar copies.  ZOH: the exact
// zero-order-hold input term; the records then carry x where they carry
// Delta x for the first-order term.  GT: the type of dy and of du, ddelta,
// dz (fp32, or the I/O type: read as given, written as the fp32 values
// rounded once).
template <typename T, int N, int K, bool HAS_Z, bool SOFTPLUS, bool VEC, bool ZOH, typename GT = float>
__global__ void __launch_bounds__(kThreads, 12) scan_bwd_kernel(BwdParams p) {
    using Sh = BwdShape<T, N, K>;
    constexpr int S = Sh::S, G = Sh::G, SLOTS = Sh::SLOTS, CH = Sh::CH;
    constexpr int EPT = Sh::EPT, TPR = Sh::TPR, ES = Sh::ES;
    constexpr int SP = (S + 1) / 2, KP = K * SP;   // state pairs per channel, per thread
    extern __shared__ __align__(16) unsigned char smem[];
    float* BB = reinterpret_cast<float*>(smem + Sh::OFF_BC);   // [kTT][N]
    float* CC = BB + kTT * N;
    float* P = reinterpret_cast<float*>(smem + Sh::OFF_P);     // [SLOTS][P_ROW]
    auto wrec = [&](int c, int j) -> float4& {
        return *reinterpret_cast<float4*>(smem + Sh::OFF_W + c * Sh::REC_ROW + j * 16);
    };
    constexpr int LANE_U = Sh::LANE_U;
    auto rrec = [&](int c, int j, int lane) -> float4& {
        return *reinterpret_cast<float4*>(smem + Sh::OFF_R + c * Sh::R_ROW +
                                          (lane * LANE_U + j) * 16);
    };

    const int tid = threadIdx.x;
    const int slot = tid / G, gi = tid % G, n0 = gi * S;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int64_t L = p.L;
    // this CTA's chunk of the sequence, its initial state and incoming adjoint
    const int cz = (int)blockIdx.z;
    const int64_t t_lo = (int64_t)cz * p.chunk_len;
    const int64_t t_hi = L - t_lo < p.chunk_len ? L : t_lo + p.chunk_len;
    const int64_t chunk_off = (int64_t)cz * p.batch * p.dim * N;
    const float* h0p = cz == 0 ? p.h0 : p.hc + chunk_off;
    const float* dlastp = cz == p.nchunks - 1 ? p.dlast : p.xc + chunk_off;
    float* dh0p = cz == 0 ? p.dh0 : nullptr;
    // recurrence role: channels slot + k SLOTS of the CTA, states n0 .. n0+S-1
    bool act[K];
    int64_t crow[K];                 // flat channel b * dim + d (0 when inactive)
    float* ckp[K];
    float2 A2[KP], g[KP], dA[KP], h[KP];   // A log2(e), adjoint, dA sums, state
    float2 IA[KP];                          // 1 / A (ZOH; 0 where A = 0)
#pragma unroll
    for (int k = 0; k < K; k++) {
        const int64_t d = d0 + slot + k * SLOTS;
        act[k] = d < p.dim;
        crow[k] = act[k] ? b * p.dim + d : 0;
        ckp[k] = p.ckpt + crow[k] * p.ntiles * N + n0;
        auto a2 = [&](int i) { return (act[k] && i < S) ? p.A[d * N + n0 + i] * kLog2e : 0.0f; };
        auto ia = [&](int i) {
            const float av = (act[k] && i < S) ? p.A[d * N + n0 + i] : 0.0f;
            return (ZOH && av != 0.0f) ? 1.0f / av : 0.0f;
        };
        auto g0 = [&](int i) {
            return (act[k] && i < S && dlastp) ? dlastp[crow[k] * N + n0 + i] : 0.0f;
        };
        auto s0 = [&](int i) { return (act[k] && i < S && h0p) ? h0p[crow[k] * N + n0 + i] : 0.0f; };
#pragma unroll
        for (int pi = 0; pi < SP; pi++) {
            A2[k * SP + pi] = make_float2(a2(2 * pi), a2(2 * pi + 1));
            IA[k * SP + pi] = make_float2(ia(2 * pi), ia(2 * pi + 1));
            g[k * SP + pi] = make_float2(g0(2 * pi), g0(2 * pi + 1));
            h[k * SP + pi] = make_float2(s0(2 * pi), s0(2 * pi + 1));   // the forward's start
            dA[k * SP + pi] = f2(0.0f);
        }
    }
    // staging role: tokens sj .. sj+EPT-1 of channel sc of the CTA
    const int sc = tid / TPR, sj = (tid % TPR) * EPT;
    const bool okc = d0 + sc < p.dim;
    const int64_t srow = (b * p.dim + (okc ? d0 + sc : 0)) * L;   // row start in (batch, dim, L)
    const float bias_c = (p.bias && okc) ? p.bias[d0 + sc] : 0.0f;
    const float D_c = (p.D && okc) ? p.D[d0 + sc] : 0.0f;
    const T* bu = static_cast<const T*>(p.u);
    const T* bdl = static_cast<const T*>(p.delta);
    const T* bz = static_cast<const T*>(p.z);
    const T* bB = static_cast<const T*>(p.B) + b * L * N;
    const T* bC = static_cast<const T*>(p.C) + b * L * N;
    unsigned char* raw = smem + Sh::OFF_RAW + (sc * kTT + sj) * ES;
    unsigned char* rawdy = smem + Sh::OFF_DY + (sc * kTT + sj) * (int)sizeof(GT);
    const GT* gdy = static_cast<const GT*>(p.dy);

    // Copy tile [t0, t0 + kTT)'s inputs into the raw buffers (asynchronously
    // when VEC); `full` adds z, dy and C.
    auto load_tile = [&](int64_t t0, bool full) {
        if constexpr (VEC) {
            const int64_t g0 = srow + t0 + sj;
            cp_async_bytes<EPT * ES>(raw, bu + g0, okc);
            cp_async_bytes<EPT * ES>(raw + Sh::RAW_PLANE, bdl + g0, okc);
            if (full && HAS_Z) cp_async_bytes<EPT * ES>(raw + 2 * Sh::RAW_PLANE, bz + g0, okc);
            if (full) cp_async_bytes<EPT * (int)sizeof(GT)>(rawdy, gdy + g0, okc);
            constexpr int BCQ = kTT * N * ES / 16;   // 16-byte chunks of one tile of B
            for (int i = tid; i < (full ? 2 : 1) * BCQ; i += kThreads) {
                const int which = i / BCQ, q = i % BCQ;
                cp_async_bytes<16>(smem + (which ? Sh::OFF_RC : Sh::OFF_RB) + q * 16,
                                   (which ? bC : bB) + t0 * N + q * (16 / ES), true);
            }
        } else {
            T* ru = reinterpret_cast<T*>(raw);
#pragma unroll
            for (int e = 0; e < EPT; e++) {
                const int64_t t = t0 + sj + e;
                const bool ok = okc && t < L;
                ru[e] = ok ? bu[srow + t] : io<T>::from_f32(0.0f);
                reinterpret_cast<T*>(raw + Sh::RAW_PLANE)[e] = ok ? bdl[srow + t] : io<T>::from_f32(0.0f);
                if (full && HAS_Z)
                    reinterpret_cast<T*>(raw + 2 * Sh::RAW_PLANE)[e] = ok ? bz[srow + t] : io<T>::from_f32(0.0f);
                if (full) reinterpret_cast<GT*>(rawdy)[e] = ok ? gdy[srow + t] : io<GT>::from_f32(0.0f);
            }
            for (int i = tid; i < (full ? 2 : 1) * kTT * N; i += kThreads) {
                const int which = i / (kTT * N), q = i % (kTT * N);
                const bool ok = t0 + q / N < L;
                reinterpret_cast<T*>(smem + (which ? Sh::OFF_RC : Sh::OFF_RB))[q] =
                    ok ? (which ? bC : bB)[t0 * N + q] : io<T>::from_f32(0.0f);
            }
        }
    };

    // Raw tile -> the records the recurrence reads.  Outside the sequence or
    // the channel range everything is 0: Delta = 0 makes a = 1 and the input
    // term 0, and ds = 0 adds nothing to g, so padded tokens leave the state
    // and the adjoint unchanged.  `ex` keeps (x, dz factor, softplus') of the
    // thread's own elements for its epilogue.
    auto put = [&](int64_t t0, bool full, float (&ex)[EPT][3]) {
        float xr[EPT], vr[EPT], zr[EPT], dyr[EPT];
        lds_row<T, EPT>(raw, xr);
        lds_row<T, EPT>(raw + Sh::RAW_PLANE, vr);
        if (full && HAS_Z) lds_row<T, EPT>(raw + 2 * Sh::RAW_PLANE, zr);
        if (full) lds_row<GT, EPT>(rawdy, dyr);
#pragma unroll
        for (int e = 0; e < EPT; e++) {
            const bool ok = okc && t0 + sj + e < L;
            const float v = vr[e] + bias_c;
            const float dt = ok ? (SOFTPLUS ? softplus(v) : v) : 0.0f;
            float ds = full ? dyr[e] : 0.0f, dzf = 0.0f;
            if (full && HAS_Z) {
                const float sg = sigmoid(zr[e]);
                ds = dyr[e] * zr[e] * sg;
                dzf = dyr[e] * sg * fmaf(zr[e], 1.0f - sg, 1.0f);
            }
            wrec(sc, sj + e) = make_float4(dt, ZOH ? xr[e] : dt * xr[e], ds, 0.0f);
            if (full) {
                ex[e][0] = xr[e];
                ex[e][1] = dzf;
                ex[e][2] = (SOFTPLUS && ok) ? sigmoid(v) : 1.0f;
            }
        }
        const T* rb = reinterpret_cast<const T*>(smem + Sh::OFF_RB);
        const T* rc = reinterpret_cast<const T*>(smem + Sh::OFF_RC);
        for (int i = tid; i < kTT * N; i += kThreads) {
            BB[i] = io<T>::to_f32(rb[i]);
            if (full) CC[i] = io<T>::to_f32(rc[i]);
        }
    };
    float ex[EPT][3];

    // ---- pass 1: forward over T1-token tiles, checkpoint at every kTT tokens ----
    {
        constexpr int T1 = Sh::T1, EPT1 = Sh::EPT1, TPR1 = Sh::TPR1;
        const int sc1 = tid / TPR1, sj1 = (tid % TPR1) * EPT1;
        const bool okc1 = d0 + sc1 < p.dim;
        const int64_t goff1 = (b * p.dim + (okc1 ? d0 + sc1 : 0)) * L + sj1;
        const float bias1 = (p.bias && okc1) ? p.bias[d0 + sc1] : 0.0f;
        unsigned char* raw1 = smem + Sh::OFF1_RAW + (sc1 * T1 + sj1) * ES;
        // (Delta, Delta x) of channel c, token j of the tile ((Delta, x) with ZOH)
        auto w1rec = [&](int c, int j) -> float2& {
            return *reinterpret_cast<float2*>(smem + Sh::OFF1_W + c * Sh::W1_ROW + j * 8);
        };
        auto load1 = [&](int64_t t0) {
            const int64_t gt = goff1 + t0;
            if constexpr (VEC) {
                // 16-byte pieces of the thread's EPT1 tokens; with L % kTT == 0
                // each piece lies wholly inside or wholly past the sequence
                constexpr int PE = 16 / ES;   // elements per piece
#pragma unroll
                for (int q = 0; q < EPT1 / PE; q++) {
                    const bool ok = okc1 && t0 + sj1 + q * PE < L;
                    cp_async_bytes<16>(raw1 + q * 16, bu + (ok ? gt + q * PE : 0), ok);
                    cp_async_bytes<16>(raw1 + Sh::RAW1_PLANE + q * 16, bdl + (ok ? gt + q * PE : 0), ok);
                }
                constexpr int BCQ1 = T1 * N * ES / 16;
                for (int i = tid; i < BCQ1; i += kThreads) {
                    const bool ok = t0 + (int64_t)i * (16 / ES) / N < L;
                    cp_async_bytes<16>(smem + Sh::OFF1_RB + i * 16, bB + (ok ? t0 * N + i * (16 / ES) : 0), ok);
                }
            } else {
                const T zero = io<T>::from_f32(0.0f);
#pragma unroll 8
                for (int e = 0; e < EPT1; e++) {
                    const bool ok = okc1 && t0 + sj1 + e < L;
                    reinterpret_cast<T*>(raw1)[e] = ok ? bu[gt + e] : zero;
                    reinterpret_cast<T*>(raw1 + Sh::RAW1_PLANE)[e] = ok ? bdl[gt + e] : zero;
                }
                for (int i = tid; i < T1 * N; i += kThreads) {
                    const bool ok = t0 + i / N < L;
                    reinterpret_cast<T*>(smem + Sh::OFF1_RB)[i] = ok ? bB[t0 * N + i] : zero;
                }
            }
        };
        auto put1 = [&](int64_t t0) {
#pragma unroll
            for (int e0 = 0; e0 < EPT1; e0 += 8) {
                float xr[8], vr[8];
                lds_row<T, 8>(raw1 + e0 * ES, xr);
                lds_row<T, 8>(raw1 + Sh::RAW1_PLANE + e0 * ES, vr);
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const bool ok = okc1 && t0 + sj1 + e0 + e < L;
                    const float v = vr[e] + bias1;
                    const float dt = ok ? (SOFTPLUS ? softplus(v) : v) : 0.0f;
                    w1rec(sc1, sj1 + e0 + e) = make_float2(dt, ZOH ? xr[e] : dt * xr[e]);
                }
            }
            const T* rb = reinterpret_cast<const T*>(smem + Sh::OFF1_RB);
            float* bb1 = reinterpret_cast<float*>(smem + Sh::OFF1_B);
            for (int i = tid; i < T1 * N; i += kThreads) bb1[i] = io<T>::to_f32(rb[i]);
        };
        const float* bb1 = reinterpret_cast<const float*>(smem + Sh::OFF1_B);
        const int64_t k1_lo = t_lo / T1, k1_hi = (t_hi + T1 - 1) / T1;   // t_lo: a multiple of T1
        if (k1_hi > k1_lo) load1(k1_lo * T1);
        for (int64_t k1 = k1_lo; k1 < k1_hi; k1++) {
            const int64_t t0 = k1 * T1;
            if constexpr (VEC) cp_async_wait_all();
            __syncthreads();             // raw tile complete, previous tile's records consumed
            put1(t0);
            __syncthreads();
            if (k1 + 1 < k1_hi) load1(t0 + T1);
#pragma unroll
            for (int j = 0; j < T1; j++) {
                if (j % kTT == 0) {      // the state before each kTT-token tile
                    const int64_t kt = t0 / kTT + j / kTT;
                    if (kt < p.ntiles) {
#pragma unroll
                        for (int k = 0; k < K; k++)
                            if (act[k]) st_pairs<S>(ckp[k] + kt * N, h + k * SP);
                    }
                }
                float2 Bv[SP];
                ld_pairs<S>(bb1 + j * N + n0, Bv);
#pragma unroll
                for (int k = 0; k < K; k++) {
                    const float2 w = w1rec(slot + k * SLOTS, j);
#pragma unroll
                    for (int pi = 0; pi < SP; pi++) {
                        const int q = k * SP + pi;
                        const float2 e = __fmul2_rn(f2(w.x), A2[q]);
                        const float2 a = ex2x2(e);
                        float2 in = __fmul2_rn(f2(w.y), Bv[pi]);
                        if constexpr (ZOH) in = __fmul2_rn(zoh_weight(a, e, f2(w.x), IA[q]), in);
                        h[q] = __ffma2_rn(a, h[q], in);
                    }
                }
            }
        }
        __syncthreads();                 // pass 1's buffers overlap pass 2's
    }

    // ---- pass 2: tiles in reverse ----
    float dD_acc = 0.0f, db_acc = 0.0f;
    const bool vec_red = N % 4 == 0 &&
        ((reinterpret_cast<uintptr_t>(p.dB) | reinterpret_cast<uintptr_t>(p.dC)) & 15) == 0;
    float2 hc[KP];   // the checkpoint of the tile processed next
    auto load_ckpt = [&](int64_t kt) {
#pragma unroll
        for (int k = 0; k < K; k++) {
            if (act[k]) {
                ld_pairs<S>(ckp[k] + kt * N, hc + k * SP);
            } else {
#pragma unroll
                for (int pi = 0; pi < SP; pi++) hc[k * SP + pi] = f2(0.0f);
            }
        }
    };
    const int64_t kt_lo = t_lo / kTT, kt_hi = (t_hi + kTT - 1) / kTT;
    if (kt_hi > kt_lo) {
        load_tile((kt_hi - 1) * kTT, true);
        load_ckpt(kt_hi - 1);
    }
    for (int64_t kt = kt_hi - 1; kt >= kt_lo; kt--) {
        const int64_t t0 = kt * kTT;
        if constexpr (VEC) cp_async_wait_all();
        __syncthreads();                 // raw tile complete, the previous tile's epilogue done
        put(t0, true, ex);
        float2 hs[kTT + 1][KP];          // the state before the tile, then after each token
#pragma unroll
        for (int q = 0; q < KP; q++) hs[0][q] = hc[q];
        __syncthreads();
        if (kt > kt_lo) {                // the tile before, in flight while this one computes
            load_tile(t0 - kTT, true);
            load_ckpt(kt - 1);
        }
#pragma unroll
        for (int j = 0; j < kTT; j++) {
            float2 Bv[SP];
            ld_pairs<S>(BB + j * N + n0, Bv);
#pragma unroll
            for (int k = 0; k < K; k++) {
                const float4 w = wrec(slot + k * SLOTS, j);
#pragma unroll
                for (int pi = 0; pi < SP; pi++) {
                    const int q = k * SP + pi;
                    const float2 e = __fmul2_rn(f2(w.x), A2[q]);
                    const float2 a = ex2x2(e);
                    float2 in = __fmul2_rn(f2(w.y), Bv[pi]);
                    if constexpr (ZOH) in = __fmul2_rn(zoh_weight(a, e, f2(w.x), IA[q]), in);
                    hs[j + 1][q] = __ffma2_rn(a, hs[j][q], in);
                }
            }
        }
        // the adjoint, backwards through the tile
#pragma unroll
        for (int j = kTT - 1; j >= 0; j--) {
            float2 Bv[SP], Cv[SP], pb[SP], pc[SP];
            ld_pairs<S>(BB + j * N + n0, Bv);
            ld_pairs<S>(CC + j * N + n0, Cv);
#pragma unroll
            for (int k = 0; k < K; k++) {
                const float4 w = wrec(slot + k * SLOTS, j);   // Delta, Delta x (ZOH: x), ds
                const float2 dt = f2(w.x), dtx = f2(w.y), ds = f2(w.z);
                float2 sa = f2(0.0f), qa = f2(0.0f), ra = f2(0.0f), va = f2(0.0f);
#pragma unroll
                for (int pi = 0; pi < SP; pi++) {
                    const int q = k * SP + pi;
                    const float2 e = __fmul2_rn(dt, A2[q]);
                    const float2 a = ex2x2(e);
                    g[q] = __ffma2_rn(ds, Cv[pi], g[q]);                      // + ds C
                    if constexpr (HAS_Z) sa = __ffma2_rn(Cv[pi], hs[j + 1][q], sa);
                    pc[pi] = k == 0 ? __fmul2_rn(ds, hs[j + 1][q]) : __ffma2_rn(ds, hs[j + 1][q], pc[pi]);
                    const float2 ga = __fmul2_rn(g[q], a);
                    if constexpr (ZOH) {
                        const float2 wq = zoh_weight(a, e, dt, IA[q]);
                        const float2 gw = __fmul2_rn(g[q], wq);
                        qa = __ffma2_rn(gw, Bv[pi], qa);                      // g w B
                        pb[pi] = k == 0 ? __fmul2_rn(gw, dtx) : __ffma2_rn(gw, dtx, pb[pi]);
                        va = __ffma2_rn(ga, Bv[pi], va);                      // g a B
                        const float2 gwa = __fmul2_rn(g[q], zoh_weight_da(a, e, dt, IA[q], wq));
                        dA[q] = __ffma2_rn(gwa, __fmul2_rn(Bv[pi], dtx), dA[q]);   // g dw/dA B x
                    } else {
                        qa = __ffma2_rn(g[q], Bv[pi], qa);
                        pb[pi] = k == 0 ? __fmul2_rn(g[q], dtx) : __ffma2_rn(g[q], dtx, pb[pi]);
                    }
                    const float2 pp = __fmul2_rn(ga, hs[j][q]);              // g a h_(t-1)
                    ra = __ffma2_rn(A2[q], pp, ra);
                    dA[q] = __ffma2_rn(dt, pp, dA[q]);
                    g[q] = ga;
                }
                rrec(slot + k * SLOTS, j, gi) =
                    make_float4(sa.x + sa.y, qa.x + qa.y, ra.x + ra.y, ZOH ? va.x + va.y : 0.0f);
            }
            st_pairs<S>(P + slot * Sh::P_ROW + j * 2 * N + n0, pb);
            st_pairs<S>(P + slot * Sh::P_ROW + j * 2 * N + N + n0, pc);
        }
        __syncthreads();
        // dB, dC of the tile: the sums over the CTA's slots, added to the batch row
        if (vec_red) {
            constexpr int NQ = N % 4 == 0 ? N / 4 : 1, NV = kTT * 2 * NQ;
            for (int o = tid; o < NV; o += kThreads) {
                const int j = o / (2 * NQ), which = (o / NQ) % 2, qd = o % NQ;
                const float* src = P + j * 2 * N + which * N + qd * 4;
                float4 v = *reinterpret_cast<const float4*>(src);
                float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
#pragma unroll
                for (int sl = 1; sl < SLOTS; sl++) {
                    v = *reinterpret_cast<const float4*>(src + sl * Sh::P_ROW);
                    lo = __fadd2_rn(lo, make_float2(v.x, v.y));
                    hi = __fadd2_rn(hi, make_float2(v.z, v.w));
                }
                const float4 acc = make_float4(lo.x, lo.y, hi.x, hi.y);
                if (t0 + j < L) {
                    float* dst = (which ? p.dC : p.dB) + (b * L + t0 + j) * N + qd * 4;
                    atomicAdd(reinterpret_cast<float4*>(dst), acc);
                }
            }
        } else {
            for (int o = tid; o < kTT * 2 * N; o += kThreads) {
                const int j = o / (2 * N), which = (o / N) % 2, n = o % N;
                const float* src = P + j * 2 * N + which * N + n;
                float acc = 0.0f;
                for (int sl = 0; sl < SLOTS; sl++) acc += src[sl * Sh::P_ROW];
                if (t0 + j < L) atomicAdd((which ? p.dC : p.dB) + (b * L + t0 + j) * N + n, acc);
            }
        }
        // the thread's own elements: du, ddelta, dz, and the dD, delta_bias sums
        {
            float dxo[EPT], dvo[EPT], dzo[EPT];
#pragma unroll
            for (int e = 0; e < EPT; e++) {
                const int j = sj + e;
                float4 rs = rrec(sc, j, 0);
#pragma unroll
                for (int l = 1; l < G; l++) {
                    const float4 v = rrec(sc, j, l);
                    rs.x += v.x; rs.y += v.y; rs.z += v.z;
                    if constexpr (ZOH) rs.w += v.w;
                }
                const float4 w = wrec(sc, j);
                if constexpr (ZOH) {
                    dxo[e] = fmaf(w.z, D_c, rs.y);                             // ds D + sum g w B
                    dvo[e] = fmaf(ex[e][0], rs.w, rs.z * kLn2) * ex[e][2];     // (r + x v) softplus'
                } else {
                    dxo[e] = fmaf(w.z, D_c, w.x * rs.y);                       // ds D + Delta q
                    dvo[e] = fmaf(ex[e][0], rs.y, rs.z * kLn2) * ex[e][2];     // (r + x q) softplus'
                }
                dzo[e] = ex[e][1] * fmaf(D_c, ex[e][0], rs.x);                 // dy (s + D x) silu'
                if (okc && t0 + j < L) {
                    dD_acc = fmaf(w.z, ex[e][0], dD_acc);
                    db_acc += dvo[e];
                }
            }
            if (okc) {
                const int64_t rem = L - (t0 + sj);
                const int valid = rem < EPT ? (int)rem : EPT;
                stg_row<GT, EPT, VEC>(static_cast<GT*>(p.du) + srow + t0 + sj, dxo, valid);
                stg_row<GT, EPT, VEC>(static_cast<GT*>(p.ddelta) + srow + t0 + sj, dvo, valid);
                if constexpr (HAS_Z) stg_row<GT, EPT, VEC>(static_cast<GT*>(p.dz) + srow + t0 + sj, dzo, valid);
            }
        }
    }

    // ---- per-channel and per-state sums ----
#pragma unroll
    for (int off = 1; off < TPR; off <<= 1) {   // the TPR adjacent lanes staging one channel
        dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, off);
        db_acc += __shfl_xor_sync(0xffffffffu, db_acc, off);
    }
    if (tid % TPR == 0 && okc) {
        if (p.dD) atomicAdd(p.dD + d0 + sc, dD_acc);
        if (p.dbias) atomicAdd(p.dbias + d0 + sc, db_acc);
    }
#pragma unroll
    for (int k = 0; k < K; k++) {
        if (!act[k]) continue;
        const int64_t d = d0 + slot + k * SLOTS;
#pragma unroll
        for (int i = 0; i < S; i++) {
            const float2 da = dA[k * SP + i / 2], gg = g[k * SP + i / 2];
            atomicAdd(p.dA + d * N + n0 + i, i % 2 ? da.y : da.x);
            if (dh0p) dh0p[crow[k] * N + n0 + i] = i % 2 ? gg.y : gg.x;
        }
    }
}

constexpr float kWalkCut = 9.094947017729282e-13f;   // 2^-40
constexpr int kAggThreads = 128;
constexpr int kWalkBlock = 8;   // tokens whose inputs are loaded before they are walked

// Chunked backward, step 1.  Thread: S = min(N, 4) states of one channel
// (flat row b dim + d) in chunk blockIdx.y.  The same Delta, decay, input
// weight and ds as scan_bwd_kernel:
//   F  = sum_t (prod_(r > t) a_r) w_t B_t x_t   over the chunk's tokens t
//        (walked back from its end: F += W w B x, then W *= a)
//   Q  = sum_t (prod_(r <= t) a_r) ds_t C_t     (walked on from its start:
//        W *= a, then Q += W ds C)
//   PF, PQ = the W each walk ends with: the product of all the chunk's decays
//        when it walked the whole chunk; below 2^-40 when it stopped early,
//        where the terms left out and the product are below 2^-40 of what
//        the carry keeps.
template <typename T, int N, bool HAS_Z, bool SOFTPLUS, bool ZOH, typename GT>
__global__ void __launch_bounds__(kAggThreads) scan_bwd_chunk_agg_kernel(BwdParams p) {
    constexpr int S = N < 4 ? N : 4, G = N / S;
    const int64_t rows = p.batch * p.dim;
    const int64_t i = (int64_t)blockIdx.x * kAggThreads + threadIdx.x;
    if (i >= rows * G) return;
    const int64_t row = i / G, b = row / p.dim, d = row % p.dim;
    const int n0 = (int)(i % G) * S;
    const int cz = (int)blockIdx.y;
    const int64_t L = p.L;
    const int64_t t_lo = (int64_t)cz * p.chunk_len;
    const int64_t t_hi = L - t_lo < p.chunk_len ? L : t_lo + p.chunk_len;
    float A2[S], IA[S];
#pragma unroll
    for (int j = 0; j < S; j++) {
        const float av = p.A[d * N + n0 + j];
        A2[j] = av * kLog2e;
        IA[j] = (ZOH && av != 0.0f) ? 1.0f / av : 0.0f;
    }
    const float bias = p.bias ? p.bias[d] : 0.0f;
    const T* u = static_cast<const T*>(p.u) + row * L;
    const T* dl = static_cast<const T*>(p.delta) + row * L;
    const T* z = HAS_Z ? static_cast<const T*>(p.z) + row * L : nullptr;
    const GT* dy = static_cast<const GT*>(p.dy) + row * L;
    const T* Bm = static_cast<const T*>(p.B) + b * L * N + n0;
    const T* Cm = static_cast<const T*>(p.C) + b * L * N + n0;
    auto delta_at = [&](int64_t t) {
        const float v = io<T>::to_f32(dl[t]) + bias;
        return SOFTPLUS ? softplus(v) : v;
    };
    auto decay = [&](float dt, int j, float& e) {
        e = dt * A2[j];
        return ex2(e);
    };
    auto below_cut = [&](const float (&W)[S]) {
        bool all = true;
#pragma unroll
        for (int j = 0; j < S; j++) all = all && W[j] < kWalkCut;   // NaN keeps walking
        return all;
    };

    // forward map: back from the chunk's end
    float Fv[S], W[S];
#pragma unroll
    for (int j = 0; j < S; j++) { Fv[j] = 0.0f; W[j] = 1.0f; }
    for (int64_t tb = t_hi - 1; tb >= t_lo; tb -= kWalkBlock) {
        float dtv[kWalkBlock], xv[kWalkBlock], Bv[kWalkBlock][S];
#pragma unroll
        for (int k = 0; k < kWalkBlock; k++) {
            const int64_t t = tb - k;
            const bool ok = t >= t_lo;
            dtv[k] = ok ? delta_at(t) : 0.0f;
            xv[k] = ok ? io<T>::to_f32(u[t]) : 0.0f;
#pragma unroll
            for (int j = 0; j < S; j++) Bv[k][j] = ok ? io<T>::to_f32(Bm[t * N + j]) : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kWalkBlock; k++) {
#pragma unroll
            for (int j = 0; j < S; j++) {
                float e;
                const float a = decay(dtv[k], j, e);
                float wgt = dtv[k];
                if constexpr (ZOH)
                    wgt = zoh_weight(f2(a), f2(e), f2(dtv[k]), f2(IA[j])).x;
                Fv[j] = fmaf(W[j], wgt * Bv[k][j] * xv[k], Fv[j]);
                W[j] *= a;
            }
        }
        if (below_cut(W)) break;
    }
    const int64_t o = ((int64_t)cz * rows + row) * N + n0;
    float* F = p.agg;
    float* PF = F + (int64_t)p.nchunks * rows * N;
    float* Q = PF + (int64_t)p.nchunks * rows * N;
    float* PQ = Q + (int64_t)p.nchunks * rows * N;
#pragma unroll
    for (int j = 0; j < S; j++) { F[o + j] = Fv[j]; PF[o + j] = W[j]; }

    // adjoint map: on from the chunk's start
    float Qv[S];
#pragma unroll
    for (int j = 0; j < S; j++) { Qv[j] = 0.0f; W[j] = 1.0f; }
    for (int64_t tb = t_lo; tb < t_hi; tb += kWalkBlock) {
        float dtv[kWalkBlock], dsv[kWalkBlock], Cv[kWalkBlock][S];
#pragma unroll
        for (int k = 0; k < kWalkBlock; k++) {
            const int64_t t = tb + k;
            const bool ok = t < t_hi;
            dtv[k] = ok ? delta_at(t) : 0.0f;
            float ds = ok ? io<GT>::to_f32(dy[t]) : 0.0f;
            if (HAS_Z && ok) {
                const float zv = io<T>::to_f32(z[t]);
                ds = ds * zv * sigmoid(zv);
            }
            dsv[k] = ds;
#pragma unroll
            for (int j = 0; j < S; j++) Cv[k][j] = ok ? io<T>::to_f32(Cm[t * N + j]) : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kWalkBlock; k++) {
#pragma unroll
            for (int j = 0; j < S; j++) {
                float e;
                W[j] *= decay(dtv[k], j, e);
                Qv[j] = fmaf(W[j], dsv[k] * Cv[k][j], Qv[j]);
            }
        }
        if (below_cut(W)) break;
    }
#pragma unroll
    for (int j = 0; j < S; j++) { Q[o + j] = Qv[j]; PQ[o + j] = W[j]; }
}

// Chunked backward, step 2.  Thread: one (channel, state).  The state before
// every chunk, H[z + 1] = F[z] + PF[z] H[z] from H[0] = h0 (0 if none), and
// the adjoint flowing into every chunk from the ones after it,
// X[z - 1] = Q[z] + PQ[z] X[z] from X[nchunks - 1] = dlast (0 if none).
// H[0] and X[nchunks - 1] are not stored (the kernel reads h0, dlast).
template <int N>
__global__ void __launch_bounds__(kAggThreads) scan_bwd_chunk_carry_kernel(BwdParams p) {
    const int64_t cells = p.batch * p.dim * N;
    const int64_t i = (int64_t)blockIdx.x * kAggThreads + threadIdx.x;
    if (i >= cells) return;
    const int nc = p.nchunks;
    const float* F = p.agg;
    const float* PF = F + (int64_t)nc * cells;
    const float* Q = PF + (int64_t)nc * cells;
    const float* PQ = Q + (int64_t)nc * cells;
    float h = p.h0 ? p.h0[i] : 0.0f;
    for (int c = 0; c + 1 < nc; c++) {
        h = fmaf(PF[c * cells + i], h, F[c * cells + i]);
        p.hc[(c + 1) * cells + i] = h;
    }
    float x = p.dlast ? p.dlast[i] : 0.0f;
    for (int c = nc - 1; c > 0; c--) {
        x = fmaf(PQ[c * cells + i], x, Q[c * cells + i]);
        p.xc[(c - 1) * cells + i] = x;
    }
}

}  // namespace bwd
}  // namespace ssm
