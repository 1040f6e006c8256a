// Backward selective scan (gradients for training), with recomputation.
//
// The forward pass keeps no state for the backward pass; the backward pass
// recomputes the forward states on chip instead of reading an expanded state
// from memory ("State Spaces, Selectively - Mamba", papermap, "The
// hardware-aware scan").  Per channel, G = N / S adjacent lanes of a warp
// hold S states each (S = min(N, 4)); the sums over a channel's states
// (the output s_t, dDelta_t, dx_t) are warp shuffles within the G lanes:
//
//   pass 1  the forward recurrence over the whole sequence, writing only the
//           state at the start of every 8-token tile to the workspace
//           (batch x dim x ceil(L/8) x N fp32 checkpoints);
//   (each 8-token tile's inputs are staged in shared memory by the whole CTA
//   with coalesced loads, Delta computed once per element; the loads of the
//   next tile are issued into registers while the current tile computes)
//   pass 2  the tiles in reverse order: the tile's states are recomputed
//           from its checkpoint into shared memory, then the adjoint
//           recurrence runs backwards through the tile:
//             ds_t = dy_t silu(z_t), dz_t = dy_t s_t silu'(z_t)
//             g_n += ds_t C_tn                       (adjoint of h_tn)
//             dDelta_t = sum_n g_n (A_n a_tn h_(t-1)n + B_tn x_t)
//             dx_t = ds_t D + sum_n g_n Delta_t B_tn
//             dA_n += g_n Delta_t a_tn h_(t-1)n,     g_n *= a_tn
//           with dB_tn = g_n Delta_t x_t and dC_tn = ds_t h_tn summed over
//           the CTA's channels at the end of the tile (from the tile's
//           states and adjoints kept in shared memory) and added to the
//           batch row's dB, dC with one atomic per (t, n) per CTA.
//   dA, dD and delta_bias's gradient are summed per thread over the
//   sequence and added per CTA with atomics; gradients are fp32.
#pragma once

#include "common.cuh"

namespace ssm {
namespace bwd {

constexpr int kThreads = 64;    // threads per CTA (more, smaller CTAs: more warps per SM)
constexpr int kTT = 8;          // tokens per tile

struct BwdParams {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;      // may be null
    const void* z;       // may be null
    const float* bias;   // may be null
    const float* dy;     // (batch, dim, L) fp32
    const float* dlast;  // (batch, dim, N) fp32, may be null
    float* du;           // (batch, dim, L)
    float* ddelta;       // (batch, dim, L)
    float* dz;           // (batch, dim, L), null when z is null
    float* dA;           // (dim, N), accumulated: zeroed by the host
    float* dB;           // (batch, L, N), accumulated
    float* dC;           // (batch, L, N), accumulated
    float* dD;           // (dim), accumulated, may be null when D is null
    float* dbias;        // (dim), accumulated, may be null
    float* dh0;          // (batch, dim, N), may be null
    float* ckpt;         // workspace: (batch, dim, ntiles, N)
    int64_t batch, dim, L, ntiles;
};

template <int N> struct BwdShape {
    static constexpr int S = N < 4 ? N : 4;    // states per thread
    static constexpr int G = N / S;            // threads per channel
    static constexpr int CH = kThreads / G;    // channels per CTA
    // [kTT + 1][kThreads][S]: row 0 the state before the tile, then the
    // tile's states; the adjoints used for dB in rows 0 .. kTT-1 of a second
    // such array; then ds_t and Delta_t x_t per channel and token
    static constexpr int TILE = (kTT + 1) * kThreads * S * 4;
    static constexpr int OFF_G = TILE;
    static constexpr int OFF_DS = 2 * TILE;
    static constexpr int OFF_DX = OFF_DS + kTT * CH * 4;
    // the tile's inputs, staged with coalesced loads: per channel a row of
    // kTT + 1 floats (x = u, Delta, v = delta + bias, z, dy), and B, C rows
    static constexpr int ROW = kTT + 1;
    static constexpr int OFF_IN = OFF_DX + kTT * CH * 4;
    static constexpr int IN_PLANE = CH * ROW * 4;
    static constexpr int OFF_BC = OFF_IN + 5 * IN_PLANE;
    static constexpr int SMEM = OFF_BC + 2 * kTT * N * 4;
};

__device__ __forceinline__ float sigmoid(float v) { return rcp(1.0f + ex2(-v * kLog2e)); }

// sum over the G lanes of a channel (adjacent, G a power of two)
template <int G>
__device__ __forceinline__ float chan_sum(float v) {
#pragma unroll
    for (int off = 1; off < G; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <typename T, int N, bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(kThreads) scan_bwd_kernel(BwdParams p) {
    using Sh = BwdShape<N>;
    constexpr int S = Sh::S, G = Sh::G, CH = Sh::CH;
    extern __shared__ __align__(16) unsigned char smem[];
    float* Hs = reinterpret_cast<float*>(smem);
    float* Gs = reinterpret_cast<float*>(smem + Sh::OFF_G);
    float* DS = reinterpret_cast<float*>(smem + Sh::OFF_DS);     // [kTT][CH]
    float* DX = reinterpret_cast<float*>(smem + Sh::OFF_DX);     // [kTT][CH]
    float* XU = reinterpret_cast<float*>(smem + Sh::OFF_IN);                    // [CH][ROW] x
    float* DT = reinterpret_cast<float*>(smem + Sh::OFF_IN + Sh::IN_PLANE);     // Delta
    float* VV = reinterpret_cast<float*>(smem + Sh::OFF_IN + 2 * Sh::IN_PLANE); // delta + bias
    float* ZZ = reinterpret_cast<float*>(smem + Sh::OFF_IN + 3 * Sh::IN_PLANE); // z
    float* DY = reinterpret_cast<float*>(smem + Sh::OFF_IN + 4 * Sh::IN_PLANE); // dy
    float* BB = reinterpret_cast<float*>(smem + Sh::OFF_BC);                    // [kTT][N]
    float* CC = BB + kTT * N;
    constexpr int ROW = Sh::ROW;

    const int tid = threadIdx.x;
    const int lc = tid / G, gi = tid % G;          // channel within the CTA, state slice
    const int n0 = gi * S;
    const int64_t b = blockIdx.y;
    const int64_t d = (int64_t)blockIdx.x * CH + lc;
    const bool active = d < p.dim;
    const int64_t dd = active ? d : 0;
    const int64_t c = b * p.dim + dd;     // flat channel
    const int64_t L = p.L;
    float* ck = p.ckpt + c * p.ntiles * N + n0;

    float A[S], A2[S];
#pragma unroll
    for (int n = 0; n < S; n++) {
        A[n] = active ? p.A[dd * N + n0 + n] : 0.0f;
        A2[n] = A[n] * kLog2e;
    }
    const float Dv = (active && p.D) ? p.D[dd] : 0.0f;
    // stage tokens [t0, t0 + nt) of the CTA's channels: consecutive threads
    // take consecutive tokens of a row; `full` also stages z, dy and C
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const T* bu = static_cast<const T*>(p.u);
    const T* bdl = static_cast<const T*>(p.delta);
    const T* bz = static_cast<const T*>(p.z);
    const T* bB = static_cast<const T*>(p.B) + b * L * N;
    const T* bC = static_cast<const T*>(p.C) + b * L * N;
    // A tile's inputs are fetched into registers (`fetch`, global loads in
    // flight while the previous tile computes) and written to shared memory
    // later (`put`).
    constexpr int E = (CH * kTT + kThreads - 1) / kThreads;   // elements per thread
    constexpr int EB = (kTT * N + kThreads - 1) / kThreads;
    float rx[E], rv[E], rz[E], rd[E], rb[EB], rc[EB];
    auto fetch = [&](int64_t t0, int nt, bool full) {
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = tid + e * kThreads;
            const int cl = i / kTT, j = i % kTT;
            const bool ok = i < CH * kTT && d0 + cl < p.dim && j < nt;
            const int64_t gi2 = ((b * p.dim + d0 + cl) * L + t0 + j);
            rx[e] = ok ? io<T>::load(bu, gi2) : 0.0f;
            rv[e] = ok ? io<T>::load(bdl, gi2) + ((p.bias) ? p.bias[d0 + cl] : 0.0f) : 0.0f;
            rz[e] = (full && ok && HAS_Z) ? io<T>::load(bz, gi2) : 0.0f;
            rd[e] = (full && ok) ? p.dy[gi2] : 0.0f;
        }
#pragma unroll
        for (int e = 0; e < EB; e++) {
            const int i = tid + e * kThreads;
            const bool ok = i < kTT * N && i / N < nt;
            rb[e] = ok ? io<T>::load(bB, t0 * N + i) : 0.0f;
            rc[e] = (full && ok) ? io<T>::load(bC, t0 * N + i) : 0.0f;
        }
    };
    auto put = [&](int nt, bool full) {
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = tid + e * kThreads;
            if (i < CH * kTT) {
                const int cl = i / kTT, j = i % kTT;
                const bool ok = d0 + cl < p.dim && j < nt;
                XU[cl * ROW + j] = rx[e];
                VV[cl * ROW + j] = rv[e];
                DT[cl * ROW + j] = ok ? (SOFTPLUS ? softplus(rv[e]) : rv[e]) : 0.0f;
                if (full) {
                    ZZ[cl * ROW + j] = rz[e];
                    DY[cl * ROW + j] = rd[e];
                }
            }
        }
#pragma unroll
        for (int e = 0; e < EB; e++) {
            const int i = tid + e * kThreads;
            if (i < kTT * N) {
                BB[i] = rb[e];
                if (full) CC[i] = rc[e];
            }
        }
    };

    // ---- pass 1: forward, checkpoint every tile ----
    float h[S];
#pragma unroll
    for (int n = 0; n < S; n++) h[n] = 0.0f;
    if (p.ntiles > 0) fetch(0, (int)(L < kTT ? L : kTT), false);
    for (int64_t k = 0; k < p.ntiles; k++) {
        const int64_t t0 = k * kTT;
        const int nt = (int)(L - t0 < kTT ? L - t0 : kTT);
        if (active) {
#pragma unroll
            for (int n = 0; n < S; n++) ck[k * N + n] = h[n];
        }
        put(nt, false);
        __syncthreads();
        if (k + 1 < p.ntiles) {
            const int64_t t1 = t0 + kTT;
            fetch(t1, (int)(L - t1 < kTT ? L - t1 : kTT), false);
        }
        for (int j = 0; j < nt; j++) {
            const float dt = DT[lc * ROW + j];
            const float dtx = dt * XU[lc * ROW + j];
#pragma unroll
            for (int n = 0; n < S; n++) h[n] = fmaf(ex2(dt * A2[n]), h[n], dtx * BB[j * N + n0 + n]);
        }
        __syncthreads();
    }

    // ---- pass 2: tiles in reverse ----
    float g[S], dA[S];
#pragma unroll
    for (int n = 0; n < S; n++) {
        g[n] = (active && p.dlast) ? p.dlast[c * N + n0 + n] : 0.0f;
        dA[n] = 0.0f;
    }
    float dD = 0.0f, dbias = 0.0f;
    if (p.ntiles > 0) {
        const int64_t tl = (p.ntiles - 1) * kTT;
        fetch(tl, (int)(L - tl < kTT ? L - tl : kTT), true);
    }
    for (int64_t k = p.ntiles - 1; k >= 0; k--) {
        const int64_t t0 = k * kTT;
        const int nt = (int)(L - t0 < kTT ? L - t0 : kTT);
        put(nt, true);
        // recompute the tile's states (row 0: the state before the tile)
#pragma unroll
        for (int n = 0; n < S; n++) Hs[tid * S + n] = h[n] = active ? ck[k * N + n] : 0.0f;
        __syncthreads();
        if (k > 0) fetch(t0 - kTT, kTT, true);   // the next tile back, in flight during this one
        for (int j = 0; j < nt; j++) {
            const float dt = DT[lc * ROW + j];
            const float dtx = dt * XU[lc * ROW + j];
            float* hs = Hs + ((j + 1) * kThreads + tid) * S;
#pragma unroll
            for (int n = 0; n < S; n++) {
                h[n] = fmaf(ex2(dt * A2[n]), h[n], dtx * BB[j * N + n0 + n]);
                hs[n] = h[n];
            }
        }
        // adjoint recurrence, backwards through the tile
        for (int j = nt - 1; j >= 0; j--) {
            const int64_t t = t0 + j;
            const float v = VV[lc * ROW + j];
            const float dt = DT[lc * ROW + j];
            const float x = XU[lc * ROW + j];
            const float* ht = Hs + ((j + 1) * kThreads + tid) * S;
            const float* hp = Hs + (j * kThreads + tid) * S;
            float Cv[S], Bv[S];
            float sp = 0.0f;
#pragma unroll
            for (int n = 0; n < S; n++) {
                Cv[n] = CC[j * N + n0 + n];
                Bv[n] = BB[j * N + n0 + n];
                sp = fmaf(Cv[n], ht[n], sp);
            }
            const float s = fmaf(Dv, x, chan_sum<G>(sp));
            const float dyv = DY[lc * ROW + j];
            float ds = dyv;
            if constexpr (HAS_Z) {
                const float zv = ZZ[lc * ROW + j];
                const float sg = sigmoid(zv);
                ds = dyv * zv * sg;
                if (active && gi == 0) p.dz[c * L + t] = dyv * s * sg * fmaf(zv, 1.0f - sg, 1.0f);
            }
            float dxp = 0.0f, ddtp = 0.0f;
            float* gs = Gs + (j * kThreads + tid) * S;
#pragma unroll
            for (int n = 0; n < S; n++) {
                const float a = ex2(dt * A2[n]);
                g[n] = fmaf(ds, Cv[n], g[n]);
                gs[n] = g[n];
                const float gah = g[n] * a * hp[n];
                ddtp = fmaf(A[n], gah, fmaf(g[n], Bv[n] * x, ddtp));
                dxp = fmaf(g[n] * dt, Bv[n], dxp);
                dA[n] = fmaf(dt, gah, dA[n]);
                g[n] *= a;
            }
            const float ddt = chan_sum<G>(ddtp);
            const float dx = fmaf(ds, Dv, chan_sum<G>(dxp));
            const float dv = SOFTPLUS ? ddt * sigmoid(v) : ddt;
            if (gi == 0) {
                DS[j * CH + lc] = ds;
                DX[j * CH + lc] = dt * x;
                dD = fmaf(ds, x, dD);
                dbias += dv;
                if (active) {
                    p.du[c * L + t] = dx;
                    p.ddelta[c * L + t] = dv;
                }
            }
        }
        __syncthreads();
        // dB_tn = sum_c g_n Delta_t x_t, dC_tn = sum_c ds_t h_tn over the CTA's channels
        for (int o = tid; o < nt * N; o += kThreads) {
            const int j = o / N, n = o % N;
            const int gn = n / S, sn = n % S;
            float sb = 0.0f, sc = 0.0f;
            for (int cc = 0; cc < CH; cc++) {
                const int th = cc * G + gn;
                sb = fmaf(Gs[(j * kThreads + th) * S + sn], DX[j * CH + cc], sb);
                sc = fmaf(DS[j * CH + cc], Hs[((j + 1) * kThreads + th) * S + sn], sc);
            }
            atomicAdd(p.dB + (b * L + t0 + j) * N + n, sb);
            atomicAdd(p.dC + (b * L + t0 + j) * N + n, sc);
        }
        __syncthreads();
    }
    if (active) {
#pragma unroll
        for (int n = 0; n < S; n++) atomicAdd(p.dA + dd * N + n0 + n, dA[n]);
        if (gi == 0) {
            if (p.dD) atomicAdd(p.dD + dd, dD);
            if (p.dbias) atomicAdd(p.dbias + dd, dbias);
        }
        if (p.dh0)
#pragma unroll
            for (int n = 0; n < S; n++) p.dh0[c * N + n0 + n] = g[n];
    }
}

}  // namespace bwd
}  // namespace ssm
