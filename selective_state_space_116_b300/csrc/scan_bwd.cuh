// Backward selective scan (gradients for training), with recomputation.
//
// The forward pass keeps no state for the backward pass; the backward pass
// recomputes the forward states on chip instead of reading an expanded state
// from memory ("State Spaces, Selectively - Mamba", papermap, "The
// hardware-aware scan").  Per channel (one thread, all N states in
// registers):
//
//   pass 1  the forward recurrence over the whole sequence, writing only the
//           state at the start of every 8-token tile to the workspace
//           (batch x dim x ceil(L/8) x N fp32 checkpoints);
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

constexpr int kCH = 64;    // channels (threads) per CTA
constexpr int kTT = 8;     // tokens per tile

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
    static constexpr int NP = N + 4;   // padded row of one channel's states
    // rows: the state before the tile, then the tile's kTT states
    static constexpr int TILE = (kTT + 1) * kCH * NP * 4;
    static constexpr int OFF_G = TILE;
    static constexpr int OFF_DS = 2 * TILE;
    static constexpr int OFF_DX = OFF_DS + kTT * kCH * 4;
    static constexpr int SMEM = OFF_DX + kTT * kCH * 4;
};

__device__ __forceinline__ float sigmoid(float v) { return rcp(1.0f + ex2(-v * kLog2e)); }

template <typename T, int N, bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(kCH) scan_bwd_kernel(BwdParams p) {
    using Sh = BwdShape<N>;
    extern __shared__ __align__(16) unsigned char smem[];
    float* Hs = reinterpret_cast<float*>(smem);                  // [kTT + 1][kCH][NP] h_(t0-1), h_t
    float* Gs = reinterpret_cast<float*>(smem + Sh::OFF_G);      // [kTT + 1][kCH][NP] g used for dB_t (rows 0..kTT-1)
    float* DS = reinterpret_cast<float*>(smem + Sh::OFF_DS);     // [kTT][kCH] ds_t
    float* DX = reinterpret_cast<float*>(smem + Sh::OFF_DX);     // [kTT][kCH] Delta_t x_t

    const int tid = threadIdx.x;
    const int64_t b = blockIdx.y;
    const int64_t d = (int64_t)blockIdx.x * kCH + tid;
    const bool active = d < p.dim;
    const int64_t dd = active ? d : 0;
    const int64_t c = b * p.dim + dd;     // flat channel
    const int64_t L = p.L;
    const T* gu = static_cast<const T*>(p.u) + c * L;
    const T* gdl = static_cast<const T*>(p.delta) + c * L;
    const T* gz = HAS_Z ? static_cast<const T*>(p.z) + c * L : nullptr;
    const T* gB = static_cast<const T*>(p.B) + b * L * N;
    const T* gC = static_cast<const T*>(p.C) + b * L * N;
    const float* gdy = p.dy + c * L;
    float* ck = p.ckpt + c * p.ntiles * N;

    float A[N], A2[N];
#pragma unroll
    for (int n = 0; n < N; n++) {
        A[n] = active ? p.A[dd * N + n] : 0.0f;
        A2[n] = A[n] * kLog2e;
    }
    const float bias = (active && p.bias) ? p.bias[dd] : 0.0f;
    const float Dv = (active && p.D) ? p.D[dd] : 0.0f;
    auto delta_of = [&](int64_t t, float& v) {
        v = io<T>::load(gdl, t) + bias;
        return SOFTPLUS ? softplus(v) : v;
    };

    // ---- pass 1: forward, checkpoint every tile ----
    float h[N];
#pragma unroll
    for (int n = 0; n < N; n++) h[n] = 0.0f;
    if (active) {
        for (int64_t t = 0; t < L; t++) {
            if (t % kTT == 0) {
#pragma unroll
                for (int n = 0; n < N; n++) ck[(t / kTT) * N + n] = h[n];
            }
            float v;
            const float dt = delta_of(t, v);
            const float dtx = dt * io<T>::load(gu, t);
#pragma unroll
            for (int n = 0; n < N; n++)
                h[n] = fmaf(ex2(dt * A2[n]), h[n], dtx * io<T>::load(gB, t * N + n));
        }
    }

    // ---- pass 2: tiles in reverse ----
    float g[N], dA[N];
#pragma unroll
    for (int n = 0; n < N; n++) {
        g[n] = (active && p.dlast) ? p.dlast[c * N + n] : 0.0f;
        dA[n] = 0.0f;
    }
    float dD = 0.0f, dbias = 0.0f;
    for (int64_t k = p.ntiles - 1; k >= 0; k--) {
        const int64_t t0 = k * kTT;
        const int nt = (int)(L - t0 < kTT ? L - t0 : kTT);
        // recompute the tile's states (row 0: the state before the tile)
        {
            float* hs = Hs + tid * Sh::NP;
#pragma unroll
            for (int n = 0; n < N; n++) hs[n] = h[n] = active ? ck[k * N + n] : 0.0f;
        }
        for (int j = 0; j < nt; j++) {
            float v;
            const float dt = active ? delta_of(t0 + j, v) : 0.0f;
            const float x = active ? io<T>::load(gu, t0 + j) : 0.0f;
            float* hs = Hs + ((j + 1) * kCH + tid) * Sh::NP;
#pragma unroll
            for (int n = 0; n < N; n++) {
                const float bv = active ? io<T>::load(gB, (t0 + j) * N + n) : 0.0f;
                h[n] = fmaf(ex2(dt * A2[n]), h[n], dt * x * bv);
                hs[n] = h[n];
            }
        }
        // adjoint recurrence, backwards through the tile
        for (int j = nt - 1; j >= 0; j--) {
            const int64_t t = t0 + j;
            float v = 0.0f;
            const float dt = active ? delta_of(t, v) : 0.0f;
            const float x = active ? io<T>::load(gu, t) : 0.0f;
            const float* ht = Hs + ((j + 1) * kCH + tid) * Sh::NP;
            const float* hp = Hs + (j * kCH + tid) * Sh::NP;
            float s = Dv * x;
            float Cv[N];
#pragma unroll
            for (int n = 0; n < N; n++) {
                Cv[n] = active ? io<T>::load(gC, t * N + n) : 0.0f;
                s = fmaf(Cv[n], ht[n], s);
            }
            const float dyv = active ? gdy[t] : 0.0f;
            float ds = dyv;
            if constexpr (HAS_Z) {
                const float zv = active ? io<T>::load(gz, t) : 0.0f;
                const float sg = sigmoid(zv);
                ds = dyv * zv * sg;
                if (active) p.dz[c * L + t] = dyv * s * sg * fmaf(zv, 1.0f - sg, 1.0f);
            }
            dD = fmaf(ds, x, dD);
            float dx = ds * Dv, ddt = 0.0f;
            float* gs = Gs + (j * kCH + tid) * Sh::NP;
#pragma unroll
            for (int n = 0; n < N; n++) {
                const float bv = active ? io<T>::load(gB, t * N + n) : 0.0f;
                const float a = ex2(dt * A2[n]);
                g[n] = fmaf(ds, Cv[n], g[n]);
                gs[n] = g[n];
                const float gah = g[n] * a * hp[n];
                ddt = fmaf(A[n], gah, fmaf(g[n], bv * x, ddt));
                dx = fmaf(g[n] * dt, bv, dx);
                dA[n] = fmaf(dt, gah, dA[n]);
                g[n] *= a;
            }
            DS[j * kCH + tid] = ds;
            DX[j * kCH + tid] = dt * x;
            const float dv = SOFTPLUS ? ddt * sigmoid(v) : ddt;
            dbias += dv;
            if (active) {
                p.du[c * L + t] = dx;
                p.ddelta[c * L + t] = dv;
            }
        }
        __syncthreads();
        // dB_tn = sum_c g_n Delta_t x_t, dC_tn = sum_c ds_t h_tn over the CTA's channels
        for (int o = tid; o < nt * N; o += kCH) {
            const int j = o / N, n = o % N;
            float sb = 0.0f, sc = 0.0f;
            for (int cc = 0; cc < kCH; cc++) {
                sb = fmaf(Gs[(j * kCH + cc) * Sh::NP + n], DX[j * kCH + cc], sb);
                sc = fmaf(DS[j * kCH + cc], Hs[((j + 1) * kCH + cc) * Sh::NP + n], sc);
            }
            atomicAdd(p.dB + (b * L + t0 + j) * N + n, sb);
            atomicAdd(p.dC + (b * L + t0 + j) * N + n, sc);
        }
        __syncthreads();
    }
    if (active) {
#pragma unroll
        for (int n = 0; n < N; n++) atomicAdd(p.dA + dd * N + n, dA[n]);
        if (p.dD) atomicAdd(p.dD + dd, dD);
        if (p.dbias) atomicAdd(p.dbias + dd, dbias);
        if (p.dh0)
#pragma unroll
            for (int n = 0; n < N; n++) p.dh0[c * N + n] = g[n];
    }
}

}  // namespace bwd
}  // namespace ssm
