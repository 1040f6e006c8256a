// Forward selective scan, channel-parallel kernel.
//
// Mapping: one thread owns one channel (b, d) and keeps all N state entries
// h[0..N) in registers for the whole sequence, so the expanded state
// (batch x dim x L x N) never leaves the SM.  A CTA owns kChannels channels
// of one batch row and walks the sequence in tiles of kTile tokens: the
// tile's u / delta / z rows and its B / C rows (shared by every channel of
// the batch row) are staged in shared memory with coalesced loads, each
// thread runs the recurrence over the tile, and y goes back through shared
// memory for coalesced stores.
#pragma once

#include "common.cuh"

namespace ssm {

struct ScanParams {
    const void* u;
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
};

namespace v1 {

constexpr int kChannels = 64;   // threads per CTA = channels per CTA
constexpr int kTile = 64;       // tokens per staged tile

template <typename T>
struct Layout {
    static constexpr int kRow = kTile + 16 / (int)sizeof(T);  // padded row, elements
    static constexpr int kRowBytes = kRow * (int)sizeof(T);
    static constexpr int kPlane = kChannels * kRowBytes;       // one (channel x token) plane
};

template <typename T, int N>
constexpr size_t smem_bytes(bool has_z) {
    return (size_t)(has_z ? 3 : 2) * Layout<T>::kPlane + 2u * kTile * N * sizeof(float);
}

// Copy a (kChannels x kTile) tile of a (batch, dim, L) tensor into a padded
// shared-memory plane; out-of-range rows and columns read as zero.
template <typename T, bool VEC>
__device__ __forceinline__ void load_plane(T* plane, const T* g, int64_t row0, int rows,
                                           int64_t L, int64_t t0) {
    if constexpr (VEC) {
        constexpr int kEpv = 16 / sizeof(T);            // elements per 16-byte vector
        constexpr int kVpr = kTile / kEpv;              // vectors per row
        for (int i = threadIdx.x; i < kChannels * kVpr; i += kChannels) {
            const int r = i / kVpr, c = i % kVpr;
            const int64_t t = t0 + (int64_t)c * kEpv;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < rows && t < L)   // L is a multiple of kEpv on this path
                v = *reinterpret_cast<const uint4*>(g + (row0 + r) * L + t);
            *reinterpret_cast<uint4*>(plane + r * Layout<T>::kRow + c * kEpv) = v;
        }
    } else {
        for (int i = threadIdx.x; i < kChannels * kTile; i += kChannels) {
            const int r = i / kTile, c = i % kTile;
            const int64_t t = t0 + c;
            T v = io<T>::from_f32(0.0f);
            if (r < rows && t < L) v = g[(row0 + r) * L + t];
            plane[r * Layout<T>::kRow + c] = v;
        }
    }
}

template <typename T, bool VEC>
__device__ __forceinline__ void store_plane(T* g, const T* plane, int64_t row0, int rows,
                                            int64_t L, int64_t t0) {
    if constexpr (VEC) {
        constexpr int kEpv = 16 / sizeof(T);
        constexpr int kVpr = kTile / kEpv;
        for (int i = threadIdx.x; i < kChannels * kVpr; i += kChannels) {
            const int r = i / kVpr, c = i % kVpr;
            const int64_t t = t0 + (int64_t)c * kEpv;
            if (r < rows && t < L)
                *reinterpret_cast<uint4*>(g + (row0 + r) * L + t) =
                    *reinterpret_cast<const uint4*>(plane + r * Layout<T>::kRow + c * kEpv);
        }
    } else {
        for (int i = threadIdx.x; i < kChannels * kTile; i += kChannels) {
            const int r = i / kTile, c = i % kTile;
            const int64_t t = t0 + c;
            if (r < rows && t < L) g[(row0 + r) * L + t] = plane[r * Layout<T>::kRow + c];
        }
    }
}

template <typename T, int N, bool HAS_Z, bool SOFTPLUS, bool VEC>
__global__ void __launch_bounds__(kChannels) scan_fwd_kernel(ScanParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    T* s_u = reinterpret_cast<T*>(smem);                        // u, then y in place
    T* s_dl = reinterpret_cast<T*>(smem + Layout<T>::kPlane);
    T* s_z = reinterpret_cast<T*>(smem + 2 * Layout<T>::kPlane);
    float* s_B = reinterpret_cast<float*>(smem + (HAS_Z ? 3 : 2) * Layout<T>::kPlane);
    float* s_C = s_B + kTile * N;

    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * kChannels;
    const int rows = (int)(p.dim - d0 < kChannels ? p.dim - d0 : kChannels);
    const int r = threadIdx.x;
    const int64_t d = d0 + r;
    const bool active = r < rows;
    const int64_t row0 = b * p.dim + d0;          // first (b, d) row of this CTA
    const int64_t L = p.L;

    // Per-channel constants.  A is pre-scaled by log2(e) so exp(Delta A) = 2^(Delta A').
    float A2[N];
#pragma unroll
    for (int n = 0; n < N; n++) A2[n] = active ? p.A[d * N + n] * kLog2e : 0.0f;
    const float Dv = (active && p.D) ? p.D[d] : 0.0f;
    const float bias = (active && p.bias) ? p.bias[d] : 0.0f;

    float h[N];
#pragma unroll
    for (int n = 0; n < N; n++) h[n] = 0.0f;

    const T* gu = static_cast<const T*>(p.u);
    const T* gdl = static_cast<const T*>(p.delta);
    const T* gz = static_cast<const T*>(p.z);
    const T* gB = static_cast<const T*>(p.B) + b * L * N;
    const T* gC = static_cast<const T*>(p.C) + b * L * N;
    T* gy = static_cast<T*>(p.y);

    for (int64_t t0 = 0; t0 < L; t0 += kTile) {
        const int tl = (int)(L - t0 < kTile ? L - t0 : kTile);
        load_plane<T, VEC>(s_u, gu, row0, rows, L, t0);
        load_plane<T, VEC>(s_dl, gdl, row0, rows, L, t0);
        if constexpr (HAS_Z) load_plane<T, VEC>(s_z, gz, row0, rows, L, t0);
        for (int i = threadIdx.x; i < kTile * N; i += kChannels) {
            const bool in = i < tl * N;
            s_B[i] = in ? io<T>::load(gB, t0 * N + i) : 0.0f;
            s_C[i] = in ? io<T>::load(gC, t0 * N + i) : 0.0f;
        }
        __syncthreads();

        T* my_u = s_u + r * Layout<T>::kRow;
        const T* my_dl = s_dl + r * Layout<T>::kRow;
        const T* my_z = s_z + r * Layout<T>::kRow;
        for (int t = 0; t < tl; t++) {
            const float x = io<T>::to_f32(my_u[t]);
            const float v = io<T>::to_f32(my_dl[t]) + bias;
            const float dt = SOFTPLUS ? softplus(v) : v;
            const float dtx = dt * x;
            const float* Bt = s_B + t * N;
            const float* Ct = s_C + t * N;
            float y0 = 0.0f, y1 = 0.0f;
            if constexpr (N == 1) {
                h[0] = fmaf(ex2(dt * A2[0]), h[0], dtx * Bt[0]);
                y0 = Ct[0] * h[0];
            } else {
                const float2 dt2 = make_float2(dt, dt);
                const float2 dtx2 = make_float2(dtx, dtx);
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int n = 0; n < N; n += 2) {
                    const float2 e = __fmul2_rn(dt2, make_float2(A2[n], A2[n + 1]));
                    const float2 a = make_float2(ex2(e.x), ex2(e.y));
                    const float2 bb = __fmul2_rn(dtx2, *reinterpret_cast<const float2*>(Bt + n));
                    const float2 hn = __ffma2_rn(a, make_float2(h[n], h[n + 1]), bb);
                    h[n] = hn.x;
                    h[n + 1] = hn.y;
                    acc = __ffma2_rn(*reinterpret_cast<const float2*>(Ct + n), hn, acc);
                }
                y0 = acc.x;
                y1 = acc.y;
            }
            float yv = fmaf(Dv, x, y0 + y1);
            if constexpr (HAS_Z) yv *= silu(io<T>::to_f32(my_z[t]));
            my_u[t] = io<T>::from_f32(yv);   // y overwrites u in place: same thread, same slot
        }
        __syncthreads();
        store_plane<T, VEC>(gy, s_u, row0, rows, L, t0);
        __syncthreads();
    }

    if (active && p.last_state) {
#pragma unroll
        for (int n = 0; n < N; n++) p.last_state[(row0 + r) * N + n] = h[n];
    }
}

}  // namespace v1
}  // namespace ssm
