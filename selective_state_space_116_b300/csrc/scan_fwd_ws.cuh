// Forward selective scan, warp-specialised state-split kernel (bf16 I/O,
// N = 16, L % 16 == 0).
//
// The arithmetic is the state-split scan of scan_fwd.cuh (8 states per
// thread, two threads per channel, B and C broadcast from shared memory), but
// the phases that kernel runs one after the other between CTA barriers run
// here concurrently in separate warps, handing 16-token blocks to one another
// through mbarrier rings (one arrival per warp, bounded waits):
//
//   warp 16       producer: one thread issues the TMA copies of the block's
//                 u, delta, z (16-token x 128-channel boxes, 32-byte swizzle)
//                 and the bulk copies of its B and C rows
//   warps 8-11    prologue, thread c for channel c: Delta = softplus(delta +
//                 bias) and Delta u for the 16 tokens, and the B, C rows
//                 staged as fp32 in the layout the recurrence reads
//   warps 0-7     recurrence: warp w serves channels 32 (w % 4) .. + 31 and
//                 states 8 (w / 4) .. + 7; per token one 2^x per state, the
//                 state update and the partial C.h
//   warps 12-15   epilogue, thread c for channel c: the two partial sums,
//                 D u, silu(z), bf16 store
// Each SM sub-partition (warp % 4) gets the same mix: two recurrence warps,
// one prologue and one epilogue warp.
//
// The CTA's work is a contiguous range of (channel group, block) units in the
// balanced persistent order of the state-split kernel (head of its last group
// first, its first group's continuation last, carries handed over through
// the workspace).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "scan_fwd.cuh"
#include "scan_fwd_tc.cuh"

namespace ssm {
namespace ws {

using tc::bulk_load;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::raw_off;
using tc::role_sync;
using tc::smem_u32;
using tc::tma_load_3d;
using tc::TmaMaps;

constexpr int kRecWarps = 8;
constexpr int kWarpPro = 8, kWarpEpi = 12, kWarpProd = 16;
constexpr int kThreads = 17 * 32;
constexpr int kCH = 128;        // channels per group
constexpr int kN = 16;          // states
constexpr int kS = 8;           // states per recurrence thread
constexpr int kTB = 16;         // tokens per block (= TMA box)
constexpr int kRawSlots = 5;
constexpr int kOpSlots = 4;
constexpr int kYSlots = 3;
static_assert(tc::kTT == kTB && tc::kCH == kCH, "the TMA boxes of the tensor-core kernel are reused");

// Raw block: u, delta, z planes (128 rows x 32 bytes, 32-byte swizzle), then
// the B and C rows of the 16 tokens.
constexpr int kPlaneBytes = kCH * kTB * 2;
constexpr int kRawBC = kTB * kN * 2;
constexpr int kOffTileB = 3 * kPlaneBytes, kOffTileC = kOffTileB + kRawBC;
constexpr int kTileBytes = (kOffTileC + kRawBC + 1023) / 1024 * 1024;
// Operand slot: (Delta, Delta u) per channel and token, rows padded to 144
// bytes; then B and C in fp32 as [token][state group][B 8 | C 8].
constexpr int kWRow = kTB * 8 + 16;
constexpr int kOffBC = kCH * kWRow;
constexpr int kSlotBytes = kOffBC + kTB * 2 * 2 * kS * 4;
// Partial outputs: [state group][channel] rows of 16 fp32, padded to 80 bytes.
constexpr int kYRow = kTB * 4 + 16;
constexpr int kYBytes = 2 * kCH * kYRow;
constexpr int kOffY = kOpSlots * kSlotBytes;
constexpr int kOffRaw = (kOffY + kYSlots * kYBytes + 1023) / 1024 * 1024;
constexpr int kSmemUsed = kOffRaw + kRawSlots * kTileBytes;
constexpr int kSmem = kSmemUsed + 1024;   // room to align the base to 1 KB
static_assert(kSmem <= 226 * 1024, "shared memory");
static_assert(kSlotBytes % 16 == 0 && kYBytes % 16 == 0 && kTileBytes % 1024 == 0, "alignment");

struct Bars {
    uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];
    uint64_t op_full[kOpSlots], op_empty[kOpSlots];
    uint64_t yp_full[kYSlots], yp_empty[kYSlots];
    int failed;   // a bounded wait of this CTA gave up
    int ok;       // the carry hand-over arrived
};

// The CTA's (group, block) range and the walk over it, as in scan_fwd_tc.cuh
// but with 16-token blocks.
struct Parts {
    int64_t s, e, nblk, g_first, g_last;
    __device__ explicit Parts(const ScanParams& p) {
        nblk = p.L / kTB;
        const int64_t W = p.ngroups * nblk;
        s = W * blockIdx.x / gridDim.x;
        e = W * (blockIdx.x + 1) / gridDim.x;
        g_first = s / nblk;
        g_last = s < e ? (e - 1) / nblk : g_first - 1;
    }
    __device__ void range(int64_t grp, int64_t& b0, int64_t& b1) const {
        const int64_t lo = grp * nblk;
        b0 = (s > lo ? s : lo) - lo;
        b1 = (e < lo + nblk ? e : lo + nblk) - lo;
    }
};

struct Cursor {
    int64_t grp, b0, b1, kb, i, b, d0;
    __device__ Cursor(const Parts& pt, const ScanParams& p) : grp(pt.g_last), i(0) { enter(pt, p); }
    __device__ void enter(const Parts& pt, const ScanParams& p) {
        if (grp >= pt.g_first) {
            pt.range(grp, b0, b1);
            b = grp / p.groups_per_row;
            d0 = (grp - b * p.groups_per_row) * kCH;
        } else {
            b0 = b1 = 0;
        }
        kb = b0;
    }
    __device__ bool valid(const Parts& pt) const { return grp >= pt.g_first; }
    __device__ void next(const Parts& pt, const ScanParams& p) {
        i++;
        if (++kb == b1) {
            --grp;
            enter(pt, p);
        }
    }
};

__device__ __forceinline__ bool wait_or_fail(uint64_t* m, uint32_t parity, Bars& br,
                                             const ScanParams& p) {
    if (mbar_wait(m, parity, &br.failed)) return true;
    atomicExch(p.status, kStatusTimeout);
    return false;
}
__device__ __forceinline__ uint32_t full_parity(int64_t k) { return (uint32_t)(k & 1); }
__device__ __forceinline__ uint32_t empty_parity(int64_t k) { return (uint32_t)((k + 1) & 1); }

template <bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(kThreads, 1)
    scan_fwd_ws_kernel(ScanParams p, const __grid_constant__ TmaMaps maps) {
    using bf16 = __nv_bfloat16;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars br;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        br.failed = 0;
        for (int i = 0; i < kRawSlots; i++) {
            mbar_init(&br.raw_full[i], 1);    // the producer's expect_tx
            mbar_init(&br.raw_empty[i], 8);   // 4 prologue + 4 epilogue warps
        }
        for (int i = 0; i < kOpSlots; i++) {
            mbar_init(&br.op_full[i], 4);             // prologue warps
            mbar_init(&br.op_empty[i], kRecWarps);
        }
        for (int i = 0; i < kYSlots; i++) {
            mbar_init(&br.yp_full[i], kRecWarps);
            mbar_init(&br.yp_empty[i], 4);            // epilogue warps
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const Parts parts(p);
    const int64_t L = p.L;

    if (warp < kRecWarps) {
        // ---------------- recurrence ----------------
        const int g = warp >> 2, c = (warp & 3) * 32 + lane;
        int64_t i = 0;
        for (int64_t grp = parts.g_last; grp >= parts.g_first; grp--) {
            int64_t b0, b1;
            parts.range(grp, b0, b1);
            const int64_t b = grp / p.groups_per_row;
            const int64_t d0 = (grp - b * p.groups_per_row) * kCH;
            const int64_t row0 = b * p.dim + d0;
            const bool active = d0 + c < p.dim;
            float A2[kS], h[kS];
#pragma unroll
            for (int j = 0; j < kS; j++)   // exp(Delta A) = 2^(Delta A log2 e)
                A2[j] = active ? p.A[(d0 + c) * kN + g * kS + j] * kLog2e : 0.0f;
            if (b0 == 0) {
#pragma unroll
                for (int j = 0; j < kS; j++) h[j] = 0.0f;
            } else {
                if (tid == 0) {
                    const bool ok = ssm::seq::wait_flag(p.flags + grp);
                    if (!ok) atomicExch(p.status, kStatusTimeout);
                    __threadfence();
                    br.ok = ok;
                }
                role_sync(1, 32 * kRecWarps);
                const bool ok = br.ok;
                const float* src = p.carry + (grp * kCH + c) * kN + g * kS;
#pragma unroll
                for (int j = 0; j < kS; j++) h[j] = ok ? __ldcg(src + j) : __int_as_float(0x7fc00000);
            }
            for (int64_t kb = b0; kb < b1; kb++, i++) {
                const int o = (int)(i % kOpSlots), ys = (int)(i % kYSlots);
                wait_or_fail(&br.op_full[o], full_parity(i / kOpSlots), br, p);
                if (i >= kYSlots) wait_or_fail(&br.yp_empty[ys], empty_parity(i / kYSlots), br, p);
                const unsigned char* sl = smem + o * kSlotBytes;
                const float4* wrow = reinterpret_cast<const float4*>(sl + c * kWRow);
                const float* bcf = reinterpret_cast<const float*>(sl + kOffBC) + g * 2 * kS;
                float* yrow = reinterpret_cast<float*>(smem + kOffY + ys * kYBytes + (g * kCH + c) * kYRow);
                ssm::seq::scan_tokens<kS, 2 * 2 * kS, kTB>(wrow, bcf, h, A2, yrow);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&br.op_empty[o]);
                    mbar_arrive(&br.yp_full[ys]);
                }
            }
            // the part's final state
            if (b1 * kTB == L) {
                if (active && p.last_state) {
                    float* dst = p.last_state + (row0 + c) * kN + g * kS;
#pragma unroll
                    for (int j = 0; j < kS; j++) dst[j] = h[j];
                }
            } else if (b1 > b0) {
                float* dst = p.carry + (grp * kCH + c) * kN + g * kS;
#pragma unroll
                for (int j = 0; j < kS; j++) __stcg(dst + j, h[j]);
                __threadfence();
                role_sync(1, 32 * kRecWarps);
                if (tid == 0)
                    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + grp), "r"(1u)
                                 : "memory");
            }
        }
    } else if (warp < kWarpEpi) {
        // ---------------- prologue ----------------
        const int c = tid - kWarpPro * 32;   // channel within the group
        float bias = 0.0f;
        int64_t bias_grp = -1;
        for (Cursor pc(parts, p); pc.valid(parts); pc.next(parts, p)) {
            const int64_t d0 = pc.d0;
            if (pc.grp != bias_grp) {
                bias_grp = pc.grp;
                bias = (d0 + c < p.dim && p.bias) ? p.bias[d0 + c] : 0.0f;
                if (SOFTPLUS) bias *= kLog2e;
            }
            const int rs = (int)(pc.i % kRawSlots), o = (int)(pc.i % kOpSlots);
            wait_or_fail(&br.raw_full[rs], full_parity(pc.i / kRawSlots), br, p);
            if (pc.i >= kOpSlots) wait_or_fail(&br.op_empty[o], empty_parity(pc.i / kOpSlots), br, p);
            const unsigned char* r = smem + kOffRaw + rs * kTileBytes;
            unsigned char* sl = smem + o * kSlotBytes;
            float4* wrow = reinterpret_cast<float4*>(sl + c * kWRow);
#pragma unroll
            for (int k = 0; k < 2; k++) {   // tokens 8k .. 8k + 7
                float uv[8], dv[8];
                ssm::seq::unpack8<bf16>(r + raw_off(c, k), uv);
                ssm::seq::unpack8<bf16>(r + kPlaneBytes + raw_off(c, k), dv);
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    float dt0, dt1;
                    if constexpr (SOFTPLUS) {
                        dt0 = ssm::seq::softplus_log2(fmaf(dv[t], kLog2e, bias));
                        dt1 = ssm::seq::softplus_log2(fmaf(dv[t + 1], kLog2e, bias));
                    } else {
                        dt0 = dv[t] + bias;
                        dt1 = dv[t + 1] + bias;
                    }
                    wrow[k * 4 + t / 2] = make_float4(dt0, dt0 * uv[t], dt1, dt1 * uv[t + 1]);
                }
            }
            {   // B and C of the block as fp32, [token][state group][B 8 | C 8]: 4 values a thread
                const int i0 = c * 4;
                const int which = i0 / (kTB * kN), e0 = i0 % (kTB * kN);
                const int t = e0 / kN, n = e0 % kN;
                const uint2 q = *reinterpret_cast<const uint2*>(r + kOffTileB + which * kRawBC + e0 * 2);
                const float4 v = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                                             __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
                float* bcf = reinterpret_cast<float*>(sl + kOffBC);
                *reinterpret_cast<float4*>(bcf + (t * 2 + n / kS) * 2 * kS + which * kS + n % kS) = v;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&br.op_full[o]);
                mbar_arrive(&br.raw_empty[rs]);
            }
        }
    } else if (warp < kWarpProd) {
        // ---------------- epilogue ----------------
        const int c = tid - kWarpEpi * 32;   // channel within the group
        for (Cursor ec(parts, p); ec.valid(parts); ec.next(parts, p)) {
            const int64_t b = ec.b, d0 = ec.d0;
            const int rs = (int)(ec.i % kRawSlots), ys = (int)(ec.i % kYSlots);
            wait_or_fail(&br.yp_full[ys], full_parity(ec.i / kYSlots), br, p);
            float y[kTB];
            {
                const float4* y0 = reinterpret_cast<const float4*>(smem + kOffY + ys * kYBytes + c * kYRow);
                const float4* y1 = reinterpret_cast<const float4*>(smem + kOffY + ys * kYBytes + (kCH + c) * kYRow);
#pragma unroll
                for (int j = 0; j < kTB / 4; j++) {
                    const float4 a = y0[j], bq = y1[j];
                    y[4 * j] = a.x + bq.x;
                    y[4 * j + 1] = a.y + bq.y;
                    y[4 * j + 2] = a.z + bq.z;
                    y[4 * j + 3] = a.w + bq.w;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&br.yp_empty[ys]);
            const unsigned char* r = smem + kOffRaw + rs * kTileBytes;
            const bool active = d0 + c < p.dim;
            const float Dv = (active && p.D) ? p.D[d0 + c] : 0.0f;
            uint4 ov[2];
#pragma unroll
            for (int hf = 0; hf < 2; hf++) {   // tokens 8 hf .. 8 hf + 7
                float uv[8];
                ssm::seq::unpack8<bf16>(r + raw_off(c, hf), uv);
                float yy[8];
#pragma unroll
                for (int t = 0; t < 8; t++) yy[t] = fmaf(Dv, uv[t], y[8 * hf + t]);
                if constexpr (HAS_Z) {
                    float zv[8];
                    ssm::seq::unpack8<bf16>(r + 2 * kPlaneBytes + raw_off(c, hf), zv);
#pragma unroll
                    for (int t = 0; t < 8; t++) yy[t] *= ssm::seq::gate<bf16>(zv[t]);
                }
                unsigned* o32 = reinterpret_cast<unsigned*>(&ov[hf]);
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(yy[2 * t], yy[2 * t + 1]);
                    o32[t] = *reinterpret_cast<const unsigned*>(&pr);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&br.raw_empty[rs]);
            if (active) {
                uint4* gy = reinterpret_cast<uint4*>(static_cast<bf16*>(p.y) + (b * p.dim + d0 + c) * L +
                                                     ec.kb * kTB);
                gy[0] = ov[0];
                gy[1] = ov[1];
            }
        }
    } else {
        // ---------------- producer: raw blocks (one thread) ----------------
        if (lane == 0) {
            int64_t T = 0;
            for (Cursor cu(parts, p); cu.valid(parts); cu.next(parts, p), T++) {
                const int slot = (int)(T % kRawSlots);
                if (T >= kRawSlots) wait_or_fail(&br.raw_empty[slot], empty_parity(T / kRawSlots), br, p);
                unsigned char* r = smem + kOffRaw + slot * kTileBytes;
                const int64_t t0 = cu.kb * kTB;
                const bf16* gB = static_cast<const bf16*>(p.B) + (cu.b * L + t0) * kN;
                const bf16* gC = static_cast<const bf16*>(p.C) + (cu.b * L + t0) * kN;
                mbar_expect_tx(&br.raw_full[slot], (HAS_Z ? 3 : 2) * kPlaneBytes + 2 * kRawBC);
                tma_load_3d(r, &maps.u, (int)t0, (int)cu.d0, (int)cu.b, &br.raw_full[slot]);
                tma_load_3d(r + kPlaneBytes, &maps.delta, (int)t0, (int)cu.d0, (int)cu.b, &br.raw_full[slot]);
                if (HAS_Z)
                    tma_load_3d(r + 2 * kPlaneBytes, &maps.z, (int)t0, (int)cu.d0, (int)cu.b, &br.raw_full[slot]);
                bulk_load(r + kOffTileB, gB, kRawBC, &br.raw_full[slot]);
                bulk_load(r + kOffTileC, gC, kRawBC, &br.raw_full[slot]);
            }
            // the shared memory is released when the CTA exits: let the last
            // copies land even if the pipeline gave up
            volatile int never = 0;
            for (int64_t k = T - kRawSlots < 0 ? 0 : T - kRawSlots; k < T; k++)
                mbar_wait(&br.raw_full[k % kRawSlots], full_parity(k / kRawSlots), &never);
        }
    }
    __syncthreads();
}

}  // namespace ws
}  // namespace ssm
