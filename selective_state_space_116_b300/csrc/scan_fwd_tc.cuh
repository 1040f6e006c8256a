// Forward selective scan with the tensor cores distributing B and C (bf16
// I/O, N = 16).
//
// The state-split kernel in scan_fwd.cuh is bound by shared-memory
// bandwidth: every thread reads the token's B and C rows (64 bytes per thread
// per token), although all channels of a batch row share them.  Here the
// tensor cores read B and C once per CTA and hand every channel its values
// in tensor memory, where each thread reads its own lane:
//
//   input term   bb[c, (t, n)] = (Delta u)[c, t] * B[t, n]: over a block of 8
//                tokens this is the GEMM  A1 x Bexp^T  with A1[c, t] =
//                (Delta u)[c, t] and the block-diagonal Bexp[(t, n), t'] =
//                B[t, n] [t = t']  (M = 128 channels, N = 128, K = 8)
//   C broadcast  Cb[c, (t, n)] = C[t, n] for every channel c: the GEMM
//                ones x Cexp^T with ones[c, k] = [k = 0] and Cexp[(t, n), k]
//                = C[t, n] [k = 0]  (same shape)
//
// Both are kind::tf32 MMAs (B, C and 1 are exact in tf32; Delta u is rounded
// to tf32's 10-bit mantissa, a relative error of 2^-11 on the input term that
// the bf16 output then rounds at 2^-9).  The recurrence h = exp(Delta A) h +
// bb and the output sum y = sum_n C h + D u stay on the CUDA cores in fp32,
// with the state in registers.  The output contraction is not put on the
// tensor cores: per token it is a dot product of 16, and as an MMA it needs
// K = (tokens x states) against a block-diagonal C, i.e. 16 small MMAs per
// block, which cost more tensor-core time than the recurrence takes.
//
// Thread mapping: 256 threads, 8 warps.  Warp w serves tensor-memory lanes
// 32 (w % 4) .. + 31, i.e. channels 32 (w % 4) + lane of the CTA's 128, and
// state half g = w / 4 (states 8g .. 8g + 7).  Warps 0-3 also compute the
// prologue (Delta = softplus(delta + bias), Delta u) of the block three
// steps ahead; warps 4-7 place B and C on the block diagonals and finish the
// output (sum of the two halves, D u skip term, silu(z) gate, bf16 store) of
// the block just scanned.  One elected thread issues the MMAs.
//
// Pipeline, per step k (one block of 8 tokens):
//   recurrence(k)   tcgen05.ld bb, Cb -> registers; partial C.h -> smem
//   the MMA thread waits for the commit of step k-1 (the MMAs of block k+1)
//   barrier
//   MMAs of block k+2 -> tensor-memory buffer (k+2) % 2; commit
//   prologue(k+3) | B/C diagonals(k+3) and output(k)
//   cp.async of the raw u, delta, z, B, C of block k+6
// Rings: 2 x 256 tensor-memory columns, 4 operand slots, 2 partial-sum
// buffers, 8 raw blocks.  Every wait is bounded.
#pragma once

#include "common.cuh"
#include "scan_fwd.cuh"

namespace ssm {
namespace tc {

constexpr int kThreads = 512;  // 16 warps: 4 state quarters x 4 tensor-memory lane quarters
constexpr int kCH = 128;        // channels per group = tensor-memory lanes = MMA M
constexpr int kN = 16;          // states
constexpr int kTB = 8;          // tokens per block (one MMA pair, one pipeline step)
constexpr int kTT = 32;         // tokens per raw input tile (4 blocks)
constexpr int kNSLOT = 4;       // operand slots (A1, W, Bexp, Cexp)
constexpr int kNTILE = 3;       // raw input tiles in flight
constexpr int kTmemCols = 512;  // 2 buffers x (128 bb + 128 Cb) columns

// Operands are K-major without swizzle: 8 x 16-byte core matrices, the next
// core matrix along K 128 bytes on, the next 8 rows 256 bytes on.
__host__ __device__ constexpr int kmaj(int row, int k) {
    return (row >> 3) * 256 + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4;
}
// Column (= Bexp / Cexp row) of token t, state n within a block: each thread's
// 4 states x 8 tokens are 32 consecutive columns.
__host__ __device__ constexpr int bcol(int t, int n) { return (n >> 2) * 32 + t * 4 + (n & 3); }
constexpr int kOpBytes = 128 * kTB * 4;     // one 128 x 8 tf32 operand
constexpr int kSlotBytes = 4 * kOpBytes;    // A1 = Delta u, W = Delta, Bexp, Cexp
constexpr int kOffW = kOpBytes, kOffBexp = 2 * kOpBytes, kOffCexp = 3 * kOpBytes;
constexpr int kYRow = 48;                   // 8 fp32 partial sums + 16 bytes of padding
constexpr int kYBytes = 4 * kCH * kYRow;    // the four state quarters
constexpr int kRawRow = kTT * 2 + 16;       // one channel's 32 bf16 tokens, padded
constexpr int kRawPlane = kCH * kRawRow;
constexpr int kRawBC = kTT * kN * 2;        // 32 tokens x 16 states bf16
constexpr int kTileBytes = 3 * kRawPlane + 2 * kRawBC;
constexpr int kOffOnes = kNSLOT * kSlotBytes;
constexpr int kOffY = kOffOnes + kOpBytes;
constexpr int kOffRaw = kOffY + 2 * kYBytes;
constexpr int kSmem = kOffRaw + kNTILE * kTileBytes;
static_assert(kSmem <= 226 * 1024, "shared memory");

// instruction descriptor, kind::tf32, fp32 accumulate, both operands K-major
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(mbar))
        : "memory");
}
__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* m, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count)
                 : "memory");
}
// Bounded wait for phase `parity` of an mbarrier; false if it gave up.  Once
// a wait of the CTA has given up (*failed set) later waits return at once, so
// a broken pipeline ends the kernel quickly instead of waiting step by step.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity, volatile int* failed) {
    if (*failed) return false;
    for (long it = 0; it < (1l << 22); it++) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(smem_u32(m)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    *failed = 1;
    return false;
}

#define SSM_TMEM_LD32(addr, v, o)                                                              \
    asm volatile(                                                                              \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"   \
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" \
        : "=r"(v[o + 0]), "=r"(v[o + 1]), "=r"(v[o + 2]), "=r"(v[o + 3]), "=r"(v[o + 4]),      \
          "=r"(v[o + 5]), "=r"(v[o + 6]), "=r"(v[o + 7]), "=r"(v[o + 8]), "=r"(v[o + 9]),      \
          "=r"(v[o + 10]), "=r"(v[o + 11]), "=r"(v[o + 12]), "=r"(v[o + 13]),                  \
          "=r"(v[o + 14]), "=r"(v[o + 15]), "=r"(v[o + 16]), "=r"(v[o + 17]),                  \
          "=r"(v[o + 18]), "=r"(v[o + 19]), "=r"(v[o + 20]), "=r"(v[o + 21]),                  \
          "=r"(v[o + 22]), "=r"(v[o + 23]), "=r"(v[o + 24]), "=r"(v[o + 25]),                  \
          "=r"(v[o + 26]), "=r"(v[o + 27]), "=r"(v[o + 28]), "=r"(v[o + 29]),                  \
          "=r"(v[o + 30]), "=r"(v[o + 31])                                                     \
        : "r"(addr))
#define SSM_TMEM_ST32(addr, v, o)                                                              \
    asm volatile(                                                                              \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"    \
        "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"     \
        "%32};" ::"r"(addr),                                                                   \
        "r"(v[o + 0]), "r"(v[o + 1]), "r"(v[o + 2]), "r"(v[o + 3]), "r"(v[o + 4]),             \
        "r"(v[o + 5]), "r"(v[o + 6]), "r"(v[o + 7]), "r"(v[o + 8]), "r"(v[o + 9]),             \
        "r"(v[o + 10]), "r"(v[o + 11]), "r"(v[o + 12]), "r"(v[o + 13]), "r"(v[o + 14]),        \
        "r"(v[o + 15]), "r"(v[o + 16]), "r"(v[o + 17]), "r"(v[o + 18]), "r"(v[o + 19]),        \
        "r"(v[o + 20]), "r"(v[o + 21]), "r"(v[o + 22]), "r"(v[o + 23]), "r"(v[o + 24]),        \
        "r"(v[o + 25]), "r"(v[o + 26]), "r"(v[o + 27]), "r"(v[o + 28]), "r"(v[o + 29]),        \
        "r"(v[o + 30]), "r"(v[o + 31])                                                         \
        : "memory")

__device__ __forceinline__ float to_tf32(float x) {   // round to nearest, ties away
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

struct Shared {
    uint64_t mbar[4];
    uint32_t taddr;
    int ok;
    int failed;   // a bounded wait of this CTA gave up
};

// One part: channel group `grp`, blocks [b0, b1) of its 8-token blocks.
// `S` is the CTA's running step counter (mbarrier slot and phase).
template <bool HAS_Z, bool SOFTPLUS>
__device__ __forceinline__ void tc_part(const ScanParams& p, unsigned char* smem, Shared& sh,
                                        int64_t grp, int64_t b0, int64_t b1, uint32_t& S) {
    using bf16 = __nv_bfloat16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, s4 = warp >> 2;
    const int c = q * 32 + lane;                       // this thread's channel in the group
    const int64_t b = grp / p.groups_per_row;
    const int64_t d0 = (grp % p.groups_per_row) * kCH;
    const int rows = (int)(p.dim - d0 < kCH ? p.dim - d0 : kCH);
    const int64_t row0 = b * p.dim + d0;
    const int64_t L = p.L;
    const int nb = (int)(b1 - b0);
    const bool active = c < rows;

    const bf16* gu = static_cast<const bf16*>(p.u);
    const bf16* gdl = static_cast<const bf16*>(p.delta);
    const bf16* gz = static_cast<const bf16*>(p.z);
    const bf16* gB = static_cast<const bf16*>(p.B) + b * L * kN;
    const bf16* gC = static_cast<const bf16*>(p.C) + b * L * kN;
    bf16* gy = static_cast<bf16*>(p.y);

    float A2[4], h[4];
#pragma unroll
    for (int j = 0; j < 4; j++)   // exp(Delta A) = 2^(Delta A log2 e)
        A2[j] = active ? p.A[(d0 + c) * kN + s4 * 4 + j] * kLog2e : 0.0f;
    float bias = (active && p.bias) ? p.bias[d0 + c] : 0.0f;
    if (SOFTPLUS) bias *= kLog2e;
    const float Dv = (active && p.D) ? p.D[d0 + c] : 0.0f;

    // raw inputs of tile j (blocks 4j .. 4j+3) into ring slot j % kNTILE,
    // 64 bytes per channel row; zero past the last channel
    auto load_tile = [&](int j) {
        unsigned char* r = smem + kOffRaw + (j % kNTILE) * kTileBytes;
        const int kb0 = 4 * j;
        const int nblk = nb - kb0 < 4 ? nb - kb0 : 4;     // blocks of this tile in the part
        const int64_t t0 = (b0 + kb0) * kTB;
        const int nplanes = HAS_Z ? 3 : 2;
        // one 16-byte chunk (8 bf16 tokens) per block: chunk ck of a row is
        // block 4j + ck, present only for ck < nblk
        for (int i = tid; i < nplanes * kCH * 4; i += kThreads) {
            const int pl = i / (kCH * 4), rem = i % (kCH * 4), ch = rem >> 2, ck = rem & 3;
            if (ck >= nblk) continue;
            const bf16* src = pl == 0 ? gu : (pl == 1 ? gdl : gz);
            const bool ok = ch < rows;
            ssm::seq::cp_async16(r + pl * kRawPlane + ch * kRawRow + ck * 16,
                                 ok ? static_cast<const void*>(src + (row0 + ch) * L + t0 + ck * 8)
                                    : src,
                                 ok ? 16 : 0);
        }
        for (int i = tid; i < 2 * nblk * 16; i += kThreads) {   // B, C: 16 chunks per block
            const int which = i / (nblk * 16), e = (i % (nblk * 16)) * 8;
            const bf16* src = (which == 0 ? gB : gC) + t0 * kN + e;
            ssm::seq::cp_async16(r + 3 * kRawPlane + which * kRawBC + e * 2, src, 16);
        }
    };

    // initial state: zero, or the state handed over by the CTA before
    if (b0 == 0) {
#pragma unroll
        for (int j = 0; j < 4; j++) h[j] = 0.0f;
    } else {
        if (tid == 0) {
            const bool ok = ssm::seq::wait_flag(p.flags + grp);
            if (!ok) atomicExch(p.status, kStatusTimeout);
            __threadfence();
            sh.ok = ok;
        }
        __syncthreads();
        const bool ok = sh.ok;
        const float* src = p.carry + (grp * kCH + c) * kN + s4 * 4;
#pragma unroll
        for (int j = 0; j < 4; j++) h[j] = ok ? __ldcg(src + j) : __int_as_float(0x7fc00000);
    }

    // Tile j is requested at step 4j - 7 (tile 0 before the first step) and
    // first read at step 4j - 3; one cp.async group per step, so at every
    // step all but the three newest groups must be complete.
    load_tile(0);
    ssm::seq::cp_async_commit();
    for (int i = 0; i < 3; i++) ssm::seq::cp_async_commit();

    const uint32_t tbase = sh.taddr;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;

    for (int k = -3; k < nb; k++, S++) {
        asm volatile("cp.async.wait_group 3;\n" ::: "memory");

        // ---- recurrence of block k: states 4 s4 .. 4 s4 + 3 ----
        if (k >= 0) {
            const uint32_t col = tbase + lane_base + (uint32_t)((k & 1) * 256 + s4 * 32);
            uint32_t v[32], cv[32];
            SSM_TMEM_LD32(col, v, 0);
            SSM_TMEM_LD32(col + 128, cv, 0);
            const unsigned char* wsl = smem + (k % kNSLOT) * kSlotBytes + kOffW;
            const float4 dA = *reinterpret_cast<const float4*>(wsl + kmaj(c, 0));
            const float4 dB = *reinterpret_cast<const float4*>(wsl + kmaj(c, 4));
            const float dts[8] = {dA.x, dA.y, dA.z, dA.w, dB.x, dB.y, dB.z, dB.w};
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            float yp[8];
#pragma unroll
            for (int t = 0; t < kTB; t++) {
                const float2 dt2 = make_float2(dts[t], dts[t]);
                const float2 e0 = __fmul2_rn(dt2, make_float2(A2[0], A2[1]));
                const float2 e1 = __fmul2_rn(dt2, make_float2(A2[2], A2[3]));
                const float2 a0 = make_float2(ex2(e0.x), ex2(e0.y));
                const float2 a1 = make_float2(ex2(e1.x), ex2(e1.y));
                const float2 h0 = __ffma2_rn(a0, make_float2(h[0], h[1]),
                                             make_float2(__uint_as_float(v[t * 4]),
                                                         __uint_as_float(v[t * 4 + 1])));
                const float2 h1 = __ffma2_rn(a1, make_float2(h[2], h[3]),
                                             make_float2(__uint_as_float(v[t * 4 + 2]),
                                                         __uint_as_float(v[t * 4 + 3])));
                h[0] = h0.x; h[1] = h0.y; h[2] = h1.x; h[3] = h1.y;
                float2 acc = __fmul2_rn(make_float2(__uint_as_float(cv[t * 4]),
                                                    __uint_as_float(cv[t * 4 + 1])), h0);
                acc = __ffma2_rn(make_float2(__uint_as_float(cv[t * 4 + 2]),
                                             __uint_as_float(cv[t * 4 + 3])), h1, acc);
                yp[t] = acc.x + acc.y;
            }
            float4* ydst = reinterpret_cast<float4*>(smem + kOffY + (k & 1) * kYBytes +
                                                     (s4 * kCH + c) * kYRow);
            ydst[0] = make_float4(yp[0], yp[1], yp[2], yp[3]);
            ydst[1] = make_float4(yp[4], yp[5], yp[6], yp[7]);
            if (k == nb - 1) {   // the part's final state
                if (b1 * kTB == L) {
                    if (active && p.last_state) {
                        float* dst = p.last_state + (row0 + c) * kN + s4 * 4;
#pragma unroll
                        for (int j = 0; j < 4; j++) dst[j] = h[j];
                    }
                } else {
                    float* dst = p.carry + (grp * kCH + c) * kN + s4 * 4;
#pragma unroll
                    for (int j = 0; j < 4; j++) __stcg(dst + j, h[j]);
                    __threadfence();
                }
            }
        }
        // step k-1's MMAs (block k+1, read from the next step on): only the
        // issuing thread waits, and the barrier passes the completion on
        if (tid == 0 && S >= 1 &&
            !mbar_wait(&sh.mbar[(S - 1) & 3], ((S - 1) >> 2) & 1, &sh.failed))
            atomicExch(p.status, kStatusTimeout);
        fence_before();
        __syncthreads();
        fence_after();

        // ---- MMAs of block k+2 (one thread) ----
        if (tid == 0) {
            if (k == nb - 1 && b1 * kTB != L)
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + grp), "r"(1u)
                             : "memory");
            const int k2 = k + 2;
            if (k2 >= 0 && k2 < nb) {
                const unsigned char* sl = smem + (k2 % kNSLOT) * kSlotBytes;
                const uint32_t d = tbase + (uint32_t)((k2 & 1) * 256);
                mma_ss(d, sdesc(smem_u32(sl), 128, 256), sdesc(smem_u32(sl + kOffBexp), 128, 256),
                       idesc_tf32(128, 128), 0);
                mma_ss(d + 128, sdesc(smem_u32(smem + kOffOnes), 128, 256),
                       sdesc(smem_u32(sl + kOffCexp), 128, 256), idesc_tf32(128, 128), 0);
            }
            mma_commit(&sh.mbar[S & 3]);
        }

        const int k3 = k + 3;
        if (s4 == 0) {
            // ---- prologue of block k+3: Delta and Delta u ----
            if (k3 < nb) {
                const unsigned char* r = smem + kOffRaw + ((k3 >> 2) % kNTILE) * kTileBytes +
                                         c * kRawRow + (k3 & 3) * 16;
                float uv[8], dv[8];
                ssm::seq::unpack8<bf16>(r, uv);
                ssm::seq::unpack8<bf16>(r + kRawPlane, dv);
                float dt[8], du[8];
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    if constexpr (SOFTPLUS) dt[t] = ssm::seq::softplus_log2(fmaf(dv[t], kLog2e, bias));
                    else dt[t] = dv[t] + bias;
                    du[t] = to_tf32(dt[t] * uv[t]);
                }
                unsigned char* sl = smem + (k3 % kNSLOT) * kSlotBytes;
                *reinterpret_cast<float4*>(sl + kmaj(c, 0)) = make_float4(du[0], du[1], du[2], du[3]);
                *reinterpret_cast<float4*>(sl + kmaj(c, 4)) = make_float4(du[4], du[5], du[6], du[7]);
                *reinterpret_cast<float4*>(sl + kOffW + kmaj(c, 0)) = make_float4(dt[0], dt[1], dt[2], dt[3]);
                *reinterpret_cast<float4*>(sl + kOffW + kmaj(c, 4)) = make_float4(dt[4], dt[5], dt[6], dt[7]);
            }
        } else if (s4 == 1) {
            // ---- B and C of block k+3 onto their block diagonals ----
            if (k3 < nb) {
                const unsigned char* r = smem + kOffRaw + ((k3 >> 2) % kNTILE) * kTileBytes +
                                         3 * kRawPlane + (k3 & 3) * 256;
                unsigned char* sl = smem + (k3 % kNSLOT) * kSlotBytes;
                const int i = c;                   // one B and one C value per thread
                const int t = i >> 4, n = i & 15;
                const int row = bcol(t, n);
                const float bv = __bfloat162float(reinterpret_cast<const bf16*>(r)[i]);
                const float cv = __bfloat162float(reinterpret_cast<const bf16*>(r + kRawBC)[i]);
                *reinterpret_cast<float*>(sl + kOffBexp + kmaj(row, t)) = bv;
                *reinterpret_cast<float*>(sl + kOffCexp + kmaj(row, 0)) = cv;
            }
        } else if (k >= 0) {
            // ---- output of block k: tokens 4 (s4 - 2) .. + 3 of channel c ----
            const int half = s4 - 2;
            const unsigned char* yb = smem + kOffY + (k & 1) * kYBytes + c * kYRow + half * 16;
            float4 acc = *reinterpret_cast<const float4*>(yb);
#pragma unroll
            for (int qq = 1; qq < 4; qq++) {
                const float4 a = *reinterpret_cast<const float4*>(yb + qq * kCH * kYRow);
                acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
            }
            float ys[4] = {acc.x, acc.y, acc.z, acc.w};
            const unsigned char* r = smem + kOffRaw + ((k >> 2) % kNTILE) * kTileBytes +
                                     c * kRawRow + (k & 3) * 16 + half * 8;
            const uint2 uq = *reinterpret_cast<const uint2*>(r);
            const float uv[4] = {__uint_as_float(uq.x << 16), __uint_as_float(uq.x & 0xffff0000u),
                                 __uint_as_float(uq.y << 16), __uint_as_float(uq.y & 0xffff0000u)};
#pragma unroll
            for (int t = 0; t < 4; t++) ys[t] = fmaf(Dv, uv[t], ys[t]);
            if constexpr (HAS_Z) {
                const uint2 zq = *reinterpret_cast<const uint2*>(r + 2 * kRawPlane);
                const float zv[4] = {__uint_as_float(zq.x << 16), __uint_as_float(zq.x & 0xffff0000u),
                                     __uint_as_float(zq.y << 16), __uint_as_float(zq.y & 0xffff0000u)};
#pragma unroll
                for (int t = 0; t < 4; t++) ys[t] *= ssm::seq::gate<bf16>(zv[t]);
            }
            if (active) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(ys[0], ys[1]);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(ys[2], ys[3]);
                uint2 o;
                o.x = *reinterpret_cast<const unsigned*>(&lo);
                o.y = *reinterpret_cast<const unsigned*>(&hi);
                *reinterpret_cast<uint2*>(gy + (row0 + c) * L + (b0 + k) * kTB + half * 4) = o;
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

        // ---- raw inputs of tile (k+7)/4 ----
        if (((k + 7) & 3) == 0) {
            const int j = (k + 7) >> 2;
            if (j >= 1 && 4 * j < nb) load_tile(j);
        }
        ssm::seq::cp_async_commit();
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    // the last MMAs of the part (issued at step nb-3) were waited for at step nb-2
    __syncthreads();
}

// Persistent, balanced schedule over (channel group, 8-token block) work,
// as for the state-split kernel; one CTA per SM (it holds all 512 columns
// of tensor memory).
template <bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(kThreads, 1) scan_fwd_tc_kernel(ScanParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ Shared sh;
    const int tid = threadIdx.x;

    // zero the operand slots once (only the block diagonals of Bexp and Cexp
    // are ever written again); the ones operand has a 1 in column 0 of every row
    for (int i = tid * 16; i < kOffY; i += kThreads * 16)
        *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid < kCH) *reinterpret_cast<float*>(smem + kOffOnes + kmaj(tid, 0)) = 1.0f;
    if (tid < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sh.taddr)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        sh.failed = 0;
        for (int i = 0; i < 4; i++) mbar_init(&sh.mbar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    fence_before();
    __syncthreads();
    fence_after();

    const int64_t nblk = p.L / kTB;
    const int64_t W = p.ngroups * nblk;
    const int64_t s = W * blockIdx.x / gridDim.x;
    const int64_t e = W * (blockIdx.x + 1) / gridDim.x;
    uint32_t S = 0;
    if (s < e) {
        const int64_t g_first = s / nblk, g_last = (e - 1) / nblk;
        for (int64_t grp = g_last; grp >= g_first; grp--) {
            const int64_t lo = grp * nblk;
            const int64_t b0 = (s > lo ? s : lo) - lo;
            const int64_t b1 = (e < lo + nblk ? e : lo + nblk) - lo;
            tc_part<HAS_Z, SOFTPLUS>(p, smem, sh, grp, b0, b1, S);
        }
    }

    fence_before();
    __syncthreads();
    if (tid < 32) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(sh.taddr),
                     "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc
}  // namespace ssm
