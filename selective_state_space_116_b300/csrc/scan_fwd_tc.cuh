// Forward selective scan with the tensor cores distributing B and C (bf16
// I/O, N = 16): an asynchronous, warp-specialised pipeline.
//
// The state-split kernel in scan_fwd.cuh is bound by shared-memory
// bandwidth: every thread reads the token's B and C rows (64 bytes per thread
// per token), although all channels of a batch row share them.  Here the
// tensor cores read B and C once per CTA and hand every channel its values
// in tensor memory, where each thread reads its own lane:
//
//   input term   bb[c, (t, n)] = (Delta u)[c, t] * B[t, n]: over a block of 8
//                tokens the GEMM  A1 x Bexp^T  with A1[c, t] = (Delta u)[c, t]
//                and the block-diagonal Bexp[(t, n), t'] = B[t, n] [t = t']
//                (M = 128 channels, N = 128, K = 8)
//   C broadcast  Cb[c, (t, n)] = C[t, n] for every channel c: the GEMM
//                ones x Cexp^T with ones[c, k] = [k = 0] and Cexp[(t, n), k]
//                = C[t, n] [k = 0]  (same shape)
//
// Both are kind::tf32 MMAs (B, C and 1 are exact in tf32; Delta u is rounded
// to tf32's 10-bit mantissa, a relative error of 2^-11 on the input term that
// the bf16 output then rounds at 2^-9).  The recurrence h = exp(Delta A) h +
// bb and the output sum y = sum_n C h + D u stay on the CUDA cores in fp32,
// with the state in registers.  (The output contraction is not put on the
// tensor cores: per token it is a dot product of 16, and as an MMA it needs
// K = tokens x states against a block-diagonal C, 16 small MMAs per block,
// which cost more tensor-core time than the recurrence takes.)
//
// Roles (512 threads, 16 warps, one CTA per SM holding all 512 columns of
// tensor memory); every hand-off is an mbarrier ring, with one arrival per
// warp, and no CTA-wide barrier runs inside the loop:
//   warp 0        producer: one thread issues the TMA copies of 16-token
//                 tiles (u, delta, z as 128-channel x 16-token boxes with
//                 32-byte swizzle; the B and C rows as bulk copies) into a
//                 ring of tiles
//   warp 1        one thread issues the two MMAs of every 8-token block into
//                 a ring of 2 tensor-memory buffers (256 columns each)
//   warps 2-3     epilogue: the sum of the two state halves' partial outputs,
//                 D u skip term, silu(z) gate, bf16 store (2 channels a thread)
//   warps 4-7     prologue, thread c for channel c: Delta = softplus(delta +
//                 bias), Delta u into the A1 operand, Delta for the
//                 recurrence, B and C onto their block diagonals (ring of
//                 operand slots)
//   warps 8-15    recurrence: warp w serves tensor-memory lanes 32 (w % 4) ..
//                 + 31 (channels) and state half (w - 8) / 4; each thread
//                 loads its bb and C values with tcgen05.ld (the next two
//                 tokens' load in flight while it computes the current two),
//                 advances its 8 states and writes its partial C.h
// Every wait is bounded; a wait that gives up marks the CTA failed, later
// waits return at once, and the workspace status word reports it.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "scan_fwd.cuh"

namespace ssm {
namespace tc {

constexpr int kThreads = 512;
constexpr int kCH = 128;        // channels per group = tensor-memory lanes = MMA M
constexpr int kN = 16;          // states
constexpr int kTB = 8;          // tokens per block (one MMA pair)
constexpr int kBPT = 2;         // blocks per raw tile
constexpr int kTT = kTB * kBPT; // tokens per raw tile
constexpr int kRawSlots = 7;    // raw tiles in flight
constexpr int kOpSlots = 4;     // operand slots in flight
constexpr int kYSlots = 4;      // partial-output slots in flight
constexpr int kRecWarps = 8;
constexpr int kTmemCols = 512;  // 2 buffers x (128 bb + 128 Cb) columns

// Operands are K-major without swizzle: 8 x 16-byte core matrices, the next
// core matrix along K 128 bytes on, the next 8 rows 256 bytes on.
__host__ __device__ constexpr int kmaj(int row, int k) {
    return (row >> 3) * 256 + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4;
}
// Column (= Bexp / Cexp row) of token t, state n within a block: the 8 states
// x 8 tokens of each state half are 64 consecutive columns.
__host__ __device__ constexpr int bcol(int t, int n) { return (n >> 3) * 64 + t * 8 + (n & 7); }
constexpr int kOpBytes = 128 * kTB * 4;     // one 128 x 8 tf32 operand
constexpr int kSlotBytes = 4 * kOpBytes;    // A1 = Delta u, W = Delta, Bexp, Cexp
constexpr int kOffW = kOpBytes, kOffBexp = 2 * kOpBytes, kOffCexp = 3 * kOpBytes;
constexpr int kYRow = 48;                   // 8 fp32 partial sums + 16 bytes of padding
constexpr int kYBytes = 2 * kCH * kYRow;    // both state halves of one block
// Raw tile: the u, delta, z planes as TMA writes a 16-token x 128-channel box
// (32-byte rows, the two 16-byte halves of row r swapped when bit 2 of r is
// set: the 32-byte swizzle, which keeps 8 consecutive rows' reads of one
// half on distinct banks), then the B and C rows of the 16 tokens.
constexpr int kPlaneBytes = kCH * kTT * 2;
constexpr int kRawBC = kTT * kN * 2;        // 16 tokens x 16 states bf16
constexpr int kOffTileB = 3 * kPlaneBytes, kOffTileC = kOffTileB + kRawBC;
constexpr int kTileBytes = (kOffTileC + kRawBC + 1023) / 1024 * 1024;
__host__ __device__ constexpr int raw_off(int c, int blk) { return c * 32 + ((blk ^ (c >> 2)) & 1) * 16; }
constexpr int kOffOnes = kOpSlots * kSlotBytes;
constexpr int kOffY = kOffOnes + kOpBytes;
constexpr int kOffRaw = kOffY + kYSlots * kYBytes;
constexpr int kSmemUsed = kOffRaw + kRawSlots * kTileBytes;
constexpr int kSmem = kSmemUsed + 1024;   // room to align the base to 1 KB
static_assert(kSmem <= 226 * 1024, "shared memory");
static_assert(kOffRaw % 1024 == 0 && kTileBytes % 1024 == 0, "swizzled planes need 1 KB alignment");

// tensor maps of u, delta, z: (L, dim, batch) bf16, box (16, 128, 1), 32-byte swizzle
struct TmaMaps {
    CUtensorMap u, delta, z;
};

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
#define SSM_TMEM_LD16(addr, v)                                                                 \
    asm volatile(                                                                              \
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"   \
        "%13,%14,%15}, [%16];"                                                                 \
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),  \
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),           \
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])                                                \
        : "r"(addr))
__device__ __forceinline__ float to_tf32(float x) {   // round to nearest, ties away
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}


__device__ __forceinline__ void mbar_arrive(uint64_t* m) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(m)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* m, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes)
                 : "memory");
}
// TMA: box at (x, y, z) of a 3-D tensor map -> shared memory, completion
// counted in bytes on the mbarrier
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* m) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(m))
        : "memory");
}
// bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* m) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(m))
        : "memory");
}
// barrier over the `count` threads of a role (ids 1.. ; 0 is __syncthreads)
__device__ __forceinline__ void role_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

struct Bars {
    uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];
    uint64_t op_full[kOpSlots], op_empty[kOpSlots];
    uint64_t d_full[2], d_empty[2], yp_full[kYSlots], yp_empty[kYSlots];
    uint32_t taddr;
    int failed;   // a bounded wait of this CTA gave up
    int ok;       // the carry hand-over arrived
};

// The CTA's share of the (channel group, 8-token block) work, walked by every
// role in the same order (as in scan_fwd_kernel of scan_fwd.cuh): the head
// of its last group, its whole groups, the continuation of its first group.
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

// Position in that walk: block kb of group grp (part [b0, b1); batch row b,
// first channel d0), the CTA-wide block counter i and raw-tile counter T.
struct Cursor {
    int64_t grp, b0, b1, kb, i, T, b, d0;
    __device__ Cursor(const Parts& pt, const ScanParams& p) : grp(pt.g_last), i(0), T(0) {
        enter(pt, p);
    }
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
    __device__ int blk() const { return (int)((kb - b0) & (kBPT - 1)); }
    __device__ bool tile_last() const { return blk() == kBPT - 1 || kb == b1 - 1; }
    __device__ void next(const Parts& pt, const ScanParams& p) {
        if (tile_last()) T++;
        i++;
        if (++kb == b1) {
            --grp;
            enter(pt, p);
        }
    }
};
static_assert((kBPT & (kBPT - 1)) == 0, "blocks per tile: a power of two");

__device__ __forceinline__ bool wait_or_fail(uint64_t* m, uint32_t parity, Bars& br,
                                             const ScanParams& p) {
    if (mbar_wait(m, parity, &br.failed)) return true;
    atomicExch(p.status, kStatusTimeout);
    return false;
}
// phase parity of the k-th use (k = 0, 1, ...) of a ring slot: the full
// barrier's phase k, and the empty barrier's phase k - 1 (k >= 1)
__device__ __forceinline__ uint32_t full_parity(int64_t k) { return (uint32_t)(k & 1); }
__device__ __forceinline__ uint32_t empty_parity(int64_t k) { return (uint32_t)((k + 1) & 1); }

// wait for this thread's tensor-memory loads; the "+r" operands keep every use
// of the loaded registers after the wait
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[16], uint32_t (&w)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                   "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                   "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(w[0]), "+r"(w[1]),
                   "+r"(w[2]), "+r"(w[3]), "+r"(w[4]), "+r"(w[5]), "+r"(w[6]), "+r"(w[7]),
                   "+r"(w[8]), "+r"(w[9]), "+r"(w[10]), "+r"(w[11]), "+r"(w[12]), "+r"(w[13]),
                   "+r"(w[14]), "+r"(w[15])
                 :
                 : "memory");
}

template <bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(kThreads, 1)
    scan_fwd_tc_kernel(ScanParams p, const __grid_constant__ TmaMaps maps) {
    using bf16 = __nv_bfloat16;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars br;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // zero the operand slots once (only the block diagonals of Bexp and Cexp
    // are ever written again); the ones operand has a 1 in column 0 of every row
    for (int i = tid * 16; i < kOffY; i += kThreads * 16)
        *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid < kCH) *reinterpret_cast<float*>(smem + kOffOnes + kmaj(tid, 0)) = 1.0f;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&br.taddr)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        br.failed = 0;
        for (int i = 0; i < kRawSlots; i++) {
            mbar_init(&br.raw_full[i], 1);    // the producer's expect_tx
            mbar_init(&br.raw_empty[i], 6);   // 4 prologue + 2 epilogue warps
        }
        for (int i = 0; i < kOpSlots; i++) {
            mbar_init(&br.op_full[i], 4);                  // prologue warps
            mbar_init(&br.op_empty[i], 1 + kRecWarps);     // MMA commit + recurrence warps
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&br.d_full[i], 1);                   // MMA commit
            mbar_init(&br.d_empty[i], kRecWarps);
        }
        for (int i = 0; i < kYSlots; i++) {
            mbar_init(&br.yp_full[i], kRecWarps);
            mbar_init(&br.yp_empty[i], 2);                 // epilogue warps
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    fence_before();
    __syncthreads();
    fence_after();

    const Parts parts(p);
    const uint32_t tbase = br.taddr;
    const int64_t L = p.L;

    if (warp == 0) {
        // ---------------- producer: raw input tiles (one thread) ----------------
        if (lane == 0) {
            int64_t T = 0;   // CTA-wide tile counter
            for (int64_t grp = parts.g_last; grp >= parts.g_first; grp--) {
                int64_t b0, b1;
                parts.range(grp, b0, b1);
                const int64_t b = grp / p.groups_per_row;
                const int d0 = (int)((grp % p.groups_per_row) * kCH);
                const bf16* gB = static_cast<const bf16*>(p.B) + b * L * kN;
                const bf16* gC = static_cast<const bf16*>(p.C) + b * L * kN;
                const int nb = (int)(b1 - b0);
                for (int j = 0; j * kBPT < nb; j++, T++) {
                    const int slot = (int)(T % kRawSlots);
                    if (T >= kRawSlots) wait_or_fail(&br.raw_empty[slot], empty_parity(T / kRawSlots), br, p);
                    unsigned char* r = smem + kOffRaw + slot * kTileBytes;
                    const int nblk = nb - j * kBPT < kBPT ? nb - j * kBPT : kBPT;
                    const int64_t t0 = (b0 + (int64_t)j * kBPT) * kTB;
                    const uint32_t bc = (uint32_t)(nblk * kTB * kN * 2);
                    mbar_expect_tx(&br.raw_full[slot], (HAS_Z ? 3 : 2) * kPlaneBytes + 2 * bc);
                    tma_load_3d(r, &maps.u, (int)t0, d0, (int)b, &br.raw_full[slot]);
                    tma_load_3d(r + kPlaneBytes, &maps.delta, (int)t0, d0, (int)b, &br.raw_full[slot]);
                    if (HAS_Z) tma_load_3d(r + 2 * kPlaneBytes, &maps.z, (int)t0, d0, (int)b, &br.raw_full[slot]);
                    bulk_load(r + kOffTileB, gB + t0 * kN, bc, &br.raw_full[slot]);
                    bulk_load(r + kOffTileC, gC + t0 * kN, bc, &br.raw_full[slot]);
                }
            }
            // the shared memory is released when the CTA exits: let the last
            // copies land even if the pipeline gave up
            volatile int never = 0;
            for (int64_t k = T - kRawSlots < 0 ? 0 : T - kRawSlots; k < T; k++)
                mbar_wait(&br.raw_full[k % kRawSlots], full_parity(k / kRawSlots), &never);
        }
    } else if (warp == 1) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            int64_t i = 0;   // CTA-wide block counter
            for (Cursor cu(parts, p); cu.valid(parts); cu.next(parts, p), i++) {
                const int o = (int)(i % kOpSlots), bf = (int)(i & 1);
                wait_or_fail(&br.op_full[o], full_parity(i / kOpSlots), br, p);
                if (i >= 2) wait_or_fail(&br.d_empty[bf], empty_parity(i / 2), br, p);
                fence_after();
                const unsigned char* sl = smem + o * kSlotBytes;
                const uint32_t d = tbase + (uint32_t)(bf * 256);
                mma_ss(d, sdesc(smem_u32(sl), 128, 256), sdesc(smem_u32(sl + kOffBexp), 128, 256),
                       idesc_tf32(128, 128), 0);
                mma_ss(d + 128, sdesc(smem_u32(smem + kOffOnes), 128, 256),
                       sdesc(smem_u32(sl + kOffCexp), 128, 256), idesc_tf32(128, 128), 0);
                mma_commit(&br.d_full[bf]);
                mma_commit(&br.op_empty[o]);
            }
            // the tensor memory is freed below: let the last MMAs finish even
            // if the pipeline gave up
            if (i > 0) {
                volatile int never = 0;
                mbar_wait(&br.d_full[(i - 1) & 1], full_parity((i - 1) / 2), &never);
            }
        }
    } else if (warp == 2 || warp == 3) {
        // ---------------- epilogue ----------------
        for (Cursor ec(parts, p); ec.valid(parts); ec.next(parts, p)) {
            const int64_t b = ec.b, d0 = ec.d0;
            const int rs = (int)(ec.T % kRawSlots), ys = (int)(ec.i % kYSlots), blk = ec.blk();
            wait_or_fail(&br.yp_full[ys], full_parity(ec.i / kYSlots), br, p);
            float y[2][8];
#pragma unroll
            for (int k = 0; k < 2; k++) {   // channels tid - 64 and tid
                const int c = tid - 64 + 64 * k;
                const unsigned char* yb = smem + kOffY + ys * kYBytes + c * kYRow;
                const float4 a0 = *reinterpret_cast<const float4*>(yb);
                const float4 a1 = *reinterpret_cast<const float4*>(yb + 16);
                const float4 b0v = *reinterpret_cast<const float4*>(yb + kCH * kYRow);
                const float4 b1v = *reinterpret_cast<const float4*>(yb + kCH * kYRow + 16);
                y[k][0] = a0.x + b0v.x; y[k][1] = a0.y + b0v.y; y[k][2] = a0.z + b0v.z; y[k][3] = a0.w + b0v.w;
                y[k][4] = a1.x + b1v.x; y[k][5] = a1.y + b1v.y; y[k][6] = a1.z + b1v.z; y[k][7] = a1.w + b1v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&br.yp_empty[ys]);
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const int c = tid - 64 + 64 * k;
                const bool active = d0 + c < p.dim;
                const float Dv = (active && p.D) ? p.D[d0 + c] : 0.0f;
                const unsigned char* r = smem + kOffRaw + rs * kTileBytes + raw_off(c, blk);
                float uv[8];
                ssm::seq::unpack8<bf16>(r, uv);
#pragma unroll
                for (int t = 0; t < 8; t++) y[k][t] = fmaf(Dv, uv[t], y[k][t]);
                if constexpr (HAS_Z) {
                    float zv[8];
                    ssm::seq::unpack8<bf16>(r + 2 * kPlaneBytes, zv);
#pragma unroll
                    for (int t = 0; t < 8; t++) y[k][t] *= ssm::seq::gate<bf16>(zv[t]);
                }
                if (active) {
                    uint4 ov;
                    unsigned* o32 = reinterpret_cast<unsigned*>(&ov);
#pragma unroll
                    for (int t = 0; t < 4; t++) {
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(y[k][2 * t], y[k][2 * t + 1]);
                        o32[t] = *reinterpret_cast<const unsigned*>(&pr);
                    }
                    bf16* gy = static_cast<bf16*>(p.y);
                    *reinterpret_cast<uint4*>(gy + (b * p.dim + d0 + c) * L + ec.kb * kTB) = ov;
                }
            }
            if (ec.tile_last()) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&br.raw_empty[rs]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- prologue ----------------
        const int c = tid - 128;   // channel within the group
        float bias = 0.0f;
        int64_t bias_grp = -1;
        for (Cursor pc(parts, p); pc.valid(parts); pc.next(parts, p)) {
            const int64_t d0 = pc.d0;
            if (pc.grp != bias_grp) {
                bias_grp = pc.grp;
                bias = (d0 + c < p.dim && p.bias) ? p.bias[d0 + c] : 0.0f;
                if (SOFTPLUS) bias *= kLog2e;
            }
            const int rs = (int)(pc.T % kRawSlots), o = (int)(pc.i % kOpSlots), blk = pc.blk();
            if (blk == 0) wait_or_fail(&br.raw_full[rs], full_parity(pc.T / kRawSlots), br, p);
            if (pc.i >= kOpSlots) wait_or_fail(&br.op_empty[o], empty_parity(pc.i / kOpSlots), br, p);
            const unsigned char* r = smem + kOffRaw + rs * kTileBytes;
            unsigned char* sl = smem + o * kSlotBytes;
            float uv[8], dv[8];
            ssm::seq::unpack8<bf16>(r + raw_off(c, blk), uv);
            ssm::seq::unpack8<bf16>(r + kPlaneBytes + raw_off(c, blk), dv);
            float dt[8], du[8];
#pragma unroll
            for (int t = 0; t < 8; t++) {
                if constexpr (SOFTPLUS) dt[t] = ssm::seq::softplus_log2(fmaf(dv[t], kLog2e, bias));
                else dt[t] = dv[t] + bias;
                du[t] = to_tf32(dt[t] * uv[t]);
            }
            *reinterpret_cast<float4*>(sl + kmaj(c, 0)) = make_float4(du[0], du[1], du[2], du[3]);
            *reinterpret_cast<float4*>(sl + kmaj(c, 4)) = make_float4(du[4], du[5], du[6], du[7]);
            *reinterpret_cast<float4*>(sl + kOffW + kmaj(c, 0)) = make_float4(dt[0], dt[1], dt[2], dt[3]);
            *reinterpret_cast<float4*>(sl + kOffW + kmaj(c, 4)) = make_float4(dt[4], dt[5], dt[6], dt[7]);
            {   // B and C element c of the block onto the block diagonals
                const unsigned char* rb = r + kOffTileB + blk * 256;
                const int t = c >> 4, n = c & 15, row = bcol(t, n);
                const float bv = __bfloat162float(reinterpret_cast<const bf16*>(rb)[c]);
                const float cv = __bfloat162float(reinterpret_cast<const bf16*>(rb + kRawBC)[c]);
                *reinterpret_cast<float*>(sl + kOffBexp + kmaj(row, t)) = bv;
                *reinterpret_cast<float*>(sl + kOffCexp + kmaj(row, 0)) = cv;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&br.op_full[o]);
                if (pc.tile_last()) mbar_arrive(&br.raw_empty[rs]);
            }
        }
    } else if (warp >= 8) {
        // ---------------- recurrence ----------------
        const int g = (warp - 8) >> 2, q = warp & 3;
        const int c = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int64_t i = 0;
        for (int64_t grp = parts.g_last; grp >= parts.g_first; grp--) {
            int64_t b0, b1;
            parts.range(grp, b0, b1);
            const int64_t b = grp / p.groups_per_row;
            const int64_t d0 = (grp % p.groups_per_row) * kCH;
            const int64_t row0 = b * p.dim + d0;
            const bool active = d0 + c < p.dim;
            float A2[8], h[8];
#pragma unroll
            for (int j = 0; j < 8; j++)   // exp(Delta A) = 2^(Delta A log2 e)
                A2[j] = active ? p.A[(d0 + c) * kN + g * 8 + j] * kLog2e : 0.0f;
            if (b0 == 0) {
#pragma unroll
                for (int j = 0; j < 8; j++) h[j] = 0.0f;
            } else {
                if (tid == 256) {
                    const bool ok = ssm::seq::wait_flag(p.flags + grp);
                    if (!ok) atomicExch(p.status, kStatusTimeout);
                    __threadfence();
                    br.ok = ok;
                }
                role_sync(2, 32 * kRecWarps);
                const bool ok = br.ok;
                const float* src = p.carry + (grp * kCH + c) * kN + g * 8;
#pragma unroll
                for (int j = 0; j < 8; j++) h[j] = ok ? __ldcg(src + j) : __int_as_float(0x7fc00000);
            }
            for (int64_t kb = b0; kb < b1; kb++, i++) {
                const int o = (int)(i % kOpSlots), bf = (int)(i & 1), ys = (int)(i % kYSlots);
                wait_or_fail(&br.op_full[o], full_parity(i / kOpSlots), br, p);
                wait_or_fail(&br.d_full[bf], full_parity(i / 2), br, p);
                __syncwarp();
                fence_after();
                const unsigned char* wsl = smem + o * kSlotBytes + kOffW;
                const float4 dA = *reinterpret_cast<const float4*>(wsl + kmaj(c, 0));
                const float4 dB = *reinterpret_cast<const float4*>(wsl + kmaj(c, 4));
                const float dts[8] = {dA.x, dA.y, dA.z, dA.w, dB.x, dB.y, dB.z, dB.w};
                const uint32_t col = tbase + lane_base + (uint32_t)(bf * 256 + g * 64);
                uint32_t v[2][16], cv[2][16];
                SSM_TMEM_LD16(col, v[0]);
                SSM_TMEM_LD16(col + 128, cv[0]);
                float yp[8];
#pragma unroll
                for (int qt = 0; qt < 4; qt++) {   // two tokens (16 columns) at a time
                    const int cur = qt & 1;
                    tmem_wait_ld(v[cur], cv[cur]);
                    if (qt < 3) {
                        SSM_TMEM_LD16(col + (qt + 1) * 16, v[cur ^ 1]);
                        SSM_TMEM_LD16(col + 128 + (qt + 1) * 16, cv[cur ^ 1]);
                    } else {   // all of the block's bb, Cb and Delta are in registers
                        fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&br.d_empty[bf]);
                            mbar_arrive(&br.op_empty[o]);
                        }
                    }
#pragma unroll
                    for (int tt = 0; tt < 2; tt++) {
                        const float2 dt2 = make_float2(dts[qt * 2 + tt], dts[qt * 2 + tt]);
                        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            const float2 e = __fmul2_rn(dt2, make_float2(A2[j], A2[j + 1]));
                            const float2 a = make_float2(ex2(e.x), ex2(e.y));
                            const float2 bb = make_float2(__uint_as_float(v[cur][tt * 8 + j]),
                                                          __uint_as_float(v[cur][tt * 8 + j + 1]));
                            const float2 hn = __ffma2_rn(a, make_float2(h[j], h[j + 1]), bb);
                            h[j] = hn.x;
                            h[j + 1] = hn.y;
                            acc = __ffma2_rn(make_float2(__uint_as_float(cv[cur][tt * 8 + j]),
                                                         __uint_as_float(cv[cur][tt * 8 + j + 1])),
                                             hn, acc);
                        }
                        yp[qt * 2 + tt] = acc.x + acc.y;
                    }
                }
                // this half's partial output sums -> the block's slot
                if (i >= kYSlots) wait_or_fail(&br.yp_empty[ys], empty_parity(i / kYSlots), br, p);
                float4* ydst = reinterpret_cast<float4*>(smem + kOffY + ys * kYBytes + (g * kCH + c) * kYRow);
                ydst[0] = make_float4(yp[0], yp[1], yp[2], yp[3]);
                ydst[1] = make_float4(yp[4], yp[5], yp[6], yp[7]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&br.yp_full[ys]);
            }
            // the part's final state
            if (b1 * kTB == L) {
                if (active && p.last_state) {
                    float* dst = p.last_state + (row0 + c) * kN + g * 8;
#pragma unroll
                    for (int j = 0; j < 8; j++) dst[j] = h[j];
                }
            } else if (b1 > b0) {
                float* dst = p.carry + (grp * kCH + c) * kN + g * 8;
#pragma unroll
                for (int j = 0; j < 8; j++) __stcg(dst + j, h[j]);
                __threadfence();
                role_sync(2, 32 * kRecWarps);
                if (tid == 256)
                    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + grp), "r"(1u)
                                 : "memory");
            }
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(br.taddr),
                     "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc
}  // namespace ssm
