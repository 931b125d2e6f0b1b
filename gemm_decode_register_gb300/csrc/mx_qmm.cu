// mx_qmm.cu -- prefill GEMM over block-float weights on the 5th-generation
// tensor cores (tcgen05), sm_103a.
//
//   Y[m][n] = bf16_rne( sum_k X[m][k] * W[n][k] ),  X bf16, fp32 accumulate.
//
// The pages move block-float dequantisation onto the GPU and feed the
// matrix units from it ("MLxcel 0.8 release", section "Decoding block-float
// formats in software": NVFP4 prefill 3.1x from GPU dequant + WMMA; talk
// slide 12).  Here each CTA owns a 256 x 256 output tile and streams K in
// 64-wide k-blocks through a 3-stage shared-memory ring:
//
//   warp 0      TMA: two 128 x 64 bf16 tiles of X per stage (128-byte swizzle)
//   warp 1      one elected thread issues tcgen05.mma.kind::f16 (bf16 x bf16
//               -> fp32): per k-block 4 K=16 steps for each of the two M=128
//               halves, both sharing the decoded weight tile; the fp32
//               accumulators live in tensor memory (2 x 256 columns)
//   warps 2-9   decoders: thread d loads the packed codes and block scales of
//               weight row n0+d for the k-block, decodes them exactly to bf16
//               (code * scale has at most 6 significant bits) and stores the
//               128-byte row in the same 128-byte-swizzled K-major layout TMA
//               produces; then the epilogue: tcgen05.ld of the accumulator,
//               NVFP4 tensor scale, round to bf16, store.
//
// Every mbarrier wait is bounded (about two seconds of %globaltimer); a wait
// that gives up sets MX_DEVERR_TIMEOUT in the device error word, the CTA
// drains what it has in flight, writes NaN to its Y tile and returns.
#include <cuda.h>

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

constexpr int QMM_BM = 256;   // two M=128 halves
constexpr int QMM_BN = 256;   // UMMA N
constexpr int QMM_BK = 64;    // bf16 elements per 128-byte swizzle row
constexpr int QMM_STAGES = 3;
constexpr int QMM_PF = 4;  // k-blocks of codes each decoder keeps in flight
constexpr int QMM_THREADS = 320;  // 10 warps
constexpr int QMM_A_BYTES = 128 * QMM_BK * 2;         // one M=128 half
constexpr int QMM_B_BYTES = QMM_BN * QMM_BK * 2;
constexpr int QMM_C_BYTES = QMM_BN * 32;  // packed 4-bit codes of one weight tile per k-block

// Per-format stage layout: [X half 0][X half 1][decoded W (bf16)][packed codes].
// The 4-bit formats bring their codes in by TMA with the X tiles; MXFP8
// (twice the code bytes, which would not leave room for three stages) loads
// them per thread.
template <int FMT>
struct QmmGeo {
    static constexpr bool TMA_CODES = FMT != FMT_MXFP8;
    static constexpr int C_BYTES = TMA_CODES ? QMM_C_BYTES : 0;
    static constexpr int STAGE = 2 * QMM_A_BYTES + QMM_B_BYTES + C_BYTES;
    static constexpr int SMEM = QMM_STAGES * STAGE + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(STAGE % 1024 == 0, "stages keep 1024-byte alignment");
};
constexpr unsigned long long QMM_WAIT_NS = 2000000000ull;

// ------------------------------------------------------------ primitives

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait on a phase; false when it timed out or (with
// respect_abort) when another role of the CTA has given up.  Drains of work
// already in flight pass respect_abort = false so they still wait for it.
__device__ __noinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                       unsigned long long limit_ns, bool respect_abort = true)
{
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u) {
            if (respect_abort && *abort_flag) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                 "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (rows of 128 bytes), sm_100 descriptor version.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 D,
// M = 128, N = 256.
__host__ __device__ constexpr uint32_t qmm_idesc()
{
    return (1u << 4)               // D format fp32
           | (1u << 7)             // A format bf16
           | (1u << 10)            // B format bf16
           | ((QMM_BN >> 3) << 17)  // N / 8
           | ((128 >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
                   "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
                   "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
                   "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------ decode

// Codes + scales of one weight row for one 64-wide k-block.
template <int FMT>
struct QRow;
template <>
struct QRow<FMT_MXFP4> {
    uint4 c[2];
    uint32_t s;  // 2 E8M0 bytes
};
template <>
struct QRow<FMT_NVFP4> {
    uint4 c[2];
    uint32_t s;  // 4 E4M3 bytes
};
template <>
struct QRow<FMT_MXFP8> {
    uint4 c[4];
    uint32_t s;  // 2 E8M0 bytes
};

template <int FMT>
__device__ __forceinline__ void qrow_load(const uint8_t *crow, const uint8_t *srow, int kb, QRow<FMT> &r)
{
    if constexpr (FMT == FMT_MXFP8) {
        const uint4 *p = reinterpret_cast<const uint4 *>(crow + (size_t)kb * 64);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.c[i] = __ldg(p + i);
        r.s = ld_nc_u16(srow + 2 * kb);
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(crow + (size_t)kb * 32);
        r.c[0] = __ldg(p);
        r.c[1] = __ldg(p + 1);
        if constexpr (FMT == FMT_NVFP4) r.s = ld_nc_u32(srow + 4 * kb);
        else r.s = ld_nc_u16(srow + 2 * kb);
    }
}

__device__ __forceinline__ uint32_t scaled_bf16x2(uint32_t h2, float s)
{
    return f32x2_to_bf16x2(__fmul_rn(f16_lo_to_f32(h2), s), __fmul_rn(f16_hi_to_f32(h2), s));
}

// Exact f16x2 -> bf16x2 of (value * 2^-112) for values decoded from E2M1 or
// E4M3: those are zero or normal f16 numbers with at most 3 mantissa bits
// (f16 bits 7-9), so the f16 exponent and mantissa bits, moved 3 places
// right, are a normal bf16 number 2^-112 times the value (bf16 bias 127 =
// f16 bias 15 + 112) and zero stays zero; the signs are kept in place.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_m112(uint32_t h2)
{
    return ((h2 & 0x7F807F80u) >> 3) | (h2 & 0x80008000u);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16x2 holding 2^(e-15) twice, for e in [-111, 142] (normal bf16).
__device__ __forceinline__ uint32_t bf16x2_pow2_m15(int e)
{
    const uint32_t b = (uint32_t)(e + 112) << 7;
    return b | (b << 16);
}

// Decode the row's 64 elements to bf16 and store the 128-byte row at
// `row_base` (row r of a 128-byte-swizzled tile: chunk c at c ^ (r & 7)).
// Fast path: hardware cvt to f16, exact move to bf16 (scaled by 2^-112),
// one bf16 multiply by the block scale times 2^112 (exact: the result has at
// most 6 significant bits and stays in bf16's range).  Scales outside the
// fast path's range (E8M0 below 2 (10 for MXFP8) or above 142, NaN scales)
// use exact fp32 products.
template <int FMT>
__device__ __forceinline__ void qrow_store(const QRow<FMT> &r, uint8_t *row_base, int row)
{
    const int sw = row & 7;
    if constexpr (FMT == FMT_MXFP8) {
        // fast path while every product stays a normal bf16 number
        const uint32_t e0 = r.s & 0xFFu, e1 = (r.s >> 8) & 0xFFu;
        if (e0 - 10u <= 132u && e1 - 10u <= 132u) {
            const uint32_t m0 = bf16x2_pow2_m15((int)e0), m1 = bf16x2_pow2_m15((int)e1);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t m = i < 2 ? m0 : m1;
                const uint32_t w[4] = {r.c[i].x, r.c[i].y, r.c[i].z, r.c[i].w};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t h0, h1, h2, h3;
                    e4m3x4_to_f16x2(w[2 * half], h0, h1);
                    e4m3x4_to_f16x2(w[2 * half + 1], h2, h3);
                    uint4 o;
                    o.x = bf16x2_mul(f16x2_to_bf16x2_m112(h0), m);
                    o.y = bf16x2_mul(f16x2_to_bf16x2_m112(h1), m);
                    o.z = bf16x2_mul(f16x2_to_bf16x2_m112(h2), m);
                    o.w = bf16x2_mul(f16x2_to_bf16x2_m112(h3), m);
                    const int chunk = 2 * i + half;
                    *reinterpret_cast<uint4 *>(row_base + ((chunk ^ sw) << 4)) = o;
                }
            }
            return;
        }
        float s0, s1;
        e8m0x2_to_f32(r.s, s0, s1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float s = i < 2 ? s0 : s1;
            const uint32_t w[4] = {r.c[i].x, r.c[i].y, r.c[i].z, r.c[i].w};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 o;
                o.x = scaled_bf16x2(e4m3x2_to_f16x2(w[2 * half]), s);
                o.y = scaled_bf16x2(e4m3x2_to_f16x2(w[2 * half] >> 16), s);
                o.z = scaled_bf16x2(e4m3x2_to_f16x2(w[2 * half + 1]), s);
                o.w = scaled_bf16x2(e4m3x2_to_f16x2(w[2 * half + 1] >> 16), s);
                const int chunk = 2 * i + half;
                *reinterpret_cast<uint4 *>(row_base + ((chunk ^ sw) << 4)) = o;
            }
        }
    } else {
        // per 16-element quarter: the bf16x2 multiplier (fast path) or fp32 scale
        uint32_t mul[4];
        bool fast;
        if constexpr (FMT == FMT_NVFP4) {
            // E4M3 scale s: bf16(s * 2^112) is exact (4 significant bits); NaN codes are 0x7F / 0xFF
            fast = ((r.s & 0x7F7F7F7Fu) + 0x01010101u & 0x80808080u) == 0u;  // no byte is S.1111.111
            const uint32_t a = e4m3x2_to_f16x2(r.s), b = e4m3x2_to_f16x2(r.s >> 16);
            const uint32_t a2 = f16x2_to_bf16x2_m112(a), b2 = f16x2_to_bf16x2_m112(b);
            // f16x2_to_bf16x2_m112 gives s * 2^-112: square the shift away with 2^224 as two 2^112 factors
            const uint32_t p112 = bf16x2_pow2_m15(127);  // 2^112
            const uint32_t as = bf16x2_mul(bf16x2_mul(a2, p112), p112);
            const uint32_t bs = bf16x2_mul(bf16x2_mul(b2, p112), p112);
            mul[0] = (as & 0xFFFFu) | (as << 16);
            mul[1] = (as >> 16) | (as & 0xFFFF0000u);
            mul[2] = (bs & 0xFFFFu) | (bs << 16);
            mul[3] = (bs >> 16) | (bs & 0xFFFF0000u);
        } else {
            const uint32_t e0 = r.s & 0xFFu, e1 = (r.s >> 8) & 0xFFu;
            fast = e0 - 2u <= 140u && e1 - 2u <= 140u;  // 2 <= e <= 142: products normal bf16
            mul[0] = mul[1] = bf16x2_pow2_m15((int)e0);
            mul[2] = mul[3] = bf16x2_pow2_m15((int)e1);
        }
        if (fast) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t w[4] = {r.c[i].x, r.c[i].y, r.c[i].z, r.c[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // word j of 16-byte half i: elements 32i + 8j .. +7 (16-element block 2i + j/2)
                    const uint32_t m = mul[2 * i + (j >> 1)];
                    uint32_t h0, h1, h2, h3;
                    e2m1x8_to_f16x2(w[j], h0, h1, h2, h3);
                    uint4 o;
                    o.x = bf16x2_mul(f16x2_to_bf16x2_m112(h0), m);
                    o.y = bf16x2_mul(f16x2_to_bf16x2_m112(h1), m);
                    o.z = bf16x2_mul(f16x2_to_bf16x2_m112(h2), m);
                    o.w = bf16x2_mul(f16x2_to_bf16x2_m112(h3), m);
                    const int chunk = 4 * i + j;
                    *reinterpret_cast<uint4 *>(row_base + ((chunk ^ sw) << 4)) = o;
                }
            }
            return;
        }
        float sc[4];
        if constexpr (FMT == FMT_NVFP4) {
            const uint32_t a = e4m3x2_to_f16x2(r.s), b = e4m3x2_to_f16x2(r.s >> 16);
            sc[0] = f16_lo_to_f32(a);
            sc[1] = f16_hi_to_f32(a);
            sc[2] = f16_lo_to_f32(b);
            sc[3] = f16_hi_to_f32(b);
        } else {
            e8m0x2_to_f32(r.s, sc[0], sc[2]);
            sc[1] = sc[0];
            sc[3] = sc[2];
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t w[4] = {r.c[i].x, r.c[i].y, r.c[i].z, r.c[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float s = sc[2 * i + (j >> 1)];
                uint4 o;
                o.x = scaled_bf16x2(e2m1x2_to_f16x2(w[j]), s);
                o.y = scaled_bf16x2(e2m1x2_to_f16x2(w[j] >> 8), s);
                o.z = scaled_bf16x2(e2m1x2_to_f16x2(w[j] >> 16), s);
                o.w = scaled_bf16x2(e2m1x2_to_f16x2(w[j] >> 24), s);
                const int chunk = 4 * i + j;
                *reinterpret_cast<uint4 *>(row_base + ((chunk ^ sw) << 4)) = o;
            }
        }
    }
}

// ------------------------------------------------------------ kernel

struct QmmArgs {
    const uint8_t *codes;
    const uint8_t *scales;
    uint16_t *Y;
    int *err;
    int M, N, K;
    unsigned long long wait_ns;
};

template <int FMT>
__global__ void __launch_bounds__(QMM_THREADS, 1) qmm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                             const __grid_constant__ CUtensorMap tmap_c, QmmArgs a)
{
    using QG = QmmGeo<FMT>;
    constexpr int QMM_STAGE_BYTES = QG::STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + QMM_STAGES * QMM_STAGE_BYTES);
    uint64_t *full_a = bars;                    // [STAGES] TMA bytes landed
    uint64_t *full_b = bars + QMM_STAGES;       // [STAGES] decoded tile stored (8 warps)
    uint64_t *empty = bars + 2 * QMM_STAGES;    // [STAGES] MMAs that read the stage finished
    uint64_t *acc_full = bars + 3 * QMM_STAGES; // accumulators complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * QMM_STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (a.M + QMM_BM - 1) / QMM_BM;
    const int m0 = (blockIdx.x % m_tiles) * QMM_BM;
    const int n0 = (blockIdx.x / m_tiles) * QMM_BN;
    const int KB = a.K / QMM_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < QMM_STAGES; ++s) {
            mbar_init(&full_a[s], 1);
            mbar_init(&full_b[s], 8);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();
    pdl_wait();  // X and Y may be used by the neighbouring kernels

    int issued_a = 0;  // producer: stages whose TMA was issued
    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % QMM_STAGES;
                if (kb >= QMM_STAGES && !mbar_wait(&empty[s], ((kb / QMM_STAGES) - 1) & 1, abort_flag, a.wait_ns))
                    break;
                uint8_t *st = smem + s * QMM_STAGE_BYTES;
                mbar_arrive_expect_tx(&full_a[s], 2 * QMM_A_BYTES + QG::C_BYTES);
                tma_load_2d(st, &tmap_x, kb * QMM_BK, m0, &full_a[s]);
                tma_load_2d(st + QMM_A_BYTES, &tmap_x, kb * QMM_BK, m0 + 128, &full_a[s]);
                if constexpr (QG::TMA_CODES)  // 256 weight rows x 32 code bytes
                    tma_load_2d(st + 2 * QMM_A_BYTES + QMM_B_BYTES, &tmap_c, kb * 32, n0, &full_a[s]);
                issued_a = kb + 1;
            }
            // drain: every issued TMA must land before the CTA may exit
            for (int kb = (issued_a > QMM_STAGES ? issued_a - QMM_STAGES : 0); kb < issued_a; ++kb)
                mbar_wait(&full_a[kb % QMM_STAGES], (kb / QMM_STAGES) & 1, abort_flag, a.wait_ns, false);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = qmm_idesc();
            int done = 0;
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % QMM_STAGES;
                const uint32_t ph = (kb / QMM_STAGES) & 1;
                if (!mbar_wait(&full_a[s], ph, abort_flag, a.wait_ns)) break;
                if (!mbar_wait(&full_b[s], ph, abort_flag, a.wait_ns)) break;
                tc_fence_after();
                const uint32_t sa0 = smem_u32(smem + s * QMM_STAGE_BYTES);
                const uint32_t sa1 = sa0 + QMM_A_BYTES;
                const uint32_t sb = sa0 + 2 * QMM_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < QMM_BK / 16; ++kk) {
                    const uint64_t bd = sw128_desc(sb + kk * 32);
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                    umma_bf16(tmem, sw128_desc(sa0 + kk * 32), bd, idesc, acc);
                    umma_bf16(tmem + QMM_BN, sw128_desc(sa1 + kk * 32), bd, idesc, acc);
                }
                umma_commit(&empty[s]);
                done = kb + 1;
            }
            umma_commit(acc_full);  // fires once every MMA issued so far has completed
            (void)done;
        }
    } else {
        // ---------------- decoders (warps 2..9), one weight row per thread
        const int d = threadIdx.x - 64;  // 0..255
        const int n = n0 + d;
        const size_t rb = FMT == FMT_MXFP8 ? (size_t)a.K : (size_t)a.K / 2;
        const size_t sb = FMT == FMT_NVFP4 ? (size_t)(a.K / 16) : (size_t)(a.K / 32);
        const uint8_t *crow = a.codes + (size_t)n * rb;
        const uint8_t *srow = a.scales + (size_t)n * sb;
        if constexpr (QG::TMA_CODES) {
            // codes arrive by TMA with the stage; the scale bytes of the next
            // QMM_PF k-blocks stay in flight in registers
            constexpr int SPK = FMT == FMT_NVFP4 ? 4 : 2;  // scale bytes per k-block
            uint32_t sv[QMM_PF];
#pragma unroll
            for (int j = 0; j < QMM_PF; ++j)
                if (j < KB) sv[j] = SPK == 4 ? ld_nc_u32(srow + 4 * j) : ld_nc_u16(srow + 2 * j);
            for (int kb0 = 0; kb0 < KB; kb0 += QMM_PF) {
#pragma unroll
                for (int j = 0; j < QMM_PF; ++j) {
                    const int kb = kb0 + j;
                    if (kb >= KB) break;
                    const int s = kb % QMM_STAGES;
                    // the stage's TMA was issued after the MMAs released it, so its
                    // arrival also means the decoded-tile slot is free
                    if (!mbar_wait(&full_a[s], (kb / QMM_STAGES) & 1, abort_flag, a.wait_ns)) goto decode_done;
                    uint8_t *stage = smem + s * QMM_STAGE_BYTES;
                    const uint4 *cp = reinterpret_cast<const uint4 *>(stage + 2 * QMM_A_BYTES + QMM_B_BYTES + d * 32);
                    QRow<FMT> rr;
                    rr.c[0] = cp[0];
                    rr.c[1] = cp[1];
                    rr.s = sv[j];
                    if (kb + QMM_PF < KB)
                        sv[j] = SPK == 4 ? ld_nc_u32(srow + 4 * (kb + QMM_PF)) : ld_nc_u16(srow + 2 * (kb + QMM_PF));
                    qrow_store<FMT>(rr, stage + 2 * QMM_A_BYTES + d * 128, d);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full_b[s]);
                }
            }
        } else {
            // codes and scales of the next QMM_PF k-blocks stay in flight in registers
            QRow<FMT> r[QMM_PF];
#pragma unroll
            for (int j = 0; j < QMM_PF; ++j)
                if (j < KB) qrow_load<FMT>(crow, srow, j, r[j]);
            for (int kb0 = 0; kb0 < KB; kb0 += QMM_PF) {
#pragma unroll
                for (int j = 0; j < QMM_PF; ++j) {
                    const int kb = kb0 + j;
                    if (kb >= KB) break;
                    const int s = kb % QMM_STAGES;
                    if (kb >= QMM_STAGES &&
                        !mbar_wait(&empty[s], ((kb / QMM_STAGES) - 1) & 1, abort_flag, a.wait_ns))
                        goto decode_done;
                    uint8_t *b_tile = smem + s * QMM_STAGE_BYTES + 2 * QMM_A_BYTES;
                    qrow_store<FMT>(r[j], b_tile + d * 128, d);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full_b[s]);
                    if (kb + QMM_PF < KB) qrow_load<FMT>(crow, srow, kb + QMM_PF, r[j]);
                }
            }
        }
    decode_done:;
    }

    // ---------------- epilogue (decoder warps): TMEM -> bf16 -> Y
    if (warp >= 2) {
        // the MMAs must have finished (even on abort) before TMEM is read or freed
        const bool ok = mbar_wait(acc_full, 0, abort_flag, a.wait_ns, false) && !*abort_flag;
        tc_fence_after();
        const int half = warp < 6 ? 0 : 1;      // accumulator (M half)
        const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
        const int m = m0 + half * 128 + quarter * 32 + lane;
        float g = 1.0f;
        if (FMT == FMT_NVFP4) g = load_f32_unaligned(a.scales + (size_t)a.N * (a.K / 16));
        uint16_t *yrow = a.Y + (size_t)m * a.N + n0;
        const bool store = m < a.M;  // rows past M were zero-filled by TMA
        for (int c = 0; c < QMM_BN; c += 32) {
            uint32_t v[32];
            if (ok) {
                tmem_ld32(tmem + half * QMM_BN + c + ((uint32_t)(quarter * 32) << 16), v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0x7FC00000u;
            }
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float lo = __uint_as_float(v[2 * i]), hi = __uint_as_float(v[2 * i + 1]);
                if (FMT == FMT_NVFP4) {
                    lo = __fmul_rn(lo, g);
                    hi = __fmul_rn(hi, g);
                }
                o[i] = f32x2_to_bf16x2(lo, hi);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(yrow + c);
            if (store) {
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) set_device_error(a.err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// ------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

template <int FMT>
static cudaError_t run_qmm(const DeviceState &ds, cudaStream_t st, const CUtensorMap &map, const CUtensorMap &cmap,
                           const QmmArgs &a)
{
    using QG = QmmGeo<FMT>;
    if (QG::SMEM > ds.max_smem_optin) return cudaErrorInvalidValue;
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(qmm_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, QG::SMEM);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    const int grid = ((a.M + QMM_BM - 1) / QMM_BM) * (a.N / QMM_BN);
    return launch_k(qmm_kernel<FMT>, dim3(grid), dim3(QMM_THREADS), (size_t)QG::SMEM, st, map, cmap, a);
}

cudaError_t launch_qmm(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *X, uint16_t *Y, int M, int N, int K)
{
    if (N % QMM_BN != 0 || K % QMM_BK != 0) return cudaErrorInvalidValue;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)QMM_BK, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(X), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // packed codes of the 4-bit formats: [N][K/2] bytes, box of 32 bytes x 256 rows
    CUtensorMap cmap;
    if (fmt != FMT_MXFP8) {
        const cuuint64_t cdims[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
        const cuuint64_t cstrides[1] = {(cuuint64_t)K / 2};
        const cuuint32_t cbox[2] = {32u, (cuuint32_t)QMM_BN};
        r = enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), cdims, cstrides, cbox, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    } else {
        cmap = map;  // unused
    }
    QmmArgs a;
    a.codes = codes;
    a.scales = scales;
    a.Y = Y;
    a.err = ds.err;
    a.M = M;
    a.N = N;
    a.K = K;
    a.wait_ns = QMM_WAIT_NS;
    if (fmt == FMT_MXFP4) return run_qmm<FMT_MXFP4>(ds, st, map, cmap, a);
    if (fmt == FMT_MXFP8) return run_qmm<FMT_MXFP8>(ds, st, map, cmap, a);
    return run_qmm<FMT_NVFP4>(ds, st, map, cmap, a);
}

}  // namespace mx
