// mx_qmm_bs.cu -- prefill GEMM over block-float activations and weights on
// the block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4 / mxf4 /
// mxf4nvf4), sm_103a; and the tensor pipe's dense peak per MMA kind.
//
//   Y[m][n] = bf16_rne( sum_k Xq[m][k] * W[n][k] ),  fp32 accumulation,
//
// where Xq holds block-float activations in the weights' format (the output
// of mx_quantize) and both operands keep their codes and block scales: the
// tensor core multiplies the codes and applies the scales itself, so nothing
// is decoded.  The pages quantise block-float on Blackwell with the hardware
// NVFP4 / MXFP4 converter (manual page "Building from source", CUDA build
// options, "GPU architecture auto-detection"); talk slide 8 sets FP4 on
// Blackwell tensor cores against software decode elsewhere.
//
// One CTA owns a 128 x BN output tile (BN = 128 or 256) and streams K in
// k-blocks of 128 bytes per row (128 MXFP8 elements, 256 MXFP4 / NVFP4):
//   warp 0      X and W codes of a k-block by TMA (128-byte swizzle) into a
//               ring of shared-memory stages
//   warp 1      allocates tensor memory; one thread issues 4 MMAs per k-block
//               (K = 32 for MXFP8, 64 for the 4-bit formats) and commits each
//               k-block to the stage's and the scale slot's empty barriers
//               and, every 16 / (scale bytes per row per k-block) k-blocks,
//               the X and W block scales of the next k-blocks as 16 bytes per
//               row (TMA, into a ring of scale stages)
//   warps 2-5   block scales: each warp reads the scale bytes of its rows
//               from a scale stage (contiguous 16-byte loads) and writes them
//               to a ring of scale slots in tensor memory (tcgen05.st), one
//               slot per k-block; then the epilogue:
//               tcgen05.ld of its accumulator lanes, NVFP4 tensor scales,
//               round to bf16, store.
// Scale layout in tensor memory: a 128-row chunk of scales covers 4 scale
// blocks along K (one byte each in a 32-bit cell, the MMA's scale-factor ID
// picks the byte) and takes 4 columns.  X (operand A): row r at lane r,
// column r / 32 of the chunk (each 32-lane quarter of the tensor core reads
// its own rows); the bytes are written to all 4 columns.  W (operand B):
// every lane quarter reads the scales of all the tile's W rows, so row n is
// at lane n % 32, column n / 32 of the chunk, in each of the 4 quarters
// (measured: with W rows at lane n the products were right only where the
// output row and column fell in the same quarter).  A 256-row W tile takes
// two chunks in consecutive column groups.  Every wait is bounded (two seconds of
// %globaltimer); a wait that gives up sets MX_DEVERR_TIMEOUT, the CTA drains
// its copies in flight, writes NaN and returns.
#include "../../include/mx.h"
#include "mx_internal.h"
#include "mx_tc.cuh"

namespace mx {

constexpr unsigned long long BS_WAIT_NS = 2000000000ull;
constexpr int BS_KB_BYTES = 128;  // code bytes per row per k-block
constexpr int BS_SMEM_LIMIT = 232448;

// ------------------------------------------------------------ primitives

__device__ __forceinline__ void umma1_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st_x4v(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
                 "r"(v2), "r"(v3)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// MMA kinds: the three block-scaled ones of the formats, plus the unscaled
// bf16 and E4M3 kinds for the peak measurement.
enum : int { BSK_BF16 = 0, BSK_E4M3 = 1, BSK_MXF8 = 2, BSK_MXF4 = 3, BSK_NVF4 = 4 };

template <int KIND>
__device__ __forceinline__ void umma1(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                      uint32_t acc)
{
    if constexpr (KIND == BSK_BF16) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(idesc), "r"(acc)
                     : "memory");
    } else if constexpr (KIND == BSK_E4M3) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(idesc), "r"(acc)
                     : "memory");
    } else if constexpr (KIND == BSK_MXF8) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], "
                     "p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
                     : "memory");
    } else if constexpr (KIND == BSK_MXF4) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], "
                     "p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
                     : "memory");
    } else {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
                     "p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
                     : "memory");
    }
}

// Instruction descriptor for M = 128, N = n, K-major A and B.
//   unscaled kinds: D format fp32 (bits 4-5 = 1), A / B formats at 7 / 10
//     (bf16 = 1 in kind::f16; E4M3 = 0 in kind::f8f6f4)
//   block-scaled kinds: scale-factor IDs of B (bits 4-5) and A (29-30), A / B
//     formats (E4M3 = 0 in kind::mxf8f6f4, E2M1 = 1 in kind::mxf4 and
//     kind::mxf4nvf4), scale type at bit 23 (1 = UE8M0, 0 = UE4M3)
//   N / 8 at bits 17-22, M / 16 at 24-28.
template <int KIND>
__host__ __device__ constexpr uint32_t bs_idesc(int n, uint32_t sfa_id = 0, uint32_t sfb_id = 0)
{
    const uint32_t shape = ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    if (KIND == BSK_BF16) return (1u << 4) | (1u << 7) | (1u << 10) | shape;
    if (KIND == BSK_E4M3) return (1u << 4) | shape;
    const uint32_t fmt = KIND == BSK_MXF8 ? 0u : 1u;
    const uint32_t ue8m0 = KIND == BSK_NVF4 ? 0u : 1u;
    return (sfb_id << 4) | (fmt << 7) | (fmt << 10) | (ue8m0 << 23) | shape | (sfa_id << 29);
}

// ------------------------------------------------------------ peak

// Operand stages of the microbenchmark: A 128 rows x 128 B, then B 256 rows
// x 128 B (48 KB); four of them.
constexpr int PEAK_STAGE = (128 + 256) * 128;
constexpr int PEAK_STAGES = 4;

// One CTA per SM issues `iters` k-blocks of 4 MMAs of 128 x 256 x K on
// shared-memory operands into tensor memory, block scales 1.0 for the scaled
// kinds: the dense rate of the tensor pipe for that kind.  Mode bits `fill`
// (the kind's bits 8-11, see mx_mma_peak): 1 random finite operands instead
// of zeros; 2 the MMAs rotate through the stages (3 when 4 is set) instead of
// using one; 4 warps 1-3 meanwhile store 16-byte vectors into the fourth
// stage at full rate; 8 they store into unused tensor-memory columns
// instead.  A wait that runs past 10 s sets the error word.
template <int KIND>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int fill, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *a = smem;              // 128 rows x 128 B
    uint8_t *b = smem + 128 * 128;  // 256 rows x 128 B
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + PEAK_STAGES * PEAK_STAGE);
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(slot + 1);
    const int warp = threadIdx.x >> 5;
    // operands: zeros, or (fill) hashed bits kept finite for the kind (bf16
    // magnitudes below 1, E4M3 without its NaN code and the sign, any FP4 code)
    const uint32_t keep = KIND == BSK_BF16 ? 0x3F7F3F7Fu : (KIND <= BSK_MXF8 ? 0x77777777u : 0xFFFFFFFFu);
    for (int i = threadIdx.x; i < PEAK_STAGES * PEAK_STAGE / 16; i += blockDim.x) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (fill & 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t h = (uint32_t)(4 * i + j) * 0x9E3779B1u + 0x7F4A7C15u;
                h ^= h >> 15;
                h *= 0x2C1B3C6Du;
                h ^= h >> 12;
                w[j] = h & keep;
            }
        }
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if constexpr (KIND >= BSK_MXF8) {
        // scales 1.0 in columns 256 .. 271 (each warp its lane quarter)
        const uint32_t one = KIND == BSK_NVF4 ? 0x38383838u : 0x7F7F7F7Fu;
        for (int c = 0; c < 16; c += 4) tmem_st_x4(tmem + ((uint32_t)(32 * warp) << 16) + 256u + (uint32_t)c, one);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp >= 1 && (fill & 12)) {
        // traffic beside the MMAs: shared-memory stores into the last stage,
        // or tensor-memory stores into columns 264-503 (the warp's lanes)
        const uint32_t lane = threadIdx.x & 31;
        if (fill & 4) {
            uint4 *dst = reinterpret_cast<uint4 *>(smem + (PEAK_STAGES - 1) * PEAK_STAGE);
            for (int i = 0; i < iters * 32; ++i)
                dst[(i * 96 + (warp - 1) * 32 + (int)lane) % (PEAK_STAGE / 16)] = make_uint4((uint32_t)i, lane, 0u, 0u);
        } else {
            for (int i = 0; i < iters * 16; ++i)
                tmem_st_x4(tmem + ((uint32_t)(32 * warp) << 16) + 264u + (uint32_t)((i * 4) % 240), (uint32_t)i);
            tmem_wait_st();
        }
    }
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = bs_idesc<KIND>(256);
        const uint32_t sa0 = smem_u32(a), sb0 = smem_u32(b);
        const int nst = (fill & 2) ? ((fill & 4) ? PEAK_STAGES - 1 : PEAK_STAGES) : 1;
        for (int i = 0; i < iters; ++i) {
            const uint32_t so = (uint32_t)(i % nst) * (uint32_t)PEAK_STAGE;
            const uint32_t sa = sa0 + so, sb = sb0 + so;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma1<KIND>(tmem, sw128_desc(sa + 32 * kk), sw128_desc(sb + 32 * kk), idesc, tmem + 256u, tmem + 260u,
                            (i | kk) != 0);
        }
        umma1_commit(bar);
        if (!mbar_wait(bar, 0, abort_flag, 10000000000ull, false)) set_device_error(err, DEVERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

// K of one MMA for each kind.
__host__ __device__ constexpr int mma_k(int kind) { return kind == BSK_BF16 ? 16 : kind <= BSK_MXF8 ? 32 : 64; }

template <int KIND>
static cudaError_t run_peak(const DeviceState &ds, cudaStream_t st, int iters, int fill, float *ms)
{
    // more shared memory than two CTAs could share: one CTA (and one
    // tensor-memory allocation) per SM
    const size_t smem = PEAK_STAGES * PEAK_STAGE + 2048;
    cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaEvent_t e0, e1;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess) return e;
    if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
        cudaEventDestroy(e0);
        return e;
    }
    e = cudaEventRecord(e0, st);
    if (e == cudaSuccess) e = launch_k(mma_peak_kernel<KIND>, dim3(ds.num_sms), dim3(128), smem, st, iters, fill, ds.err);
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return e;
}

// ------------------------------------------------------------ GEMM

template <int FMT>
struct BsFmt {
    static constexpr int KIND = FMT == FMT_MXFP8 ? BSK_MXF8 : FMT == FMT_MXFP4 ? BSK_MXF4 : BSK_NVF4;
    static constexpr int KB_ELEMS = FMT == FMT_MXFP8 ? 128 : 256;  // elements per k-block
    static constexpr int SPB = FMT == FMT_MXFP8 ? 4 : FMT == FMT_MXFP4 ? 8 : 16;  // scale bytes per row per k-block
    static constexpr int CH = SPB / 4;                                          // 4-byte scale chunks per k-block
    static constexpr int SG = 16 / SPB;                                         // k-blocks per 16-byte scale stage
};

template <int FMT, int BN>
struct BsGeo {
    static constexpr int A_BYTES = 128 * BS_KB_BYTES;
    static constexpr int B_BYTES = BN * BS_KB_BYTES;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int ST = 4;                                 // scale stages (16 bytes per X and W row)
    static constexpr int SC_STAGE = (128 + BN) * 16;
    static constexpr int S_FIT = (BS_SMEM_LIMIT - 2048 - ST * SC_STAGE) / STAGE;
    static constexpr int S = S_FIT > 6 ? 6 : S_FIT;
    static constexpr int RB = BN / 128;                          // 128-row chunks of W per tile
    static constexpr int SLOT_COLS = 4 * BsFmt<FMT>::CH * (1 + RB);
    // scale slots in tensor memory: the writers load a k-block's scales from
    // L2 while the MMAs work through the R - 1 slots ahead of it
    static constexpr int R = (512 - BN) / SLOT_COLS > 8 ? 8 : (512 - BN) / SLOT_COLS;
    static constexpr int TMEM_COLS = BN + R * SLOT_COLS <= 256 ? 256 : 512;
    // warps: 0 TMA, 1 MMA, 2-5 scale writers, 6-13 epilogue; at most four
    // warps per scheduler, so 128 registers a thread fit each one's file
    static constexpr int THREADS = 448;
    static constexpr int OFF_SC = S * STAGE;
    static constexpr int OFF_BAR = OFF_SC + ST * SC_STAGE;
    static constexpr int SMEM = 1024 + OFF_BAR + 512;
    static_assert((2 * S + 2 * R + 2 * ST + 2) * 8 + 8 <= 512, "barrier area");
    static_assert(BN + R * SLOT_COLS <= 512, "tensor memory");
    static_assert(SMEM <= BS_SMEM_LIMIT, "shared memory");
    static_assert(S >= 2 && R >= 2, "pipeline depth");
};

struct BsArgs {
    const uint8_t *scales;   // W block scales [N][K / block] (+ NVFP4 tensor scale)
    const uint8_t *xscales;  // X block scales [M][K / block] (+ NVFP4 tensor scale)
    uint16_t *Y;             // bf16 [M][N]
    int *err;
    int M, N, K;
    unsigned long long wait_ns;
};

// Word w (0..3) of a 16-byte vector (w a compile-time constant after
// unrolling).
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int w)
{
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

template <int FMT, int BN>
__global__ void __maxnreg__(128) qmm_bs_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                        const __grid_constant__ CUtensorMap tmap_w,
                                                        const __grid_constant__ CUtensorMap tmap_xs,
                                                        const __grid_constant__ CUtensorMap tmap_ws, BsArgs a)
{
    using G = BsGeo<FMT, BN>;
    using F = BsFmt<FMT>;
    constexpr int S = G::S, R = G::R, RB = G::RB, CH = F::CH, ST = G::ST, SG = F::SG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *scs = smem + G::OFF_SC;    // [ST] scale stages: 128 X rows then BN W rows, 16 bytes each
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + G::OFF_BAR);
    uint64_t *full = bars;              // [S] X and W codes of a stage landed (TMA bytes)
    uint64_t *empty = bars + S;         // [S] the MMAs that read the stage finished
    uint64_t *sf_full = bars + 2 * S;   // [R] the 4 scale warps wrote the slot
    uint64_t *sf_empty = sf_full + R;   // [R] the MMAs that read the slot finished
    uint64_t *sc_full = sf_full + 2 * R;  // [ST] a scale stage landed (TMA bytes)
    uint64_t *sc_empty = sc_full + ST;    // [ST] the 4 scale warps read it
    uint64_t *acc_full = sc_full + 2 * ST;  // the MMAs of a tile completed
    uint64_t *acc_empty = acc_full + 1;     // the 8 epilogue warps read the accumulator
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (a.M + 127) / 128;
    const int tiles = m_tiles * (a.N / BN);
    const int KB = a.K / F::KB_ELEMS;
    const int nsc = (KB + SG - 1) / SG;  // scale stages per tile
    // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ... (consecutive
    // tiles share a W column block, read by neighbouring CTAs at once)
    const int my_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile_m0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) % m_tiles * 128; };
    auto tile_n0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) / m_tiles * BN; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&sf_full[r], 4);
            mbar_init(&sf_empty[r], 1);
        }
        for (int u = 0; u < ST; ++u) {
            mbar_init(&sc_full[u], 1);
            mbar_init(&sc_empty[u], 4);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(G::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sf_col0 = (uint32_t)BN;  // scale slots follow the accumulator columns
    pdl_trigger();
    pdl_wait();  // the activations (and their scales) come from the previous kernel

    if (warp == 0) {
        // ---------------- codes and scales producer, across the CTA's tiles
        if (lane == 0) {
            int issued = 0, sissued = 0;  // k-blocks and scale stages issued, counted over tiles
            bool go = true;
            for (int i = 0; i < my_tiles && go; ++i) {
                const int m0 = tile_m0(i), n0 = tile_n0(i);
                for (int kb = 0; kb < KB; ++kb) {
                    const int g = i * KB + kb, s = g % S;
                    if (kb % SG == 0) {
                        // the scale stage of k-blocks kb .. kb + SG - 1
                        const int t = i * nsc + kb / SG, u = t % ST;
                        if (t >= ST && !mbar_wait(&sc_empty[u], ((t / ST) - 1) & 1, abort_flag, a.wait_ns)) {
                            go = false;
                            break;
                        }
                        uint8_t *sc = scs + u * G::SC_STAGE;
                        mbar_arrive_expect_tx(&sc_full[u], (uint32_t)G::SC_STAGE);
                        tma_load_2d(sc, &tmap_xs, 16 * (kb / SG), m0, &sc_full[u]);
                        tma_load_2d(sc + 128 * 16, &tmap_ws, 16 * (kb / SG), n0, &sc_full[u]);
                        sissued = t + 1;
                    }
                    if (g >= S && !mbar_wait(&empty[s], ((g / S) - 1) & 1, abort_flag, a.wait_ns)) {
                        go = false;
                        break;
                    }
                    uint8_t *st = smem + s * G::STAGE;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)G::STAGE);
                    tma_load_2d(st, &tmap_x, kb * BS_KB_BYTES, m0, &full[s]);
                    tma_load_2d(st + G::A_BYTES, &tmap_w, kb * BS_KB_BYTES, n0, &full[s]);
                    issued = g + 1;
                }
            }
            // every issued load must land before the CTA may exit
            for (int g = (issued > S ? issued - S : 0); g < issued; ++g)
                mbar_wait(&full[g % S], (g / S) & 1, abort_flag, BS_WAIT_NS, false);
            for (int t = (sissued > ST ? sissued - ST : 0); t < sissued; ++t)
                mbar_wait(&sc_full[t % ST], (t / ST) & 1, abort_flag, BS_WAIT_NS, false);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: a tile's k-blocks into the accumulator once
        // the epilogue has read the previous tile out of it
        if (lane == 0) {
            bool go = true;
            for (int i = 0; i < my_tiles && go; ++i) {
                if (i > 0 && !mbar_wait(acc_empty, (i - 1) & 1, abort_flag, a.wait_ns)) {
                    go = false;
                    break;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    const int g = i * KB + kb, s = g % S, r = g % R;
                    if (!mbar_wait(&full[s], (g / S) & 1, abort_flag, a.wait_ns) ||
                        !mbar_wait(&sf_full[r], (g / R) & 1, abort_flag, a.wait_ns)) {
                        go = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * G::STAGE), sb = sa + G::A_BYTES;
                    const uint32_t sfa = tmem + sf_col0 + (uint32_t)(r * G::SLOT_COLS);
                    const uint32_t sfb = sfa + (uint32_t)(4 * CH);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // the scale chunk and byte of MMA kk: MXFP8 one 32-element block
                        // (chunk 0, byte kk); MXFP4 two (chunk kk / 2, bytes 2 (kk % 2)
                        // and up); NVFP4 four 16-element blocks (chunk kk, byte 0)
                        const int c = FMT == FMT_MXFP8 ? 0 : FMT == FMT_MXFP4 ? kk >> 1 : kk;
                        const uint32_t id = FMT == FMT_MXFP8 ? (uint32_t)kk : FMT == FMT_MXFP4 ? 2u * (kk & 1) : 0u;
                        const uint32_t idesc = bs_idesc<F::KIND>(BN, id, id);
                        umma1<F::KIND>(tmem, sw128_desc(sa + 32 * kk), sw128_desc(sb + 32 * kk), idesc,
                                       sfa + (uint32_t)(4 * c), sfb + (uint32_t)(4 * c * RB), (kb | kk) != 0);
                    }
                    umma1_commit(&empty[s]);
                    umma1_commit(&sf_empty[r]);
                }
                if (go) umma1_commit(acc_full);  // fires once the tile's MMAs have completed
            }
            // after giving up: let the epilogue see the MMAs issued so far
            // complete (it writes NaN) before the tensor memory is released
            if (!go) umma1_commit(acc_full);
        }
    } else if (warp < 6) {
        // ---------------- scale writers (warps 2-5: lane quarter q = warp % 4)
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        bool go = true;
        for (int i = 0; i < my_tiles && go; ++i) {
            for (int tl = 0; tl < nsc && go; ++tl) {
                const int t = i * nsc + tl, u = t % ST;
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&sc_full[u], (t / ST) & 1, abort_flag, a.wait_ns);
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                    go = false;
                    break;
                }
                // X row 32 q + lane; W rows 128 j + 32 i + lane (the same in every warp)
                const uint8_t *sc = scs + u * G::SC_STAGE;
                const uint4 xv = *reinterpret_cast<const uint4 *>(sc + 16 * (32 * q + lane));
                uint4 wv[RB][4];
#pragma unroll
                for (int j = 0; j < RB; ++j)
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii)
                        wv[j][ii] = *reinterpret_cast<const uint4 *>(sc + 16 * (128 + 128 * j + 32 * ii + lane));
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc_empty[u]);
#pragma unroll
                for (int jj = 0; jj < SG; ++jj) {
                    const int kb = tl * SG + jj;
                    if (kb >= KB) break;
                    const int g = i * KB + kb, r = g % R;
                    if (lane == 0 && g >= R) ok = mbar_wait(&sf_empty[r], ((g / R) - 1) & 1, abort_flag, a.wait_ns);
                    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                        go = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = tmem + lane_base + sf_col0 + (uint32_t)(r * G::SLOT_COLS);
#pragma unroll
                    for (int c = 0; c < CH; ++c) {
                        const int w = jj * CH + c;  // word of the 16 bytes
                        tmem_st_x4(base + (uint32_t)(4 * c), word_of(xv, w));
#pragma unroll
                        for (int j = 0; j < RB; ++j)
                            tmem_st_x4v(base + (uint32_t)(4 * CH + 4 * (c * RB + j)), word_of(wv[j][0], w),
                                        word_of(wv[j][1], w), word_of(wv[j][2], w), word_of(wv[j][3], w));
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sf_full[r]);
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 6-13: lane quarter q = warp % 4,
        // column half h): the warp's half tile row is read out of tensor
        // memory into registers (bf16) and the accumulator handed back
        // before the stores, so the next tile's MMAs overlap them
        const int q = warp & 3, h = (warp - 6) >> 2;
        constexpr int HC = BN / 2;  // columns per warp
        float g = 1.0f;
        if (FMT == FMT_NVFP4) {
            g = load_f32_unaligned(a.scales + (size_t)a.N * (a.K / 16));
            g = __fmul_rn(g, load_f32_unaligned(a.xscales + (size_t)a.M * (a.K / 16)));
        }
        bool live = true;
        for (int i = 0; i < my_tiles; ++i) {
            const int row = tile_m0(i) + 32 * q + lane, n0 = tile_n0(i) + h * HC;
            if (live) live = mbar_wait(acc_full, i & 1, abort_flag, BS_WAIT_NS, false) && !*abort_flag;
            uint32_t o[HC / 2];
            if (live) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < HC / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HC + 32 * c), v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float lo = __uint_as_float(v[2 * j]), hi = __uint_as_float(v[2 * j + 1]);
                        if (FMT == FMT_NVFP4) {
                            lo = __fmul_rn(lo, g);
                            hi = __fmul_rn(hi, g);
                        }
                        o[16 * c + j] = f32x2_to_bf16x2(lo, hi);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            } else {
#pragma unroll
                for (int j = 0; j < HC / 2; ++j) o[j] = 0x7FC07FC0u;  // a call that gave up writes NaN
            }
            if (row < a.M) {
                uint4 *dst = reinterpret_cast<uint4 *>(a.Y + (size_t)row * a.N + n0);
#pragma unroll
                for (int j = 0; j < HC / 8; ++j)
                    dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) set_device_error(a.err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G::TMEM_COLS)
                     : "memory");
    }
}

// Codes as [rows][row bytes] uint8 with boxes of one k-block (128 bytes) x
// box_rows rows, 128-byte swizzle; rows past `rows` read as zero.
static cudaError_t encode_codes_map(const uint8_t *codes, long long rows, long long row_bytes, int box_rows,
                                    CUtensorMap &map)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)BS_KB_BYTES, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Block scales as [rows][scale bytes per row] uint8 with boxes of 16 bytes x
// box_rows rows, no swizzle; rows past `rows` read as zero.
static cudaError_t encode_scales_map(const uint8_t *scales, long long rows, long long row_bytes, int box_rows,
                                     CUtensorMap &map)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {16u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(scales), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int FMT, int BN>
static cudaError_t run_qmm_bs(const DeviceState &ds, cudaStream_t st, const uint8_t *codes, const uint8_t *scales,
                              const uint8_t *xcodes, const uint8_t *xscales, uint16_t *Y, int M, int N, int K)
{
    using G = BsGeo<FMT, BN>;
    if (G::SMEM > ds.max_smem_optin) return cudaErrorInvalidValue;
    const long long row_bytes = FMT == FMT_MXFP8 ? K : K / 2;
    const long long srow_bytes = K / (FMT == FMT_NVFP4 ? 16 : 32);
    CUtensorMap xmap, wmap, xsmap, wsmap;
    cudaError_t e = encode_codes_map(xcodes, M, row_bytes, 128, xmap);
    if (e != cudaSuccess) return e;
    if ((e = encode_codes_map(codes, N, row_bytes, BN, wmap)) != cudaSuccess) return e;
    if ((e = encode_scales_map(xscales, M, srow_bytes, 128, xsmap)) != cudaSuccess) return e;
    if ((e = encode_scales_map(scales, N, srow_bytes, BN, wsmap)) != cudaSuccess) return e;
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        e = cudaFuncSetAttribute(qmm_bs_kernel<FMT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    BsArgs a;
    a.scales = scales;
    a.xscales = xscales;
    a.Y = Y;
    a.err = ds.err;
    a.M = M;
    a.N = N;
    a.K = K;
    a.wait_ns = BS_WAIT_NS;
    // persistent CTAs, one per SM, each taking every num_sms-th tile
    const int tiles = ((M + 127) / 128) * (N / BN);
    const int ctas = tiles < ds.num_sms ? tiles : ds.num_sms;
    return launch_k(qmm_bs_kernel<FMT, BN>, dim3(ctas), dim3(G::THREADS), (size_t)G::SMEM, st, xmap, wmap, xsmap,
                    wsmap, a);
}

}  // namespace mx

using namespace mx;

extern "C" int mx_qmm_qx(int fmt, const void *codes, const void *scales, const void *xcodes, const void *xscales,
                         void *Y, int M, int N, int K)
{
    if (fmt != MX_FMT_MXFP4 && fmt != MX_FMT_MXFP8 && fmt != MX_FMT_NVFP4) return MX_EUNSUPPORTED;
    if (!codes || !scales || !xcodes || !xscales || !Y) return MX_EINVAL;
    if (M <= 0 || N <= 0 || K <= 0 || K % (fmt == MX_FMT_NVFP4 ? 16 : 32) != 0) return MX_EINVAL;
    // whole k-blocks, and scale rows whose byte stride the scale TMA can take
    // (a multiple of 16 bytes)
    if (N % 128 != 0 || K % (fmt == MX_FMT_NVFP4 ? 256 : 512) != 0) return MX_EUNSUPPORTED;
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(codes) || !a16(scales) || !a16(xcodes) || !a16(xscales) || !a16(Y)) return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    cudaStream_t st = current_stream();
    const uint8_t *c = static_cast<const uint8_t *>(codes), *s = static_cast<const uint8_t *>(scales);
    const uint8_t *xc = static_cast<const uint8_t *>(xcodes), *xs = static_cast<const uint8_t *>(xscales);
    uint16_t *y = static_cast<uint16_t *>(Y);
    cudaError_t e;
    const bool wide = N % 256 == 0;
    if (fmt == MX_FMT_MXFP8)
        e = wide ? run_qmm_bs<FMT_MXFP8, 256>(*ds, st, c, s, xc, xs, y, M, N, K)
                 : run_qmm_bs<FMT_MXFP8, 128>(*ds, st, c, s, xc, xs, y, M, N, K);
    else if (fmt == MX_FMT_MXFP4)
        e = wide ? run_qmm_bs<FMT_MXFP4, 256>(*ds, st, c, s, xc, xs, y, M, N, K)
                 : run_qmm_bs<FMT_MXFP4, 128>(*ds, st, c, s, xc, xs, y, M, N, K);
    else
        e = wide ? run_qmm_bs<FMT_NVFP4, 256>(*ds, st, c, s, xc, xs, y, M, N, K)
                 : run_qmm_bs<FMT_NVFP4, 128>(*ds, st, c, s, xc, xs, y, M, N, K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return e == cudaSuccess ? MX_OK : MX_ECUDA;
}

extern "C" int mx_mma_peak(int kind, int iters, float *ms)
{
    const int fill = (kind >> 8) & 15;  // MX_PEAK_FILLED / _ROTATE / _SMEM_STORES / _TMEM_STORES
    kind &= ~0xF00;
    if (kind < 0 || kind > 4 || !ms || iters <= 0) return MX_EINVAL;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    cudaStream_t st = current_stream();
    cudaError_t e;
    switch (kind) {
    case BSK_BF16: e = run_peak<BSK_BF16>(*ds, st, iters, fill, ms); break;
    case BSK_E4M3: e = run_peak<BSK_E4M3>(*ds, st, iters, fill, ms); break;
    case BSK_MXF8: e = run_peak<BSK_MXF8>(*ds, st, iters, fill, ms); break;
    case BSK_MXF4: e = run_peak<BSK_MXF4>(*ds, st, iters, fill, ms); break;
    default: e = run_peak<BSK_NVF4>(*ds, st, iters, fill, ms); break;
    }
    return e == cudaSuccess ? MX_OK : MX_ECUDA;
}
