// mx_qmm.cu -- prefill GEMM over block-float weights on the 5th-generation
// tensor cores (tcgen05, CTA pairs), sm_103a.
//
//   Y[m][n] = bf16_rne( sum_k X[m][k] * W[n][k] ),  X bf16, fp32 accumulate.
//
// The pages move block-float dequantisation onto the GPU and feed the
// matrix units from it ("MLxcel 0.8 release", section "Decoding block-float
// formats in software": NVFP4 prefill 3.1x from GPU dequant + WMMA; talk
// slide 12).  Here a cluster of two CTAs (a CTA pair on neighbouring SMs)
// owns a (256 * NACC) x 256 output tile and runs tcgen05.mma.cta_group::2
// with M = 256, N = 256, K = 16: CTA r holds rows 128r .. 128r+127 of each
// 256-row slab of X (its half of operand A) and weight rows
// n0 + 128r .. +127 decoded to bf16 (its half of operand B); the pair's MMA
// reads both CTAs' shared memory and CTA r's tensor memory receives its 128
// rows of the accumulator.  Against one CTA running 128 x 256 MMAs this
// halves each SM's decode work and shared-memory operand reads per flop.
// Per CTA, K streams in 64-wide k-blocks through three rings of shared
// memory (X slabs, decoded weights, packed codes with their scales):
//
//   warp 0      codes of the CTA's 128 weight rows by TMA, and their block
//               scales through registers into shared memory
//   warp 1      CTA 0: one thread issues the pair's MMAs (NACC accumulators
//               of 256 columns sharing the decoded weights) and commits each
//               k-block to the empty barriers of both CTAs
//   warps 2-    decoders, in groups of 8 warps (one group for 512-row tiles,
//               two taking alternate k-blocks for 256-row tiles, whose MMAs
//               are twice as fast per k-block): two threads per weight row,
//               32 elements each; they decode the codes exactly to bf16
//               (code * scale has at most 6 significant bits) into the
//               128-byte-swizzled K-major layout TMA produces; CTA 0's warps
//               then arrive on CTA 0's barrier, CTA 1's signal it with a
//               16-byte bulk copy that completes there.  Then the epilogue:
//               tcgen05.ld of the CTA's accumulator rows, NVFP4 tensor
//               scale, round to bf16, store.
//   last warp   X: NACC 128 x 64 bf16 slabs per k-block by TMA (128-byte
//               swizzle); both CTAs' slabs complete on CTA 0's barrier
//
// Every mbarrier wait is bounded (about two seconds of %globaltimer); a wait
// that gives up sets MX_DEVERR_TIMEOUT in the device error word, the CTA
// drains what it has in flight, both CTAs of the pair write NaN to their Y
// rows and return.
#include <atomic>

#include "mx_internal.h"
#include "mx_tc.cuh"

namespace mx {

constexpr int QMM_BN = 256;                    // UMMA N: 128 weight rows from each CTA
constexpr int QMM_BK = 64;                     // bf16 elements per 128-byte swizzle row
constexpr int QMM_X_BYTES = 128 * QMM_BK * 2;  // a CTA's 128 rows of one 256-row X slab
constexpr int QMM_W_BYTES = 128 * QMM_BK * 2;  // a CTA's 128 decoded weight rows
constexpr int QMM_SMEM_LIMIT = 232448;         // 227 KB of dynamic shared memory per CTA
constexpr unsigned long long QMM_WAIT_NS = 2000000000ull;
// control words after the barriers: TMEM base, abort flag, X k-blocks loaded,
// X k-blocks taken, decoded k-blocks taken from CTA 1, and the count of
// signals each of up to 16 decoder warps issued
constexpr int QMM_CTRL_WORDS = 5 + 16;

// Per-format, per-tile-height geometry.  Three rings of k-blocks:
//   X ring (SX slots): NACC slabs of 128 x 64 bf16 X rows, by TMA;
//   D ring (SD slots): the decoded 128 x 64 bf16 weight tile;
//   C ring (SC slots): the packed codes (TMA) and block scales of a k-block.
// A D slot is held from its decode through the hand-over to CTA 0 until the
// MMA finishes; a C slot only until its codes are decoded.
template <int FMT, int NACC, bool GROUPED = false>
struct QmmGeo {
    static constexpr int BM = 256 * NACC;  // output rows per pair tile
    static constexpr int CODE_ROW = FMT == FMT_MXFP8 ? QMM_BK : QMM_BK / 2;  // code bytes per row per k-block
    static constexpr int C_BYTES = 128 * CODE_ROW;
    static constexpr int SPK = FMT == FMT_NVFP4 ? 4 : 2;  // scale bytes per row per k-block
    static constexpr int SC_BYTES = 128 * SPK;
    static constexpr int X_STAGE = NACC * QMM_X_BYTES;
    // decoder groups: with 256-row tiles one group of 8 warps decoding a
    // k-block at a time cannot keep up with the MMAs (its warps are latency
    // bound), so two groups take alternate k-blocks; grouped tiles (up to 512
    // rows, often only 256 used) take two groups as well
    static constexpr int NG = (NACC == 1 || GROUPED) ? 2 : 1;
    static constexpr int SX = NACC == 2 ? 4 : 8;  // 256-row tiles: X slabs land late under load, go deeper
    static constexpr int SD = NACC == 2 ? (NG == 2 ? 4 : 5) : 4;
    static constexpr int SC_MAX = 4;  // codes ring depth cap
    static constexpr int THREADS = 96 + 256 * NG;  // codes producer, MMA, X producer, decoders
    static constexpr int SPF = 4;     // k-blocks of block scales the producer keeps in flight
    static constexpr int RESERVED = 1024 /*align*/ + 128 /*signal landing*/ + 512 /*barriers*/;
    static constexpr int C_FIT = (QMM_SMEM_LIMIT - RESERVED - SX * X_STAGE - SD * QMM_W_BYTES) / (C_BYTES + SC_BYTES);
    static constexpr int SC = C_FIT > SC_MAX ? SC_MAX : C_FIT;
    // layout: [X ring][D ring][codes ring][scales ring][signal landing][barriers]
    static constexpr int OFF_D = SX * X_STAGE;
    static constexpr int OFF_C = OFF_D + SD * QMM_W_BYTES;
    static constexpr int OFF_S = OFF_C + SC * C_BYTES;
    static constexpr int OFF_SIG = OFF_S + SC * SC_BYTES;
    static constexpr int OFF_BAR = OFF_SIG + 128;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;
    static constexpr int TMEM_COLS = 256 * NACC;
    static_assert(OFF_C % 1024 == 0 && OFF_S % 128 == 0 && OFF_SIG % 128 == 0, "ring alignment");
    static_assert(SC >= 2, "codes ring too shallow");
    // each ring slot is always used by the same decoder group (so a group
    // never waits on a phase two completions ahead of the barrier)
    static_assert(SC % NG == 0 && SD % NG == 0, "ring depth and decoder groups");
    static_assert((2 * SX + 2 * SC + 3 * SD + 1) * 8 + 4 * QMM_CTRL_WORDS <= 512, "barrier area");
    static_assert(SMEM <= QMM_SMEM_LIMIT, "shared memory");
};

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 D,
// M = 256 (the pair), N = 256.
__host__ __device__ constexpr uint32_t qmm_idesc()
{
    return (1u << 4)                // D format fp32
           | (1u << 7)              // A format bf16
           | (1u << 10)             // B format bf16
           | ((QMM_BN >> 3) << 17)  // N / 8
           | ((256 >> 4) << 24);    // M / 16
}

// ------------------------------------------------------------ decode

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

__device__ __forceinline__ void store_chunk(uint8_t *row_base, int chunk, int sw, uint32_t x, uint32_t y,
                                            uint32_t z, uint32_t w)
{
    *reinterpret_cast<uint4 *>(row_base + ((chunk ^ sw) << 4)) = make_uint4(x, y, z, w);
}

// Decode 32 elements of one weight row (half `half` of a 64-wide k-block)
// to bf16 and store them as chunks 4*half .. 4*half+3 of the row's 128 bytes
// at `row_base` (row r of a 128-byte-swizzled tile: chunk c at c ^ (r & 7)).
// w[]: the packed codes (4 words for E2M1, 8 for E4M3); sbits: the block
// scale byte (MX) or the two E4M3 scale bytes (NVFP4).
// Fast path: hardware cvt to f16, exact move to bf16 (scaled by 2^-112), one
// bf16 multiply by the block scale times 2^112 (exact: the result has at most
// 6 significant bits and stays a normal bf16 number).  Scales outside its
// range (E8M0 below 2 (10 for MXFP8) or above 142, NaN scales) use exact fp32
// products.
template <int FMT>
__device__ __forceinline__ void qhalf_store(const uint32_t *w, uint32_t sbits, uint8_t *row_base, int half, int sw)
{
    if constexpr (FMT == FMT_MXFP8) {
        const uint32_t e = sbits & 0xFFu;
        // An E4M3 NaN byte (S.1111.111) converts to an f16 NaN, which the
        // exact move would turn into a finite bf16: a half row holding one
        // takes the fp32 path, which keeps it NaN.  (b & 0x7F) + 1 sets bit 7
        // of its byte only for 0x7F, and never carries into the next byte.
        uint32_t nan_probe = 0u;
#pragma unroll
        for (int c = 0; c < 8; ++c) nan_probe |= (w[c] & 0x7F7F7F7Fu) + 0x01010101u;
        if (e - 10u <= 132u && (nan_probe & 0x80808080u) == 0u) {
            const uint32_t m = bf16x2_pow2_m15((int)e);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t h0, h1, h2, h3;
                e4m3x4_to_f16x2(w[2 * c], h0, h1);
                e4m3x4_to_f16x2(w[2 * c + 1], h2, h3);
                store_chunk(row_base, 4 * half + c, sw, bf16x2_mul(f16x2_to_bf16x2_m112(h0), m),
                            bf16x2_mul(f16x2_to_bf16x2_m112(h1), m), bf16x2_mul(f16x2_to_bf16x2_m112(h2), m),
                            bf16x2_mul(f16x2_to_bf16x2_m112(h3), m));
            }
            return;
        }
        const float s = e8m0_to_f32(e);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            store_chunk(row_base, 4 * half + c, sw, scaled_bf16x2(e4m3x2_to_f16x2(w[2 * c]), s),
                        scaled_bf16x2(e4m3x2_to_f16x2(w[2 * c] >> 16), s),
                        scaled_bf16x2(e4m3x2_to_f16x2(w[2 * c + 1]), s),
                        scaled_bf16x2(e4m3x2_to_f16x2(w[2 * c + 1] >> 16), s));
    } else {
        // multiplier of words 0-1 (m0) and 2-3 (m1): one 32-element E8M0
        // block, or two 16-element E4M3 blocks
        uint32_t m0, m1;
        bool fast;
        if constexpr (FMT == FMT_NVFP4) {
            // E4M3 scale s: bf16(s * 2^112) is exact (4 significant bits); NaN codes are 0x7F / 0xFF
            fast = (((sbits & 0x7F7Fu) + 0x0101u) & 0x8080u) == 0u;
            const uint32_t a2 = f16x2_to_bf16x2_m112(e4m3x2_to_f16x2(sbits));
            // a2 holds s * 2^-112: multiply by 2^112 twice to get s * 2^112
            const uint32_t p112 = bf16x2_pow2_m15(127);
            const uint32_t as = bf16x2_mul(bf16x2_mul(a2, p112), p112);
            m0 = (as & 0xFFFFu) | (as << 16);
            m1 = (as >> 16) | (as & 0xFFFF0000u);
        } else {
            const uint32_t e = sbits & 0xFFu;
            fast = e - 2u <= 140u;  // 2 <= e <= 142: products normal bf16
            m0 = m1 = bf16x2_pow2_m15((int)e);
        }
        if (fast) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // word j: elements 8j .. 8j+7 of the half row
                const uint32_t m = j < 2 ? m0 : m1;
                uint32_t h0, h1, h2, h3;
                e2m1x8_to_f16x2(w[j], h0, h1, h2, h3);
                store_chunk(row_base, 4 * half + j, sw, bf16x2_mul(f16x2_to_bf16x2_m112(h0), m),
                            bf16x2_mul(f16x2_to_bf16x2_m112(h1), m), bf16x2_mul(f16x2_to_bf16x2_m112(h2), m),
                            bf16x2_mul(f16x2_to_bf16x2_m112(h3), m));
            }
            return;
        }
        float s0, s1;
        if constexpr (FMT == FMT_NVFP4) {
            const uint32_t a = e4m3x2_to_f16x2(sbits);
            s0 = f16_lo_to_f32(a);
            s1 = f16_hi_to_f32(a);
        } else {
            s0 = s1 = e8m0_to_f32(sbits);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float s = j < 2 ? s0 : s1;
            store_chunk(row_base, 4 * half + j, sw, scaled_bf16x2(e2m1x2_to_f16x2(w[j]), s),
                        scaled_bf16x2(e2m1x2_to_f16x2(w[j] >> 8), s),
                        scaled_bf16x2(e2m1x2_to_f16x2(w[j] >> 16), s),
                        scaled_bf16x2(e2m1x2_to_f16x2(w[j] >> 24), s));
        }
    }
}

// ------------------------------------------------------------ kernel

// One row's block scales of one k-block: 2 E8M0 bytes or 4 E4M3 bytes.
template <int SPK>
__device__ __forceinline__ uint32_t scale_load(const uint8_t *p)
{
    return SPK == 4 ? ld_nc_u32(p) : ld_nc_u16(p);
}

// The SPK block-scale bytes of k-block kb of one weight row (`row`: its
// scales, nsc bytes).  Bytes past the row's scales (a last k-block that K
// only partly covers) and rows past the weights read as 1.0: their codes are
// zero-filled by the TMA, so they add zero.  `wide`: rows are SPK-aligned,
// so a whole k-block's scales come in one load.
template <int SPK>
__device__ __forceinline__ uint32_t scale_load_edge(const uint8_t *row, bool row_ok, int kb, int nsc, bool wide)
{
    constexpr uint32_t one = SPK == 4 ? 0x38383838u : 0x7F7Fu;  // E4M3 1.0 / E8M0 1.0
    if (!row_ok) return one;
    const int b0 = kb * SPK;
    if (wide && b0 + SPK <= nsc) return scale_load<SPK>(row + b0);
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < SPK; ++j) v |= (b0 + j < nsc ? ld_nc_u8(row + b0 + j) : (one & 0xFFu)) << (8 * j);
    return v;
}

// What a pair tile computes and where its rows go.
constexpr int QMM_DENSE = 0;        // Y[M][N] = X W^T
constexpr int QMM_GROUPED = 1;      // expert groups of sorted rows (up to 512); row i of group g -> Y[slot_of[r0 + i]]
constexpr int QMM_GROUPED_GLU = 2;  // as 1, but CTA 0 takes gate rows, CTA 1 up rows; h = SwiGLU -> H[r0 + i]

struct QmmArgs {
    const uint8_t *scales;
    uint16_t *Y;  // dense / grouped: [rows][N]; SwiGLU: h [rows][N / 2]
    int *err;
    int M, N, K;  // grouped: N weight rows per expert, M rows of the gathered X
    int wrows;    // weight rows in the codes tensor (N, or E * N for expert stacks)
    int ystore;   // 2: Y rows 32-byte aligned (32-byte stores); 1: 16-byte; 0: 2-byte stores
    unsigned long long wait_ns;   // limit of a pipeline wait (producer / consumer)
    unsigned long long drain_ns;  // limit of a wait for copies already in flight
    int stall_x;                  // test hook: issue no X loads, so the MMA issuer's first wait times out
    // grouped modes: the routing tables (written by the moe_group_route kernels)
    const int *groups;   // [0] = number of tiles G; from word 4 on: G x {expert, first sorted row, rows, 0}
    const int *slot_of;  // sorted row -> slot (QMM_GROUPED)
    int E;               // experts
    int ntile;           // column tiles per group tile
};

// silu(g) * u rounded to bf16 for the prefill SwiGLU epilogue: the same
// formula as swiglu_bf16 (sigmoid from e^-|g|, so nothing overflows) with the
// fast exponent and division intrinsics; the epilogue of a 256-row tile
// evaluates it 32768 times per CTA after the last MMA, where the exactly
// rounded division dominated the tile's tail.  The result differs from
// swiglu_bf16's by at most one bf16 unit, and only near rounding boundaries.
__device__ __forceinline__ uint32_t swiglu_bf16_fast(float g, float u)
{
    const float e = __expf(-fabsf(g));
    const float sig = __fdividef(g >= 0.0f ? 1.0f : e, 1.0f + e);
    return f32x2_to_bf16x2(g * sig * u, 0.0f) & 0xFFFFu;
}

// 32 bf16 outputs of one row (o: 16 bf16 pairs) at dst, of which the first
// `valid` are stored (a last column tile that N only partly covers); ystore:
// see QmmArgs.
__device__ __forceinline__ void store_row32(uint16_t *dst, const uint32_t *o, int valid, int ystore);

// 32 contiguous bytes to global memory (32-byte aligned address).
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v)
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                 "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void store_row32(uint16_t *dst, const uint32_t *o, int valid, int ystore)
{
    if (valid >= 32 && ystore == 2) {
        st_global_v8(dst, o);
        st_global_v8(dst + 16, o + 8);
    } else if (valid >= 32 && ystore == 1) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int j = 0; j < 4; ++j) d4[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (2 * j < valid) dst[2 * j] = (uint16_t)(o[j] & 0xFFFFu);
            if (2 * j + 1 < valid) dst[2 * j + 1] = (uint16_t)(o[j] >> 16);
        }
    }
}

template <int FMT, int NACC, int MODE>
__global__ void __launch_bounds__(QmmGeo<FMT, NACC, MODE != QMM_DENSE>::THREADS, 1) qmm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                             const __grid_constant__ CUtensorMap tmap_c, QmmArgs a)
{
    using QG = QmmGeo<FMT, NACC, MODE != QMM_DENSE>;
    constexpr int SX = QG::SX, SD = QG::SD, SC = QG::SC, SPK = QG::SPK;
    constexpr uint32_t SIG_BYTES = 8 * 16;  // one 16-byte signal per decoder warp of CTA 1
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *xring = smem;
    uint8_t *dring = smem + QG::OFF_D;
    uint8_t *cring = smem + QG::OFF_C;
    uint8_t *sring = smem + QG::OFF_S;
    uint8_t *sig = smem + QG::OFF_SIG;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + QG::OFF_BAR);
    uint64_t *full_x = bars;                // [SX] (CTA 0) both CTAs' X slabs landed: 2 arrivals + bytes
    uint64_t *empty_x = bars + SX;          // [SX] the pair's MMAs that read the X slot finished
    uint64_t *full_c = bars + 2 * SX;       // [SC] this CTA's codes (TMA) and scales landed
    uint64_t *empty_c = full_c + SC;        // [SC] this CTA's decoders read the codes (8 warps)
    uint64_t *dec_full = full_c + 2 * SC;   // [SD] this CTA's decoded tile stored (8 warps)
    uint64_t *peer_full = dec_full + SD;    // [SD] (CTA 0) CTA 1's decoded tile stored (8 signals)
    uint64_t *empty_d = dec_full + 2 * SD;  // [SD] the pair's MMAs that read the D slot finished
    uint64_t *acc_full = dec_full + 3 * SD; // accumulators complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *x_issued = reinterpret_cast<volatile int *>(tmem_slot + 2);  // X k-blocks this CTA loaded
    volatile int *x_taken = reinterpret_cast<volatile int *>(tmem_slot + 3);   // (CTA 0) X k-blocks the MMAs took
    volatile int *peer_taken = reinterpret_cast<volatile int *>(tmem_slot + 4);  // (CTA 0) k-blocks whose CTA 1 half the MMAs took
    volatile int *sig_issued = reinterpret_cast<volatile int *>(tmem_slot + 5);  // (CTA 1) [8 NG] signals each decoder warp issued

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x();
    const int KB = (a.K + QMM_BK - 1) / QMM_BK;  // the last k-block may be partly past K
    // m0: first X row of the tile; n0: first output column; wrow: first of
    // this CTA's 128 weight rows (over all experts); rows: valid tile rows
    int m0, n0, wrow, rows, expert = 0;
    if constexpr (MODE == QMM_DENSE) {
        const int m_tiles = (a.M + QG::BM - 1) / QG::BM;
        m0 = (cid % m_tiles) * QG::BM;
        n0 = (cid / m_tiles) * QMM_BN;
        wrow = n0 + 128 * (int)rank;
        rows = a.M - m0;
    } else {
        // the routing tables come from the previous kernel; a grid sized for
        // the most tiles any routing can make leaves the spare pairs idle
        pdl_wait();
        const int g = cid / a.ntile, nt = cid - g * a.ntile;
        if (g >= __ldcg(a.groups)) return;  // both CTAs of the pair see the same g
        const int4 t = __ldcg(reinterpret_cast<const int4 *>(a.groups + 4) + g);
        expert = t.x;
        m0 = t.y;
        rows = t.z;
        if constexpr (MODE == QMM_GROUPED) {
            n0 = nt * QMM_BN;
            wrow = expert * a.N + n0 + 128 * (int)rank;
        } else {
            n0 = nt * 128;  // h columns; gate rows n0.. (CTA 0), up rows N/2 + n0.. (CTA 1)
            wrow = expert * a.N + (int)rank * (a.N / 2) + n0;
        }
    }
    // 256-row halves of the tile that hold rows: a grouped tile of at most 256
    // rows skips the second half's X slabs, MMAs and epilogue
    const int nh = (MODE == QMM_DENSE || rows > 256) ? NACC : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; ++s) {
            mbar_init(&full_x[s], 2);
            mbar_init(&empty_x[s], 1);
        }
        for (int s = 0; s < SC; ++s) {
            mbar_init(&full_c[s], 2);
            mbar_init(&empty_c[s], 8);
        }
        for (int s = 0; s < SD; ++s) {
            mbar_init(&dec_full[s], 8);
            mbar_init(&peer_full[s], 1);
            mbar_init(&empty_d[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        *x_issued = 0;
        *x_taken = 0;
        *peer_taken = 0;
        for (int w = 0; w < 8 * QG::NG; ++w) sig_issued[w] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // first use of each peer_full: its one arrival, and the signal bytes to wait for
        for (int s = 0; s < SD; ++s) mbar_arrive_expect_tx(&peer_full[s], SIG_BYTES);
    }
    cluster_sync_all();  // both CTAs' barriers exist before either signals remotely
    if (warp == 1) {
        // one warp of each CTA allocates the pair's columns together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(QG::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();
    if constexpr (MODE == QMM_DENSE) pdl_wait();  // X and Y may be used by the neighbouring kernels

    if (warp == 2 + 8 * QG::NG) {
        // ---------------- X producer: both CTAs' slabs complete on CTA 0's
        // barrier, each CTA adding one arrival and its own bytes
        if (lane == 0) {
            const uint32_t fx0 = map_to_cta(smem_u32(full_x), 0);
            int issued = 0;
            for (int kb = 0; kb < KB && !a.stall_x; ++kb) {
                const int s = kb % SX;
                if (kb >= SX && !mbar_wait(&empty_x[s], ((kb / SX) - 1) & 1, abort_flag, a.wait_ns)) break;
                const uint32_t bar = fx0 + 8u * (uint32_t)s;
                mbar_arrive_expect_tx_cluster(bar, (uint32_t)(nh * QMM_X_BYTES));
#pragma unroll
                for (int h = 0; h < NACC; ++h)
                    if (h < nh)
                        tma_load_2d_pair(xring + s * QG::X_STAGE + h * QMM_X_BYTES, &tmap_x, kb * QMM_BK,
                                         m0 + 256 * h + 128 * (int)rank, bar);
                issued = kb + 1;
            }
            *x_issued = issued;
        }
    } else if (warp == 0) {
        // ---------------- codes producer: codes by TMA (lane 0), block scales
        // (whole warp, QG::SPF k-blocks in flight).  The scales come through
        // shared memory so that the decoders hold no global loads in flight.
        const int nsc = a.K / (FMT == FMT_NVFP4 ? 16 : 32);  // scale bytes per weight row
        const bool wide = nsc % SPK == 0;
        const uint8_t *srow[4];
        bool rok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = wrow + lane + 32 * i;
            rok[i] = r < a.wrows;
            srow[i] = a.scales + (size_t)(rok[i] ? r : 0) * nsc;
        }
        uint32_t pv[QG::SPF][4];
#pragma unroll
        for (int j = 0; j < QG::SPF; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (j < KB) pv[j][i] = scale_load_edge<SPK>(srow[i], rok[i], j, nsc, wide);
        int issued = 0;
        bool go = true;
        for (int kb0 = 0; kb0 < KB && go; kb0 += QG::SPF) {
#pragma unroll
            for (int j = 0; j < QG::SPF; ++j) {
                const int kb = kb0 + j;
                if (kb >= KB) break;
                const int s = kb % SC;
                int ok = 1;
                if (lane == 0 && kb >= SC) ok = mbar_wait(&empty_c[s], ((kb / SC) - 1) & 1, abort_flag, a.wait_ns);
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                    go = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full_c[s], QG::C_BYTES);
                    tma_load_2d(cring + s * QG::C_BYTES, &tmap_c, kb * QG::CODE_ROW, wrow, &full_c[s]);
                }
                uint8_t *sc = sring + s * QG::SC_BYTES;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (SPK == 4) *reinterpret_cast<uint32_t *>(sc + 4 * (lane + 32 * i)) = pv[j][i];
                    else *reinterpret_cast<uint16_t *>(sc + 2 * (lane + 32 * i)) = (uint16_t)pv[j][i];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_c[s]);
                issued = kb + 1;
                if (kb + QG::SPF < KB)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        pv[j][i] = scale_load_edge<SPK>(srow[i], rok[i], kb + QG::SPF, nsc, wide);
            }
        }
        // drain: every issued codes TMA must land before the CTA may exit
        if (lane == 0)
            for (int kb = (issued > SC ? issued - SC : 0); kb < issued; ++kb)
                mbar_wait(&full_c[kb % SC], (kb / SC) & 1, abort_flag, a.drain_ns, false);
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) {
            // ---------------- MMA issuer (CTA 0)
            constexpr uint32_t idesc = qmm_idesc();
            int taken = 0, ptaken = 0;
            for (int kb = 0; kb < KB; ++kb) {
                const int sx = kb % SX, sd = kb % SD;
                if (!mbar_wait(&full_x[sx], (kb / SX) & 1, abort_flag, a.wait_ns)) break;
                taken = kb + 1;
                if (!mbar_wait(&dec_full[sd], (kb / SD) & 1, abort_flag, a.wait_ns)) break;
                if (!mbar_wait(&peer_full[sd], (kb / SD) & 1, abort_flag, a.wait_ns)) break;
                ptaken = kb + 1;
                // arm the slot's next use: its arrival, and the signal bytes to wait for
                mbar_arrive_expect_tx(&peer_full[sd], SIG_BYTES);
                tc_fence_after();
                const uint32_t xa = smem_u32(xring + sx * QG::X_STAGE);
                const uint32_t da = smem_u32(dring + sd * QMM_W_BYTES);
#pragma unroll
                for (int kk = 0; kk < QMM_BK / 16; ++kk) {
                    const uint64_t bd = sw128_desc(da + kk * 32);
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
                    for (int h = 0; h < NACC; ++h)
                        if (h < nh)
                            umma2_bf16(tmem + h * QMM_BN, sw128_desc(xa + h * QMM_X_BYTES + kk * 32), bd, idesc,
                                       acc);
                }
                umma2_commit_both(&empty_x[sx]);
                umma2_commit_both(&empty_d[sd]);
            }
            umma2_commit_both(acc_full);  // fires once every MMA issued so far has completed
            *x_taken = taken;
            *peer_taken = ptaken;
        }
    } else {
        // ---------------- decoders (warps 2 ..): group grp (8 warps) takes
        // k-blocks grp, grp + NG, ...; its thread d decodes half (d & 1) of
        // weight row wrow + (d >> 1).  CTA 0's decoders arrive on their own
        // barrier; CTA 1's signal CTA 0 with a 16-byte bulk copy.
        const int dw = warp - 2, grp = dw >> 3, dl = dw & 7;
        const int d = 32 * dl + lane;
        const int row = d >> 1, half = d & 1;
        const uint32_t sig0 = map_to_cta(smem_u32(sig + 16 * dl), 0);
        const uint32_t pf0 = map_to_cta(smem_u32(peer_full), 0);
        int nsig = 0;  // (CTA 1, lane 0) signals issued
        for (int kb = grp; kb < KB; kb += QG::NG) {
            const int sc = kb % SC, sd = kb % SD;
            if (!mbar_wait(&full_c[sc], (kb / SC) & 1, abort_flag, a.wait_ns)) break;
            const uint8_t *cp = cring + sc * QG::C_BYTES + row * QG::CODE_ROW + half * (QG::CODE_ROW / 2);
            uint32_t w[FMT == FMT_MXFP8 ? 8 : 4];
            if constexpr (FMT == FMT_MXFP8) {
                // the two 16-byte reads in a row-dependent order spread a
                // warp's reads over all banks
                const int f = (row >> 1) & 1;
                const uint4 v0 = *reinterpret_cast<const uint4 *>(cp + 16 * f);
                const uint4 v1 = *reinterpret_cast<const uint4 *>(cp + 16 * (f ^ 1));
                const uint4 lo = f ? v1 : v0, hi = f ? v0 : v1;
                w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
                w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
            } else {
                const uint4 v = *reinterpret_cast<const uint4 *>(cp);
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            }
            const uint8_t *scp = sring + sc * QG::SC_BYTES + SPK * row + (SPK / 2) * half;
            const uint32_t sbits = SPK == 4 ? *reinterpret_cast<const uint16_t *>(scp) : *scp;
            // the codes slot may be refilled (by TMA) once every warp has read it
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_c[sc]);
            // the decoded slot is free once the pair's MMAs of k-block kb - SD finished
            if (kb >= SD && !mbar_wait(&empty_d[sd], ((kb / SD) - 1) & 1, abort_flag, a.wait_ns)) break;
            uint8_t *dslot = dring + sd * QMM_W_BYTES;
            qhalf_store<FMT>(w, sbits, dslot + row * 128, half, row & 7);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) {
                    mbar_arrive(&dec_full[sd]);
                } else {
                    bulk_signal(sig0, dslot + 16 * dl, pf0 + 8u * (uint32_t)sd);
                    ++nsig;
                }
            }
        }
        if (lane == 0 && rank == 1) sig_issued[dw] = nsig;  // read by CTA 0 if the pair gives up
    }

    // ---------------- epilogue (decoder warps): TMEM -> bf16 -> Y
    bool acc_ok = true;
    if (warp >= 2 && warp < 2 + 8 * QG::NG) {
        // the MMAs must have finished (even on abort) before TMEM is read or freed
        acc_ok = mbar_wait(acc_full, 0, abort_flag, a.drain_ns, false);
    }
    // every role of both CTAs is done: settle whether the pair gave up
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const int aborted = *abort_flag | ld_cluster_s32(map_to_cta(smem_u32((const void *)abort_flag), rank ^ 1u));
    if (aborted && rank == 0 && threadIdx.x == 32 * (2 + 8 * QG::NG)) {
        // X slabs the MMAs did not take may still be landing in either CTA:
        // supply the arrival of a CTA that did not load a k-block, then wait
        // for each outstanding slot (its bytes complete on this barrier)
        const int i0 = *x_issued, i1 = ld_cluster_s32(map_to_cta(smem_u32((const void *)x_issued), 1u));
        const int hi = i0 > i1 ? i0 : i1;
        for (int kb = *x_taken; kb < hi; ++kb) {
            const int s = kb % SX;
            if (kb >= i0) mbar_arrive_expect_tx_cluster(smem_u32(&full_x[s]), 0);
            if (kb >= i1) mbar_arrive_expect_tx_cluster(smem_u32(&full_x[s]), 0);
            mbar_wait(&full_x[s], (kb / SX) & 1, abort_flag, a.drain_ns, false);
        }
        // CTA 1's 16-byte signals of decoded k-blocks the MMAs did not take
        // may still be landing on this CTA's peer_full barriers.  CTA 1's
        // decoder warps published how many they issued (group g's warps
        // signal k-blocks g, g + NG, ...).  A signal for k-block kb is only
        // issued once the MMAs of kb - SD finished, so every outstanding one
        // belongs to [taken, taken + SD), whose phases are armed for 8
        // signals: complete the bytes of the signals never issued, then wait
        // for the phase, after which none is in flight.
        const int pt = *peer_taken;
        for (int kb = pt; kb < pt + SD && kb < KB; ++kb) {
            const int grp = kb % QG::NG, idx = kb / QG::NG;
            int n = 0;
            for (int w = 0; w < 8; ++w)
                n += ld_cluster_s32(map_to_cta(smem_u32((const void *)(sig_issued + 8 * grp + w)), 1u)) > idx;
            if (n == 0) continue;
            if (n < 8) mbar_complete_tx(&peer_full[kb % SD], 16u * (uint32_t)(8 - n));
            mbar_wait(&peer_full[kb % SD], (kb / SD) & 1, abort_flag, a.drain_ns, false);
        }
    }
    if (warp >= 2 && warp < 2 + 8 * QG::NG) {
        const bool ok = acc_ok && !aborted;
        const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31 (a warp reads its own quarter)
        const int group = (warp - 2) >> 2;  // which of the 2 * NG column ranges
        constexpr int NCG = 2 * QG::NG;
        float g = 1.0f;
        if (FMT == FMT_NVFP4) {
            const size_t blocks = (size_t)(MODE == QMM_DENSE ? 1 : a.E) * a.N * (a.K / 16);
            g = load_f32_unaligned(a.scales + blocks + 4 * (size_t)expert);
        }
        if constexpr (MODE == QMM_GROUPED_GLU) {
            // in accumulator h, columns c (gate) and 128 + c (up) of a row hold
            // the same h column
            const int hw = a.N / 2;
            constexpr int PER = NACC * 128 / NCG;
            for (int cc = group * PER; cc < (group + 1) * PER; cc += 32) {
                const int h = cc / 128, c = cc % 128;
                if (h >= nh) continue;  // warp-uniform
                const int i = 256 * h + 128 * (int)rank + 32 * quarter + lane;  // tile row
                const uint32_t tb = tmem + (uint32_t)(h * QMM_BN) + ((uint32_t)(quarter * 32) << 16);
                uint32_t vg[32], vu[32];
                if (ok) {
                    tmem_ld32(tb + (uint32_t)c, vg);
                    tmem_ld32(tb + (uint32_t)(128 + c), vu);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) vg[j] = vu[j] = 0x7FC00000u;
                }
                uint32_t o[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float g0 = __uint_as_float(vg[2 * j]), g1 = __uint_as_float(vg[2 * j + 1]);
                    float u0 = __uint_as_float(vu[2 * j]), u1 = __uint_as_float(vu[2 * j + 1]);
                    if (FMT == FMT_NVFP4) {
                        g0 = __fmul_rn(g0, g);
                        g1 = __fmul_rn(g1, g);
                        u0 = __fmul_rn(u0, g);
                        u1 = __fmul_rn(u1, g);
                    }
                    o[j] = swiglu_bf16_fast(g0, u0) | (swiglu_bf16_fast(g1, u1) << 16);
                }
                if (i < rows && n0 + c < hw)
                    store_row32(a.Y + (size_t)(m0 + i) * hw + n0 + c, o, hw - (n0 + c), a.ystore);
            }
        } else {
            for (int c = group * (NACC * 256 / NCG); c < (group + 1) * (NACC * 256 / NCG); c += 32) {
                const int h = c / QMM_BN, nc = c % QMM_BN;
                if (h >= nh) continue;  // warp-uniform
                const int i = 256 * h + 128 * (int)rank + 32 * quarter + lane;  // tile row
                uint32_t v[32];
                if (ok) {
                    tmem_ld32(tmem + (uint32_t)c + ((uint32_t)(quarter * 32) << 16), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0x7FC00000u;
                }
                uint32_t o[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float lo = __uint_as_float(v[2 * j]), hi = __uint_as_float(v[2 * j + 1]);
                    if (FMT == FMT_NVFP4) {
                        lo = __fmul_rn(lo, g);
                        hi = __fmul_rn(hi, g);
                    }
                    o[j] = f32x2_to_bf16x2(lo, hi);
                }
                if (i < rows) {  // dense: rows past M were zero-filled by TMA
                    // a lane writes 64 bytes of its own row, so every store
                    // instruction touches 32 rows: the fewer instructions the
                    // better (measured: prefill up projection 1680 -> 1731 TFLOP/s)
                    const size_t yrow = MODE == QMM_DENSE ? (size_t)(m0 + i) : (size_t)__ldcg(a.slot_of + m0 + i);
                    if (n0 + nc < a.N) store_row32(a.Y + yrow * a.N + n0 + nc, o, a.N - (n0 + nc), a.ystore);
                }
            }
        }
    }
    // neither CTA frees tensor memory or exits while its peer may still use it
    tc_fence_before();
    cluster_sync_all();
    if (threadIdx.x == 0 && *abort_flag) set_device_error(a.err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(QG::TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------ host

// Test hook state (mx_debug_qmm_stall): process-wide, read at each launch.
static std::atomic<int> g_stall_x{0};
static std::atomic<unsigned long long> g_wait_ns{0};

void set_qmm_stall(int stall_x, unsigned long long wait_ns)
{
    g_stall_x.store(stall_x ? 1 : 0);
    g_wait_ns.store(wait_ns);
}

static void qmm_wait_args(QmmArgs &a)
{
    const unsigned long long w = g_wait_ns.load();
    a.wait_ns = w ? w : QMM_WAIT_NS;
    a.drain_ns = QMM_WAIT_NS;
    a.stall_x = g_stall_x.load();
}

template <int FMT, int NACC, int MODE>
static cudaError_t run_qmm(const DeviceState &ds, cudaStream_t st, const CUtensorMap &xmap, const CUtensorMap &cmap,
                           const QmmArgs &a, int pairs)
{
    using QG = QmmGeo<FMT, NACC, MODE != QMM_DENSE>;
    if (QG::SMEM > ds.max_smem_optin) return cudaErrorInvalidValue;
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(qmm_kernel<FMT, NACC, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             QG::SMEM);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(QG::THREADS);
    cfg.dynamicSmemBytes = QG::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, qmm_kernel<FMT, NACC, MODE>, xmap, cmap, a);
}

// Pair tiles of 512 rows halve each SM's decode and shared-memory writes per
// flop against 256-row tiles but come in half as many; take them unless the
// coarser wave quantisation costs more.  On GB300 a 256-row tile takes about
// 0.83 times as long as a 512-row one (M = 4096, N = 28672, K = 8192: 85 us
// against 102 us per wave of num_sms / 2 pairs).
static int qmm_nacc(const DeviceState &ds, int M, int N)
{
    if (M <= 256) return 1;
    const long long slots = ds.num_sms / 2 > 0 ? ds.num_sms / 2 : 1;
    const long long p1 = (long long)((M + 255) / 256) * ((N + QMM_BN - 1) / QMM_BN);
    const long long p2 = (long long)((M + 511) / 512) * ((N + QMM_BN - 1) / QMM_BN);
    const long long w1 = (p1 + slots - 1) / slots, w2 = (p2 + slots - 1) / slots;
    return w2 * 120 <= w1 * 100 ? 2 : 1;
}

template <int FMT>
static cudaError_t run_qmm_fmt(const DeviceState &ds, cudaStream_t st, const CUtensorMap &xmap,
                               const CUtensorMap &cmap, const QmmArgs &a)
{
    const int n_tiles = (a.N + QMM_BN - 1) / QMM_BN;
    if (qmm_nacc(ds, a.M, a.N) == 2)
        return run_qmm<FMT, 2, QMM_DENSE>(ds, st, xmap, cmap, a, ((a.M + 511) / 512) * n_tiles);
    return run_qmm<FMT, 1, QMM_DENSE>(ds, st, xmap, cmap, a, ((a.M + 255) / 256) * n_tiles);
}

// X: [rows][K] bf16, boxes of 64 x 128 rows, 128-byte swizzle; rows past
// `rows` read as zero.  Codes: [wrows][row bytes], boxes of one k-block's
// bytes x 128 rows.
static cudaError_t encode_maps(int fmt, const uint16_t *X, long long rows, const uint8_t *codes, long long wrows,
                               int K, CUtensorMap &xmap, CUtensorMap &cmap)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)QMM_BK, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(X), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const cuuint64_t row_bytes = fmt == FMT_MXFP8 ? (cuuint64_t)K : (cuuint64_t)K / 2;
    const cuuint64_t cdims[2] = {row_bytes, (cuuint64_t)wrows};
    const cuuint64_t cstrides[1] = {row_bytes};
    const cuuint32_t cbox[2] = {fmt == FMT_MXFP8 ? (cuuint32_t)QMM_BK : (cuuint32_t)QMM_BK / 2, 128u};
    r = enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), cdims, cstrides, cbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Shapes the TMA loads can take: codes rows (K/2 or K bytes) and X rows (2K
// bytes) a multiple of 16 bytes apart, i.e. K % 32 == 0 (the MX block; NVFP4
// with K % 32 == 16 is out).
bool qmm_shape_ok(int fmt, int K) { return K > 0 && K % 32 == 0; }

// Widest epilogue store the output rows allow: 32 bytes when Y and every row
// (width elements of bf16) are 32-byte aligned, 16 bytes when 16-byte
// aligned, else 2-byte stores.
static int y_store_width(const void *Y, int width)
{
    const uintptr_t y = reinterpret_cast<uintptr_t>(Y);
    if ((y & 31u) == 0 && width % 16 == 0) return 2;
    if ((y & 15u) == 0 && width % 8 == 0) return 1;
    return 0;
}

cudaError_t launch_qmm_grouped(const DeviceState &ds, cudaStream_t st, int fmt, bool swiglu, const uint8_t *codes,
                               const uint8_t *scales, const uint16_t *Xs, int rows, const int *groups,
                               int max_groups, const int *slot_of, uint16_t *Y, int E, int N, int K)
{
    if (!qmm_shape_ok(fmt, K) || (swiglu && N % 2 != 0)) return cudaErrorInvalidValue;
    if (max_groups <= 0) return cudaSuccess;
    CUtensorMap xmap, cmap;
    cudaError_t e = encode_maps(fmt, Xs, rows, codes, (long long)E * N, K, xmap, cmap);
    if (e != cudaSuccess) return e;
    QmmArgs a;
    a.scales = scales;
    a.Y = Y;
    a.err = ds.err;
    a.M = rows;
    a.N = N;
    a.K = K;
    qmm_wait_args(a);
    const int yw = swiglu ? N / 2 : N;  // output row width
    a.wrows = E * N;
    a.ystore = y_store_width(Y, yw);
    a.groups = groups;
    a.slot_of = slot_of;
    a.E = E;
    a.ntile = swiglu ? (N / 2 + 127) / 128 : (N + QMM_BN - 1) / QMM_BN;
    const int pairs = max_groups * a.ntile;
    if (swiglu) {
        if (fmt == FMT_MXFP4) return run_qmm<FMT_MXFP4, 2, QMM_GROUPED_GLU>(ds, st, xmap, cmap, a, pairs);
        if (fmt == FMT_MXFP8) return run_qmm<FMT_MXFP8, 2, QMM_GROUPED_GLU>(ds, st, xmap, cmap, a, pairs);
        return run_qmm<FMT_NVFP4, 2, QMM_GROUPED_GLU>(ds, st, xmap, cmap, a, pairs);
    }
    if (fmt == FMT_MXFP4) return run_qmm<FMT_MXFP4, 2, QMM_GROUPED>(ds, st, xmap, cmap, a, pairs);
    if (fmt == FMT_MXFP8) return run_qmm<FMT_MXFP8, 2, QMM_GROUPED>(ds, st, xmap, cmap, a, pairs);
    return run_qmm<FMT_NVFP4, 2, QMM_GROUPED>(ds, st, xmap, cmap, a, pairs);
}

cudaError_t launch_qmm(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *X, uint16_t *Y, int M, int N, int K)
{
    if (!qmm_shape_ok(fmt, K)) return cudaErrorInvalidValue;
    CUtensorMap xmap, cmap;
    cudaError_t e = encode_maps(fmt, X, M, codes, N, K, xmap, cmap);
    if (e != cudaSuccess) return e;
    QmmArgs a;
    a.scales = scales;
    a.Y = Y;
    a.err = ds.err;
    a.M = M;
    a.N = N;
    a.K = K;
    qmm_wait_args(a);
    a.wrows = N;
    a.ystore = y_store_width(Y, N);
    a.groups = nullptr;
    a.slot_of = nullptr;
    a.E = 1;
    a.ntile = 0;
    if (fmt == FMT_MXFP4) return run_qmm_fmt<FMT_MXFP4>(ds, st, xmap, cmap, a);
    if (fmt == FMT_MXFP8) return run_qmm_fmt<FMT_MXFP8>(ds, st, xmap, cmap, a);
    return run_qmm_fmt<FMT_NVFP4>(ds, st, xmap, cmap, a);
}

}  // namespace mx
