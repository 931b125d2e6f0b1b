// mx_qmv_core.cuh -- device pieces shared by the decode-GEMV kernels
// (direct-load and streaming variants): activation staging, the m16n8k16
// fragment mapping for block-float weights, and the warp reductions.
//
// What is computed: y[t][n] = sum_k x[t][k] * W[n][k] for a handful of
// tokens t, with W streamed from HBM exactly once per call ("MLxcel 0.8
// release", section "Profiling set the porting order": in dense decode one
// GEMV kernel takes 95% of GPU time and runs at the memory roofline; talk
// slide 13).  The weight is never materialised: each 32-element block of
// codes is decoded in registers and its block scale is applied to the
// block's partial sum.
//
// sm_103a design.  Decoding dominates the instruction budget of a GEMV at
// HBM speed (about 12 G weights/ms at 6.4 TB/s of MXFP4), so the
// multiply-accumulate runs on the tensor pipe: codes are converted by
// cvt.rn.f16x2.e2m1x2 / .e4m3x2 straight into the A fragment of an
// m16n8k16 f16 MMA with fp32 accumulation, and the activations, scaled per
// token by a power of two so that the largest magnitude lies in [1, 2),
// form the B fragment (exact for elements within 2^14 of the token's
// largest; smaller ones become f16 subnormals with an absolute error of at
// most 2^-25 times that largest magnitude, and those below 2^-24 of it
// flush to zero).  To keep one block scale per MMA output while loads stay
// contiguous, the 16 A rows of an MMA are (weight row, block) pairs and the
// 8 B columns are (token, block) pairs with the same block set:
//
//     BPM = 8 / MC blocks per MMA, MC = tokens per pass (1, 2, 4 or 8)
//     A row a (0..15): weight row  (a / 8) * MC + (a % 8) / BPM,  block a % BPM
//     B col n (0..7):  token       n / BPM,                        block n % BPM
//
// Only entries whose A-row block equals the B-column block are used; the
// others are discarded (the tensor pipe has ample headroom).  Lane
// (g = lane/4, q = lane%4) then reads, for A rows g and g+8, the 4-byte
// (MXFP4) or 8-byte (MXFP8) slice [8q, 8q+8) of the block: for MC = 1 the 32
// lanes read 128 contiguous bytes of one row per load.  Inside a 32-element
// unit, fragment slot p = 8q + 4s + i (MMA step s, element i) holds element
// p for MX formats and element 16s + 4q + i for NVFP4, so each MMA step
// stays inside one 16-element NVFP4 block; the staged activations use the
// same permutation.
#pragma once

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

constexpr int QMV_WARPS = 16;
constexpr int QMV_THREADS = QMV_WARPS * 32;
// Pipeline depth (MMA iterations loaded ahead) of the dense and MoE kernels.
template <int FMT>
__host__ __device__ constexpr int dense_uf() { return FMT == FMT_MXFP8 ? 6 : 8; }
constexpr int MOE_UF = 4;

// f16 row stride of staged activations: units*32 rounded so that the byte
// stride is an odd multiple of 64 (conflict-free B loads for 8 tokens).
__host__ __device__ inline int stage_stride(int K)
{
    int U = (K + 31) / 32;
    int ks = U * 32;
    if ((ks / 32) % 2 == 0) ks += 32;
    return ks;
}


// -------------------------------------------------------------- staging

// Stage activation rows (bf16 -> scaled f16, permuted per unit) into
// shared memory.  Row r of xs holds elements [0, len) of source row src[r]
// (or r when src is null) of x, whose rows are ld elements apart.  sh[r]
// receives the per-row power-of-two exponent: the staged values are
// x * 2^-sh[r] with the largest finite magnitude in [1, 2).  bf16 has 8
// significant bits and f16 11, so an element is staged exactly when it is
// at least 2^-14 times that largest magnitude (an f16 normal); smaller ones
// become f16 subnormals (absolute error at most 2^-25 times the largest) and
// those below 2^-24 times it become zero.  Infinities and NaNs do not set
// the scale and stay infinities and NaNs.  Elements past len up to the next
// 32-element unit are zero.
// len and ld are multiples of 8 and x is 16-byte aligned (K is a multiple
// of the block), so every 8-element chunk is one aligned 16-byte load that
// lies wholly inside or wholly past len.
// When the rows fit in registers (<= 8 chunks of 8 elements per thread)
// global memory is read once and the chunks stay in registers; otherwise the
// raw bf16 chunks are parked in xs and converted there in place.
constexpr int STAGE_REG_CHUNKS = 8;

// Elements k0 .. k0+7 (k0 a multiple of 8) of staged row `row` (xs + r*ks),
// scaled by f and rounded to f16; zero when the chunk lies past len.
__device__ __forceinline__ void stage_store(uint16_t *row, int k0, int len, uint4 v, float f, int fmt)
{
    const int p0 = k0 & 31;
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    if (k0 < len) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            out[j] = f32x2_to_f16x2(__uint_as_float(w[j] << 16) * f, __uint_as_float(w[j] & 0xFFFF0000u) * f);
    }
    row += k0 - p0;
    if (fmt == FMT_NVFP4) {
        // slots of elements p0, p0+2 are adjacent, and those of p0+4, p0+6
        const int s0 = 8 * ((p0 & 15) >> 2) + 4 * (p0 >> 4);
        *reinterpret_cast<uint2 *>(row + s0) = make_uint2(out[0], out[1]);
        *reinterpret_cast<uint2 *>(row + s0 + 8) = make_uint2(out[2], out[3]);
    } else {
        *reinterpret_cast<uint4 *>(row + p0) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// Magnitude bits of a bf16 value for the row maximum; an infinity or a NaN
// counts as zero (it must not set the scale of the finite elements).
__device__ __forceinline__ unsigned fin_mag(uint32_t h)
{
    h &= 0x7FFFu;
    return h >= 0x7F80u ? 0u : h;
}

// Running per-half maximum of bf16 magnitudes: |m| = max(|m|, |w|) in each
// half (the sign bits are meaningless; mask them off at the end).  A NaN
// operand loses to the other one, so NaNs never enter; an infinity does.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t w)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(m), "r"(w));
    return d;
}

__device__ __forceinline__ uint32_t absmax_chunk(uint32_t m, uint4 v)
{
    return absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m, v.x), v.y), v.z), v.w);
}

// Largest finite magnitude (bf16 bits) of the 8 elements of a chunk,
// element by element (the path taken when an infinity was seen).
__device__ __forceinline__ unsigned chunk_mag_exact(uint4 v)
{
    unsigned m = max(max(fin_mag(v.x), fin_mag(v.x >> 16)), max(fin_mag(v.y), fin_mag(v.y >> 16)));
    return max(m, max(max(fin_mag(v.z), fin_mag(v.z >> 16)), max(fin_mag(v.w), fin_mag(v.w >> 16))));
}

struct NoMid {
    __device__ void operator()() const {}
};

// Power-of-two exponent of a row from its maximum (bf16 magnitude bits).
__device__ __forceinline__ int stage_shift(unsigned mb)
{
    const int ef = (int)(mb >> 7);
    return (mb == 0u || ef == 255) ? 0 : (ef == 0 ? -126 : ef - 127);
}

// Thread layout of the staging: a pass covers RP rows (a power of two up to
// 16) with TPR = blockDim / RP threads per row (whole warps: blockDim is a
// power of two of at least 512, QMV_THREADS in every caller, so that the warp
// reduction of a row's maximum never mixes rows); thread (tr, tc) takes
// chunks tc, tc + TPR, ... of row tr + p * RP in pass p.  A thread's j-th chunk is step q = j % NQ of pass p = j / NQ.
// Shifts only: a division costs a long dependent chain at kernel start.
struct StageMap {
    int rp, tpr, tr, tc, npass, nq;
    __device__ __forceinline__ StageMap(int nrows, int cpr)
    {
        const int lrp = nrows <= 1 ? 0 : nrows <= 2 ? 1 : nrows <= 4 ? 2 : nrows <= 8 ? 3 : 4;
        const int ltpr = (31 - __clz((int)blockDim.x)) - lrp;
        rp = 1 << lrp;
        tpr = 1 << ltpr;
        tr = (int)threadIdx.x >> ltpr;
        tc = (int)threadIdx.x & (tpr - 1);
        npass = (nrows + rp - 1) >> lrp;
        nq = (cpr + tpr - 1) >> ltpr;
    }
};

// The max of a pass: lanes hold their own finite maxima (a lane that saw an
// infinity contributes 0 here and publishes its chunks exactly later), the
// warp (one row) reduces them and lane 0 publishes.
__device__ __forceinline__ void publish_pass(uint32_t m2, int r, int nrows, unsigned *maxbits, bool &bad)
{
    unsigned m = max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu);
    if (m >= 0x7F80u) {
        bad = true;
        m = 0u;
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0 && m != 0u && r < nrows) atomicMax(&maxbits[r], m);
}

// mid() runs once the activation loads are in flight and before they are
// used: a caller issues its weight copies there, so that the activations do
// not queue behind them in the memory system.
template <int FMT, class Mid = NoMid>
__device__ void stage_x(const uint16_t *__restrict__ x, size_t ld, int len, int nrows, const int *src,
                        uint16_t *xs, int ks, int *sh, unsigned *maxbits, const Mid &mid = Mid())
{
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) maxbits[r] = 0u;
    __syncthreads();
    // 8-element chunks per row (whole units; one all-zero chunk when len is 0)
    const int cpr = len > 0 ? (len + 31) / 32 * 4 : 1;
    const StageMap mp(nrows, cpr);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    auto load = [&](int r, int c) {
        if (r >= nrows || c * 8 >= len) return zero;
        return *reinterpret_cast<const uint4 *>(x + (size_t)(src ? src[r] : r) * ld + c * 8);
    };
    bool bad = false;
    const int nj = mp.npass * mp.nq;  // chunks per thread
    if (nj <= STAGE_REG_CHUNKS) {
        uint4 cache[STAGE_REG_CHUNKS];
        {
            int p = 0, q = 0;
#pragma unroll
            for (int j = 0; j < STAGE_REG_CHUNKS; ++j) {
                cache[j] = j < nj ? load(mp.tr + p * mp.rp, mp.tc + q * mp.tpr) : zero;
                if (++q == mp.nq) {
                    q = 0;
                    ++p;
                }
            }
        }
        mid();
        {
            int p = 0, q = 0;
            uint32_t m2 = 0u;
#pragma unroll
            for (int j = 0; j < STAGE_REG_CHUNKS; ++j) {
                if (j >= nj) break;
                m2 = absmax_chunk(m2, cache[j]);
                if (++q == mp.nq) {
                    publish_pass(m2, mp.tr + p * mp.rp, nrows, maxbits, bad);
                    m2 = 0u;
                    q = 0;
                    ++p;
                }
            }
        }
        if (bad) {
            int p = 0, q = 0;
#pragma unroll
            for (int j = 0; j < STAGE_REG_CHUNKS; ++j) {
                if (j >= nj) break;
                const int r = mp.tr + p * mp.rp;
                const unsigned m = chunk_mag_exact(cache[j]);
                if (r < nrows && m != 0u) atomicMax(&maxbits[r], m);
                if (++q == mp.nq) {
                    q = 0;
                    ++p;
                }
            }
        }
        __syncthreads();
        // every thread derives its row's exponent (the row's first thread
        // records it); the caller synchronises before sh is read
        int p = 0, q = 0;
        float f = 1.0f;
#pragma unroll
        for (int j = 0; j < STAGE_REG_CHUNKS; ++j) {
            if (j >= nj) break;
            const int r = mp.tr + p * mp.rp, c = mp.tc + q * mp.tpr;
            if (q == 0 && r < nrows) {
                const int e = stage_shift(maxbits[r]);
                if (mp.tc == 0) sh[r] = e;
                f = pow2f(-e);
            }
            if (r < nrows && c < cpr) stage_store(xs + (size_t)r * ks, c * 8, len, cache[j], f, FMT);
            if (++q == mp.nq) {
                q = 0;
                ++p;
            }
        }
        return;
    }
    mid();
    // pass 1: raw bf16 chunks into xs (element k of row r at xs[r*ks + k])
    // and the maxima, eight loads in flight per thread
    for (int p = 0; p < mp.npass; ++p) {
        const int r = mp.tr + p * mp.rp;
        uint32_t m2 = 0u;
        for (int q0 = 0; q0 < mp.nq; q0 += STAGE_REG_CHUNKS) {
            uint4 cache[STAGE_REG_CHUNKS];
#pragma unroll
            for (int j = 0; j < STAGE_REG_CHUNKS; ++j) {
                const int c = mp.tc + (q0 + j) * mp.tpr;
                cache[j] = c < cpr ? load(r, c) : zero;
            }
#pragma unroll
            for (int j = 0; j < STAGE_REG_CHUNKS; ++j) {
                const int c = mp.tc + (q0 + j) * mp.tpr;
                m2 = absmax_chunk(m2, cache[j]);
                if (r < nrows && c < cpr) *reinterpret_cast<uint4 *>(xs + (size_t)r * ks + c * 8) = cache[j];
            }
        }
        bool bad_p = false;
        publish_pass(m2, r, nrows, maxbits, bad_p);
        if (bad_p) {
            bad = true;
            for (int c = mp.tc; c < cpr && r < nrows; c += mp.tpr) {
                const unsigned m = chunk_mag_exact(*reinterpret_cast<const uint4 *>(xs + (size_t)r * ks + c * 8));
                if (m != 0u) atomicMax(&maxbits[r], m);
            }
        }
    }
    __syncthreads();
    // pass 2: convert in place.  MX layouts keep every element where it is
    // (a thread rewrites its own chunks); NVFP4 permutes within a 32-element
    // unit, so a thread takes whole units (reads all four chunks first).
    for (int p = 0; p < mp.npass; ++p) {
        const int r = mp.tr + p * mp.rp;
        if (r >= nrows) continue;
        uint16_t *row = xs + (size_t)r * ks;
        const int e = stage_shift(maxbits[r]);
        if (mp.tc == 0) sh[r] = e;
        const float f = pow2f(-e);
        if (FMT != FMT_NVFP4) {
            for (int c = mp.tc; c < cpr; c += mp.tpr)
                stage_store(row, c * 8, len, *reinterpret_cast<const uint4 *>(row + c * 8), f, FMT);
        } else {
            for (int u = mp.tc; u < cpr / 4; u += mp.tpr) {
                uint4 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = *reinterpret_cast<const uint4 *>(row + u * 32 + 8 * q);
#pragma unroll
                for (int q = 0; q < 4; ++q) stage_store(row, u * 32 + 8 * q, len, v[q], f, FMT);
            }
        }
    }
}

// Split of a token's power of two 2^sh: MX formats fold 2^min(sh, 0) into
// the block scales inside the loop (see compute_unit) and multiply the
// finished sum by 2^max(sh, 0); NVFP4 applies all of 2^sh to the finished
// sum (an E4M3 block scale times a partial of at most 2^9 cannot leave
// fp32's range).
template <int FMT>
__device__ __forceinline__ int sh_fold(int sh) { return FMT == FMT_NVFP4 ? 0 : min(sh, 0); }
template <int FMT>
__device__ __forceinline__ int sh_final(int sh) { return FMT == FMT_NVFP4 ? sh : max(sh, 0); }

// Token (0..MC-1) of the lane's accumulator column c: the m16n8k16 D
// fragment holds columns 2q and 2q + 1.
template <int MC>
__device__ __forceinline__ int acc_token(int c)
{
    return (2 * (threadIdx.x & 3) + c) / (8 / MC);
}

// -------------------------------------------------------------- loads

template <int FMT>
struct Ld;

template <>
struct Ld<FMT_MXFP4> {
    uint32_t c[2];
    uint32_t s;  // scale bytes of A rows g (low byte) and g+8
};
template <>
struct Ld<FMT_NVFP4> {
    uint32_t c[2];
    uint32_t s[2];  // two E4M3 block scales per A row (low byte: step 0)
};
template <>
struct Ld<FMT_MXFP8> {
    uint2 c[2];
    uint32_t s;
};

// Per-lane constants of one tile.
struct TileCtx {
    const uint8_t *cp[2];  // code pointer of A rows g, g+8, lane offset applied
    const uint8_t *sp[2];  // block-scale row pointer
    bool rv[2];            // weight row exists
    int b;                 // block offset within an MMA group
    int U;                 // 32-element units per row
    int KB16;              // NVFP4 16-element blocks per row
};

template <int FMT>
__device__ __forceinline__ void load_unit(const TileCtx &t, int u, bool ok, Ld<FMT> &l)
{
    if constexpr (FMT == FMT_MXFP4) {
        uint32_t s0 = 127u, s1 = 127u;
        l.c[0] = l.c[1] = 0u;
        if (ok && t.rv[0]) { l.c[0] = ld_nc_u32(t.cp[0] + (size_t)u * 16); s0 = ld_nc_u8(t.sp[0] + u); }
        if (ok && t.rv[1]) { l.c[1] = ld_nc_u32(t.cp[1] + (size_t)u * 16); s1 = ld_nc_u8(t.sp[1] + u); }
        l.s = s0 | (s1 << 8);
    } else if constexpr (FMT == FMT_MXFP8) {
        uint32_t s0 = 127u, s1 = 127u;
        l.c[0] = l.c[1] = make_uint2(0u, 0u);
        if (ok && t.rv[0]) { l.c[0] = ld_nc_u64(t.cp[0] + (size_t)u * 32); s0 = ld_nc_u8(t.sp[0] + u); }
        if (ok && t.rv[1]) { l.c[1] = ld_nc_u64(t.cp[1] + (size_t)u * 32); s1 = ld_nc_u8(t.sp[1] + u); }
        l.s = s0 | (s1 << 8);
    } else {
        const bool two = 2 * u + 1 < t.KB16;  // the unit's second 16-block exists
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t c = 0u, s = 0x3838u;  // E4M3 1.0, 1.0
            if (ok && t.rv[h]) {
                const uint8_t *cp = t.cp[h] + (size_t)u * 16;
                const uint8_t *sp = t.sp[h] + 2 * u;
                c = ld_nc_u16(cp);
                s = ld_nc_u8(sp) | 0x3800u;
                if (two) {
                    c |= ld_nc_u16(cp + 8) << 16;
                    s = (s & 0xFFu) | (ld_nc_u8(sp + 1) << 8);
                }
            }
            l.c[h] = c;
            l.s[h] = s;
        }
    }
}

// acc[h][c] += d (row half h, column c) times the block scale of half h
// (times the column's fold factor).
template <bool FOLD>
__device__ __forceinline__ void mx_accumulate(const float (&d)[4], float s0, float s1, const float (&f)[2],
                                              float (&acc)[2][2])
{
    if constexpr (FOLD) {
        acc[0][0] = fmaf(d[0], s0 * f[0], acc[0][0]);
        acc[0][1] = fmaf(d[1], s0 * f[1], acc[0][1]);
        acc[1][0] = fmaf(d[2], s1 * f[0], acc[1][0]);
        acc[1][1] = fmaf(d[3], s1 * f[1], acc[1][1]);
    } else {
        acc[0][0] = fmaf(d[0], s0, acc[0][0]);
        acc[0][1] = fmaf(d[1], s0, acc[0][1]);
        acc[1][0] = fmaf(d[2], s1, acc[1][0]);
        acc[1][1] = fmaf(d[3], s1, acc[1][1]);
    }
}

// One MMA group: BPM units (one per A-row block offset) -> acc[h][c].
// ok = false: the lane's unit lies outside the work; its fragments may hold
// stale data, so nothing is accumulated (the quad that shares the A rows
// and B column has the same ok).
// FOLD (MX formats): the E8M0 block scale of accumulator column c is
// multiplied by f[c] = 2^min(sh, 0) of that column's token first, so a block
// partial enters the sum already in the output's scale.  A token whose
// activations are all below 1 is staged scaled up by 2^-sh; without the
// fold a huge block scale (E8M0 above ~245) could overflow the fp32 partial
// that the final 2^sh would have brought back into range.  f <= 1, so the
// folded scale never overflows (a zero partial times it stays zero).
template <int FMT, bool FOLD = false>
__device__ __forceinline__ void compute_unit(const Ld<FMT> &l, const uint32_t (&B)[4], float (&acc)[2][2],
                                             bool ok = true, const float (&f)[2] = {1.f, 1.f})
{
    const float z[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (FMT == FMT_MXFP8) {
        float d[4];
        uint32_t a[4];
        // step 0 uses word .x of each A row, step 1 word .y
        e4m3x4_to_f16x2(l.c[0].x, a[0], a[2]);
        e4m3x4_to_f16x2(l.c[1].x, a[1], a[3]);
        mma_f16_16816(d, a, B[0], B[1], z);
        e4m3x4_to_f16x2(l.c[0].y, a[0], a[2]);
        e4m3x4_to_f16x2(l.c[1].y, a[1], a[3]);
        mma_f16_16816(d, a, B[2], B[3], d);
        float s0, s1;
        e8m0x2_to_f32(l.s, s0, s1);
        if (ok) mx_accumulate<FOLD>(d, s0, s1, f, acc);
    } else {
        // bytes 0,1 of a row's word feed MMA step 0 (A cols 2q.. and 2q+8..),
        // bytes 2,3 feed step 1
        uint32_t a0[4], a1[4];
        e2m1x8_to_f16x2(l.c[0], a0[0], a0[2], a1[0], a1[2]);
        e2m1x8_to_f16x2(l.c[1], a0[1], a0[3], a1[1], a1[3]);
        if constexpr (FMT == FMT_MXFP4) {
            float d[4];
            mma_f16_16816(d, a0, B[0], B[1], z);
            mma_f16_16816(d, a1, B[2], B[3], d);
            float s0, s1;
            e8m0x2_to_f32(l.s, s0, s1);
            if (ok) mx_accumulate<FOLD>(d, s0, s1, f, acc);
        } else {
            float d0[4], d1[4];
            mma_f16_16816(d0, a0, B[0], B[1], z);
            mma_f16_16816(d1, a1, B[2], B[3], z);
            const uint32_t f0 = e4m3x2_to_f16x2(l.s[0]), f1 = e4m3x2_to_f16x2(l.s[1]);
            const float s00 = f16_lo_to_f32(f0), s01 = f16_hi_to_f32(f0);
            const float s10 = f16_lo_to_f32(f1), s11 = f16_hi_to_f32(f1);
            if (ok) {
                acc[0][0] = fmaf(d1[0], s01, fmaf(d0[0], s00, acc[0][0]));
                acc[0][1] = fmaf(d1[1], s01, fmaf(d0[1], s00, acc[0][1]));
                acc[1][0] = fmaf(d1[2], s11, fmaf(d0[2], s10, acc[1][0]));
                acc[1][1] = fmaf(d1[3], s11, fmaf(d0[3], s10, acc[1][1]));
            }
        }
    }
}

// Stream MMA iterations [it0, it1) of one tile (2*MC weight rows from row0)
// and accumulate the lane's fragment partial sums into acc[h][c].
// xrow: this lane's B-column activation row in xs, or -1 for a padding
// column.
// FOLD, f: see compute_unit.
template <int FMT, int MC, int UF, bool FOLD = false>
__device__ __forceinline__ void qmv_tile(const uint8_t *__restrict__ codes,
                                         const uint8_t *__restrict__ scales, int N, int K,
                                         int row0, int it0, int it1, const uint16_t *xs, int ks,
                                         int xrow, float (&acc)[2][2], const float (&f)[2] = {1.f, 1.f})
{
    constexpr int BPM = 8 / MC;
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    TileCtx t;
    t.b = g % BPM;
    t.U = (K + 31) / 32;
    t.KB16 = K / 16;
    const size_t rb = FMT == FMT_MXFP8 ? (size_t)K : (size_t)K / 2;
    const size_t sb = FMT == FMT_NVFP4 ? (size_t)(K / 16) : (size_t)(K / 32);
    const int lane_off = FMT == FMT_MXFP8 ? 8 * q : (FMT == FMT_NVFP4 ? 2 * q : 4 * q);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = row0 + h * MC + g / BPM;
        t.rv[h] = row < N;
        const int rr = t.rv[h] ? row : 0;
        t.cp[h] = codes + (size_t)rr * rb + lane_off;
        t.sp[h] = scales + (size_t)rr * sb;
    }
    const uint16_t *xp = xrow >= 0 ? xs + (size_t)xrow * ks + 8 * q : nullptr;

    Ld<FMT> cur[UF], nxt[UF];
#pragma unroll
    for (int j = 0; j < UF; ++j) {
        const int it = it0 + j, u = it * BPM + t.b;
        load_unit<FMT>(t, u, it < it1 && u < t.U, cur[j]);
    }
    for (int itb = it0; itb < it1; itb += UF) {
        const bool more = itb + UF < it1;
#pragma unroll
        for (int j = 0; j < UF; ++j) {
            const int it = itb + UF + j, u = it * BPM + t.b;
            if (more) load_unit<FMT>(t, u, it < it1 && u < t.U, nxt[j]);
        }
#pragma unroll
        for (int j = 0; j < UF; ++j) {
            const int it = itb + j, u = it * BPM + t.b;
            if (it < it1) {
                uint32_t B[4] = {0u, 0u, 0u, 0u};
                if (xp && u < t.U) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xp + (size_t)u * 32);
                    B[0] = v.x; B[1] = v.y; B[2] = v.z; B[3] = v.w;
                }
                compute_unit<FMT, FOLD>(cur[j], B, acc, true, f);
            }
        }
        if (more) {
#pragma unroll
            for (int j = 0; j < UF; ++j) cur[j] = nxt[j];
        }
    }
}

// Reduce a lane's fragment partials over the lanes that share a
// (weight row, token) pair.  After the call, lanes for which
// tile_out() returns true hold finished sums in v[h][c].
template <int MC>
__device__ __forceinline__ void qmv_warp_reduce(const float (&acc)[2][2], float (&v)[2][2])
{
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if constexpr (MC == 8) {
            v[h][0] = acc[h][0];
            v[h][1] = acc[h][1];
        } else {
            float x;
            if constexpr (MC == 1) x = (q == (g >> 1)) ? acc[h][g & 1] : 0.f;
            else if constexpr (MC == 2) x = ((q & 1) == ((g >> 1) & 1)) ? acc[h][g & 1] : 0.f;
            else x = acc[h][g & 1];
            if constexpr (MC == 1) {
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 16);
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 8);
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 2);
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
            } else if constexpr (MC == 2) {
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 8);
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
            } else {
                x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
            }
            v[h][0] = x;
            v[h][1] = 0.f;
        }
    }
}

// Which (tile row r, token t) a lane's finished v[h][c] belongs to; false
// when the lane holds no finished value for it.
template <int MC>
__device__ __forceinline__ bool tile_out(int h, int c, int &r, int &t)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    constexpr int BPM = 8 / MC;
    r = h * MC + g / BPM;
    if constexpr (MC == 8) {
        t = 2 * q + c;
        return true;
    } else if constexpr (MC == 1) {
        t = 0;
        return c == 0 && lane == 0;  // after the full-warp sum lane 0 holds both rows
    } else if constexpr (MC == 2) {
        t = q >> 1;
        return c == 0 && (g & 3) == 0 && (q & 1) == 0;
    } else {
        t = q;
        return c == 0 && (g & 1) == 0;
    }
}

// The lane's B column: which token (0..MC-1) it carries.
template <int MC>
__device__ __forceinline__ int lane_token()
{
    return ((threadIdx.x & 31) >> 2) / (8 / MC);
}

__device__ __forceinline__ int warp_incl_scan(int v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Exclusive prefix sum of a[0..n) in shared memory (whole block calls);
// returns the total.  tmp: >= 33 ints of shared scratch.
__device__ inline int block_excl_scan(int *a, int n, int *tmp)
{
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int s = 0;
    for (int i = lo; i < hi; ++i) s += a[i];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int inc = warp_incl_scan(s);
    if (lane == 31) tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? tmp[lane] : 0;
        int wi = warp_incl_scan(w);
        if (lane < nw) tmp[lane] = wi - w;
        if (lane == 31) tmp[32] = wi;
    }
    __syncthreads();
    int run = tmp[warp] + inc - s;
    for (int i = lo; i < hi; ++i) {
        int v = a[i];
        a[i] = run;
        run += v;
    }
    const int total = tmp[32];
    __syncthreads();
    return total;
}

// Shared-memory arrays of the MoE routing step.
struct RouteSmem {
    int *cnt;       // [E]  per-expert counts, then first index in `sorted`
    int *wgs;       // [E]  first work group of each expert
    int *pos;       // [E]  placement cursors
    int *sorted;    // [P]  valid slots grouped by expert, increasing slot order inside a group
    int *wg_e;      // [P]  work group -> expert
    int *wg_first;  // [P]  work group -> first index in `sorted`
    int *wg_mc;     // [P]  work group -> member count (1..cap)
    int *tmp;       // [40] scan scratch
};

// Group the routed slots by expert on the device (every CTA computes the
// same result from expert_ids; nothing is copied to the host).  Slots with
// an id outside [0, E) are left out.  Work group w serves expert wg_e[w]
// for the slots sorted[wg_first[w] .. + wg_mc[w]), at most `cap` of them,
// so an expert routed from several tokens is streamed once per group.
// Whole block calls; returns the number of work groups.
__device__ inline int moe_route(const int32_t *ids, int P, int E, int cap, const RouteSmem &r)
{
    if (P <= 32) {
        // one warp, same result: groups in expert order, slots of an expert
        // in slot order
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int e = lane < P ? ids[lane] : -1;
            const bool valid = lane < P && e >= 0 && e < E;
            const int key = valid ? e : -1 - lane;
            const unsigned m = __match_any_sync(0xFFFFFFFFu, key);
            const int cnt = __popc(m), rank = __popc(m & ((1u << lane) - 1u));
            const bool leader = valid && rank == 0;
            const int nsub = leader ? (cnt + cap - 1) / cap : 0;
            // groups and slots of the experts below mine
            int gbase = 0, sbase = 0, nwg = 0;
            for (int j = 0; j < 32; ++j) {
                const int ej = __shfl_sync(0xFFFFFFFFu, key, j);
                const int lj = __shfl_sync(0xFFFFFFFFu, (int)leader, j);
                const int nj = __shfl_sync(0xFFFFFFFFu, nsub, j);
                const int cj = __shfl_sync(0xFFFFFFFFu, cnt, j);
                if (lj) {
                    nwg += nj;
                    if (ej < key) {
                        gbase += nj;
                        sbase += cj;
                    }
                }
            }
            const int lead_lane = __ffs(m) - 1;
            const int my_sbase = __shfl_sync(0xFFFFFFFFu, sbase, lead_lane);
            if (valid) r.sorted[my_sbase + rank] = lane;
            if (leader)
                for (int c = 0; c < nsub; ++c) {
                    r.wg_e[gbase + c] = e;
                    r.wg_first[gbase + c] = sbase + cap * c;
                    r.wg_mc[gbase + c] = min(cap, cnt - cap * c);
                }
            if (lane == 0) r.tmp[0] = nwg;
        }
        __syncthreads();
        return r.tmp[0];
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) r.cnt[e] = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int e = ids[p];
        if (e >= 0 && e < E) atomicAdd(&r.cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) r.wgs[e] = (r.cnt[e] + cap - 1) / cap;
    __syncthreads();
    const int nwg = block_excl_scan(r.wgs, E, r.tmp);
    block_excl_scan(r.cnt, E, r.tmp);  // counts -> starts
    for (int e = threadIdx.x; e < E; e += blockDim.x) r.pos[e] = r.cnt[e];
    __syncthreads();
    // stable placement (one warp, in slot order)
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        for (int base = 0; base < P; base += 32) {
            const int p = base + lane;
            int e = p < P ? ids[p] : -1;
            const bool valid = p < P && e >= 0 && e < E;
            if (!valid) e = -1 - (p & 0xFFFF);  // distinct keys for invalid lanes
            const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
            const int rank = __popc(m & ((1u << lane) - 1u));
            int at = 0;
            if (valid) at = r.pos[e] + rank;
            __syncwarp();
            if (valid) {
                r.sorted[at] = p;
                if (rank == 0) r.pos[e] += __popc(m);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int n = (e + 1 < E ? r.cnt[e + 1] : r.pos[e]) - r.cnt[e];  // members of e
        for (int c = 0; c * cap < n; ++c) {
            const int w = r.wgs[e] + c;
            r.wg_e[w] = e;
            r.wg_first[w] = r.cnt[e] + cap * c;
            r.wg_mc[w] = min(cap, n - cap * c);
        }
    }
    __syncthreads();
    return nwg;
}

}  // namespace mx
