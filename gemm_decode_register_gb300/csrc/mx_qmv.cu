// mx_qmv.cu -- decode GEMV (qmv) and MoE decode GEMV over block-float weights.
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
// token by a power of two into fp16 range (exact for bf16 inputs), form
// the B fragment.  To keep one block scale per MMA output while loads stay
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

int qmv_stage_bytes(int rows, int K)
{
    long long b = (long long)rows * stage_stride(K) * 2;
    return b > (1 << 30) ? -1 : (int)b;
}

// -------------------------------------------------------------- staging

// Stage activation rows (bf16 -> scaled f16, permuted per unit) into
// shared memory.  Row r of xs is source row src[r] (or r when src is null)
// of x [.][K].  sh[r] receives the per-row power-of-two exponent: the
// staged values are x * 2^-sh[r] with max |.| in [1, 2).
template <int FMT>
__device__ void stage_x(const uint16_t *__restrict__ x, int K, int nrows, const int *src,
                        uint16_t *xs, int ks, int *sh, unsigned *maxbits)
{
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) maxbits[r] = 0u;
    __syncthreads();
    // pass 1: largest magnitude per row (as bf16 bits; NaN > inf > finite)
    const int kp = K / 2;  // bf16 pairs per row
    for (int r = 0; r < nrows; ++r) {
        const uint32_t *row = reinterpret_cast<const uint32_t *>(x + (size_t)(src ? src[r] : r) * K);
        unsigned m = 0;
        for (int i = threadIdx.x; i < kp; i += blockDim.x) {
            uint32_t v = row[i];
            m = max(m, max(v & 0x7FFFu, (v >> 16) & 0x7FFFu));
        }
        if (m) atomicMax(&maxbits[r], m);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
        unsigned mb = maxbits[r];
        int ef = (int)(mb >> 7);
        int s = 0;
        if (mb != 0u && ef != 255) s = ef == 0 ? -126 : ef - 127;
        sh[r] = s;
    }
    __syncthreads();
    // pass 2: convert and permute (zero past K)
    const int U = (K + 31) / 32;
    const int pairs = U * 16;
    for (int idx = threadIdx.x; idx < nrows * pairs; idx += blockDim.x) {
        const int r = idx / pairs, pp = idx - r * pairs;
        const int k = 2 * pp;
        const int u = k >> 5, p = k & 31;
        int slot = p;
        if (FMT == FMT_NVFP4) slot = 8 * ((p & 15) >> 2) + 4 * (p >> 4) + (p & 3);
        uint32_t out = 0u;
        if (k < K) {
            uint32_t v = reinterpret_cast<const uint32_t *>(x + (size_t)(src ? src[r] : r) * K)[pp];
            float f = pow2f(-sh[r]);
            out = f32x2_to_f16x2(bf16_to_f32(v & 0xFFFFu) * f, bf16_to_f32(v >> 16) * f);
        }
        *reinterpret_cast<uint32_t *>(xs + (size_t)r * ks + u * 32 + slot) = out;
    }
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

// One MMA group: BPM units (one per A-row block offset) -> acc[h][c].
template <int FMT>
__device__ __forceinline__ void compute_unit(const Ld<FMT> &l, const uint32_t (&B)[4], float (&acc)[2][2])
{
    const float z[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (FMT == FMT_MXFP8) {
        float d[4];
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2(l.c[0].x);
        a[1] = e4m3x2_to_f16x2(l.c[1].x);
        a[2] = e4m3x2_to_f16x2(l.c[0].x >> 16);
        a[3] = e4m3x2_to_f16x2(l.c[1].x >> 16);
        mma_f16_16816(d, a, B[0], B[1], z);
        a[0] = e4m3x2_to_f16x2(l.c[0].y);
        a[1] = e4m3x2_to_f16x2(l.c[1].y);
        a[2] = e4m3x2_to_f16x2(l.c[0].y >> 16);
        a[3] = e4m3x2_to_f16x2(l.c[1].y >> 16);
        mma_f16_16816(d, a, B[2], B[3], d);
        float s0, s1;
        e8m0x2_to_f32(l.s, s0, s1);
        acc[0][0] = fmaf(d[0], s0, acc[0][0]);
        acc[0][1] = fmaf(d[1], s0, acc[0][1]);
        acc[1][0] = fmaf(d[2], s1, acc[1][0]);
        acc[1][1] = fmaf(d[3], s1, acc[1][1]);
    } else {
        uint32_t a0[4], a1[4];
        a0[0] = e2m1x2_to_f16x2(l.c[0]);
        a0[1] = e2m1x2_to_f16x2(l.c[1]);
        a0[2] = e2m1x2_to_f16x2(l.c[0] >> 8);
        a0[3] = e2m1x2_to_f16x2(l.c[1] >> 8);
        a1[0] = e2m1x2_to_f16x2(l.c[0] >> 16);
        a1[1] = e2m1x2_to_f16x2(l.c[1] >> 16);
        a1[2] = e2m1x2_to_f16x2(l.c[0] >> 24);
        a1[3] = e2m1x2_to_f16x2(l.c[1] >> 24);
        if constexpr (FMT == FMT_MXFP4) {
            float d[4];
            mma_f16_16816(d, a0, B[0], B[1], z);
            mma_f16_16816(d, a1, B[2], B[3], d);
            float s0, s1;
            e8m0x2_to_f32(l.s, s0, s1);
            acc[0][0] = fmaf(d[0], s0, acc[0][0]);
            acc[0][1] = fmaf(d[1], s0, acc[0][1]);
            acc[1][0] = fmaf(d[2], s1, acc[1][0]);
            acc[1][1] = fmaf(d[3], s1, acc[1][1]);
        } else {
            float d0[4], d1[4];
            mma_f16_16816(d0, a0, B[0], B[1], z);
            mma_f16_16816(d1, a1, B[2], B[3], z);
            const uint32_t f0 = e4m3x2_to_f16x2(l.s[0]), f1 = e4m3x2_to_f16x2(l.s[1]);
            const float s00 = f16_lo_to_f32(f0), s01 = f16_hi_to_f32(f0);
            const float s10 = f16_lo_to_f32(f1), s11 = f16_hi_to_f32(f1);
            acc[0][0] = fmaf(d1[0], s01, fmaf(d0[0], s00, acc[0][0]));
            acc[0][1] = fmaf(d1[1], s01, fmaf(d0[1], s00, acc[0][1]));
            acc[1][0] = fmaf(d1[2], s11, fmaf(d0[2], s10, acc[1][0]));
            acc[1][1] = fmaf(d1[3], s11, fmaf(d0[3], s10, acc[1][1]));
        }
    }
}

// Stream MMA iterations [it0, it1) of one tile (2*MC weight rows from row0)
// and accumulate the lane's fragment partial sums into acc[h][c].
// xrow: this lane's B-column activation row in xs, or -1 for a padding
// column.
template <int FMT, int MC, int UF>
__device__ __forceinline__ void qmv_tile(const uint8_t *__restrict__ codes,
                                         const uint8_t *__restrict__ scales, int N, int K,
                                         int row0, int it0, int it1, const uint16_t *xs, int ks,
                                         int xrow, float (&acc)[2][2])
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
                compute_unit<FMT>(cur[j], B, acc);
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

// -------------------------------------------------------------- dense qmv

struct QmvArgs {
    const uint8_t *codes;
    const uint8_t *scales;
    const uint16_t *x;  // bf16 [M][K]
    float *y;           // [M][N]
    int N, K;
    int m0, mc;  // token chunk
    int wk;      // warps that split K for one tile (divides QMV_WARPS)
    int tiles;   // ceil(N / (2*MC))
    int ks;      // staged row stride
};

template <int FMT, int MC>
__global__ void __launch_bounds__(QMV_THREADS, 1) qmv_kernel(QmvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + (size_t)MC * a.ks * 2);  // [warps][2MC][MC]
    int *sh = reinterpret_cast<int *>(red + QMV_WARPS * 2 * MC * MC);     // [MC]
    unsigned *maxbits = reinterpret_cast<unsigned *>(sh + 8);              // [MC]

    stage_x<FMT>(a.x + (size_t)a.m0 * a.K, a.K, a.mc, nullptr, xs, a.ks, sh, maxbits);
    __syncthreads();

    constexpr int BPM = 8 / MC;
    constexpr int RT = 2 * MC;
    const int warp = threadIdx.x >> 5;
    const int wr = warp / a.wk, wkk = warp - wr * a.wk;
    const int WR = QMV_WARPS / a.wk;
    const int U = (a.K + 31) / 32;
    const int iters = (U + BPM - 1) / BPM;
    const int per = (iters + a.wk - 1) / a.wk;
    const int it0 = min(iters, wkk * per), it1 = min(iters, it0 + per);
    const int tok = lane_token<MC>();
    const int xrow = tok < a.mc ? tok : -1;
    float g = 1.0f;
    if (FMT == FMT_NVFP4) g = load_f32_unaligned(a.scales + (size_t)a.N * (a.K / 16));

    for (int base = blockIdx.x * WR; base < a.tiles; base += gridDim.x * WR) {
        const int tile = base + wr;
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (tile < a.tiles)
            qmv_tile<FMT, MC, dense_uf<FMT>()>(a.codes, a.scales, a.N, a.K, tile * RT, it0, it1, xs,
                                                a.ks, xrow, acc);
        float v[2][2];
        qmv_warp_reduce<MC>(acc, v);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                int r, t;
                if (tile_out<MC>(h, c, r, t)) red[(warp * RT + r) * MC + t] = v[h][c];
            }
        __syncthreads();
        for (int i = threadIdx.x; i < WR * RT * MC; i += blockDim.x) {
            const int w = i / (RT * MC), rt = i - w * RT * MC, r = rt / MC, t = rt - r * MC;
            const int row = (base + w) * RT + r;
            if (base + w < a.tiles && row < a.N && t < a.mc) {
                float s = 0.f;
                for (int k = 0; k < a.wk; ++k) s += red[((w * a.wk + k) * RT + r) * MC + t];
                s *= pow2f(sh[t]);
                if (FMT == FMT_NVFP4) s *= g;
                a.y[(size_t)(a.m0 + t) * a.N + row] = s;
            }
        }
        __syncthreads();
    }
}

template <int FMT, int MC>
static cudaError_t run_qmv(const DeviceState &ds, cudaStream_t st, const QmvArgs &a)
{
    const size_t smem = (size_t)MC * a.ks * 2 + QMV_WARPS * 2 * MC * MC * 4 + 16 * 4;
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(qmv_kernel<FMT, MC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ds.max_smem_optin);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    const int WR = QMV_WARPS / a.wk;
    int rounds = (a.tiles + WR - 1) / WR;
    int grid = rounds < ds.num_sms ? rounds : ds.num_sms;
    qmv_kernel<FMT, MC><<<grid, QMV_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

template <int FMT>
static cudaError_t qmv_dispatch(const DeviceState &ds, cudaStream_t st, QmvArgs a, int MC)
{
    switch (MC) {
    case 1: return run_qmv<FMT, 1>(ds, st, a);
    case 2: return run_qmv<FMT, 2>(ds, st, a);
    case 4: return run_qmv<FMT, 4>(ds, st, a);
    default: return run_qmv<FMT, 8>(ds, st, a);
    }
}

static int round_mc(int m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : 8; }

cudaError_t launch_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K)
{
    const int ks = stage_stride(K);
    // tokens per pass: up to 8, bounded by shared memory
    auto bytes = [&](int mc) { return (size_t)mc * ks * 2 + QMV_WARPS * 2 * mc * mc * 4 + 64; };
    int cap = 8;
    while (cap > 1 && bytes(cap) > (size_t)ds.max_smem_optin) cap >>= 1;
    if (bytes(1) > (size_t)ds.max_smem_optin) return cudaErrorInvalidValue;
    for (int m0 = 0; m0 < M; m0 += cap) {
        const int mc = M - m0 < cap ? M - m0 : cap;
        const int MC = round_mc(mc);
        QmvArgs a;
        a.codes = codes;
        a.scales = scales;
        a.x = x;
        a.y = y;
        a.N = N;
        a.K = K;
        a.m0 = m0;
        a.mc = mc;
        a.ks = ks;
        a.tiles = (N + 2 * MC - 1) / (2 * MC);
        // K split: aim for >= 8 MMA iterations per warp
        const int iters = ((K + 31) / 32 + (8 / MC) - 1) / (8 / MC);
        int wk = 1;
        while (wk < QMV_WARPS && iters / (wk * 2) >= 8) wk *= 2;
        // keep enough tiles in flight when the matrix is short
        while (wk < QMV_WARPS && (long long)a.tiles * wk < 2LL * ds.num_sms * QMV_WARPS &&
               iters / (wk * 2) >= 2)
            wk *= 2;
        a.wk = wk;
        cudaError_t e;
        if (fmt == FMT_MXFP4) e = qmv_dispatch<FMT_MXFP4>(ds, st, a, MC);
        else if (fmt == FMT_MXFP8) e = qmv_dispatch<FMT_MXFP8>(ds, st, a, MC);
        else e = qmv_dispatch<FMT_NVFP4>(ds, st, a, MC);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// -------------------------------------------------------------- MoE qmv
//
// Routing on the device: every CTA reads expert_ids, groups the slots by
// expert (stable counting sort), and splits each expert's slots into work
// groups of at most 8.  A work item is (work group, tile of 2*MC rows); a
// warp streams the tile's rows of that expert once for all the group's
// tokens.  Experts that no slot routes to are never read.

struct MoeArgs {
    const uint8_t *codes;   // expert 0
    const uint8_t *scales;  // expert 0
    const uint16_t *x;      // bf16 [T][K]
    const int32_t *ids;     // [T*topk]
    float *y;               // [T*topk][N]
    int *err;
    int T, E, topk, N, K;
    int ks;
};

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
__device__ int block_excl_scan(int *a, int n, int *tmp)
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

template <int FMT, int MC>
__device__ __forceinline__ void moe_item(const MoeArgs &a, const uint8_t *ec, const uint8_t *es, float g,
                                         int tile, const int *mem, int mc, const uint16_t *xs,
                                         const int *sh)
{
    constexpr int RT = 2 * MC;
    const int U = (a.K + 31) / 32;
    const int iters = (U + (8 / MC) - 1) / (8 / MC);
    const int tok = lane_token<MC>();
    const int xrow = tok < mc ? mem[tok] / a.topk : -1;
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    qmv_tile<FMT, MC, MOE_UF>(ec, es, a.N, a.K, tile * RT, 0, iters, xs, a.ks, xrow, acc);
    float v[2][2];
    qmv_warp_reduce<MC>(acc, v);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            int r, t;
            if (tile_out<MC>(h, c, r, t)) {
                const int row = tile * RT + r;
                if (row < a.N && t < mc) {
                    const int slot = mem[t];
                    float s = v[h][c] * pow2f(sh[slot / a.topk]);
                    if (FMT == FMT_NVFP4) s *= g;
                    a.y[(size_t)slot * a.N + row] = s;
                }
            }
        }
}

template <int FMT>
__global__ void __launch_bounds__(QMV_THREADS, 1) moe_qmv_kernel(MoeArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int P = a.T * a.topk;
    // shared layout
    int *cnt = reinterpret_cast<int *>(smem);  // [E] counts -> starts
    int *wgs = cnt + a.E;                     // [E] work-group starts
    int *pos = wgs + a.E;                     // [E] placement cursors
    int *sorted = pos + a.E;                  // [P] slots grouped by expert
    int *wg_e = sorted + P;                   // [P] work group -> expert
    int *wg_first = wg_e + P;                 // [P] work group -> first index in sorted
    int *wg_mc = wg_first + P;                // [P]
    int *item0 = wg_mc + P;                   // [P + 1] first item of each work group
    int *tmp = item0 + P + 1;                 // [40]
    int *sh = tmp + 40;                       // [T] per-row exponents
    unsigned *maxbits = reinterpret_cast<unsigned *>(sh + a.T);  // [T]
    uint16_t *xs = reinterpret_cast<uint16_t *>(
        smem + ((((size_t)(3 * a.E + 5 * P + 41 + 2 * a.T) * 4) + 15) & ~(size_t)15));

    for (int e = threadIdx.x; e < a.E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int e = a.ids[p];
        if (e >= 0 && e < a.E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) wgs[e] = (cnt[e] + 7) >> 3;
    __syncthreads();
    const int nwg = block_excl_scan(wgs, a.E, tmp);
    block_excl_scan(cnt, a.E, tmp);  // cnt -> starts
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) pos[e] = cnt[e];
    __syncthreads();
    // stable placement (one warp, in slot order)
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        for (int base = 0; base < P; base += 32) {
            const int p = base + lane;
            int e = p < P ? a.ids[p] : -1;
            const bool valid = p < P && e >= 0 && e < a.E;
            if (!valid) e = -1 - (p & 0xFFFF);  // distinct keys for invalid lanes
            const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
            const int rank = __popc(m & ((1u << lane) - 1u));
            int at = 0;
            if (valid) at = pos[e] + rank;
            __syncwarp();
            if (valid) {
                sorted[at] = p;
                if (rank == 0) pos[e] += __popc(m);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // work groups
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        const int n = (e + 1 < a.E ? cnt[e + 1] : pos[e]) - cnt[e];  // members of e
        for (int c = 0; c * 8 < n; ++c) {
            const int w = wgs[e] + c;
            wg_e[w] = e;
            wg_first[w] = cnt[e] + 8 * c;
            wg_mc[w] = min(8, n - 8 * c);
        }
    }
    __syncthreads();
    for (int w = threadIdx.x; w < nwg; w += blockDim.x) {
        const int mcw = wg_mc[w];
        const int MCw = mcw <= 1 ? 1 : mcw <= 2 ? 2 : mcw <= 4 ? 4 : 8;
        item0[w] = (a.N + 2 * MCw - 1) / (2 * MCw);
    }
    __syncthreads();
    const int items = block_excl_scan(item0, nwg, tmp);
    if (threadIdx.x == 0) item0[nwg] = items;
    // invalid ids: flag and fill with NaN (rows split over CTAs)
    for (int p = blockIdx.x; p < P; p += gridDim.x) {
        const int e = a.ids[p];
        if (e < 0 || e >= a.E) {
            if (threadIdx.x == 0) set_device_error(a.err, DEVERR_BAD_EXPERT);
            for (int n = threadIdx.x; n < a.N; n += blockDim.x) a.y[(size_t)p * a.N + n] = __int_as_float(0x7FC00000);
        }
    }
    stage_x<FMT>(a.x, a.K, a.T, nullptr, xs, a.ks, sh, maxbits);
    __syncthreads();

    const size_t rb = FMT == FMT_MXFP8 ? (size_t)a.K : (size_t)a.K / 2;
    const size_t sbytes = FMT == FMT_NVFP4 ? (size_t)(a.K / 16) : (size_t)(a.K / 32);
    const int warp = threadIdx.x >> 5;
    for (int it = blockIdx.x * QMV_WARPS + warp; it < items; it += gridDim.x * QMV_WARPS) {
        int lo = 0, hi = nwg - 1;  // last work group with item0 <= it
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (item0[mid] <= it) lo = mid;
            else hi = mid - 1;
        }
        const int w = lo, tile = it - item0[w];
        const int e = wg_e[w], mc = wg_mc[w];
        const int *mem = sorted + wg_first[w];
        const uint8_t *ec = a.codes + (size_t)e * a.N * rb;
        const uint8_t *es = a.scales + (size_t)e * a.N * sbytes;
        float g = 1.0f;
        if (FMT == FMT_NVFP4) g = load_f32_unaligned(a.scales + (size_t)a.E * a.N * sbytes + 4 * (size_t)e);
        if (mc <= 1) moe_item<FMT, 1>(a, ec, es, g, tile, mem, mc, xs, sh);
        else if (mc <= 2) moe_item<FMT, 2>(a, ec, es, g, tile, mem, mc, xs, sh);
        else if (mc <= 4) moe_item<FMT, 4>(a, ec, es, g, tile, mem, mc, xs, sh);
        else moe_item<FMT, 8>(a, ec, es, g, tile, mem, mc, xs, sh);
    }
}

static size_t moe_smem_bytes(int T, int E, int P, int ks)
{
    size_t head = (((size_t)(3 * E + 5 * P + 41 + 2 * T) * 4) + 15) & ~(size_t)15;
    return head + (size_t)T * ks * 2;
}

template <int FMT>
static cudaError_t run_moe(const DeviceState &ds, cudaStream_t st, const MoeArgs &a, size_t smem)
{
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(moe_qmv_kernel<FMT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ds.max_smem_optin);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    moe_qmv_kernel<FMT><<<ds.num_sms, QMV_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_moe_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, const uint16_t *x, const int32_t *ids, float *y,
                           int T, int E, int topk, int N, int K)
{
    MoeArgs a;
    a.codes = codes;
    a.scales = scales;
    a.x = x;
    a.ids = ids;
    a.y = y;
    a.err = ds.err;
    a.T = T;
    a.E = E;
    a.topk = topk;
    a.N = N;
    a.K = K;
    a.ks = stage_stride(K);
    const size_t smem = moe_smem_bytes(T, E, T * topk, a.ks);
    if (smem > (size_t)ds.max_smem_optin) return cudaErrorInvalidValue;
    if (fmt == FMT_MXFP4) return run_moe<FMT_MXFP4>(ds, st, a, smem);
    if (fmt == FMT_MXFP8) return run_moe<FMT_MXFP8>(ds, st, a, smem);
    return run_moe<FMT_NVFP4>(ds, st, a, smem);
}

}  // namespace mx
