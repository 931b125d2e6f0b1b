// mx_stream.cuh -- the weight stream shared by the streaming decode GEMV
// kernels (dense: mx_qmv_stream.cu, MoE: mx_moe_stream.cu).
//
// Same arithmetic as the direct-load kernels (mx_qmv_core.cuh: codes decoded
// by cvt into m16n8k16 fragments, block scale applied per block), but the
// weight bytes reach the SM through a per-warp shared-memory ring fed by
// 16-byte cp.async copies: every warp keeps S - 1 ~2.4 KB stages (codes plus
// block scales of its rows) in flight while it decodes one, so that the
// bytes outstanding per SM cost no registers, and each copy instruction
// moves 512 contiguous bytes.
//
// Work is cut into units (2*MC weight rows x a run of K) that each warp
// streams back to back: the ring runs continuously across units.
#pragma once
#include <algorithm>

#include "mx_qmv_core.cuh"

namespace mx {
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage geometry for one (format, tokens-per-pass) pair.
template <int FMT, int MC>
struct SGeo {
    static constexpr int BPM = 8 / MC;                             // units per MMA
    static constexpr int RT = 2 * MC;                              // weight rows per tile
    static constexpr int UCB = FMT == FMT_MXFP8 ? 32 : 16;        // code bytes per 32-element unit
    static constexpr int IPS = FMT == FMT_MXFP8 ? 4 : 8;          // MMA iterations per stage
    static constexpr int UPS = IPS * BPM;                          // units per row per stage
    static constexpr int CB = UPS * UCB;                           // code bytes per row per stage
    static constexpr int SPU = FMT == FMT_NVFP4 ? 2 : 1;           // scale bytes per unit
    static constexpr int SB = UPS * SPU;                           // scale bytes per row per stage
    // Paired units (MC <= 4): lane group g decodes, for tile row g / HB, the
    // units 2j and 2j + 1 (j = g % HB) of each MMA iteration as A rows g and
    // g + 8; the two block scales are adjacent bytes and only the two
    // accumulators of matching blocks are kept.  MC = 8 (one unit per MMA
    // iteration and row) keeps A rows g and g + 8 as tile rows g and 8 + g.
    static constexpr bool PAIR = MC <= 4;
    static constexpr int HB = PAIR ? BPM / 2 : 1;                 // lane groups per tile row
    // Shared-memory offset of tile row r: rows are CB bytes plus a pad whose
    // size spreads the 8 lane groups' loads of one iteration over the banks.
    __host__ __device__ static constexpr int row_base(int r)
    {
        return !PAIR ? r * (CB + (FMT == FMT_MXFP8 ? 256 : 128) / MC)
               : FMT == FMT_MXFP8 ? r * (CB + 32)
                                  : r * CB + 16 * ((r & 1) + (r >> 1) * 2 * HB);
    }
    static constexpr int CODE_BYTES = (row_base(RT - 1) + CB + 15) / 16 * 16;
    static constexpr int STAGE_BYTES = CODE_BYTES + RT * SB;
    // ring depth: one stage in decode, the rest in flight (short tiles leave
    // room in shared memory for a deeper ring)
    static constexpr int STAGES = MC <= 2 ? 4 : 3;
    static constexpr int PIECES = RT * CB / 16;                    // 16-byte code copies per stage
    static constexpr int SWORDS = RT * SB / 4;                     // 4-byte scale copies per stage
    static_assert(PIECES % 32 == 0, "code copies per lane");
    static_assert(STAGE_BYTES % 16 == 0, "stage alignment");
};

// One unit of a warp's stream.
struct SUnit {
    const uint8_t *codes;   // matrix (expert) base
    const uint8_t *scales;  // block-scale base
    int row0;               // first weight row of the tile
    int ub, ul;             // units [ub, ul)
    // Tile row r (of 2*MC) is weight row row0 + r % MC + (r / MC) * jump,
    // valid while row0 + r % MC < lim (and the row is inside the matrix):
    // jump = MC, lim = N for a contiguous tile; jump = lim = I pairs gate row
    // i with up row I + i.
    int jump, lim;
};

template <int FMT, int MC>
__device__ __forceinline__ int unit_stages(const SUnit &u)
{
    using G = SGeo<FMT, MC>;
    return u.ul > u.ub ? (u.ul - u.ub + G::UPS - 1) / G::UPS : 0;
}

// A lane's share of the copies of one unit, resolved once per unit:
// source pointers at the unit's first stage, bytes left in the row after
// them (<= 0: nothing to copy), and destination offsets within a ring slot.
template <int FMT, int MC>
struct CopyPlan {
    using G = SGeo<FMT, MC>;
    static constexpr int NP = G::PIECES / 32;
    static constexpr int NW = (G::SWORDS + 31) / 32;
    const uint8_t *src[NP];
    int left[NP];
    const uint8_t *ssrc[NW];
    int sleft[NW];
};

// Lane constants of the copy mapping (independent of the unit).
template <int FMT, int MC>
struct CopyLane {
    using G = SGeo<FMT, MC>;
    int row[CopyPlan<FMT, MC>::NP], off[CopyPlan<FMT, MC>::NP], dst[CopyPlan<FMT, MC>::NP];
    int srow[CopyPlan<FMT, MC>::NW], soff[CopyPlan<FMT, MC>::NW];
    __device__ __forceinline__ CopyLane()
    {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < CopyPlan<FMT, MC>::NP; ++j) {
            const int p = lane + 32 * j;
            row[j] = p / (G::CB / 16);
            off[j] = (p % (G::CB / 16)) * 16;
            dst[j] = G::row_base(row[j]) + off[j];
        }
#pragma unroll
        for (int j = 0; j < CopyPlan<FMT, MC>::NW; ++j) {
            const int w = lane + 32 * j;
            srow[j] = w < G::SWORDS ? w / (G::SB / 4) : 0;
            soff[j] = (w % (G::SB / 4)) * 4;
        }
    }
};

template <int FMT, int MC>
__device__ __forceinline__ void plan_copies(const SUnit &u, const CopyLane<FMT, MC> &cl, int N, int RB, int KS,
                                            CopyPlan<FMT, MC> &c)
{
    using G = SGeo<FMT, MC>;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < c.NP; ++j) {
        const int base = u.row0 + cl.row[j] % MC;
        const int grow = base + (cl.row[j] / MC) * u.jump;
        const bool ok = base < u.lim && grow < N;
        const int col = u.ub * G::UCB + cl.off[j];
        c.src[j] = u.codes + (size_t)(ok ? grow : 0) * RB + col;
        c.left[j] = ok ? RB - col : 0;
    }
#pragma unroll
    for (int j = 0; j < c.NW; ++j) {
        const int base = u.row0 + cl.srow[j] % MC;
        const int grow = base + (cl.srow[j] / MC) * u.jump;
        const bool ok = base < u.lim && grow < N;
        const int col = u.ub * G::SPU + cl.soff[j];
        c.ssrc[j] = u.scales + (size_t)(ok ? grow : 0) * KS + col;
        c.sleft[j] = (ok && lane + 32 * j < G::SWORDS) ? KS - col : 0;
    }
}

// Copy stage s of the planned unit into the ring slot at shared address dst.
template <int FMT, int MC>
__device__ __forceinline__ void copy_stage(const CopyPlan<FMT, MC> &c, const CopyLane<FMT, MC> &cl, int s,
                                           uint32_t dst)
{
    using G = SGeo<FMT, MC>;
    const int cs = s * G::CB, ss = s * G::SB;
#pragma unroll
    for (int j = 0; j < c.NP; ++j)
        if (cs < c.left[j]) cp_async16(dst + cl.dst[j], c.src[j] + cs);
#pragma unroll
    for (int j = 0; j < c.NW; ++j)
        if (ss < c.sleft[j]) cp_async4(dst + G::CODE_BYTES + cl.srow[j] * G::SB + cl.soff[j], c.ssrc[j] + ss);
}

// One MMA group of the paired-unit layout: A row g holds unit 2j and A row
// g + 8 unit 2j + 1 of the same weight row (l.s: their scales, low byte
// first; NVFP4: two bytes each).  Only the products of matching blocks are
// accumulated: acc[0][0] (unit 2j, B column 2q) and acc[1][1] (unit 2j + 1,
// B column 2q + 1); on lanes with q % HB == j both belong to token q / HB.
// ok = false: the lane's units lie outside the work (nothing accumulated).
// FOLD, f: as compute_unit (f[0] = f[1] here: one token per lane).
template <int FMT, bool FOLD>
__device__ __forceinline__ void compute_pair(const Ld<FMT> &l, const uint32_t (&B)[4], float (&acc)[2][2], bool ok,
                                             const float (&f)[2])
{
    const float z[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (FMT == FMT_MXFP8) {
        float d[4];
        uint32_t a[4];
        e4m3x4_to_f16x2(l.c[0].x, a[0], a[2]);
        e4m3x4_to_f16x2(l.c[1].x, a[1], a[3]);
        mma_f16_16816(d, a, B[0], B[1], z);
        e4m3x4_to_f16x2(l.c[0].y, a[0], a[2]);
        e4m3x4_to_f16x2(l.c[1].y, a[1], a[3]);
        mma_f16_16816(d, a, B[2], B[3], d);
        float s0, s1;
        e8m0x2_to_f32(l.s, s0, s1);
        if (ok) {
            acc[0][0] = fmaf(d[0], FOLD ? s0 * f[0] : s0, acc[0][0]);
            acc[1][1] = fmaf(d[3], FOLD ? s1 * f[1] : s1, acc[1][1]);
        }
    } else {
        uint32_t a0[4], a1[4];
        e2m1x8_to_f16x2(l.c[0], a0[0], a0[2], a1[0], a1[2]);
        e2m1x8_to_f16x2(l.c[1], a0[1], a0[3], a1[1], a1[3]);
        if constexpr (FMT == FMT_MXFP4) {
            float d[4];
            mma_f16_16816(d, a0, B[0], B[1], z);
            mma_f16_16816(d, a1, B[2], B[3], d);
            float s0, s1;
            e8m0x2_to_f32(l.s, s0, s1);
            if (ok) {
                acc[0][0] = fmaf(d[0], FOLD ? s0 * f[0] : s0, acc[0][0]);
                acc[1][1] = fmaf(d[3], FOLD ? s1 * f[1] : s1, acc[1][1]);
            }
        } else {
            // MMA step s covers 16-element block s of each unit
            float d0[4], d1[4];
            mma_f16_16816(d0, a0, B[0], B[1], z);
            mma_f16_16816(d1, a1, B[2], B[3], z);
            const uint32_t f0 = e4m3x2_to_f16x2(l.s[0]), f1 = e4m3x2_to_f16x2(l.s[1]);
            if (ok) {
                acc[0][0] = fmaf(d1[0], f16_hi_to_f32(f0), fmaf(d0[0], f16_lo_to_f32(f0), acc[0][0]));
                acc[1][1] = fmaf(d1[3], f16_hi_to_f32(f1), fmaf(d0[3], f16_lo_to_f32(f1), acc[1][1]));
            }
        }
    }
}

// End of a tile in the paired-unit layout: adds each tile row's HB lane
// groups (the lanes with q % HB == j hold a (row, token) pair's two
// accumulators, the others none).  Returns true on the lane left holding
// tile row r and token t, with the sum in v.
template <int MC>
__device__ __forceinline__ bool pair_reduce(const float (&acc)[2][2], float &v, int &r, int &t)
{
    constexpr int HB = 4 / MC;
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    float x = q % HB == g % HB ? acc[0][0] + acc[1][1] : 0.f;
    if constexpr (MC == 1) {
        // lanes 16r + 5j (j = 0..3) hold row r
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 8);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 2);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
        r = g >> 2;
        t = 0;
        v = x;
        return (lane & 15) == 0;
    } else if constexpr (MC == 2) {
        // lanes 8r + 2t and 8r + 2t + 5 hold (row r, token t)
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
        r = g >> 1;
        t = q >> 1;
        v = x;
        return (lane & 5) == 0;
    } else {
        r = g;
        t = q;
        v = x;
        return true;
    }
}

// Decode-and-multiply one stage from shared memory into acc.
// xrow: the lane's staged activation row (-1: padding column); xu0: the
// first unit held by the staged activations.  FULL: every unit of the stage
// lies inside the unit's range (no per-iteration checks).  FOLD, f: see
// compute_unit.
template <int FMT, int MC, bool FULL, bool FOLD>
__device__ __forceinline__ void compute_stage_impl(const SUnit &u, int s, const uint8_t *buf, const uint16_t *xs,
                                                   int ks, int xu0, int xrow, float (&acc)[2][2],
                                                   const float (&f)[2])
{
    using G = SGeo<FMT, MC>;
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int b = g % G::BPM;
    const int u0 = u.ub + s * G::UPS;
    const int lane_off = FMT == FMT_MXFP8 ? 8 * q : (FMT == FMT_NVFP4 ? 2 * q : 4 * q);
    const uint16_t *xp = xrow >= 0 ? xs + (size_t)xrow * ks + 8 * q + (size_t)(u0 + b - xu0) * 32 : nullptr;
    if constexpr (G::PAIR) {
        const int rr = g / G::HB, j = g % G::HB;  // tile row; its units 2j, 2j + 1 of each iteration
        const uint8_t *a0 = buf + G::row_base(rr) + 2 * j * G::UCB + lane_off;
        const uint8_t *sp = buf + G::CODE_BYTES + rr * G::SB + 2 * j * G::SPU;
#pragma unroll
        for (int it = 0; it < G::IPS; ++it) {
            const int rel = it * G::BPM;
            bool ok_a = true, ok_b = true;
            if constexpr (!FULL) {
                if (rel >= u.ul - u0) break;  // warp-uniform end of the unit
                ok_a = u0 + rel + 2 * j < u.ul;
                ok_b = u0 + rel + b < u.ul;
            }
            Ld<FMT> l;
            if constexpr (FMT == FMT_MXFP4) {
                l.c[0] = *reinterpret_cast<const uint32_t *>(a0 + rel * 16);
                l.c[1] = *reinterpret_cast<const uint32_t *>(a0 + rel * 16 + 16);
                l.s = *reinterpret_cast<const uint16_t *>(sp + rel);
            } else if constexpr (FMT == FMT_MXFP8) {
                l.c[0] = *reinterpret_cast<const uint2 *>(a0 + rel * 32);
                l.c[1] = *reinterpret_cast<const uint2 *>(a0 + rel * 32 + 32);
                l.s = *reinterpret_cast<const uint16_t *>(sp + rel);
            } else {
                l.c[0] = __byte_perm(*reinterpret_cast<const uint16_t *>(a0 + rel * 16),
                                     *reinterpret_cast<const uint16_t *>(a0 + rel * 16 + 8), 0x5410);
                l.c[1] = __byte_perm(*reinterpret_cast<const uint16_t *>(a0 + rel * 16 + 16),
                                     *reinterpret_cast<const uint16_t *>(a0 + rel * 16 + 24), 0x5410);
                const uint32_t w = *reinterpret_cast<const uint32_t *>(sp + rel * 2);
                l.s[0] = w & 0xFFFFu;
                l.s[1] = w >> 16;
            }
            uint32_t B[4] = {0u, 0u, 0u, 0u};
            if (xp && ok_b) {
                const uint4 v = *reinterpret_cast<const uint4 *>(xp + (size_t)rel * 32);
                B[0] = v.x;
                B[1] = v.y;
                B[2] = v.z;
                B[3] = v.w;
            }
            compute_pair<FMT, FOLD>(l, B, acc, ok_a, f);
        }
        return;
    }
    const int r0 = g / G::BPM, r1 = MC + g / G::BPM;
    const uint8_t *a0 = buf + G::row_base(r0) + b * G::UCB + lane_off;
    const uint8_t *a1 = buf + G::row_base(r1) + b * G::UCB + lane_off;
    const uint8_t *s0 = buf + G::CODE_BYTES + r0 * G::SB + b * G::SPU;
    const uint8_t *s1 = buf + G::CODE_BYTES + r1 * G::SB + b * G::SPU;
#pragma unroll
    for (int it = 0; it < G::IPS; ++it) {
        const int rel = it * G::BPM;
        bool ok = true;
        if constexpr (!FULL) {
            if (rel >= u.ul - u0) break;  // warp-uniform end of the unit
            ok = u0 + rel + b < u.ul;
        }
        Ld<FMT> l;
        if constexpr (FMT == FMT_MXFP4) {
            l.c[0] = *reinterpret_cast<const uint32_t *>(a0 + rel * 16);
            l.c[1] = *reinterpret_cast<const uint32_t *>(a1 + rel * 16);
            l.s = __byte_perm(s0[rel], s1[rel], 0x0040);
        } else if constexpr (FMT == FMT_MXFP8) {
            l.c[0] = *reinterpret_cast<const uint2 *>(a0 + rel * 32);
            l.c[1] = *reinterpret_cast<const uint2 *>(a1 + rel * 32);
            l.s = __byte_perm(s0[rel], s1[rel], 0x0040);
        } else {
            l.c[0] = __byte_perm(*reinterpret_cast<const uint16_t *>(a0 + rel * 16),
                                 *reinterpret_cast<const uint16_t *>(a0 + rel * 16 + 8), 0x5410);
            l.c[1] = __byte_perm(*reinterpret_cast<const uint16_t *>(a1 + rel * 16),
                                 *reinterpret_cast<const uint16_t *>(a1 + rel * 16 + 8), 0x5410);
            l.s[0] = *reinterpret_cast<const uint16_t *>(s0 + rel * 2);
            l.s[1] = *reinterpret_cast<const uint16_t *>(s1 + rel * 2);
        }
        uint32_t B[4] = {0u, 0u, 0u, 0u};
        if (xp && ok) {
            const uint4 v = *reinterpret_cast<const uint4 *>(xp + (size_t)rel * 32);
            B[0] = v.x;
            B[1] = v.y;
            B[2] = v.z;
            B[3] = v.w;
        }
        compute_unit<FMT, FOLD>(l, B, acc, ok, f);
    }
}

template <int FMT, int MC, bool FOLD>
__device__ __forceinline__ void compute_stage(const SUnit &u, int s, const uint8_t *buf, const uint16_t *xs,
                                              int ks, int xu0, int xrow, float (&acc)[2][2], const float (&f)[2])
{
    using G = SGeo<FMT, MC>;
    if (u.ul - (u.ub + s * G::UPS) >= G::UPS)
        compute_stage_impl<FMT, MC, true, FOLD>(u, s, buf, xs, ks, xu0, xrow, acc, f);
    else
        compute_stage_impl<FMT, MC, false, FOLD>(u, s, buf, xs, ks, xu0, xrow, acc, f);
}

// A warp's stream of units through its ring of S slots: copies run S-1
// stages ahead of the decode.  prime() issues the first copies (it may run
// before the activations are staged: the weights do not depend on them);
// run() decodes every stage and refills the ring as it goes.
// next(i) -> SUnit for the warp's unit i.
template <int FMT, int MC, class Next, int S = SGeo<FMT, MC>::STAGES>
struct Streamer {
    using G = SGeo<FMT, MC>;
    static_assert(S >= 2, "ring depth");
    const Next &next;
    int n_units, N, RB, KS;
    uint32_t ring_s;
    CopyLane<FMT, MC> cl;
    CopyPlan<FMT, MC> plan;
    int iu = -1, is = 0, ins = 0, slot_issue = 0;

    __device__ __forceinline__ Streamer(const Next &nx, int n, uint8_t *ring, int n_rows, int rb, int kscale)
        : next(nx), n_units(n), N(n_rows), RB(rb), KS(kscale), ring_s(smem_addr(ring))
    {
    }

    __device__ __forceinline__ void issue()
    {
        while (iu < n_units && (iu < 0 || is >= ins)) {
            ++iu;
            is = 0;
            if (iu < n_units) {
                const SUnit u = next(iu);
                ins = unit_stages<FMT, MC>(u);
                plan_copies<FMT, MC>(u, cl, N, RB, KS, plan);
            }
        }
        if (iu < n_units) {
            copy_stage<FMT, MC>(plan, cl, is, ring_s + slot_issue * G::STAGE_BYTES);
            ++is;
        }
        cp_async_commit();
        slot_issue = slot_issue + 1 == S ? 0 : slot_issue + 1;
    }

    // Issue `n` of the S - 1 stages in flight when the stream starts (n over
    // all calls before run() adds up to S - 1).
    __device__ __forceinline__ void prime(int n = S - 1)
    {
#pragma unroll
        for (int s = 0; s < S - 1; ++s)
            if (s < n) issue();
    }

    // xrow_of(i): the lane's activation row for unit i; done(i, acc): the
    // lane's fragment partial sums at the end of unit i; fold_of(i, f): the
    // fold factors of the lane's accumulator columns in unit i (FOLD only).
    template <bool FOLD, class XRow, class Done, class Fold>
    __device__ __forceinline__ void run(const XRow &xrow_of, const Done &done, const Fold &fold_of,
                                        const uint8_t *ring, const uint16_t *xs, int ks, int xu0)
    {
        int slot = 0;
        for (int cu = 0; cu < n_units; ++cu) {
            const SUnit cd = next(cu);
            const int nst = unit_stages<FMT, MC>(cd);
            const int xrow = xrow_of(cu);
            float f[2] = {1.f, 1.f};
            if constexpr (FOLD) fold_of(cu, f);
            float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            for (int cs = 0; cs < nst; ++cs) {
                cp_async_wait<S - 2>();
                __syncwarp();
                issue();  // refills the slot consumed one stage ago
                compute_stage<FMT, MC, FOLD>(cd, cs, ring + slot * G::STAGE_BYTES, xs, ks, xu0, xrow, acc, f);
                slot = slot + 1 == S ? 0 : slot + 1;
            }
            done(cu, acc);
        }
        cp_async_wait<0>();
        __syncwarp();
    }
};

// Rows must be 128-element aligned for the 16-byte copies of codes and the
// 4-byte copies of scales.
inline bool stream_ok(int, int K) { return K % 128 == 0; }

}  // namespace mx
