// mx_qmv_stream.cu -- decode GEMV and MoE decode GEMV, streaming variant.
//
// Same arithmetic as the direct-load kernels (mx_qmv_core.cuh: codes decoded
// by cvt into m16n8k16 fragments, block scale applied per block), but the
// weight bytes reach the SM through a per-warp shared-memory ring fed by
// 16-byte cp.async copies: every warp keeps two ~2.4 KB stages (codes plus
// block scales of its rows) in flight while it decodes the third, so an SM
// with 16 warps has ~80 KB of HBM reads outstanding without spending
// registers on them, and each copy instruction moves 512 contiguous bytes.
//
// Work is cut into units (2*MC weight rows x a run of K) that each warp
// streams back to back: the ring runs continuously across units.
//   * dense: a CTA's tiles go to its warps whole and round-robin when that
//     balances them; otherwise the CTA's stages (tile-major) are dealt out
//     in equal contiguous runs, so a tile's K is cut only where two runs
//     meet, and the pieces' partial sums are added in K order in shared
//     memory.  When the tokens' activations do not fit in shared memory, K
//     is also split across CTAs (windows); the windows' partial sums go to a
//     device workspace and the last CTA of a tile group adds them in window
//     order (deterministic).
//   * MoE: units are (work group of up to MC slots routed to one expert,
//     tile) over the whole K of that expert.
#include <algorithm>

#include "mx_qmv_core.cuh"

namespace mx {

constexpr int ST_RED_BUDGET = 24 * 1024;

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
    static constexpr int RS = CB + (FMT == FMT_MXFP8 ? 256 : 128) / MC;  // padded row stride
    static constexpr int SPU = FMT == FMT_NVFP4 ? 2 : 1;           // scale bytes per unit
    static constexpr int SB = UPS * SPU;                           // scale bytes per row per stage
    static constexpr int CODE_BYTES = RT * RS;
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
    int row[CopyPlan<FMT, MC>::NP], off[CopyPlan<FMT, MC>::NP];
    int srow[CopyPlan<FMT, MC>::NW], soff[CopyPlan<FMT, MC>::NW];
    __device__ __forceinline__ CopyLane()
    {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < CopyPlan<FMT, MC>::NP; ++j) {
            const int p = lane + 32 * j;
            row[j] = p / (G::CB / 16);
            off[j] = (p % (G::CB / 16)) * 16;
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
        if (cs < c.left[j]) cp_async16(dst + cl.row[j] * G::RS + cl.off[j], c.src[j] + cs);
#pragma unroll
    for (int j = 0; j < c.NW; ++j)
        if (ss < c.sleft[j]) cp_async4(dst + G::CODE_BYTES + cl.srow[j] * G::SB + cl.soff[j], c.ssrc[j] + ss);
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
    const int r0 = g / G::BPM, r1 = MC + g / G::BPM;
    const int u0 = u.ub + s * G::UPS;
    const int lane_off = FMT == FMT_MXFP8 ? 8 * q : (FMT == FMT_NVFP4 ? 2 * q : 4 * q);
    const uint8_t *a0 = buf + r0 * G::RS + b * G::UCB + lane_off;
    const uint8_t *a1 = buf + r1 * G::RS + b * G::UCB + lane_off;
    const uint8_t *s0 = buf + G::CODE_BYTES + r0 * G::SB + b * G::SPU;
    const uint8_t *s1 = buf + G::CODE_BYTES + r1 * G::SB + b * G::SPU;
    const uint16_t *xp = xrow >= 0 ? xs + (size_t)xrow * ks + 8 * q + (size_t)(u0 + b - xu0) * 32 : nullptr;
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

// A warp's stream of units through its ring: copies run S-1 stages ahead
// of the decode.  prime() issues the first copies (it may run before the
// activations are staged: the weights do not depend on them); run()
// decodes every stage and refills the ring as it goes.
// next(i) -> SUnit for the warp's unit i.
template <int FMT, int MC, class Next>
struct Streamer {
    using G = SGeo<FMT, MC>;
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
        slot_issue = slot_issue + 1 == G::STAGES ? 0 : slot_issue + 1;
    }

    // Issue `n` of the STAGES - 1 stages in flight when the stream starts
    // (n over all calls before run() adds up to STAGES - 1).
    __device__ __forceinline__ void prime(int n = G::STAGES - 1)
    {
#pragma unroll
        for (int s = 0; s < G::STAGES - 1; ++s)
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
                cp_async_wait<G::STAGES - 2>();
                __syncwarp();
                issue();  // refills the slot consumed one stage ago
                compute_stage<FMT, MC, FOLD>(cd, cs, ring + slot * G::STAGE_BYTES, xs, ks, xu0, xrow, acc, f);
                slot = slot + 1 == G::STAGES ? 0 : slot + 1;
            }
            done(cu, acc);
        }
        cp_async_wait<0>();
        __syncwarp();
    }
};

// ------------------------------------------------------------------ dense

struct QmvSArgs {
    const uint8_t *codes;
    const uint8_t *scales;
    const uint16_t *x;  // bf16 [M][K]
    float *y;           // [M][N]
    float *ws;          // window partials [nwin][mc][N]
    int *ws_count;      // [G]
    int N, K;
    int m0, mc;
    int tiles;     // ceil(N / RT)
    int G;         // CTAs per window
    int nwin;      // K windows
    int WU;        // units per window (multiple of UPS)
    int pmax;      // partial-sum slots per tile (pieces a tile's K may be cut into)
    int split;     // 0: whole tiles per warp; 1, 2: equal runs of stages per warp,
                   // a piece's slot 1: (warp - the tile's first warp), 2: its stage offset
    int ntl_max;   // tiles per CTA (upper bound)
    int ks;        // staged row stride (f16 elements)
};

template <int FMT, int MC>
__global__ void __launch_bounds__(QMV_THREADS, 1) qmv_stream_kernel(QmvSArgs a)
{
    using G = SGeo<FMT, MC>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    size_t off = (size_t)MC * a.ks * 2;
    int *sh = reinterpret_cast<int *>(smem + off);
    unsigned *maxbits = reinterpret_cast<unsigned *>(sh + 8);
    int *flag = reinterpret_cast<int *>(maxbits + 8);
    off += 80;
    float *red = reinterpret_cast<float *>(smem + off);
    off += (((size_t)a.ntl_max * a.pmax * G::RT * MC * 4) + 15) & ~(size_t)15;
    uint8_t *rings = smem + off;

    const int gb = blockIdx.x % a.G, win = blockIdx.x / a.G;
    const int U = (a.K + 31) / 32;
    const int xu0 = win * a.WU, xu1 = min(U, xu0 + a.WU);
    const int len = min(a.K - xu0 * 32, (xu1 - xu0) * 32);

    const int warp = threadIdx.x >> 5;
    const int ntl = gb < a.tiles ? (a.tiles - gb + a.G - 1) / a.G : 0;
    // The CTA's work is its tiles' stages in tile-major order (S of them).
    // Whole tiles go round-robin to the warps when that balances them (many
    // tiles); otherwise each warp takes an equal contiguous run, so the warps
    // finish together and a tile's K is cut only where runs meet (cutting
    // rows finer measured slower).  A piece's partial sums go to a slot of
    // its tile; the slots are added in K order.
    const int spw = (xu1 - xu0 + G::UPS - 1) / G::UPS;  // stages per row in this window
    const long long S = (long long)ntl * spw;
    long long lo_w = 0, hi_w = 0;
    int t_first = 0, n_my = 0;
    if (a.split) {
        lo_w = S * warp / QMV_WARPS;
        hi_w = S * (warp + 1) / QMV_WARPS;
        if (hi_w > lo_w) {
            t_first = (int)(lo_w / spw);
            n_my = (int)((hi_w - 1) / spw) - t_first + 1;
        }
    } else {
        t_first = warp;
        n_my = warp < ntl ? (ntl - warp + QMV_WARPS - 1) / QMV_WARPS : 0;
    }
    const int RB = FMT == FMT_MXFP8 ? a.K : a.K / 2;
    const int KS = FMT == FMT_NVFP4 ? a.K / 16 : a.K / 32;
    const int tok = lane_token<MC>();
    const int xrow = tok < a.mc ? tok : -1;

    // unit i of this warp: tile t, stages [lo, hi) of the CTA's sequence
    auto unit_tile = [&](int i) { return a.split ? t_first + i : warp + QMV_WARPS * i; };
    auto next = [&](int i) {
        const int t = unit_tile(i);
        SUnit u;
        u.codes = a.codes;
        u.scales = a.scales;
        u.row0 = (gb + t * a.G) * G::RT;
        if (a.split) {
            const long long t0 = (long long)t * spw;
            const long long lo = lo_w > t0 ? lo_w : t0, hi = hi_w < t0 + spw ? hi_w : t0 + spw;
            u.ub = xu0 + (int)(lo - t0) * G::UPS;
            u.ul = min(xu1, xu0 + (int)(hi - t0) * G::UPS);
        } else {
            u.ub = xu0;
            u.ul = xu1;
        }
        u.jump = MC;
        u.lim = a.N;
        return u;
    };
    auto slot_of = [&](int i) {
        if (!a.split) return 0;
        const long long t0 = (long long)unit_tile(i) * spw;
        if (lo_w <= t0) return 0;
        if (a.split == 2) return (int)(lo_w - t0);
        // the warp whose run holds the tile's first stage
        const int wf = (int)((QMV_WARPS * (t0 + 1) + S - 1) / S) - 1;
        return warp - wf;
    };
    auto xrow_of = [&](int) { return xrow; };
    auto done = [&](int i, const float (&acc)[2][2]) {
        const size_t v = (size_t)unit_tile(i) * a.pmax + slot_of(i);
        float vv[2][2];
        qmv_warp_reduce<MC>(acc, vv);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                int r, t;
                if (tile_out<MC>(h, c, r, t)) red[(v * G::RT + r) * MC + t] = vv[h][c];
            }
    };
    pdl_trigger();
    uint8_t *ring = rings + (size_t)warp * G::STAGES * G::STAGE_BYTES;
    Streamer<FMT, MC, decltype(next)> st(next, n_my, ring, a.N, RB, KS);
    // One stage of weight copies overlaps the previous kernel's tail; the
    // rest is issued once the activation loads are in flight (behind a
    // ring's worth of weight copies the activations take microseconds
    // longer to arrive).
    st.prime(1);
    pdl_wait();
    stage_x<FMT>(a.x + (size_t)a.m0 * a.K + (size_t)xu0 * 32, (size_t)a.K, len, a.mc, nullptr, xs, a.ks, sh,
                 maxbits, [&]() { st.prime(G::STAGES - 2); });
    for (int i = threadIdx.x; i < ntl * a.pmax * G::RT * MC; i += blockDim.x) red[i] = 0.f;  // unused slots add 0
    __syncthreads();
    // fold factors of the lane's accumulator columns (the same in every
    // unit); the fold is on when a token was staged scaled up, a decision
    // every CTA takes alike
    float fcol[2];
    bool fold = false;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int t = acc_token<MC>(c);
        fcol[c] = t < a.mc ? pow2f(sh_fold<FMT>(sh[t])) : 1.0f;
    }
    for (int t = 0; t < a.mc; ++t) fold |= sh_fold<FMT>(sh[t]) < 0;
    auto fold_of = [&](int, float (&f)[2]) {
        f[0] = fcol[0];
        f[1] = fcol[1];
    };
    if (fold)
        st.template run<true>(xrow_of, done, fold_of, ring, xs, a.ks, xu0);
    else
        st.template run<false>(xrow_of, done, fold_of, ring, xs, a.ks, xu0);
    __syncthreads();

    float g = 1.0f;
    if (FMT == FMT_NVFP4) g = load_f32_unaligned(a.scales + (size_t)a.N * (a.K / 16));
    const int total = ntl * G::RT * a.mc;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int ti = idx / (G::RT * a.mc), rt = idx - ti * G::RT * a.mc;
        const int r = rt / a.mc, t = rt - r * a.mc;
        const int row = (gb + ti * a.G) * G::RT + r;
        if (row >= a.N) continue;
        float s = 0.f;
        for (int c = 0; c < a.pmax; ++c) s += red[((size_t)(ti * a.pmax + c) * G::RT + r) * MC + t];
        s *= pow2f(sh_final<FMT>(sh[t]));
        if (a.nwin == 1) {
            if (FMT == FMT_NVFP4) s *= g;
            a.y[(size_t)(a.m0 + t) * a.N + row] = s;
        } else {
            a.ws[((size_t)win * a.mc + t) * a.N + row] = s;
        }
    }
    if (a.nwin == 1) return;
    // split-K over windows: the last CTA of this tile group adds the windows
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *flag = atomicAdd(&a.ws_count[gb], 1) == a.nwin - 1;
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int ti = idx / (G::RT * a.mc), rt = idx - ti * G::RT * a.mc;
        const int r = rt / a.mc, t = rt - r * a.mc;
        const int row = (gb + ti * a.G) * G::RT + r;
        if (row >= a.N) continue;
        float s = 0.f;
        for (int w = 0; w < a.nwin; ++w) s += __ldcg(&a.ws[((size_t)w * a.mc + t) * a.N + row]);
        if (FMT == FMT_NVFP4) s *= g;
        a.y[(size_t)(a.m0 + t) * a.N + row] = s;
    }
    if (threadIdx.x == 0) atomicExch(&a.ws_count[gb], 0);
}

template <int FMT, int MC>
static cudaError_t run_qmv_stream(const DeviceState &ds, cudaStream_t st, QmvSArgs a, size_t smem)
{
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(qmv_stream_kernel<FMT, MC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, ds.max_smem_optin);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    return launch_k(qmv_stream_kernel<FMT, MC>, dim3(a.G * a.nwin), dim3(QMV_THREADS), smem, st, a);
}

// Plan and launch one token chunk; returns cudaErrorNotSupported when the
// streaming kernel cannot take this shape (the caller falls back).  With a
// query, nothing is launched: the workspace the launch would use is
// reported instead.
template <int FMT, int MC>
static cudaError_t plan_qmv_stream(const DeviceState &ds, cudaStream_t st, const uint8_t *codes,
                                   const uint8_t *scales, const uint16_t *x, float *y, int m0, int mc, int N, int K,
                                   QmvScratchNeed *query = nullptr)
{
    using G = SGeo<FMT, MC>;
    const int U = K / 32;
    const int rings = QMV_WARPS * G::STAGES * G::STAGE_BYTES;
    const int tiles = (N + G::RT - 1) / G::RT;
    // reduction slots needed at most (one window, 16 chunks per tile)
    const long long red_est =
        std::min<long long>(ST_RED_BUDGET, (long long)((tiles + ds.num_sms - 1) / ds.num_sms) * 16 * G::RT * MC * 4);
    const long long avail = (long long)ds.max_smem_optin - rings - red_est - 128;
    if (avail < 8192) return cudaErrorNotSupported;
    // K windows so that the staged activations fit
    int nwin = 1, WU = 0, ks = 0;
    for (;; ++nwin) {
        WU = (U + nwin - 1) / nwin;
        WU = (WU + G::UPS - 1) / G::UPS * G::UPS;
        ks = WU * 32;
        if ((ks / 32) % 2 == 0) ks += 32;
        if ((long long)MC * ks * 2 <= avail) break;
        if (nwin > 64) return cudaErrorNotSupported;
    }
    nwin = (U + WU - 1) / WU;
    QmvSArgs a;
    a.codes = codes;
    a.scales = scales;
    a.x = x;
    a.y = y;
    a.ws = ds.ws;
    a.ws_count = ds.ws_count;
    a.N = N;
    a.K = K;
    a.m0 = m0;
    a.mc = mc;
    a.tiles = (N + G::RT - 1) / G::RT;
    a.nwin = nwin;
    a.G = nwin == 1 ? ds.num_sms : (ds.num_sms / nwin > 0 ? ds.num_sms / nwin : 1);
    if (a.G > a.tiles) a.G = a.tiles;
    a.WU = WU;
    a.ntl_max = (a.tiles + a.G - 1) / a.G;
    // K windows add their partial sums through the calling stream's workspace:
    // without one attached, or when it is too small, the chunk falls back to
    // the direct-load kernel (which needs none)
    if (nwin > 1 && ((size_t)nwin * mc * N > ds.ws_floats || a.G > ds.ws_counters)) return cudaErrorNotSupported;
    if (nwin > 1 && !query && (ds.ws == nullptr || ds.ws_count == nullptr)) return cudaErrorNotSupported;
    // work split: whole tiles round-robin when the busiest warp has at most
    // 5 % more than the average; else equal runs of stages (a tile cut into
    // at most pmax pieces when every warp's run has a stage, else one slot
    // per stage offset)
    const int spw = (WU + G::UPS - 1) / G::UPS;  // stages per row per window
    const int spw_last = (U - (nwin - 1) * WU + G::UPS - 1) / G::UPS;  // the last window may be shorter
    const int ntl_min = a.tiles / a.G;
    const long long s_min = (long long)ntl_min * std::min(spw, spw_last);
    const long long busiest = (long long)((a.ntl_max + QMV_WARPS - 1) / QMV_WARPS) * QMV_WARPS;
    if (a.ntl_max >= QMV_WARPS && busiest * 100 <= (long long)a.ntl_max * 105) {
        a.split = 0;
        a.pmax = 1;
    } else if (s_min >= QMV_WARPS) {
        a.split = 1;
        const long long q = s_min / QMV_WARPS;  // shortest run (stages)
        a.pmax = (int)std::min<long long>(spw, (spw + q - 1) / q + 1);
    } else {
        a.split = 2;
        a.pmax = spw;
    }
    const long long per = (long long)a.ntl_max * a.pmax * G::RT * MC * 4;
    const long long red_cap = (long long)ds.max_smem_optin - rings - 128 - (long long)MC * ks * 2;
    if (per > red_cap) return cudaErrorNotSupported;
    a.ks = ks;
    const size_t red = (((size_t)a.ntl_max * a.pmax * G::RT * MC * 4) + 15) & ~(size_t)15;
    const size_t smem = (size_t)MC * ks * 2 + 80 + red + rings;
    if (smem > (size_t)ds.max_smem_optin) return cudaErrorNotSupported;
    if (query) {
        query->floats = nwin > 1 ? (size_t)nwin * mc * N : 0;
        query->counters = nwin > 1 ? a.G : 0;
        return cudaSuccess;
    }
    return run_qmv_stream<FMT, MC>(ds, st, a, smem);
}

static int round_mc_s(int m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : 8; }

template <int FMT>
static cudaError_t qmv_stream_chunk(const DeviceState &ds, cudaStream_t st, const uint8_t *codes,
                                    const uint8_t *scales, const uint16_t *x, float *y, int m0, int mc, int N, int K,
                                    QmvScratchNeed *query = nullptr)
{
    switch (round_mc_s(mc)) {
    case 1: return plan_qmv_stream<FMT, 1>(ds, st, codes, scales, x, y, m0, mc, N, K, query);
    case 2: return plan_qmv_stream<FMT, 2>(ds, st, codes, scales, x, y, m0, mc, N, K, query);
    case 4: return plan_qmv_stream<FMT, 4>(ds, st, codes, scales, x, y, m0, mc, N, K, query);
    default: return plan_qmv_stream<FMT, 8>(ds, st, codes, scales, x, y, m0, mc, N, K, query);
    }
}

// Rows must be 128-element aligned for the 16-byte copies of codes and the
// 4-byte copies of scales.
static bool stream_ok(int, int K) { return K % 128 == 0; }

cudaError_t launch_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K)
{
    if (!stream_ok(fmt, K)) return launch_qmv_direct(ds, st, fmt, codes, scales, x, y, M, N, K);
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mc = M - m0 < 8 ? M - m0 : 8;
        cudaError_t e;
        if (fmt == FMT_MXFP4) e = qmv_stream_chunk<FMT_MXFP4>(ds, st, codes, scales, x, y, m0, mc, N, K);
        else if (fmt == FMT_MXFP8) e = qmv_stream_chunk<FMT_MXFP8>(ds, st, codes, scales, x, y, m0, mc, N, K);
        else e = qmv_stream_chunk<FMT_NVFP4>(ds, st, codes, scales, x, y, m0, mc, N, K);
        if (e == cudaErrorNotSupported)
            e = launch_qmv_direct(ds, st, fmt, codes, scales, x + (size_t)m0 * K, y + (size_t)m0 * N, mc, N, K);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

QmvScratchNeed qmv_scratch_need(const DeviceState &ds, int fmt, int M, int N, int K)
{
    QmvScratchNeed need;
    if (!stream_ok(fmt, K)) return need;  // the direct-load kernels use no workspace
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mc = M - m0 < 8 ? M - m0 : 8;
        QmvScratchNeed q;
        cudaError_t e;
        if (fmt == FMT_MXFP4) e = qmv_stream_chunk<FMT_MXFP4>(ds, nullptr, nullptr, nullptr, nullptr, nullptr, m0, mc, N, K, &q);
        else if (fmt == FMT_MXFP8) e = qmv_stream_chunk<FMT_MXFP8>(ds, nullptr, nullptr, nullptr, nullptr, nullptr, m0, mc, N, K, &q);
        else e = qmv_stream_chunk<FMT_NVFP4>(ds, nullptr, nullptr, nullptr, nullptr, nullptr, m0, mc, N, K, &q);
        if (e != cudaSuccess) continue;  // that chunk falls back to the direct-load kernel
        if (q.floats > need.floats) need.floats = q.floats;
        if (q.counters > need.counters) need.counters = q.counters;
    }
    return need;
}

// ------------------------------------------------------------------ MoE

// What the MoE kernel computes from the routed products (see the ABI):
//   MOE_PLAIN          y[slot][n]            (mx_moe_qmv)
//   MOE_GATE_UP_SWIGLU h[slot][i] = swiglu(gate row i, up row I + i)
//   MOE_DOWN_COMBINE   out[t][n] = sum_j r[t][j] * (W_e(t,j) h[t*topk + j])[n]
enum : int { MOE_PLAIN = 0, MOE_GATE_UP_SWIGLU = 1, MOE_DOWN_COMBINE = 2 };

struct MoeSArgs {
    const uint8_t *codes;
    const uint8_t *scales;
    const uint16_t *x;  // bf16 [XR][K]: tokens (plain, gate-up) or slots (down-combine)
    const int32_t *ids;
    float *y;           // plain: [T*topk][N]
    uint16_t *h;        // gate-up: bf16 [T*topk][I]
    const float *rw;    // down-combine: router weights [T][topk]
    float *out;         // down-combine: [T][N]
    float *ws;          // down-combine: per-slot partials [T*topk][N]
    int *ws_count;      // down-combine: per-tile arrival counters
    int *err;
    int T, E, topk, N, K;
    int I;              // gate-up: intermediate size (N = 2 I weight rows per expert)
    int ks;
};

template <int MODE>
__host__ __device__ inline int moe_xrows(int T, int topk)
{
    return MODE == MOE_DOWN_COMBINE ? T * topk : T;
}

template <int FMT, int MC, int MODE>
__global__ void __launch_bounds__(QMV_THREADS, 1) moe_stream_kernel(MoeSArgs a)
{
    using G = SGeo<FMT, MC>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int P = a.T * a.topk;
    const int XR = moe_xrows<MODE>(a.T, a.topk);
    int *cnt = reinterpret_cast<int *>(smem);
    int *wgs = cnt + a.E;
    int *pos = wgs + a.E;
    int *sorted = pos + a.E;
    int *wg_e = sorted + P;
    int *wg_first = wg_e + P;
    int *wg_mc = wg_first + P;
    int *tmp = wg_mc + P;
    int *sh = tmp + 40;
    unsigned *maxbits = reinterpret_cast<unsigned *>(sh + XR);
    size_t off = (((size_t)(3 * a.E + 4 * P + 40 + 2 * XR) * 4) + 15) & ~(size_t)15;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + off);
    off += (size_t)XR * a.ks * 2;
    uint8_t *rings = smem + off;

    // The routing and the routed experts' weights do not depend on the
    // previous kernel (no kernel of this library writes expert ids; the
    // caller's ids are complete when the call is issued): the grouping and
    // the first weight copies overlap its tail.  Activations and outputs wait.
    pdl_trigger();
    RouteSmem rs{cnt, wgs, pos, sorted, wg_e, wg_first, wg_mc, tmp};
    const int nwg = moe_route(a.ids, P, a.E, MC, rs);
    if (MODE == MOE_DOWN_COMBINE && nwg == 0) {
        // no valid slot at all: every token's sum has a NaN term
        pdl_wait();
        if (blockIdx.x == 0 && threadIdx.x == 0) set_device_error(a.err, DEVERR_BAD_EXPERT);
        for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)a.T * a.N;
             i += (size_t)gridDim.x * blockDim.x)
            a.out[i] = __int_as_float(0x7FC00000);
        return;
    }

    // weight rows per expert, and tiles of rows per work group
    const int R = MODE == MOE_GATE_UP_SWIGLU ? 2 * a.I : a.N;
    const int tiles = MODE == MOE_GATE_UP_SWIGLU ? (a.I + MC - 1) / MC : (a.N + G::RT - 1) / G::RT;
    const int items = nwg * tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * QMV_WARPS + warp, stride = gridDim.x * QMV_WARPS;
    const int n_my = gw < items ? (items - gw + stride - 1) / stride : 0;
    const int RB = FMT == FMT_MXFP8 ? a.K : a.K / 2;
    const int KS = FMT == FMT_NVFP4 ? a.K / 16 : a.K / 32;
    const int U = (a.K + 31) / 32;
    const int tok = lane_token<MC>();

    auto next = [&](int i) {
        const int item = gw + stride * i;
        const int w = item / tiles, tile = item - w * tiles;
        const int e = wg_e[w];
        SUnit u;
        u.codes = a.codes + (size_t)e * R * RB;
        u.scales = a.scales + (size_t)e * R * KS;
        u.ub = 0;
        u.ul = U;
        if (MODE == MOE_GATE_UP_SWIGLU) {
            u.row0 = tile * MC;
            u.jump = a.I;
            u.lim = a.I;
        } else {
            u.row0 = tile * G::RT;
            u.jump = MC;
            u.lim = a.N;
        }
        return u;
    };
    // staged activation row of a work-group member
    auto xrow_of_slot = [&](int slot) { return MODE == MOE_DOWN_COMBINE ? slot : slot / a.topk; };
    auto xrow_of = [&](int i) {
        const int w = (gw + stride * i) / tiles;
        return tok < wg_mc[w] ? xrow_of_slot(sorted[wg_first[w] + tok]) : -1;
    };
    auto done = [&](int i, const float (&acc)[2][2]) {
        const int item = gw + stride * i;
        const int w = item / tiles, tile = item - w * tiles;
        float vv[2][2];
        qmv_warp_reduce<MC>(acc, vv);
        float g = 1.0f;
        if (FMT == FMT_NVFP4)
            g = load_f32_unaligned(a.scales + (size_t)a.E * R * KS + 4 * (size_t)wg_e[w]);
        if constexpr (MODE == MOE_GATE_UP_SWIGLU) {
            // the lane holding gate row i of a token also holds its up row
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                int r, t;
                if (tile_out<MC>(0, c, r, t)) {
                    const int irow = tile * MC + r;
                    if (irow < a.I && t < wg_mc[w]) {
                        const int slot = sorted[wg_first[w] + t];
                        const float f = pow2f(sh_final<FMT>(sh[slot / a.topk]));
                        float gv = vv[0][c] * f, uv = vv[1][c] * f;
                        if (FMT == FMT_NVFP4) {
                            gv *= g;
                            uv *= g;
                        }
                        a.h[(size_t)slot * a.I + irow] = (uint16_t)swiglu_bf16(gv, uv);
                    }
                }
            }
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    int r, t;
                    if (tile_out<MC>(h, c, r, t)) {
                        const int row = tile * G::RT + r;
                        if (row < a.N && t < wg_mc[w]) {
                            const int slot = sorted[wg_first[w] + t];
                            float s = vv[h][c] * pow2f(sh_final<FMT>(sh[xrow_of_slot(slot)]));
                            if (FMT == FMT_NVFP4) s *= g;
                            if (MODE == MOE_PLAIN) a.y[(size_t)slot * a.N + row] = s;
                            else a.ws[(size_t)slot * a.N + row] = s;
                        }
                    }
                }
        }
    };
    uint8_t *ring = rings + (size_t)warp * G::STAGES * G::STAGE_BYTES;
    Streamer<FMT, MC, decltype(next)> st(next, n_my, ring, R, RB, KS);
    st.prime(1);
    pdl_wait();
    for (int p = blockIdx.x; p < P; p += gridDim.x) {
        const int e = a.ids[p];
        if (e < 0 || e >= a.E) {
            if (threadIdx.x == 0) set_device_error(a.err, DEVERR_BAD_EXPERT);
            if (MODE == MOE_PLAIN)
                for (int n = threadIdx.x; n < a.N; n += blockDim.x) a.y[(size_t)p * a.N + n] = __int_as_float(0x7FC00000);
            if (MODE == MOE_GATE_UP_SWIGLU)
                for (int i = threadIdx.x; i < a.I; i += blockDim.x) a.h[(size_t)p * a.I + i] = 0x7FC0u;
        }
    }
    // the rest of the weight copies are issued once the activation loads are in flight
    stage_x<FMT>(a.x, (size_t)a.K, a.K, XR, nullptr, xs, a.ks, sh, maxbits, [&]() { st.prime(G::STAGES - 2); });
    __syncthreads();
    // fold factors per unit (the members of its work group); the fold is on
    // when a staged row was scaled up, a decision every CTA takes alike
    bool fold = false;
    for (int r = 0; r < XR; ++r) fold |= sh_fold<FMT>(sh[r]) < 0;
    auto fold_of = [&](int i, float (&f)[2]) {
        const int w = (gw + stride * i) / tiles;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int t = acc_token<MC>(c);
            f[c] = t < wg_mc[w] ? pow2f(sh_fold<FMT>(sh[xrow_of_slot(sorted[wg_first[w] + t])])) : 1.0f;
        }
    };
    if (fold)
        st.template run<true>(xrow_of, done, fold_of, ring, xs, a.ks, 0);
    else
        st.template run<false>(xrow_of, done, fold_of, ring, xs, a.ks, 0);

    if constexpr (MODE == MOE_DOWN_COMBINE) {
        // Each tile gets one unit per work group.  The warp that completes a
        // tile's last unit sums the slots' partials in slot order, weighted
        // by the router, and re-arms the tile's counter.
        __threadfence();
        __syncwarp();
        for (int i = 0; i < n_my; ++i) {
            const int tile = (gw + stride * i) % tiles;
            int last = 0;
            if (lane == 0) last = atomicAdd(&a.ws_count[tile], 1) == nwg - 1;
            if (!__shfl_sync(0xFFFFFFFFu, last, 0)) continue;
            __threadfence();
            for (int idx = lane; idx < G::RT * a.T; idx += 32) {
                const int t = idx / G::RT, row = tile * G::RT + (idx - t * G::RT);
                if (row >= a.N) continue;
                float s = 0.f;
                for (int j = 0; j < a.topk; ++j) {
                    const int p = t * a.topk + j;
                    const int e = a.ids[p];
                    const float v = (e >= 0 && e < a.E) ? __ldcg(&a.ws[(size_t)p * a.N + row]) : __int_as_float(0x7FC00000);
                    s = fmaf(a.rw[p], v, s);
                }
                a.out[(size_t)t * a.N + row] = s;
            }
            if (lane == 0) a.ws_count[tile] = 0;
        }
    }
}

template <int FMT, int MC, int MODE>
static cudaError_t run_moe_stream(const DeviceState &ds, cudaStream_t st, const MoeSArgs &a)
{
    using G = SGeo<FMT, MC>;
    const int P = a.T * a.topk;
    const int XR = moe_xrows<MODE>(a.T, a.topk);
    const size_t head = (((size_t)(3 * a.E + 4 * P + 40 + 2 * XR) * 4) + 15) & ~(size_t)15;
    const size_t smem = head + (size_t)XR * a.ks * 2 + (size_t)QMV_WARPS * G::STAGES * G::STAGE_BYTES;
    if (smem > (size_t)ds.max_smem_optin) return cudaErrorNotSupported;
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(moe_stream_kernel<FMT, MC, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, ds.max_smem_optin);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    return launch_k(moe_stream_kernel<FMT, MC, MODE>, dim3(ds.num_sms), dim3(QMV_THREADS), smem, st, a);
}

template <int FMT, int MODE>
static cudaError_t moe_stream_dispatch(const DeviceState &ds, cudaStream_t st, const MoeSArgs &a, int MC)
{
    switch (MC) {
    case 1: return run_moe_stream<FMT, 1, MODE>(ds, st, a);
    case 2: return run_moe_stream<FMT, 2, MODE>(ds, st, a);
    case 4: return run_moe_stream<FMT, 4, MODE>(ds, st, a);
    default: return run_moe_stream<FMT, 8, MODE>(ds, st, a);
    }
}

template <int MODE>
static cudaError_t moe_stream_fmt(const DeviceState &ds, cudaStream_t st, int fmt, const MoeSArgs &a, int MC)
{
    if (fmt == FMT_MXFP4) return moe_stream_dispatch<FMT_MXFP4, MODE>(ds, st, a, MC);
    if (fmt == FMT_MXFP8) return moe_stream_dispatch<FMT_MXFP8, MODE>(ds, st, a, MC);
    return moe_stream_dispatch<FMT_NVFP4, MODE>(ds, st, a, MC);
}

static MoeSArgs moe_args(const DeviceState &ds, const uint8_t *codes, const uint8_t *scales, const uint16_t *x,
                         const int32_t *ids, int T, int E, int topk, int N, int K)
{
    MoeSArgs a = {};
    a.codes = codes;
    a.scales = scales;
    a.x = x;
    a.ids = ids;
    a.err = ds.err;
    a.T = T;
    a.E = E;
    a.topk = topk;
    a.N = N;
    a.K = K;
    a.ks = stage_stride(K);
    return a;
}

// A work group holds the slots of one expert, at most one per token when
// each token's experts are distinct, so the pass width follows the tokens;
// but at least 4: for the short rows of MoE experts (K of a few thousand)
// the 8-row stages of width 4 keep more bytes in flight per warp than the
// 2-row stages of width 1, which outweighs the unused MMA columns
// (measured on GB300, 128 experts, K = 2048 and 768: 10.0 against 11.0 us
// for gate-up, 9.8 against 16.8 us for the fused down projection at T = 1).
static int moe_mc(int T) { return T <= 4 ? 4 : 8; }

// The fused down projection's groups hold up to one slot per token as well;
// from three tokens on, the 16-row stages of width 8 measure faster.
static int moe_mc_down(int T) { return T <= 2 ? 4 : 8; }

cudaError_t launch_moe_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, const uint16_t *x, const int32_t *ids, float *y, int T, int E,
                           int topk, int N, int K)
{
    if (stream_ok(fmt, K)) {
        MoeSArgs a = moe_args(ds, codes, scales, x, ids, T, E, topk, N, K);
        a.y = y;
        const cudaError_t e = moe_stream_fmt<MOE_PLAIN>(ds, st, fmt, a, moe_mc(T));
        if (e != cudaErrorNotSupported) return e;
    }
    return launch_moe_qmv_direct(ds, st, fmt, codes, scales, x, ids, y, T, E, topk, N, K);
}

cudaError_t launch_moe_gate_up_swiglu(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                                      const uint8_t *scales, const uint16_t *x, const int32_t *ids, uint16_t *h,
                                      int T, int E, int topk, int I, int K)
{
    if (!stream_ok(fmt, K)) {
        // rows not 128-element aligned: the direct-load MoE kernel writes the
        // gate and up products to the workspace, then the SwiGLU glue (the
        // same silu and rounding) forms h
        if ((size_t)T * topk * 2 * I > ds.ws_floats || ds.ws == nullptr) return cudaErrorInvalidValue;
        cudaError_t e = launch_moe_qmv_direct(ds, st, fmt, codes, scales, x, ids, ds.ws, T, E, topk, 2 * I, K);
        if (e != cudaSuccess) return e;
        return launch_swiglu(ds, st, ds.ws, h, T * topk, I);
    }
    MoeSArgs a = moe_args(ds, codes, scales, x, ids, T, E, topk, 2 * I, K);
    a.h = h;
    a.I = I;
    const cudaError_t e = moe_stream_fmt<MOE_GATE_UP_SWIGLU>(ds, st, fmt, a, moe_mc(T));
    return e == cudaErrorNotSupported ? cudaErrorInvalidValue : e;
}

cudaError_t launch_moe_down_combine(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                                    const uint8_t *scales, const uint16_t *h, const int32_t *ids, const float *rw,
                                    float *out, int T, int E, int topk, int N, int K)
{
    if (!stream_ok(fmt, K)) {
        // rows not 128-element aligned: per-slot down products from the
        // direct-load MoE kernel through the workspace, then the router
        // combine (fused multiply-adds in slot order, as the fused kernel)
        if ((size_t)T * topk * N > ds.ws_floats || ds.ws == nullptr) return cudaErrorInvalidValue;
        cudaError_t e = launch_moe_qmv_direct(ds, st, fmt, codes, scales, h, ids, ds.ws, T * topk, E, 1, N, K);
        if (e != cudaSuccess) return e;
        return launch_moe_combine(ds, st, ds.ws, rw, out, T, topk, N);
    }
    const int MC = moe_mc_down(T);
    const int RT = 2 * MC;
    if ((size_t)T * topk * N > ds.ws_floats || (N + RT - 1) / RT > ds.ws_counters || ds.ws == nullptr)
        return cudaErrorInvalidValue;
    MoeSArgs a = moe_args(ds, codes, scales, h, ids, T, E, topk, N, K);
    a.rw = rw;
    a.out = out;
    a.ws = ds.ws;
    a.ws_count = ds.ws_count;
    const cudaError_t e = moe_stream_fmt<MOE_DOWN_COMBINE>(ds, st, fmt, a, MC);
    return e == cudaErrorNotSupported ? cudaErrorInvalidValue : e;
}

}  // namespace mx
