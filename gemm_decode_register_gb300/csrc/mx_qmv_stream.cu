// mx_qmv_stream.cu -- decode GEMV, streaming variant (the weight stream of
// mx_stream.cuh).
//
// A CTA's tiles go to its warps whole and round-robin when that balances
// them; otherwise the CTA's stages (tile-major) are dealt out in equal
// contiguous runs, so a tile's K is cut only where two runs meet, and the
// pieces' partial sums are added in K order in shared memory.  When the
// tokens' activations do not fit in shared memory, K is also split across
// CTAs (windows); the windows' partial sums go to a device workspace and
// the last CTA of a tile group adds them in window order (deterministic).
#include "mx_stream.cuh"

namespace mx {

constexpr int ST_RED_BUDGET = 24 * 1024;
// K windows at most (rows up to 2^20 elements at 8 tokens per pass need ~160)
constexpr int ST_MAX_WINDOWS = 1024;

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
    int G;         // CTAs per window (grid: G x nwin)
    int tq, tr;    // tiles / G, tiles % G
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

    // (The set-up below avoids integer division where it can: at kernel
    // start a division is a long dependent chain on the critical path.)
    const int gb = blockIdx.x, win = blockIdx.y;
    const int U = (a.K + 31) / 32;
    const int xu0 = win * a.WU, xu1 = min(U, xu0 + a.WU);
    const int len = min(a.K - xu0 * 32, (xu1 - xu0) * 32);

    const int warp = threadIdx.x >> 5;
    const int ntl = gb < a.tiles ? a.tq + (gb < a.tr ? 1 : 0) : 0;
    // The CTA's work is its tiles' stages in tile-major order (S of them).
    // Whole tiles go round-robin to the warps when that balances them (many
    // tiles); otherwise each warp takes an equal contiguous run, so the warps
    // finish together and a tile's K is cut only where runs meet (cutting
    // rows finer measured slower).  A piece's partial sums go to a slot of
    // its tile; the slots are added in K order.
    // (32-bit counts: the planner keeps ntl * spw far below 2^27.)
    const int spw = (xu1 - xu0 + G::UPS - 1) / G::UPS;  // stages per row in this window
    const int S = ntl * spw;
    int lo_w = 0, hi_w = 0;
    int t_first = 0, n_my = 0;
    if (a.split) {
        lo_w = S * warp / QMV_WARPS;
        hi_w = S * (warp + 1) / QMV_WARPS;
        if (hi_w > lo_w) {
            t_first = lo_w / spw;
            n_my = (hi_w - 1) / spw - t_first + 1;
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
            const int t0 = t * spw;
            const int lo = lo_w > t0 ? lo_w : t0, hi = hi_w < t0 + spw ? hi_w : t0 + spw;
            u.ub = xu0 + (lo - t0) * G::UPS;
            u.ul = min(xu1, xu0 + (hi - t0) * G::UPS);
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
        const int t0 = unit_tile(i) * spw;
        if (lo_w <= t0) return 0;
        if (a.split == 2) return lo_w - t0;
        // the warp whose run holds the tile's first stage
        const int wf = (QMV_WARPS * (t0 + 1) + S - 1) / S - 1;
        return warp - wf;
    };
    auto xrow_of = [&](int) { return xrow; };
    auto done = [&](int i, const float (&acc)[2][2]) {
        const size_t v = (size_t)unit_tile(i) * a.pmax + slot_of(i);
        if constexpr (G::PAIR) {
            float x;
            int r, t;
            if (pair_reduce<MC>(acc, x, r, t)) red[(v * G::RT + r) * MC + t] = x;
        } else {
            float vv[2][2];
            qmv_warp_reduce<MC>(acc, vv);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    int r, t;
                    if (tile_out<MC>(h, c, r, t)) red[(v * G::RT + r) * MC + t] = vv[h][c];
                }
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
    return launch_k(qmv_stream_kernel<FMT, MC>, dim3(a.G, a.nwin), dim3(QMV_THREADS), smem, st, a);
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
        if (nwin > ST_MAX_WINDOWS) return cudaErrorNotSupported;
    }
    nwin = (U + WU - 1) / WU;
    if (nwin > 1) {
        // Windows are needed anyway: one more of them is worth it when that
        // lets the activation staging keep a thread's chunks in registers (at
        // most 8 chunks of 8 elements per thread: rows padded to a power of
        // two share the 512 threads) and its busiest CTA has no more stages
        // (measured: 4 tokens, K = 28672, 3 -> 4 windows 29.3 -> 27.5 us; 8
        // tokens, 6 -> 7 windows with one stage more, 47.3 -> 50.5 us).
        const int rp = mc <= 1 ? 1 : mc <= 2 ? 2 : mc <= 4 ? 4 : mc <= 8 ? 8 : 16;
        auto in_regs = [&](int wu) { return (long long)wu * rp * 4 <= (long long)QMV_THREADS * STAGE_REG_CHUNKS; };
        auto busiest = [&](int wu) {
            const int nw = (U + wu - 1) / wu;
            const int g = std::max(1, std::min(ds.num_sms / nw, tiles));
            return (long long)((tiles + g - 1) / g) * ((wu + G::UPS - 1) / G::UPS);
        };
        if (!in_regs(WU) && nwin < ST_MAX_WINDOWS) {
            int wu = (U + nwin) / (nwin + 1);
            wu = (wu + G::UPS - 1) / G::UPS * G::UPS;
            if (in_regs(wu) && busiest(wu) <= busiest(WU)) WU = wu;
        }
        ks = WU * 32;
        if ((ks / 32) % 2 == 0) ks += 32;
        nwin = (U + WU - 1) / WU;
    }
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
    // The partial-sum slots of a CTA's tile pieces must fit beside its staged
    // activations: when they do not (few tiles per CTA cut into many pieces
    // over a long window), one more window shrinks the staging and is tried.
    for (int attempt = 0;; ++attempt) {
        a.nwin = nwin;
        a.G = nwin == 1 ? ds.num_sms : (ds.num_sms / nwin > 0 ? ds.num_sms / nwin : 1);
        if (a.G > a.tiles) a.G = a.tiles;
        a.tq = a.tiles / a.G;
        a.tr = a.tiles % a.G;
        a.WU = WU;
        a.ntl_max = (a.tiles + a.G - 1) / a.G;
        // K windows add their partial sums through the calling stream's
        // workspace: without one attached, or when it is too small, the chunk
        // falls back to the direct-load kernel (which needs none)
        if (nwin > 1 && ((size_t)nwin * mc * N > ds.ws_floats || a.G > ds.ws_counters))
            return cudaErrorNotSupported;
        if (nwin > 1 && !query && (ds.ws == nullptr || ds.ws_count == nullptr)) return cudaErrorNotSupported;
        // work split: whole tiles round-robin when the busiest warp has at
        // most 5 % more than the average; else equal runs of stages (a tile
        // cut into at most pmax pieces when every warp's run has a stage, else
        // one slot per stage offset)
        const int spw = (WU + G::UPS - 1) / G::UPS;                     // stages per row per window
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
        if ((long long)a.ntl_max * spw * QMV_WARPS >= (1LL << 27)) return cudaErrorNotSupported;  // 32-bit counts
        const long long per = (long long)a.ntl_max * a.pmax * G::RT * MC * 4;
        const long long red_cap = (long long)ds.max_smem_optin - rings - 128 - (long long)MC * ks * 2;
        if (per <= red_cap) break;
        if (nwin >= ST_MAX_WINDOWS || attempt >= 16) return cudaErrorNotSupported;
        WU = (U + nwin) / (nwin + 1);
        WU = (WU + G::UPS - 1) / G::UPS * G::UPS;
        ks = WU * 32;
        if ((ks / 32) % 2 == 0) ks += 32;
        nwin = (U + WU - 1) / WU;
    }
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

// One group of up to 8 tokens: the streaming kernel, else the direct-load
// kernel (one pass over the weights, no workspace), else - for rows too long
// for the direct kernel's staging, whose K windows' partial sums exceed the
// workspace - the two halves of the group on their own (fewer tokens per
// pass need less workspace).  With a query, nothing is launched and the
// workspace the launches would use is merged into *query.
static cudaError_t qmv_group(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                             const uint8_t *scales, const uint16_t *x, float *y, int m0, int mc, int N, int K,
                             QmvScratchNeed *query)
{
    QmvScratchNeed q;
    QmvScratchNeed *qp = query ? &q : nullptr;
    cudaError_t e;
    if (fmt == FMT_MXFP4) e = qmv_stream_chunk<FMT_MXFP4>(ds, st, codes, scales, x, y, m0, mc, N, K, qp);
    else if (fmt == FMT_MXFP8) e = qmv_stream_chunk<FMT_MXFP8>(ds, st, codes, scales, x, y, m0, mc, N, K, qp);
    else e = qmv_stream_chunk<FMT_NVFP4>(ds, st, codes, scales, x, y, m0, mc, N, K, qp);
    if (e == cudaSuccess && query) {
        if (q.floats > query->floats) query->floats = q.floats;
        if (q.counters > query->counters) query->counters = q.counters;
    }
    if (e != cudaErrorNotSupported) return e;
    if (qmv_direct_fits(ds, K))
        return query ? cudaSuccess
                     : launch_qmv_direct(ds, st, fmt, codes, scales, x + (size_t)m0 * K, y + (size_t)m0 * N, mc, N, K);
    if (mc == 1) return cudaErrorInvalidValue;
    const int h = mc / 2;
    e = qmv_group(ds, st, fmt, codes, scales, x, y, m0, h, N, K, query);
    if (e != cudaSuccess) return e;
    return qmv_group(ds, st, fmt, codes, scales, x, y, m0 + h, mc - h, N, K, query);
}

cudaError_t launch_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K)
{
    if (!stream_ok(fmt, K)) return launch_qmv_direct(ds, st, fmt, codes, scales, x, y, M, N, K);
    for (int m0 = 0; m0 < M; m0 += 8) {
        const cudaError_t e = qmv_group(ds, st, fmt, codes, scales, x, y, m0, M - m0 < 8 ? M - m0 : 8, N, K, nullptr);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

QmvScratchNeed qmv_scratch_need(const DeviceState &ds, int fmt, int M, int N, int K)
{
    QmvScratchNeed need;
    if (!stream_ok(fmt, K)) return need;  // the direct-load kernels use no workspace
    for (int m0 = 0; m0 < M; m0 += 8)
        qmv_group(ds, nullptr, fmt, nullptr, nullptr, nullptr, nullptr, m0, M - m0 < 8 ? M - m0 : 8, N, K, &need);
    return need;
}

}  // namespace mx
