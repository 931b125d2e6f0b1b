// mx_qmv.cu -- decode GEMV and MoE decode GEMV, direct-load variant: each
// lane loads its own 4-byte fragment slices straight from global memory.
// It serves every legal shape; the streaming variant (mx_qmv_stream.cu)
// takes the shapes whose rows are 128-element aligned.
#include "mx_qmv_core.cuh"

namespace mx {

int qmv_stage_bytes(int rows, int K)
{
    long long b = (long long)rows * stage_stride(K) * 2;
    return b > (1 << 30) ? -1 : (int)b;
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

    pdl_trigger();
    pdl_wait();
    stage_x<FMT>(a.x + (size_t)a.m0 * a.K, (size_t)a.K, a.K, a.mc, nullptr, xs, a.ks, sh, maxbits);
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
    // fold factors of the lane's accumulator columns; the fold is on when a
    // token was staged scaled up (the same decision in every CTA)
    float f[2];
    bool fold = false;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int t = acc_token<MC>(c);
        f[c] = t < a.mc ? pow2f(sh_fold<FMT>(sh[t])) : 1.0f;
    }
    for (int t = 0; t < a.mc; ++t) fold |= sh_fold<FMT>(sh[t]) < 0;

    for (int base = blockIdx.x * WR; base < a.tiles; base += gridDim.x * WR) {
        const int tile = base + wr;
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (tile < a.tiles) {
            if (fold)
                qmv_tile<FMT, MC, dense_uf<FMT>(), true>(a.codes, a.scales, a.N, a.K, tile * RT, it0, it1, xs,
                                                          a.ks, xrow, acc, f);
            else
                qmv_tile<FMT, MC, dense_uf<FMT>()>(a.codes, a.scales, a.N, a.K, tile * RT, it0, it1, xs,
                                                    a.ks, xrow, acc);
        }
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
                s *= pow2f(sh_final<FMT>(sh[t]));
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
    return launch_k(qmv_kernel<FMT, MC>, dim3(grid), dim3(QMV_THREADS), smem, st, a);
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

// shared memory of a pass of mc tokens: staged rows and the warps' partials
static size_t qmv_direct_bytes(int K, int mc)
{
    return (size_t)mc * stage_stride(K) * 2 + QMV_WARPS * 2 * mc * mc * 4 + 64;
}

bool qmv_direct_fits(const DeviceState &ds, int K) { return qmv_direct_bytes(K, 1) <= (size_t)ds.max_smem_optin; }

cudaError_t launch_qmv_direct(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K)
{
    const int ks = stage_stride(K);
    // tokens per pass: up to 8, bounded by shared memory
    int cap = 8;
    while (cap > 1 && qmv_direct_bytes(K, cap) > (size_t)ds.max_smem_optin) cap >>= 1;
    if (!qmv_direct_fits(ds, K)) return cudaErrorInvalidValue;
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
    float f[2];
    bool fold = false;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int t = acc_token<MC>(c);
        f[c] = t < mc ? pow2f(sh_fold<FMT>(sh[mem[t] / a.topk])) : 1.0f;
        fold |= f[c] != 1.0f;
    }
    if (__any_sync(0xFFFFFFFFu, fold))
        qmv_tile<FMT, MC, MOE_UF, true>(ec, es, a.N, a.K, tile * RT, 0, iters, xs, a.ks, xrow, acc, f);
    else
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
                    float s = v[h][c] * pow2f(sh_final<FMT>(sh[slot / a.topk]));
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

    pdl_trigger();
    pdl_wait();
    RouteSmem rs{cnt, wgs, pos, sorted, wg_e, wg_first, wg_mc, tmp};
    const int nwg = moe_route(a.ids, P, a.E, 8, rs);
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
    stage_x<FMT>(a.x, (size_t)a.K, a.K, a.T, nullptr, xs, a.ks, sh, maxbits);
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
    return launch_k(moe_qmv_kernel<FMT>, dim3(ds.num_sms), dim3(QMV_THREADS), smem, st, a);
}

cudaError_t launch_moe_qmv_direct(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
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
