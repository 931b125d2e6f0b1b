// mx_moe_stream.cu -- MoE decode GEMV (plain, fused gate-up + SwiGLU, fused
// down + router combine), streaming variant (the weight stream of
// mx_stream.cuh).  Units are (work group of up to MC slots routed to one
// expert, tile) over the whole K of that expert.
#include "mx_stream.cuh"

namespace mx {

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
    int lc;             // down-combine: partials summed in shared memory (1) or through ws (0)
    int ntile_max;      // down-combine, lc: row tiles per CTA at most
};

template <int MODE>
__host__ __device__ inline int moe_xrows(int T, int topk)
{
    return MODE == MOE_DOWN_COMBINE ? T * topk : T;
}

// S: ring depth of each warp (stages).
template <int FMT, int MC, int MODE, int S>
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
    // the whole ring's weight copies overlap its tail.  Activations and
    // outputs wait (their L2 prefetch is issued first).
    pdl_trigger();
    prefetch_l2(a.x, (size_t)XR * a.K * 2);  // the activation rows, ahead of the weight stream
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
    // Work items (work group w, row tile): dealt over every warp of the grid;
    // or, with the CTA-local combine of the down projection, every group of
    // this CTA's tiles (blockIdx.x, + gridDim.x, ...) over this CTA's warps,
    // so that a tile's partial sums meet in shared memory.
    const bool lc = MODE == MOE_DOWN_COMBINE && a.lc;
    const int ntile_c = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int n_local = ntile_c * nwg;
    const int n_my = lc ? (warp < n_local ? (n_local - warp + QMV_WARPS - 1) / QMV_WARPS : 0)
                        : (gw < items ? (items - gw + stride - 1) / stride : 0);
    auto item_at = [&](int i, int &w, int &tile, int &ti) {
        if (lc) {
            const int j = warp + QMV_WARPS * i;
            ti = j / nwg;
            w = j - ti * nwg;
            tile = (int)blockIdx.x + ti * (int)gridDim.x;
        } else {
            const int item = gw + stride * i;
            w = item / tiles;
            tile = item - w * tiles;
            ti = 0;
        }
    };
    const int RB = FMT == FMT_MXFP8 ? a.K : a.K / 2;
    const int KS = FMT == FMT_NVFP4 ? a.K / 16 : a.K / 32;
    const int U = (a.K + 31) / 32;
    const int tok = lane_token<MC>();

    auto next = [&](int i) {
        int w, tile, ti;
        item_at(i, w, tile, ti);
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
        int w, tile, ti;
        item_at(i, w, tile, ti);
        return tok < wg_mc[w] ? xrow_of_slot(sorted[wg_first[w] + tok]) : -1;
    };
    float *part = reinterpret_cast<float *>(rings + (size_t)QMV_WARPS * S * G::STAGE_BYTES);  // lc: [ntile][P][RT]
    auto done = [&](int i, const float (&acc)[2][2]) {
        int w, tile, ti;
        item_at(i, w, tile, ti);
        float g = 1.0f;
        if (FMT == FMT_NVFP4)
            g = load_f32_unaligned(a.scales + (size_t)a.E * R * KS + 4 * (size_t)wg_e[w]);
        if constexpr (G::PAIR) {
            // every lane holds tile row r for token t (MC = 4: no lanes to add)
            static_assert(MC == 4, "paired MoE tiles of 4 slots");
            float v;
            int r, t;
            pair_reduce<MC>(acc, v, r, t);
            if constexpr (MODE == MOE_GATE_UP_SWIGLU) {
                // gate row i (tile row r < MC) is paired with up row I + i
                // (tile row MC + r), two lane groups further
                const float up = __shfl_down_sync(0xFFFFFFFFu, v, 16);
                const int irow = tile * MC + r;
                if (r < MC && irow < a.I && t < wg_mc[w]) {
                    const int slot = sorted[wg_first[w] + t];
                    const float fs = pow2f(sh_final<FMT>(sh[slot / a.topk]));
                    float gv = v * fs, uv = up * fs;
                    if (FMT == FMT_NVFP4) {
                        gv *= g;
                        uv *= g;
                    }
                    a.h[(size_t)slot * a.I + irow] = (uint16_t)swiglu_bf16(gv, uv);
                }
            } else {
                const int row = tile * G::RT + r;
                if (row < a.N && t < wg_mc[w]) {
                    const int slot = sorted[wg_first[w] + t];
                    float sv = v * pow2f(sh_final<FMT>(sh[xrow_of_slot(slot)]));
                    if (FMT == FMT_NVFP4) sv *= g;
                    if (MODE == MOE_PLAIN) a.y[(size_t)slot * a.N + row] = sv;
                    else if (lc) part[((size_t)ti * P + slot) * G::RT + r] = sv;
                    else a.ws[(size_t)slot * a.N + row] = sv;
                }
            }
            return;
        }
        float vv[2][2];
        qmv_warp_reduce<MC>(acc, vv);
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
                            else if (lc) part[((size_t)ti * P + slot) * G::RT + r] = s;
                            else a.ws[(size_t)slot * a.N + row] = s;
                        }
                    }
                }
        }
    };
    uint8_t *ring = rings + (size_t)warp * S * G::STAGE_BYTES;
    Streamer<FMT, MC, decltype(next), S> st(next, n_my, ring, R, RB, KS);
    st.prime(S - 1);
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
    stage_x<FMT>(a.x, (size_t)a.K, a.K, XR, nullptr, xs, a.ks, sh, maxbits);
    __syncthreads();
    // fold factors per unit (the members of its work group); the fold is on
    // when a staged row was scaled up, a decision every CTA takes alike
    bool fold = false;
    for (int r = 0; r < XR; ++r) fold |= sh_fold<FMT>(sh[r]) < 0;
    auto fold_of = [&](int i, float (&f)[2]) {
        int w, tile, ti;
        item_at(i, w, tile, ti);
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

    if (MODE == MOE_DOWN_COMBINE && lc) {
        // The CTA's tiles: each slot's partials sit in shared memory; sum them
        // in slot order, weighted by the router (a slot routed nowhere is NaN).
        __syncthreads();
        for (int idx = threadIdx.x; idx < ntile_c * a.T * G::RT; idx += blockDim.x) {
            const int ti = idx / (a.T * G::RT), rem = idx - ti * (a.T * G::RT);
            const int t = rem / G::RT, r = rem - t * G::RT;
            const int row = ((int)blockIdx.x + ti * (int)gridDim.x) * G::RT + r;
            if (row >= a.N) continue;
            float s = 0.f;
            for (int j = 0; j < a.topk; ++j) {
                const int p = t * a.topk + j;
                const int e = a.ids[p];
                const float v = (e >= 0 && e < a.E) ? part[((size_t)ti * P + p) * G::RT + r] : __int_as_float(0x7FC00000);
                s = fmaf(a.rw[p], v, s);
            }
            a.out[(size_t)t * a.N + row] = s;
        }
    } else if constexpr (MODE == MOE_DOWN_COMBINE) {
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

template <int FMT, int MC, int MODE, int S>
static cudaError_t launch_moe_stream(const DeviceState &ds, cudaStream_t st, const MoeSArgs &a, size_t smem)
{
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(moe_stream_kernel<FMT, MC, MODE, S>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, ds.max_smem_optin);
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    return launch_k(moe_stream_kernel<FMT, MC, MODE, S>, dim3(ds.num_sms), dim3(QMV_THREADS), smem, st, a);
}

// Work groups of 4 slots stream an expert's rows in units of a few stages
// (K of a few thousand): a ring of MOE_DEEP stages holds a whole unit in
// flight when shared memory allows, else the default depth; groups of 8
// slots (16-row stages) take one stage more than the default when it fits
// (4 tokens, down projection: layer 31.6 -> 31.2 us).
constexpr int MOE_DEEP = 5;
constexpr int MOE_DEEP8 = 4;

template <int FMT, int MC, int MODE>
static cudaError_t run_moe_stream(const DeviceState &ds, cudaStream_t st, const MoeSArgs &a0)
{
    using G = SGeo<FMT, MC>;
    MoeSArgs a = a0;
    const int P = a.T * a.topk;
    const int XR = moe_xrows<MODE>(a.T, a.topk);
    const size_t head = (((size_t)(3 * a.E + 4 * P + 40 + 2 * XR) * 4) + 15) & ~(size_t)15;
    const size_t base = head + (size_t)XR * a.ks * 2;
    const size_t lim = (size_t)ds.max_smem_optin;
    // down projection: the CTA-local combine when its partials fit next to the ring
    size_t part = 0;
    if (MODE == MOE_DOWN_COMBINE) {
        const int tiles = (a.N + G::RT - 1) / G::RT;
        a.ntile_max = (tiles + ds.num_sms - 1) / ds.num_sms;
        part = (((size_t)a.ntile_max * P * G::RT * 4) + 15) & ~(size_t)15;
        a.lc = base + (size_t)QMV_WARPS * G::STAGES * G::STAGE_BYTES + part <= lim;
        if (!a.lc) part = 0;
    }
    constexpr int DEEP = MC == 4 ? MOE_DEEP : MOE_DEEP8;
    const size_t deep = base + (size_t)QMV_WARPS * DEEP * G::STAGE_BYTES + part;
    if (deep <= lim) return launch_moe_stream<FMT, MC, MODE, DEEP>(ds, st, a, deep);
    const size_t smem = base + (size_t)QMV_WARPS * G::STAGES * G::STAGE_BYTES + part;
    if (smem > lim) return cudaErrorNotSupported;
    return launch_moe_stream<FMT, MC, MODE, G::STAGES>(ds, st, a, smem);
}

// Work groups of 4 or 8 slots (see moe_mc).
template <int FMT, int MODE>
static cudaError_t moe_stream_dispatch(const DeviceState &ds, cudaStream_t st, const MoeSArgs &a, int MC)
{
    return MC == 4 ? run_moe_stream<FMT, 4, MODE>(ds, st, a) : run_moe_stream<FMT, 8, MODE>(ds, st, a);
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
    if (stream_ok(fmt, K)) {
        MoeSArgs a = moe_args(ds, codes, scales, x, ids, T, E, topk, 2 * I, K);
        a.h = h;
        a.I = I;
        const cudaError_t e = moe_stream_fmt<MOE_GATE_UP_SWIGLU>(ds, st, fmt, a, moe_mc(T));
        if (e != cudaErrorNotSupported) return e;
    }
    // rows not 128-element aligned, or too long to stage beside the ring: the
    // direct-load MoE kernel writes the gate and up products to the
    // workspace, then the SwiGLU glue (the same silu and rounding) forms h
    if ((size_t)T * topk * 2 * I > ds.ws_floats || ds.ws == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = launch_moe_qmv_direct(ds, st, fmt, codes, scales, x, ids, ds.ws, T, E, topk, 2 * I, K);
    if (e != cudaSuccess) return e;
    return launch_swiglu(ds, st, ds.ws, h, T * topk, I);
}

cudaError_t launch_moe_down_combine(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                                    const uint8_t *scales, const uint16_t *h, const int32_t *ids, const float *rw,
                                    float *out, int T, int E, int topk, int N, int K)
{
    if ((size_t)T * topk * N > ds.ws_floats || ds.ws == nullptr) return cudaErrorInvalidValue;
    if (stream_ok(fmt, K)) {
        const int MC = moe_mc_down(T);
        const int RT = 2 * MC;
        if ((N + RT - 1) / RT > ds.ws_counters) return cudaErrorInvalidValue;
        MoeSArgs a = moe_args(ds, codes, scales, h, ids, T, E, topk, N, K);
        a.rw = rw;
        a.out = out;
        a.ws = ds.ws;
        a.ws_count = ds.ws_count;
        const cudaError_t e = moe_stream_fmt<MOE_DOWN_COMBINE>(ds, st, fmt, a, MC);
        if (e != cudaErrorNotSupported) return e;
    }
    // rows not 128-element aligned, or too long to stage beside the ring:
    // per-slot down products from the direct-load MoE kernel through the
    // workspace, then the router combine (fused multiply-adds in slot order,
    // as the fused kernel)
    cudaError_t e = launch_moe_qmv_direct(ds, st, fmt, codes, scales, h, ids, ds.ws, T * topk, E, 1, N, K);
    if (e != cudaSuccess) return e;
    return launch_moe_combine(ds, st, ds.ws, rw, out, T, topk, N);
}

}  // namespace mx
