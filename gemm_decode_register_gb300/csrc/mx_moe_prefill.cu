// mx_moe_prefill.cu -- expert-batched MoE prefill: the routed (token, slot)
// rows are grouped by expert on the device, gathered into expert order and
// run through the pair tensor-core GEMM (qmm_kernel, grouped modes) one
// group tile of up to 512 rows at a time (two 256-row accumulators sharing
// each decoded weight tile; a tile of at most 256 rows runs only the first),
// so that each expert's weights are decoded once per 512 routed rows instead
// of once per token.
//
// The pages read only the experts a token is routed to (talk "High-
// performance LLM/VLM inference on AMD Strix Halo with mlxcel engine",
// slide 4) and name MoE prefill as the weak spot once dense prefill moved to
// the matrix units ("MLxcel 0.8 release", section "Bandwidth utilisation per
// model"); grouping by expert is what lets a routed expert's rows share one
// pass over its block-float weights.
//
// Launches (all with programmatic dependent launch; each waits for the one
// before it before touching the workspace).  Up to 256 experts:
//   moe_count_kernel         per chunk of 128 slots: its rows per expert
//   moe_scan_kernel          one block: per expert, the exclusive prefix of
//                            the chunks' counts; exclusive scans over the
//                            experts, the group tile table
//   moe_place_gather_kernel  per chunk: each slot's sorted row (its chunk's
//                            first row of the expert plus a cursor), and the
//                            chunk's X rows copied into expert order
// More experts:
//   moe_group_route_kernel   one block: per-expert counts, exclusive scans,
//                            the group tile table, sorted row -> slot
//   gather_rows_kernel       X rows into expert order (bf16, 16-byte copies)
// Then:
//   qmm_kernel (grouped)     per group tile and column tile; output rows
//                            scattered back to slot order, or (SwiGLU mode)
//                            h in expert order
//   combine_bf16_kernel      (FFN) router-weighted sum over a token's slots
//
// Workspace (caller-owned, 256-byte aligned), in this order:
//   groups   16 + 16 * max_groups bytes: tile count, valid rows, tiles
//   slot_of  4 * S bytes (S = T * topk)
//   blk      (up to 256 experts) 4 * E * (CP + 1) bytes: per expert, the
//            chunks' counts, then their first sorted rows (row stride CP,
//            the chunk count rounded up to 128), and pos[E]
//   xs       2 * S * K bytes: gathered activations (the FFN's down
//            projection writes its per-slot outputs here afterwards)
//   hs       2 * S * I bytes (FFN only): SwiGLU output in expert order
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

constexpr int GROUP_ROWS = 512;  // rows of a group tile (two 256-row pair MMAs sharing the decoded weights)
constexpr int ROUTE_THREADS = 1024;
constexpr int ROUTE_SMALL_E = 256;   // experts the multi-block routing takes
constexpr int ROUTE_CHUNK = 128;     // slots per counting / placing block
constexpr int GATHER_THREADS = 512;   // threads of a placing block (one warp per copied row)

// Chunks of ROUTE_CHUNK slots, and the row stride of their count table.
static int route_chunks(long long S) { return (int)((S + ROUTE_CHUNK - 1) / ROUTE_CHUNK); }
static int route_stride(int C) { return (C + 127) / 128 * 128; }

// Byte offset of the count table (right after slot_of) and its size.
static size_t route_table_offset(size_t off_slot, long long S) { return align256(off_slot + 4 * (size_t)S); }
static size_t route_table_bytes(long long S, int E)
{
    return E <= ROUTE_SMALL_E ? 4 * (size_t)E * (route_stride(route_chunks(S)) + 1) : 0;
}


MoeGroupPlan moe_group_plan(int T, int E, int topk, int K, int I)
{
    MoeGroupPlan p;
    const long long S = (long long)T * topk;
    const long long active = S < E ? S : E;
    // sum over experts of ceil(rows_e / G) <= (S + (G - 1) * active experts) / G
    p.S = (int)S;
    p.max_groups = (int)((S + (long long)(GROUP_ROWS - 1) * active) / GROUP_ROWS);
    p.off_groups = 0;
    p.off_slot = align256(16 + 16 * (size_t)p.max_groups);
    p.off_xs = align256(route_table_offset(p.off_slot, S) + route_table_bytes(S, E));
    p.off_hs = align256(p.off_xs + 2 * (size_t)S * K);
    p.bytes = I > 0 ? align256(p.off_hs + 2 * (size_t)S * I) : p.off_hs;
    return p;
}

// Exclusive scans of the per-expert row counts cnt[] and tile counts
// (ceil(cnt / GROUP_ROWS)) into pos[] and tile0[], the group tile table, and the
// totals in groups[0] (tiles) and groups[1] (rows).  Thread tid owns experts
// [tid * per, tid * per + per).  Ends with the block synchronised.
__device__ void route_scan_tiles(const int *cnt, int *pos, int *tile0, int E, int *groups)
{
    __shared__ int wsum_r[32], wsum_t[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (E + ROUTE_THREADS - 1) / ROUTE_THREADS;
    const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
    int rsum = 0, tsum = 0;
    for (int e = e0; e < e1; ++e) {
        rsum += cnt[e];
        tsum += (cnt[e] + GROUP_ROWS - 1) / GROUP_ROWS;
    }
    int rinc = rsum, tinc = tsum;  // inclusive scans within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int rv = __shfl_up_sync(0xFFFFFFFFu, rinc, o), tv = __shfl_up_sync(0xFFFFFFFFu, tinc, o);
        if (lane >= o) {
            rinc += rv;
            tinc += tv;
        }
    }
    if (lane == 31) {
        wsum_r[warp] = rinc;
        wsum_t[warp] = tinc;
    }
    __syncthreads();
    if (warp == 0) {
        int r = wsum_r[lane], t = wsum_t[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int rv = __shfl_up_sync(0xFFFFFFFFu, r, o), tv = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o) {
                r += rv;
                t += tv;
            }
        }
        wsum_r[lane] = r;  // inclusive over warps
        wsum_t[lane] = t;
    }
    __syncthreads();
    int rpre = rinc - rsum + (warp > 0 ? wsum_r[warp - 1] : 0);
    int tpre = tinc - tsum + (warp > 0 ? wsum_t[warp - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        pos[e] = rpre;
        tile0[e] = tpre;
        rpre += cnt[e];
        tpre += (cnt[e] + GROUP_ROWS - 1) / GROUP_ROWS;
    }
    if (tid == 0) {
        groups[0] = wsum_t[31];  // tiles
        groups[1] = wsum_r[31];  // rows with a valid expert
    }
    __syncthreads();
    int4 *tiles = reinterpret_cast<int4 *>(groups + 4);
    for (int e = tid; e < E; e += ROUTE_THREADS) {
        const int n = cnt[e];
        for (int i = 0; i * GROUP_ROWS < n; ++i)
            tiles[tile0[e] + i] = make_int4(e, pos[e] + i * GROUP_ROWS, min(GROUP_ROWS, n - i * GROUP_ROWS), 0);
    }
    __syncthreads();
}

__device__ __forceinline__ void nan_row(uint16_t *ynan, int s, int w)
{
    uint4 *row = reinterpret_cast<uint4 *>(ynan + (size_t)s * w);
    for (int c = 0; c < w / 8; ++c) row[c] = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
}

// One block, any E <= 4096.  Slots with an expert id outside [0, E) are left
// out of every group; they set DEVERR_BAD_EXPERT and, when ynan is given,
// their output row of ynan_w bf16 values is written as NaN.  An expert's
// rows are placed in no particular order (each output row depends on its
// own X row only, so the order does not change the result).
__global__ void __launch_bounds__(ROUTE_THREADS) moe_group_route_kernel(const int32_t *__restrict__ ids, int S, int E,
                                                                        int *__restrict__ groups,
                                                                        int *__restrict__ slot_of, uint16_t *ynan,
                                                                        int ynan_w, int *err)
{
    extern __shared__ int route_smem[];
    int *cnt = route_smem;            // [E] rows per expert
    int *pos = route_smem + E;        // [E] first sorted row, then the placement cursor
    int *tile0 = route_smem + 2 * E;  // [E] first group tile
    __shared__ int bad;
    const int tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();  // the ids may come from the previous kernel; the tables may still be read by it
    for (int e = tid; e < E; e += ROUTE_THREADS) cnt[e] = 0;
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int s = tid; s < S; s += ROUTE_THREADS) {
        const int e = ids[s];
        if ((unsigned)e < (unsigned)E) {
            atomicAdd(&cnt[e], 1);
        } else {
            bad = 1;
            if (ynan) nan_row(ynan, s, ynan_w);
        }
    }
    __syncthreads();
    route_scan_tiles(cnt, pos, tile0, E, groups);
    for (int s = tid; s < S; s += ROUTE_THREADS) {
        const int e = ids[s];
        if ((unsigned)e < (unsigned)E) slot_of[atomicAdd(&pos[e], 1)] = s;
    }
    if (tid == 0 && bad) set_device_error(err, DEVERR_BAD_EXPERT);
}

// Rows per expert of chunk blockIdx.x (ROUTE_CHUNK slots, one per thread)
// into blk[e][chunk] (row stride CP).  Slots with an expert id outside
// [0, E) count nowhere; they set DEVERR_BAD_EXPERT and, when ynan is given,
// their output row of ynan_w bf16 values is written as NaN.
__global__ void __launch_bounds__(ROUTE_CHUNK) moe_count_kernel(const int32_t *__restrict__ ids, int S, int E, int CP,
                                                                int *__restrict__ blk, uint16_t *ynan, int ynan_w,
                                                                int *err)
{
    __shared__ int hist[ROUTE_SMALL_E];
    const int tid = threadIdx.x, c = blockIdx.x;
    const int s = c * ROUTE_CHUNK + tid;
    pdl_trigger();
    pdl_wait();  // the ids may come from the previous kernel; the count table may still be read by it
    const int e = s < S ? ids[s] : 0;
    for (int i = tid; i < E; i += ROUTE_CHUNK) hist[i] = 0;
    __syncthreads();
    if (s < S) {
        if ((unsigned)e < (unsigned)E) {
            atomicAdd(&hist[e], 1);
        } else {
            set_device_error(err, DEVERR_BAD_EXPERT);
            if (ynan) nan_row(ynan, s, ynan_w);
        }
    }
    __syncthreads();
    for (int i = tid; i < E; i += ROUTE_CHUNK) blk[(size_t)i * CP + c] = hist[i];
}

// Four consecutive entries of a count row, those at chunk C and beyond as 0.
__device__ __forceinline__ int4 load_counts(const int *row, int c0, int C)
{
    int4 v = __ldcg(reinterpret_cast<const int4 *>(row + c0));
    if (c0 + 0 >= C) v.x = 0;
    if (c0 + 1 >= C) v.y = 0;
    if (c0 + 2 >= C) v.z = 0;
    if (c0 + 3 >= C) v.w = 0;
    return v;
}

// One block of ROUTE_THREADS: per expert e, blk[e][c] becomes the number of
// e's rows in chunks before c.  tpe lanes of a warp share an expert's row,
// which they read in rounds of tpe consecutive 16-byte pieces (4 chunks
// each; coalesced), scanning each round across the lanes and carrying its
// total into the next; the experts' totals then give the exclusive scans,
// the group tile table (groups) and pos[e] (the expert's first sorted row)
// in posg.
__global__ void __launch_bounds__(ROUTE_THREADS) moe_scan_kernel(int *__restrict__ blk, int C, int CP, int E,
                                                                 int *__restrict__ groups, int *__restrict__ posg)
{
    __shared__ int cnt[ROUTE_SMALL_E], pos[ROUTE_SMALL_E], tile0[ROUTE_SMALL_E];
    const int tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    int tpe = 32;  // lanes per expert: a power of two, within one warp
    while (tpe > 1 && tpe * E > ROUTE_THREADS) tpe >>= 1;
    const int e = tid / tpe, j = tid - e * tpe;
    const bool mine = e < E;
    int *row = blk + (size_t)(mine ? e : 0) * CP;
    const int rounds = CP / (4 * tpe);  // at least 1: CP is a multiple of 128
    int carry = 0;
    for (int r0 = 0; r0 < rounds; r0 += 8) {
        int4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            v[u] = mine && r0 + u < rounds ? load_counts(row, 4 * ((r0 + u) * tpe + j), C) : make_int4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (r0 + u >= rounds) break;  // the same for every lane
            const int sum = v[u].x + v[u].y + v[u].z + v[u].w;
            int inc = sum;  // inclusive scan of the round over the expert's lanes
            for (int o = 1; o < tpe; o <<= 1) {
                const int t = __shfl_up_sync(0xFFFFFFFFu, inc, o, tpe);
                if (j >= o) inc += t;
            }
            const int total = __shfl_sync(0xFFFFFFFFu, inc, tpe - 1, tpe);
            int run = carry + inc - sum;
            int4 o4;
            o4.x = run;
            run += v[u].x;
            o4.y = run;
            run += v[u].y;
            o4.z = run;
            run += v[u].z;
            o4.w = run;
            if (mine) *reinterpret_cast<int4 *>(row + 4 * ((r0 + u) * tpe + j)) = o4;
            carry += total;
        }
    }
    if (mine && j == 0) cnt[e] = carry;
    __syncthreads();
    route_scan_tiles(cnt, pos, tile0, E, groups);
    for (int i = tid; i < E; i += ROUTE_THREADS) posg[i] = pos[i];
}

// Chunk blockIdx.x: each valid slot takes the next sorted row of its expert
// (the chunk's first row of that expert, blk, plus a cursor; an expert's
// rows are in no particular order: each output row depends on its own X row
// only), records slot_of, and the chunk's X rows are copied to their sorted
// rows (one warp per row, 16-byte copies, eight in flight per lane).
__global__ void __launch_bounds__(GATHER_THREADS) moe_place_gather_kernel(
    const int32_t *__restrict__ ids, int S, int E, const int *__restrict__ blk, int CP, const int *__restrict__ posg,
    int *__restrict__ slot_of, const uint16_t *__restrict__ x, int topk, int K, uint16_t *__restrict__ xs)
{
    __shared__ int cur[ROUTE_SMALL_E];
    __shared__ int prow[ROUTE_CHUNK];
    const int tid = threadIdx.x, c = blockIdx.x;
    const int s = c * ROUTE_CHUNK + tid;
    pdl_trigger();
    pdl_wait();
    const int e = tid < ROUTE_CHUNK && s < S ? ids[s] : -1;
    for (int i = tid; i < E; i += GATHER_THREADS) cur[i] = __ldcg(posg + i) + __ldcg(blk + (size_t)i * CP + c);
    __syncthreads();
    if (tid < ROUTE_CHUNK) {
        int p = -1;
        if ((unsigned)e < (unsigned)E) {
            p = atomicAdd(&cur[e], 1);
            slot_of[p] = s;
        }
        prow[tid] = p;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int vec = K / 8;  // 16-byte chunks per row
    for (int i = warp; i < ROUTE_CHUNK; i += GATHER_THREADS / 32) {
        const int p = prow[i];
        if (p < 0) continue;
        const int t = (c * ROUTE_CHUNK + i) / topk;
        // x may have been written by the kernel before this one: coherent (L2) loads
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * K);
        uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)p * K);
        int k = lane;
        for (; k + 224 < vec; k += 256) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + k + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u) dst[k + 32 * u] = v[u];
        }
        for (; k < vec; k += 32) dst[k] = __ldcg(src + k);
    }
}

// xs[p] = x[slot_of[p] / topk] for the valid sorted rows, one warp per row.
__global__ void gather_rows_kernel(const uint16_t *__restrict__ x, const int *__restrict__ groups,
                                   const int *__restrict__ slot_of, int topk, int K, uint16_t *__restrict__ xs)
{
    pdl_trigger();
    pdl_wait();
    const int rows = __ldcg(groups + 1);
    const int wpb = blockDim.x >> 5, lane = threadIdx.x & 31;
    const int vec = K / 8;  // 16-byte chunks per row
    for (int p = blockIdx.x * wpb + (threadIdx.x >> 5); p < rows; p += gridDim.x * wpb) {
        const int t = __ldcg(slot_of + p) / topk;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * K);
        uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)p * K);
        // x may have been written by the kernel before this one: coherent (L2) loads
        for (int c = lane; c < vec; c += 32) dst[c] = __ldcg(src + c);
    }
}

// out[t][n] = sum_j r[t][j] * yd[t * topk + j][n] (fmaf in slot order), yd
// bf16; NaN for a token with an expert id outside [0, E).  Eight columns per
// thread.
__global__ void combine_bf16_kernel(const uint16_t *__restrict__ yd, const float *__restrict__ r,
                                    const int32_t *__restrict__ ids, int E, float *__restrict__ out, int T, int topk,
                                    int N)
{
    pdl_trigger();
    pdl_wait();
    const int n8 = N / 8;
    const size_t total = (size_t)T * n8;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / n8), c = (int)(i - (size_t)t * n8);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        bool bad = false;
        for (int j = 0; j < topk; ++j) {
            const int s = t * topk + j;
            bad |= (unsigned)ids[s] >= (unsigned)E;
            const float w = r[s];
            const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(yd + (size_t)s * N) + c);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = fmaf(w, __uint_as_float(u[q] << 16), acc[2 * q]);
                acc[2 * q + 1] = fmaf(w, __uint_as_float(u[q] & 0xFFFF0000u), acc[2 * q + 1]);
            }
        }
        if (bad)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = __int_as_float(0x7FC00000);
        float4 *o = reinterpret_cast<float4 *>(out + (size_t)t * N) + 2 * c;
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

static cudaError_t route_and_gather(const DeviceState &ds, cudaStream_t st, const MoeGroupPlan &p, uint8_t *ws,
                                    const uint16_t *x, const int32_t *ids, int E, int topk, int K, uint16_t *ynan,
                                    int ynan_w)
{
    int *groups = reinterpret_cast<int *>(ws + p.off_groups);
    int *slot_of = reinterpret_cast<int *>(ws + p.off_slot);
    uint16_t *xs = reinterpret_cast<uint16_t *>(ws + p.off_xs);
    if (E <= ROUTE_SMALL_E) {
        const int C = route_chunks(p.S), CP = route_stride(C);
        int *blk = reinterpret_cast<int *>(ws + route_table_offset(p.off_slot, p.S));
        int *posg = blk + (size_t)E * CP;
        cudaError_t e = launch_k(moe_count_kernel, dim3(C), dim3(ROUTE_CHUNK), 0, st, ids, p.S, E, CP, blk, ynan,
                                 ynan_w, ds.err);
        if (e != cudaSuccess) return e;
        e = launch_k(moe_scan_kernel, dim3(1), dim3(ROUTE_THREADS), 0, st, blk, C, CP, E, groups, posg);
        if (e != cudaSuccess) return e;
        return launch_k(moe_place_gather_kernel, dim3(C), dim3(GATHER_THREADS), 0, st, ids, p.S, E,
                        (const int *)blk, CP, (const int *)posg, slot_of, x, topk, K, xs);
    }
    // three [E] int tables: up to 48 KiB, plus the static shared memory
    static int configured_dev[64] = {0};
    if (ds.device < 64 && !configured_dev[ds.device]) {
        cudaError_t e = cudaFuncSetAttribute(moe_group_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             3 * MOE_MAX_EXPERTS * (int)sizeof(int));
        if (e != cudaSuccess) return e;
        configured_dev[ds.device] = 1;
    }
    cudaError_t e = launch_k(moe_group_route_kernel, dim3(1), dim3(ROUTE_THREADS), (size_t)3 * E * sizeof(int), st,
                             ids, p.S, E, groups, slot_of, ynan, ynan_w, ds.err);
    if (e != cudaSuccess) return e;
    int blocks = (p.S + 7) / 8;  // 8 warps (rows) per block
    const int cap = ds.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_k(gather_rows_kernel, dim3(blocks), dim3(256), 0, st, x, (const int *)groups, (const int *)slot_of,
                    topk, K, xs);
}

cudaError_t launch_moe_qmm(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, const uint16_t *x, const int32_t *ids, uint16_t *y, int T, int E,
                           int topk, int N, int K, void *workspace)
{
    const MoeGroupPlan p = moe_group_plan(T, E, topk, K, 0);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e = route_and_gather(ds, st, p, ws, x, ids, E, topk, K, y, N);
    if (e != cudaSuccess) return e;
    return launch_qmm_grouped(ds, st, fmt, false, codes, scales, reinterpret_cast<const uint16_t *>(ws + p.off_xs),
                              p.S, reinterpret_cast<const int *>(ws + p.off_groups), p.max_groups,
                              reinterpret_cast<const int *>(ws + p.off_slot), y, E, N, K);
}

cudaError_t launch_moe_ffn_prefill(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *gu_codes,
                                   const uint8_t *gu_scales, const uint8_t *dn_codes, const uint8_t *dn_scales,
                                   const uint16_t *x, const int32_t *ids, const float *rw, float *out, int T, int E,
                                   int topk, int H, int I, void *workspace)
{
    const MoeGroupPlan p = moe_group_plan(T, E, topk, H, I);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int *groups = reinterpret_cast<const int *>(ws + p.off_groups);
    const int *slot_of = reinterpret_cast<const int *>(ws + p.off_slot);
    uint16_t *xs = reinterpret_cast<uint16_t *>(ws + p.off_xs);
    uint16_t *hs = reinterpret_cast<uint16_t *>(ws + p.off_hs);
    cudaError_t e = route_and_gather(ds, st, p, ws, x, ids, E, topk, H, nullptr, 0);
    if (e != cudaSuccess) return e;
    // gate and up rows of each routed expert, SwiGLU in the epilogue: h in expert order
    e = launch_qmm_grouped(ds, st, fmt, true, gu_codes, gu_scales, xs, p.S, groups, p.max_groups, slot_of, hs, E,
                           2 * I, H);
    if (e != cudaSuccess) return e;
    // down rows: outputs back to slot order, over the gathered activations (no longer needed)
    e = launch_qmm_grouped(ds, st, fmt, false, dn_codes, dn_scales, hs, p.S, groups, p.max_groups, slot_of, xs, E, H,
                           I);
    if (e != cudaSuccess) return e;
    size_t blocks = ((size_t)T * (H / 8) + 255) / 256;
    const size_t cap = (size_t)ds.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return launch_k(combine_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, (const uint16_t *)xs, rw, ids, E,
                    out, T, topk, H);
}

}  // namespace mx
