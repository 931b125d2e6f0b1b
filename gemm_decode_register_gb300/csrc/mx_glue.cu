// mx_glue.cu -- the small kernels around the hot path: exact dequantisation
// (the decode exposed for exactness tests), SwiGLU between the MoE gate-up
// and down projections, and the router-weighted combine.
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

// W[n][k] = fp32(code * scale): 8 consecutive elements per thread.
// Exact: an E2M1 or E4M3 value times a power of two (MX) or an E4M3 scale
// (NVFP4) has at most 6 significant bits and stays in fp32 range except for
// true overflow, which rounds to inf as IEEE requires.  NVFP4 then applies
// the fp32 tensor scale with one round-to-nearest-even multiply.
template <int FMT>
__global__ void dequant_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales,
                               float *__restrict__ W, int N, int K)
{
    pdl_trigger();
    pdl_wait();
    const size_t groups = (size_t)N * (K / 8);
    float g = 1.0f;
    if (FMT == FMT_NVFP4) g = load_f32_unaligned(scales + (size_t)N * (K / 16));
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < groups;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t n = i / (K / 8);
        const int k0 = (int)(i - n * (K / 8)) * 8;
        float v[8];
        if constexpr (FMT == FMT_MXFP8) {
            const uint2 c = *reinterpret_cast<const uint2 *>(codes + n * K + k0);
            uint32_t h[4] = {e4m3x2_to_f16x2(c.x), e4m3x2_to_f16x2(c.x >> 16), e4m3x2_to_f16x2(c.y),
                             e4m3x2_to_f16x2(c.y >> 16)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] = f16_lo_to_f32(h[j]);
                v[2 * j + 1] = f16_hi_to_f32(h[j]);
            }
        } else {
            const uint32_t c = *reinterpret_cast<const uint32_t *>(codes + n * (K / 2) + k0 / 2);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t h = e2m1x2_to_f16x2(c >> (8 * j));
                v[2 * j] = f16_lo_to_f32(h);
                v[2 * j + 1] = f16_hi_to_f32(h);
            }
        }
        float s;
        if constexpr (FMT == FMT_NVFP4) s = e4m3_to_f32(scales[n * (K / 16) + k0 / 16]);
        else s = e8m0_to_f32(scales[n * (K / 32) + k0 / 32]);
        float4 o0, o1;
        float *o = &o0.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __fmul_rn(v[j], s);
        o = &o1.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __fmul_rn(v[4 + j], s);
        if constexpr (FMT == FMT_NVFP4) {
            o0.x = __fmul_rn(o0.x, g); o0.y = __fmul_rn(o0.y, g); o0.z = __fmul_rn(o0.z, g); o0.w = __fmul_rn(o0.w, g);
            o1.x = __fmul_rn(o1.x, g); o1.y = __fmul_rn(o1.y, g); o1.z = __fmul_rn(o1.z, g); o1.w = __fmul_rn(o1.w, g);
        }
        float4 *dst = reinterpret_cast<float4 *>(W + n * K + k0);
        dst[0] = o0;
        dst[1] = o1;
    }
}

cudaError_t launch_dequant(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, float *W, int N, int K)
{
    const size_t groups = (size_t)N * (K / 8);
    size_t blocks = (groups + 255) / 256;
    const size_t cap = (size_t)ds.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    if (fmt == FMT_MXFP4) return launch_k(dequant_kernel<FMT_MXFP4>, dim3((unsigned)blocks), dim3(256), 0, st, codes, scales, W, N, K);
    if (fmt == FMT_MXFP8) return launch_k(dequant_kernel<FMT_MXFP8>, dim3((unsigned)blocks), dim3(256), 0, st, codes, scales, W, N, K);
    return launch_k(dequant_kernel<FMT_NVFP4>, dim3((unsigned)blocks), dim3(256), 0, st, codes, scales, W, N, K);
}

// h = bf16(silu(gate) * up) (swiglu_bf16).
__global__ void swiglu_kernel(const float *__restrict__ gu, uint16_t *__restrict__ h, int Q, int I)
{
    pdl_trigger();
    pdl_wait();
    const size_t total = (size_t)Q * I;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t q = i / I, j = i - q * I;
        h[i] = (uint16_t)swiglu_bf16(gu[q * 2 * I + j], gu[q * 2 * I + I + j]);
    }
}

cudaError_t launch_swiglu(const DeviceState &ds, cudaStream_t st, const float *gu, uint16_t *h,
                          int Q, int I)
{
    size_t blocks = ((size_t)Q * I + 255) / 256;
    const size_t cap = (size_t)ds.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return launch_k(swiglu_kernel, dim3((unsigned)blocks), dim3(256), 0, st, gu, h, Q, I);
}

// out[t][n] = sum_j r[t][j] * yd[t*topk + j][n] (fp32, increasing j).
__global__ void combine_kernel(const float *__restrict__ yd, const float *__restrict__ r,
                               float *__restrict__ out, int T, int topk, int N)
{
    pdl_trigger();
    pdl_wait();
    const size_t total = (size_t)T * N;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / N, n = i - t * N;
        float acc = 0.f;
        for (int j = 0; j < topk; ++j) acc = fmaf(r[t * topk + j], yd[(t * topk + j) * N + n], acc);
        out[i] = acc;
    }
}

cudaError_t launch_moe_combine(const DeviceState &ds, cudaStream_t st, const float *yd,
                               const float *r, float *out, int T, int topk, int N)
{
    size_t blocks = ((size_t)T * N + 255) / 256;
    const size_t cap = (size_t)ds.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return launch_k(combine_kernel, dim3((unsigned)blocks), dim3(256), 0, st, yd, r, out, T, topk, N);
}

}  // namespace mx
