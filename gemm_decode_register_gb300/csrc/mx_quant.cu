// mx_quant.cu -- on-device block-float quantisation of bf16 activations to
// MXFP4 / MXFP8 / NVFP4 (the reverse of the decode the matmul kernels do).
//
// The pages run block-float quantisation on the GPU's hardware NVFP4 /
// MXFP4 converter on Blackwell (manual page "Building from source", CUDA
// build options, "GPU architecture auto-detection") and re-quantise FP8
// block checkpoints to MXFP8 (manual, ROCm status table).  The procedure,
// which the pages leave open, is the plain reading of the format
// definitions:
//   MXFP4 / MXFP8 (OCP MX v1.0 conversion): per block of 32, shared exponent
//     e = floor(log2(amax)) - emax_elem (2 for E2M1, 8 for E4M3), at least
//     -127 (amax = 0 or a bf16 subnormal gives -127); scale byte e + 127;
//     elements x * 2^-e (exact in fp32) converted nearest-even with
//     saturation by the hardware converter (cvt.rn.satfinite).
//   NVFP4: g = fp32(G / 2688), G = the largest finite |x| of the tensor
//     (g = 1 when G = 0), written after the scales; per block of 16,
//     s = E4M3(fp32(amax / fp32(6 g))) and elements fp32(x / fp32(s g)) to
//     E2M1 (all zero when s g = 0).
//   A block holding a NaN or an infinity gets a NaN scale (E8M0 0xFF, E4M3
//   0x7F) and zero codes; every zero code is +0.
// One thread per block: MX reads 64 bytes and writes 16 (MXFP4) or 32
// (MXFP8) bytes of codes and one scale byte; the kernel is HBM-bound
// (2 bytes read and 0.53-1.03 bytes written per element).
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

// Eight fp32 values to eight E2M1 codes, v[0] in the lowest nibble, each
// nearest-even with saturation (the converter puts its first operand in the
// high nibble of the byte).
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float (&v)[8])
{
    uint32_t d;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(d)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return d;
}

// Four fp32 values to four E4M3 codes, v[0] in the lowest byte.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float v0, float v1, float v2, float v3)
{
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v1), "f"(v0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v3), "f"(v2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// -0 codes (the sign bit alone) become +0: eight E2M1 nibbles, four E4M3 bytes.
__device__ __forceinline__ uint32_t e2m1x8_plus_zero(uint32_t w)
{
    const uint32_t t = w & 0x77777777u;
    const uint32_t zero = ~(t | (t >> 1) | (t >> 2)) & 0x11111111u;  // bit 4i: nibble i has magnitude 0
    return w & ~(zero << 3);
}

__device__ __forceinline__ uint32_t e4m3x4_plus_zero(uint32_t w)
{
    const uint32_t t = w & 0x7F7F7F7Fu;
    const uint32_t nonzero = (t + 0x7F7F7F7Fu) & 0x80808080u;  // bit 7 of byte i: magnitude i non-zero
    return w & (nonzero | 0x7F7F7F7Fu);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Largest |bits| of the bf16 pairs in w[0..n) (bf16 magnitudes compare as
// integers) and whether any of them is an infinity or a NaN.  One packed
// maximum of magnitudes per pair: a NaN operand makes that half NaN (the
// .NaN form) and an infinity is the largest magnitude, so the result is
// 0x7F80 or above exactly when the block holds either.
template <int N>
__device__ __forceinline__ uint32_t bf16_amax(const uint32_t (&w)[N], bool &nonfinite)
{
    uint32_t m2 = 0u;
#pragma unroll
    for (int i = 0; i < N; ++i) asm("max.NaN.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w[i]));
    const uint32_t m = max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu);
    nonfinite = m >= 0x7F80u;
    return m;
}

// Largest finite magnitude bits of the bf16 pairs of a 16-byte vector: a
// packed maximum of magnitudes (NaNs lose to the other operand), redone
// element by element when an infinity (or an all-NaN pair) came out on top.
__device__ __forceinline__ uint32_t vec_fin_amax(const uint4 &v)
{
    uint32_t m2;
    asm("{\n\t.reg .b32 t, u;\n\t"
        "max.xorsign.abs.bf16x2 t, %1, %2;\n\t"
        "max.xorsign.abs.bf16x2 u, %3, %4;\n\t"
        "max.xorsign.abs.bf16x2 %0, t, u;\n\t}"
        : "=r"(m2)
        : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
    uint32_t m = max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu);
    if (m >= 0x7F80u) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        m = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = w[j] & 0x7FFFu, hi = (w[j] >> 16) & 0x7FFFu;
            if (lo < 0x7F80u) m = max(m, lo);
            if (hi < 0x7F80u) m = max(m, hi);
        }
    }
    return m;
}

constexpr int AMAX_THREADS = 256;
constexpr int AMAX_UNROLL = 4;  // independent 16-byte loads in flight per thread

// G: the largest finite |x| over the tensor, as fp32 bits, by atomicMax into
// *gbits (zeroed by the host before the launch): each block reduces its
// share in registers and shared memory and adds one atomic.
__global__ void __launch_bounds__(AMAX_THREADS) quant_amax_kernel(const uint16_t *__restrict__ x, long long n8,
                                                                  unsigned *gbits)
{
    __shared__ uint32_t wmax[AMAX_THREADS / 32];
    pdl_trigger();
    pdl_wait();
    const uint4 *v = reinterpret_cast<const uint4 *>(x);
    const long long stride = (long long)gridDim.x * AMAX_THREADS;
    long long i = blockIdx.x * (long long)AMAX_THREADS + threadIdx.x;
    uint32_t m = 0;
    for (; i + (AMAX_UNROLL - 1) * stride < n8; i += AMAX_UNROLL * stride) {
        uint4 r[AMAX_UNROLL];
#pragma unroll
        for (int u = 0; u < AMAX_UNROLL; ++u) r[u] = __ldcg(v + i + u * stride);  // kept in L2 for the block pass
#pragma unroll
        for (int u = 0; u < AMAX_UNROLL; ++u) m = max(m, vec_fin_amax(r[u]));
    }
    for (; i < n8; i += stride) m = max(m, vec_fin_amax(__ldcg(v + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < AMAX_THREADS / 32 ? wmax[threadIdx.x] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (threadIdx.x == 0 && m) atomicMax(gbits, m << 16);
    }
}

// Eight quotients x_i / den to E2M1 codes, identical to converting the
// correctly rounded fp32 quotients Q_i.  With r = rcp(den) correctly rounded,
// rl = r (1 - 2^-21) and rh = r (1 + 2^-21) (both rounded), the products
// x_i rl and x_i rh (rounded) lie on either side of Q_i: each differs from
// x_i / den by the factor 1 -/+ 2^-21 and four roundings of at most 2^-24, and
// Q_i from x_i / den by one.  E2M1 conversion is monotone, so equal codes at
// both ends are the code of Q_i (the code of the plain product is not needed).
// Otherwise (rare: a quotient near a rounding boundary of E2M1, or rh beyond
// the fp32 range) the eight are divided after all; so are they when r
// overflows (den below 2^-128: a tensor whose largest magnitude is below
// about 2^-117).
__device__ __forceinline__ uint32_t e2m1x8_of_quotients(const float (&x)[8], float den, float rl, float rh)
{
    float lo[8], hi[8];
    if (rl <= 3.4028234663852886e38f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo[i] = __fmul_rn(x[i], rl);
            hi[i] = __fmul_rn(x[i], rh);
        }
        const uint32_t c = f32x8_to_e2m1x8(lo);
        if (f32x8_to_e2m1x8(hi) == c) return c;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) lo[i] = __fdiv_rn(x[i], den);
    return f32x8_to_e2m1x8(lo);
}

// One block's codes (NC 32-bit words) and scale byte from its W bf16 pairs.
template <int FMT, int W, int NC>
__device__ __forceinline__ uint32_t quant_block(const uint32_t (&w)[W], float g, float d6, uint32_t (&c)[NC])
{
#pragma unroll
    for (int i = 0; i < NC; ++i) c[i] = 0;
    bool nonfinite;
    const uint32_t amax = bf16_amax(w, nonfinite);
    if (nonfinite) return FMT == FMT_NVFP4 ? 0x7Fu : 0xFFu;
    if constexpr (FMT == FMT_NVFP4) {
        const float t = __fdiv_rn(__uint_as_float(amax << 16), d6);
        const uint32_t sbyte = f32x4_to_e4m3x4(t, 0.0f, 0.0f, 0.0f) & 0xFFu;
        const float den = __fmul_rn(f16_lo_to_f32(e4m3x2_to_f16x2(sbyte)), g);  // s exactly, times g
        if (den != 0.0f) {
            const float rcp = __frcp_rn(den);
            const float rl = __fmul_rn(rcp, 1.0f - 0x1p-21f), rh = __fmul_rn(rcp, 1.0f + 0x1p-21f);
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[2 * j] = bf16_lo(w[4 * i + j]);
                    v[2 * j + 1] = bf16_hi(w[4 * i + j]);
                }
                c[i] = e2m1x8_plus_zero(e2m1x8_of_quotients(v, den, rl, rh));
            }
        }
        return sbyte;
    } else {
        constexpr int EMAX = FMT == FMT_MXFP8 ? 8 : 2;
        const int E = (int)(amax >> 7);  // bf16 exponent field of amax
        const int e = E == 0 ? -127 : max(E - 127 - EMAX, -127);
        const float mul = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, a normal fp32
        if constexpr (FMT == FMT_MXFP8) {
#pragma unroll
            for (int i = 0; i < NC; ++i)
                c[i] = e4m3x4_plus_zero(f32x4_to_e4m3x4(bf16_lo(w[2 * i]) * mul, bf16_hi(w[2 * i]) * mul,
                                                        bf16_lo(w[2 * i + 1]) * mul, bf16_hi(w[2 * i + 1]) * mul));
        } else {
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[2 * j] = bf16_lo(w[4 * i + j]) * mul;  // exact
                    v[2 * j + 1] = bf16_hi(w[4 * i + j]) * mul;
                }
                c[i] = e2m1x8_plus_zero(f32x8_to_e2m1x8(v));
            }
        }
        return (uint32_t)(e + 127);
    }
}

// Each thread takes P consecutive blocks per step (P = 2 for NVFP4, so that
// every thread, as for the MX formats, reads 64 contiguous bytes per step).
template <int FMT>
__global__ void quantize_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ codes,
                                uint8_t *__restrict__ scales, long long nblocks, const unsigned *gbits)
{
    constexpr int B = FMT == FMT_NVFP4 ? 16 : 32;          // elements per block
    constexpr int W = B / 2;                                 // bf16 pairs per block
    constexpr int NC = FMT == FMT_MXFP8 ? B / 4 : B / 8;     // 32-bit code words per block
    constexpr int P = FMT == FMT_NVFP4 ? 2 : 1;              // blocks per thread and step
    pdl_trigger();
    pdl_wait();
    float g = 1.0f, d6 = 6.0f;
    if constexpr (FMT == FMT_NVFP4) {
        const float G = __uint_as_float(__ldcg(gbits));
        if (G > 0.0f) g = __fdiv_rn(G, 2688.0f);
        d6 = __fmul_rn(6.0f, g);
        if (blockIdx.x == 0 && threadIdx.x == 0) {  // the tensor scale, after the block scales (any alignment)
            const uint32_t gb = __float_as_uint(g);
            uint8_t *p = scales + nblocks;
            p[0] = (uint8_t)gb;
            p[1] = (uint8_t)(gb >> 8);
            p[2] = (uint8_t)(gb >> 16);
            p[3] = (uint8_t)(gb >> 24);
        }
    }
    const long long nsteps = (nblocks + P - 1) / P;
    for (long long st = blockIdx.x * (long long)blockDim.x + threadIdx.x; st < nsteps;
         st += (long long)gridDim.x * blockDim.x) {
        const long long b0 = st * P;
        const int nb = nblocks - b0 < P ? (int)(nblocks - b0) : P;
        uint32_t w[P][W];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (b0 + p) * B);
#pragma unroll
            for (int i = 0; i < W / 4; ++i) {
                const uint4 v = p < nb ? __ldcs(src + i) : make_uint4(0u, 0u, 0u, 0u);
                w[p][4 * i] = v.x;
                w[p][4 * i + 1] = v.y;
                w[p][4 * i + 2] = v.z;
                w[p][4 * i + 3] = v.w;
            }
        }
        uint32_t c[P][NC], sb[P];
#pragma unroll
        for (int p = 0; p < P; ++p) sb[p] = quant_block<FMT, W, NC>(w[p], g, d6, c[p]);
        if constexpr (FMT == FMT_MXFP8) {
            scales[b0] = (uint8_t)sb[0];
            uint4 *dst = reinterpret_cast<uint4 *>(codes + b0 * 32);
            dst[0] = make_uint4(c[0][0], c[0][1], c[0][2], c[0][3]);
            dst[1] = make_uint4(c[0][4], c[0][5], c[0][6], c[0][7]);
        } else if constexpr (FMT == FMT_MXFP4) {
            scales[b0] = (uint8_t)sb[0];
            *reinterpret_cast<uint4 *>(codes + b0 * 16) = make_uint4(c[0][0], c[0][1], c[0][2], c[0][3]);
        } else if (nb == 2) {
            *reinterpret_cast<uint16_t *>(scales + b0) = (uint16_t)(sb[0] | (sb[1] << 8));
            *reinterpret_cast<uint4 *>(codes + b0 * 8) = make_uint4(c[0][0], c[0][1], c[1][0], c[1][1]);
        } else {
            scales[b0] = (uint8_t)sb[0];
            *reinterpret_cast<uint2 *>(codes + b0 * 8) = make_uint2(c[0][0], c[0][1]);
        }
    }
}

cudaError_t launch_quantize(const DeviceState &ds, cudaStream_t st, int fmt, const uint16_t *x, uint8_t *codes,
                            uint8_t *scales, int M, int K)
{
    const int B = fmt == FMT_NVFP4 ? 16 : 32;
    const long long nblocks = (long long)M * (K / B);
    const long long steps = fmt == FMT_NVFP4 ? (nblocks + 1) / 2 : nblocks;  // see quantize_kernel
    long long grid = (steps + 255) / 256;
    const long long cap = (long long)ds.num_sms * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    unsigned *gbits = ds.amax;  // the calling stream's tensor-maximum word (NVFP4 only)
    if (fmt == FMT_NVFP4) {
        if (gbits == nullptr) return cudaErrorInvalidValue;
        cudaError_t e = cudaMemsetAsync(gbits, 0, sizeof(unsigned), st);
        if (e != cudaSuccess) return e;
        const long long n8 = (long long)M * K / 8;
        long long g2 = (n8 + AMAX_THREADS * AMAX_UNROLL - 1) / (AMAX_THREADS * AMAX_UNROLL);
        const long long cap2 = (long long)ds.num_sms * (2048 / AMAX_THREADS);  // one wave
        if (g2 > cap2) g2 = cap2;
        if (g2 < 1) g2 = 1;
        e = launch_k(quant_amax_kernel, dim3((unsigned)g2), dim3(AMAX_THREADS), 0, st, x, n8, gbits);
        if (e != cudaSuccess) return e;
        return launch_k(quantize_kernel<FMT_NVFP4>, dim3((unsigned)grid), dim3(256), 0, st, x, codes, scales,
                        nblocks, (const unsigned *)gbits);
    }
    if (fmt == FMT_MXFP8)
        return launch_k(quantize_kernel<FMT_MXFP8>, dim3((unsigned)grid), dim3(256), 0, st, x, codes, scales,
                        nblocks, (const unsigned *)gbits);
    return launch_k(quantize_kernel<FMT_MXFP4>, dim3((unsigned)grid), dim3(256), 0, st, x, codes, scales, nblocks,
                    (const unsigned *)gbits);
}

}  // namespace mx
