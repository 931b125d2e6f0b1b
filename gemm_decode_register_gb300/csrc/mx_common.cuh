// mx_common.cuh -- device helpers shared by the sm_103a kernels: exact
// block-float decodes, scale conversions and the m16n8k16 tensor op.
//
// E2M1 decode ("MLxcel 0.8 release", section "Decoding block-float formats
// in software"; Strix Halo talk, slide 12): the pages place each E2M1
// nibble into fp16 sign/exponent/mantissa bits and fix the exponent offset
// with one multiply.  sm_103a has that conversion in hardware:
// cvt.rn.f16x2.e2m1x2 turns one byte (two nibbles) into two exact fp16
// values (0, +-0.5 .. +-6 are all normal fp16 numbers), so no corrective
// multiply is needed.  E4M3 likewise converts exactly to fp16
// (cvt.rn.f16x2.e4m3x2), and E8M0 exactly to bf16 (cvt.rn.bf16x2.ue8m0x2;
// 2^-127 becomes a bf16 subnormal, 0xFF a NaN).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// Launch a kernel of this library with programmatic stream serialisation
// (see pdl_trigger / pdl_wait).
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                   Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

namespace mx {

enum : int { FMT_MXFP4 = 0, FMT_MXFP8 = 1, FMT_NVFP4 = 2 };
enum : int { DEVERR_BAD_EXPERT = 0x1, DEVERR_TIMEOUT = 0x2 };

// ------------------------------------------------------------- conversions

// Two E2M1 nibbles (low nibble = first element) -> f16x2 (low half = first).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte)
{
    uint32_t out;
    asm("{\n\t.reg .b8 lo, hi;\n\t"
        "mov.b16 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, lo;\n\t}"
        : "=r"(out)
        : "h"((unsigned short)(byte & 0xFFu)));
    return out;
}

// Eight E2M1 nibbles of a word (nibble i = element i) -> four f16x2 words
// (word j holds elements 2j, 2j+1).  The bytes are split with a vector
// move, so the conversion reads them in place.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t &o0, uint32_t &o1, uint32_t &o2,
                                                uint32_t &o3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(w));
}

// Four E4M3 bytes of a word -> two f16x2 words (elements 0,1 and 2,3).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t &o0, uint32_t &o1)
{
    asm("{\n\t.reg .b16 h0, h1;\n\t"
        "mov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
        : "=r"(o0), "=r"(o1)
        : "r"(w));
}

// Two E4M3 bytes (low byte = first element) -> f16x2 (low half = first).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"((unsigned short)(two_bytes & 0xFFFFu)));
    return out;
}

// Two E8M0 bytes -> bf16x2 (exact).
__device__ __forceinline__ uint32_t ue8m0x2_to_bf16x2(uint32_t two_bytes)
{
    uint32_t out;
    asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(out) : "h"((unsigned short)(two_bytes & 0xFFFFu)));
    return out;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2)
{
    float f;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2)
{
    float f;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tcvt.f32.f16 %0, u;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

// bf16 bits (low 16) -> fp32, exact.
__device__ __forceinline__ float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

// E8M0 byte -> fp32 2^(e-127), exact (2^-127 kept as a subnormal, 0xFF NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e)
{
    return bf16_to_f32(ue8m0x2_to_bf16x2(e & 0xFFu) & 0xFFFFu);
}

// Two E8M0 bytes (low byte first) -> two fp32.
__device__ __forceinline__ void e8m0x2_to_f32(uint32_t two_bytes, float &a, float &b)
{
    uint32_t v = ue8m0x2_to_bf16x2(two_bytes);
    a = __uint_as_float(v << 16);
    b = __uint_as_float(v & 0xFFFF0000u);
}

// E4M3 byte -> fp32, exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) { return f16_lo_to_f32(e4m3x2_to_f16x2(b & 0xFFu)); }

// Two fp32 -> f16x2 (round to nearest even; lo in the low half).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi)
{
    uint32_t out;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

// Two fp32 -> bf16x2 (round to nearest even; lo in the low half).
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi)
{
    uint32_t out;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

// Exact 2^e as fp32 for e in [-149, 127]; 0 below, +inf above.
__device__ __forceinline__ float pow2f(int e)
{
    if (e > 127) return __uint_as_float(0x7F800000u);
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.0f;
}

// ---------------------------------------------------------- tensor op

// D = A(16x16, f16, row) * B(16x8, f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1, const float (&c)[4])
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]),
                   "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// ---------------------------------------------------------- launch overlap
//
// Programmatic dependent launch: every kernel of this library lets the next
// kernel on its stream start as soon as it begins (pdl_trigger), and waits
// for the previous kernel's completion and memory (pdl_wait) before it reads
// activations or writes outputs.  Weights (codes, block scales) and MoE
// expert ids may be read before the wait: no kernel of this library writes
// them, and the ABI requires them to be complete when a call is issued.
// Both are no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Ask L2 for the 128-byte lines of [p, p + bytes), the block's threads taking
// every blockDim-th line.  A prefetch moves nothing into the SM and has no
// effect on what later loads return (L2 is where the previous kernel's
// writes land), so it may be issued before griddepcontrol.wait: data that
// the previous kernel has not touched then starts its way from HBM ahead of
// the weight stream instead of queueing behind it.
__device__ __forceinline__ void prefetch_l2(const void *p, size_t bytes)
{
    const char *c = static_cast<const char *>(p);
    for (size_t o = (size_t)threadIdx.x * 128; o < bytes; o += (size_t)blockDim.x * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
}

// ---------------------------------------------------------- activation

// SwiGLU of one (gate, up) pair rounded to bf16 (bits in the low half):
// bf16(silu(g) * u) in fp32 arithmetic, silu(v) = v * sigmoid(v) with the
// sigmoid evaluated from e = exp(-|v|) (CUDA's expf, never overflows) as
// 1 / (1 + e) for v >= 0 and e / (1 + e) below, correctly rounded division.
__device__ __forceinline__ uint32_t swiglu_bf16(float g, float u)
{
    const float e = expf(-fabsf(g));
    const float sig = __fdiv_rn(g >= 0.0f ? 1.0f : e, __fadd_rn(1.0f, e));
    const float p = __fmul_rn(__fmul_rn(g, sig), u);
    return f32x2_to_bf16x2(p, 0.0f) & 0xFFFFu;
}

// ---------------------------------------------------------- misc

__device__ __forceinline__ void set_device_error(int *err, int bits)
{
    if (err) atomicOr(err, bits);
}

// Read a possibly unaligned little-endian fp32 from global memory.
__device__ __forceinline__ float load_f32_unaligned(const uint8_t *p)
{
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    return __uint_as_float(u);
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_nc_u64(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_nc_u16(const void *p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.b16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_nc_u8(const void *p)
{
    unsigned short v;
    asm volatile("ld.global.nc.b8 %0, [%1];" : "=h"(v) : "l"(p));
    return v & 0xFFu;
}

}  // namespace mx
