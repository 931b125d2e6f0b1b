/*
 * mx.h -- C ABI of the block-float decode-in-kernel matmul library
 * (libmxgemm.so, sm_103a).
 *
 * The operation: y = x . W^T where the weight W[N][K] is stored as packed
 * low-precision codes plus one shared scale per block, and is decoded
 * inside the kernel.  Formats ("MLxcel 0.8 release", section "Decoding
 * block-float formats in software"; talk "High-performance LLM/VLM
 * inference on AMD Strix Halo with mlxcel engine", slide 7 "AMD Strix
 * Halo: The Target Platform" and slide 12 "Software Decode for Block Float
 * Formats" name MXFP4, MXFP8 and NVFP4 and fix the E2M1 element as 1 sign,
 * 2 exponent and 1 mantissa bit, decoded exactly; the rest follows the
 * OCP MX v1.0 and NVFP4 definitions those pages refer to):
 *
 *   MX_FMT_MXFP4  E2M1 codes, 2 per byte, one E8M0 scale per 32 elements
 *   MX_FMT_MXFP8  E4M3 codes, 1 per byte, one E8M0 scale per 32 elements
 *   MX_FMT_NVFP4  E2M1 codes, 2 per byte, one E4M3 scale per 16 elements,
 *                 times one fp32 per-tensor scale
 *
 * Layouts (all row-major, little-endian):
 *   codes   uint8 [N][K/2] (4-bit formats: element k in byte k/2, even k in
 *           the low nibble) or [N][K] (MXFP8).
 *   scales  uint8 [N][K/block].  NVFP4: the fp32 per-tensor scale follows
 *           immediately after these N*K/16 bytes (any alignment).
 *   x, X    bf16 [M][K];  y fp32 [M][N];  Y bf16 [M][N].
 *   MoE     expert e's codes start at e*N*(bytes per row), its scales at
 *           e*N*(K/block); NVFP4 stacks carry E fp32 tensor scales after the
 *           whole [E][N][K/16] scale block, one per expert.
 *
 * Values: E8M0 byte e = 2^(e-127), 0xFF = NaN; E4M3 has bias 7, no
 * infinities, S.1111.111 = NaN, max 448.  Decoding is exact (see
 * mx_dequant).  Products accumulate in fp32; their rounding order is the
 * kernel's, not a fixed sequential one.
 *
 * Ownership and execution: every pointer is a caller-owned DEVICE pointer
 * on the current CUDA device.  Calls are asynchronous on the stream set with
 * mx_set_stream (per host thread; default: the legacy default stream),
 * re-entrant across host threads and streams, and return as soon as the
 * kernels are queued.  The device error word is a variable of the library
 * image.  Calls whose kernels pass partial sums through global memory
 * (mx_qmv when K is split across CTAs, mx_moe_gate_up_swiglu for rows the
 * streaming kernel cannot take, mx_moe_down_combine, NVFP4 mx_quantize) use a 16 MiB workspace slot of the stream they are issued on,
 * so calls on different streams never share one; a stream's slot is
 * allocated and cleared by the first such call on it (cudaMalloc, with the
 * calling thread switched to relaxed capture mode for it, so that first call
 * may come inside a stream capture) and kept until the process exits.  The
 * per-thread default stream gets one slot per host thread.  A captured graph
 * keeps using the slot of the stream it was captured on: do not replay it
 * concurrently with itself or with calls on that stream.  mx_qmv_noalloc
 * never allocates.
 *
 * Errors: 0 on success, otherwise a negative MX_E* code; the call then
 * launched nothing.  Faults found on the device (an expert id out of range,
 * a pipeline wait that timed out) do not trap: the kernel writes NaN to the
 * affected outputs, sets a bit in the device error word and returns;
 * mx_device_error() reads and clears it.
 */
#ifndef MX_H
#define MX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum mx_fmt { MX_FMT_MXFP4 = 0, MX_FMT_MXFP8 = 1, MX_FMT_NVFP4 = 2 };

enum mx_status {
    MX_OK = 0,
    MX_EINVAL = -1,       /* null pointer, a size <= 0, K not a multiple of the block */
    MX_EUNSUPPORTED = -2, /* unknown format, or a size beyond what the kernel handles */
    MX_EALIGN = -3,       /* a pointer is not 16-byte aligned */
    MX_ECUDA = -4,        /* a CUDA runtime call or the launch failed */
    MX_EDEVICE = -5       /* (mx_device_error only) a device-side check fired */
};

/* Device error word bits, as returned by mx_device_error(). */
#define MX_DEVERR_BAD_EXPERT 0x1 /* an expert id outside [0, E); that slot's y rows are NaN */
#define MX_DEVERR_TIMEOUT 0x2    /* a bounded pipeline wait gave up; that tile of Y is NaN */

/* Decode GEMV for a few tokens (the memory-bound decode step; "MLxcel 0.8
 * release", section "Profiling set the porting order": the qmv kernel is 95%
 * of dense decode GPU time):
 *   y[m][n] = sum_k x[m][k] * W[n][k],   m < M, n < N.
 * x bf16 [M][K], y fp32 [M][N].  Any M >= 1 is accepted; the weight is
 * streamed once per group of up to 8 tokens (groups of rows longer than
 * about 10^5 elements whose K windows' partial sums exceed the stream's
 * workspace run as smaller groups).  K must be a multiple of 32
 * (MXFP4, MXFP8) or 16 (NVFP4); K <= 2^20.  codes, scales, x, y 16-byte
 * aligned. */
int mx_qmv(int fmt, const void *codes, const void *scales, const void *x, float *y, int M, int N,
           int K);

/* MoE decode GEMV over routed experts only (talk slide 4 "UMA Advantage for
 * MoE Architecture": each token reads only its active experts; manual page
 * "Building from source", ROCm status table: single-token MoE decode runs
 * a gate-up kernel then a down kernel):
 *   y[t][j][n] = sum_k x[t][k] * W_{e}[n][k],  e = expert_ids[t][j].
 * expert_codes / expert_scales hold E stacked [N][K] weights (layout
 * above); x bf16 [T][K]; expert_ids int32 [T][topk]; y fp32 [T][topk][N].
 * Slots that share an expert are served by one pass over that expert's
 * weights.  The routing is read on the device (no host copy).  T*topk <=
 * 1024, E <= 4096; the T rows of x (padded bf16) and the routing tables
 * must fit one CTA's shared memory (about 110,000 elements of K for one
 * token, proportionally fewer for more), else MX_EUNSUPPORTED.  The fused
 * MoE calls have the same bound on their staged rows (x's T rows for
 * mx_moe_gate_up_swiglu, h's T*topk rows for mx_moe_down_combine); rows too
 * long for their streaming kernels run through the direct-load kernel and
 * the workspace instead.  The ids are read as soon as the kernel starts, before it
 * waits for the preceding kernel on the stream (the routed experts' weights
 * start streaming under that kernel's tail): they must be complete when the
 * call is issued, i.e. not written by a kernel that lets its dependents start
 * early (no kernel of this library writes expert ids; activations and outputs
 * do wait).  The same holds for mx_moe_gate_up_swiglu and
 * mx_moe_down_combine.  An id outside [0, E) sets MX_DEVERR_BAD_EXPERT and fills that
 * slot's N outputs with NaN.  For the down projection call with T' = T*topk
 * rows of x, topk = 1 and the ids flattened to [T*topk][1]. */
int mx_moe_qmv(int fmt, const void *expert_codes, const void *expert_scales, const void *x,
               const int32_t *expert_ids, float *y, int T, int E, int topk, int N, int K);

/* Fused MoE FFN, first half: gate and up projections of the routed experts
 * with the SwiGLU applied as the outputs are formed (the pages' fused MoE
 * decode: manual page "Building from source", ROCm status table, a gate-up
 * kernel then a down kernel per layer; talk slide 13 "Porting Order Set by
 * Profiling", the fused-MoE port):
 *   h[t][j][i] = bf16_rne( silu(g) * u ),  g = sum_k x[t][k] * W_e[i][k],
 *                                          u = sum_k x[t][k] * W_e[I + i][k],
 * e = expert_ids[t][j].  Each expert's weight is [2I][K]: rows 0..I-1 gate,
 * rows I..2I-1 up (NVFP4: E fp32 tensor scales after the whole
 * [E][2I][K/16] scale block).  x bf16 [T][K]; h bf16 [T][topk][I].  silu and
 * the rounding are those of mx_swiglu, so h equals mx_swiglu applied to
 * mx_moe_qmv's output with N = 2I.  When K is not a multiple of 128, or
 * the staged rows of x do not fit beside the streaming kernel's weight ring,
 * the products come from the direct-load MoE kernel through the calling
 * stream's workspace slot, then the SwiGLU glue (two launches; T*topk*2I <=
 * 4 Mi floats).  Other limits and the bad-id behaviour (h rows NaN) as in
 * mx_moe_qmv.  codes, scales, x, h 16-byte aligned; ids 4-byte aligned. */
int mx_moe_gate_up_swiglu(int fmt, const void *expert_codes, const void *expert_scales, const void *x,
                          const int32_t *expert_ids, void *h, int T, int E, int topk, int I, int K);

/* Fused MoE FFN, second half: down projection of each routed slot and the
 * router-weighted sum over the token's slots:
 *   out[t][n] = sum_j r[t][j] * ( sum_k h[t*topk + j][k] * W_e[n][k] ),
 * e = expert_ids[t][j], summed over j in increasing order with fused
 * multiply-adds (as mx_moe_combine).  Expert weights [N][K]; h bf16
 * [T*topk][K] (mx_moe_gate_up_swiglu's output, K = I); r fp32 [T][topk];
 * out fp32 [T][N].  Slots that share an expert are served by one pass over
 * its weights; the per-slot partial sums of a row tile meet in the shared
 * memory of the CTA that takes all of that tile's work groups when they fit
 * there, else they go through the library's device workspace slot of the
 * calling stream (T*topk*N <= 4 Mi floats, counters re-armed by the call
 * itself); either way the sum runs in slot order.  A bad id sets MX_DEVERR_BAD_EXPERT and makes that token's
 * outputs NaN.  When K is not a multiple of 128, or the staged rows of h do
 * not fit beside the streaming kernel's weight ring, the per-slot products
 * come from the direct-load MoE kernel, then the router combine (two
 * launches).
 * h, out, codes, scales 16-byte aligned,
 * ids and r 4-byte aligned.  Calls on one stream run in order; calls on
 * different streams use different workspace slots. */
int mx_moe_down_combine(int fmt, const void *expert_codes, const void *expert_scales, const void *h,
                        const int32_t *expert_ids, const float *router_weights, float *out, int T, int E,
                        int topk, int N, int K);

/* Prefill GEMM over the same weights (release post, section "Decoding
 * block-float formats in software": dequantise on the GPU and multiply on
 * matrix units):
 *   Y[m][n] = bf16_rne( sum_k X[m][k] * W[n][k] ),  fp32 accumulation.
 * X bf16 [M][K], Y bf16 [M][N].  The weight tile is decoded exactly to bf16
 * in shared memory and multiplied by tcgen05 tensor-core MMA with the
 * accumulator in tensor memory.  Any M >= 1 and N >= 1 (a last column tile
 * that N only partly covers is masked); K a multiple of 32 (the TMA loads
 * need code rows a multiple of 16 bytes apart: NVFP4 with K % 32 == 16 gives
 * MX_EUNSUPPORTED); the NVFP4 tensor scale is applied in the epilogue. */
int mx_qmm(int fmt, const void *codes, const void *scales, const void *X, void *Y, int M, int N,
           int K);

/* Prefill GEMM over block-float activations on the block-scaled tensor
 * cores (manual page "Building from source", CUDA build options: on
 * Blackwell, block-float quantisation runs on the hardware NVFP4 / MXFP4
 * converter; talk slide 8 "ROCm on RDNA 3.5 vs. Metal vs. CUDA": FP4 on
 * Blackwell tensor cores):
 *   Y[m][n] = bf16_rne( sum_k Xq[m][k] * W[n][k] ),  fp32 accumulation,
 * where Xq is the block-float activation given by xcodes / xscales in the
 * weights' format and layout ([M][K] codes, [M][K/block] scales, NVFP4: the
 * fp32 tensor scale after the M*K/16 scale bytes; e.g. mx_quantize's
 * output).  Nothing is decoded: tcgen05.mma kind::mxf8f6f4 (MXFP8),
 * kind::mxf4 (MXFP4) or kind::mxf4nvf4 with 16-element blocks (NVFP4)
 * multiplies the codes and applies both operands' block scales; the NVFP4
 * tensor scales multiply the fp32 sum.  NVFP4 block scales are read as
 * unsigned E4M3 (mx_quantize never writes a negative one).  Any M >= 1; N a
 * multiple of 128 and K of 512 (MXFP4, MXFP8: scale rows a multiple of 16
 * bytes) or 256 (NVFP4), else MX_EUNSUPPORTED.  All pointers 16-byte aligned.  A pipeline wait that
 * times out sets MX_DEVERR_TIMEOUT and makes that output tile NaN. */
int mx_qmm_qx(int fmt, const void *codes, const void *scales, const void *xcodes, const void *xscales, void *Y,
              int M, int N, int K);

/* Expert-batched MoE prefill (grouped GEMM): the mx_moe_qmv operation for
 * many tokens, on the tensor cores.
 *   y[t][j][n] = bf16_rne( sum_k x[t][k] * W_e[n][k] ),  e = expert_ids[t][j],
 * x bf16 [T][K], y bf16 [T][topk][N], expert stacks as in mx_moe_qmv.  The
 * pages read only the experts a token is routed to (talk slide 4) and name
 * MoE prefill as the weak spot once dense prefill runs on the matrix units
 * (release post, section "Bandwidth utilisation per model"); here the
 * (token, slot) rows are grouped by expert on the device, gathered into
 * expert order and multiplied in tiles of up to 512 rows as in mx_qmm, so
 * each expert's weights are decoded once per 512 routed rows.  Launches: for
 * up to 256 experts, per-chunk row counts, one scan block (the group tile
 * table) and the placement of each row with the gather of its x row; for
 * more experts, one routing block and the gather; then the grouped GEMM.
 * workspace: caller-owned device memory of at least
 * mx_moe_qmm_workspace_size(T, E, topk, K) bytes, 256-byte aligned (else
 * MX_EINVAL / MX_EALIGN); the call overwrites it, so calls sharing one
 * workspace must not overlap.  Any N; K a multiple of 32 (as mx_qmm), T*topk
 * <= 2^24, E <= 4096, E*N < 2^31 (else MX_EUNSUPPORTED).  An id outside [0, E)
 * sets MX_DEVERR_BAD_EXPERT and fills that slot's N outputs with NaN.
 * codes, scales, x, y 16-byte aligned; ids 4-byte aligned.  For a down
 * projection pass T' = T*topk rows, topk = 1. */
size_t mx_moe_qmm_workspace_size(int T, int E, int topk, int K);
int mx_moe_qmm(int fmt, const void *expert_codes, const void *expert_scales, const void *x,
               const int32_t *expert_ids, void *y, int T, int E, int topk, int N, int K, void *workspace,
               size_t workspace_bytes);

/* Expert-batched MoE FFN prefill, one call:
 *   h[t][j]  = bf16_rne( silu(W_gu,e[0:I] x[t]) * (W_gu,e[I:2I] x[t]) )   (as mx_moe_gate_up_swiglu,
 *              with the fast exponent and division: within one bf16 unit of it)
 *   yd[t][j] = bf16_rne( W_dn,e h[t][j] )
 *   out[t][n] = sum_j r[t][j] * yd[t][j][n]  (fp32 fused multiply-adds in slot order)
 * e = expert_ids[t][j]; gate-up stacks [E][2I][H], down stacks [E][H][I];
 * x bf16 [T][H]; r fp32 [T][topk]; out fp32 [T][H].  Launches: routing and
 * gather (as mx_moe_qmm), grouped gate-up GEMM with the SwiGLU in its epilogue (CTA pairs
 * whose two halves hold gate row i and up row I + i), grouped down GEMM,
 * combine.  workspace: at least mx_moe_ffn_prefill_workspace_size(T, E,
 * topk, H, I) bytes, 256-byte aligned.  H and I multiples of 32 (each is the
 * K of one of the GEMMs); other limits as mx_moe_qmm.  A bad id sets MX_DEVERR_BAD_EXPERT and makes that
 * token's outputs NaN.  Pointers 16-byte aligned; ids and r 4-byte. */
size_t mx_moe_ffn_prefill_workspace_size(int T, int E, int topk, int H, int I);
int mx_moe_ffn_prefill(int fmt, const void *gate_up_codes, const void *gate_up_scales, const void *down_codes,
                       const void *down_scales, const void *x, const int32_t *expert_ids,
                       const float *router_weights, float *out, int T, int E, int topk, int H, int I,
                       void *workspace, size_t workspace_bytes);

/* On-device block-float quantisation of bf16 activations, the reverse of the
 * decode (manual page "Building from source", CUDA build options: on
 * Blackwell, block-float quantisation runs on the hardware NVFP4 / MXFP4
 * converter; ROCm status table: FP8 block checkpoints are re-quantised to
 * MXFP8).  x bf16 [M][K] in; codes and scales out in the layouts above
 * (NVFP4: the fp32 tensor scale is written after the M*K/16 scale bytes).
 *   MXFP4 / MXFP8 (OCP MX v1.0 conversion): per 32 elements the scale is
 *     2^e, e = floor(log2(max |x|)) - emax (2 for E2M1, 8 for E4M3), at
 *     least -127; each element x / 2^e rounded to nearest-even in the
 *     element format, saturating at its largest finite value.
 *   NVFP4: g = fp32(G / 2688), G the largest finite |x| of the whole tensor
 *     (1 when G = 0); per 16 elements s = E4M3(fp32(max |x| / fp32(6 g)))
 *     and each element fp32(x / fp32(s g)) rounded to E2M1 (zero codes when
 *     s g = 0).  Two launches (tensor maximum, then the blocks); the
 *     maximum goes through a word of the calling stream's workspace slot.
 *   A block holding a NaN or an infinity gets a NaN scale (0xFF / 0x7F) and
 *   zero codes; a zero result is stored as +0.
 * K a multiple of the block (else MX_EINVAL); x and codes 16-byte aligned. */
int mx_quantize(int fmt, const void *x, void *codes, void *scales, int M, int K);

/* ---- support calls (not on the pages; part of this library's contract) */

/* Stream for subsequent calls from this host thread (a cudaStream_t; NULL =
 * the legacy default stream). */
int mx_set_stream(void *cuda_stream);

/* Bit-exact dequantisation W[n][k] = fp32(code * scale) (NVFP4: then one
 * round-to-nearest-even multiply by the fp32 tensor scale), W fp32 [N][K].
 * Exposes the kernels' decode for exactness tests. */
int mx_dequant(int fmt, const void *codes, const void *scales, float *W, int N, int K);

/* MoE FFN glue used between the two projections:
 *   h[q][i] = bf16_rne( silu(gu[q][i]) * gu[q][I + i] ),  silu(v) = v / (1 + e^-v),
 * gu fp32 [Q][2I] (gate rows then up rows), h bf16 [Q][I].  Evaluated in
 * fp32 as v * sigmoid(v) with the sigmoid formed from e^-|v|, so it never
 * overflows. */
int mx_swiglu(const float *gu, void *h, int Q, int I);

/* Router-weighted combine: out[t][n] = sum_j r[t][j] * yd[t*topk + j][n],
 * yd fp32 [T*topk][N], r fp32 [T][topk], out fp32 [T][N]. */
int mx_moe_combine(const float *yd, const float *r, float *out, int T, int topk, int N);

/* Decode GEMV for callers that cannot allocate device memory.  Same
 * operation, arguments, layouts and errors as mx_qmv, which cudaMalloc's a
 * 16 MiB workspace slot on the first call on a stream whose shape splits K
 * across CTAs; some callers cannot allow
 * that (an engine whose own allocator already owns the whole device pool, or
 * a latency-critical decode loop that cannot take the device
 * synchronisation of a first-call allocation).  This variant allocates
 * nothing: its split-K workspace is a fixed ~1 MiB array inside the library
 * image (262,144 fp32 partial sums plus 4,096 counters), held by every GPU
 * that loads the library until the process exits.  A group of 8 tokens whose
 * workspace would not fit (many tokens times large N with K split into
 * windows) runs on the slower direct-load kernel, which needs none, or, when
 * its rows are too long for that kernel's staging, as two smaller groups
 * (each needing less workspace), so every shape mx_qmv takes is served.  The first call on a device looks up the array's
 * device address and the device attributes; make that first call before any
 * stream capture.  Every call shares the one array, so two calls that
 * overlap on the GPU (for example on two streams) race; each call clears
 * the counters it uses before launching.  No counterpart on the pages: this
 * is an interface variant of mx_qmv, not a different computation. */
int mx_qmv_noalloc(int fmt, const void *codes, const void *scales, const void *x, float *y, int M, int N,
                   int K);

/* Measurement support: the dense rate of this GPU's tensor pipe for one MMA
 * kind, the denominator of the prefill GEMMs' roofline.  One CTA per SM
 * issues iters x 4 tcgen05.mma of 128 x 256 x K (cta_group::1) on
 * shared-memory operands into tensor memory; *ms receives the elapsed time
 * (CUDA events on the calling thread's stream).  kind: 0 bf16 (kind::f16,
 * K = 16), 1 E4M3 (kind::f8f6f4, K = 32), 2 MXFP8 (kind::mxf8f6f4
 * block-scaled, K = 32), 3 MXFP4 (kind::mxf4, K = 64), 4 NVFP4
 * (kind::mxf4nvf4, 16-element blocks, K = 64); the operands are zeros,
 * or, with MX_PEAK_FILLED added to kind, hashed bits kept finite (bf16 below
 * 1 in magnitude, E4M3 without the NaN code, any FP4 code) with unit block
 * scales.  Added flags probe what a GEMM's pipeline adds: MX_PEAK_ROTATE
 * rotates the MMAs through four 48 KB operand stages (three with
 * MX_PEAK_SMEM_STORES); MX_PEAK_SMEM_STORES has three other warps store
 * 16-byte vectors into the fourth stage at full rate meanwhile, and
 * MX_PEAK_TMEM_STORES has them store into unused tensor-memory columns
 * instead.  FLOPs of a call: 2 * 128 * 256 * K * 4 * iters * (number of
 * SMs).  MX_EINVAL for another kind.  Synchronises the stream. */
#define MX_PEAK_FILLED 0x100
#define MX_PEAK_ROTATE 0x200
#define MX_PEAK_SMEM_STORES 0x400
#define MX_PEAK_TMEM_STORES 0x800
int mx_mma_peak(int kind, int iters, float *ms);

/* Test hook for the bounded waits of the tensor-core kernels (mx_qmm,
 * mx_moe_qmm, mx_moe_ffn_prefill); the pages' fault handling (talk slide 10
 * "70 Fixes to the ROCm Fork", GPU fault handling: waits that used to block
 * forever after a fault now give up and report it).  With stall != 0, every
 * later launch of those kernels from this process issues none of its
 * activation loads, so the MMA issuer's first wait can only end by timing
 * out: the pair then writes NaN to its output tile, sets MX_DEVERR_TIMEOUT
 * and returns with nothing in flight.  wait_ns is the limit of a pipeline
 * wait (0: the default of 2 s); waits for copies already in flight keep the
 * 2 s limit.  mx_debug_qmm_stall(0, 0) restores normal operation.  For
 * tests only: not to be used while other threads launch those kernels. */
int mx_debug_qmm_stall(int stall, unsigned long long wait_ns);

/* Synchronise the calling thread's stream, then return the device error
 * word of the current device (0 = none; MX_DEVERR_* bits) and clear it.
 * Returns MX_ECUDA if the synchronisation fails. */
int mx_device_error(void);

/* Static description of a status code. */
const char *mx_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* MX_H */
