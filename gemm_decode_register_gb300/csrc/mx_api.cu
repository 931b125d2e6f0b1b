// mx_api.cu -- the C ABI declared in include/mx.h: argument validation,
// per-thread stream, per-device state, per-stream workspace slots and the
// device error word.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "../../include/mx.h"
#include "mx_internal.h"

namespace mx {

static thread_local cudaStream_t t_stream = nullptr;
static std::mutex g_mu;
static DeviceState g_dev[64];

// The device error word: a module variable, so it exists (zeroed) on every
// device the library is loaded on and needs no allocation.  [0] is the word;
// the rest pads it to a sector of its own.
static __device__ __align__(256) int g_err_word[64];

cudaStream_t current_stream() { return t_stream; }

DeviceState *device_state()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &ds = g_dev[dev];
    if (ds.device == dev) return &ds;
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return nullptr;
    void *err = nullptr;
    if (cudaGetSymbolAddress(&err, g_err_word) != cudaSuccess || err == nullptr) return nullptr;
    ds.num_sms = sms;
    ds.max_smem_optin = smem;
    ds.err = static_cast<int *>(err);
    ds.device = dev;
    return &ds;
}

// ---- per-stream workspace slots
//
// Calls whose kernels pass partial sums through global memory (mx_qmv with K
// split across CTAs, mx_moe_down_combine, NVFP4 mx_quantize) each use the
// slot of the stream they are issued on, so calls on different streams never
// share one.  A slot is made on the first such call on a stream and kept
// until the process exits.  The per-thread default stream is one stream per
// host thread, so its slots are also keyed by the thread.
namespace {

struct StreamSlot {
    cudaStream_t stream;
    std::thread::id thread;  // only for cudaStreamPerThread
    char *mem;
};

struct DeviceSlots {
    std::vector<StreamSlot> slots;
    cudaStream_t zero_stream = nullptr;  // private stream that clears new slots
};

DeviceSlots g_slots[64];

// Restores the calling thread's stream-capture mode on scope exit.
struct RelaxedCapture {
    cudaStreamCaptureMode prev = cudaStreamCaptureModeRelaxed;
    RelaxedCapture() { cudaThreadExchangeStreamCaptureMode(&prev); }
    ~RelaxedCapture() { cudaThreadExchangeStreamCaptureMode(&prev); }
};

char *new_slot(DeviceSlots &d)
{
    // cudaMalloc is not a stream operation: in relaxed mode it is allowed
    // while a stream of this thread is being captured, and the memory is not
    // part of the graph.  The slot is cleared on a private stream and waited
    // for here, so the clearing is neither captured nor ordered against the
    // caller's streams.
    RelaxedCapture relaxed;
    if (d.zero_stream == nullptr && cudaStreamCreateWithFlags(&d.zero_stream, cudaStreamNonBlocking) != cudaSuccess)
        return nullptr;
    void *p = nullptr;
    if (cudaMalloc(&p, SLOT_BYTES) != cudaSuccess) return nullptr;
    if (cudaMemsetAsync(p, 0, SLOT_BYTES, d.zero_stream) != cudaSuccess ||
        cudaStreamSynchronize(d.zero_stream) != cudaSuccess) {
        cudaFree(p);
        return nullptr;
    }
    return static_cast<char *>(p);
}

}  // namespace

bool attach_stream_workspace(DeviceState &v, cudaStream_t st)
{
    if (v.device < 0 || v.device >= 64) return false;
    const std::thread::id tid = st == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id();
    char *mem = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DeviceSlots &d = g_slots[v.device];
        for (const StreamSlot &s : d.slots)
            if (s.stream == st && s.thread == tid) {
                mem = s.mem;
                break;
            }
        if (mem == nullptr) {
            mem = new_slot(d);
            if (mem == nullptr) return false;
            d.slots.push_back(StreamSlot{st, tid, mem});
        }
    }
    v.amax = reinterpret_cast<unsigned *>(mem);
    v.ws = reinterpret_cast<float *>(mem + 256);
    v.ws_count = reinterpret_cast<int *>(v.ws + WS_FLOATS);
    v.ws_floats = WS_FLOATS;
    v.ws_counters = WS_COUNTERS;
    return true;
}

}  // namespace mx

using namespace mx;

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static int block_of(int fmt) { return fmt == MX_FMT_NVFP4 ? 16 : 32; }
static bool fmt_ok(int fmt) { return fmt == MX_FMT_MXFP4 || fmt == MX_FMT_MXFP8 || fmt == MX_FMT_NVFP4; }

static int finish(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ECUDA; }

extern "C" int mx_set_stream(void *cuda_stream)
{
    t_stream = static_cast<cudaStream_t>(cuda_stream);
    return MX_OK;
}

extern "C" int mx_qmv(int fmt, const void *codes, const void *scales, const void *x, float *y, int M,
                      int N, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!codes || !scales || !x || !y) return MX_EINVAL;
    if (M <= 0 || N <= 0 || K <= 0 || K % block_of(fmt) != 0) return MX_EINVAL;
    if (K > QMV_MAX_K) return MX_EUNSUPPORTED;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(y)) return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    // a workspace slot only for shapes that split K across CTAs
    DeviceState v = *ds;
    v.ws_floats = WS_FLOATS;
    v.ws_counters = WS_COUNTERS;
    const QmvScratchNeed need = qmv_scratch_need(v, fmt, M, N, K);
    if ((need.floats > 0 || need.counters > 0) && !attach_stream_workspace(v, t_stream)) return MX_ECUDA;
    cudaError_t e = launch_qmv(v, t_stream, fmt, static_cast<const uint8_t *>(codes),
                               static_cast<const uint8_t *>(scales), static_cast<const uint16_t *>(x), y,
                               M, N, K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

extern "C" int mx_moe_qmv(int fmt, const void *expert_codes, const void *expert_scales, const void *x,
                          const int32_t *expert_ids, float *y, int T, int E, int topk, int N, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!expert_codes || !expert_scales || !x || !expert_ids || !y) return MX_EINVAL;
    if (T <= 0 || E <= 0 || topk <= 0 || N <= 0 || K <= 0 || topk > E || K % block_of(fmt) != 0)
        return MX_EINVAL;
    if ((long long)T * topk > MOE_MAX_SLOTS || E > MOE_MAX_EXPERTS || K > QMV_MAX_K)
        return MX_EUNSUPPORTED;
    if (!aligned16(expert_codes) || !aligned16(expert_scales) || !aligned16(x) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u))
        return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    cudaError_t e = launch_moe_qmv(*ds, t_stream, fmt, static_cast<const uint8_t *>(expert_codes),
                                   static_cast<const uint8_t *>(expert_scales),
                                   static_cast<const uint16_t *>(x), expert_ids, y, T, E, topk, N, K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

extern "C" int mx_moe_gate_up_swiglu(int fmt, const void *expert_codes, const void *expert_scales, const void *x,
                                     const int32_t *expert_ids, void *h, int T, int E, int topk, int I, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!expert_codes || !expert_scales || !x || !expert_ids || !h) return MX_EINVAL;
    if (T <= 0 || E <= 0 || topk <= 0 || I <= 0 || K <= 0 || topk > E || K % block_of(fmt) != 0)
        return MX_EINVAL;
    if ((long long)T * topk > MOE_MAX_SLOTS || E > MOE_MAX_EXPERTS || K > QMV_MAX_K) return MX_EUNSUPPORTED;
    if (!aligned16(expert_codes) || !aligned16(expert_scales) || !aligned16(x) || !aligned16(h) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u))
        return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    DeviceState v = *ds;  // rows the streaming kernel cannot take: gate/up products pass through the workspace
    if (!attach_stream_workspace(v, t_stream)) return MX_ECUDA;
    cudaError_t e = launch_moe_gate_up_swiglu(v, t_stream, fmt, static_cast<const uint8_t *>(expert_codes),
                                              static_cast<const uint8_t *>(expert_scales),
                                              static_cast<const uint16_t *>(x), expert_ids,
                                              static_cast<uint16_t *>(h), T, E, topk, I, K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

extern "C" int mx_moe_down_combine(int fmt, const void *expert_codes, const void *expert_scales, const void *h,
                                   const int32_t *expert_ids, const float *router_weights, float *out, int T,
                                   int E, int topk, int N, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!expert_codes || !expert_scales || !h || !expert_ids || !router_weights || !out) return MX_EINVAL;
    if (T <= 0 || E <= 0 || topk <= 0 || N <= 0 || K <= 0 || topk > E || K % block_of(fmt) != 0)
        return MX_EINVAL;
    if ((long long)T * topk > MOE_MAX_SLOTS || E > MOE_MAX_EXPERTS || K > QMV_MAX_K) return MX_EUNSUPPORTED;
    if (!aligned16(expert_codes) || !aligned16(expert_scales) || !aligned16(h) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u) || (reinterpret_cast<uintptr_t>(router_weights) & 3u))
        return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    DeviceState v = *ds;
    if (!attach_stream_workspace(v, t_stream)) return MX_ECUDA;
    cudaError_t e = launch_moe_down_combine(v, t_stream, fmt, static_cast<const uint8_t *>(expert_codes),
                                            static_cast<const uint8_t *>(expert_scales),
                                            static_cast<const uint16_t *>(h), expert_ids, router_weights, out, T,
                                            E, topk, N, K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

extern "C" int mx_qmm(int fmt, const void *codes, const void *scales, const void *X, void *Y, int M,
                      int N, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!codes || !scales || !X || !Y) return MX_EINVAL;
    if (M <= 0 || N <= 0 || K <= 0 || K % block_of(fmt) != 0) return MX_EINVAL;
    if (!qmm_shape_ok(fmt, K)) return MX_EUNSUPPORTED;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(X) || !aligned16(Y)) return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    cudaError_t e = launch_qmm(*ds, t_stream, fmt, static_cast<const uint8_t *>(codes),
                               static_cast<const uint8_t *>(scales), static_cast<const uint16_t *>(X),
                               static_cast<uint16_t *>(Y), M, N, K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

// Expert-batched prefill: limits beyond mx_moe_qmv's.
static constexpr long long PREFILL_MAX_SLOTS = 1ll << 24;  // T * topk

static bool prefill_sizes_ok(long long T, long long E, long long topk)
{
    return T * topk <= PREFILL_MAX_SLOTS && E <= MOE_MAX_EXPERTS;
}

extern "C" size_t mx_moe_qmm_workspace_size(int T, int E, int topk, int K)
{
    if (T <= 0 || E <= 0 || topk <= 0 || K <= 0 || topk > E || !prefill_sizes_ok(T, E, topk)) return 0;
    return moe_group_plan(T, E, topk, K, 0).bytes;
}

extern "C" int mx_moe_qmm(int fmt, const void *expert_codes, const void *expert_scales, const void *x,
                          const int32_t *expert_ids, void *y, int T, int E, int topk, int N, int K, void *workspace,
                          size_t workspace_bytes)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!expert_codes || !expert_scales || !x || !expert_ids || !y || !workspace) return MX_EINVAL;
    if (T <= 0 || E <= 0 || topk <= 0 || N <= 0 || K <= 0 || topk > E || K % block_of(fmt) != 0)
        return MX_EINVAL;
    if (!qmm_shape_ok(fmt, K) || !prefill_sizes_ok(T, E, topk) || (long long)E * N > 0x7FFFFFFFll)
        return MX_EUNSUPPORTED;
    if (workspace_bytes < moe_group_plan(T, E, topk, K, 0).bytes) return MX_EINVAL;
    if (!aligned16(expert_codes) || !aligned16(expert_scales) || !aligned16(x) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    cudaError_t e = launch_moe_qmm(*ds, t_stream, fmt, static_cast<const uint8_t *>(expert_codes),
                                   static_cast<const uint8_t *>(expert_scales), static_cast<const uint16_t *>(x),
                                   expert_ids, static_cast<uint16_t *>(y), T, E, topk, N, K, workspace);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

extern "C" size_t mx_moe_ffn_prefill_workspace_size(int T, int E, int topk, int H, int I)
{
    if (T <= 0 || E <= 0 || topk <= 0 || H <= 0 || I <= 0 || topk > E || !prefill_sizes_ok(T, E, topk)) return 0;
    return moe_group_plan(T, E, topk, H, I).bytes;
}

extern "C" int mx_moe_ffn_prefill(int fmt, const void *gate_up_codes, const void *gate_up_scales,
                                  const void *down_codes, const void *down_scales, const void *x,
                                  const int32_t *expert_ids, const float *router_weights, float *out, int T, int E,
                                  int topk, int H, int I, void *workspace, size_t workspace_bytes)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!gate_up_codes || !gate_up_scales || !down_codes || !down_scales || !x || !expert_ids || !router_weights ||
        !out || !workspace)
        return MX_EINVAL;
    if (T <= 0 || E <= 0 || topk <= 0 || H <= 0 || I <= 0 || topk > E || H % block_of(fmt) != 0 ||
        I % block_of(fmt) != 0)
        return MX_EINVAL;
    if (!qmm_shape_ok(fmt, H) || !qmm_shape_ok(fmt, I) || !prefill_sizes_ok(T, E, topk) ||
        (long long)E * 2 * I > 0x7FFFFFFFll ||
        (long long)E * H > 0x7FFFFFFFll)
        return MX_EUNSUPPORTED;
    if (workspace_bytes < moe_group_plan(T, E, topk, H, I).bytes) return MX_EINVAL;
    if (!aligned16(gate_up_codes) || !aligned16(gate_up_scales) || !aligned16(down_codes) ||
        !aligned16(down_scales) || !aligned16(x) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u) || (reinterpret_cast<uintptr_t>(router_weights) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    cudaError_t e = launch_moe_ffn_prefill(
        *ds, t_stream, fmt, static_cast<const uint8_t *>(gate_up_codes), static_cast<const uint8_t *>(gate_up_scales),
        static_cast<const uint8_t *>(down_codes), static_cast<const uint8_t *>(down_scales),
        static_cast<const uint16_t *>(x), expert_ids, router_weights, out, T, E, topk, H, I, workspace);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return finish(e);
}

namespace mx {
// mx_quant.cu
cudaError_t launch_quantize(const DeviceState &ds, cudaStream_t st, int fmt, const uint16_t *x, uint8_t *codes,
                            uint8_t *scales, int M, int K);
}  // namespace mx

extern "C" int mx_quantize(int fmt, const void *x, void *codes, void *scales, int M, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!x || !codes || !scales) return MX_EINVAL;
    if (M <= 0 || K <= 0 || K % block_of(fmt) != 0) return MX_EINVAL;
    if (!aligned16(x) || !aligned16(codes)) return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    DeviceState v = *ds;
    if (fmt == MX_FMT_NVFP4 && !attach_stream_workspace(v, t_stream)) return MX_ECUDA;
    return finish(launch_quantize(v, t_stream, fmt, static_cast<const uint16_t *>(x), static_cast<uint8_t *>(codes),
                                  static_cast<uint8_t *>(scales), M, K));
}

extern "C" int mx_dequant(int fmt, const void *codes, const void *scales, float *W, int N, int K)
{
    if (!fmt_ok(fmt)) return MX_EUNSUPPORTED;
    if (!codes || !scales || !W) return MX_EINVAL;
    if (N <= 0 || K <= 0 || K % block_of(fmt) != 0) return MX_EINVAL;
    if (!aligned16(codes) || !aligned16(W)) return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    return finish(launch_dequant(*ds, t_stream, fmt, static_cast<const uint8_t *>(codes),
                                 static_cast<const uint8_t *>(scales), W, N, K));
}

extern "C" int mx_swiglu(const float *gu, void *h, int Q, int I)
{
    if (!gu || !h) return MX_EINVAL;
    if (Q <= 0 || I <= 0) return MX_EINVAL;
    if ((reinterpret_cast<uintptr_t>(gu) & 3u) || (reinterpret_cast<uintptr_t>(h) & 1u)) return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    return finish(launch_swiglu(*ds, t_stream, gu, static_cast<uint16_t *>(h), Q, I));
}

extern "C" int mx_moe_combine(const float *yd, const float *r, float *out, int T, int topk, int N)
{
    if (!yd || !r || !out) return MX_EINVAL;
    if (T <= 0 || topk <= 0 || N <= 0) return MX_EINVAL;
    if ((reinterpret_cast<uintptr_t>(yd) & 3u) || (reinterpret_cast<uintptr_t>(r) & 3u) ||
        (reinterpret_cast<uintptr_t>(out) & 3u))
        return MX_EALIGN;
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    return finish(launch_moe_combine(*ds, t_stream, yd, r, out, T, topk, N));
}

extern "C" int mx_debug_qmm_stall(int stall, unsigned long long wait_ns)
{
    set_qmm_stall(stall, wait_ns);
    return MX_OK;
}

extern "C" int mx_device_error(void)
{
    DeviceState *ds = device_state();
    if (!ds) return MX_ECUDA;
    int word = 0;
    if (cudaMemcpyAsync(&word, ds->err, sizeof word, cudaMemcpyDeviceToHost, t_stream) != cudaSuccess ||
        cudaStreamSynchronize(t_stream) != cudaSuccess)
        return MX_ECUDA;
    if (word && (cudaMemsetAsync(ds->err, 0, sizeof word, t_stream) != cudaSuccess ||
                 cudaStreamSynchronize(t_stream) != cudaSuccess))
        return MX_ECUDA;
    return word;
}

extern "C" const char *mx_strerror(int status)
{
    switch (status) {
    case MX_OK: return "ok";
    case MX_EINVAL: return "invalid argument (null pointer, size <= 0, or K not a multiple of the block)";
    case MX_EUNSUPPORTED: return "unsupported format or size";
    case MX_EALIGN: return "pointer not 16-byte aligned";
    case MX_ECUDA: return "CUDA runtime error";
    case MX_EDEVICE: return "device-side check fired";
    default: return "unknown status";
    }
}
