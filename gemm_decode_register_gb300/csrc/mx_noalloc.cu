// mx_noalloc.cu -- mx_qmv_noalloc: the decode GEMV for callers that must
// not allocate device memory.
//
// mx_qmv takes its split-K workspace from a 16 MiB slot it cudaMalloc's on
// the first call on a stream that needs one.  Some callers cannot allow
// that: a serving engine that has already handed the whole device pool to
// its own allocator (a cudaMalloc there fails or breaks its accounting), or
// a latency-critical decode loop where the implicit device synchronisation
// of a first-call cudaMalloc is not acceptable.  This entry point runs the
// same kernels but keeps the workspace in the file-scope array below, which
// is part of the library image: every GPU that loads the library holds it
// (about 1 MiB) until the process exits, and no call allocates.
#include <mutex>

#include "../../include/mx.h"
#include "mx_internal.h"

namespace mx {

// Window partial sums, then the arrival counters.
constexpr size_t NA_FLOATS = (size_t)1 << 18;  // 1 MiB of fp32 partials
constexpr int NA_COUNTERS = WS_COUNTERS;
constexpr size_t NA_BYTES = NA_FLOATS * 4 + (size_t)NA_COUNTERS * 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_BYTES];

namespace {

struct NoAllocDevice {
    bool ready = false;
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_na_mu;
NoAllocDevice g_na[64];

// Set-up on the first call on a device (that device current): device
// attributes and the device address of the scratch array.  In host code the
// array's name is only a host-side handle, so the address must come from
// cudaGetSymbolAddress.
const NoAllocDevice *noalloc_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_na_mu);
    NoAllocDevice &d = g_na[dev];
    if (d.ready) return &d;
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return nullptr;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    d.device = dev;
    d.num_sms = sms;
    d.max_smem_optin = smem;
    d.scratch = static_cast<unsigned char *>(p);
    d.ready = true;
    return &d;
}

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" int mx_qmv_noalloc(int fmt, const void *codes, const void *scales, const void *x, float *y, int M,
                              int N, int K)
{
    if (fmt != MX_FMT_MXFP4 && fmt != MX_FMT_MXFP8 && fmt != MX_FMT_NVFP4) return MX_EUNSUPPORTED;
    if (!codes || !scales || !x || !y) return MX_EINVAL;
    if (M <= 0 || N <= 0 || K <= 0 || K % (fmt == MX_FMT_NVFP4 ? 16 : 32) != 0) return MX_EINVAL;
    if (K > QMV_MAX_K) return MX_EUNSUPPORTED;
    auto aligned16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(y)) return MX_EALIGN;
    const NoAllocDevice *d = noalloc_device();
    if (!d) return MX_ECUDA;
    DeviceState ds;  // a view of this device without the allocating per-device state
    ds.device = d->device;
    ds.num_sms = d->num_sms;
    ds.max_smem_optin = d->max_smem_optin;
    ds.err = nullptr;  // the qmv kernels never write the error word
    ds.ws = reinterpret_cast<float *>(d->scratch);
    ds.ws_count = reinterpret_cast<int *>(d->scratch + NA_FLOATS * 4);
    ds.ws_floats = NA_FLOATS;
    ds.ws_counters = NA_COUNTERS;
    // A group of 8 tokens whose split-K partial sums would not fit the array
    // runs on the direct-load kernel instead, which needs no workspace; the
    // query reports what the groups that do use the array need.
    const QmvScratchNeed need = qmv_scratch_need(ds, fmt, M, N, K);
    cudaStream_t st = current_stream();
    // the array keeps the last call's contents: the arrival counters must
    // start at zero (a cleared range, not an allocation)
    if (need.counters > 0 &&
        cudaMemsetAsync(ds.ws_count, 0, sizeof(int) * (size_t)need.counters, st) != cudaSuccess)
        return MX_ECUDA;
    const cudaError_t e = launch_qmv(ds, st, fmt, static_cast<const uint8_t *>(codes),
                                     static_cast<const uint8_t *>(scales), static_cast<const uint16_t *>(x), y, M, N,
                                     K);
    if (e == cudaErrorInvalidValue) return MX_EUNSUPPORTED;
    return e == cudaSuccess ? MX_OK : MX_ECUDA;
}
