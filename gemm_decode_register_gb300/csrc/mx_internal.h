// mx_internal.h -- host-side declarations shared by the library's
// translation units (launchers, per-device state).  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mx {

// Per-device state, created on first use of a device, plus (in the copy a
// call works on) the workspace slot of the calling stream.
struct DeviceState {
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;    // bytes of dynamic shared memory a block may opt into
    int *err = nullptr;        // device error word (shared by every stream of the device)
    float *ws = nullptr;       // split-K / per-slot partial sums (ws_floats floats)
    int *ws_count = nullptr;   // arrival counters (ws_counters ints, kept at zero between calls)
    unsigned *amax = nullptr;  // NVFP4 quantiser: the tensor maximum's bits
    size_t ws_floats = 0;      // capacities: 0 = no workspace attached
    int ws_counters = 0;
};

// Workspace slot of one stream: NVFP4 tensor-maximum word (256 bytes), partial
// sums, arrival counters.
constexpr size_t WS_FLOATS = (size_t)4 << 20;  // 16 MiB
constexpr int WS_COUNTERS = 4096;
constexpr size_t SLOT_BYTES = 256 + WS_FLOATS * 4 + WS_COUNTERS * 4;

DeviceState *device_state();  // current device; nullptr on CUDA error
cudaStream_t current_stream();

// Point v's workspace at the slot of stream st (allocated, zeroed, on the
// first call that needs one on this stream; the calling thread is switched
// to relaxed capture mode for that, so a first call inside a stream capture
// works too).  false on a CUDA error.
bool attach_stream_workspace(DeviceState &v, cudaStream_t st);

// Launchers: validated arguments in, a CUDA error code out.  The plain
// launch_qmv / launch_moe_qmv pick the streaming kernels when the shape
// allows and fall back to the direct-load kernels otherwise.
cudaError_t launch_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K);
cudaError_t launch_moe_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, const uint16_t *x, const int32_t *ids, float *y,
                           int T, int E, int topk, int N, int K);
// Whether the direct-load kernel can stage a token's row of K elements.
bool qmv_direct_fits(const DeviceState &ds, int K);
cudaError_t launch_qmv_direct(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                              const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K);
cudaError_t launch_moe_qmv_direct(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                                  const uint8_t *scales, const uint16_t *x, const int32_t *ids, float *y,
                                  int T, int E, int topk, int N, int K);
cudaError_t launch_dequant(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, float *W, int N, int K);
cudaError_t launch_swiglu(const DeviceState &ds, cudaStream_t st, const float *gu, uint16_t *h,
                          int Q, int I);
cudaError_t launch_moe_combine(const DeviceState &ds, cudaStream_t st, const float *yd,
                               const float *r, float *out, int T, int topk, int N);
cudaError_t launch_moe_gate_up_swiglu(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                                      const uint8_t *scales, const uint16_t *x, const int32_t *ids, uint16_t *h,
                                      int T, int E, int topk, int I, int K);
cudaError_t launch_moe_down_combine(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                                    const uint8_t *scales, const uint16_t *h, const int32_t *ids, const float *rw,
                                    float *out, int T, int E, int topk, int N, int K);
cudaError_t launch_qmm(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *X, uint16_t *Y, int M, int N, int K);

// K the tensor-core GEMMs take (their TMA loads need rows 16-byte apart).
bool qmm_shape_ok(int fmt, int K);

// Grouped (expert-batched) prefill: routes on the device, gathers the
// routed rows into expert order and runs the pair GEMM per group tile.
// Y / h / per-slot outputs are bf16.
cudaError_t launch_qmm_grouped(const DeviceState &ds, cudaStream_t st, int fmt, bool swiglu, const uint8_t *codes,
                               const uint8_t *scales, const uint16_t *Xs, int rows, const int *groups,
                               int max_groups, const int *slot_of, uint16_t *Y, int E, int N, int K);

// Byte offsets of the grouped-prefill workspace (caller-owned, 256-byte aligned).
struct MoeGroupPlan {
    int S = 0;           // routed rows (T * topk)
    int max_groups = 0;  // most group tiles any routing can make
    size_t off_groups = 0, off_slot = 0, off_xs = 0, off_hs = 0, bytes = 0;
};
MoeGroupPlan moe_group_plan(int T, int E, int topk, int K, int I /* 0: no FFN */);
cudaError_t launch_moe_qmm(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, const uint16_t *x, const int32_t *ids, uint16_t *y, int T, int E,
                           int topk, int N, int K, void *workspace);
cudaError_t launch_moe_ffn_prefill(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *gu_codes,
                                   const uint8_t *gu_scales, const uint8_t *dn_codes, const uint8_t *dn_scales,
                                   const uint16_t *x, const int32_t *ids, const float *rw, float *out, int T, int E,
                                   int topk, int H, int I, void *workspace);

// Test hook of the tensor-core kernels' bounded waits (mx_debug_qmm_stall).
void set_qmm_stall(int stall_x, unsigned long long wait_ns);

// Limits checked on the host.
constexpr int QMV_MAX_K = 1 << 20;
constexpr int MOE_MAX_SLOTS = 1024;  // T * topk
constexpr int MOE_MAX_EXPERTS = 4096;

// Split-K workspace a launch_qmv call would use (0 when it needs none).
struct QmvScratchNeed {
    size_t floats = 0;  // window partial sums
    int counters = 0;   // arrival counters, zero before the launch
};
QmvScratchNeed qmv_scratch_need(const DeviceState &ds, int fmt, int M, int N, int K);

// Shared-memory bytes the qmv kernel needs to stage `rows` activation rows
// of length K (f16, padded), or -1 if that cannot fit.
int qmv_stage_bytes(int rows, int K);

}  // namespace mx
