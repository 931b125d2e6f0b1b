// mx_internal.h -- host-side declarations shared by the library's
// translation units (launchers, per-device state).  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mx {

// Per-device state, created on first use of a device.
struct DeviceState {
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;  // bytes of dynamic shared memory a block may opt into
    int *err = nullptr;      // device error word (first int of the scratch block)
    float *ws = nullptr;     // split-K partial sums (WS_FLOATS floats)
    int *ws_count = nullptr; // split-K arrival counters (WS_COUNTERS ints, kept at zero between calls)
};

// Device scratch: error word (256 bytes), split-K partials, counters.
constexpr size_t WS_FLOATS = (size_t)4 << 20;  // 16 MiB
constexpr int WS_COUNTERS = 4096;
constexpr size_t SCRATCH_BYTES = 256 + WS_FLOATS * 4 + WS_COUNTERS * 4;

DeviceState *device_state();  // current device; nullptr on CUDA error
cudaStream_t current_stream();

// Launchers: validated arguments in, a CUDA error code out.  The plain
// launch_qmv / launch_moe_qmv pick the streaming kernels when the shape
// allows and fall back to the direct-load kernels otherwise.
cudaError_t launch_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                       const uint8_t *scales, const uint16_t *x, float *y, int M, int N, int K);
cudaError_t launch_moe_qmv(const DeviceState &ds, cudaStream_t st, int fmt, const uint8_t *codes,
                           const uint8_t *scales, const uint16_t *x, const int32_t *ids, float *y,
                           int T, int E, int topk, int N, int K);
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
