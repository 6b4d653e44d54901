// launch.h -- host-side declarations shared by the C-ABI layer and the kernel
// translation units (launchers, workspace layout, device status).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fmca {

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout (both paths):
//   [0, align256(B*G*s*e*4))          per-chunk states, fp32 [B][G][s][e]
//   [that, + B*Gp*s*e*4)              state prefix sums / n, Gp = G (causal)
//                                     or 1 (bidirectional); fp32 on the SIMT
//                                     path, bf16 on the tensor-core path
inline size_t workspace_bytes(int B, int n, int s, int e, int C, int causal) {
  const size_t G = (size_t)(n / C);
  const size_t se = (size_t)s * (size_t)e;
  const size_t Gp = causal ? G : 1;
  return align256(sizeof(float) * (size_t)B * G * se) +
         align256(sizeof(float) * (size_t)B * Gp * se);
}

// Both return 0 on success, nonzero when a launch failed.
// `events` (may be NULL) holds launch-count + 1 cudaEvent_t handles recorded
// before the first kernel and after each kernel.
int launch_simt_forward(const void *Z, const void *V, const void *U, const float *gamma,
                        const float *beta, void *O, int B, int n, int s, int e, int C,
                        int causal, int dtype_bf16, void *workspace, cudaStream_t stream,
                        cudaEvent_t const *events = nullptr);

int launch_tc_forward(const void *Z, const void *V, const void *U, const float *gamma,
                      const float *beta, void *O, int B, int n, int s, int e, int C, int causal,
                      void *workspace, cudaStream_t stream, cudaEvent_t const *events = nullptr);

inline bool record_event(cudaEvent_t const *events, int i, cudaStream_t stream) {
  return events == nullptr || cudaEventRecord(events[i], stream) == cudaSuccess;
}

// Shapes the tensor-core path covers.
bool tc_supported(int B, int n, int s, int e, int C);
int tc_launch_count();
constexpr int kSimtLaunches = 3;

// Device-side status word (tensor-core kernels' bounded waits).
int read_and_clear_device_status(cudaStream_t stream, int32_t *where);
int launch_timeout_selftest(int limit_us, cudaStream_t stream);

}  // namespace fmca
