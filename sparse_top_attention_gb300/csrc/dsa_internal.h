// Launchers shared between the kernel translation units and the C-ABI layer.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

struct Problem {
  int T, H, S_kv, W;
  float scale;
  bool delta_residual;  // out holds [2, T, H, 512]: rounded output, then its residual
  bool deterministic;   // dkv summed as 64-bit fixed point (order-independent)
  int d_qk = 576;        // q / kv row width: 576 (512 V + 64 rope) or 512 (V only)
  // Varlen batch (device arrays of B + 1 offsets), or nullptr for one sequence.
  const int32_t* cu_q = nullptr;
  const int32_t* cu_kv = nullptr;
  int B = 0;
};

// Byte offsets inside the backward workspace (256-byte aligned pieces).
struct BwdWorkspace {
  size_t dkv_acc;   // fp32 [S_kv, 576], or int64 [S_kv, 576] in 2^-32 units when deterministic
  size_t det_count; // u32 [S_kv]     deterministic only: valid slots naming each KV row
  size_t det_max;   // u32 [1]        deterministic only: largest |add| of the call (fp32 bits)
  size_t zero_bytes;  // end of the region zeroed before the backward (from dkv_acc = 0)
  size_t idxc;      // int32 [T, W]   compacted rows
  size_t count;     // int32 [T]
  size_t delta;     // fp32 [T, H]    rowsum(dout * out), written by the main stage one item ahead
  size_t dsink_t;   // fp32 [T, H]    -p_sink * delta (exact delta), from the main stage
  size_t cfix;      // fp32 [T, H]    scale * (exact delta - delta from out), from the main stage
  size_t sp;        // bf16 [T, nbmax, 64G, 128]: per (token, 128-slot block) the
                    // dS' rows (32G heads) then the P rows (32G heads), slots
                    // contiguous; G = ceil(H / 32), nbmax = ceil(W / 128)
  size_t total;
};
// Kernel attributes (the dynamic shared-memory limit) hold per device, so
// each launcher records in a bitmask which devices it has set up.  Device
// ordinals past 63 are set up on every call.
inline int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}
inline bool device_needs_setup(const std::atomic<uint64_t>& done, int dev) {
  return dev < 0 || dev >= 64 || (done.load(std::memory_order_acquire) & (1ull << dev)) == 0;
}
inline void mark_device_setup(std::atomic<uint64_t>& done, int dev) {
  if (dev >= 0 && dev < 64) done.fetch_or(1ull << dev, std::memory_order_release);
}

// SMs of the current device: the grid size of the persistent kernels.
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1;
  return n;
}

inline int bwd_groups(int H) { return (H + 31) / 32; }
inline int bwd_nbmax(int W) { return (W + 127) / 128; }
BwdWorkspace bwd_workspace_layout(const Problem& p);
// Validates the problem as every entry point does, then gives the backward's
// workspace size; the status is that of the failed check.
dsa_status_t bwd_workspace_checked(const dsa_problem_t* problem, size_t* bytes);

cudaError_t launch_fwd(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                       const int32_t* len, const float* sink, void* out, float* lse,
                       cudaStream_t s);

cudaError_t launch_compact(const Problem& p, const int32_t* idx, const int32_t* len,
                           int32_t* idx_out, int32_t* count_out, cudaStream_t s,
                           unsigned int* row_refs = nullptr);

// Backward stages; stage mask bit 0 = preprocess, 1 = main, 2 = finalize.
enum : int { kBwdPre = 1, kBwdMain = 2, kBwdFinal = 4, kBwdAll = 7 };
cudaError_t launch_bwd(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                       const int32_t* len, const float* sink, const void* out, const float* lse,
                       const void* dout, void* dq, void* dkv, float* dsink, void* ws,
                       cudaStream_t s, int stages);

// One small kernel whose barrier waits run out after limit_ns (the bounded-
// wait self-test behind dsa_wait_selftest).
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s);

// Device error words (one per translation unit): read-and-clear after a sync.
// 0x1xx are wait timeouts (the low byte says where); kErrDetRange is the
// deterministic accumulator's range check.
constexpr unsigned int kErrDetRange = 0x4FFu;
unsigned int fwd_take_error();
unsigned int bwd_take_error();

}  // namespace dsa
