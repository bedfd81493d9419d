// dsa_bwd_no_alloc: the backward pass with its workspace in a fixed, file-scope
// device array instead of caller-provided memory.
//
// Some callers cannot allocate device memory when they call the backward:
//   - a plain C host program that owns only the input and output buffers and
//     has no allocator of its own;
//   - a serving loop that runs under a fixed memory budget and must not let a
//     cudaMalloc synchronise the device in the middle of its pipeline.
// This entry point lets them run the same kernels, at the price of one
// fixed-size array that every GPU loading this library keeps until the
// process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace {

// Largest workspace this entry point can serve: 64 MiB.  For example this
// covers T = 128 tokens at H = 128 with the 640-slot DeepSeek-V4 layout.
constexpr size_t kNoAllocBytes = static_cast<size_t>(64) << 20;

// The workspace itself.  In host code this name is only a stand-in for the
// symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_no_alloc_workspace[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device with that device current.
dsa_status_t workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_workspace) != cudaSuccess || p == nullptr)
      return DSA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" dsa_status_t dsa_bwd_no_alloc(const dsa_problem_t* problem, const void* q,
                                         const void* kv, const int32_t* topk_idxs,
                                         const int32_t* topk_length, const float* sink,
                                         const void* out, const float* lse, const void* dout,
                                         void* dq, void* dkv, float* dsink, void* stream) {
  // The problem is checked exactly as dsa_bwd checks it (same status codes);
  // only then is its workspace compared with the array.
  size_t need = 0;
  const dsa_status_t chk = dsa::bwd_workspace_checked(problem, &need);
  if (chk != DSA_OK) return chk;
  if (need > kNoAllocBytes) return DSA_ERR_WORKSPACE;
  void* ws = nullptr;
  const dsa_status_t st = workspace_address(&ws);
  if (st != DSA_OK) return st;
  return dsa_bwd(problem, q, kv, topk_idxs, topk_length, sink, out, lse, dout, dq, dkv, dsink, ws,
                 kNoAllocBytes, stream);
}
