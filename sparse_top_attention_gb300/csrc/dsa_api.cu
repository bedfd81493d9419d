// C-ABI entry points declared in include/dsa.h: argument validation, then
// launches on the caller's stream.  Nothing here allocates device memory.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace {

constexpr int kMaxWForward = 2048;  // matches the forward kernel's shared slot list

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status_t check_problem(const dsa_problem_t* p) {
  if (p == nullptr) return DSA_ERR_INVALID_ARG;
  if (p->T < 0 || p->H < 1 || p->S_kv < 1 || p->W < 1) return DSA_ERR_INVALID_ARG;
  if ((p->flags & ~(DSA_FLAG_DELTA_RESIDUAL | DSA_FLAG_DETERMINISTIC)) != 0u)
    return DSA_ERR_INVALID_ARG;
  if (!(p->scale == p->scale)) return DSA_ERR_INVALID_ARG;  // NaN scale
  if ((p->d_qk != 576 && p->d_qk != 512) || p->d_v != 512) return DSA_ERR_UNSUPPORTED;
  if (p->H > 128) return DSA_ERR_UNSUPPORTED;
  // The backward addresses accumulator rows with 32-bit element offsets.
  if (static_cast<int64_t>(p->S_kv) * p->d_qk > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

dsa::Problem to_internal(const dsa_problem_t* p) {
  dsa::Problem q{p->T, p->H, p->S_kv, p->W, p->scale,
                 (p->flags & DSA_FLAG_DELTA_RESIDUAL) != 0u,
                 (p->flags & DSA_FLAG_DETERMINISTIC) != 0u};
  q.d_qk = p->d_qk;
  return q;
}

dsa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// A varlen batch: B >= 1 sequences, both offset arrays given and 4-byte
// aligned.  Their contents stay on the device; the kernels clamp them.
dsa_status_t apply_varlen(const dsa_varlen_t* v, dsa::Problem* p) {
  if (v == nullptr) return DSA_OK;
  if (v->B < 1 || v->cu_seqlens_q == nullptr || v->cu_seqlens_kv == nullptr)
    return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(v->cu_seqlens_q) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(v->cu_seqlens_kv) & 3u) != 0)
    return DSA_ERR_ALIGNMENT;
  p->cu_q = v->cu_seqlens_q;
  p->cu_kv = v->cu_seqlens_kv;
  p->B = v->B;
  return DSA_OK;
}

}  // namespace

namespace dsa {
dsa_status_t bwd_workspace_checked(const dsa_problem_t* problem, size_t* bytes) {
  const dsa_status_t st = check_problem(problem);
  if (st != DSA_OK) return st;
  *bytes = bwd_workspace_layout(to_internal(problem)).total;
  return DSA_OK;
}
}  // namespace dsa

extern "C" {

static dsa_status_t fwd_impl(const dsa_problem_t* problem, const dsa_varlen_t* varlen,
                             const void* q, const void* kv, const int32_t* topk_idxs,
                             const int32_t* topk_length, const float* sink, void* out, float* lse,
                             void* stream) {
  dsa_status_t st = check_problem(problem);
  if (st != DSA_OK) return st;
  dsa::Problem p = to_internal(problem);
  st = apply_varlen(varlen, &p);
  if (st != DSA_OK) return st;
  if (problem->W > kMaxWForward) return DSA_ERR_UNSUPPORTED;
  if (problem->T == 0) return DSA_OK;
  if (!q || !kv || !topk_idxs || !out || !lse) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(topk_idxs) || !aligned16(out) ||
      !aligned16(lse) || (topk_length && !aligned16(topk_length)) || (sink && !aligned16(sink)))
    return DSA_ERR_ALIGNMENT;
  return from_cuda(dsa::launch_fwd(p, q, kv, topk_idxs, topk_length, sink, out, lse,
                                   static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_fwd(const dsa_problem_t* problem, const void* q, const void* kv,
                     const int32_t* topk_idxs, const int32_t* topk_length, const float* sink,
                     void* out, float* lse, void* stream) {
  return fwd_impl(problem, nullptr, q, kv, topk_idxs, topk_length, sink, out, lse, stream);
}

dsa_status_t dsa_fwd_varlen(const dsa_problem_t* problem, const dsa_varlen_t* varlen,
                            const void* q, const void* kv, const int32_t* topk_idxs,
                            const int32_t* topk_length, const float* sink, void* out, float* lse,
                            void* stream) {
  if (varlen == nullptr) return DSA_ERR_INVALID_ARG;
  return fwd_impl(problem, varlen, q, kv, topk_idxs, topk_length, sink, out, lse, stream);
}

size_t dsa_bwd_workspace_bytes(const dsa_problem_t* problem) {
  size_t n = 0;
  return dsa::bwd_workspace_checked(problem, &n) == DSA_OK ? n : 0;
}

static dsa_status_t bwd_stages(const dsa_problem_t* problem, const void* q, const void* kv,
                               const int32_t* topk_idxs, const int32_t* topk_length,
                               const float* sink, const void* out, const float* lse,
                               const void* dout, void* dq, void* dkv, float* dsink,
                               void* workspace, size_t workspace_bytes, void* stream, int stages,
                               const dsa_varlen_t* varlen = nullptr) {
  dsa_status_t st = check_problem(problem);
  if (st != DSA_OK) return st;
  dsa::Problem p = to_internal(problem);
  st = apply_varlen(varlen, &p);
  if (st != DSA_OK) return st;
  if (!kv || !dkv) return DSA_ERR_INVALID_ARG;
  if ((sink == nullptr) != (dsink == nullptr)) return DSA_ERR_INVALID_ARG;
  if (problem->T > 0 && (!q || !topk_idxs || !out || !lse || !dout || !dq))
    return DSA_ERR_INVALID_ARG;
  const size_t need = dsa::bwd_workspace_layout(p).total;
  if (workspace == nullptr || workspace_bytes < need) return DSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DSA_ERR_ALIGNMENT;
  const void* ptrs[] = {q, kv, topk_idxs, topk_length, sink, out, lse, dout, dq, dkv, dsink};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return DSA_ERR_ALIGNMENT;
  return from_cuda(dsa::launch_bwd(p, q, kv, topk_idxs, topk_length, sink, out, lse, dout, dq, dkv,
                                   dsink, workspace, static_cast<cudaStream_t>(stream), stages));
}

#define DSA_BWD_ARGS_DECL                                                                 \
  const dsa_problem_t *problem, const void *q, const void *kv, const int32_t *topk_idxs, \
      const int32_t *topk_length, const float *sink, const void *out, const float *lse,  \
      const void *dout, void *dq, void *dkv, float *dsink, void *workspace,              \
      size_t workspace_bytes, void *stream
#define DSA_BWD_ARGS \
  problem, q, kv, topk_idxs, topk_length, sink, out, lse, dout, dq, dkv, dsink, workspace, \
      workspace_bytes, stream

dsa_status_t dsa_bwd(DSA_BWD_ARGS_DECL) { return bwd_stages(DSA_BWD_ARGS, dsa::kBwdAll); }
dsa_status_t dsa_bwd_preprocess(DSA_BWD_ARGS_DECL) { return bwd_stages(DSA_BWD_ARGS, dsa::kBwdPre); }
dsa_status_t dsa_bwd_main(DSA_BWD_ARGS_DECL) { return bwd_stages(DSA_BWD_ARGS, dsa::kBwdMain); }
dsa_status_t dsa_bwd_finalize(DSA_BWD_ARGS_DECL) { return bwd_stages(DSA_BWD_ARGS, dsa::kBwdFinal); }

dsa_status_t dsa_bwd_varlen(const dsa_problem_t* problem, const dsa_varlen_t* varlen,
                            const void* q, const void* kv, const int32_t* topk_idxs,
                            const int32_t* topk_length, const float* sink, const void* out,
                            const float* lse, const void* dout, void* dq, void* dkv, float* dsink,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (varlen == nullptr) return DSA_ERR_INVALID_ARG;
  return bwd_stages(DSA_BWD_ARGS, dsa::kBwdAll, varlen);
}

dsa_status_t dsa_topk_compact(const dsa_problem_t* problem, const int32_t* topk_idxs,
                              const int32_t* topk_length, int32_t* idx_out, int32_t* count_out,
                              void* stream) {
  dsa_status_t st = check_problem(problem);
  if (st != DSA_OK) return st;
  if (problem->T == 0) return DSA_OK;
  if (!topk_idxs || !idx_out || !count_out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(topk_idxs) || !aligned16(idx_out) || !aligned16(count_out) ||
      (topk_length && !aligned16(topk_length)))
    return DSA_ERR_ALIGNMENT;
  return from_cuda(dsa::launch_compact(to_internal(problem), topk_idxs, topk_length, idx_out,
                                       count_out, static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_wait_selftest(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return DSA_ERR_INVALID_ARG;
  return from_cuda(dsa::launch_wait_selftest(static_cast<uint64_t>(limit_us) * 1000u,
                                             static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  const unsigned int a = dsa::fwd_take_error();
  const unsigned int b = dsa::bwd_take_error();
  if (a == 0xFFFFFFFFu || b == 0xFFFFFFFFu) return DSA_ERR_CUDA;
  if (a != 0) return DSA_ERR_DEVICE_TIMEOUT;
  if (b == dsa::kErrDetRange) return DSA_ERR_RANGE;
  if (b != 0) return DSA_ERR_DEVICE_TIMEOUT;
  return DSA_OK;
}

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported problem for this build";
    case DSA_ERR_ALIGNMENT: return "device pointer not 16-byte aligned (workspace: 256)";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSA_ERR_CUDA: return "CUDA runtime error";
    case DSA_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on an internal barrier";
    case DSA_ERR_RANGE: return "a deterministic dkv row may have left the accumulator's range";
  }
  return "unknown status";
}

int dsa_version(void) { return 100; }

}  // extern "C"
