// Shapes, limits and the slot-validity rule shared by the CUDA kernels.
#pragma once

#include <cstdint>

#include "dsa_ptx.cuh"

namespace dsa {

constexpr int kDqk = 576;         // q / kv row width (512 + 64)
constexpr int kDv = 512;          // V = kv[:, :512]
constexpr int kRowBytes = kDqk * 2;
constexpr int kChunks = kDqk / 64;  // 64-column (128-byte) chunks of a row
constexpr int kBlk = 128;         // gathered slots per block (UMMA M)
// Rows of a block one gather warp issues: 3 warps share the 32 groups of 4 rows.
constexpr int kRowGroups = (kBlk / 4 + 2) / 3;
constexpr int kMaxW = 2048;       // index slots per token supported by the forward
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kFltMax = 3.402823466e38f;

// Validity of slot j of a token (cuDNN frontend "DSA backward SM90: fix three
// top-k and attention-sink boundary failures", Why item 2; cuDNN frontend
// "DSA bwd SM100 fix dropped dKV gradients when topk width > total_S_kv"):
// the index value must lie in [0, S_kv) and the slot must lie before the
// clamped top-k length.  The column position is never compared with S_kv.
__device__ __forceinline__ bool slot_valid(int32_t idx, int j, int len, int S_kv) {
  return idx >= 0 && idx < S_kv && j < len;
}

// Effective length of a token's slot list: W without a length array,
// otherwise topk_length[t] clamped to [0, W].
__device__ __forceinline__ int slot_len(const int32_t* topk_length, int t, int W) {
  if (topk_length == nullptr) return W;
  const int n = topk_length[t];
  return n < 0 ? 0 : (n > W ? W : n);
}

// The KV rows a token may index: all S_kv rows, or in a varlen batch the rows
// of the token's own sequence.  Sequence b holds tokens cu_q[b] <= t <
// cu_q[b + 1] and KV rows cu_kv[b] <= r < cu_kv[b + 1]; its indices count
// from cu_kv[b].  The range is clamped into [0, S_kv], and a token outside
// every sequence gets an empty range, so malformed arrays cannot reach
// outside kv.
struct KvRange {
  int lo, n;
};
__device__ __forceinline__ KvRange kv_range(const int32_t* cu_q, const int32_t* cu_kv, int B, int t,
                                            int S_kv) {
  if (cu_q == nullptr) return {0, S_kv};
  int lo = 0, hi = B - 1;  // the last sequence whose first token is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  if (t < cu_q[lo] || t >= cu_q[lo + 1]) return {0, 0};
  const int a = min(max(cu_kv[lo], 0), S_kv);
  const int e = min(max(cu_kv[lo + 1], a), S_kv);
  return {a, e - a};
}

// Block-wide compaction of one token's valid rows, in slot order.
// All `nthreads` threads (a multiple of 32) must call it.  `warp_counts`
// is shared scratch of nthreads/32 ints.  Writes up to `cap` entries to
// `list` (shared or global) and returns the total valid count.  Slot j is
// valid when 0 <= idx < kv.n; its entry is the KV row kv.lo + idx.
__device__ __forceinline__ int compact_token(const int32_t* __restrict__ idx_row, int W, int len,
                                             KvRange kv, int32_t* list, int cap, int* warp_counts,
                                             int tid, int nthreads) {
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  int base = 0;
  for (int j0 = 0; j0 < W; j0 += nthreads) {
    const int j = j0 + tid;
    int32_t v = -1;
    bool ok = false;
    if (j < W) {
      v = idx_row[j];
      ok = slot_valid(v, j, len, kv.n);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) warp_counts[warp] = __popc(bal);
    __syncthreads();
    int off = base, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int c = warp_counts[w];
      if (w < warp) off += c;
      tot += c;
    }
    const int pos = off + __popc(bal & lt_mask);
    if (ok && pos < cap) list[pos] = kv.lo + v;
    base += tot;
    __syncthreads();
  }
  return base;
}

// compact_token on a row that each thread has already read into registers:
// vals[i] is entry i * nthreads + tid (W <= kN * nthreads).  Reading the row
// early lets its latency overlap other set-up work.
template <int kN>
__device__ __forceinline__ void load_index_row(const int32_t* __restrict__ idx_row, int W, int tid,
                                               int nthreads, int32_t (&vals)[kN]) {
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    const int j = i * nthreads + tid;
    vals[i] = j < W ? idx_row[j] : -1;
  }
}

// Compacts a register-held index row (element i * nthreads + tid in vals[i])
// with `nthreads` threads (whole warps, thread ids 0..nthreads-1 within the
// group) that synchronise on named barrier `bar`.
template <int kN>
__device__ __forceinline__ int compact_token_regs(const int32_t (&vals)[kN], int W, int len,
                                                  KvRange kv, int32_t* list, int cap,
                                                  int* warp_counts, int tid, int nthreads,
                                                  int bar) {
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    if (i * nthreads >= W) break;
    const int j = i * nthreads + tid;
    const int32_t v = vals[i];
    const bool ok = j < W && slot_valid(v, j, len, kv.n);
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) warp_counts[warp] = __popc(bal);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthreads) : "memory");
    int off = base, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int c = warp_counts[w];
      if (w < warp) off += c;
      tot += c;
    }
    const int pos = off + __popc(bal & lt_mask);
    if (ok && pos < cap) list[pos] = kv.lo + v;
    base += tot;
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthreads) : "memory");
  }
  return base;
}

// Number of valid slots of one index row, counted by one warp (every lane
// gets the count).  The same rule as the compaction: slot j < min(len, W)
// holding an index in [0, kv.n).
__device__ __forceinline__ int warp_count_valid(const int32_t* __restrict__ idx_row, int W,
                                                int len, KvRange kv, int lane) {
  const int lim = len < W ? len : W;
  int n = 0;
  for (int j0 = 0; j0 < lim; j0 += 128) {
    int32_t v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q * 32 + lane;
      v[q] = j < lim ? idx_row[j] : -1;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) n += __popc(__ballot_sync(0xffffffffu, v[q] >= 0 && v[q] < kv.n));
  }
  return n;
}

}  // namespace dsa
