// Sparse MLA (DSA) backward for sm_103a.
//
// Kernels, queued in order on the caller's stream:
//   memset      dkv accumulator <- 0 (fp32, or int64 fixed point)
//   k_compact   a1: valid KV rows of every token, in slot order, and counts
//   k_bwd_pre   b1: delta = rowsum(dout * out), lse*log2(e), gate and the
//               per-(t,h) d_sink terms (FlashAttention "dpsum" preprocess)
//   k_bwd_dq    b2-b5: per (token, 64-head group; 32 heads when H <= 32)
//               recompute P, form dS, accumulate dQ in TMEM and store dq;
//               write the dS' and P
//               tiles of every 128-slot block to a bf16 scratch.  One
//               persistent CTA per SM walks the (token, group) items.
//   k_bwd_dkv   b6: per token, dKV_blk^T = [Q^T | dO^T] [dS'; P] over all
//               heads at once, scatter-added into the fp32 accumulator
//   k_dkv_cast  fp32 accumulator -> bf16 dkv (k_dkv_cast_fixed for the int64
//               fixed-point accumulator of DSA_FLAG_DETERMINISTIC)
//   k_dsink     b7: d_sink[h] = sum_t (-p_sink * delta), fixed order
//
// Math per (t, h) and valid slot j.  The forward's lse excludes the sink;
// gate = sigma(lse - sink):
//   P_j  = exp(s_j - lse) * gate
//   dP_j = dout . V_j
//   dS_j = P_j * (dP_j - delta)
//   dq   = scale * sum_j dS_j KV_j
//   dkv[idx_j] += scale * dS_j q + P_j [dout, 0]
//   dsink = -sum_t sigma(sink - lse) * delta
// Sources:
//   - cuDNN frontend "DSA backward SM90: fix three top-k and attention-sink
//     boundary failures": Summary 1-3, Why 1-3, "Not addressed" (delta from
//     the bf16 out; P recomputed without an online softmax, live columns
//     satisfy s - lse <= 0).
//   - flash-attention "[CuTe, SM100] Support 1..128 Q heads in sparse MLA via
//     in-kernel TMA padding", Agent Notes: padded heads give dS = 0, and the
//     d_sink reduce only covers the real heads.
//   - cuDNN frontend "DSA bwd SM100 fix dropped dKV gradients when topk
//     width > total_S_kv": a dkv contribution is judged by the index value
//     and the top-k bound only.
//
// Rows are D = 576 columns (512 V + 64 rope) or 512 (no rope part); the
// kernels are templates over D.
// k_bwd_dq tiles, transposed like the forward: gathered rows are UMMA M
// (128) and the 64 heads of the group are N (32 heads, and half the N,
// when H <= 32).
//   [S^T | dP^T] = KV_blk . [Q^T | dO^T]  M=128 N=128 K=512, then S^T += rope part (N=64, K=64)
//   dQ^T += KV_blk^T . dS'^T             ceil(D/128) x (M=128 N=64 K=128)
// where dS' = scale * dS.  dS'^T and P^T tiles are written to the scratch.
// A block of 128 consecutive KV rows (the sliding window) is loaded by 2-D
// TMA; other blocks row by row with cp.async.  Q and dO of 64 heads do not
// fit beside a 128-row KV block, so each S / dP step brings its 64-column
// (Q, dO) chunk pair in by TMA through a 4-stage ring.  Two softmax
// warpgroups split the 64 heads of each gathered row.
// k_bwd_dkv tiles, per 128-slot block of one token, d rows on the M side:
//   dKV_blk^T[d, slots] = [Q^T | dO^T][d, 2 x 32G] . [dS'; P][2 x 32G, slots]
// (dO^T is zero for the 64 rope rows), so the dKV GEMM sees all heads at once
// and each valid slot gets one partial per token.  Its fp32 adds go through
// shared memory so that each warp reduction covers 128 floats of one row.
#include <cmath>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_tmap.h"

namespace dsa {

BwdWorkspace bwd_workspace_layout(const Problem& p) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  BwdWorkspace w{};
  size_t off = 0;
  const size_t TH = static_cast<size_t>(p.T) * p.H;
  w.dkv_acc = off; off = up(off + static_cast<size_t>(p.S_kv) * p.d_qk * (p.deterministic ? 8 : 4));
  w.idxc = off;    off = up(off + static_cast<size_t>(p.T) * p.W * 4);
  w.count = off;   off = up(off + static_cast<size_t>(p.T) * 4);
  w.lse2 = off;    off = up(off + TH * 4);
  w.gate = off;    off = up(off + TH * 4);
  w.delta = off;   off = up(off + TH * 4);
  w.dsink_t = off; off = up(off + TH * 4);
  w.sp = off;
  off = up(off + static_cast<size_t>(p.T) * bwd_nbmax(p.W) * 64 * bwd_groups(p.H) * 128 * 2);
  w.total = off;
  return w;
}

namespace {

__device__ unsigned int g_err_bwd;

// ------------------------------------------------------------------ a1

constexpr int kCompactThreads = 256;

__global__ void __launch_bounds__(kCompactThreads)
k_compact(const int32_t* __restrict__ topk_idxs, const int32_t* __restrict__ topk_length,
          int32_t* __restrict__ idx_out, int32_t* __restrict__ count_out, int W, int S_kv,
          const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int B) {
  __shared__ int warp_counts[kCompactThreads / 32];
  const int t = blockIdx.x;
  const int len = slot_len(topk_length, t, W);
  const KvRange kvr = kv_range(cu_q, cu_kv, B, t, S_kv);
  const int n = compact_token(topk_idxs + static_cast<size_t>(t) * W, W, len, kvr,
                              idx_out + static_cast<size_t>(t) * W, W, warp_counts, threadIdx.x,
                              kCompactThreads);
  if (threadIdx.x == 0) count_out[t] = n;
}

// ------------------------------------------------------------------ b1

// One warp per (t, h) row: delta = sum_d dout*out over the 512 V columns.
__global__ void __launch_bounds__(256)
k_bwd_pre(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
          const float* __restrict__ lse, const float* __restrict__ sink,
          const int32_t* __restrict__ count, float* __restrict__ lse2_o,
          float* __restrict__ gate_o, float* __restrict__ delta_o, float* __restrict__ dsink_t,
          int T, int H, int residual) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(T) * H) return;
  const int t = static_cast<int>(row / H), h = static_cast<int>(row - static_cast<long long>(t) * H);
  const uint4* o4 = reinterpret_cast<const uint4*>(out + row * kDv);
  const uint4* d4 = reinterpret_cast<const uint4*>(dout + row * kDv);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 a = o4[lane + 32 * i], b = d4[lane + 32 * i];
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(a2[k]), fb = __bfloat1622float2(b2[k]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
  if (residual) {  // delta from out + its rounding residual (about fp32 O)
    const uint4* l4 = reinterpret_cast<const uint4*>(out + static_cast<size_t>(T) * H * kDv + row * kDv);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 a = l4[lane + 32 * i], b = d4[lane + 32 * i];
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(a2[k]), fb = __bfloat1622float2(b2[k]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    const bool empty = count[t] == 0;
    const float l = lse[row];
    const float sk = sink != nullptr ? sink[h] : -INFINITY;
    // An empty row has no attention term: the sink holds the whole
    // denominator (p_sink = 1) and P is zero.
    const float gate = empty ? 0.f : stable_sigmoid(l - sk);
    const float p_sink = empty ? 1.f : stable_sigmoid(sk - l);
    lse2_o[row] = empty ? 0.f : l * kLog2e;
    gate_o[row] = gate;
    delta_o[row] = acc;
    dsink_t[row] = -p_sink * acc;
  }
}

// ------------------------------------------------------------------ b2-b4: dq, dS', P

constexpr int kSoftmax = 256;            // warps 0-7: row (warp & 3) * 32 + lane, half (warp >> 2) of the heads
constexpr int kMmaWarp = 8;
constexpr int kIssuer = 288;             // lane 0 of warp 9
constexpr int kProducers = 96;           // warps 9-11
constexpr int kLoaderWarp = 12;          // lane 0 streams the (Q, dO) chunk pairs
constexpr int kThreads = kSoftmax + 32 + kProducers + 32;
constexpr int kKVChunk = kBlk * 128;     // 16 KB
constexpr int kMaxStages = 8;
constexpr int kMaxHG = 64;
constexpr uint32_t kTmemCols = 512;

// Head group of an item: 64 heads, or 32 when H <= 32 (less padding: the
// Q/dO ring stages halve and the MMAs narrow).
template <int kHG>
struct DqHeads {
  static_assert(kHG == 64 || kHG == 32, "head group");
  static constexpr int kHT = kHG / 2;          // heads per softmax thread
  static constexpr int kHChunk = kHG * 128;    // 64 columns of kHG head rows
  static constexpr int kStage = 2 * kHChunk;   // Q chunk x (rows 0..kHG-1), then dO chunk x
  static constexpr int kStages = kHG == 64 ? 4 : 8;  // ring of (Q, dO) chunk pairs
  // TMEM: [S^T | dP^T] (2 x kHG columns), then dQ^T (5 tiles x kHG columns).
  static constexpr uint32_t kColS = 0, kColdP = kHG, kColdQ = 2 * kHG;
};

struct Misc {
  uint64_t kv_full[kChunks];
  uint64_t kv_free[kChunks];
  uint64_t qd_full[kMaxStages], qd_free[kMaxStages];
  uint64_t s_full, ds_full, rope_done, dsp_free, dq_full, mma_done;
  // per head of the item: (log2(gate) - lse * log2(e), delta), so that
  // P = exp2(s * scale * log2(e) + x) and one 16-byte load serves two heads
  alignas(16) float2 cd[kMaxHG];
  uint32_t tmem_base;
  int abort_flag;
};

// Shared-memory layout for rows of kD columns (576 = 512 V + 64 rope, or 512).
// With a rope chunk, position p of the gathered block holds d-chunk x(p):
// p = 0 the rope columns 512..575 (reused for the P tile once the rope part
// of dQ is done), p = 1..8 the V chunks 0..7; blocks are gathered and
// consumed in the order p = 1..8, 0 because position 0 is released last.
// Without one, position p holds V chunk p and P has a tile of its own.
// Q and dO do not stay resident: their chunk x comes in by TMA into a ring
// stage for each S / dP step.
template <int kD, int kHG>
struct DqLayout {
  using Hd = DqHeads<kHG>;
  static constexpr int kHChunk = Hd::kHChunk, kStage = Hd::kStage, kStages = Hd::kStages;
  static constexpr int kCh = kD / 64;
  static constexpr bool kRope = kCh > 8;
  static constexpr int kDT = (kD + 127) / 128;   // 128-row d tiles of dQ^T
  static constexpr int kOffKV = 0;
  static constexpr int kOffQD = kOffKV + kCh * kKVChunk;
  static constexpr int kOffdS = kOffQD + kStages * kStage;  // 2 sub-tiles of 64 slots
  static constexpr int kOffP = kRope ? kOffKV : kOffdS + 2 * kHChunk;
  static constexpr int kOffMisc = kRope ? kOffdS + 2 * kHChunk : kOffP + 2 * kHChunk;
  static constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQD % 1024 == 0 && kOffdS % 1024 == 0 && kOffP % 1024 == 0, "alignment");
};

template <unsigned int* kErr>
__device__ __forceinline__ void mbar_wait_final(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(kErr, 0u, 0x1FFu);
      return;
    }
  }
}

template <bool kRope>
__device__ __forceinline__ int dchunk_of_pos(int pos) {
  return kRope ? (pos == 0 ? 8 : pos - 1) : pos;
}
// Gather / S-GEMM order of the shared positions: V chunks first, rope last.
template <bool kRope>
__device__ __forceinline__ int pos_of_step(int i) {
  return kRope ? (i == kChunks - 1 ? 0 : i + 1) : i;
}

// Byte offset of element (head row h, slot) in a [kHG rows x 128 slots] bf16
// tile kept as two 128B-swizzled sub-tiles of 64 slots: the layout of dS' and
// P (K-major B for dQ^T; stored to the scratch by TMA, 32 rows x 64 slots
// per box).
template <int kHG>
__device__ __forceinline__ uint32_t hs_tile_off(uint32_t h, uint32_t slot) {
  const uint32_t col = slot & 63u;
  return (slot >> 6) * (kHG * 128u) + h * 128u +
         ((((col >> 3) ^ (h & 7u)) << 4) | ((col & 7u) << 1));
}

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Items are (token, kHG-head group) pairs; the scratch keeps its rows per
// 32-head group (G32 groups: dS' rows first, then P rows).
template <int kD, int kHG>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_dq(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
         const __grid_constant__ CUtensorMap tm_sp, const __grid_constant__ CUtensorMap tm_kv,
         const __nv_bfloat16* __restrict__ kv,
         const int32_t* __restrict__ idxc, const int32_t* __restrict__ count,
         const float* __restrict__ lse2_g, const float* __restrict__ gate_g,
         const float* __restrict__ delta_g, __nv_bfloat16* __restrict__ dq, int T, int H, int W,
         float scale, int G, int G32, int box_heads, int nbmax) {
  using L = DqLayout<kD, kHG>;
  using Hd = DqHeads<kHG>;
  constexpr int kCh = L::kCh, kDT = L::kDT, kOffKV = L::kOffKV, kOffQD = L::kOffQD,
                kOffdS = L::kOffdS, kOffP = L::kOffP, kOffMisc = L::kOffMisc;
  constexpr int kHChunk = Hd::kHChunk, kStage = Hd::kStage, kStages = Hd::kStages, kHT = Hd::kHT;
  constexpr uint32_t kColS = Hd::kColS, kColdP = Hd::kColdP, kColdQ = Hd::kColdQ;
  constexpr bool kRope = L::kRope;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (tid == 0) atomicCAS(&g_err_bwd, 0u, 0x2FFu);
    return;
  }
  Misc& m = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const FailState fs{&g_err_bwd, &m.abort_flag};
  // Persistent: CTA c takes items c, c + gridDim.x, ... of the (token, head
  // group) list.  Every role walks the same items; barrier phases follow
  // running counts of blocks, of S / dP steps (the Q / dO ring) and of
  // non-empty items.
  const int n_items = T * G;

  if (tid == 0) {
    for (int c = 0; c < kCh; ++c) {
      mbar_init(smem_u32(&m.kv_full[c]), kProducers);
      mbar_init(smem_u32(&m.kv_free[c]), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&m.qd_full[s]), 1);
      mbar_init(smem_u32(&m.qd_free[s]), 1);
    }
    mbar_init(smem_u32(&m.s_full), 1);
    mbar_init(smem_u32(&m.ds_full), kSoftmax);
    mbar_init(smem_u32(&m.rope_done), 1);
    mbar_init(smem_u32(&m.dsp_free), 1);
    mbar_init(smem_u32(&m.dq_full), 1);
    mbar_init(smem_u32(&m.mma_done), 1);
    m.abort_flag = 0;
    mbar_init_fence();
  }
  // Ring rows the TMA boxes do not cover (only when H < 64) are zero; the
  // loads never write them, so once is enough.
  {
    const int per = (kHG - box_heads) * 8;  // 16-byte pieces per half stage
    for (int i = tid; i < kStages * 2 * per; i += kThreads) {
      const int half = i / per, rem = i - half * per;  // half = 2 * stage + (0: Q, 1: dO)
      const int row = (half & 1) * kHG + box_heads + rem / 8, pc = rem & 7;
      asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(
                       sbase + kOffQD + (half >> 1) * kStage + sw128_off(row, pc)),
                   "r"(0u)
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  if (warp == kMmaWarp) tmem_alloc(smem_u32(&m.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

  if (warp == kLoaderWarp) {
    // ------------------------------------------------------------ Q / dO ring
    // The (Q, dO) chunk pair of every S / dP step by TMA, each as soon as its
    // ring stage is free: the first stages of a block fill while the softmax
    // and dQ of the previous block run.
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();
      int gs = 0;
      for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
        const int t = u / G, h0 = (u - t * G) * kHG;
        const int Kt = count[t];
        if (Kt == 0) continue;
        const int nsteps = (Kt + kBlk - 1) / kBlk * kCh;
        for (int k = 0; k < nsteps; ++k, ++gs) {
          const int x = dchunk_of_pos<kRope>(pos_of_step<kRope>(k % kCh));
          const int s = gs % kStages, n = gs / kStages;
          if (n > 0) mbar_wait(smem_u32(&m.qd_free[s]), (n - 1) & 1, fs, 11);
          const uint32_t st = sbase + kOffQD + s * kStage;
          mbar_arrive_expect_tx(smem_u32(&m.qd_full[s]), (x < 8 ? 2 : 1) * box_heads * 128);
          tma_load_3d_hint(st, &tm_q, x * 64, h0, t, smem_u32(&m.qd_full[s]), keep);
          if (x < 8)
            tma_load_3d_hint(st + kHChunk, &tm_do, x * 64, h0, t, smem_u32(&m.qd_full[s]), keep);
        }
      }
    }
    __syncwarp();
  } else if (warp > kMmaWarp) {
    // ------------------------------------------------------------ KV gather
    // The KV chunk of each S / dP step: cp.async (one warp instruction = 4
    // whole 128 B row pieces) into the 128B-swizzled chunk tile, or by 2-D
    // TMA for a block of consecutive rows.
    const int pw = warp - (kMmaWarp + 1);
    const uint64_t keep = l2_evict_last();
    int gb = 0;  // blocks so far
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G;
      const int Kt = count[t];
      if (Kt == 0) continue;
      const int nblk = (Kt + kBlk - 1) / kBlk;
      const int32_t* rows = idxc + static_cast<size_t>(t) * W;
      for (int b = 0; b < nblk; ++b, ++gb) {
        // This lane's rows of the block, read once (before the wait on the
        // first chunk, so the reads overlap it) and reused by all chunks.
        const __nv_bfloat16* src[kRowGroups];
        uint32_t dst[kRowGroups], nbytes[kRowGroups];
#pragma unroll
        for (int k = 0; k < kRowGroups; ++k) {
          const int g = pw + 3 * k;
          const int row = g * 4 + (lane >> 3), pc = lane & 7;
          const int slot = b * kBlk + row;
          const bool ok = g < kBlk / 4 && slot < Kt;
          const int r = ok ? rows[slot] : 0;
          src[k] = kv + static_cast<size_t>(r) * kD + pc * 8;
          dst[k] = sw128_off(row & (kBlk - 1), pc);
          nbytes[k] = ok ? 16u : 0u;
        }
        // A full block of consecutive KV rows (the sliding window) comes in
        // with one 2-D TMA load per chunk instead of 128 row copies.
        bool contig = false;
        int r0 = 0;
        if (b * kBlk + kBlk <= Kt) {
          r0 = rows[b * kBlk];
          bool mine = true;
          for (int i = tid - kIssuer; i < kBlk; i += kProducers) mine &= rows[b * kBlk + i] == r0 + i;
          contig = !named_bar_or(2, kProducers, !mine);
        }
        for (int i = 0; i < kCh; ++i) {
          const int pos = pos_of_step<kRope>(i);
          const int x = dchunk_of_pos<kRope>(pos);
          if (gb > 0) mbar_wait(smem_u32(&m.kv_free[pos]), (gb - 1) & 1, fs, 1);
          if (contig) {
            if (tid == kIssuer) {
              mbar_arrive_expect_tx(smem_u32(&m.kv_full[pos]), kKVChunk);
              tma_load_2d_hint(sbase + kOffKV + pos * kKVChunk, &tm_kv, x * 64, r0,
                               smem_u32(&m.kv_full[pos]), keep);
            } else {
              mbar_arrive(smem_u32(&m.kv_full[pos]));
            }
            continue;
          }
#pragma unroll
          for (int k = 0; k < kRowGroups; ++k)
            if (pw + 3 * k < kBlk / 4)
              cp_async_16_hint(sbase + kOffKV + pos * kKVChunk + dst[k], src[k] + x * 64,
                               nbytes[k], keep);
          cp_async_arrive(smem_u32(&m.kv_full[pos]));
        }
      }
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ UMMA issue
    if (lane == 0) {
      const uint32_t idSdP = idesc_bf16(128, 2 * kHG, false, false);  // [S^T | dP^T]
      const uint32_t idS = idesc_bf16(128, kHG, false, false);         // S^T, rope part
      const uint32_t idQ = idesc_bf16(128, kHG, true, false);  // dQ^T: A MN-major, B K-major
      int it = 0, gb = 0, gs = 0;
      for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
        const int t = u / G;
        const int Kt = count[t];
        if (Kt == 0) continue;
        const int nblk = (Kt + kBlk - 1) / kBlk;
        for (int b = 0; b < nblk; ++b, ++gb) {
          for (int i = 0; i < kCh; ++i, ++gs) {
            const int pos = pos_of_step<kRope>(i);
            const int x = dchunk_of_pos<kRope>(pos);
            const int s = gs % kStages, n = gs / kStages;
            mbar_wait(smem_u32(&m.kv_full[pos]), gb & 1, fs, 3);
            mbar_wait(smem_u32(&m.qd_full[s]), n & 1, fs, 2);
            fence_proxy_async_smem();  // cp.async (generic proxy) -> UMMA (async proxy)
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t a = sdesc_sw128(sbase + kOffKV + pos * kKVChunk + k * 32, 16, 1024);
              // V chunks: S and dP in one N = 128 MMA (B rows: the Q heads,
              // then the dO heads); the rope chunk adds to S only.
              const uint64_t bqd = sdesc_sw128(sbase + kOffQD + s * kStage + k * 32, 16, 1024);
              umma_ss(tmem + kColS, a, bqd, x < 8 ? idSdP : idS, (i | k) != 0);
            }
            umma_commit(smem_u32(&m.qd_free[s]));
          }
          umma_commit(smem_u32(&m.s_full));
          // dS' of this block; for the first block of an item this also
          // orders the softmax warps' read-out of the previous dQ^T first
          mbar_wait(smem_u32(&m.ds_full), gb & 1, fs, 4);
          tc_fence_after();
          // dQ^T chunks: rope first (its second 64-row atom reads V chunk 0 as
          // filler rows that are never stored), then d rows 0..511.
          for (int jj = 0; jj < kDT; ++jj) {
            const int j = kRope ? ((jj == 0) ? 4 : jj - 1) : jj;
            const int pos0 = (j == 4) ? 0 : (kRope ? 1 + 2 * j : 2 * j);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t a =
                  sdesc_sw128(sbase + kOffKV + pos0 * kKVChunk + kk * 2048, kKVChunk, 1024);
              const uint64_t bs =
                  sdesc_sw128(sbase + kOffdS + (kk >> 2) * kHChunk + (kk & 3) * 32, 16, 1024);
              umma_ss(tmem + kColdQ + j * kHG, a, bs, idQ, (b | kk) != 0);
            }
            if (j == 4) {
              umma_commit(smem_u32(&m.rope_done));
            } else {
              umma_commit(smem_u32(&m.kv_free[pos0]));
              umma_commit(smem_u32(&m.kv_free[pos0 + 1]));
            }
          }
          umma_commit(smem_u32(&m.dsp_free));
        }
        umma_commit(smem_u32(&m.dq_full));
        ++it;
      }
      if (it > 0) {  // all MMAs retired before the TMEM is freed
        umma_commit(smem_u32(&m.mma_done));
        mbar_wait_final<&g_err_bwd>(smem_u32(&m.mma_done), 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ P, dS', dq
    // Thread (warp w, lane l) owns gathered row (w & 3) * 32 + l of the
    // block (its TMEM lane) and heads hb .. hb + kHT - 1, hb = kHT * (w >> 2): two
    // warps per SM sub-partition share the exp2 / FMA work of a block.
    const float sl2 = scale * kLog2e;
    const size_t spr = static_cast<size_t>(64) * G32;  // scratch rows per (token, block)
    const int row = (warp & 3) * 32 + lane, hb = (warp >> 2) * kHT;
    int it = 0, gb = 0;
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G, h0 = (u - t * G) * kHG;
      const int nh = min(kHG, H - h0);
      const int Kt = count[t];
      if (Kt == 0) {  // empty row: dq = 0, nothing for dkv
        for (int v = tid; v < nh * (kD / 8); v += kSoftmax) {
          const int h = v / (kD / 8), c = v - h * (kD / 8);
          *reinterpret_cast<uint4*>(dq + (static_cast<size_t>(t) * H + h0 + h) * kD + c * 8) =
              make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int nblk = (Kt + kBlk - 1) / kBlk;
      if (tid < kHG) {
        // Padded heads get gate 0, hence P = dS = 0: they add nothing anywhere.
        const bool real = tid < nh;
        const size_t r = static_cast<size_t>(t) * H + h0 + tid;
        const float gt = real ? gate_g[r] : 0.f;
        m.cd[tid] = make_float2(gt > 0.f ? log2f(gt) - lse2_g[r] : -INFINITY,
                                real ? delta_g[r] : 0.f);
      }
      named_bar_sync(1, kSoftmax);
      for (int b = 0; b < nblk; ++b, ++gb) {
        mbar_wait(smem_u32(&m.s_full), gb & 1, fs, 7);
        tc_fence_after();
        const bool valid = b * kBlk + row < Kt;
        uint32_t rs[kHT], rd[kHT];
        if constexpr (kHT == 32)
          tmem_ld32x2_sync(tmem + lane_base + kColS + hb, rs, tmem + lane_base + kColdP + hb, rd);
        else
          tmem_ld16x2_sync(tmem + lane_base + kColS + hb, rs, tmem + lane_base + kColdP + hb, rd);
        float dsv[kHT];
        uint32_t pk[kHT / 2];  // P as bf16 pairs (heads hb + 2i, hb + 2i + 1)
        const float4* cd4 = reinterpret_cast<const float4*>(m.cd + hb);
#pragma unroll
        for (int i = 0; i < kHT; i += 2) {
          const float4 c = cd4[i / 2];  // heads hb + i, hb + i + 1
          // Live columns satisfy s - lse <= 0, so exp2 never overflows here;
          // rows past the valid count hold zero KV (finite dP) and get P = 0.
          const float p0 = valid ? ex2_approx(fmaf(__uint_as_float(rs[i]), sl2, c.x)) : 0.f;
          const float p1 = valid ? ex2_approx(fmaf(__uint_as_float(rs[i + 1]), sl2, c.z)) : 0.f;
          dsv[i] = p0 * (__uint_as_float(rd[i]) - c.y) * scale;
          dsv[i + 1] = p1 * (__uint_as_float(rd[i + 1]) - c.w) * scale;
          pk[i / 2] = pack_bf16x2(p0, p1);
        }
        if (gb > 0) mbar_wait(smem_u32(&m.dsp_free), (gb - 1) & 1, fs, 8);
        // thread 0 finished reading the previous block's tiles out (bulk wait below)
        named_bar_sync(1, kSoftmax);
#pragma unroll
        for (int i = 0; i < kHT; ++i) {
          const __nv_bfloat16 v = __float2bfloat16_rn(dsv[i]);
          st_shared_b16(sbase + kOffdS + hs_tile_off<kHG>(hb + i, row),
                        *reinterpret_cast<const uint16_t*>(&v));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&m.ds_full));
        // With a rope chunk, P goes into position 0 once the rope part of dQ
        // has read the rope rows.
        if constexpr (kRope) mbar_wait(smem_u32(&m.rope_done), gb & 1, fs, 9);
#pragma unroll
        for (int i = 0; i < kHT / 2; ++i) {
          st_shared_b16(sbase + kOffP + hs_tile_off<kHG>(hb + 2 * i, row),
                        static_cast<uint16_t>(pk[i]));
          st_shared_b16(sbase + kOffP + hs_tile_off<kHG>(hb + 2 * i + 1, row),
                        static_cast<uint16_t>(pk[i] >> 16));
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kSoftmax);
        if (tid == 0) {
          // dS' and P rows of this head group -> the (token, block) scratch
          // tile, in boxes of 32 heads that hold at least one real head
          const int row0 = static_cast<int>((static_cast<size_t>(t) * nbmax + b) * spr) + h0;
          const uint64_t pol = l2_evict_first();
          for (int half = 0; half < 2; ++half)
            for (int g2 = 0; g2 * 32 < nh; ++g2) {
              tma_store_2d_hint(&tm_sp, half * 64, row0 + g2 * 32,
                                sbase + kOffdS + half * kHChunk + g2 * 4096, pol);
              tma_store_2d_hint(&tm_sp, half * 64, row0 + 32 * G32 + g2 * 32,
                                sbase + kOffP + half * kHChunk + g2 * 4096, pol);
            }
          bulk_commit();
          bulk_wait_read();
          if constexpr (kRope) mbar_arrive(smem_u32(&m.kv_free[0]));  // position 0 may take the next rope rows
        }
      }
      // dQ^T -> dq (bf16), straight from registers: for each head, a warp
      // writes 32 consecutive d of that head's row.
      mbar_wait(smem_u32(&m.dq_full), it & 1, fs, 10);
      tc_fence_after();
      __nv_bfloat16* dq_t = dq + (static_cast<size_t>(t) * H + h0) * kD;
      for (int j = 0; j < kDT; ++j) {
        const int d = j * 128 + row;
        uint32_t v[kHT];
        if constexpr (kHT == 32)
          tmem_ld32_sync(tmem + lane_base + kColdQ + j * kHG + hb, v);
        else
          tmem_ld16_sync(tmem + lane_base + kColdQ + j * kHG + hb, v);
        if (d < kD) {
#pragma unroll
          for (int i = 0; i < kHT; ++i) {
            const int h = hb + i;
            if (h < nh) dq_t[static_cast<size_t>(h) * kD + d] = __float2bfloat16_rn(__uint_as_float(v[i]));
          }
        }
      }
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ b5-b6: dKV

// One CTA per token, every head at once:
//   dKV^T[d, slot] = sum_h Q[h, d] dS'[h, slot] + sum_h dO[h, d] P[h, slot]
// M = 128 d rows per chunk (4 V chunks + the rope chunk), N = 128 slots of a
// block, K = 32G heads of dS' plus 32G heads of P.  A = [Q^T | dO^T] chunk
// (MN-major, from q/dout by 3-D TMA), B = the (token, block) scratch tile
// written by k_bwd_dq (MN-major).  With d on the TMEM lanes, each warp-level
// atomic adds 128 contiguous bytes of one KV row, and there is one partial per
// valid slot, however many head groups there are.
namespace dkv {
constexpr int kDrainWarps = 16;             // 4 per sub-partition, 32 slots each
constexpr int kThreads = (kDrainWarps + 2) * 32;
constexpr int kTmaWarp = kDrainWarps, kMmaWarp = kDrainWarps + 1;
constexpr int kBTile = 64 * 4 * 128 * 2;    // up to 256 rows x 128 slots bf16 = 64 KB
constexpr int kAStage = 4 * 128 * 128;      // Q and dO, 2 boxes each of up to 128 heads x 64 d
constexpr int kOffB = 0;
constexpr int kOffA = kOffB + kBTile;       // 2 stages
// Drain staging: per slot quarter, 16 slots x 128 d fp32, so that one warp
// reduction covers 128 contiguous floats of one KV row.
constexpr int kStageQ = 16 * 128 * 4;
constexpr int kOffStage = kOffA + 2 * kAStage;
constexpr int kOffMisc = kOffStage + 4 * kStageQ;
constexpr uint32_t kTmemCols = 256;         // 2 accumulators of 128 columns

struct Misc {
  uint64_t b_full, b_empty, a_full[2], a_empty[2], d_full[2], d_empty[2], mma_done;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffA % 1024 == 0, "alignment");
}  // namespace dkv

// kDet: the accumulator is int64 in units of 2^-32 and the adds are integer
// adds, so the sum does not depend on their order (bitwise reproducible).
template <bool kDet, int kD>
__global__ void __launch_bounds__(dkv::kThreads, 1)
k_bwd_dkv(const __grid_constant__ CUtensorMap tm_qa, const __grid_constant__ CUtensorMap tm_doa,
          const __grid_constant__ CUtensorMap tm_spb, const int32_t* __restrict__ idxc,
          const int32_t* __restrict__ count, void* __restrict__ dkv_acc, int T, int H, int W,
          int G, int box_heads, int nbmax) {
  using dkv::kDrainWarps;
  using dkv::kTmaWarp;
  using dkv::kMmaWarp;
  using dkv::kOffB;
  using dkv::kOffA;
  using dkv::kAStage;
  constexpr int kNT = (kD + 127) / 128;  // 128-row d tiles (the last may be a 64-row rope tile)
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (tid == 0) atomicCAS(&g_err_bwd, 0u, 0x3FFu);
    return;
  }
  // CTA c takes tokens c, c + gridDim.x, ... (one token each when the grid
  // is T); barrier phases follow running counts of blocks and of (block,
  // d tile) units, so with fewer CTAs the TMA warp loads the next token's
  // tiles while the drain finishes this one.
  dkv::Misc& m = *reinterpret_cast<dkv::Misc*>(smem + dkv::kOffMisc);
  const FailState fs{&g_err_bwd, &m.abort_flag};
  const int HP = 32 * G;                          // padded head rows per half
  const uint32_t a_half = static_cast<uint32_t>(HP) * 128;  // one 64-d box of HP rows
  const uint32_t b_half = static_cast<uint32_t>(2 * HP) * 128;  // one 64-slot box

  if (tid == 0) {
    mbar_init(smem_u32(&m.b_full), 1);
    mbar_init(smem_u32(&m.b_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&m.a_full[i]), 1);
      mbar_init(smem_u32(&m.a_empty[i]), 1);
      mbar_init(smem_u32(&m.d_full[i]), 1);
      mbar_init(smem_u32(&m.d_empty[i]), kDrainWarps * 32);
    }
    mbar_init(smem_u32(&m.mma_done), 1);
    m.abort_flag = 0;
    mbar_init_fence();
  }
  // A rows past H inside the padded head range stay zero (the TMA box covers
  // only H rows): the matching scratch rows are zero, and 0 * garbage could
  // be NaN.
  if (box_heads < HP) {
    for (int i = tid; i < 2 * 4 * (HP - box_heads) * 8; i += dkv::kThreads) {
      const int per = (HP - box_heads) * 8;
      const int sb = i / per, rem = i - sb * per;  // sb: stage * 4 + box
      const int row = box_heads + rem / 8, pc = rem & 7;
      const uint32_t base = sbase + kOffA + (sb >> 2) * kAStage + (sb & 3) * a_half;
      asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(base + sw128_off(row, pc)),
                   "r"(0u)
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  if (warp == kMmaWarp) tmem_alloc(smem_u32(&m.tmem_base), dkv::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;
  const size_t spr = static_cast<size_t>(2 * HP);

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int gb = 0;  // blocks so far
      for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const int Kt = count[t];
        if (Kt == 0) continue;
        const int nblk = (Kt + kBlk - 1) / kBlk;
        for (int b = 0; b < nblk; ++b, ++gb) {
          if (gb > 0) mbar_wait(smem_u32(&m.b_empty), (gb - 1) & 1, fs, 20);
          mbar_arrive_expect_tx(smem_u32(&m.b_full), 2 * b_half);
          const int row0 = static_cast<int>((static_cast<size_t>(t) * nbmax + b) * spr);
          const uint64_t pol = l2_evict_first();
          tma_load_2d_hint(sbase + kOffB, &tm_spb, 0, row0, smem_u32(&m.b_full), pol);
          tma_load_2d_hint(sbase + kOffB + b_half, &tm_spb, 64, row0, smem_u32(&m.b_full), pol);
          for (int n = 0; n < kNT; ++n) {
            const int u = gb * kNT + n, st = u & 1, use = u >> 1;
            if (use > 0) mbar_wait(smem_u32(&m.a_empty[st]), (use - 1) & 1, fs, 21);
            const uint32_t base = sbase + kOffA + st * kAStage;
            const int nd = n < 4 ? 2 : 1;  // 64-d boxes in this chunk
            const uint32_t bytes = (n < 4 ? 4u : 1u) * box_heads * 128u;
            mbar_arrive_expect_tx(smem_u32(&m.a_full[st]), bytes);
            for (int k = 0; k < nd; ++k)
              tma_load_3d(base + k * a_half, &tm_qa, n * 128 + k * 64, 0, t,
                          smem_u32(&m.a_full[st]));
            if (n < 4)
              for (int k = 0; k < 2; ++k)
                tma_load_3d(base + (2 + k) * a_half, &tm_doa, n * 128 + k * 64, 0, t,
                            smem_u32(&m.a_full[st]));
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t id = idesc_bf16(128, kBlk, true, true);
      int gb = 0;
      for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const int Kt = count[t];
        if (Kt == 0) continue;
        const int nblk = (Kt + kBlk - 1) / kBlk;
        for (int b = 0; b < nblk; ++b, ++gb) {
          mbar_wait(smem_u32(&m.b_full), gb & 1, fs, 22);
          for (int n = 0; n < kNT; ++n) {
            const int u = gb * kNT + n, st = u & 1, use = u >> 1;
            mbar_wait(smem_u32(&m.a_full[st]), use & 1, fs, 23);
            if (use > 0) mbar_wait(smem_u32(&m.d_empty[st]), (use - 1) & 1, fs, 24);
            tc_fence_after();
            const uint32_t base = sbase + kOffA + st * kAStage;
            const uint32_t d_t = tmem + st * kBlk;
            // dS' . Q part: A = Q^T (M = d), B = scratch rows 0..HP-1
            for (int kk = 0; kk < HP / 16; ++kk) {
              const uint64_t a = sdesc_sw128(base + kk * 2048, a_half, 1024);
              const uint64_t bb = sdesc_sw128(sbase + kOffB + kk * 2048, b_half, 1024);
              umma_ss(d_t, a, bb, id, kk != 0);
            }
            if (n < 4) {  // P . dO part: A = dO^T, B = scratch rows HP..2HP-1
              for (int kk = 0; kk < HP / 16; ++kk) {
                const uint64_t a = sdesc_sw128(base + 2 * a_half + kk * 2048, a_half, 1024);
                const uint64_t bb =
                    sdesc_sw128(sbase + kOffB + HP * 128 + kk * 2048, b_half, 1024);
                umma_ss(d_t, a, bb, id, 1);
              }
            }
            umma_commit(smem_u32(&m.a_empty[st]));
            umma_commit(smem_u32(&m.d_full[st]));
          }
          umma_commit(smem_u32(&m.b_empty));
        }
      }
      if (gb > 0) {  // all MMAs retired before the TMEM is freed
        umma_commit(smem_u32(&m.mma_done));
        mbar_wait_final<&g_err_bwd>(smem_u32(&m.mma_done), 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ drain
    // Warp w reads TMEM lanes 32 (w % 4) .. +31 (d rows of the chunk) and
    // slot columns 32 (w / 4) .. +31.
    const int sp = warp & 3, quarter = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    const uint64_t keep = l2_evict_last();
    int gb = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      const int Kt = count[t];
      if (Kt == 0) continue;
      const int nblk = (Kt + kBlk - 1) / kBlk;
      const int32_t* rows = idxc + static_cast<size_t>(t) * W;
      for (int b = 0; b < nblk; ++b, ++gb) {
        const int s0 = b * kBlk + quarter * 32;
        const int nvalid = max(0, min(32, Kt - s0));
        // Lane s holds the accumulator offset of slot s0 + s; shuffles hand it
        // to the whole warp without a shared-memory round trip per add.
        const uint32_t roff = lane < nvalid ? static_cast<uint32_t>(rows[s0 + lane]) * kD : 0u;
        for (int n = 0; n < kNT; ++n) {
          const int u = gb * kNT + n, st = u & 1, use = u >> 1;
          mbar_wait(smem_u32(&m.d_full[st]), use & 1, fs, 25);
          tc_fence_after();
          uint32_t v[32];
          tmem_ld32_sync(tmem + lane_base + st * kBlk + quarter * 32, v);
          tc_fence_before();
          mbar_arrive(smem_u32(&m.d_empty[st]));
          const int d = n * 128 + sp * 32 + lane;
          if (kDet && (n < 4 || d < kD)) {
            {
              unsigned long long* dst = static_cast<unsigned long long*>(dkv_acc) + d;
#pragma unroll
              for (int s = 0; s < 32; ++s) {
                const uint32_t o = __shfl_sync(0xffffffffu, roff, s);
                if (s < nvalid) red_add_fixed32(dst + o, __uint_as_float(v[s]), keep);
              }
            }
          }
          if constexpr (!kDet) {
            // The quarter's four warps hold d rows 32 sp .. of the tile for the
            // same 32 slots.  Through shared memory, 16 slots at a time, each
            // warp then adds whole 128-float rows: 4 slots per warp, 32 lanes x
            // 4 floats each (the fast reduction pattern).
            float* stg = reinterpret_cast<float*>(smem + dkv::kOffStage) + quarter * (16 * 128);
            const int dt = n * 128;  // first d of the tile
            const bool lane_ok = dt + lane * 4 < kD;  // the rope tile has 64 columns
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int s = 0; s < 16; ++s) stg[s * 128 + sp * 32 + lane] = __uint_as_float(v[half * 16 + s]);
              named_bar_sync(1 + quarter, 128);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int sl = sp * 4 + j;            // slot within the half
                const int s = half * 16 + sl;         // slot within the quarter
                const float4 f = *reinterpret_cast<const float4*>(stg + sl * 128 + lane * 4);
                const uint32_t o = __shfl_sync(0xffffffffu, roff, s);
                if (s < nvalid && lane_ok)
                  red_add_v4_f32_hint(static_cast<float*>(dkv_acc) + o + dt + lane * 4, f, keep);
              }
              named_bar_sync(1 + quarter, 128);
            }
          }
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, dkv::kTmemCols);
}

// ------------------------------------------------------------------ casts and reductions

__global__ void __launch_bounds__(256)
k_dkv_cast(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dkv, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 o;
  o.x = pack_bf16x2(a.x, a.y);
  o.y = pack_bf16x2(a.z, a.w);
  o.z = pack_bf16x2(b.x, b.y);
  o.w = pack_bf16x2(b.z, b.w);
  reinterpret_cast<uint4*>(dkv)[i] = o;
}

// The fixed-point accumulator (int64, units of 2^-32) -> bf16 dkv.
__global__ void __launch_bounds__(256)
k_dkv_cast_fixed(const long long* __restrict__ acc, __nv_bfloat16* __restrict__ dkv, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  float f[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = fixed32_to_float(acc[8 * i + j]);
  uint4 o;
  o.x = pack_bf16x2(f[0], f[1]);
  o.y = pack_bf16x2(f[2], f[3]);
  o.z = pack_bf16x2(f[4], f[5]);
  o.w = pack_bf16x2(f[6], f[7]);
  reinterpret_cast<uint4*>(dkv)[i] = o;
}

// d_sink[h] = sum over t of the per-row terms, in a fixed order (deterministic).
__global__ void __launch_bounds__(256)
k_dsink(const float* __restrict__ dsink_t, float* __restrict__ dsink, int T, int H) {
  __shared__ float red[256];
  const int h = blockIdx.x;
  float acc = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) acc += dsink_t[static_cast<size_t>(t) * H + h];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsink[h] = red[0];
}

}  // namespace

cudaError_t launch_compact(const Problem& p, const int32_t* idx, const int32_t* len,
                           int32_t* idx_out, int32_t* count_out, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  k_compact<<<p.T, kCompactThreads, 0, s>>>(idx, len, idx_out, count_out, p.W, p.S_kv, p.cu_q,
                                            p.cu_kv, p.B);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                       const int32_t* len, const float* sink, const void* out, const float* lse,
                       const void* dout, void* dq, void* dkv, float* dsink, void* ws,
                       cudaStream_t s, int stages) {
  static std::atomic<uint64_t> attr_done{0};
  const int dev = current_device();
  if (device_needs_setup(attr_done, dev)) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_dq<576, 64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqLayout<576, 64>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_bwd_dq<512, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DqLayout<512, 64>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_bwd_dq<576, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DqLayout<576, 32>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_bwd_dq<512, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DqLayout<512, 32>::kSmemBytes);
    void (*dkv_kernels[])(CUtensorMap, CUtensorMap, CUtensorMap, const int32_t*, const int32_t*,
                          void*, int, int, int, int, int, int) = {
        k_bwd_dkv<false, 576>, k_bwd_dkv<true, 576>, k_bwd_dkv<false, 512>, k_bwd_dkv<true, 512>};
    for (auto k : dkv_kernels)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
    if (e != cudaSuccess) return e;
    mark_device_setup(attr_done, dev);
  }
  const BwdWorkspace L = bwd_workspace_layout(p);
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* acc = base + L.dkv_acc;
  int32_t* idxc = reinterpret_cast<int32_t*>(base + L.idxc);
  int32_t* count = reinterpret_cast<int32_t*>(base + L.count);
  float* lse2 = reinterpret_cast<float*>(base + L.lse2);
  float* gate = reinterpret_cast<float*>(base + L.gate);
  float* delta = reinterpret_cast<float*>(base + L.delta);
  float* dsink_t = reinterpret_cast<float*>(base + L.dsink_t);
  const size_t acc_bytes = static_cast<size_t>(p.S_kv) * p.d_qk * (p.deterministic ? 8 : 4);
  cudaError_t e = cudaSuccess;
  if (stages & kBwdPre) {
    e = cudaMemsetAsync(acc, 0, acc_bytes, s);
    if (e != cudaSuccess) return e;
    if (p.T > 0) {
      e = launch_compact(p, idx, len, idxc, count, s);
      if (e != cudaSuccess) return e;
      const long long rows = static_cast<long long>(p.T) * p.H;
      k_bwd_pre<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse,
          sink, count, lse2, gate, delta, dsink_t, p.T, p.H, p.delta_residual ? 1 : 0);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  if ((stages & kBwdMain) && p.T > 0) {
    const int G32 = bwd_groups(p.H), nbmax = bwd_nbmax(p.W);
    // 64-head items, or 32-head items when that is all there is
    const int hg = p.H <= 32 ? 32 : 64;
    const int G = (p.H + hg - 1) / hg;
    __nv_bfloat16* sp = reinterpret_cast<__nv_bfloat16*>(base + L.sp);
    const long long sp_rows = static_cast<long long>(p.T) * nbmax * 64 * G32;
    CUtensorMap tm_q, tm_do, tm_sp_st, tm_kv;
    const int box_heads = p.H < hg ? p.H : hg;  // never larger than the tensor
    e = make_head_tile_map(&tm_q, q, p.T, p.H, p.d_qk, box_heads);
    if (e == cudaSuccess) e = make_head_tile_map(&tm_do, dout, p.T, p.H, kDv, box_heads);
    if (e == cudaSuccess) e = make_matrix_map(&tm_sp_st, sp, sp_rows, kBlk, 32);
    if (e == cudaSuccess) e = make_matrix_map(&tm_kv, kv, p.S_kv, p.d_qk, kBlk);
    if (e != cudaSuccess) return e;
    auto kern = hg == 32 ? (p.d_qk == 512 ? k_bwd_dq<512, 32> : k_bwd_dq<576, 32>)
                         : (p.d_qk == 512 ? k_bwd_dq<512, 64> : k_bwd_dq<576, 64>);
    const int smem = hg == 32 ? (p.d_qk == 512 ? DqLayout<512, 32>::kSmemBytes
                                               : DqLayout<576, 32>::kSmemBytes)
                              : (p.d_qk == 512 ? DqLayout<512, 64>::kSmemBytes
                                               : DqLayout<576, 64>::kSmemBytes);
    // persistent: at most one CTA per SM, each walking its share of the items
    const long long items = static_cast<long long>(p.T) * G;
    const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
    kern<<<grid, kThreads, smem, s>>>(
        tm_q, tm_do, tm_sp_st, tm_kv, static_cast<const __nv_bfloat16*>(kv), idxc, count, lse2,
        gate,
        delta, static_cast<__nv_bfloat16*>(dq), p.T, p.H, p.W, p.scale, G, G32, box_heads, nbmax);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if ((stages & kBwdFinal) && p.T > 0) {
    const int G = bwd_groups(p.H), nbmax = bwd_nbmax(p.W);
    __nv_bfloat16* sp = reinterpret_cast<__nv_bfloat16*>(base + L.sp);
    const long long sp_rows = static_cast<long long>(p.T) * nbmax * 64 * G;
    CUtensorMap tm_qa, tm_doa, tm_sp_ld;
    const int HP = 32 * G;
    const int box_all = p.H < HP ? p.H : HP;
    e = make_head_tile_map(&tm_qa, q, p.T, p.H, p.d_qk, box_all);
    if (e == cudaSuccess) e = make_head_tile_map(&tm_doa, dout, p.T, p.H, kDv, box_all);
    if (e == cudaSuccess) e = make_matrix_map(&tm_sp_ld, sp, sp_rows, kBlk, 2 * HP);
    if (e != cudaSuccess) return e;
    auto kern = p.d_qk == 512 ? (p.deterministic ? k_bwd_dkv<true, 512> : k_bwd_dkv<false, 512>)
                              : (p.deterministic ? k_bwd_dkv<true, 576> : k_bwd_dkv<false, 576>);
    // One CTA per token lets the hardware balance the uneven token costs
    // (measured faster for the fp32 path); the int64 path gains more from
    // persistent CTAs that prefetch the next token.
    const int grid = p.deterministic && p.T > sm_count() ? sm_count() : p.T;
    kern<<<grid, dkv::kThreads, dkv::kSmemBytes, s>>>(
        tm_qa, tm_doa, tm_sp_ld, idxc, count, acc, p.T, p.H, p.W, G, box_all, nbmax);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdFinal) {
    const long long n8 = static_cast<long long>(p.S_kv) * p.d_qk / 8;
    if (p.deterministic)
      k_dkv_cast_fixed<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(
          static_cast<const long long*>(acc), static_cast<__nv_bfloat16*>(dkv), n8);
    else
      k_dkv_cast<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(
          static_cast<const float*>(acc), static_cast<__nv_bfloat16*>(dkv), n8);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (dsink != nullptr) {
      k_dsink<<<p.H, 256, 0, s>>>(dsink_t, dsink, p.T, p.H);
      e = cudaGetLastError();
    }
  }
  return e;
}

unsigned int bwd_take_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_bwd, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v) cudaMemcpyToSymbol(g_err_bwd, &zero, sizeof(zero));
  return v;
}

}  // namespace dsa
