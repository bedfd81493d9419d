// Sparse MLA (DSA) backward for sm_103a.
//
// Kernels, queued in order on the caller's stream:
//   memset      dkv accumulator <- 0 (fp32, or int64 fixed point)
//   k_compact   a1: valid KV rows of every token, in slot order, and counts
//   k_bwd_dq    b1-b5: per (token, 64-head group; 32 heads when H <= 32)
//               delta_a = rowsum(dout * out) (the FlashAttention "dpsum"
//               preprocess, formed by the softmax warps one item ahead while
//               the current item's last S / dP GEMMs run), recompute P, form
//               dS, accumulate dQ in TMEM and store dq with the exact-delta
//               correction; write the dS' and P tiles of every 128-slot block
//               to a bf16 scratch.  Persistent CTAs, twice as many as SMs,
//               walk the (token, group) items.
//   k_bwd_dkv   b6: per token, dKV_blk^T = [Q^T | dO^T] [dS''; P] over all
//               heads at once (dS'' = dS' - c P, the exact-delta fixup),
//               scatter-added into the fp32 accumulator; persistent CTAs,
//               twice as many as SMs, walk the tokens
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
  if (p.deterministic) {  // the range bound per KV row, zeroed with the accumulator
    w.det_count = off; off = up(off + static_cast<size_t>(p.S_kv) * 4);
    w.det_max = off;   off = up(off + 4);
  }
  w.zero_bytes = off;
  w.idxc = off;    off = up(off + static_cast<size_t>(p.T) * p.W * 4);
  w.count = off;   off = up(off + static_cast<size_t>(p.T) * 4);
  w.delta = off;   off = up(off + TH * 4);
  w.dsink_t = off; off = up(off + TH * 4);
  w.cfix = off;    off = up(off + TH * 4);
  w.sp = off;
  off = up(off + static_cast<size_t>(p.T) * bwd_nbmax(p.W) * 64 * bwd_groups(p.H) * 128 * 2);
  w.total = off;
  return w;
}

namespace {

__device__ unsigned int g_err_bwd;

// ------------------------------------------------------------------ a1

constexpr int kCompactThreads = 256;

// With `row_refs` (deterministic mode), also counts how many valid slots name
// each KV row: the number of adds every element of that row receives.
__global__ void __launch_bounds__(kCompactThreads)
k_compact(const int32_t* __restrict__ topk_idxs, const int32_t* __restrict__ topk_length,
          int32_t* __restrict__ idx_out, int32_t* __restrict__ count_out, int W, int S_kv,
          const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int B,
          unsigned int* __restrict__ row_refs) {
  __shared__ int warp_counts[kCompactThreads / 32];
  const int t = blockIdx.x;
  const int len = slot_len(topk_length, t, W);
  const KvRange kvr = kv_range(cu_q, cu_kv, B, t, S_kv);
  int32_t* list = idx_out + static_cast<size_t>(t) * W;
  const int n = compact_token(topk_idxs + static_cast<size_t>(t) * W, W, len, kvr, list, W,
                              warp_counts, threadIdx.x, kCompactThreads);
  if (threadIdx.x == 0) count_out[t] = n;
  if (row_refs != nullptr)  // the list is complete: compact_token ends on a barrier
    for (int i = threadIdx.x; i < n; i += kCompactThreads) atomicAdd(row_refs + list[i], 1u);
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
constexpr int kOnesBytes = 2048;         // bf16 ones: two 8-slot groups of 128-byte rows

// Head group of an item: 64 heads, or 32 when H <= 32 (less padding: the
// Q/dO ring stages halve and the MMAs narrow).
template <int kHG>
struct DqHeads {
  static_assert(kHG == 64 || kHG == 32, "head group");
  static constexpr int kHT = kHG / 2;          // heads per softmax thread
  static constexpr int kHChunk = kHG * 128;    // 64 columns of kHG head rows
  static constexpr int kStage = 2 * kHChunk;   // Q chunk x (rows 0..kHG-1), then dO chunk x
  static constexpr int kStages = kHG == 64 ? 4 : 8;  // ring of (Q, dO) chunk pairs
  // TMEM: [S^T | dP^T] (2 x kHG columns), then dQ^T (kHG columns per 128-row
  // d tile).  The tile after the four V tiles is the rope tile (D = 576),
  // 2 x kHG wide: its second half accumulates KV_rope^T . P^T.  At D = 512
  // the same columns hold sigma, the per-head sum of the stored dS'.
  static constexpr uint32_t kColS = 0, kColdP = kHG, kColdQ = 2 * kHG;
  static constexpr uint32_t kColTail = kColdQ + 4 * kHG;
};

struct Misc {
  uint64_t kv_full[kChunks];
  uint64_t kv_free[kChunks];
  uint64_t qd_full[kMaxStages], qd_free[kMaxStages];
  uint64_t s_full, ds_full, dsp_free, dq_full, mma_done;
  // per head of the item: (log2(gate) - lse * log2(e), delta), so that
  // P = exp2(s * scale * log2(e) + x) and one 16-byte load serves two heads;
  // in the epilogue: (sigma, c)
  alignas(16) float2 cd[kMaxHG];
  uint32_t tmem_base;
  int abort_flag;
};

// Shared-memory layout for rows of kD columns (576 = 512 V + 64 rope, or 512).
// With a rope chunk, position p of the gathered block holds d-chunk x(p):
// p = 0 the rope columns 512..575, p = 1..8 the V chunks 0..7; blocks are
// gathered and consumed in the order p = 1..8, 0.  Without one, position p
// holds V chunk p.
// Q and dO do not stay resident: their chunk x comes in by TMA into a ring
// stage for each S / dP step (64-head items with a rope chunk keep three
// stages, so that P has a tile of its own beside dS').
// The dS'/P tile is two 64-slot halves, each kHG dS' rows followed by kHG P
// rows (128B-swizzled, slots contiguous): K-major B of the dQ MMAs (the
// rope tile reads both row sets as one N = 2 kHG operand) and the source of
// the scratch stores.
// The ones tile is the A operand of the rows that sum dS' over the slots:
// the rope tile's filler rows (D = 576, placed above the KV tile so that
// every step's LBO reaches it) or a tile of its own (D = 512, placed first).
template <int kD, int kHG>
struct DqLayout {
  using Hd = DqHeads<kHG>;
  static constexpr int kHChunk = Hd::kHChunk, kStage = Hd::kStage;
  static constexpr int kCh = kD / 64;
  static constexpr bool kRope = kCh > 8;
  static constexpr int kStages = (kRope && kHG == 64) ? 3 : Hd::kStages;
  static constexpr int kDT = (kD + 127) / 128;   // 128-row d tiles of dQ^T
  static constexpr int kOffKV = kRope ? 0 : kOnesBytes;
  static constexpr int kOffQD = kOffKV + kCh * kKVChunk;
  static constexpr int kOffSP = kOffQD + kStages * kStage;
  static constexpr int kOffOnes = kRope ? kOffSP + 4 * kHChunk : 0;
  static constexpr int kOffMisc = kRope ? kOffOnes + kOnesBytes : kOffSP + 4 * kHChunk;
  static constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQD % 1024 == 0 && kOffSP % 1024 == 0 && kOffOnes % 1024 == 0, "alignment");
  // The rope tile's LBO (filler rows -> ones tile) must fit the descriptor's
  // 14-bit field of 16-byte units.
  static_assert(!kRope || kOffOnes - kOffKV < (1 << 18), "LBO range");
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

// Byte offset of element (row, slot) of the dS'/P tile: rows 0..kHG-1 are
// the heads' dS', rows kHG..2 kHG-1 their P; each 64-slot half is a
// 128B-swizzled [2 kHG rows x 64 slots] tile (stored to the scratch by TMA,
// 32 rows x 64 slots per box).
template <int kHG>
__device__ __forceinline__ uint32_t hs_tile_off(uint32_t r, uint32_t slot) {
  const uint32_t col = slot & 63u;
  return (slot >> 6) * (2u * kHG * 128u) + r * 128u +
         ((((col >> 3) ^ (r & 7u)) << 4) | ((col & 7u) << 1));
}

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Items are (token, kHG-head group) pairs; the scratch keeps its rows per
// 32-head group (G32 groups: dS' rows first, then P rows).
//
// Exact delta without a second pass.  dS' is formed with delta_a, the delta
// of the bf16 out (item_delta below).  The exact delta, sum_j P_j dP_j in fp32, is
// the one the cuDNN page "DSA backward SM90: fix three top-k and
// attention-sink boundary failures" ("Not addressed") measures as the
// accurate form; that page notes it needs every P_j dP_j before any dS_j.
// Here the gradients are linear in delta, so it is applied afterwards:
//   sigma_h = sum_j dS'_j            (fp32 dS': the MMA sums the stored bf16
//                                     dS' through rows of a ones tile, and the
//                                     softmax threads add the bf16 rounding
//                                     remainders they kept)
//   c_h     = sigma_h - scale * delta_a * p_sink = scale * (delta - delta_a)
//   dq      = sum_j dS'_j KV_j - c_h [out, sum_j P_j KV_j[512:]]
//   dS''_j  = dS'_j - c_h P_j        (k_bwd_dkv, before its dKV GEMM)
//   dsink  += -p_sink (delta - delta_a)
// The first-order terms of the bf16 rounding of out drop out, which matters
// where the attention is one-hot and dS is all rounding noise.
template <int kD, int kHG>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_dq(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
         const __grid_constant__ CUtensorMap tm_sp, const __grid_constant__ CUtensorMap tm_kv,
         const __nv_bfloat16* __restrict__ kv,
         const int32_t* __restrict__ idxc, const int32_t* __restrict__ count,
         const float* __restrict__ lse, const float* __restrict__ sink,
         const __nv_bfloat16* __restrict__ dout, int residual, const __nv_bfloat16* __restrict__ out,
         float* __restrict__ delta_g,
         float* __restrict__ dsink_t, float* __restrict__ cfix_g,
         __nv_bfloat16* __restrict__ dq, int T, int H, int W,
         float scale, int G, int G32, int box_heads, int nbmax) {
  using L = DqLayout<kD, kHG>;
  using Hd = DqHeads<kHG>;
  constexpr int kCh = L::kCh, kDT = L::kDT, kOffKV = L::kOffKV, kOffQD = L::kOffQD,
                kOffSP = L::kOffSP, kOffOnes = L::kOffOnes, kOffMisc = L::kOffMisc;
  constexpr int kHChunk = Hd::kHChunk, kStage = Hd::kStage, kStages = L::kStages, kHT = Hd::kHT;
  constexpr uint32_t kColS = Hd::kColS, kColdP = Hd::kColdP, kColdQ = Hd::kColdQ,
                     kColTail = Hd::kColTail;
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
  // The ones tile (bf16 1.0 = 0x3F80).
  for (int i = tid; i < kOnesBytes / 16; i += kThreads)
    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + kOffOnes + i * 16),
                 "r"(0x3F803F80u)
                 : "memory");
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
        // the item's out rows, read by the dq correction at its end
        bulk_prefetch_l2(out + (static_cast<size_t>(t) * H + h0) * kDv,
                         static_cast<uint32_t>(min(kHG, H - h0)) * kDv * 2u);
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
    // The issuing thread's bookkeeping sits between MMAs: ring stages are
    // followed incrementally and descriptors stepped by constants (the start
    // address field counts 16-byte units).
    if (lane == 0) {
      const uint32_t idSdP = idesc_bf16(128, 2 * kHG, false, false);  // [S^T | dP^T]
      const uint32_t idS = idesc_bf16(128, kHG, false, false);         // S^T, rope part
      const uint32_t idQ = idesc_bf16(128, kHG, true, false);  // dQ^T: A MN-major, B K-major
      const uint32_t idQ2 = idesc_bf16(128, 2 * kHG, true, false);  // rope tile: B = [dS'; P]
      const uint32_t kvfull0 = smem_u32(&m.kv_full[0]), kvfree0 = smem_u32(&m.kv_free[0]);
      const uint32_t qdfull0 = smem_u32(&m.qd_full[0]), qdfree0 = smem_u32(&m.qd_free[0]);
      const uint64_t dkv0 = sdesc_sw128(sbase + kOffKV, 16, 1024);   // KV chunk, K-major
      const uint64_t dqd0 = sdesc_sw128(sbase + kOffQD, 16, 1024);   // (Q, dO) stage, K-major
      const uint64_t dsp0 = sdesc_sw128(sbase + kOffSP, 16, 1024);   // [dS'; P], K-major
      int it = 0, gb = 0;
      int qs = 0, qn = 0;  // ring stage of the next S / dP step and its fill count
      for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
        const int t = u / G;
        const int Kt = count[t];
        if (Kt == 0) continue;
        const int nblk = (Kt + kBlk - 1) / kBlk;
        for (int b = 0; b < nblk; ++b, ++gb) {
#pragma unroll
          for (int i = 0; i < kCh; ++i) {
            const int pos = pos_of_step<kRope>(i);
            mbar_wait(kvfull0 + 8 * pos, gb & 1, fs, 3);
            mbar_wait(qdfull0 + 8 * qs, qn & 1, fs, 2);
            fence_proxy_async_smem();  // cp.async (generic proxy) -> UMMA (async proxy)
            tc_fence_after();
            // V chunks: S and dP in one N = 128 MMA (B rows: the Q heads, then
            // the dO heads); the rope chunk adds to S only.
            const uint64_t a0 = dkv0 + static_cast<uint64_t>(pos * (kKVChunk >> 4));
            const uint64_t b0 = dqd0 + static_cast<uint64_t>(qs * (kStage >> 4));
            const uint32_t id = dchunk_of_pos<kRope>(pos) < 8 ? idSdP : idS;
#pragma unroll
            for (int k = 0; k < 4; ++k) umma_ss(tmem + kColS, a0 + 2 * k, b0 + 2 * k, id, (i | k) != 0);
            umma_commit(qdfree0 + 8 * qs);
            if (++qs == kStages) { qs = 0; ++qn; }
          }
          umma_commit(smem_u32(&m.s_full));
          // dS' and P of this block; for the first block of an item this also
          // orders the softmax warps' read-out of the previous dQ^T first
          mbar_wait(smem_u32(&m.ds_full), gb & 1, fs, 4);
          tc_fence_after();
          // dQ^T chunks: rope first, then d rows 0..511.  The rope tile's B
          // is [dS'; P] (N = 2 kHG), so its second half accumulates
          // KV_rope^T . P^T; its 64 filler rows (d 576..639) read the ones
          // tile, so they accumulate sigma = sum over slots of dS' (and of P).
          // (Its LBO reaches the ones tile from each step's start, so the LBO
          // field falls by what the start field gains.)
#pragma unroll 1
          for (int jj = 0; jj < kDT; ++jj) {
            const int j = kRope ? ((jj == 0) ? 4 : jj - 1) : jj;
            const int pos0 = (j == 4) ? 0 : (kRope ? 1 + 2 * j : 2 * j);
            const uint32_t a_addr = kOffKV + pos0 * kKVChunk;
            const uint64_t da = (j == 4) ? sdesc_sw128(sbase + a_addr, kOffOnes - a_addr, 1024)
                                         : sdesc_sw128(sbase + a_addr, kKVChunk, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t step = static_cast<uint64_t>(kk * (2048 >> 4));
              const uint64_t a = (j == 4) ? da + step - (step << 16) : da + step;
              const uint64_t bs =
                  dsp0 + static_cast<uint64_t>((kk >> 2) * ((2 * kHChunk) >> 4) + (kk & 3) * 2);
              umma_ss(tmem + kColdQ + j * kHG, a, bs, j == 4 ? idQ2 : idQ, (b | kk) != 0);
            }
            umma_commit(kvfree0 + 8 * pos0);
            if (j != 4) umma_commit(kvfree0 + 8 * (pos0 + 1));
          }
          if constexpr (!kRope) {
            // sigma without a rope tile: rows 0..63 of A are the ones tile,
            // rows 64..127 (never read) the first dS' rows.
            const uint64_t a = sdesc_sw128(sbase + kOffOnes, kOffSP - kOffOnes, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bs =
                  dsp0 + static_cast<uint64_t>((kk >> 2) * ((2 * kHChunk) >> 4) + (kk & 3) * 2);
              umma_ss(tmem + kColTail, a, bs, idQ, (b | kk) != 0);
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
    const size_t lo_off = residual ? static_cast<size_t>(T) * H * kDv : 0;  // residual half
    // delta_a = rowsum(dout * out) of an item's heads (with out's rounding
    // residual when the forward stored it): to dst[h * stride] for every head
    // of the group (0 for padded heads) when `all`, else for the real heads
    // only.  Warp w takes heads w, w + 8, ..., two per round, so that eight
    // 16-byte loads per lane are in flight; lane l reads pieces l and l + 32
    // of a row, so each warp load covers 512 contiguous bytes.  The softmax
    // warps compute the next item's values while they wait for the last
    // S / dP GEMMs of this one (and a CTA's first item's before it starts).
    auto item_delta = [&](int t, int h0, int nh, float* dst, int stride, bool all) {
      const size_t base = (static_cast<size_t>(t) * H + h0) * kDv;
      auto dot8 = [](const uint4& a, const uint4& b, float acc) {
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 fa = __bfloat1622float2(a2[k]), fb = __bfloat1622float2(b2[k]);
          acc = fmaf(fa.x, fb.x, acc);
          acc = fmaf(fa.y, fb.y, acc);
        }
        return acc;
      };
      // the out rows, then (with the residual flag) a second pass over the
      // residual rows, so that only eight loads per lane are live at a time
#pragma unroll 1
      for (int pass = 0; pass < (residual ? 2 : 1); ++pass) {
        const size_t ob = base + (pass ? lo_off : 0);
#pragma unroll
        for (int r = 0; r < kHG / 16; ++r) {
          uint4 o[2][2], d[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int hh = warp + 8 * (2 * r + j);
            const bool ok = hh < nh;
            const uint4* o4 = reinterpret_cast<const uint4*>(out + ob + static_cast<size_t>(hh) * kDv);
            const uint4* d4 = reinterpret_cast<const uint4*>(dout + base + static_cast<size_t>(hh) * kDv);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint4 z = make_uint4(0, 0, 0, 0);
              o[j][k] = ok ? __ldg(o4 + lane + 32 * k) : z;
              d[j][k] = ok ? __ldg(d4 + lane + 32 * k) : z;
            }
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float acc = dot8(o[j][1], d[j][1], dot8(o[j][0], d[j][0], 0.f));
#pragma unroll
            for (int x = 16; x > 0; x >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
            const int hh = warp + 8 * (2 * r + j);
            if (lane == 0 && (all || hh < nh)) {
              float* p = dst + hh * stride;
              *p = pass ? *p + acc : acc;
            }
          }
        }
      }
    };
    int it = 0, gb = 0;
    bool ahead = false;  // this item's delta_a is already in delta_g
    // this item's delta_a -> m.cd[h].y (0 for padded heads)
    auto load_delta = [&](int t, int h0, int nh) {
      if (ahead) {
        if (tid < kHG) m.cd[tid].y = tid < nh ? __ldcg(delta_g + static_cast<size_t>(t) * H + h0 + tid) : 0.f;
      } else {
        item_delta(t, h0, nh, &m.cd[0].y, 2, true);
      }
      ahead = false;
    };
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G, h0 = (u - t * G) * kHG;
      const int nh = min(kHG, H - h0);
      const int Kt = count[t];
      if (Kt == 0) {  // empty row: dq = 0, nothing for dkv; the sink holds the
                      // whole denominator (p_sink = 1), so dsink_t = -delta_a
        load_delta(t, h0, nh);
        named_bar_sync(1, kSoftmax);
        if (tid < nh) dsink_t[static_cast<size_t>(t) * H + h0 + tid] = -m.cd[tid].y;
        for (int v = tid; v < nh * (kD / 8); v += kSoftmax) {
          const int h = v / (kD / 8), c = v - h * (kD / 8);
          *reinterpret_cast<uint4*>(dq + (static_cast<size_t>(t) * H + h0 + h) * kD + c * 8) =
              make_uint4(0, 0, 0, 0);
        }
        named_bar_sync(1, kSoftmax);  // m.cd is rewritten at the next item's start
        continue;
      }
      const int nblk = (Kt + kBlk - 1) / kBlk;
      load_delta(t, h0, nh);
      named_bar_sync(1, kSoftmax);
      float gate_h = 0.f, dsink_h = 0.f;  // thread tid < nh: head h0 + tid, for the epilogue
      if (tid < kHG) {
        // Padded heads get gate 0, hence P = dS = 0: they add nothing anywhere.
        float x = -INFINITY;  // log2(gate) - lse * log2(e)
        if (tid < nh) {
          const size_t r = static_cast<size_t>(t) * H + h0 + tid;
          const float l = lse[r];
          const float sk = sink != nullptr ? sink[h0 + tid] : -INFINITY;
          gate_h = stable_sigmoid(l - sk);
          dsink_h = -stable_sigmoid(sk - l) * m.cd[tid].y;  // -p_sink * delta_a
          if (gate_h > 0.f) x = log2f(gate_h) - l * kLog2e;
        }
        m.cd[tid].x = x;
      }
      named_bar_sync(1, kSoftmax);
      // Per head, this row's sum over the item's blocks of the bf16 rounding
      // remainder of dS' (dS' - bf16(dS')): sigma from the MMA sums the
      // stored bf16 values, and these remainders bring it to fp32 accuracy.
      __nv_bfloat162 eacc[kHT / 2];
#pragma unroll
      for (int i = 0; i < kHT / 2; ++i) eacc[i] = __float2bfloat162_rn(0.f);
      for (int b = 0; b < nblk; ++b, ++gb) {
        if (b == nblk - 1 && u + static_cast<int>(gridDim.x) < n_items) {
          // the next item's delta_a, while this block's S / dP GEMMs run
          const int un = u + gridDim.x, tn = un / G, hn = (un - tn * G) * kHG;
          item_delta(tn, hn, min(kHG, H - hn), delta_g + static_cast<size_t>(tn) * H + hn, 1,
                     false);
          ahead = true;
        }
        mbar_wait(smem_u32(&m.s_full), gb & 1, fs, 7);
        tc_fence_after();
        const bool valid = b * kBlk + row < Kt;
        uint32_t pk[kHT / 2];  // P as bf16 pairs (heads hb + 2i, hb + 2i + 1)
        uint32_t dk[kHT / 2];  // dS' as bf16 pairs
        const float4* cd4 = reinterpret_cast<const float4*>(m.cd + hb);
        // 16 heads at a time, so that only 32 loaded TMEM values are live
#pragma unroll
        for (int hh = 0; hh < kHT; hh += 16) {
          uint32_t rs[16], rd[16];
          tmem_ld16x2_sync(tmem + lane_base + kColS + hb + hh, rs,
                           tmem + lane_base + kColdP + hb + hh, rd);
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float4 c = cd4[(hh + i) / 2];  // heads hb + hh + i, + 1
            // Live columns satisfy s - lse <= 0, so exp2 never overflows here;
            // rows past the valid count hold zero KV (finite dP) and get P = 0.
            const float p0 = valid ? ex2_approx(fmaf(__uint_as_float(rs[i]), sl2, c.x)) : 0.f;
            const float p1 = valid ? ex2_approx(fmaf(__uint_as_float(rs[i + 1]), sl2, c.z)) : 0.f;
            const float ds0 = p0 * (__uint_as_float(rd[i]) - c.y) * scale;
            const float ds1 = p1 * (__uint_as_float(rd[i + 1]) - c.w) * scale;
            const int q = (hh + i) / 2;
            pk[q] = pack_bf16x2(p0, p1);
            dk[q] = pack_bf16x2(ds0, ds1);
            const float r0 = ds0 - __uint_as_float(dk[q] << 16);
            const float r1 = ds1 - __uint_as_float(dk[q] & 0xFFFF0000u);
            eacc[q] = __hadd2(eacc[q], __floats2bfloat162_rn(r0, r1));
          }
        }
        if (gb > 0) mbar_wait(smem_u32(&m.dsp_free), (gb - 1) & 1, fs, 8);
        // thread 0 finished reading the previous block's tiles out (bulk wait below)
        named_bar_sync(1, kSoftmax);
#pragma unroll
        for (int i = 0; i < kHT / 2; ++i) {
          st_shared_b16(sbase + kOffSP + hs_tile_off<kHG>(hb + 2 * i, row),
                        static_cast<uint16_t>(dk[i]));
          st_shared_b16(sbase + kOffSP + hs_tile_off<kHG>(hb + 2 * i + 1, row),
                        static_cast<uint16_t>(dk[i] >> 16));
        }
#pragma unroll
        for (int i = 0; i < kHT / 2; ++i) {
          st_shared_b16(sbase + kOffSP + hs_tile_off<kHG>(kHG + hb + 2 * i, row),
                        static_cast<uint16_t>(pk[i]));
          st_shared_b16(sbase + kOffSP + hs_tile_off<kHG>(kHG + hb + 2 * i + 1, row),
                        static_cast<uint16_t>(pk[i] >> 16));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&m.ds_full));
        named_bar_sync(1, kSoftmax);
        if (tid == 0) {
          // dS' and P rows of this head group -> the (token, block) scratch
          // tile, in boxes of 32 heads that hold at least one real head
          const int row0 = static_cast<int>((static_cast<size_t>(t) * nbmax + b) * spr) + h0;
          const uint64_t pol = l2_evict_first();
          for (int half = 0; half < 2; ++half)
            for (int g2 = 0; g2 * 32 < nh; ++g2) {
              const uint32_t src = sbase + kOffSP + half * (2 * kHChunk) + g2 * 4096;
              tma_store_2d_hint(&tm_sp, half * 64, row0 + g2 * 32, src, pol);
              tma_store_2d_hint(&tm_sp, half * 64, row0 + 32 * G32 + g2 * 32, src + kHChunk, pol);
            }
          bulk_commit();
          bulk_wait_read();
        }
      }
      // ---------------------------------------------------------- epilogue
      // The rounding remainders, summed over this warp's 32 rows: a butterfly
      // reduce-scatter leaves lane L with head hb + (L mod kHT).
      float esum_mine;
      {
        float ev[kHT];
#pragma unroll
        for (int i = 0; i < kHT / 2; ++i) {
          ev[2 * i] = __low2float(eacc[i]);
          ev[2 * i + 1] = __high2float(eacc[i]);
        }
#pragma unroll
        for (int o = 16; o >= kHT; o >>= 1) {
#pragma unroll
          for (int i = 0; i < kHT; ++i) ev[i] += __shfl_xor_sync(0xffffffffu, ev[i], o);
        }
#pragma unroll
        for (int o = kHT / 2; o > 0; o >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < o; ++i) {
            const float keep = up ? ev[i + o] : ev[i];
            const float send = up ? ev[i] : ev[i + o];
            ev[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        esum_mine = ev[0];
      }
      // The out values of the dq correction, for this warp's 32 d rows of
      // each V tile and its kHT heads, as 16-byte pieces (lane L: piece
      // L + 32 k is head (L + 32 k) / 4, d columns 8 ((L + 32 k) % 4) ..),
      // redistributed through shared memory below.  Two tiles in flight at
      // a time (the first two while the last dQ MMAs run).
      const __nv_bfloat16* out_t = out + (static_cast<size_t>(t) * H + h0) * kDv;
      constexpr int kPieces = kHT / 8;  // per lane per tile
      auto load_out = [&](int j, uint4 (&dst)[kPieces]) {
#pragma unroll
        for (int k = 0; k < kPieces; ++k) {
          const int pc = lane + 32 * k, hh = hb + pc / 4;
          dst[k] = hh < nh ? __ldg(reinterpret_cast<const uint4*>(
                                 out_t + static_cast<size_t>(hh) * kDv + j * 128 +
                                 (warp & 3) * 32 + (pc & 3) * 8))
                           : make_uint4(0, 0, 0, 0);
        }
      };
      uint4 opc[2][kPieces];
      load_out(0, opc[0]);
      load_out(1, opc[1]);
      mbar_wait(smem_u32(&m.dq_full), it & 1, fs, 10);
      tc_fence_after();
      // The four row warps' remainder sums meet in the dS'/P tile (after the
      // out slices below, 8 warps x kHT x 64 bytes).  The tile is free once
      // thread 0 has seen the last block's scratch stores read it: its bulk
      // wait precedes this barrier.
      float* esum = reinterpret_cast<float*>(smem + kOffSP + 8 * kHT * 64);  // [4][kHG]
      named_bar_sync(1, kSoftmax);
      if (lane < kHT) esum[(warp & 3) * kHG + hb + lane] = esum_mine;
      // sigma per head: the rope tile's filler rows (64..127), or rows 0..63
      // of the separate sum tile without a rope chunk.
      if ((warp & 3) == (kRope ? 2 : 0)) {
        uint32_t v[kHT];
        if constexpr (kHT == 32)
          tmem_ld32_sync(tmem + lane_base + kColTail + hb, v);
        else
          tmem_ld16_sync(tmem + lane_base + kColTail + hb, v);
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < kHT; ++i) m.cd[hb + i].x = __uint_as_float(v[i]);
        }
      }
      named_bar_sync(1, kSoftmax);
      if (tid < kHG) {
        float c = 0.f;
        if (tid < nh) {
          const size_t r = static_cast<size_t>(t) * H + h0 + tid;
          const float sig = m.cd[tid].x + ((esum[tid] + esum[kHG + tid]) +
                                           (esum[2 * kHG + tid] + esum[3 * kHG + tid]));
          c = sig + scale * dsink_h;             // dsink_h = -p_sink * delta_a
          cfix_g[r] = c;                         // = scale * (delta - delta_a)
          const float eps = scale != 0.f ? c / scale : 0.f;
          dsink_t[r] = dsink_h - (1.f - gate_h) * eps;  // p_sink = 1 - gate
        }
        m.cd[tid].y = c;
      }
      named_bar_sync(1, kSoftmax);
      // dQ^T -> dq (bf16) straight from registers, with the delta correction:
      // for each head, a warp writes 32 consecutive d of that head's row.
      __nv_bfloat16* dq_t = dq + (static_cast<size_t>(t) * H + h0) * kD;
      // this warp's [kHT heads x 32 d] bf16 slice of out, 64 bytes per head
      const uint32_t oslice = sbase + kOffSP + warp * (kHT * 64);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int d = j * 128 + row;
#pragma unroll
        for (int k = 0; k < kPieces; ++k) {
          const int pc = lane + 32 * k;
          const uint4 x = opc[j & 1][k];
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(oslice + pc * 16), "r"(x.x),
                       "r"(x.y), "r"(x.z), "r"(x.w)
                       : "memory");
        }
        if (j < 2) load_out(j + 2, opc[j & 1]);
        __syncwarp();
        float o[kHT];
#pragma unroll
        for (int i = 0; i < kHT; ++i) {
          uint16_t b;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(b) : "r"(oslice + i * 64 + lane * 2));
          o[i] = __uint_as_float(static_cast<uint32_t>(b) << 16);
        }
        __syncwarp();  // the slice is rewritten for the next tile
        uint32_t v[kHT];
        if constexpr (kHT == 32)
          tmem_ld32_sync(tmem + lane_base + kColdQ + j * kHG + hb, v);
        else
          tmem_ld16_sync(tmem + lane_base + kColdQ + j * kHG + hb, v);
#pragma unroll
        for (int i = 0; i < kHT; ++i) {
          const int h = hb + i;
          if (h < nh)
            dq_t[static_cast<size_t>(h) * kD + d] =
                __float2bfloat16_rn(fmaf(-m.cd[h].y, o[i], __uint_as_float(v[i])));
        }
      }
      if constexpr (kRope) {
        if ((warp & 3) < 2) {  // rows 0..63: d 512..575
          const int d = 512 + row;
#pragma unroll
          for (int hh = 0; hh < kHT; hh += 16) {
            uint32_t v[16], w[16];
            tmem_ld16x2_sync(tmem + lane_base + kColTail + hb + hh, v,
                             tmem + lane_base + kColTail + kHG + hb + hh, w);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int h = hb + hh + i;
              if (h < nh)
                dq_t[static_cast<size_t>(h) * kD + d] = __float2bfloat16_rn(
                    fmaf(-m.cd[h].y, __uint_as_float(w[i]), __uint_as_float(v[i])));
            }
          }
        }
      }
      named_bar_sync(1, kSoftmax);  // m.cd is rewritten at the next item's start
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ b5-b6: dKV

// Per token (a CTA walks tokens), every head at once:
//   dKV^T[d, slot] = sum_h Q[h, d] dS'[h, slot] + sum_h dO[h, d] P[h, slot]
// M = 128 d rows per chunk (4 V chunks + the rope chunk), N = 128 slots of a
// block, K = 32G heads of dS' plus 32G heads of P.  A = [Q^T | dO^T] chunk
// (MN-major, from q/dout by 3-D TMA), B = the (token, block) scratch tile
// written by k_bwd_dq (MN-major).  With d on the TMEM lanes, each warp-level
// atomic adds 128 contiguous bytes of one KV row, and there is one partial per
// valid slot, however many head groups there are.
// Before the GEMM of a block, the fixup warps apply the delta correction of
// k_bwd_dq to the loaded tile: dS'' = dS' - c_h P per head row.
namespace dkv {
constexpr int kDrainWarps = 16;             // 4 per sub-partition, 32 slots each
constexpr int kFixWarps = 8;                // the dS' correction of each loaded tile
constexpr int kThreads = (kDrainWarps + 2 + kFixWarps) * 32;
constexpr int kTmaWarp = kDrainWarps, kMmaWarp = kDrainWarps + 1, kFixWarp0 = kDrainWarps + 2;
constexpr int kBTile = 64 * 4 * 128 * 2;    // up to 256 rows x 128 slots bf16 = 64 KB
constexpr int kAStage = 4 * 128 * 128;      // Q and dO, 2 boxes each of up to 128 heads x 64 d
constexpr int kOffB = 0;
constexpr int kOffA = kOffB + kBTile;       // 2 stages
// Drain staging: per slot quarter, 16 slots x 128 d fp32, so that one warp
// reduction covers 128 contiguous floats of one KV row.
constexpr int kStageQ = 16 * 128 * 4;
constexpr int kOffStage = kOffA + 2 * kAStage;
constexpr int kOffMisc = kOffStage + 4 * kStageQ;
constexpr uint32_t kTmemCols = 512;         // 4 accumulators of 128 columns

struct Misc {
  uint64_t b_full, b_fixed, b_empty, a_full[2], a_empty[2], d_full[4], d_empty[4], mma_done;
  float c[128];       // the token's per-head correction c_h (0 past H)
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
          const int32_t* __restrict__ count, const float* __restrict__ cfix,
          void* __restrict__ dkv_acc, unsigned int* __restrict__ row_max, int T, int H, int W,
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
    mbar_init(smem_u32(&m.b_fixed), dkv::kFixWarps * 32);
    mbar_init(smem_u32(&m.b_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&m.a_full[i]), 1);
      mbar_init(smem_u32(&m.a_empty[i]), 1);
    }
    for (int i = 0; i < 4; ++i) {
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
      // Descriptors are built once and stepped by constants (the start
      // address field counts 16-byte units); the two A stages alternate by
      // parity and the four accumulators go round in turn.
      const uint32_t id = idesc_bf16(128, kBlk, true, true);
      const uint64_t da0 = sdesc_sw128(sbase + kOffA, a_half, 1024);   // Q^T / dO^T, MN-major
      const uint64_t db0 = sdesc_sw128(sbase + kOffB, b_half, 1024);   // [dS''; P], MN-major
      const uint64_t a_dO = static_cast<uint64_t>((2 * a_half) >> 4);  // dO^T after the two Q^T boxes
      const uint64_t b_P = static_cast<uint64_t>((HP * 128) >> 4);     // P rows after the dS'' rows
      const int nk = HP / 16;
      const uint32_t afull0 = smem_u32(&m.a_full[0]), aempty0 = smem_u32(&m.a_empty[0]);
      const uint32_t dfull0 = smem_u32(&m.d_full[0]), dempty0 = smem_u32(&m.d_empty[0]);
      int gb = 0, use = 0, st = 0;  // A stage of the next d tile, and its use count
      int sd = 0, used = 0;         // accumulator of the next d tile, and its use count
      for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const int Kt = count[t];
        if (Kt == 0) continue;
        const int nblk = (Kt + kBlk - 1) / kBlk;
        for (int b = 0; b < nblk; ++b, ++gb) {
          // The P rows are final as loaded: the first tile's P . dO part runs
          // while the fixup warps still correct the dS' rows.
          mbar_wait(smem_u32(&m.b_full), gb & 1, fs, 22);
          for (int n = 0; n < kNT; ++n) {
            mbar_wait(afull0 + 8 * st, use & 1, fs, 23);
            if (used > 0) mbar_wait(dempty0 + 8 * sd, (used - 1) & 1, fs, 24);
            tc_fence_after();
            const uint64_t da = da0 + static_cast<uint64_t>((st * kAStage) >> 4);
            const uint32_t d_t = tmem + sd * kBlk;
            // P . dO part (V tiles): A = dO^T, B = scratch rows HP..2HP-1
            if (n < 4) {
              for (int kk = 0; kk < nk; ++kk)
                umma_ss(d_t, da + a_dO + 128 * kk, db0 + b_P + 128 * kk, id, kk != 0);
            }
            if (n == 0) {
              mbar_wait(smem_u32(&m.b_fixed), gb & 1, fs, 27);
              tc_fence_after();
            }
            // dS'' . Q part: A = Q^T (M = d), B = scratch rows 0..HP-1
            for (int kk = 0; kk < nk; ++kk)
              umma_ss(d_t, da + 128 * kk, db0 + 128 * kk, id, n < 4 || kk != 0);
            umma_commit(aempty0 + 8 * st);
            umma_commit(dfull0 + 8 * sd);
            st ^= 1;
            use += st == 0;
            sd = (sd + 1) & 3;
            used += sd == 0;
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
  } else if (warp >= dkv::kFixWarp0) {
    // ------------------------------------------------------------ dS' fixup
    // dS'' = dS' - c_h P on every 16-byte piece of the loaded tile: row h of
    // the dS' rows and row HP + h of the P rows share their swizzle phase, so
    // the same piece index holds the same slots in both.
    const int ftid = tid - dkv::kFixWarp0 * 32;
    constexpr int kFixThreads = dkv::kFixWarps * 32;
    int gb = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      const int Kt = count[t];
      if (Kt == 0) continue;
      const int nblk = (Kt + kBlk - 1) / kBlk;
      named_bar_sync(6, kFixThreads);  // the previous token's pieces are all done
      for (int h = ftid; h < HP; h += kFixThreads)
        m.c[h] = h < H ? cfix[static_cast<size_t>(t) * H + h] : 0.f;
      named_bar_sync(6, kFixThreads);
      for (int b = 0; b < nblk; ++b, ++gb) {
        mbar_wait(smem_u32(&m.b_full), gb & 1, fs, 26);
        // 16 HP pieces of 16 bytes (a multiple of kFixThreads, since HP is a
        // multiple of 32).  Whole rounds of four independent pieces, loads
        // first so that their latencies overlap (all of them at HP = 64 and
        // 128), then one piece at a time for the rest (HP = 32 and 96).
        const int npce = 16 * HP;
        auto piece_addr = [&](int pce, float& cp) {
          const int box = pce / (8 * HP), rem = pce - box * 8 * HP;
          cp = m.c[rem >> 3];
          return sbase + kOffB + box * b_half + rem * 16;
        };
        auto fix_piece = [&](uint32_t a, float cp, uint32_t (&dw)[4], const uint32_t (&pw)[4]) {
          if (cp == 0.f) return;  // padded heads, or nothing to correct
          // packed bf16 FMA, one rounding: -c (bf16) * P + dS'
          const __nv_bfloat162 nc = __float2bfloat162_rn(-cp);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 r =
                __hfma2(nc, *reinterpret_cast<const __nv_bfloat162*>(&pw[k]),
                        *reinterpret_cast<const __nv_bfloat162*>(&dw[k]));
            dw[k] = *reinterpret_cast<const uint32_t*>(&r);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(dw[0]), "r"(dw[1]),
                       "r"(dw[2]), "r"(dw[3])
                       : "memory");
        };
        auto ld4 = [](uint32_t a, uint32_t (&w)[4]) {
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(a));
        };
        const uint32_t p_off = static_cast<uint32_t>(HP) * 128u;  // P rows after the dS' rows
        int p0 = ftid;
        for (; p0 + 3 * kFixThreads < npce; p0 += 4 * kFixThreads) {
          uint32_t a[4], dw[4][4], pw[4][4];
          float c[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            a[u] = piece_addr(p0 + u * kFixThreads, c[u]);
            ld4(a[u], dw[u]);
            ld4(a[u] + p_off, pw[u]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) fix_piece(a[u], c[u], dw[u], pw[u]);
        }
        for (; p0 < npce; p0 += kFixThreads) {
          uint32_t dw[4], pw[4];
          float c;
          const uint32_t a = piece_addr(p0, c);
          ld4(a, dw);
          ld4(a + p_off, pw);
          fix_piece(a, c, dw, pw);
        }
        fence_proxy_async_smem();  // generic-proxy writes -> the UMMA reads
        mbar_arrive(smem_u32(&m.b_fixed));
      }
    }
  } else {
    // ------------------------------------------------------------ drain
    // Warp w reads TMEM lanes 32 (w % 4) .. +31 (d rows of the chunk) and
    // slot columns 32 (w / 4) .. +31.
    const int sp = warp & 3, quarter = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    const uint64_t keep = l2_evict_last();
    uint32_t vmax = 0;  // kDet: largest |v| added by this thread (fp32 bits)
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
          const int u = gb * kNT + n, st = u & 3, use = u >> 2;
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
                if (s < nvalid) {
                  const float f = __uint_as_float(v[s]);
                  red_add_fixed32(dst + o, f, keep);
                  // largest |v| this thread adds (non-negative floats order
                  // like their bit patterns; NaN counts as the largest)
                  vmax = max(vmax, __float_as_uint(fabsf(f)));
                }
              }
            }
          }
          if constexpr (!kDet) {
            // The quarter's four warps hold d rows 32 sp .. of the tile for the
            // same 32 slots.  Through shared memory, 16 slots at a time, each
            // warp then adds whole 128-float rows: 4 slots per warp, 32 lanes x
            // 4 floats each (the fast reduction pattern).
            float* stg = reinterpret_cast<float*>(smem + dkv::kOffStage) + quarter * (16 * 128);
            float* acc = static_cast<float*>(dkv_acc);
            if (kD > 512 && n == kNT - 1) {
              // The 64-column rope tile: only TMEM lanes 0..63 (sp 0 and 1)
              // hold its d rows.  Those two warps stage all 32 slots at once
              // (32 x 64 floats), and each reduction then covers two slots,
              // lanes 0..15 one row and lanes 16..31 the next: half the
              // staging, barriers and reductions of a full tile.
              if (sp < 2) {
#pragma unroll
                for (int s = 0; s < 32; ++s) stg[s * 64 + sp * 32 + lane] = __uint_as_float(v[s]);
              }
              named_bar_sync(1 + quarter, 128);
              const int c4 = (lane & 15) * 4;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int s = sp * 8 + 2 * j + (lane >> 4);  // slot within the quarter
                const float4 f = *reinterpret_cast<const float4*>(stg + s * 64 + c4);
                const uint32_t o = __shfl_sync(0xffffffffu, roff, s);
                if (s < nvalid) red_add_v4_f32_hint(acc + o + 512 + c4, f, keep);
              }
              named_bar_sync(1 + quarter, 128);
            } else {
              const int dt = n * 128;  // first d of the tile (a full 128-column tile)
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
                  if (s < nvalid) red_add_v4_f32_hint(acc + o + dt + lane * 4, f, keep);
                }
                named_bar_sync(1 + quarter, 128);
              }
            }
          }
        }
        __syncwarp();
      }
    }
    if constexpr (kDet) {  // one atomic per warp for the range check
      const uint32_t mx = redux_max_u32(vmax);
      if (lane == 0 && mx != 0) atomicMax(row_max, mx);
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

// The fixed-point accumulator (int64, units of 2^-32) -> bf16 dkv.  Every
// element of row r received row_refs[r] adds, each at most *vmax (the
// largest |add| of the whole call) in magnitude, so its sum stayed inside the
// accumulator's +-2^31 when their product is below 2^31; otherwise the row
// may have wrapped, and the error word says so (DSA_ERR_RANGE).
__global__ void __launch_bounds__(256)
k_dkv_cast_fixed(const long long* __restrict__ acc, __nv_bfloat16* __restrict__ dkv, long long n8,
                 const unsigned int* __restrict__ row_refs,
                 const unsigned int* __restrict__ vmax, int D) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  if ((8 * i) % D == 0) {  // first piece of a row
    const long long r = 8 * i / D;
    const float bound = static_cast<float>(row_refs[r]) * __uint_as_float(*vmax);
    if (!(bound < 2147483648.0f)) atomicCAS(&g_err_bwd, 0u, kErrDetRange);
  }
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

// ------------------------------------------------------------------ wait self-test

// Two waits on barriers that nothing completes: thread 0 with a short limit,
// thread 32 with the ordinary one.  The first gives up, records a timeout in
// the error word and raises the abort flag, which ends the second wait at its
// next check; then the kernel returns and the context stays usable.
__global__ void __launch_bounds__(64) k_wait_selftest(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  const FailState fs{&g_err_bwd, &abort_flag};
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar[0]), 0, fs, 0x30, limit_ns);
  if (threadIdx.x == 32) mbar_wait(smem_u32(&bar[1]), 0, fs, 0x31);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
  k_wait_selftest<<<1, 64, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_compact(const Problem& p, const int32_t* idx, const int32_t* len,
                           int32_t* idx_out, int32_t* count_out, cudaStream_t s,
                           unsigned int* row_refs) {
  if (p.T == 0) return cudaSuccess;
  k_compact<<<p.T, kCompactThreads, 0, s>>>(idx, len, idx_out, count_out, p.W, p.S_kv, p.cu_q,
                                            p.cu_kv, p.B, row_refs);
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
                          const float*, void*, unsigned int*, int, int, int, int, int, int) = {
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
  unsigned int* row_refs =
      p.deterministic ? reinterpret_cast<unsigned int*>(base + L.det_count) : nullptr;
  unsigned int* row_max =
      p.deterministic ? reinterpret_cast<unsigned int*>(base + L.det_max) : nullptr;
  int32_t* idxc = reinterpret_cast<int32_t*>(base + L.idxc);
  int32_t* count = reinterpret_cast<int32_t*>(base + L.count);
  float* delta = reinterpret_cast<float*>(base + L.delta);
  float* dsink_t = reinterpret_cast<float*>(base + L.dsink_t);
  float* cfix = reinterpret_cast<float*>(base + L.cfix);
  cudaError_t e = cudaSuccess;
  if (stages & kBwdPre) {
    e = cudaMemsetAsync(acc, 0, L.zero_bytes - L.dkv_acc, s);
    if (e != cudaSuccess) return e;
    if (p.T > 0) {
      e = launch_compact(p, idx, len, idxc, count, s, row_refs);
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
    // Persistent CTAs, twice as many as SMs. The shared memory holds one per
    // SM, so the second half runs as a second wave: each starts on whichever
    // SM frees first, which evens out the end of the kernel (0.6 % at the
    // 8192-token, 128-head workload).
    const long long items = static_cast<long long>(p.T) * G;
    const int grid = static_cast<int>(items < 2 * sm_count() ? items : 2 * sm_count());
    kern<<<grid, kThreads, smem, s>>>(
        tm_q, tm_do, tm_sp_st, tm_kv, static_cast<const __nv_bfloat16*>(kv), idxc, count, lse,
        sink, static_cast<const __nv_bfloat16*>(dout), p.delta_residual ? 1 : 0,
        static_cast<const __nv_bfloat16*>(out), delta, dsink_t, cfix,
        static_cast<__nv_bfloat16*>(dq), p.T, p.H, p.W, p.scale, G, G32, box_heads, nbmax);
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
    // Persistent CTAs walking the tokens, twice as many as SMs: the TMA warp
    // loads the next token's tiles while the drain finishes this one, and
    // the second CTA of an SM (resident once the first exits) evens out the
    // tail.  Measured at T = 8192: one CTA per token 2.39 ms, one per SM
    // 2.35, two per SM 2.34, four 2.35 (the int64 path: the same at all).
    const int grid = p.T > 2 * sm_count() ? 2 * sm_count() : p.T;
    kern<<<grid, dkv::kThreads, dkv::kSmemBytes, s>>>(
        tm_qa, tm_doa, tm_sp_ld, idxc, count, cfix, acc, row_max, p.T, p.H, p.W, G, box_all,
        nbmax);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdFinal) {
    const long long n8 = static_cast<long long>(p.S_kv) * p.d_qk / 8;
    if (p.deterministic)
      k_dkv_cast_fixed<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(
          static_cast<const long long*>(acc), static_cast<__nv_bfloat16*>(dkv), n8, row_refs,
          row_max, p.d_qk);
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
