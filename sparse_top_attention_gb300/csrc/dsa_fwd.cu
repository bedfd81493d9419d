// Sparse MLA (DSA) forward for sm_103a.
//
// A work item is one token t with a group of up to 64 query heads; each
// persistent CTA processes a share of the items in turn.  The token's top-k
// rows are gathered from the shared KV tensor, 128 rows at a time
// ("blocks").  The contractions use 5th-gen tensor cores with fp32
// accumulators in TMEM, in a transposed orientation: the gathered rows form
// the UMMA M dimension (128) and the heads form N (64), so a 64-head group
// fills a full-rate M=128 tile.
//   S^T[slot, h]  = sum_d KV[slot, d] * Q[h, d]          (M=128, N=64, K=D)
//   O^T[d, h]    += sum_slot V[slot, d] * P^T[slot, h]   (4 x M=128, N=64, K=128)
// with rows of D = 576 columns (512 V + 64 rope) or 512 (a template
// parameter).  The softmax runs on S^T in registers, one thread per gathered
// row and 32 heads, with a lazy rescale: a head's shift only moves when a score exceeds it
// by more than 2^8.  The sink enters at the end, as sigma(lse - sink):
//   out = O * sigma(lse - sink) / l.
// Sources:
//   - flash-attention "[CuTe, SM100] Support 1..128 Q heads in sparse MLA via
//     in-kernel TMA padding", Agent Notes: a tile serves a single token with
//     its own top-k gather list; padded heads are zero rows.
//   - cuDNN frontend "DSA backward SM90: fix three top-k and attention-sink
//     boundary failures", Summary 1-3: empty rows, padded columns masked to
//     -inf, a sink that stays finite when it saturates.
//
// Warp roles (384 threads):
//   warps 0-7  softmax and epilogue; thread (w, l) owns TMEM lane
//              32 (w % 4) + l (gathered row) and heads 32 (w / 4) .. +31, so
//              two softmax warps share each SM sub-partition's exp2 work
//   warp 8     TMEM allocation and the single UMMA-issuing thread
//   warps 9-11 per item: compact the token's index row, lane 0 of warp 9
//              loads the Q tile by TMA (3-D tensor map), then the three warps
//              gather KV rows with cp.async into 128B-swizzled shared tiles,
//              or a whole block of consecutive rows (the sliding window) with
//              2-D TMA
// The kernel is persistent: one CTA per SM walks the (token, head group)
// items, so an item's epilogue overlaps the next item's first gather.
#include <cmath>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_tmap.h"

namespace dsa {
namespace {

__device__ unsigned int g_err_fwd;

constexpr int kHG = 64;                      // heads per CTA (UMMA N)
constexpr int kSoftmax = 256;               // warps 0-7: row (warp & 3) * 32 + lane, heads 32 * (warp >> 2) + 0..31
constexpr int kMmaWarp = 8;
constexpr int kQIssuer = 288;               // lane 0 of warp 9
constexpr int kProducers = 96;              // warps 9-11
constexpr int kThreads = kSoftmax + 32 + kProducers;
constexpr int kQChunk = kHG * 128;           // one 64-column chunk of Q: 8 KB
constexpr int kKVChunk = kBlk * 128;         // one 64-column chunk of 128 rows: 16 KB
constexpr int kIdxRegs = (kMaxW + kProducers - 1) / kProducers;  // index row per producer

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T: 64 columns
constexpr uint32_t kColO = 64;    // O^T: 4 chunks x 64 columns

struct Misc {
  uint64_t kv_full[kChunks];
  uint64_t kv_free[kChunks];
  uint64_t q_full, q_free, s_full, p_full, o_done, mma_done;
  float red[2][4][kHG];   // per-warp column maxima, double-buffered by block parity
  alignas(16) float m_used[kHG];  // running shift per head (log2 units)
  float fac[kHG];         // rescale factor per head, then the output scale
  int warp_counts[kThreads / 32];
  uint32_t tmem_base;
  int abort_flag;
};

// Shared-memory layout for rows of kD columns (576 = 512 V + 64 rope, or 512).
// Chunks 0..7 of the KV tile are V (d 0..511), chunk 8 the rope columns.
template <int kD>
struct FwdLayout {
  static constexpr int kCh = kD / 64;         // 64-column chunks of a row
  static constexpr bool kRope = kCh > 8;
  static constexpr int kOffKV = 0;
  static constexpr int kOffQ = kOffKV + kCh * kKVChunk;
  static constexpr int kOffList = kOffQ + kCh * kQChunk;
  // P^T reuses the rope chunk once S is done; without one it has its own tile.
  static constexpr int kOffP = kRope ? kOffKV + 8 * kKVChunk : kOffList + kMaxW * 4;
  static constexpr int kOffMisc = kRope ? kOffList + kMaxW * 4 : kOffP + kKVChunk;
  static constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms need 1024-byte alignment");
};

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Waits on a barrier that the kernel's own tensor-core work completes,
// ignoring the abort flag but still bounded in time.
__device__ __forceinline__ void mbar_wait_final(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&g_err_fwd, 0u, 0x1FFu);
      return;
    }
  }
}

template <int kD>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
           const int32_t* __restrict__ topk_idxs, const int32_t* __restrict__ topk_length,
           const float* __restrict__ sink, __nv_bfloat16* __restrict__ out,
           float* __restrict__ lse, const __nv_bfloat16* __restrict__ kv, int T, int H, int S_kv,
           int W, float scale, int G, int residual, int box_heads,
           const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int B) {
  using L = FwdLayout<kD>;
  constexpr int kCh = L::kCh, kOffKV = L::kOffKV, kOffQ = L::kOffQ, kOffList = L::kOffList,
                kOffP = L::kOffP, kOffMisc = L::kOffMisc;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // uniform across the CTA; never expected
    if (tid == 0) atomicCAS(&g_err_fwd, 0u, 0x2FFu);
    return;
  }
  Misc& m = *reinterpret_cast<Misc*>(smem + kOffMisc);
  int32_t* list = reinterpret_cast<int32_t*>(smem + kOffList);
  const FailState fs{&g_err_fwd, &m.abort_flag};
  // Persistent: CTA c takes items c, c + gridDim.x, ... of the (token, head
  // group) list.  Every role walks the same items and finds each item's
  // valid-slot count itself; barrier phases follow running counts of
  // non-empty items (Q tile) and of blocks (everything else).
  const int n_items = T * G;
  const size_t lo_off = residual ? static_cast<size_t>(T) * H * kDv : 0;  // residual half

  if (tid == 0) {
    for (int c = 0; c < kCh; ++c) {
      mbar_init(smem_u32(&m.kv_full[c]), kProducers);
      mbar_init(smem_u32(&m.kv_free[c]), 1);
    }
    mbar_init(smem_u32(&m.q_full), 1);
    mbar_init(smem_u32(&m.q_free), 1);
    mbar_init(smem_u32(&m.s_full), 1);
    mbar_init(smem_u32(&m.p_full), kSoftmax);
    mbar_init(smem_u32(&m.o_done), 1);
    mbar_init(smem_u32(&m.mma_done), 1);
    m.abort_flag = 0;
    mbar_init_fence();
  }
  if (tid < kHG) m.m_used[tid] = -INFINITY;
  // Q tile rows that the TMA box does not cover (only when H < 64) are zero;
  // the loads never write them, so once is enough.
  for (int i = tid; i < kCh * (kHG - box_heads) * 8; i += kThreads) {
    const int per = (kHG - box_heads) * 8;
    const int c = i / per, rem = i - c * per;
    const int row = box_heads + rem / 8, pc = rem & 7;
    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + kOffQ + c * kQChunk +
                                                               sw128_off(row, pc)),
                 "r"(0u)
                 : "memory");
  }
  fence_proxy_async_smem();
  if (warp == kMmaWarp) tmem_alloc(smem_u32(&m.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp > kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Per item: compact the token's valid slots into the row list (slot
    // order), load the Q tile of the head group by TMA once the previous
    // item's S GEMMs are done with it, then gather the rows block by block:
    // cp.async 16-byte pieces into the 128B-swizzled chunk tiles (one warp
    // instruction moves 4 whole 128-byte row pieces; rows past the valid
    // count are zero-filled and their scores masked), or one 2-D TMA load
    // per chunk for a block of consecutive rows (the sliding window).
    const int ptid = tid - kQIssuer, pw = warp - (kMmaWarp + 1);
    const uint64_t keep = l2_evict_last();
    int it = 0, gb = 0;  // non-empty items and blocks so far
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G, h0 = (u - t * G) * kHG;
      int32_t idx_regs[kIdxRegs];
      load_index_row(topk_idxs + static_cast<size_t>(t) * W, W, ptid, kProducers, idx_regs);
      // Every producer has issued the previous item's last gathers (the
      // list reads) before the first barrier inside, ahead of any write.
      const int Kt = compact_token_regs(idx_regs, W, slot_len(topk_length, t, W),
                                        kv_range(cu_q, cu_kv, B, t, S_kv), list, kMaxW,
                                        m.warp_counts, ptid, kProducers, 2);
      if (Kt == 0) continue;
      const int nblk = (Kt + kBlk - 1) / kBlk;
      if (tid == kQIssuer) {
        if (it > 0) mbar_wait(smem_u32(&m.q_free), (it - 1) & 1, fs, 8);
        mbar_arrive_expect_tx(smem_u32(&m.q_full), kCh * box_heads * 128);
        const uint64_t pol = l2_evict_first();
        for (int c = 0; c < kCh; ++c)
          tma_load_3d_hint(sbase + kOffQ + c * kQChunk, &tm_q, c * 64, h0, t,
                           smem_u32(&m.q_full), pol);
      }
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
          const int r = ok ? list[slot] : 0;
          src[k] = kv + static_cast<size_t>(r) * kD + pc * 8;
          dst[k] = sw128_off(row & (kBlk - 1), pc);
          nbytes[k] = ok ? 16u : 0u;
        }
        bool contig = false;
        int r0 = 0;
        if (b * kBlk + kBlk <= Kt) {
          r0 = list[b * kBlk];
          bool mine = true;
          for (int i = ptid; i < kBlk; i += kProducers) mine &= list[b * kBlk + i] == r0 + i;
          contig = !named_bar_or(2, kProducers, !mine);
        }
        for (int c = 0; c < kCh; ++c) {
          if (gb > 0) mbar_wait(smem_u32(&m.kv_free[c]), (gb - 1) & 1, fs, 1);
          if (contig) {
            if (tid == kQIssuer) {
              mbar_arrive_expect_tx(smem_u32(&m.kv_full[c]), kKVChunk);
              tma_load_2d_hint(sbase + kOffKV + c * kKVChunk, &tm_kv, c * 64, r0,
                               smem_u32(&m.kv_full[c]), keep);
            } else {
              mbar_arrive(smem_u32(&m.kv_full[c]));
            }
            continue;
          }
#pragma unroll
          for (int k = 0; k < kRowGroups; ++k)
            if (pw + 3 * k < kBlk / 4)
              cp_async_16_hint(sbase + kOffKV + c * kKVChunk + dst[k], src[k] + c * 64,
                               nbytes[k], keep);
          cp_async_arrive(smem_u32(&m.kv_full[c]));
        }
      }
      ++it;
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ UMMA issue
    const uint32_t idS = idesc_bf16(128, kHG, false, false);
    const uint32_t idPV = idesc_bf16(128, kHG, true, true);
    const uint32_t tS = tmem + kColS, tO = tmem + kColO;
    int it = 0, gb = 0;
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G;
      const int Kt = warp_count_valid(topk_idxs + static_cast<size_t>(t) * W, W,
                                      slot_len(topk_length, t, W),
                                      kv_range(cu_q, cu_kv, B, t, S_kv), lane);
      if (Kt == 0) continue;
      const int nblk = (Kt + kBlk - 1) / kBlk;
      if (lane == 0) {
        mbar_wait(smem_u32(&m.q_full), it & 1, fs, 2);
        for (int b = 0; b < nblk; ++b) {
          const int g = gb + b;
          for (int c = 0; c < kCh; ++c) {
            mbar_wait(smem_u32(&m.kv_full[c]), g & 1, fs, 3);
            fence_proxy_async_smem();  // cp.async (generic proxy) -> UMMA (async proxy)
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t a = sdesc_sw128(sbase + kOffKV + c * kKVChunk + k * 32, 16, 1024);
              const uint64_t bq = sdesc_sw128(sbase + kOffQ + c * kQChunk + k * 32, 16, 1024);
              umma_ss(tS, a, bq, idS, (c | k) != 0);
            }
          }
          umma_commit(smem_u32(&m.s_full));
          if (b == nblk - 1) umma_commit(smem_u32(&m.q_free));  // Q read for the last time
          mbar_wait(smem_u32(&m.p_full), g & 1, fs, 4);
          tc_fence_after();
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t a =
                  sdesc_sw128(sbase + kOffKV + (2 * j) * kKVChunk + k * 2048, kKVChunk, 1024);
              const uint64_t bp = sdesc_sw128(sbase + kOffP + k * 2048, kKVChunk, 1024);
              umma_ss(tO + j * kHG, a, bp, idPV, (b | k) != 0);
            }
            umma_commit(smem_u32(&m.kv_free[2 * j]));
            umma_commit(smem_u32(&m.kv_free[2 * j + 1]));
          }
          if constexpr (L::kRope) umma_commit(smem_u32(&m.kv_free[8]));
          umma_commit(smem_u32(&m.o_done));
        }
      }
      gb += nblk;
      ++it;
      __syncwarp();
    }
    if (lane == 0 && it > 0) {  // all MMAs retired before the TMEM is freed
      umma_commit(smem_u32(&m.mma_done));
      mbar_wait_final(smem_u32(&m.mma_done), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Thread (warp w, lane l) owns gathered row (w & 3) * 32 + l of the
    // block (its TMEM lane) and heads hb .. hb + 31, hb = 32 * (w >> 2): two
    // warps per SM sub-partition share the exp2 work of a block.
    const float sl2 = scale * kLog2e;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane, hb = (warp >> 2) * 32;
    int gb = 0;
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G, h0 = (u - t * G) * kHG;
      const int nh = min(kHG, H - h0);
      const int Kt = warp_count_valid(topk_idxs + static_cast<size_t>(t) * W, W,
                                      slot_len(topk_length, t, W),
                                      kv_range(cu_q, cu_kv, B, t, S_kv), lane);
      if (Kt == 0) {  // empty row: out = 0, lse = -FLT_MAX, no tensor-core work
        for (int v = tid; v < nh * (kDv / 8); v += kSoftmax) {
          const int h = v / (kDv / 8), c = v - h * (kDv / 8);
          const size_t o = (static_cast<size_t>(t) * H + h0 + h) * kDv + c * 8;
          *reinterpret_cast<uint4*>(out + o) = make_uint4(0, 0, 0, 0);
          if (residual) *reinterpret_cast<uint4*>(out + lo_off + o) = make_uint4(0, 0, 0, 0);
        }
        if (tid < nh) lse[static_cast<size_t>(t) * H + h0 + tid] = -kFltMax;
        continue;
      }
      const int nblk = (Kt + kBlk - 1) / kBlk;
      float lp[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) lp[h] = 0.f;

      for (int b = 0; b < nblk; ++b) {
        const int g = gb + b;
        mbar_wait(smem_u32(&m.s_full), g & 1, fs, 5);
        tc_fence_after();
        uint32_t r0[32];
        tmem_ld32_sync(tmem + lane_base + kColS + hb, r0);
        const bool valid = b * kBlk + row < Kt;
        float s[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = valid ? __uint_as_float(r0[i]) * sl2 : -INFINITY;
        // Lazy rescale: a head keeps its shift unless the block's maximum
        // exceeds it by more than 2^8; the final normalisation uses the same
        // shift for O and l.  The column maxima are only needed when some
        // score is that far above its head's shift (always in the first
        // block), so one vote decides whether to compute them.
        bool above = false;
        const float4* mu4 = reinterpret_cast<const float4*>(m.m_used + hb);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 mu = mu4[i / 4];
          above |= (s[i] > mu.x + 8.f) | (s[i + 1] > mu.y + 8.f) | (s[i + 2] > mu.z + 8.f) |
                   (s[i + 3] > mu.w + 8.f);
        }
        bool any = named_bar_or(1, kSoftmax, above);
        if (any) {
          // column (per-head) maximum over the 128 gathered rows
          float* red = m.red[g & 1][warp & 3];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float mx = warp_max(s[i]);
            if (i == lane) red[hb + i] = mx;
          }
          named_bar_sync(1, kSoftmax);
          bool resc = false;
          if (tid < kHG) {
            const float bm = fmaxf(fmaxf(m.red[g & 1][0][tid], m.red[g & 1][1][tid]),
                                   fmaxf(m.red[g & 1][2][tid], m.red[g & 1][3][tid]));
            const float mo = m.m_used[tid];
            const float mn = fmaxf(mo, bm);
            resc = mn > mo + 8.f;
            m.fac[tid] = resc ? ex2_approx(mo - mn) : 1.f;
            if (resc) m.m_used[tid] = mn;
          }
          any = named_bar_or(1, kSoftmax, resc);
        }
        if (any) {
#pragma unroll
          for (int i = 0; i < 32; ++i) lp[i] *= m.fac[hb + i];
        }
        if (any && b > 0) {
          // O^T columns of heads whose shift moved: scale by 2^(old - new).
          // The previous PV finished before this block's S (in-order
          // completion), so the wait returns at once.
          mbar_wait(smem_u32(&m.o_done), (g - 1) & 1, fs, 6);
          tc_fence_after();
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
            const uint32_t ta = tmem + lane_base + kColO + j * kHG + hb;
            uint32_t r[32];
            tmem_ld32_sync(ta, r);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              r[i] = __float_as_uint(__uint_as_float(r[i]) * m.fac[hb + i]);
            tmem_st32(ta, r);
          }
          tmem_wait_st();
        }
        // P^T row as bf16 pairs; s[] is dead after this loop.
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float4 mu = mu4[i / 2];
          const float p0 = ex2_approx(s[2 * i] - mu.x);
          const float p1 = ex2_approx(s[2 * i + 1] - mu.y);
          const float p2 = ex2_approx(s[2 * i + 2] - mu.z);
          const float p3 = ex2_approx(s[2 * i + 3] - mu.w);
          lp[2 * i] += p0;
          lp[2 * i + 1] += p1;
          lp[2 * i + 2] += p2;
          lp[2 * i + 3] += p3;
          pk[i] = pack_bf16x2(p0, p1);
          pk[i + 1] = pack_bf16x2(p2, p3);
        }
        // Store into the swizzled MN-major tile that the PV UMMA reads: this
        // thread's heads are 16-byte pieces hb / 8 .. hb / 8 + 3 of its row.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t dst = sbase + kOffP + sw128_off(row, hb / 8 + c);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[4 * c]),
                       "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                       : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&m.p_full));
      }
      gb += nblk;

      // ---------------------------------------------------------- epilogue
      // l per head: a butterfly reduce-scatter leaves lane L of each warp
      // with its rows' sum for head hb + L in lp[0]; the four row warps'
      // partials meet in shared memory (both halves of red are free: the
      // block loop's last barrier came after their last reads).
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float keep = up ? lp[i + o] : lp[i];
          const float send = up ? lp[i] : lp[i + o];
          lp[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      m.red[0][warp & 3][hb + lane] = lp[0];
      named_bar_sync(1, kSoftmax);
      if (tid < kHG) {
        const float l = (m.red[0][0][tid] + m.red[0][1][tid]) + (m.red[0][2][tid] + m.red[0][3][tid]);
        const float lse_nat = (m.m_used[tid] + log2f(l)) * kLn2;
        const float sk = (sink != nullptr && tid < nh) ? sink[h0 + tid] : -INFINITY;
        const float gate = stable_sigmoid(lse_nat - sk);
        m.fac[tid] = gate / l;
        m.m_used[tid] = -INFINITY;  // the next item starts afresh
        if (tid < nh) lse[static_cast<size_t>(t) * H + h0 + tid] = lse_nat;
      }
      named_bar_sync(1, kSoftmax);
      // O^T -> out (bf16) straight from registers once the last PV is done:
      // for each head, a warp writes 32 consecutive d of that head's row.
      mbar_wait(smem_u32(&m.o_done), (gb - 1) & 1, fs, 7);
      tc_fence_after();
      __nv_bfloat16* out_t = out + (static_cast<size_t>(t) * H + h0) * kDv;
      for (int j = 0; j < 4; ++j) {
        uint32_t r[32];
        tmem_ld32_sync(tmem + lane_base + kColO + j * kHG + hb, r);
        const int d = j * 128 + row;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = hb + i;
          if (h < nh) {
            const float o = __uint_as_float(r[i]) * m.fac[h];
            const __nv_bfloat16 hi = __float2bfloat16_rn(o);
            out_t[static_cast<size_t>(h) * kDv + d] = hi;
            if (residual)
              out_t[lo_off + static_cast<size_t>(h) * kDv + d] =
                  __float2bfloat16_rn(o - __bfloat162float(hi));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                       const int32_t* len, const float* sink, void* out, float* lse,
                       cudaStream_t s) {
  static std::atomic<uint64_t> attr_done{0};
  const int dev = current_device();
  if (device_needs_setup(attr_done, dev)) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<576>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdLayout<576>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fwd_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               FwdLayout<512>::kSmemBytes);
    if (e != cudaSuccess) return e;
    mark_device_setup(attr_done, dev);
  }
  const int G = (p.H + kHG - 1) / kHG;
  const long long items = static_cast<long long>(p.T) * G;
  if (items == 0) return cudaSuccess;
  // persistent: at most one CTA per SM, each walking its share of the items
  const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
  CUtensorMap tm_q, tm_kv;
  const int box_heads = p.H < kHG ? p.H : kHG;  // never larger than the tensor
  cudaError_t e = make_head_tile_map(&tm_q, q, p.T, p.H, p.d_qk, box_heads);
  if (e == cudaSuccess) e = make_matrix_map(&tm_kv, kv, p.S_kv, p.d_qk, kBlk);
  if (e != cudaSuccess) return e;
  auto kern = p.d_qk == 512 ? fwd_kernel<512> : fwd_kernel<576>;
  const int smem = p.d_qk == 512 ? FwdLayout<512>::kSmemBytes : FwdLayout<576>::kSmemBytes;
  kern<<<grid, kThreads, smem, s>>>(
      tm_q, tm_kv, idx, len, sink, static_cast<__nv_bfloat16*>(out), lse,
      static_cast<const __nv_bfloat16*>(kv), p.T, p.H, p.S_kv, p.W, p.scale, G,
      p.delta_residual ? 1 : 0, box_heads, p.cu_q, p.cu_kv, p.B);
  return cudaGetLastError();
}

unsigned int fwd_take_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v) cudaMemcpyToSymbol(g_err_fwd, &zero, sizeof(zero));
  return v;
}

}  // namespace dsa
