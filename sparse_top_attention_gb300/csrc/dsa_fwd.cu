// Sparse MLA (DSA) forward for sm_103a.
//
// One CTA computes one token t for a group of up to 64 query heads.  The
// token's top-k rows are gathered from the shared KV tensor, 128 rows at a
// time ("blocks").  The contractions use 5th-gen tensor cores with fp32
// accumulators in TMEM, in a transposed orientation: the gathered rows form
// the UMMA M dimension (128) and the heads form N (64), so a 64-head group
// fills a full-rate M=128 tile.
//   S^T[slot, h]  = sum_d KV[slot, d] * Q[h, d]          (M=128, N=64, K=D)
//   O^T[d, h]    += sum_slot V[slot, d] * P^T[slot, h]   (4 x M=128, N=64, K=128)
// with rows of D = 576 columns (512 V + 64 rope) or 512 (a template
// parameter).  The softmax runs on S^T in registers, one thread per gathered
// row, with a lazy rescale: a head's shift only moves when a score exceeds it
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
// Warp roles (256 threads):
//   warps 0-3  softmax and epilogue; thread i owns TMEM lane i (gathered row i)
//   warp 4     TMEM allocation and the single UMMA-issuing thread
//   warps 5-7  lane 0 of warp 5 issues the Q tile TMA (3-D tensor map) at
//              kernel entry; the three warps gather KV rows with cp.async into
//              128B-swizzled shared tiles, or a whole block of consecutive
//              rows (the sliding window) with 2-D TMA
// Eight warps keep two warps per SM sub-partition, so each thread may use up
// to 255 registers.
#include <cmath>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_tmap.h"

namespace dsa {
namespace {

__device__ unsigned int g_err_fwd;

constexpr int kHG = 64;                      // heads per CTA (UMMA N)
constexpr int kThreads = 256;
constexpr int kQIssuer = 160;               // lane 0 of warp 5
constexpr int kProducers = 96;              // warps 5-7
constexpr int kQChunk = kHG * 128;           // one 64-column chunk of Q: 8 KB
constexpr int kKVChunk = kBlk * 128;         // one 64-column chunk of 128 rows: 16 KB

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T: 64 columns
constexpr uint32_t kColO = 64;    // O^T: 4 chunks x 64 columns

struct Misc {
  uint64_t kv_full[kChunks];
  uint64_t kv_free[kChunks];
  uint64_t q_full, s_full, p_full, o_done, mma_done;
  float red[2][4][kHG];   // per-warp column maxima, double-buffered by block parity
  float m_used[kHG];      // running shift per head (log2 units)
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
  const int t = blockIdx.x / G, grp = blockIdx.x - t * G;
  const int h0 = grp * kHG;
  const int nh = min(kHG, H - h0);
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // uniform across the CTA; never expected
    if (tid == 0) atomicCAS(&g_err_fwd, 0u, 0x2FFu);
    return;
  }
  Misc& m = *reinterpret_cast<Misc*>(smem + kOffMisc);
  int32_t* list = reinterpret_cast<int32_t*>(smem + kOffList);
  const FailState fs{&g_err_fwd, &m.abort_flag};

  // The Q tile of the head group (kCh chunks of [box_heads x 64 columns],
  // 128B swizzle; heads past H inside the box are zero-filled by the TMA)
  // loads from kernel entry: its issuing thread owns its barrier.  The
  // token's index row is read into registers now as well, so that both
  // latencies overlap the set-up below.
  if (tid == kQIssuer) {
    mbar_init(smem_u32(&m.q_full), 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(smem_u32(&m.q_full), kCh * box_heads * 128);
    const uint64_t pol = l2_evict_first();
    for (int c = 0; c < kCh; ++c)
      tma_load_3d_hint(sbase + kOffQ + c * kQChunk, &tm_q, c * 64, h0, t, smem_u32(&m.q_full),
                       pol);
  }
  int32_t idx_regs[kMaxW / kThreads];
  load_index_row(topk_idxs + static_cast<size_t>(t) * W, W, tid, kThreads, idx_regs);

  if (tid == 0) {
    for (int c = 0; c < kCh; ++c) {
      mbar_init(smem_u32(&m.kv_full[c]), kProducers);
      mbar_init(smem_u32(&m.kv_free[c]), 1);
    }
    mbar_init(smem_u32(&m.s_full), 1);
    mbar_init(smem_u32(&m.p_full), 128);
    mbar_init(smem_u32(&m.o_done), 1);
    mbar_init(smem_u32(&m.mma_done), 1);
    m.abort_flag = 0;
    mbar_init_fence();
  }
  if (tid < kHG) m.m_used[tid] = -INFINITY;
  // Q tile rows that the TMA box does not cover (only when H < 64) are zero.
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
  __syncthreads();

  // a1: decode and compact the valid slots of token t (slot order).
  const int len = slot_len(topk_length, t, W);
  const KvRange kvr = kv_range(cu_q, cu_kv, B, t, S_kv);
  const int Kt = compact_token_regs(idx_regs, W, len, kvr, list, kMaxW, m.warp_counts, tid,
                                    kThreads);

  const size_t lo_off = residual ? static_cast<size_t>(T) * H * kDv : 0;  // residual half
  if (Kt == 0) {  // empty row: out = 0, lse = -FLT_MAX, no tensor-core work
    for (int v = tid; v < nh * (kDv / 8); v += kThreads) {
      const int h = v / (kDv / 8), c = v - h * (kDv / 8);
      const size_t o = (static_cast<size_t>(t) * H + h0 + h) * kDv + c * 8;
      *reinterpret_cast<uint4*>(out + o) = make_uint4(0, 0, 0, 0);
      if (residual) *reinterpret_cast<uint4*>(out + lo_off + o) = make_uint4(0, 0, 0, 0);
    }
    if (tid < nh) lse[static_cast<size_t>(t) * H + h0 + tid] = -kFltMax;
    // the Q tile is still landing in this CTA's shared memory: let it finish
    if (tid == kQIssuer) mbar_wait_final(smem_u32(&m.q_full), 0);
    return;
  }
  const int nblk = (Kt + kBlk - 1) / kBlk;

  if (warp == 4) tmem_alloc(smem_u32(&m.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp >= 5) {
    // ------------------------------------------------------------ gather
    // cp.async 16-byte pieces into the 128B-swizzled chunk tiles; one warp
    // instruction moves 4 whole 128-byte row pieces.  Rows past the valid
    // count are zero-filled (their scores are masked).
    const int pw = warp - 5;
    const uint64_t keep = l2_evict_last();
    for (int b = 0; b < nblk; ++b) {
      // This lane's rows of the block, read once (before the wait on the
      // first chunk, so the reads overlap it) and reused by all 9 chunks.
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
      // A full block of consecutive KV rows (the sliding window) comes in with
      // one 2-D TMA load per chunk instead of 128 row copies.
      bool contig = false;
      int r0 = 0;
      if (b * kBlk + kBlk <= Kt) {
        r0 = list[b * kBlk];
        bool mine = true;
        for (int i = tid - kQIssuer; i < kBlk; i += kProducers) mine &= list[b * kBlk + i] == r0 + i;
        contig = !named_bar_or(2, kProducers, !mine);
      }
      for (int c = 0; c < kCh; ++c) {
        if (b > 0) mbar_wait(smem_u32(&m.kv_free[c]), (b - 1) & 1, fs, 1);
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
            cp_async_16_hint(sbase + kOffKV + c * kKVChunk + dst[k], src[k] + c * 64, nbytes[k],
                             keep);
        cp_async_arrive(smem_u32(&m.kv_full[c]));
      }
    }
    cp_async_wait_all();
  } else if (warp == 4) {
    // ------------------------------------------------------------ UMMA issue
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, kHG, false, false);
      const uint32_t idPV = idesc_bf16(128, kHG, true, true);
      const uint32_t tS = tmem + kColS, tO = tmem + kColO;
      mbar_wait(smem_u32(&m.q_full), 0, fs, 2);
      for (int b = 0; b < nblk; ++b) {
        for (int c = 0; c < kCh; ++c) {
          mbar_wait(smem_u32(&m.kv_full[c]), b & 1, fs, 3);
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
        mbar_wait(smem_u32(&m.p_full), b & 1, fs, 4);
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
      umma_commit(smem_u32(&m.mma_done));
      mbar_wait_final(smem_u32(&m.mma_done), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const float sl2 = scale * kLog2e;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS_row = tmem + lane_base + kColS;
    float lp[kHG];
#pragma unroll
    for (int h = 0; h < kHG; ++h) lp[h] = 0.f;
    __nv_bfloat16* const sP = reinterpret_cast<__nv_bfloat16*>(smem + kOffP);
    (void)sP;

    for (int b = 0; b < nblk; ++b) {
      mbar_wait(smem_u32(&m.s_full), b & 1, fs, 5);
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32x2_sync(tS_row, r0, tS_row + 32, r1);
      const bool valid = b * kBlk + tid < Kt;
      float s[kHG];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = valid ? __uint_as_float(r0[i]) * sl2 : -INFINITY;
        s[32 + i] = valid ? __uint_as_float(r1[i]) * sl2 : -INFINITY;
      }
      // Lazy rescale: a head keeps its shift unless the block's maximum
      // exceeds it by more than 2^8; the final normalisation uses the same
      // shift for O and l.  The column maxima are only needed when some score
      // is that far above its head's shift (always in the first block), so
      // one vote decides whether to compute them.
      bool above = false;
#pragma unroll
      for (int h = 0; h < kHG; ++h) above |= s[h] > m.m_used[h] + 8.f;
      bool any = named_bar_or(1, 128, above);
      if (any) {
        // column (per-head) maximum over the 128 gathered rows
        float* red = m.red[b & 1][warp];
#pragma unroll
        for (int h = 0; h < kHG; ++h) {
          const float mx = warp_max(s[h]);
          if ((h & 31) == lane) red[h] = mx;
        }
        named_bar_sync(1, 128);
        bool resc = false;
        if (tid < kHG) {
          const float bm = fmaxf(fmaxf(m.red[b & 1][0][tid], m.red[b & 1][1][tid]),
                                 fmaxf(m.red[b & 1][2][tid], m.red[b & 1][3][tid]));
          const float mo = m.m_used[tid];
          const float mn = fmaxf(mo, bm);
          resc = mn > mo + 8.f;
          m.fac[tid] = resc ? ex2_approx(mo - mn) : 1.f;
          if (resc) m.m_used[tid] = mn;
        }
        any = named_bar_or(1, 128, resc);
      }
      if (any) {
#pragma unroll
        for (int h = 0; h < kHG; ++h) lp[h] *= m.fac[h];
      }
      // P^T row as bf16 pairs; s[] is dead after this loop.
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2_approx(s[2 * i] - m.m_used[2 * i]);
        const float p1 = ex2_approx(s[2 * i + 1] - m.m_used[2 * i + 1]);
        lp[2 * i] += p0;
        lp[2 * i + 1] += p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      if (any && b > 0) {
        // O^T columns of heads whose shift moved: scale by 2^(old - new).
        mbar_wait(smem_u32(&m.o_done), (b - 1) & 1, fs, 6);
        tc_fence_after();
        for (int j = 0; j < 4; ++j) {
          for (int half = 0; half < 2; ++half) {
            const uint32_t ta = tmem + lane_base + kColO + j * kHG + half * 32;
            uint32_t r[32];
            tmem_ld32_sync(ta, r);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              r[i] = __float_as_uint(__uint_as_float(r[i]) * m.fac[half * 32 + i]);
            tmem_st32(ta, r);
          }
        }
        tmem_wait_st();
      }
      // Store into the swizzled MN-major tile that the PV UMMA reads.
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t dst = sbase + kOffP + sw128_off(tid, c);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[4 * c]),
                     "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&m.p_full));
    }

    // ------------------------------------------------------------ epilogue
    mbar_wait(smem_u32(&m.o_done), (nblk - 1) & 1, fs, 7);
    tc_fence_after();
    float* lbuf = reinterpret_cast<float*>(smem + kOffKV);  // [128][65]
#pragma unroll
    for (int h = 0; h < kHG; ++h) lbuf[tid * 65 + h] = lp[h];
    named_bar_sync(1, 128);
    if (tid < kHG) {
      float l = 0.f;
      for (int r = 0; r < kBlk; ++r) l += lbuf[r * 65 + tid];
      const float lse_nat = (m.m_used[tid] + log2f(l)) * kLn2;
      const float sk = (sink != nullptr && tid < nh) ? sink[h0 + tid] : -INFINITY;
      const float gate = stable_sigmoid(lse_nat - sk);
      m.fac[tid] = gate / l;
      if (tid < nh) lse[static_cast<size_t>(t) * H + h0 + tid] = lse_nat;
    }
    named_bar_sync(1, 128);
    // Stage bf16 rows [64][512] (and their rounding residual) over the free KV
    // tiles; the l partials there were consumed before the barrier above.
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + kOffKV);
    __nv_bfloat16* stage_lo = reinterpret_cast<__nv_bfloat16*>(smem + kOffKV + kHG * kDv * 2);
    for (int j = 0; j < 4; ++j) {
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        tmem_ld32_sync(tmem + lane_base + kColO + j * kHG + half * 32, r);
        const int d = j * 128 + tid;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = half * 32 + i;
          const float o = __uint_as_float(r[i]) * m.fac[h];
          const __nv_bfloat16 hi = __float2bfloat16_rn(o);
          stage[h * kDv + d] = hi;
          if (residual) stage_lo[h * kDv + d] = __float2bfloat16_rn(o - __bfloat162float(hi));
        }
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (tid == 0) {
      // out rows (t, h0..h0+nh) are contiguous: one bulk store per half
      const size_t o = (static_cast<size_t>(t) * H + h0) * kDv;
      const uint64_t pol = l2_evict_first();
      bulk_store_hint(out + o, smem_u32(stage), nh * kDv * 2, pol);
      if (residual) bulk_store_hint(out + lo_off + o, smem_u32(stage_lo), nh * kDv * 2, pol);
      bulk_commit();
      bulk_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                       const int32_t* len, const float* sink, void* out, float* lse,
                       cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<576>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdLayout<576>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fwd_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               FwdLayout<512>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int G = (p.H + kHG - 1) / kHG;
  const long long grid = static_cast<long long>(p.T) * G;
  if (grid == 0) return cudaSuccess;
  CUtensorMap tm_q, tm_kv;
  const int box_heads = p.H < kHG ? p.H : kHG;  // never larger than the tensor
  cudaError_t e = make_head_tile_map(&tm_q, q, p.T, p.H, p.d_qk, box_heads);
  if (e == cudaSuccess) e = make_matrix_map(&tm_kv, kv, p.S_kv, p.d_qk, kBlk);
  if (e != cudaSuccess) return e;
  auto kern = p.d_qk == 512 ? fwd_kernel<512> : fwd_kernel<576>;
  const int smem = p.d_qk == 512 ? FwdLayout<512>::kSmemBytes : FwdLayout<576>::kSmemBytes;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(
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
