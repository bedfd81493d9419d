// Sparse MLA (DSA) forward for sm_103a.
//
// A work item is one token t with a group of query heads: 64, or 32 / 16
// when H is that small (the narrowest group that holds H); each persistent
// CTA processes a share of the items in turn.  The token's top-k rows are
// gathered from the shared KV tensor, 128 rows at a time ("blocks").  The
// contractions use 5th-gen tensor cores with fp32 accumulators in TMEM, in a
// transposed orientation: the gathered rows form the UMMA M dimension (128)
// and the heads form N, so any head group fills a full-rate M=128 tile.
//   S^T[slot, h]  = sum_d KV[slot, d] * Q[h, d]          (M=128, N=HG, K=D)
//   O^T[d, h]    += sum_slot V[slot, d] * P^T[slot, h]   (4 x M=128, N=HG, K=128)
// with rows of D = 576 columns (512 V + 64 rope) or 512 (a template
// parameter).  The softmax runs on S^T in registers, one thread per gathered
// row and HG/2 heads, with a lazy rescale: a head's shift only moves when a
// score exceeds it by more than 2^8.  The sink enters at the end, as
// sigma(lse - sink):
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
//              32 (w % 4) + l (gathered row) and heads HG/2 * (w / 4) + ..,
//              so two softmax warps share each SM sub-partition's exp2 work
//   warp 8     TMEM allocation and the single UMMA-issuing thread
//   warps 9-11 per item: compact the token's index row, lane 0 of warp 9
//              loads the Q tile by TMA (3-D tensor map), then the three warps
//              gather KV rows with cp.async into 128B-swizzled shared tiles,
//              or a whole block of consecutive rows (the sliding window) with
//              2-D TMA, into a ring of chunk slots
// The kernel is persistent: one CTA per SM walks the (token, head group)
// items, so an item's epilogue overlaps the next item's first gather.
#include <cmath>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_tmap.h"

namespace dsa {
namespace {

__device__ unsigned int g_err_fwd;

constexpr int kSoftmax = 256;               // warps 0-7: row (warp & 3) * 32 + lane, heads kHT * (warp >> 2) + 0..kHT-1
constexpr int kMmaWarp = 8;
constexpr int kQIssuer = 288;               // lane 0 of warp 9
constexpr int kProducers = 96;              // warps 9-11
constexpr int kThreads = kSoftmax + 32 + kProducers;
constexpr int kKVChunk = kBlk * 128;         // one 64-column chunk of 128 rows: 16 KB
constexpr int kVUnit = 2 * kKVChunk;         // the two V chunks one P.V tile reads: 32 KB
constexpr int kIdxRegs = (kMaxW + kProducers - 1) / kProducers;  // index row per producer
constexpr int kMaxUnits = 6, kMaxRope = 2;

template <int kHG>
struct Misc {
  uint64_t v_full[kMaxUnits][2];  // per V chunk of a unit
  uint64_t v_free[kMaxUnits];
  uint64_t rope_full[kMaxRope], rope_free[kMaxRope];
  uint64_t q_full[kChunks];  // per 64-column chunk of the Q tile
  uint64_t q_free, s_full, p_full, o_done, mma_done;
  float red[2][4][kHG];   // per-warp column maxima, double-buffered by block parity
  alignas(16) float m_used[kHG];  // running shift per head (log2 units)
  float fac[kHG];         // rescale factor per head, then the output scale
  int warp_counts[kThreads / 32];
  uint32_t tmem_base;
  int abort_flag;
};

// Per head group (64 heads, or 32 / 16 when H is that small) and row width
// kD (576 = 512 V + 64 rope, or 512):
//  - V chunks live in a ring of kUnits 32 KB units, each holding the two
//    64-column chunks that one P.V tile reads (so the tile's MN-major operand
//    steps from one to the other by a fixed LBO); the rope chunk in a ring of
//    kRopeSlots 16 KB slots.  A ring longer than one block lets the next
//    block's first chunks land while this block's softmax and P.V run.
//  - P^T: for 64 heads at D = 576 it reuses the block's rope slot (MN-major,
//    heads contiguous); for 64 heads at D = 512 it has its own MN-major tile;
//    for 32 / 16 heads it is a K-major [kHG head rows x 128 slots] tile.
//    S of block g + 1 is issued after the P.V of block g, so S done means
//    that P.V is done too: one S^T buffer and one P^T tile suffice, and the
//    ring never makes the next block's S wait on a P.V issued after it.
template <int kD, int kHG>
struct FwdLayout {
  static_assert(kHG == 64 || kHG == 32 || kHG == 16, "head group");
  static constexpr int kHT = kHG / 2;          // heads per softmax thread
  static constexpr int kCh = kD / 64;          // 64-column chunks of a row
  static constexpr bool kRope = kCh > 8;
  static constexpr int kQChunk = kHG * 128;    // one 64-column chunk of Q
  static constexpr bool kPInRope = kRope && kHG == 64;
  // one Q barrier per 64-column chunk (measured faster only for the 72 KB
  // tile of 64 heads at D = 576)
  static constexpr bool kQPerChunk = kRope && kHG == 64;
  static constexpr bool kPKMajor = kHG < 64;
  static constexpr int kPTile = kPKMajor ? kHG * 256 : kKVChunk;
  static constexpr int kPBytes = kPInRope ? 0 : kPTile;
  static constexpr int kMiscBytes = (static_cast<int>(sizeof(Misc<kHG>)) + 15) / 16 * 16;
  static constexpr int kFixed = kCh * kQChunk + kPBytes + kMaxW * 4 + kMiscBytes;
  static constexpr int kAvail = 232448 - kFixed;
  // rope slots: one when P shares it; two otherwise (the rope is gathered
  // first, and a slot frees as soon as S has read it)
  static constexpr int kRopeSlots = !kRope ? 0 : (kPInRope ? 1 : 2);
  static constexpr int kUnits0 = (kAvail - kRopeSlots * kKVChunk) / kVUnit;
  static constexpr int kUnits = kUnits0 > kMaxUnits ? kMaxUnits : kUnits0;
  static constexpr int kOffV = 0;
  static constexpr int kOffRope = kOffV + kUnits * kVUnit;
  static constexpr int kOffQ = kOffRope + kRopeSlots * kKVChunk;
  static constexpr int kOffP = kPInRope ? -1 : kOffQ + kCh * kQChunk;
  static constexpr int kOffList = kOffQ + kCh * kQChunk + kPBytes;
  static constexpr int kOffMisc = kOffList + kMaxW * 4;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes;
  // TMEM: S^T (kHG columns), then O^T (4 x kHG)
  static constexpr uint32_t kColO = kHG;
  static constexpr uint32_t kTmemCols = kHG == 64 ? 512 : (kHG == 32 ? 256 : 128);
  static_assert(kColO + 4 * kHG <= kTmemCols, "TMEM columns");
  static_assert(kUnits >= 4, "one block of V chunks must fit");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQ % 1024 == 0 && (kPInRope || kOffP % 1024 == 0) && kPTile % 1024 == 0,
                "swizzle atoms need 1024-byte alignment");
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

// Byte offset of element (head h, slot) in a K-major P^T tile of kHG head
// rows: two 64-slot halves, each [kHG rows x 128 B] with the 128-byte swizzle.
template <int kHG>
__device__ __forceinline__ uint32_t pk_tile_off(uint32_t h, uint32_t slot) {
  const uint32_t col = slot & 63u;
  return (slot >> 6) * (kHG * 128u) + h * 128u + ((((col >> 3) ^ (h & 7u)) << 4) | ((col & 7u) << 1));
}

// Where chunk `step` of a block (in gather order) lives, and its d-chunk.
// Gather order: with P in the rope slot, V chunks 0..7 then the rope chunk
// (the rope slot frees last); otherwise the rope chunk first.
template <int kD, int kHG>
struct ChunkRef {
  uint32_t addr, full, free;  // shared address, its full barrier, its free barrier
  int x;                      // d-chunk (0..7 V, 8 rope)
  int use;                    // fill count of its unit / slot before this one
};
template <int kD, int kHG>
__device__ __forceinline__ ChunkRef<kD, kHG> chunk_ref(uint32_t sbase, Misc<kHG>& m, int gb,
                                                       int step) {
  using L = FwdLayout<kD, kHG>;
  ChunkRef<kD, kHG> r;
  if constexpr (L::kRope) {
    if (L::kPInRope ? step == 8 : step == 0) {
      const int slot = gb % L::kRopeSlots;
      r.addr = sbase + L::kOffRope + slot * kKVChunk;
      r.full = smem_u32(&m.rope_full[slot]);
      r.free = smem_u32(&m.rope_free[slot]);
      r.x = 8;
      r.use = gb / L::kRopeSlots;
      return r;
    }
  }
  {
    const int c = (L::kRope && !L::kPInRope) ? step - 1 : step;  // V chunk
    const int pu = gb * 4 + (c >> 1), unit = pu % L::kUnits;
    r.addr = sbase + L::kOffV + unit * kVUnit + (c & 1) * kKVChunk;
    r.full = smem_u32(&m.v_full[unit][c & 1]);
    r.free = smem_u32(&m.v_free[unit]);
    r.x = c;
    r.use = pu / L::kUnits;
  }
  return r;
}

template <int kD, int kHG>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
           const int32_t* __restrict__ topk_idxs, const int32_t* __restrict__ topk_length,
           const float* __restrict__ sink, __nv_bfloat16* __restrict__ out,
           float* __restrict__ lse, const __nv_bfloat16* __restrict__ kv, int T, int H, int S_kv,
           int W, float scale, int G, int residual, int box_heads,
           const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int B) {
  using L = FwdLayout<kD, kHG>;
  constexpr int kCh = L::kCh, kHT = L::kHT, kQChunk = L::kQChunk, kOffQ = L::kOffQ,
                kOffList = L::kOffList, kOffMisc = L::kOffMisc;
  constexpr bool kPK = L::kPKMajor;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // uniform across the CTA; never expected
    if (tid == 0) atomicCAS(&g_err_fwd, 0u, 0x2FFu);
    return;
  }
  Misc<kHG>& m = *reinterpret_cast<Misc<kHG>*>(smem + kOffMisc);
  int32_t* list = reinterpret_cast<int32_t*>(smem + kOffList);
  const FailState fs{&g_err_fwd, &m.abort_flag};
  // Persistent: CTA c takes items c, c + gridDim.x, ... of the (token, head
  // group) list.  Every role walks the same items and finds each item's
  // valid-slot count itself; barrier phases follow running counts of
  // non-empty items (Q tile) and of blocks (everything else).
  const int n_items = T * G;
  const size_t lo_off = residual ? static_cast<size_t>(T) * H * kDv : 0;  // residual half
  // P^T tile of block gb (shared address)
  auto p_tile = [&](int gb) -> uint32_t {
    if constexpr (L::kPInRope)
      return sbase + L::kOffRope;  // the single rope slot
    else
      return sbase + L::kOffP;
  };

  if (tid == 0) {
    for (int u = 0; u < L::kUnits; ++u) {
      mbar_init(smem_u32(&m.v_full[u][0]), kProducers);
      mbar_init(smem_u32(&m.v_full[u][1]), kProducers);
      mbar_init(smem_u32(&m.v_free[u]), 1);
    }
    for (int r = 0; r < L::kRopeSlots; ++r) {
      mbar_init(smem_u32(&m.rope_full[r]), kProducers);
      mbar_init(smem_u32(&m.rope_free[r]), 1);
    }
    for (int c = 0; c < kCh; ++c) mbar_init(smem_u32(&m.q_full[c]), 1);
    mbar_init(smem_u32(&m.q_free), 1);
    mbar_init(smem_u32(&m.s_full), 1);
    mbar_init(smem_u32(&m.p_full), kSoftmax);
    mbar_init(smem_u32(&m.o_done), 1);
    mbar_init(smem_u32(&m.mma_done), 1);
    m.abort_flag = 0;
    mbar_init_fence();
  }
  if (tid < kHG) m.m_used[tid] = -INFINITY;
  // Q tile rows that the TMA box does not cover (only when H < kHG) are
  // zero; the loads never write them, so once is enough.
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
  if (warp == kMmaWarp) tmem_alloc(smem_u32(&m.tmem_base), L::kTmemCols);
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
    // per chunk for a block of consecutive rows (the sliding window).  Each
    // chunk waits only for its own unit or slot of the ring.
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
        const uint64_t pol = l2_evict_first();
        // 64 heads at D = 576 (a 72 KB tile): one barrier per chunk, so that
        // S starts on the first to land; otherwise one barrier for all of it
        if constexpr (!L::kQPerChunk) mbar_arrive_expect_tx(smem_u32(&m.q_full[0]), kCh * box_heads * 128);
        for (int c = 0; c < kCh; ++c) {
          const uint32_t qb = smem_u32(&m.q_full[L::kQPerChunk ? c : 0]);
          if constexpr (L::kQPerChunk) mbar_arrive_expect_tx(qb, box_heads * 128);
          tma_load_3d_hint(sbase + kOffQ + c * kQChunk, &tm_q, c * 64, h0, t, qb, pol);
        }
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
        for (int i = 0; i < kCh; ++i) {
          const ChunkRef<kD, kHG> cr = chunk_ref<kD, kHG>(sbase, m, gb, i);
          if (cr.use > 0) mbar_wait(cr.free, (cr.use - 1) & 1, fs, 1);
          if (contig) {
            if (tid == kQIssuer) {
              mbar_arrive_expect_tx(cr.full, kKVChunk);
              tma_load_2d_hint(cr.addr, &tm_kv, cr.x * 64, r0, cr.full, keep);
            } else {
              mbar_arrive(cr.full);
            }
            continue;
          }
#pragma unroll
          for (int k = 0; k < kRowGroups; ++k)
            if (pw + 3 * k < kBlk / 4)
              cp_async_16_hint(cr.addr + dst[k], src[k] + cr.x * 64, nbytes[k], keep);
          cp_async_arrive(cr.full);
        }
      }
      ++it;
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ UMMA issue
    // Per block: S^T over the chunks as they land, then (once the softmax has
    // written P) the four P.V tiles, each releasing its unit of the ring.
    // This one thread's bookkeeping sits between MMA issues, so it follows
    // the ring incrementally (no division) and steps descriptors by
    // constants (the start address field counts 16-byte units).
    const uint32_t idS = idesc_bf16(128, kHG, false, false);
    const uint32_t idPV = idesc_bf16(128, kHG, true, !kPK);  // P^T K-major for small groups
    const uint32_t tS = tmem, tO = tmem + L::kColO;
    const uint32_t vfull0 = smem_u32(&m.v_full[0][0]), vfree0 = smem_u32(&m.v_free[0]);
    const uint32_t rfull0 = smem_u32(&m.rope_full[0]), rfree0 = smem_u32(&m.rope_free[0]);
    const uint64_t dq0 = sdesc_sw128(sbase + kOffQ, 16, 1024);            // Q, K-major
    const uint64_t dv0 = sdesc_sw128(sbase + L::kOffV, 16, 1024);         // KV, K-major (S)
    const uint64_t dvt0 = sdesc_sw128(sbase + L::kOffV, kKVChunk, 1024);  // V^T, MN-major (P.V)
    const uint64_t dr0 = sdesc_sw128(sbase + L::kOffRope, 16, 1024);      // rope chunk (S)
    const uint64_t dp0 = kPK ? sdesc_sw128(p_tile(0), 16, 1024) : sdesc_sw128(p_tile(0), kKVChunk, 1024);
    constexpr bool kRopeFirst = L::kRope && !L::kPInRope;
    // S += chunk (d-chunk x) . Q chunk x^T, once the chunk has landed
    const uint32_t qfull0 = smem_u32(&m.q_full[0]);
    int qpar = -1;  // in an item's first block: the parity of its Q chunks' barriers
    auto s_chunk = [&](uint32_t full, uint32_t parity, uint64_t da, int x, bool first) {
      mbar_wait(full, parity, fs, 3);
      if (qpar >= 0) mbar_wait(qfull0 + 8 * x, static_cast<uint32_t>(qpar), fs, 2);
      fence_proxy_async_smem();  // cp.async (generic proxy) -> UMMA (async proxy)
      tc_fence_after();
      const uint64_t db = dq0 + static_cast<uint64_t>((x * kQChunk) >> 4);
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_ss(tS, da + 2 * k, db + 2 * k, idS, (!first || k != 0) ? 1u : 0u);
    };
    int it = 0, gb = 0;
    int ub = 0, wb = 0;  // ring unit of the current block's first V pair, and its fill count
    for (int u = blockIdx.x; u < n_items; u += gridDim.x) {
      const int t = u / G;
      const int Kt = warp_count_valid(topk_idxs + static_cast<size_t>(t) * W, W,
                                      slot_len(topk_length, t, W),
                                      kv_range(cu_q, cu_kv, B, t, S_kv), lane);
      if (Kt == 0) continue;
      const int nblk = (Kt + kBlk - 1) / kBlk;
      if (lane == 0) {
        if constexpr (!L::kQPerChunk) mbar_wait(qfull0, it & 1, fs, 2);  // the Q tile at once
        for (int b = 0; b < nblk; ++b) {
          const int g = gb + b;
          // 64 heads at D = 576: S starts on each Q chunk as it lands (first
          // block only)
          qpar = (L::kQPerChunk && b == 0) ? (it & 1) : -1;
          // rope slot of this block and its fill count (one or two slots)
          const int rs = L::kRopeSlots == 2 ? (g & 1) : 0;
          const int rw = L::kRopeSlots == 2 ? (g >> 1) : g;
          if constexpr (kRopeFirst) {
            s_chunk(rfull0 + 8 * rs, rw & 1, dr0 + static_cast<uint64_t>(rs * (kKVChunk >> 4)), 8,
                    true);
            umma_commit(rfree0 + 8 * rs);  // P lives elsewhere: the slot is free once S read it
          }
          for (int j = 0; j < 4; ++j) {
            int un = ub + j, w = wb;
            if (un >= L::kUnits) { un -= L::kUnits; ++w; }
#pragma unroll
            for (int h = 0; h < 2; ++h)
              s_chunk(vfull0 + 16 * un + 8 * h, w & 1,
                      dv0 + static_cast<uint64_t>((un * kVUnit + h * kKVChunk) >> 4), 2 * j + h,
                      !kRopeFirst && j == 0 && h == 0);
          }
          if constexpr (L::kPInRope) s_chunk(rfull0, g & 1, dr0, 8, false);
          umma_commit(smem_u32(&m.s_full));
          if (b == nblk - 1) umma_commit(smem_u32(&m.q_free));  // Q read for the last time
          mbar_wait(smem_u32(&m.p_full), g & 1, fs, 4);
          tc_fence_after();
          for (int j = 0; j < 4; ++j) {
            int un = ub + j;
            if (un >= L::kUnits) un -= L::kUnits;
            const uint64_t da = dvt0 + static_cast<uint64_t>((un * kVUnit) >> 4);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t bp = kPK ? dp0 + static_cast<uint64_t>((k >> 2) * ((kHG * 128) >> 4) + (k & 3) * 2)
                                      : dp0 + static_cast<uint64_t>(k * (2048 >> 4));
              umma_ss(tO + j * kHG, da + static_cast<uint64_t>(k * (2048 >> 4)), bp, idPV,
                      (b | k) != 0);
            }
            umma_commit(vfree0 + 8 * un);  // the unit's two chunks are read
          }
          if constexpr (L::kPInRope) umma_commit(rfree0);
          umma_commit(smem_u32(&m.o_done));
          ub += 4;
          if (ub >= L::kUnits) { ub -= L::kUnits; ++wb; }
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
    // block (its TMEM lane) and heads hb .. hb + kHT - 1, hb = kHT * (w >> 2):
    // two warps per SM sub-partition share the exp2 work of a block.
    const float sl2 = scale * kLog2e;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane, hb = (warp >> 2) * kHT;
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
      float lp[kHT];
#pragma unroll
      for (int h = 0; h < kHT; ++h) lp[h] = 0.f;

      for (int b = 0; b < nblk; ++b) {
        const int g = gb + b;
        mbar_wait(smem_u32(&m.s_full), g & 1, fs, 5);
        tc_fence_after();
        uint32_t r0[kHT];
        tmem_ld_n<kHT>(tmem + lane_base + hb, r0);
        const bool valid = b * kBlk + row < Kt;
        // Lazy rescale: a head keeps its shift unless the block's maximum
        // exceeds it by more than 2^8; the final normalisation uses the same
        // shift for O and l.  P is computed with the current shifts first:
        // a score that far above its head's shift shows as p > 2^8 (always
        // in an item's first block, whose shifts are -inf).  Only then are
        // the scores read again from TMEM (this block's S^T stays there
        // until its P.V is issued), the column maxima formed and P redone.
        const float4* mu4 = reinterpret_cast<const float4*>(m.m_used + hb);
        float p[kHT];
        bool above = false;
#pragma unroll
        for (int i = 0; i < kHT; i += 4) {
          const float4 mu = mu4[i / 4];
          const float m4[4] = {mu.x, mu.y, mu.z, mu.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float sv = valid ? __uint_as_float(r0[i + k]) * sl2 : -INFINITY;
            p[i + k] = ex2_approx(sv - m4[k]);
            above |= p[i + k] > 256.f;
          }
        }
        bool any = named_bar_or(1, kSoftmax, above);
        if (any) {
          uint32_t r1[kHT];
          tmem_ld_n<kHT>(tmem + lane_base + hb, r1);
#pragma unroll
          for (int i = 0; i < kHT; ++i) p[i] = valid ? __uint_as_float(r1[i]) * sl2 : -INFINITY;
          // column (per-head) maximum over the 128 gathered rows
          float* red = m.red[g & 1][warp & 3];
#pragma unroll
          for (int i = 0; i < kHT; ++i) {
            const float mx = warp_max(p[i]);
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
          // P with the new shifts (p[] holds the scores here)
#pragma unroll
          for (int i = 0; i < kHT; i += 4) {
            const float4 mu = mu4[i / 4];
            p[i] = ex2_approx(p[i] - mu.x);
            p[i + 1] = ex2_approx(p[i + 1] - mu.y);
            p[i + 2] = ex2_approx(p[i + 2] - mu.z);
            p[i + 3] = ex2_approx(p[i + 3] - mu.w);
          }
        }
        if (any) {
#pragma unroll
          for (int i = 0; i < kHT; ++i) lp[i] *= m.fac[hb + i];
        }
        if (any && b > 0) {
          // O^T columns of heads whose shift moved: scale by 2^(old - new).
          // The previous P.V finished before this block's S (in-order
          // completion), so the wait returns at once.
          mbar_wait(smem_u32(&m.o_done), (g - 1) & 1, fs, 6);
          tc_fence_after();
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
            const uint32_t ta = tmem + lane_base + L::kColO + j * kHG + hb;
            uint32_t r[kHT];
            tmem_ld_n<kHT>(ta, r);
#pragma unroll
            for (int i = 0; i < kHT; ++i)
              r[i] = __float_as_uint(__uint_as_float(r[i]) * m.fac[hb + i]);
            tmem_st_n<kHT>(ta, r);
          }
          tmem_wait_st();
        }
        // P^T row as bf16 pairs
        uint32_t pk[kHT / 2];
#pragma unroll
        for (int i = 0; i < kHT / 2; ++i) {
          lp[2 * i] += p[2 * i];
          lp[2 * i + 1] += p[2 * i + 1];
          pk[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
        }
        const uint32_t pt = p_tile(g);
        if constexpr (!kPK) {
          // MN-major tile that the P.V UMMA reads: this thread's heads are
          // 16-byte pieces hb / 8 .. hb / 8 + 3 of its row.
#pragma unroll
          for (int c = 0; c < kHT / 8; ++c) {
            const uint32_t dst = pt + sw128_off(row, hb / 8 + c);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[4 * c]),
                         "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                         : "memory");
          }
        } else {
          // K-major tile: head rows, slots contiguous; this thread writes
          // column `row` of its kHT head rows.
#pragma unroll
          for (int i = 0; i < kHT / 2; ++i) {
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(pt + pk_tile_off<kHG>(hb + 2 * i, row)),
                         "h"(static_cast<uint16_t>(pk[i]))
                         : "memory");
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(pt + pk_tile_off<kHG>(hb + 2 * i + 1, row)),
                         "h"(static_cast<uint16_t>(pk[i] >> 16))
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&m.p_full));
      }
      gb += nblk;

      // ---------------------------------------------------------- epilogue
      // l per head: full sums across lane groups, then a butterfly
      // reduce-scatter, leave lane L of each warp with its rows' sum for head
      // hb + (L mod kHT) in lp[0]; the four row warps' partials meet in
      // shared memory (both halves of red are free: the block loop's last
      // barrier came after their last reads).
#pragma unroll
      for (int o = 16; o >= kHT; o >>= 1) {
#pragma unroll
        for (int i = 0; i < kHT; ++i) lp[i] += __shfl_xor_sync(0xffffffffu, lp[i], o);
      }
#pragma unroll
      for (int o = kHT / 2; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float keep = up ? lp[i + o] : lp[i];
          const float send = up ? lp[i] : lp[i + o];
          lp[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      if (lane < kHT) m.red[0][warp & 3][hb + lane] = lp[0];
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
      // O^T -> out (bf16) straight from registers once the last P.V is done:
      // for each head, a warp writes 32 consecutive d of that head's row.
      mbar_wait(smem_u32(&m.o_done), (gb - 1) & 1, fs, 7);
      tc_fence_after();
      __nv_bfloat16* out_t = out + (static_cast<size_t>(t) * H + h0) * kDv;
      for (int j = 0; j < 4; ++j) {
        uint32_t r[kHT];
        tmem_ld_n<kHT>(tmem + lane_base + L::kColO + j * kHG + hb, r);
        const int d = j * 128 + row;
#pragma unroll
        for (int i = 0; i < kHT; ++i) {
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
  if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
}

template <int kD, int kHG>
cudaError_t set_fwd_smem() {
  return cudaFuncSetAttribute(fwd_kernel<kD, kHG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FwdLayout<kD, kHG>::kSmemBytes);
}

template <int kD, int kHG>
cudaError_t launch_fwd_hg(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                          const int32_t* len, const float* sink, void* out, float* lse,
                          cudaStream_t s) {
  const int G = (p.H + kHG - 1) / kHG;
  const long long items = static_cast<long long>(p.T) * G;
  if (items == 0) return cudaSuccess;
  // persistent: at most one CTA per SM, each walking its share of the items
  // (twice as many CTAs, a second wave as in the backward, is no faster here)
  const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
  CUtensorMap tm_q, tm_kv;
  const int box_heads = p.H < kHG ? p.H : kHG;  // never larger than the tensor
  cudaError_t e = make_head_tile_map(&tm_q, q, p.T, p.H, p.d_qk, box_heads);
  if (e == cudaSuccess) e = make_matrix_map(&tm_kv, kv, p.S_kv, p.d_qk, kBlk);
  if (e != cudaSuccess) return e;
  fwd_kernel<kD, kHG><<<grid, kThreads, FwdLayout<kD, kHG>::kSmemBytes, s>>>(
      tm_q, tm_kv, idx, len, sink, static_cast<__nv_bfloat16*>(out), lse,
      static_cast<const __nv_bfloat16*>(kv), p.T, p.H, p.S_kv, p.W, p.scale, G,
      p.delta_residual ? 1 : 0, box_heads, p.cu_q, p.cu_kv, p.B);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const void* q, const void* kv, const int32_t* idx,
                       const int32_t* len, const float* sink, void* out, float* lse,
                       cudaStream_t s) {
  static std::atomic<uint64_t> attr_done{0};
  const int dev = current_device();
  if (device_needs_setup(attr_done, dev)) {
    cudaError_t e = set_fwd_smem<576, 64>();
    if (e == cudaSuccess) e = set_fwd_smem<512, 64>();
    if (e == cudaSuccess) e = set_fwd_smem<576, 32>();
    if (e == cudaSuccess) e = set_fwd_smem<512, 32>();
    if (e == cudaSuccess) e = set_fwd_smem<576, 16>();
    if (e == cudaSuccess) e = set_fwd_smem<512, 16>();
    if (e != cudaSuccess) return e;
    mark_device_setup(attr_done, dev);
  }
  // The narrowest head group that holds H (the same group in every item).
  const bool d512 = p.d_qk == 512;
  if (p.H <= 16)
    return d512 ? launch_fwd_hg<512, 16>(p, q, kv, idx, len, sink, out, lse, s)
                : launch_fwd_hg<576, 16>(p, q, kv, idx, len, sink, out, lse, s);
  if (p.H <= 32)
    return d512 ? launch_fwd_hg<512, 32>(p, q, kv, idx, len, sink, out, lse, s)
                : launch_fwd_hg<576, 32>(p, q, kv, idx, len, sink, out, lse, s);
  return d512 ? launch_fwd_hg<512, 64>(p, q, kv, idx, len, sink, out, lse, s)
              : launch_fwd_hg<576, 64>(p, q, kv, idx, len, sink, out, lse, s);
}

unsigned int fwd_take_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v) cudaMemcpyToSymbol(g_err_fwd, &zero, sizeof(zero));
  return v;
}

}  // namespace dsa
