// Dense MLA split-KV decode kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (FlashMLA PR #183, "Add SM80 (Ampere/A100) dense MLA
// decode kernel", section Design): for the 128 query rows of one row block
// of a request (all heads share one latent KV head), over the keys of one
// split: S = Q K^T on 576 dims, online softmax, O = P V with V = the first
// 512 dims of the same latent rows; then O / l and the split's LSE.  Keys
// come from 64-token bf16 pages through the block table.
//
// How (GB300 design, not the page's SM80 one):
//  * TMEM holds 512 fp32 columns per SM, exactly one 128 x 512 accumulator,
//    so the two CTAs of a cluster split the value dims: rank c accumulates
//    O[:, 256c : 256c+256).  Each computes the full Q K^T itself: on this
//    part distributed shared memory moves ~14 B/clk per SM, far too little
//    to share a 32 KB score tile per page between the two CTAs.
//  * Q of the row block is the MMA A operand: dims [0, 384) sit in TMEM
//    (packed bf16 pairs, written by the softmax threads once per unit), dims
//    [384, 576) in shared memory (TMA, 128-byte swizzle).
//  * One pipeline tile = one 64-key page = nine 64-dim TMA boxes.  The four
//    boxes that are also this CTA's V (dims 256c .. 256c+255) go to a "V"
//    ring and stay until P V has run; the other five go to a "K" ring that
//    is released as soon as Q K^T has run.  Each ring has two slots and its
//    own producer warp, and Q K^T reads the K-ring boxes first, so the next
//    pages keep streaming while the softmax of the current one runs.  Pages
//    a few tiles ahead are also prefetched into L2.
//  * tcgen05.mma M=128: S (N=64) and O (N=256) accumulate in TMEM.  An MMA
//    instruction costs at least ~45 cycles to issue, so N=64 is the smallest
//    score tile that keeps the tensor pipe mostly busy, and each group of
//    MMAs is issued as one fully unrolled block.  P is written as bf16 by
//    the softmax threads into swizzled shared memory.
//  * Online softmax in the log2 domain with a lazy rescale: O is rescaled
//    only when the running max grows by more than 2^8.
// Roles: warps 0-3 softmax + epilogue + Q-to-TMEM (thread = row = TMEM lane),
//        warp 4 K-ring + Q producer, warp 5 V-ring producer,
//        warp 6 MMA issuer and TMEM owner.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

// Timeline hooks: empty in the library; an instrumented build defines
// MLA_TRACE(event, tile) to record timestamps.
#ifndef MLA_TRACE
#define MLA_TRACE(ev, tile) \
  do {                       \
  } while (0)
#endif

namespace mla {
namespace dn {

constexpr int kT = 64;                             // keys per pipeline tile (one page)
constexpr int kBoxes = 9;                          // 64-dim boxes of a 576-dim row
constexpr int kKBoxes = 5;                         // boxes only Q K^T reads
constexpr int kVBoxes = 4;                         // boxes Q K^T and P V read
constexpr int kQTmemBoxes = 6;                     // Q dims [0, 384) in TMEM
constexpr int kQSmemBoxes = kBoxes - kQTmemBoxes;  // Q dims [384, 576) in shared memory
constexpr int kQBoxBytes = kRowsPerBlock * 128;    // 128 rows x 64 bf16
constexpr int kBoxBytes = kT * 128;                // 64 keys x 64 bf16
constexpr int kKSlotBytes = kKBoxes * kBoxBytes;
constexpr int kVSlotBytes = kVBoxes * kBoxBytes;
constexpr int kSlots = 2;
constexpr int kPBytes = kRowsPerBlock * kT * 2;  // one 64-key P tile, bf16

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQSmemBoxes * kQBoxBytes;
constexpr int kOffV = kOffK + kSlots * kKSlotBytes;
constexpr int kOffP = kOffV + kSlots * kVSlotBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kNumBars = 24;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 && kKSlotBytes % 1024 == 0,
              "swizzle atoms need 1024-byte alignment");

constexpr int kThreads = 224;
constexpr int kWarpK = 4, kWarpV = 5, kWarpMma = 6;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // S: [256, 320)
constexpr uint32_t kTmemQ = 320;  // Q dims [0, 384) as packed bf16 pairs: [320, 512)

enum : int {
  Q_FULL = 0,
  Q_EMPTY = 1,
  KA_FULL = 2,   // +slot
  KA_EMPTY = 4,  // +slot
  KB_FULL = 6,   // +slot
  KB_EMPTY = 8,  // +slot
  S_FULL = 10,
  S_FREE = 11,
  P_FULL = 12,  // +buffer
  P_FREE = 14,  // +buffer
  O_FULL = 16,
  O_FREE = 17,
  DRAIN = 18,
};

#ifndef MLA_DENSE_PREFETCH_PAGES
#define MLA_DENSE_PREFETCH_PAGES 0
#endif
constexpr int kPrefetch = MLA_DENSE_PREFETCH_PAGES;  // pages prefetched into L2 ahead of the TMA loads
constexpr float kTau = 8.0f;  // lazy-rescale threshold (log2 units)
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Part {
  int b0, t0, b1, t1, s0;
};

__device__ __forceinline__ Part load_part(const int32_t* sched, int idx) {
  const int32_t* e = sched + idx * MLA_SCHED_INTS;
  return Part{e[0], e[1], e[2], e[3], e[4]};
}

__device__ __forceinline__ bool unit_in_part(const Part& P, int b, int n_units) {
  return b < n_units && (b < P.b1 || (b == P.b1 && P.t1 > 0));
}

// Walk over the pipeline tiles (unit, page) of one partition.
struct Cursor {
  int b, L, k, lo, hi;  // unit, its key count, page, page range in this partition
  int u;                // ordinal of the unit within the partition
  uint32_t t;           // ordinal of the tile within the partition
  bool valid;
};

__device__ __forceinline__ void cursor_seek(const DecodeParams& p, const Part& P, Cursor& c, int from_b) {
  for (int b = from_b; unit_in_part(P, b, p.n_units); ++b) {
    const int L = max(p.lengths[b], 0);
    const int lo = (b == P.b0) ? P.t0 : 0;
    const int hi = (b == P.b1) ? P.t1 : num_tiles(L);
    if (hi > lo) {
      c.b = b;
      c.L = L;
      c.lo = lo;
      c.hi = hi;
      c.k = lo;
      c.valid = true;
      return;
    }
  }
  c.valid = false;
}

__device__ __forceinline__ void cursor_init(const DecodeParams& p, const Part& P, Cursor& c) {
  c.u = 0;
  c.t = 0;
  cursor_seek(p, P, c, P.b0);
}

__device__ __forceinline__ bool cursor_first(const Cursor& c) { return c.k == c.lo; }
__device__ __forceinline__ bool cursor_last(const Cursor& c) { return c.k == c.hi - 1; }

__device__ __forceinline__ void cursor_next(const DecodeParams& p, const Part& P, Cursor& c) {
  ++c.t;
  if (++c.k == c.hi) {
    ++c.u;
    cursor_seek(p, P, c, c.b + 1);
  }
}

// Global box held in slot position j of this rank's K ring: the other half's
// value dims, then the RoPE box.
template <int kRank>
__host__ __device__ constexpr int k_box(int j) {
  return kRank == 0 ? 4 + j : (j < 4 ? j : 8);
}

__device__ __forceinline__ void set_abort(volatile int* abort_flag, int32_t* status, int code) {
  *abort_flag = 1;
  report(status, code);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

// Prefetch one page (all 9 boxes) into L2; bad ids are skipped.
__device__ __forceinline__ void prefetch_page(const DecodeParams& p, int pg, const CUtensorMap* kv_map) {
  if (pg < 0 || pg >= p.num_pages) return;
#pragma unroll
  for (int bx = 0; bx < kBoxes; ++bx) tma_prefetch_3d(kv_map, 64 * bx, 0, pg);
}

// Page ids of 32 consecutive pages of unit c.b starting at `base`, one per lane
// (0 past the partition's range; ids outside the pool are reported and read as 0).
__device__ __forceinline__ int load_page_window(const DecodeParams& p, const Cursor& c, int base, int lane) {
  const int kk = base + lane;
  int pg = 0;
  if (kk < c.hi) {
    pg = kk < p.max_pages ? p.block_table[static_cast<size_t>(c.b) * p.max_pages + kk] : -1;
    if (pg < 0 || pg >= p.num_pages) {
      report(p.status, MLA_ERR_BAD_INDEX);
      pg = 0;
    }
  }
  return pg;
}

// Q K^T over one 64-dim box kG (4 K-steps).  The A operand (Q) comes from TMEM
// for kG < 6, else from shared memory; B is the box in a K or V ring slot.
template <int kG>
__device__ __forceinline__ void qk_box(uint32_t d, uint32_t tmem, uint64_t q_desc0, uint64_t b_desc, bool first) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, kT, false);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t b = b_desc + static_cast<uint64_t>((k * 32) >> 4);
    if constexpr (kG < kQTmemBoxes)
      umma_f16_ts(d, tmem + kTmemQ + 32 * kG + 8 * k, b, idesc, (first && k == 0) ? 0u : 1u);
    else
      umma_f16(d, q_desc0 + static_cast<uint64_t>(((kG - kQTmemBoxes) * kQBoxBytes + k * 32) >> 4), b, idesc,
               (first && k == 0) ? 0u : 1u);
  }
}

// Q K^T over this rank's K-ring boxes (first part of the score tile).
template <int kRank>
__device__ __forceinline__ void issue_qk_k(uint32_t d, uint32_t tmem, uint64_t q_desc0, uint64_t kslot) {
  qk_box<k_box<kRank>(0)>(d, tmem, q_desc0, kslot + ((0 * kBoxBytes) >> 4), true);
  qk_box<k_box<kRank>(1)>(d, tmem, q_desc0, kslot + ((1 * kBoxBytes) >> 4), false);
  qk_box<k_box<kRank>(2)>(d, tmem, q_desc0, kslot + ((2 * kBoxBytes) >> 4), false);
  qk_box<k_box<kRank>(3)>(d, tmem, q_desc0, kslot + ((3 * kBoxBytes) >> 4), false);
  qk_box<k_box<kRank>(4)>(d, tmem, q_desc0, kslot + ((4 * kBoxBytes) >> 4), false);
}

// Q K^T over this rank's V-ring boxes (second part of the score tile).
template <int kRank>
__device__ __forceinline__ void issue_qk_v(uint32_t d, uint32_t tmem, uint64_t q_desc0, uint64_t vslot) {
  qk_box<4 * kRank + 0>(d, tmem, q_desc0, vslot + ((0 * kBoxBytes) >> 4), false);
  qk_box<4 * kRank + 1>(d, tmem, q_desc0, vslot + ((1 * kBoxBytes) >> 4), false);
  qk_box<4 * kRank + 2>(d, tmem, q_desc0, vslot + ((2 * kBoxBytes) >> 4), false);
  qk_box<4 * kRank + 3>(d, tmem, q_desc0, vslot + ((3 * kBoxBytes) >> 4), false);
}

// Q row `row` of unit b, dims [0, 384) -> this thread's TMEM lane, columns
// [kTmemQ, kTmemQ + 192): column c holds dims (2c, 2c+1) as packed bf16.
__device__ __forceinline__ void load_q_to_tmem(const DecodeParams& p, const uint16_t* q, int b, int row,
                                               uint32_t taddr) {
  const bool ok = row < p.rows;
  const uint4* src = reinterpret_cast<const uint4*>(q + (static_cast<size_t>(b) * p.rows + row) * kDqk);
#pragma unroll 1
  for (int round = 0; round < 2; ++round) {
    uint4 w[24];  // all loads of the round in flight at once
#pragma unroll
    for (int i = 0; i < 24; ++i) w[i] = ok ? __ldg(src + round * 24 + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int g = 0; g < 6; ++g) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[4 * j + 0] = w[4 * g + j].x;
        v[4 * j + 1] = w[4 * g + j].y;
        v[4 * j + 2] = w[4 * g + j].z;
        v[4 * j + 3] = w[4 * g + j].w;
      }
      tmem_st16(taddr + kTmemQ + round * 96 + g * 16, v);
    }
  }
  tmem_wait_st();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    dense_decode_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kv_map,
                        const DecodeParams p, const uint16_t* __restrict__ q) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sP = smem + kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster_id = blockIdx.x >> 1;
  const int part_idx = cluster_id / p.row_blocks;
  const int rb = cluster_id - part_idx * p.row_blocks;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bars[Q_FULL], 128 + 1);  // softmax threads (TMEM part) + K producer (TMA part)
    mbar_init(&bars[Q_EMPTY], 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bars[KA_FULL + i], 1);
      mbar_init(&bars[KA_EMPTY + i], 1);
      mbar_init(&bars[KB_FULL + i], 1);
      mbar_init(&bars[KB_EMPTY + i], 1);
    }
    mbar_init(&bars[S_FULL], 1);
    mbar_init(&bars[S_FREE], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[P_FULL + i], 128);
      mbar_init(&bars[P_FREE + i], 1);
    }
    mbar_init(&bars[O_FULL], 1);
    mbar_init(&bars[O_FREE], 128);
    mbar_init(&bars[DRAIN], 1);
    fence_mbar_init_cluster();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpK && lane == 0) {
    prefetch_tmap(&q_map);
    prefetch_tmap(&kv_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  const Part P = load_part(p.sched, part_idx);

  if (warp == kWarpK || warp == kWarpV) {
    // ------------------------------------------------------------ TMA producers
    const bool is_k = (warp == kWarpK);
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    const int full_bar = is_k ? KA_FULL : KB_FULL;
    const int empty_bar = is_k ? KA_EMPTY : KB_EMPTY;
    uint8_t* ring = is_k ? sK : sV;
    const int slot_bytes = is_k ? kKSlotBytes : kVSlotBytes;
    Cursor c;
    cursor_init(p, P, c);
    bool ok = true;
    uint32_t issued[kSlots] = {0u, 0u};
    uint32_t q_issued = 0;
    int page_reg = 0, page_base = -1, cur_b = -1;
    while (ok && c.valid) {
      if (is_k && cursor_first(c)) {
        if (lane == 0) {
          if (c.u >= 1) ok = mbar_wait(&bars[Q_EMPTY], (c.u - 1) & 1, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&bars[Q_FULL], kQSmemBoxes * kQBoxBytes);
            const int row0 = c.b * p.rows + rb * kRowsPerBlock;
#pragma unroll
            for (int i = 0; i < kQSmemBoxes; ++i)
              tma_load_2d(sQ + i * kQBoxBytes, &q_map, &bars[Q_FULL], 64 * (kQTmemBoxes + i), row0, pol_q);
            ++q_issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      // page ids of the next 32 pages of this unit, one per lane; refreshed early
      // enough that the L2 prefetch kPrefetch pages ahead stays inside the window
      const bool fresh = c.b != cur_b;
      if (fresh || c.k - page_base >= 32 - kPrefetch) {
        cur_b = c.b;
        page_base = c.k;
        page_reg = load_page_window(p, c, page_base, lane);
      }
      const int page = __shfl_sync(0xffffffffu, page_reg, c.k - page_base);
      if (is_k && kPrefetch > 0) {
        int pf[kPrefetch > 0 ? kPrefetch : 1];
#pragma unroll
        for (int i = 0; i < kPrefetch; ++i)
          pf[i] = __shfl_sync(0xffffffffu, page_reg, min(c.k + 1 + i - page_base, 31));
        if (lane == 0) {
          if (fresh) {
#pragma unroll
            for (int i = 0; i + 1 < kPrefetch; ++i)
              if (c.k + 1 + i < c.hi) prefetch_page(p, pf[i], &kv_map);
          }
          if (c.k + kPrefetch < c.hi) prefetch_page(p, pf[kPrefetch - 1], &kv_map);
        }
      }
      const int s = c.t & 1;
      if (lane == 0) {
        if (c.t >= kSlots) ok = mbar_wait(&bars[empty_bar + s], ((c.t >> 1) - 1) & 1, abort_flag);
        if (ok) {
          MLA_TRACE(is_k ? 0 : 7, c.t);
          mbar_arrive_expect_tx(&bars[full_bar + s], slot_bytes);
          uint8_t* dst = ring + s * slot_bytes;
          if (is_k) {
#pragma unroll
            for (int j = 0; j < kKBoxes; ++j) {
              const int g = rank == 0 ? k_box<0>(j) : k_box<1>(j);
              tma_load_3d(dst + j * kBoxBytes, &kv_map, &bars[full_bar + s], 64 * g, 0, page, pol_kv);
            }
          } else {
#pragma unroll
            for (int j = 0; j < kVBoxes; ++j)
              tma_load_3d(dst + j * kBoxBytes, &kv_map, &bars[full_bar + s], 64 * (4 * static_cast<int>(rank) + j),
                          0, page, pol_kv);
          }
          ++issued[s];
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      cursor_next(p, P, c);
    }
    if (lane == 0) {
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // no TMA write may land after this CTA exits
      for (int s = 0; s < kSlots; ++s)
        if (issued[s] > 0) mbar_wait(&bars[full_bar + s], (issued[s] - 1) & 1, nullptr);
      if (q_issued > 0) mbar_wait(&bars[Q_FULL], (q_issued - 1) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_bf16_f32(128, 256, true);
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t vk_desc0 = sdesc_sw128(smem_u32(sV), 16, 1024);        // V boxes as K-major B of Q K^T
      const uint64_t vv_desc0 = sdesc_sw128(smem_u32(sV), kBoxBytes, 1024);  // V boxes as MN-major B of P V
      const uint64_t p_desc0 = sdesc_sw128(smem_u32(sP), 16, 1024);
      // Three jobs per tile, issued as soon as their inputs are ready, in the
      // priority P V > Q K^T (V-ring part) > Q K^T (K-ring part):
      //   QKa(t): needs the K slot, S read by the softmax of t-1, Q of the unit
      //   QKb(t): needs QKa(t) issued and the V slot; completes S(t)
      //   PV(t):  needs QKb(t) issued and P(t)
      Cursor ca, cb, cv;
      cursor_init(p, P, ca);
      cursor_init(p, P, cb);
      cursor_init(p, P, cv);
      bool ok = true;
      uint64_t t_last = globaltimer_ns();
      while (cv.valid) {
        bool progressed = false;
        if (cv.t < cb.t) {
          const int pb = cv.t & 1;
          const bool first = cursor_first(cv);
          bool ready = mbar_test_wait(&bars[P_FULL + pb], (cv.t >> 1) & 1);
          if (ready && first && cv.u >= 1) ready = mbar_test_wait(&bars[O_FREE], (cv.u - 1) & 1);
          if (ready) {
            MLA_TRACE(3, cv.t);
            tc_fence_after();
            const uint64_t a0 = p_desc0 + static_cast<uint64_t>((pb * kPBytes) >> 4);
            const uint64_t b0 = vv_desc0 + static_cast<uint64_t>((pb * kVSlotBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              umma_f16(tmem + kTmemO, a0 + static_cast<uint64_t>((kk * 32) >> 4),
                       b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (first && kk == 0) ? 0u : 1u);
            umma_commit(&bars[P_FREE + pb]);
            umma_commit(&bars[KB_EMPTY + pb]);
            if (cursor_last(cv)) umma_commit(&bars[O_FULL]);
            cursor_next(p, P, cv);
            progressed = true;
          }
        }
        if (!progressed && cb.t < ca.t) {
          const int s = cb.t & 1;
          if (mbar_test_wait(&bars[KB_FULL + s], (cb.t >> 1) & 1)) {
            MLA_TRACE(8, cb.t);
            tc_fence_after();
            const uint64_t vslot = vk_desc0 + static_cast<uint64_t>((s * kVSlotBytes) >> 4);
            if (rank == 0)
              issue_qk_v<0>(tmem + kTmemS, tmem, q_desc0, vslot);
            else
              issue_qk_v<1>(tmem + kTmemS, tmem, q_desc0, vslot);
            umma_commit(&bars[S_FULL]);
            umma_commit(&bars[KA_EMPTY + s]);
            MLA_TRACE(2, cb.t);
            if (cursor_last(cb)) umma_commit(&bars[Q_EMPTY]);
            cursor_next(p, P, cb);
            progressed = true;
          }
        }
        if (!progressed && ca.valid && ca.t == cb.t) {
          const int s = ca.t & 1;
          bool ready = true;
          if (cursor_first(ca)) ready = mbar_test_wait(&bars[Q_FULL], ca.u & 1);
          ready = ready && mbar_test_wait(&bars[KA_FULL + s], (ca.t >> 1) & 1);
          if (ready && ca.t >= 1) ready = mbar_test_wait(&bars[S_FREE], (ca.t - 1) & 1);
          if (ready) {
            MLA_TRACE(1, ca.t);
            tc_fence_after();
            const uint64_t kslot = k_desc0 + static_cast<uint64_t>((s * kKSlotBytes) >> 4);
            if (rank == 0)
              issue_qk_k<0>(tmem + kTmemS, tmem, q_desc0, kslot);
            else
              issue_qk_k<1>(tmem + kTmemS, tmem, q_desc0, kslot);
            cursor_next(p, P, ca);
            progressed = true;
          }
        }
        if (progressed) {
          t_last = globaltimer_ns();
        } else {
          if (*abort_flag || globaltimer_ns() - t_last > MLA_WAIT_LIMIT_NS) {
            ok = false;
            break;
          }
          __nanosleep(20);
        }
      }
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // every MMA has completed before TMEM is released
      umma_commit(&bars[DRAIN]);
      mbar_wait(&bars[DRAIN], 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = tid;  // row of the block == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    const int row = rb * kRowsPerBlock + r;
    const bool row_ok = row < p.rows;
    const int tok = row_ok ? row / p.h_q : 0;
    const float c_log2 = p.scale_log2;
    Cursor c;
    cursor_init(p, P, c);
    bool ok = true;
    if (c.valid) {  // Q of the first unit
      load_q_to_tmem(p, q, c.b, row, tmem + lane_base);
      tc_fence_before();
      mbar_arrive(&bars[Q_FULL]);
    }
    float m_used = -INFINITY, l_sum = 0.f;  // running max (log2 units) and fp32 row sum
    while (ok && c.valid) {
      const uint32_t t = c.t;
      const bool first = cursor_first(c), last = cursor_last(c);
      if (first) {
        m_used = -INFINITY;
        l_sum = 0.f;
      }
      const int jmax = p.causal ? (c.L - p.s_q + tok) : (c.L - 1);  // last visible key
      const int vis = jmax - c.k * kT;                                // keys 0..vis of this tile are visible
      ok = warp_wait(&bars[S_FULL], t & 1, abort_flag);
      if (!ok) break;
      if (tid == 0) MLA_TRACE(4, t);
      tc_fence_after();
      float s[kT];
      {
        uint32_t (&lo32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
        uint32_t (&hi32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
        tmem_ld32(tmem + lane_base + kTmemS, lo32);
        tmem_ld32(tmem + lane_base + kTmemS + 32u, hi32);
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(&bars[S_FREE]);
      const int b_here = c.b, u_here = c.u;
      // masked keys -> -inf; raw tile max (the scale is positive, so max commutes with it)
      if (vis < kT - 1) {
#pragma unroll
        for (int j = 0; j < kT; ++j)
          if (j > vis) s[j] = -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
      for (int j = 16; j < kT; j += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], s[j + i]);
      const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float mt = mraw * c_log2;  // -inf stays -inf
      bool rescale = false;
      float alpha = 1.f;
      if (mt > m_used + kTau) {
        alpha = ex2(m_used - mt);  // 0 when m_used == -inf
        rescale = !first;
        l_sum *= alpha;
        m_used = mt;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      uint32_t pk[kT / 2];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kT / 2; ++i) {
        const float p0 = ex2(fmaf(s[2 * i], c_log2, -mref));
        const float p1 = ex2(fmaf(s[2 * i + 1], c_log2, -mref));
        const __nv_bfloat162 hv = __floats2bfloat162_rn(p0, p1);
        pk[i] = *reinterpret_cast<const uint32_t*>(&hv);
        ls[i & 3] += p0 + p1;
      }
      l_sum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      const int pb = t & 1;
      if (t >= 2) {
        ok = warp_wait(&bars[P_FREE + pb], ((t - 2) >> 1) & 1, abort_flag);
        if (!ok) break;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O accumulated so far (through P V of the previous tile) times alpha
        ok = warp_wait(&bars[P_FREE + (pb ^ 1)], ((t - 1) >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (uint32_t c0 = 0; c0 < 256; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + kTmemO + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st16(tmem + lane_base + kTmemO + c0, v);
        }
        tmem_wait_st();
      }
      // P row: 64 keys = eight 16-byte chunks of the 128-byte swizzled row
      uint8_t* prow = sP + pb * kPBytes + r * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(prow + ((static_cast<uint32_t>(cc) ^ swz) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[P_FULL + pb]);
      if (tid == 0) MLA_TRACE(5, t);
      cursor_next(p, P, c);
      if (!last) continue;
      if (c.valid) {
        // Q of this unit is no longer read (its last Q K^T finished): stage the next unit's Q
        ok = warp_wait(&bars[Q_EMPTY], u_here & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        load_q_to_tmem(p, q, c.b, row, tmem + lane_base);
        tc_fence_before();
        mbar_arrive(&bars[Q_FULL]);
      }
      // ---- epilogue of this (unit, split)
      ok = warp_wait(&bars[O_FULL], u_here & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int s_begin = p.split_offset[b_here];
      const int nsplit = p.split_offset[b_here + 1] - s_begin;
      const int slot = s_begin + ((b_here == P.b0) ? P.s0 : 0);
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const size_t orow = static_cast<size_t>(b_here) * p.rows + row;
      const size_t arow = static_cast<size_t>(slot) * p.rows + row;
      const bool direct = (nsplit == 1);
      const bool bf16_out = direct && !p.out_fp32;
      // O half -> global through the two P buffers (free: the unit's last P V
      // has completed): each thread stages its row's 128 bytes of a column
      // chunk, then the 128 threads store 16-byte pieces so that each warp
      // writes whole 128-byte row segments.
      const int chunk_cols = bf16_out ? 64 : 32;  // 128 bytes of output per row
      const size_t base_row = direct ? static_cast<size_t>(b_here) * p.rows : static_cast<size_t>(slot) * p.rows;
#pragma unroll 1
      for (int ch = 0; ch < 256 / chunk_cols; ++ch) {
        uint8_t* stage = sP + (ch & 1) * kPBytes;
        uint32_t w[32];
        if (bf16_out) {
          uint32_t v[32];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tmem_ld32(tmem + lane_base + kTmemO + 64 * ch + 32 * hh, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const __nv_bfloat162 hv =
                  __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
              w[16 * hh + i] = *reinterpret_cast<const uint32_t*>(&hv);
            }
          }
        } else {
          tmem_ld32(tmem + lane_base + kTmemO + 32 * ch, w);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * inv_l);
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(stage + r * 128 + ((static_cast<uint32_t>(cc) ^ swz) << 4)) =
              make_uint4(w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
        named_bar_sync(1, 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int flat = tid + 128 * i;
          const int rr = flat >> 3, cc = flat & 7;
          const int rg = rb * kRowsPerBlock + rr;
          if (rg >= p.rows) continue;
          const uint4 val =
              *reinterpret_cast<const uint4*>(stage + rr * 128 + ((static_cast<uint32_t>(cc ^ (rr & 7))) << 4));
          const size_t e = (base_row + rg) * kDv + 256u * rank + static_cast<size_t>(ch) * chunk_cols;
          if (bf16_out)
            reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + e)[cc] = val;
          else
            reinterpret_cast<uint4*>((direct ? static_cast<float*>(p.out) : p.o_accum) + e)[cc] = val;
        }
      }
      named_bar_sync(1, 128);  // staging reads done before the next unit writes P
      (void)orow;
      (void)arow;
      tc_fence_before();
      mbar_arrive(&bars[O_FREE]);
      if (tid == 0) MLA_TRACE(6, t);
      if (rank == 0 && row_ok) {
        const size_t orow = static_cast<size_t>(b_here) * p.rows + row;
        const size_t arow = static_cast<size_t>(slot) * p.rows + row;
        const float lse = l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
        if (direct)
          p.lse[orow] = lse;
        else
          p.lse_accum[arow] = lse;
      }
    }
    if (!ok && lane == 0) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace dn

int dense_smem_bytes() { return dn::kSmemBytes; }
int dense_threads() { return dn::kThreads; }
const void* dense_kernel_ptr() { return reinterpret_cast<const void*>(&dn::dense_decode_kernel); }

cudaError_t launch_dense(const CUtensorMap& q_map, const CUtensorMap& kv_map, const DecodeParams& p, const void* q,
                         int num_parts, cudaStream_t stream) {
  const dim3 grid(2 * num_parts * p.row_blocks);
  dn::dense_decode_kernel<<<grid, dn::kThreads, dn::kSmemBytes, stream>>>(q_map, kv_map, p,
                                                                         static_cast<const uint16_t*>(q));
  return cudaGetLastError();
}

}  // namespace mla
