// Dense MLA split-KV decode kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (FlashMLA PR #183, "Add SM80 (Ampere/A100) dense MLA
// decode kernel", section Design): for the 128 query rows of one row block
// of a request (all heads share one latent KV head), over the keys of one
// split: S = Q K^T on 576 dims, online softmax, O = P V with V = the first
// 512 dims of the same latent rows; then O / l and the split's LSE.  Keys
// come from 64-token pages (bf16 or fp16, one or more latent KV heads)
// through the block table.
//
// How (GB300 design, not the page's SM80 one):
//  * TMEM holds 512 fp32 columns per SM, exactly one 128 x 512 accumulator,
//    so the two CTAs of a cluster split the value dims: rank c accumulates
//    O[:, 256c : 256c+256).
//  * The two CTAs take turns on the pipeline tiles (one 64-key page each):
//    tile t is "owned" by rank t & 1, which alone computes S = Q K^T for it,
//    its softmax and its P.  The owner sends P (16 KB of bf16) to the other
//    CTA with asynchronous bulk copies into distributed shared memory, and
//    both run P V for their own value half.  Every score
//    is computed once; only P crosses between the SMs.
//  * Both halves of O must use the same softmax reference.  The reference
//    after tile t is R_t = the running max (log2 units), raised only when a
//    tile's max exceeds it by more than 2^8 (lazy rescale).  Each CTA derives
//    every R_t itself, by that rule, from the raw row maxima of all tiles in
//    order: its own tiles' and the other CTA's, which arrive as 128 floats in
//    a small mailbox in distributed shared memory (one 4-byte remote store
//    per row, which takes no TMA instruction), sent as soon as the owner has
//    read the tile's scores, long before its P.  The same fp32 comparisons
//    in the same order give both CTAs the same references.  When R changes,
//    both CTAs rescale their O half in TMEM before that tile's P V.  Each CTA
//    keeps the row sum l of its own tiles only (rescaled on every reference
//    change); the two are added once per unit, before the epilogue, through
//    a second mailbox.
//  * The P V of a received tile waits only for its P to land (the P V thread
//    watches the copy's barrier) and for the softmax threads' go, given as
//    soon as the tile's reference is known.
//  * Q of the row block is the MMA A operand: dims [0, 384) sit in TMEM
//    (packed bf16 pairs), dims [384, 576) in shared memory (TMA, 128-byte
//    swizzle).  A Q warp streams a unit's nine 64-dim Q boxes through the
//    three box slots of that shared-memory buffer; the Q K^T thread moves
//    boxes 0-5 (dims [0, 384)) into TMEM with tcgen05.cp as they land, and
//    boxes 6-8 stay.  The next unit's Q is prefetched into L2 meanwhile, and
//    the softmax warps write the epilogue while Q streams in.  (Instance
//    kQV: the first unit's nine boxes load at once, boxes 0-5 staged in the
//    still-empty V ring.)
//  * One tile = nine 64-dim slices (8 KB swizzled boxes) of one page.  The
//    four that are this CTA's V half go to a 3-slot "V" ring for every tile
//    (P V reads them; for its own tiles Q K^T reads them too); the other five
//    go to a "K" slot, for own tiles only, released as soon as Q K^T has read
//    them.  Each range of consecutive slices comes in ONE TMA
//    instruction (a 5-D box of four or five slices; rank 1's K slot takes
//    two): the TMA engine's time goes mostly per instruction, so that moves
//    the same bytes with a third of the engine time of 8 KB boxes.
//  * tcgen05.mma M=128: S (N=64) and O (N=256) accumulate in TMEM; each
//    group of MMAs is one fully unrolled block of compile-time descriptors.
// Roles: warps 0-3 softmax + epilogue (thread = row = TMEM lane),
//        warp 4 K-slot producer, warp 5 V-ring producer,
//        warp 6 Q K^T issuer (and Q copies into TMEM) and TMEM owner,
//        warp 7 Q producer, warp 8 P V issuer.
//        Q K^T and P V come from two threads so that a ready P V does not
//        wait for a Q K^T block to finish issuing; they touch different TMEM
//        accumulators.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

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
constexpr int kKBoxes = 5;                         // boxes only Q K^T reads
constexpr int kVBoxes = 4;                         // boxes Q K^T and P V read
constexpr int kQTmemBoxes = 6;                     // Q dims [0, 384) in TMEM
constexpr int kQSmemBoxes = 3;                     // Q dims [384, 576) in shared memory
constexpr int kQBoxBytes = kRowsPerBlock * 128;    // 128 rows x 64 bf16
constexpr int kBoxBytes = kT * 128;                // 64 keys x 64 bf16
constexpr int kKSlotBytes = kKBoxes * kBoxBytes;
constexpr int kVSlotBytes = kVBoxes * kBoxBytes;
constexpr int kKSlots = 1;
constexpr int kVSlots = 3;
constexpr int kPBytes = kRowsPerBlock * kT * 2;    // one 64-key P tile, bf16
constexpr int kWarpPBytes = 32 * 128;              // the 32 P rows of one softmax warp
constexpr int kVecBytes = kRowsPerBlock * 4;       // one fp32 per row (references, row sums)

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQSmemBoxes * kQBoxBytes;
constexpr int kOffV = kOffK + kKSlots * kKSlotBytes;
constexpr int kOffPOwn = kOffV + kVSlots * kVSlotBytes;
constexpr int kOffPRecv = kOffPOwn + kPBytes;
constexpr int kOffRefIn = kOffPRecv + kPBytes;     // mailbox: the peer's raw tile maxima
constexpr int kOffLOut = kOffRefIn + kVecBytes;    // this CTA's row sums, staged
constexpr int kOffLIn = kOffLOut + kVecBytes;      // mailbox: the peer's row sums
constexpr int kOffBar = kOffLIn + kVecBytes;

enum : int {
  Q_EMPTY = 0,                    // the unit's last Q K^T is done: Q may be replaced
  QB_FULL = 1,                    // +slot: a Q box has landed in that slot of the Q buffer (TMA bytes)
  QB_EMPTY = QB_FULL + kQSmemBoxes,  // +slot: the box in that slot has been copied into TMEM
  K_FULL = QB_EMPTY + kQSmemBoxes,   // +slot
  K_EMPTY = K_FULL + kKSlots,     // +slot
  V_FULL = K_EMPTY + kKSlots,     // +slot
  V_EMPTY = V_FULL + kVSlots,     // +slot
  S_FULL = V_EMPTY + kVSlots,
  S_FREE,
  OWN_GO,     // softmax -> P V thread: P of an own tile written, O rescaled
  OWN_FREE,   // own P buffer reusable: own P V done + the peer's P V done (its multicast commit)
  RECV_FULL,  // the peer's P has landed (bulk-copy bytes); watched and re-armed by the P V thread
  RECV_GO,    // softmax -> P V thread: received tile's reference applied (O rescaled if it changed)
  R_FULL,     // raw-maximum mailbox filled (remote-store bytes)
  R_FREE,     // the peer has read our last references (one remote arrival per warp)
  L_FULL,     // row-sum mailbox filled (bulk-copy bytes)
  L_FREE,     // the peer has read our last row sums (one remote arrival per warp)
  PV_DONE,    // +(t&1): one completion per P V of a tile of that parity, in tile order
  O_FULL = PV_DONE + 2,
  O_FREE,
  DRAIN,
  VQ_FULL,   // V-ring Q stage: the first unit's Q boxes 0-5 have landed in the V ring
  VQ_EMPTY,  // ... and have been copied into TMEM: the V ring is free
  kNumBars
};

constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffPOwn % 1024 == 0 && kOffPRecv % 1024 == 0 &&
                  kKSlotBytes % 1024 == 0 && kVSlotBytes % 1024 == 0,
              "swizzle atoms need 1024-byte alignment");
static_assert(kOffRefIn % 16 == 0 && kOffLOut % 16 == 0 && kOffLIn % 16 == 0,
              "bulk copies need 16-byte alignment");

constexpr int kThreads = 288;
constexpr int kWarpK = 4, kWarpV = 5, kWarpMma = 6, kWarpQ = 7, kWarpPV = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // S: [256, 320)
constexpr uint32_t kTmemQ = 320;  // Q dims [0, 384) as packed bf16 pairs: [320, 512)

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

// Global box held in slot position j of this rank's K slot: the other half's
// value dims, then the RoPE box.
template <int kRank>
__host__ __device__ constexpr int k_box(int j) {
  return kRank == 0 ? 4 + j : (j < 4 ? j : 8);
}

// Wait budget of the stall-test instance (kStall): short, so that its test
// ends quickly; the other instances keep the 2 s budget of every wait.
constexpr uint64_t kStallWaitNs = 200000;  // 200 us

// tcgen05.ld of 32 columns (as tmem_ld32) that also returns the maximum of
// the 32 fp32 values this thread loaded (valid after tcgen05.wait::ld).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr));
}

__device__ __forceinline__ void set_abort(volatile int* abort_flag, int32_t* status, int code) {
  *abort_flag = 1;
  report(status, code);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, limit_ns));
}

__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait<true>(bar, parity, abort_flag, limit_ns));
}

// Page ids of 32 consecutive pages of unit c.b starting at `base`, one per lane
// (0 past the partition's range; ids outside the pool are reported and read
// as page 0, whose keys the softmax then masks).
__device__ __forceinline__ int load_page_window(const DecodeParams& p, const Cursor& c, int base, int lane) {
  const int kk = base + lane;
  int pg = 0;
  if (kk < c.hi) {
    pg = kk < p.max_pages ? p.block_table[static_cast<size_t>(c.b) * p.max_pages + kk] : -1;
    if (pg < 0 || pg >= p.num_pages) {
      report(p.status, MLA_ERR_BAD_INDEX);
      pg = -1;
    }
  }
  return pg;
}

// Q K^T over one 64-dim box kG (4 K-steps).  The A operand (Q) comes from TMEM
// for kG < 6, else from shared memory; B is the box in the K slot or V ring.
template <bool kHalf, int kG>
__device__ __forceinline__ void qk_box(uint32_t d, uint32_t tmem, uint64_t q_desc0, uint64_t b_desc, bool first) {
  constexpr uint32_t idesc = idesc_16bit_f32(128, kT, false, kHalf);
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

// Q K^T over this rank's K-slot boxes (first part of the score tile).
template <bool kHalf, int kRank>
__device__ __forceinline__ void issue_qk_k(uint32_t d, uint32_t tmem, uint64_t q_desc0, uint64_t kslot) {
  qk_box<kHalf, k_box<kRank>(0)>(d, tmem, q_desc0, kslot + ((0 * kBoxBytes) >> 4), true);
  qk_box<kHalf, k_box<kRank>(1)>(d, tmem, q_desc0, kslot + ((1 * kBoxBytes) >> 4), false);
  qk_box<kHalf, k_box<kRank>(2)>(d, tmem, q_desc0, kslot + ((2 * kBoxBytes) >> 4), false);
  qk_box<kHalf, k_box<kRank>(3)>(d, tmem, q_desc0, kslot + ((3 * kBoxBytes) >> 4), false);
  qk_box<kHalf, k_box<kRank>(4)>(d, tmem, q_desc0, kslot + ((4 * kBoxBytes) >> 4), false);
}

// Q K^T over this rank's V-ring boxes (second part of the score tile).
template <bool kHalf, int kRank>
__device__ __forceinline__ void issue_qk_v(uint32_t d, uint32_t tmem, uint64_t q_desc0, uint64_t vslot) {
  qk_box<kHalf, 4 * kRank + 0>(d, tmem, q_desc0, vslot + ((0 * kBoxBytes) >> 4), false);
  qk_box<kHalf, 4 * kRank + 1>(d, tmem, q_desc0, vslot + ((1 * kBoxBytes) >> 4), false);
  qk_box<kHalf, 4 * kRank + 2>(d, tmem, q_desc0, vslot + ((2 * kBoxBytes) >> 4), false);
  qk_box<kHalf, 4 * kRank + 3>(d, tmem, q_desc0, vslot + ((3 * kBoxBytes) >> 4), false);
}

// Two fp32 -> one packed pair of 16-bit floats (round to nearest even).
template <bool kHalf>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (kHalf) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Row r of a CTA's 128-row block -> its row within the request's s_q * h_q
// query rows (token-major); false for a padding row.  h_kv = 1: 128
// consecutive rows per block.  h_kv > 1: block rb of head group grp holds
// block_tokens whole tokens of that group's group_heads heads.
__device__ __forceinline__ bool block_row(const DecodeParams& p, int grp, int rb, int r, int& qrow, int& tok) {
  if (p.h_kv == 1) {
    qrow = rb * kRowsPerBlock + r;
    tok = qrow / p.h_q;
    return qrow < p.rows;
  }
  const int t = r / p.group_heads;
  tok = rb * p.block_tokens + t;
  qrow = tok * p.h_q + grp * p.group_heads + (r - t * p.group_heads);
  return t < p.block_tokens && tok < p.s_q;
}

// O half (this thread's row) *= alpha.
__device__ __forceinline__ void rescale_o(uint32_t taddr, float alpha) {
#pragma unroll 1
  for (uint32_t c0 = 0; c0 < 256; c0 += 16) {
    uint32_t v[16];
    tmem_ld16(taddr + kTmemO + c0, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
    tmem_st16(taddr + kTmemO + c0, v);
  }
  tmem_wait_st();
}

// O-rescale factor between two references; 1 when unchanged (also when both
// are -inf), 0 when the old one is -inf and the new one finite.
__device__ __forceinline__ float ref_alpha(float r_old, float r_new) {
  return r_new == r_old ? 1.f : ex2(r_old - r_new);
}

// kQV: the first unit's Q boxes 0-5 are staged in the (still empty) V ring
// and all nine boxes load at once (a separate instance, chosen when many
// partitions share each request, so that the other instances keep their
// code unchanged).
// kHalf: Q and KV are fp16 (else bf16).  The three maps view the 16-bit
// pool with boxes of 4, 5 and 1 consecutive 64-dim slices (kv_map, sc_map,
// rope_map).
template <bool kHalf, bool kQV, bool kStall>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    dense_decode_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kv_map,
                        const __grid_constant__ CUtensorMap sc_map, const __grid_constant__ CUtensorMap rope_map,
                        const DecodeParams p) {
  constexpr uint64_t kWaitNs = kStall ? kStallWaitNs : MLA_WAIT_LIMIT_NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sPOwn = smem + kOffPOwn;
  uint8_t* sPRecv = smem + kOffPRecv;
  float* sRefIn = reinterpret_cast<float*>(smem + kOffRefIn);
  float* sLOut = reinterpret_cast<float*>(smem + kOffLOut);
  float* sLIn = reinterpret_cast<float*>(smem + kOffLIn);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  volatile int* sBad = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);  // [2]: own tile's page outside the pool

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // Q rows staged per box: 128 (h_kv = 1) or the group's block_tokens tokens
  const uint32_t q_box_bytes =
      (p.h_kv == 1 ? kRowsPerBlock : p.group_heads * p.block_tokens) * 128u;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster_id = blockIdx.x >> 1;
  const int part_idx = cluster_id / p.row_blocks;
  const int blk = cluster_id - part_idx * p.row_blocks;
  const int grp = blk / p.blocks_per_group;  // KV head group (0 when h_kv = 1)
  const int rb = blk - grp * p.blocks_per_group;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bars[Q_EMPTY], 1);
    for (int i = 0; i < kQSmemBoxes; ++i) {
      mbar_init(&bars[QB_FULL + i], 1);
      mbar_init(&bars[QB_EMPTY + i], 1);
    }
    mbar_init(&bars[VQ_FULL], 1);
    mbar_init(&bars[VQ_EMPTY], 1);
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(&bars[K_FULL + i], 1);
      mbar_init(&bars[K_EMPTY + i], 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(&bars[V_FULL + i], 1);
      mbar_init(&bars[V_EMPTY + i], 1);
    }
    mbar_init(&bars[S_FULL], 1);
    mbar_init(&bars[S_FREE], 128);
    mbar_init(&bars[OWN_GO], 128);
    mbar_init(&bars[OWN_FREE], 2);
    mbar_init(&bars[RECV_FULL], 1);
    mbar_init(&bars[RECV_GO], 128);
    mbar_init(&bars[R_FULL], 1);
    mbar_init(&bars[R_FREE], 4);
    mbar_init(&bars[L_FULL], 1);
    mbar_init(&bars[L_FREE], 4);
    mbar_init(&bars[PV_DONE], 1);
    mbar_init(&bars[PV_DONE + 1], 1);
    mbar_init(&bars[O_FULL], 1);
    mbar_init(&bars[O_FREE], 128);
    mbar_init(&bars[DRAIN], 2);  // the Q K^T issuer and the P V issuer
    fence_mbar_init_cluster();
    // armed for the first P, references and row sums the peer will send
    mbar_arrive_expect_tx(&bars[RECV_FULL], kPBytes);
    mbar_arrive_expect_tx(&bars[R_FULL], kVecBytes);
    mbar_arrive_expect_tx(&bars[L_FULL], kVecBytes);
  }
  static_assert(kVSlots * kVSlotBytes == 6 * kQBoxBytes, "the V ring holds Q boxes 0-5 at the start");
  if (q_box_bytes < static_cast<uint32_t>(kQBoxBytes)) {
    // Q boxes of a head group cover fewer than 128 rows: the rows past them stay
    // zero (in the Q buffer, and in the V ring where the first unit's Q lands)
    for (int i = tid; i < kQSmemBoxes * kQBoxBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (kQV)
      for (int i = tid; i < 6 * kQBoxBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(sV)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpQ && lane == 0) prefetch_tmap(&q_map);
  if (warp == kWarpK && lane == 0) prefetch_tmap(&kv_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // the peer's barriers are initialised before any remote access
  cluster_wait();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  const Part P = load_part(p.sched, part_idx);
  bool aborted = false;
  uint32_t r_seen = 0, l_seen = 0;  // reference / row-sum messages received (armed phases)

  if (warp == kWarpK || warp == kWarpV) {
    // ------------------------------------------------------------ TMA producers
    const bool is_k = (warp == kWarpK);
    const uint64_t pol_kv = policy_evict_first();
    Cursor c;
    int page_reg = 0, page_base = -1, cur_b = -1;
    cursor_init(p, P, c);
    bool ok = true;
    uint32_t k_issued[kKSlots] = {}, v_issued[kVSlots] = {};
    uint32_t own_k = 0;
    while (ok && c.valid) {
      const bool mine = (c.t & 1u) == rank;
      if (!is_k || mine) {
        // page ids of the next 32 pages of this unit, one per lane
        if (c.b != cur_b || c.k - page_base >= 32) {
          cur_b = c.b;
          page_base = c.k;
          page_reg = load_page_window(p, c, page_base, lane);
        }
        const int page_raw = __shfl_sync(0xffffffffu, page_reg, c.k - page_base);
        const int page = max(page_raw, 0);  // a page outside the pool (-1) reads page 0
        if (lane == 0) {
          if (is_k) {
            const uint32_t n = own_k / kKSlots;
            const int s = static_cast<int>(own_k % kKSlots);
            if (n >= 1) ok = mbar_wait(&bars[K_EMPTY + s], (n - 1) & 1, abort_flag, kWaitNs);
            // the stall-test instance never loads its first own tile's K slot
            if (kStall && own_k == 0) {
              // nothing issued: the Q K^T thread's wait for this slot runs out
            } else if (ok) {
              // the softmax masks this own tile's keys if its page was outside
              // the pool; written once the previous own tile's Q K^T has read
              // the K slot, hence after the softmax read the entry's last use
              // (that Q K^T waited for the scores two own tiles back to be read)
              sBad[own_k & 1] = page_raw < 0 ? 1 : 0;
              __threadfence_block();
              MLA_TRACE(9, c.t);
              uint8_t* dst = sK + s * kKSlotBytes;
              mbar_arrive_expect_tx(&bars[K_FULL + s], kKSlotBytes);
              if (rank == 0) {
                tma_load_5d(dst, &sc_map, &bars[K_FULL + s], 0, 0, k_box<0>(0), grp, page, pol_kv);
              } else {
                tma_load_5d(dst, &kv_map, &bars[K_FULL + s], 0, 0, k_box<1>(0), grp, page, pol_kv);
                tma_load_5d(dst + 4 * kBoxBytes, &rope_map, &bars[K_FULL + s], 0, 0, k_box<1>(4), grp, page,
                            pol_kv);
              }
              ++k_issued[s];
            }
          } else {
            const uint32_t n = c.t / kVSlots;
            const int s = static_cast<int>(c.t % kVSlots);
            if (n >= 1) ok = mbar_wait(&bars[V_EMPTY + s], (n - 1) & 1, abort_flag, kWaitNs);
            // V-ring Q stage: the ring holds the first unit's Q until it is in TMEM
            if constexpr (kQV) {
              if (c.t == 0 && ok) ok = mbar_wait(&bars[VQ_EMPTY], 0, abort_flag, kWaitNs);
            }
            if (ok) {
              MLA_TRACE(7, c.t);
              uint8_t* dst = sV + s * kVSlotBytes;
              mbar_arrive_expect_tx(&bars[V_FULL + s], kVSlotBytes);
              tma_load_5d(dst, &kv_map, &bars[V_FULL + s], 0, 0, 4 * static_cast<int>(rank), grp, page, pol_kv);
              ++v_issued[s];
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (is_k && mine) ++own_k;
      cursor_next(p, P, c);
    }
    if (lane == 0) {
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // no TMA write may land after this CTA exits
      for (int s = 0; s < kKSlots; ++s)
        if (k_issued[s] > 0) mbar_wait(&bars[K_FULL + s], (k_issued[s] - 1) & 1, nullptr, kWaitNs);
      for (int s = 0; s < kVSlots; ++s)
        if (v_issued[s] > 0) mbar_wait(&bars[V_FULL + s], (v_issued[s] - 1) & 1, nullptr, kWaitNs);
    }
    __syncwarp();
  } else if (warp == kWarpQ) {
    // ------------------------------------------------------------ Q producer
    // Per unit, the nine 64-dim boxes of Q in order through the three slots
    // of the shared-memory Q buffer: box j goes to slot j % 3.  Boxes 0-5
    // (dims [0, 384)) are copied into TMEM by the Q K^T thread, which frees
    // the slot for box j + 3; boxes 6-8 stay until the unit's last Q K^T.
    if (kQV && lane == 0) {
      // V-ring instance.  The first unit: boxes 0-5 go into the V
      // ring, still empty at the start (the Q K^T thread copies them into TMEM
      // and frees the ring for the V producer), boxes 6-8 into the Q slots,
      // all nine at once.  Later units: box j through slot j % 3 as below.
      const uint64_t pol_q = policy_evict_last();
      Cursor c;
      cursor_init(p, P, c);
      bool ok = true;
      uint32_t qb_issued[kQSmemBoxes] = {}, vq_issued = 0;
      // box j of unit b into dst; into L2 only when bar is null
      auto q_box = [&](int b, int j, uint8_t* dst, uint64_t* bar) {
        if (p.h_kv == 1) {
          const int row0 = b * p.rows + rb * kRowsPerBlock;
          if (bar)
            tma_load_2d(dst, &q_map, bar, 64 * j, row0, pol_q);
          else
            tma_prefetch_2d(&q_map, 64 * j, row0);
        } else {
          // [batch * s_q][h_kv][group_heads][576]: block_tokens tokens of head group grp
          const int tok0 = b * p.s_q + rb * p.block_tokens;
          if (bar)
            tma_load_4d(dst, &q_map, bar, 64 * j, 0, grp, tok0, pol_q);
          else
            tma_prefetch_4d(&q_map, 64 * j, 0, grp, tok0);
        }
      };
      while (ok && c.valid) {
        if (c.u == 0) {
          mbar_arrive_expect_tx(&bars[VQ_FULL], 6 * q_box_bytes);
          for (int j = 0; j < 6; ++j) q_box(c.b, j, sV + j * kQBoxBytes, &bars[VQ_FULL]);
          ++vq_issued;
          for (int sl = 0; sl < kQSmemBoxes; ++sl) {
            mbar_arrive_expect_tx(&bars[QB_FULL + sl], q_box_bytes);
            q_box(c.b, 6 + sl, sQ + sl * kQBoxBytes, &bars[QB_FULL + sl]);
            ++qb_issued[sl];
          }
        } else {
          const int us = c.u - 1;  // units streamed through the slots before this one
          ok = mbar_wait(&bars[Q_EMPTY], (c.u - 1) & 1, abort_flag, kWaitNs);
          for (int j = 0; ok && j < 9; ++j) {
            const int sl = j % kQSmemBoxes;
            // the slot's previous box (j - 3) has been copied into TMEM (two copies a slot per streamed unit)
            if (j >= kQSmemBoxes) ok = mbar_wait(&bars[QB_EMPTY + sl], (2 * us + j / 3 - 1) & 1, abort_flag, kWaitNs);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars[QB_FULL + sl], q_box_bytes);
            q_box(c.b, j, sQ + sl * kQBoxBytes, &bars[QB_FULL + sl]);
            ++qb_issued[sl];
          }
        }
        // on to the next unit; its Q into L2 while this one is worked on
        c.t += static_cast<uint32_t>(c.hi - c.k);
        ++c.u;
        cursor_seek(p, P, c, c.b + 1);
        if (ok && c.valid)
          for (int j = 0; j < 9; ++j) q_box(c.b, j, nullptr, nullptr);
      }
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // no TMA write may land after this CTA exits
      if (vq_issued > 0) mbar_wait(&bars[VQ_FULL], 0, nullptr, kWaitNs);
      for (int sl = 0; sl < kQSmemBoxes; ++sl)
        if (qb_issued[sl] > 0) mbar_wait(&bars[QB_FULL + sl], (qb_issued[sl] - 1) & 1, nullptr, kWaitNs);
    } else if (lane == 0) {
      const uint64_t pol_q = policy_evict_last();
      Cursor c;
      cursor_init(p, P, c);
      bool ok = true;
      uint32_t qb_issued[kQSmemBoxes] = {};
      // box j of unit b into slot j % 3; into L2 only when bar is null
      auto q_box = [&](int b, int j, uint64_t* bar) {
        uint8_t* dst = sQ + (j % kQSmemBoxes) * kQBoxBytes;
        if (p.h_kv == 1) {
          const int row0 = b * p.rows + rb * kRowsPerBlock;
          if (bar)
            tma_load_2d(dst, &q_map, bar, 64 * j, row0, pol_q);
          else
            tma_prefetch_2d(&q_map, 64 * j, row0);
        } else {
          // [batch * s_q][h_kv][group_heads][576]: block_tokens tokens of head group grp
          const int tok0 = b * p.s_q + rb * p.block_tokens;
          if (bar)
            tma_load_4d(dst, &q_map, bar, 64 * j, 0, grp, tok0, pol_q);
          else
            tma_prefetch_4d(&q_map, 64 * j, 0, grp, tok0);
        }
      };
      if (c.valid)
        for (int j = 3; j < 9; ++j) q_box(c.b, j, nullptr);
      while (ok && c.valid) {
        if (c.u >= 1) ok = mbar_wait(&bars[Q_EMPTY], (c.u - 1) & 1, abort_flag, kWaitNs);
        for (int j = 0; ok && j < 9; ++j) {
          const int sl = j % kQSmemBoxes;
          // the slot's previous box (j - 3) has been copied into TMEM
          if (j >= kQSmemBoxes) ok = mbar_wait(&bars[QB_EMPTY + sl], (2 * c.u + j / 3 - 1) & 1, abort_flag, kWaitNs);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[QB_FULL + sl], q_box_bytes);
          q_box(c.b, j, &bars[QB_FULL + sl]);
          ++qb_issued[sl];
        }
        // on to the next unit; its Q into L2 while this one is worked on
        c.t += static_cast<uint32_t>(c.hi - c.k);
        ++c.u;
        cursor_seek(p, P, c, c.b + 1);
        if (ok && c.valid)
          for (int j = 0; j < 9; ++j) q_box(c.b, j, nullptr);
      }
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // no TMA write may land after this CTA exits
      for (int sl = 0; sl < kQSmemBoxes; ++sl)
        if (qb_issued[sl] > 0) mbar_wait(&bars[QB_FULL + sl], (qb_issued[sl] - 1) & 1, nullptr, kWaitNs);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ P V issuer
    // P V of every tile in order, from the own or the received P; issued by a
    // thread of its own so that a ready P V enters the tensor pipe without
    // waiting for a Q K^T block to finish issuing.
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_16bit_f32(128, 256, true, kHalf);
      const uint64_t vv_desc0 = sdesc_sw128(smem_u32(sV), kBoxBytes, 1024);  // V boxes as MN-major B of P V
      const uint64_t pown_desc = sdesc_sw128(smem_u32(sPOwn), 16, 1024);
      const uint64_t precv_desc = sdesc_sw128(smem_u32(sPRecv), 16, 1024);
      const uint16_t peer_mask = static_cast<uint16_t>(1u << peer);
      Cursor cv;
      cursor_init(p, P, cv);
      uint32_t pv_own = 0, pv_recv = 0;
      bool ok = true;
      uint64_t t_last = globaltimer_ns();
      while (cv.valid) {
        bool progressed = false;
        {
          const bool mine = (cv.t & 1u) == rank;
          const bool first = cursor_first(cv);
          const int vs = static_cast<int>(cv.t % kVSlots);
          bool ready = mine ? mbar_test_wait(&bars[OWN_GO], pv_own & 1)
                            : (mbar_test_wait(&bars[RECV_GO], pv_recv & 1) &&
                               mbar_test_wait(&bars[RECV_FULL], pv_recv & 1));
          ready = ready && mbar_test_wait(&bars[V_FULL + vs], (cv.t / kVSlots) & 1);
          if (ready && first && cv.u >= 1) ready = mbar_test_wait(&bars[O_FREE], (cv.u - 1) & 1);
          if (ready) {
            MLA_TRACE(3, cv.t);
            // armed for the next received P (it cannot be sent before this P V is done)
            if (!mine) mbar_arrive_expect_tx(&bars[RECV_FULL], kPBytes);
            tc_fence_after();
            const uint64_t a0 = mine ? pown_desc : precv_desc;
            const uint64_t b0 = vv_desc0 + static_cast<uint64_t>((vs * kVSlotBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              umma_f16(tmem + kTmemO, a0 + static_cast<uint64_t>((kk * 32) >> 4),
                       b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (first && kk == 0) ? 0u : 1u);
            umma_commit(&bars[V_EMPTY + vs]);
            umma_commit(&bars[PV_DONE + (cv.t & 1)]);
            if (mine) {
              umma_commit(&bars[OWN_FREE]);
              ++pv_own;
            } else {
              // the peer may refill our receive buffer (and reuse its own copy of that P)
              umma_commit_multicast(&bars[OWN_FREE], peer_mask);
              ++pv_recv;
            }
            if (cursor_last(cv)) umma_commit(&bars[O_FULL]);
            MLA_TRACE(16, cv.t);
            cursor_next(p, P, cv);
            progressed = true;
          }
        }
        if (progressed) {
          t_last = globaltimer_ns();
        } else if (*abort_flag || globaltimer_ns() - t_last > kWaitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
        // a P the peer already sent may still be landing in our receive buffer
        mbar_wait<true>(&bars[RECV_FULL], pv_recv & 1, nullptr, kWaitNs);
      }
      umma_commit(&bars[DRAIN]);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ Q K^T issuer
    if (lane == 0) {
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t vk_desc0 = sdesc_sw128(smem_u32(sV), 16, 1024);        // V boxes as K-major B of Q K^T
      // cq: Q K^T of own tiles, in two halves (K slot part, then V ring part
      // -> S); it steps over the peer's tiles at once and releases Q at every
      // unit end (after the unit's Q has arrived, so that the Q barriers'
      // phases stay aligned even for a unit without own tiles).  Each pass
      // issues at most one job: a landed Q box's copies into TMEM, else the
      // next Q K^T half.
      Cursor cq;
      cursor_init(p, P, cq);
      uint32_t a_own = 0;
      int q_phase = 0;          // 0: next is QKa of cq, 1: next is QKb of cq
      uint32_t qb_seen = 0;     // Q boxes seen landed (nine per unit, in order)
      bool ok = true;
      uint64_t t_last = globaltimer_ns();
      // cq onto the next own tile, releasing the Q of every unit it leaves;
      // returns false if it has to stop at a unit end whose Q has not arrived
      auto advance_q = [&]() -> bool {
        while (cq.valid) {
          const bool mine = (cq.t & 1u) == rank;
          if (mine && q_phase == 0) return true;  // at an own tile: its QKa is next
          if (!mine || q_phase == 2) {
            // leaving this tile; at the unit's end, Q of the unit is released
            if (cursor_last(cq)) {
              if (qb_seen < 9u * static_cast<uint32_t>(cq.u + 1)) return false;
              umma_commit(&bars[Q_EMPTY]);
            }
            cursor_next(p, P, cq);
            q_phase = 0;
            continue;
          }
          return true;  // own tile with QKb next
        }
        return true;
      };
      // the next Q box: boxes 0-5 are copied into TMEM (four copies of 128
      // rows x 16 dims, the K steps the MMAs read) and their slot released;
      // boxes 6-8 are only counted (they stay for the MMAs)
      auto q_copy = [&]() -> bool {
        const uint32_t uq = qb_seen / 9u, j = qb_seen % 9u, sl = j % kQSmemBoxes;
        // completion of this box's slot barrier: three per unit, except one
        // (boxes 6-8) for a first unit staged in the V ring
        const uint32_t idx = !kQV ? 3u * uq + j / 3u : (uq == 0 ? 0u : 1u + 3u * (uq - 1u) + j / 3u);
        if (!mbar_test_wait(&bars[QB_FULL + sl], idx & 1u)) return false;
        if (j < 6u) {
          tc_fence_after();
#pragma unroll
          for (uint32_t k = 0; k < 4; ++k)
            tmem_cp_128x256b(tmem + kTmemQ + 32u * j + 8u * k,
                             q_desc0 + static_cast<uint64_t>((sl * kQBoxBytes + k * 32u) >> 4));
          umma_commit(&bars[QB_EMPTY + sl]);
        }
        ++qb_seen;
        return true;
      };
      if (kQV && cq.valid) {
        // the first unit's boxes 0-5, staged in the V ring: into TMEM (once,
        // before the issue loop), then the ring goes to the V producer
        ok = mbar_wait(&bars[VQ_FULL], 0, abort_flag, kWaitNs);
        if (ok) {
          tc_fence_after();
          const uint64_t vq_desc0 = sdesc_sw128(smem_u32(sV), 16, 1024);
#pragma unroll 1
          for (uint32_t jj = 0; jj < 6; ++jj)
#pragma unroll
            for (uint32_t k = 0; k < 4; ++k)
              tmem_cp_128x256b(tmem + kTmemQ + 32u * jj + 8u * k,
                               vq_desc0 + static_cast<uint64_t>((jj * kQBoxBytes + k * 32u) >> 4));
          umma_commit(&bars[VQ_EMPTY]);
          qb_seen = 6;
        }
      }
      advance_q();
      while (ok && cq.valid) {
        bool progressed = q_copy();
        if (!progressed && cq.valid && advance_q() && cq.valid) {
          if (q_phase == 0) {
            const int ks = static_cast<int>(a_own % kKSlots);
            bool ready = qb_seen >= 9u * static_cast<uint32_t>(cq.u + 1);
            ready = ready && mbar_test_wait(&bars[K_FULL + ks], (a_own / kKSlots) & 1);
            if (ready && a_own >= 1) ready = mbar_test_wait(&bars[S_FREE], (a_own - 1) & 1);
            if (ready) {
              MLA_TRACE(1, cq.t);
              tc_fence_after();
              const uint64_t kslot = k_desc0 + static_cast<uint64_t>((ks * kKSlotBytes) >> 4);
              if (rank == 0)
                issue_qk_k<kHalf, 0>(tmem + kTmemS, tmem, q_desc0, kslot);
              else
                issue_qk_k<kHalf, 1>(tmem + kTmemS, tmem, q_desc0, kslot);
              umma_commit(&bars[K_EMPTY + ks]);
              MLA_TRACE(17, cq.t);
              ++a_own;
              q_phase = 1;
              progressed = true;
            }
          } else {
            const int vs = static_cast<int>(cq.t % kVSlots);
            if (mbar_test_wait(&bars[V_FULL + vs], (cq.t / kVSlots) & 1)) {
              MLA_TRACE(8, cq.t);
              tc_fence_after();
              const uint64_t vslot = vk_desc0 + static_cast<uint64_t>((vs * kVSlotBytes) >> 4);
              if (rank == 0)
                issue_qk_v<kHalf, 0>(tmem + kTmemS, tmem, q_desc0, vslot);
              else
                issue_qk_v<kHalf, 1>(tmem + kTmemS, tmem, q_desc0, vslot);
              umma_commit(&bars[S_FULL]);
              MLA_TRACE(2, cq.t);
              q_phase = 2;
              advance_q();
              progressed = true;
            }
          }
        }
        if (progressed) {
          t_last = globaltimer_ns();
        } else {
          // spin: a sleeping issuer reacts to a ready job far later than the job takes
          if (*abort_flag || globaltimer_ns() - t_last > kWaitNs) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // every MMA (of both issuers) has completed before TMEM is released
      umma_commit(&bars[DRAIN]);
      mbar_wait(&bars[DRAIN], 0, nullptr, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = tid;  // row of the block == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t taddr = tmem + lane_base;
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    int qrow, tok;
    const bool row_ok = block_row(p, grp, rb, r, qrow, tok);
    if (!row_ok) tok = 0;
    const float c_log2 = p.scale_log2;
    // the peer's buffers and barriers this warp sends to
    const uint32_t peer_p = mapa_shared(smem_u32(sPRecv + warp * kWarpPBytes), peer);
    const uint32_t peer_ref = mapa_shared(smem_u32(sRefIn + 32 * warp), peer);
    const uint32_t peer_l = mapa_shared(smem_u32(sLIn + 32 * warp), peer);
    const uint32_t peer_recv_full = mapa_shared(smem_u32(&bars[RECV_FULL]), peer);
    const uint32_t peer_r_full = mapa_shared(smem_u32(&bars[R_FULL]), peer);
    const uint32_t peer_r_free = mapa_shared(smem_u32(&bars[R_FREE]), peer);
    const uint32_t peer_l_full = mapa_shared(smem_u32(&bars[L_FULL]), peer);
    const uint32_t peer_l_free = mapa_shared(smem_u32(&bars[L_FREE]), peer);
    Cursor c;
    cursor_init(p, P, c);
    bool ok = true;
    uint32_t own_i = 0, recv_i = 0, units = 0;
    float r_cur = -INFINITY;  // reference (log2 units) after the last tile seen
    float l_own = 0.f;        // fp32 row sum of this CTA's own tiles, relative to r_cur

    while (ok && c.valid) {
      const uint32_t t = c.t;
      const bool first = cursor_first(c), last = cursor_last(c);
      const bool mine = (t & 1u) == rank;
      if (first) {
        r_cur = -INFINITY;
        l_own = 0.f;
      }
      float alpha;
      if (mine) {
        // ---- own tile: scores, reference, P
        const int jmax = p.causal ? (c.L - p.s_q + tok) : (c.L - 1);  // last visible key
        const int vis = jmax - c.k * kT;                                // keys 0..vis of this tile are visible
        uint64_t keep = (vis >= kT - 1 ? ~0ull : (vis < 0 ? 0ull : (~0ull >> (kT - 1 - vis))));
        ok = warp_wait(&bars[S_FULL], own_i & 1, abort_flag, kWaitNs);
        if (!ok) break;
        if (tid == 0) MLA_TRACE(4, t);
        tc_fence_after();
        // a page outside the pool (the K producer's flag): every key masked.
        // Read before S_FREE: the producer rewrites the entry only after that.
        // (Read from shared memory, not the block table: a global load here
        // sat on every own tile's critical path and cost 4-9 us per call.)
        if (sBad[own_i & 1]) keep = 0ull;
        float s[kT];
        float m_lo, m_hi;  // the loads' own maxima of the two halves
        {
          uint32_t (&lo32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
          uint32_t (&hi32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
          tmem_ld32_max(taddr + kTmemS, lo32, m_lo);
          tmem_ld32_max(taddr + kTmemS + 32u, hi32, m_hi);
          tmem_wait_ld();
        }
        tc_fence_before();
        mbar_arrive(&bars[S_FREE]);
        // masked keys (past the last visible one, or on a page outside the pool) ->
        // -inf; raw tile max (the scale is positive, so max commutes with it)
        // a tile with every key visible takes the loads' maxima; otherwise the
        // masked keys become -inf and the maximum is taken over the rest
        float mraw = fmaxf(m_lo, m_hi);
        if (keep != ~0ull) {
          const uint32_t klo = static_cast<uint32_t>(keep), khi = static_cast<uint32_t>(keep >> 32);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (!((klo >> j) & 1u)) s[j] = -INFINITY;
            if (!((khi >> j) & 1u)) s[j + 32] = -INFINITY;
          }
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
          for (int j = 16; j < kT; j += 8)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], s[j + i]);
          mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        }
        const float mt = mraw * c_log2;  // -inf stays -inf
        // the peer derives this tile's reference from its raw maximum, as we
        // do: it is sent at once and waits for nothing of the peer's
        if (own_i >= 1) {
          ok = warp_wait_cluster(&bars[R_FREE], (own_i - 1) & 1, abort_flag, kWaitNs);
          if (!ok) break;
        }
        // one 4-byte remote store per row (no TMA instruction: the TMA engine's
        // time goes per instruction, and it also carries the KV loads and P)
        st_async_f32(peer_ref + 4u * static_cast<uint32_t>(lane), mt, peer_r_full);
        if (tid == 0) MLA_TRACE(13, t);
        const float r_t = (mt > r_cur + kTau) ? mt : r_cur;
        const float mref = (r_t == -INFINITY) ? 0.f : r_t;
        // the own P buffer is free once our P V and the peer's P V of the
        // previous own tile are done (the latter also means our copy landed);
        // waited for before the exponentials, so that each 16-byte piece of P
        // is stored as soon as it is formed
        if (own_i >= 1) {
          ok = warp_wait_cluster(&bars[OWN_FREE], (own_i - 1) & 1, abort_flag, kWaitNs);
          if (!ok) break;
        }
        if (tid == 0) MLA_TRACE(14, t);
        uint8_t* prow = sPOwn + r * 128;
        // row sum in four fp32 partial sums (two packed pairs: keys 0, 1 mod 4
        // and 2, 3 mod 4), one packed add per pair of keys
        float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const float2 cl2 = make_float2(c_log2, c_log2), nref2 = make_float2(-mref, -mref);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t pk[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int i = 4 * cc + q4;
            // the two exponent offsets as one packed f32x2 FMA (the same IEEE operations)
            const float2 e = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), cl2, nref2);
            const float p0 = ex2(e.x);
            const float p1 = ex2(e.y);
            pk[q4] = pack2<kHalf>(p0, p1);
            ls2[i & 1] = __fadd2_rn(ls2[i & 1], make_float2(p0, p1));
          }
          *reinterpret_cast<uint4*>(prow + ((static_cast<uint32_t>(cc) ^ swz) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        const float rowsum = (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
        fence_proxy_async_smem();
        __syncwarp();
        // this warp's 32 P rows to the peer's receive buffer
        if (lane == 0) bulk_copy_to_cluster(peer_p, smem_u32(sPOwn + warp * kWarpPBytes), kWarpPBytes, peer_recv_full);
        if (tid == 0) MLA_TRACE(5, t);
        alpha = ref_alpha(r_cur, r_t);
        l_own = l_own * alpha + rowsum;
        r_cur = r_t;
      } else {
        // ---- received tile: its reference from the owner's raw maximum, by the
        // same rule the owner applies; its P V runs when its P lands
        ok = warp_wait_cluster(&bars[R_FULL], recv_i & 1, abort_flag, kWaitNs);
        if (!ok) break;
        if (tid == 0) mbar_arrive_expect_tx(&bars[R_FULL], kVecBytes);  // armed for the next message
        // read (and use, so the load has completed) before the mailbox is released
        const float m_in = __shfl_sync(0xffffffffu, sRefIn[r], lane);
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(peer_r_free);
        if (tid == 0) MLA_TRACE(10, t);
        const float r_t = (m_in > r_cur + kTau) ? m_in : r_cur;
        alpha = ref_alpha(r_cur, r_t);
        l_own *= alpha;
        r_cur = r_t;
      }
      // O (through P V of the previous tile) to the new reference, then go.
      // P V t-1 completes phase (t-1)/2 of the barrier of its parity; the phase
      // before it is P V t-3, which is complete here (own tile: its V slot was
      // refilled for this tile; received tile: the last own tile's P waited for
      // it), so the parity wait cannot pass on an older completion.  (With one
      // barrier for all tiles it could, while P V t-2 was still in flight.)
      if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = warp_wait(&bars[PV_DONE + ((t - 1) & 1)], ((t - 1) >> 1) & 1, abort_flag, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        rescale_o(taddr, alpha);
      }
      tc_fence_before();
      if (mine) {
        mbar_arrive(&bars[OWN_GO]);
        if (tid == 0) MLA_TRACE(12, t);
        ++own_i;
      } else {
        mbar_arrive(&bars[RECV_GO]);
        if (tid == 0) MLA_TRACE(11, t);
        ++recv_i;
      }
      const int b_here = c.b, u_here = c.u;
      cursor_next(p, P, c);
      if (!last) continue;
      // ---- row sum of the unit: ours + the peer's, both relative to r_cur
      if (units >= 1) {
        ok = warp_wait_cluster(&bars[L_FREE], (units - 1) & 1, abort_flag, kWaitNs);
        if (!ok) break;
      }
      sLOut[r] = l_own;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) bulk_copy_to_cluster(peer_l, smem_u32(sLOut + 32 * warp), 32 * 4, peer_l_full);
      ok = warp_wait_cluster(&bars[L_FULL], units & 1, abort_flag, kWaitNs);
      if (!ok) break;
      if (tid == 0) mbar_arrive_expect_tx(&bars[L_FULL], kVecBytes);
      const float l_peer = __shfl_sync(0xffffffffu, sLIn[r], lane);
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(peer_l_free);
      const float l_sum = l_own + l_peer;  // the same fp32 sum on both ranks
      ++units;
      // ---- epilogue of this (unit, split)
      // staging buffer: the own P buffer, free once both P V of our last own tile are done
      ok = warp_wait(&bars[O_FULL], u_here & 1, abort_flag, kWaitNs);
      if (ok && own_i >= 1) ok = warp_wait_cluster(&bars[OWN_FREE], (own_i - 1) & 1, abort_flag, kWaitNs);
      if (!ok) break;
      tc_fence_after();
      const int s_begin = p.split_offset[b_here];
      const int nsplit = p.split_offset[b_here + 1] - s_begin;
      const int slot = s_begin + ((b_here == P.b0) ? P.s0 : 0);
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const bool direct = (nsplit == 1);
      const bool bf16_out = direct && p.out_type != MLA_DTYPE_FP32;  // a 16-bit output (bf16 or fp16)
      const bool fp16_out = p.out_type == MLA_DTYPE_FP16;
      // O half -> global through that buffer: each thread stages its row's
      // 128 bytes of a column chunk, then the 128 threads store 16-byte pieces
      // so that each warp writes whole 128-byte row segments.
      const int chunk_cols = bf16_out ? 64 : 32;  // 128 bytes of output per row
      const size_t base_row = direct ? static_cast<size_t>(b_here) * p.rows : static_cast<size_t>(slot) * p.rows;
      uint8_t* stage = sPOwn;
#pragma unroll 1
      for (int ch = 0; ch < 256 / chunk_cols; ++ch) {
        uint32_t w[32];
        if (bf16_out) {
          uint32_t v[32];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tmem_ld32(taddr + kTmemO + 64 * ch + 32 * hh, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = __uint_as_float(v[2 * i]) * inv_l, b2 = __uint_as_float(v[2 * i + 1]) * inv_l;
              w[16 * hh + i] = fp16_out ? pack2<true>(a, b2) : pack2<false>(a, b2);
            }
          }
        } else {
          tmem_ld32(taddr + kTmemO + 32 * ch, w);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * inv_l);
        }
        named_bar_sync(1, 128);  // the previous chunk's stores have read the stage
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(stage + r * 128 + ((static_cast<uint32_t>(cc) ^ swz) << 4)) =
              make_uint4(w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
        named_bar_sync(1, 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int flat = tid + 128 * i;
          const int rr = flat >> 3, cc = flat & 7;
          int rg, rtok;
          if (!block_row(p, grp, rb, rr, rg, rtok)) continue;
          const uint4 val =
              *reinterpret_cast<const uint4*>(stage + rr * 128 + ((static_cast<uint32_t>(cc ^ (rr & 7))) << 4));
          const size_t e = (base_row + rg) * kDv + 256u * rank + static_cast<size_t>(ch) * chunk_cols;
          if (bf16_out)
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + e)[cc] = val;
          else
            reinterpret_cast<uint4*>((direct ? static_cast<float*>(p.out) : p.o_accum) + e)[cc] = val;
        }
      }
      named_bar_sync(1, 128);  // staging reads done before the next unit writes P
      tc_fence_before();
      mbar_arrive(&bars[O_FREE]);
      if (tid == 0) MLA_TRACE(6, t);
      if (rank == 0 && row_ok) {
        const float lse = l_sum > 0.f ? (r_cur + __log2f(l_sum)) * kLn2 : -INFINITY;
        if (direct)
          p.lse[static_cast<size_t>(b_here) * p.rows + qrow] = lse;
        else
          p.lse_accum[static_cast<size_t>(slot) * p.rows + qrow] = lse;
      }
    }
    if (!ok) {
      if (lane == 0) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      aborted = true;
    }
    r_seen = recv_i;
    l_seen = units;
  }

  // ------------------------------------------------------------ teardown
  // After a timeout the peer may still have a mailbox copy in flight to us:
  // give the armed ones (bounded) time to land before the cluster can exit.
  if (tid == 0 && (aborted || *abort_flag)) {
    mbar_wait<true>(&bars[R_FULL], r_seen & 1, nullptr, kWaitNs);
    mbar_wait<true>(&bars[L_FULL], l_seen & 1, nullptr, kWaitNs);
  }
  tc_fence_before();
  __syncthreads();
  cluster_arrive();  // the peer no longer touches this CTA's shared memory
  cluster_wait();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace dn

int dense_smem_bytes() { return dn::kSmemBytes; }
// kind 0: bf16, 1: fp16, 2: bf16 with the V-ring Q stage, 3: fp16 with it,
// 4: the bf16 stall-test instance (its first own tile's K slot is never
// loaded, so a wait runs out and the kernel reports MLA_ERR_TIMEOUT)
int dense_threads(int) { return dn::kThreads; }
const void* dense_kernel_ptr(int kind) {
  switch (kind) {
    case 1: return reinterpret_cast<const void*>(&dn::dense_decode_kernel<true, false, false>);
    case 2: return reinterpret_cast<const void*>(&dn::dense_decode_kernel<false, true, false>);
    case 3: return reinterpret_cast<const void*>(&dn::dense_decode_kernel<true, true, false>);
    case 4: return reinterpret_cast<const void*>(&dn::dense_decode_kernel<false, false, true>);
    default: return reinterpret_cast<const void*>(&dn::dense_decode_kernel<false, false, false>);
  }
}

cudaError_t launch_dense(const CUtensorMap& q_map, const CUtensorMap& kv_map, const CUtensorMap& sc_map,
                         const CUtensorMap& rope_map, const DecodeParams& p, int num_parts, int kind,
                         cudaStream_t stream) {
  const dim3 grid(2 * num_parts * p.row_blocks);
  switch (kind) {
    case 1:
      dn::dense_decode_kernel<true, false, false>
          <<<grid, dn::kThreads, dn::kSmemBytes, stream>>>(q_map, kv_map, sc_map, rope_map, p);
      break;
    case 2:
      dn::dense_decode_kernel<false, true, false>
          <<<grid, dn::kThreads, dn::kSmemBytes, stream>>>(q_map, kv_map, sc_map, rope_map, p);
      break;
    case 3:
      dn::dense_decode_kernel<true, true, false>
          <<<grid, dn::kThreads, dn::kSmemBytes, stream>>>(q_map, kv_map, sc_map, rope_map, p);
      break;
    case 4:
      dn::dense_decode_kernel<false, false, true>
          <<<grid, dn::kThreads, dn::kSmemBytes, stream>>>(q_map, kv_map, sc_map, rope_map, p);
      break;
    default:
      dn::dense_decode_kernel<false, false, false>
          <<<grid, dn::kThreads, dn::kSmemBytes, stream>>>(q_map, kv_map, sc_map, rope_map, p);
  }
  return cudaGetLastError();
}

}  // namespace mla
