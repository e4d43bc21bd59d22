// Sparse FP8 MLA split-KV decode for sm_103a (tcgen05 + TMEM + TMA), and the
// bit-exact record unpack.
//
// What it computes (FlashMLA PR #200, "[SM90] Add packed selected-KV sparse
// decode", sections Motivation and "SM90 packing kernel"; the attention
// itself as in FlashMLA PR #183, section Design): query token (b, i) attends
// to the records its top-k list selects.  Entry t of the list is a physical
// slot (page t/64, row t%64); -1, entries past topk_length and entries
// outside the pool are masked.  A 656-byte record holds 512 E4M3 codes, four
// fp32 scales (one per 128-dim group) and 64 bf16 RoPE values; the key is
// code * scale (NoPE) followed by the RoPE values, the value is the NoPE
// part.  Per split: S = Q K^T over 576 dims, online softmax, O = P V, then
// O / l and the split's LSE; the combine kernel merges the splits.  The same
// kernel serves two other slot sources: packed selections (slot t of unit
// u is packed record u * tiles * 64 + t, live when its mask bit is set) and
// a dense cache of FP8 records read through the block table, a unit then
// being a whole request (its s_q * h_q rows in row blocks of 128, each row
// masked at its token's causal limit).
//
// How (GB300 design):
//  * One 2-CTA cluster per (partition, row block of 128 heads).  The pair
//    splits the four 128-dim NoPE groups: rank c owns groups 2c and 2c+1 for
//    both the scores and the values (O[:, 256c : 256c+256) in its TMEM);
//    rank 0 also owns the 64 RoPE dims of the scores.
//  * Exact scores without a per-element dequantisation: the E4M3 codes are
//    staged as bf16 (every E4M3 value is a bf16 value) and each group gets
//    its own TMEM accumulator A_g = Q_g . codes_g (fp32).  The softmax
//    threads form the rank's partial score sum_g scale_g[j] * A_g[j] (+ the
//    RoPE product on rank 0) in fp32 and swap it with the peer through
//    distributed shared memory, so both ranks see the same full score.
//  * The value scale is folded into P: rank c multiplies P by scale_g[j] for
//    each of its two groups and runs one N=128 PV product per group against
//    the unscaled codes.
//  * Three producer warps gather the selected records into 128-byte-swizzled
//    tiles in a 2-stage ring: the tile's 64 slot indices first go to a small
//    shared table, then the records of the next tile are loaded while the
//    current one is converted (two tiles of scattered loads in flight).
//    Q comes by TMA.  One elected thread issues every tcgen05.mma.
//  * Online softmax in the log2 domain with a lazy rescale of O (only when
//    the running max grows by more than 2^8).
// Roles: warps 0-7 softmax + epilogue (two warps per TMEM lane quarter, a
// thread per row and half of the tile's scores), warps 8-10 gather producer,
// warp 11 MMA issuer and TMEM owner.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

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
namespace sp {

constexpr int kT = kTile;                         // selection slots per tile
constexpr int kQBoxBytes = kRowsPerBlock * 128;   // 128 rows x 64 bf16
constexpr int kBoxBytes = kT * 128;               // 64 keys x 64 bf16
constexpr int kMaxBoxes = 5;                      // rank 0: 4 NoPE boxes + RoPE; rank 1: 4 NoPE boxes
constexpr int kStages = 2;
constexpr int kStageBytes = kMaxBoxes * kBoxBytes;
constexpr int kScaleStageBytes = 2 * kT * 4;      // the rank's two group scales of 64 keys
constexpr int kXBytes = kRowsPerBlock * kT * 4;   // the peer's partial scores
constexpr int kPGroupBytes = kRowsPerBlock * kT * 2;
constexpr uint32_t kHalfX = kXBytes / 2;          // scores 32-63 of the mailbox rows
static_assert(kHalfX == kPGroupBytes && kXBytes == 2 * kPGroupBytes, "the partial is staged in the P buffer");

constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMaxBoxes * kQBoxBytes;
constexpr int kOffX = kOffKV + kStages * kStageBytes;
constexpr int kOffP = kOffX + kXBytes;
constexpr int kOffScale = kOffP + 2 * kPGroupBytes;
constexpr int kOffIdx = kOffScale + kStages * kScaleStageBytes;  // [2][64] record index or -1 (producer only)
constexpr int kVisSlots = 4;
constexpr int kOffVis = kOffIdx + 2 * kT * 4;                     // [4] 64-bit valid-slot masks
constexpr int kOffBar = kOffVis + kVisSlots * 8;
constexpr int kNumBars = 21;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffKV % 1024 == 0 && kOffX % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms need 1 KB alignment");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // score accumulators: A_{2c}, A_{2c+1}, RoPE (rank 0), 64 columns each
// [448, 452): where the two softmax threads of a row swap their halves' row
// maximum (448 + h) and row sum (450 + h): the two warps of a lane quarter
// reach the same TMEM lanes
constexpr uint32_t kTmemX = 448;

constexpr int kSoftmaxWarps = 8;
// named barriers: 1-4 pair the two softmax warps of a TMEM lane quarter
constexpr uint32_t kBarProdSync = 5, kBarProdOr = 6;
constexpr int kProducerWarps = 3;
constexpr int kMmaWarp = kSoftmaxWarps + kProducerWarps;
constexpr int kThreads = 32 * (kMmaWarp + 1);

enum : int {
  Q_FULL = 0,
  Q_EMPTY = 1,
  KV_FULL = 2,   // +stage
  KV_EMPTY = 4,  // +stage
  S_FULL = 6,
  S_FREE = 7,
  P_FULL = 8,
  P_FREE = 9,
  O_FULL = 10,
  O_FREE = 11,
  X_FULL = 12,   // +warp
  X_FREE = 16,   // +warp
  DRAIN = 20,
};

constexpr float kTau = 8.0f;  // lazy-rescale threshold (log2 units)
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

struct Part {
  int b0, t0, b1, t1, s0;
};

__device__ __forceinline__ Part load_part(const int32_t* sched, int idx) {
  const int32_t* e = sched + idx * MLA_SCHED_INTS;
  return Part{e[0], e[1], e[2], e[3], e[4]};
}

// Length of unit b as the scheduler saw it (tiles are counted from this)...
__device__ __forceinline__ int sched_len(const DecodeParams& p, int b) {
  return max(p.lengths != nullptr ? p.lengths[b] : p.default_length, 0);
}

// ...and the candidate slots that may be valid: clamped to the list size.
__device__ __forceinline__ int unit_len(const DecodeParams& p, int b) { return min(sched_len(p, b), p.topk); }

// Tile range [lo, hi) of unit b inside partition P.
__device__ __forceinline__ void unit_tiles(const Part& P, int b, int nt, int& lo, int& hi) {
  lo = (b == P.b0) ? P.t0 : 0;
  hi = (b == P.b1) ? P.t1 : nt;
}

__device__ __forceinline__ bool unit_in_part(const Part& P, int b, int n_units) {
  return b < n_units && (b < P.b1 || (b == P.b1 && P.t1 > 0));
}

// Walk over the (unit, tile) sequence of one partition.
struct Cursor {
  int b, k, lo, hi;  // unit, tile, tile range of the unit in this partition
  int u;             // ordinal of the unit within the partition
  uint32_t t;        // ordinal of the tile within the partition
  bool valid;
};

__device__ __forceinline__ void cursor_seek(const DecodeParams& p, const Part& P, Cursor& c, int from_b) {
  for (int b = from_b; unit_in_part(P, b, p.n_units); ++b) {
    int lo, hi;
    unit_tiles(P, b, num_tiles(sched_len(p, b)), lo, hi);
    if (hi > lo) {
      c.b = b;
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

__device__ __forceinline__ void cursor_next(const DecodeParams& p, const Part& P, Cursor& c) {
  ++c.t;
  if (++c.k == c.hi) {
    ++c.u;
    cursor_seek(p, P, c, c.b + 1);
  }
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

// 1 / x within 5.1% for a normal positive x below 2^126: one integer
// subtract from the bit pattern negates the exponent and takes the
// mantissa's reciprocal to first order.  Used only to rescale the rounding
// residual (relative size <= 2^-9) of a product p * x, so the result is
// within 2^-13 of p of the exact quotient.  The producer stores scales
// below the smallest normal fp32 as 0; for x = 0 the residual it scales is
// 0 (so is the product), and the term is 0.
__device__ __forceinline__ float approx_inv(float x) { return __int_as_float(0x7EF311C7 - __float_as_int(x)); }

// Wait budget of the stall-test instance of the decode kernel (kStall):
// short, so that its test ends quickly; the other instance keeps the 2 s
// budget of every wait.
constexpr uint64_t kDecodeStallWaitNs = 200000;  // 200 us

// Two E4M3 codes (bytes 0 and 1 of `pair`) -> two bf16 of the same values
// (low half = byte 0): E4M3 -> f16 -> f32 -> bf16 is exact at every step
// (3 mantissa bits, exponents well inside both formats).  (Integer moves
// plus a bf16 multiply by 2^120 measured slower than these conversions.)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t pair) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 8 E4M3 codes -> 8 bf16 of the same values.
__device__ __forceinline__ uint4 codes_to_bf16(uint2 codes) {
  return make_uint4(e4m3x2_to_bf16x2(codes.x), e4m3x2_to_bf16x2(codes.x >> 16), e4m3x2_to_bf16x2(codes.y),
                    e4m3x2_to_bf16x2(codes.y >> 16));
}

// Selection entry t of unit b as stored (no check yet); -1 past the list.
// Packed selection: the record of slot t sits at ordinal b * tiles * 64 + t
// of the packed records when its bit in the tile's valid mask is set.
// Dense FP8 cache: every token is a key; slot t of unit b is record t % 64
// of page block_table[b / unit_request_div][t / 64] (a unit is a whole
// request); a page outside the pool comes back as -2 (reported, masked).
__device__ __forceinline__ int load_slot(const DecodeParams& p, int b, int t, int L) {
  if (t >= L) return -1;
  if (p.block_table != nullptr) {
    const int pg = t / kT;
    const int page =
        pg < p.max_pages ? __ldg(p.block_table + static_cast<size_t>(b / p.unit_request_div) * p.max_pages + pg) : -1;
    return (page < 0 || page >= p.num_pages) ? -2 : page * kT + (t - pg * kT);
  }
  if (p.packed_mask != nullptr) {
    const int tiles = (p.topk + kT - 1) / kT;
    const unsigned long long m =
        __ldg(reinterpret_cast<const unsigned long long*>(p.packed_mask) + static_cast<size_t>(b) * tiles + t / kT);
    return ((m >> (t % kT)) & 1ull) ? (b * tiles * kT + t) : -1;
  }
  return __ldg(p.indices + static_cast<size_t>(b) * p.topk + t);
}

// A stored entry -> record index, or -1 when masked; an entry outside the
// pool (other than -1) is reported.
__device__ __forceinline__ int resolve_slot(const DecodeParams& p, int idx) {
  if (idx == -1) return -1;
  if (idx < 0 || idx >= p.num_pages * kT) {
    report(p.status, MLA_ERR_BAD_INDEX);
    return -1;
  }
  return idx;
}

// Q/KV box lb of rank `rank` -> first latent dim it holds.
__device__ __forceinline__ int box_dim(uint32_t rank, int lb) {
  return rank == 0 ? (lb < 4 ? 64 * lb : 512) : 256 + 64 * lb;
}

// S accumulators of one tile: kAcc = 3 (rank 0: two groups + RoPE) or 2.
// Group accumulator a reads boxes 2a, 2a+1 (8 K-steps of 16 dims); the RoPE
// accumulator reads box 4 (4 K-steps).  Fully unrolled: the descriptor
// offsets are compile-time constants.
template <int kAcc>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint64_t q_desc0, uint64_t kv_desc_stage, uint32_t idesc) {
#pragma unroll
  for (int a = 0; a < kAcc; ++a) {
    const int nks = a < 2 ? 8 : 4;
#pragma unroll
    for (int ks = 0; ks < nks; ++ks) {
      const int lb = a < 2 ? 2 * a + (ks >> 2) : 4;
      const uint32_t off_q = lb * kQBoxBytes + (ks & 3) * 32;
      const uint32_t off_k = lb * kBoxBytes + (ks & 3) * 32;
      umma_f16(tmem + kTmemS + 64u * a, q_desc0 + (off_q >> 4), kv_desc_stage + (off_k >> 4), idesc,
               ks > 0 ? 1u : 0u);
    }
  }
}

// O[:, 128g : 128g+128) += P_g (128 x 64 keys) x codes of boxes 2g, 2g+1.
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint64_t p_desc0, uint64_t v_desc_stage, uint32_t idesc,
                                         bool first) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk) {
      const uint32_t off_p = g * kPGroupBytes + kk * 32;
      const uint32_t off_v = 2 * g * kBoxBytes + kk * 2048;
      umma_f16(tmem + kTmemO + 128u * g, p_desc0 + (off_p >> 4), v_desc_stage + (off_v >> 4), idesc,
               (first && kk == 0) ? 0u : 1u);
    }
  }
}

template <bool kStall>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    sparse_decode_kernel(const __grid_constant__ CUtensorMap q_map, const DecodeParams p) {
  constexpr uint64_t kWaitNs = kStall ? kDecodeStallWaitNs : MLA_WAIT_LIMIT_NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKV = smem + kOffKV;
  uint8_t* sX = smem + kOffX;
  uint8_t* sP = smem + kOffP;
  float* sScale = reinterpret_cast<float*>(smem + kOffScale);  // [stage][2 groups][64 keys]
  int* sIdx = reinterpret_cast<int*>(smem + kOffIdx);           // [tile & 1][64 slots]
  uint32_t* sVis = reinterpret_cast<uint32_t*>(smem + kOffVis);  // [tile & 3][2 halves]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster_id = blockIdx.x >> 1;
  const int part_idx = cluster_id / p.row_blocks;
  const int rb = cluster_id - part_idx * p.row_blocks;
  const int n_boxes = rank == 0 ? 5 : 4;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bars[Q_FULL], 1);
    mbar_init(&bars[Q_EMPTY], 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars[KV_FULL + i], 32 * kProducerWarps);
      mbar_init(&bars[KV_EMPTY + i], 1);
    }
    mbar_init(&bars[S_FULL], 1);
    mbar_init(&bars[S_FREE], 32 * kSoftmaxWarps);
    mbar_init(&bars[P_FULL], 32 * kSoftmaxWarps);
    mbar_init(&bars[P_FREE], 1);
    mbar_init(&bars[O_FULL], 1);
    mbar_init(&bars[O_FREE], 32 * kSoftmaxWarps);
    for (int w = 0; w < 4; ++w) {
      mbar_init(&bars[X_FULL + w], 1);
      mbar_init(&bars[X_FREE + w], 1);
    }
    mbar_init(&bars[DRAIN], 1);
    fence_mbar_init_cluster();
    // armed for the peer's first partial scores (32 rows x 64 fp32 per warp)
    for (int w = 0; w < 4; ++w) mbar_arrive_expect_tx(&bars[X_FULL + w], 32 * kT * 4);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) prefetch_tmap(&q_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // the peer's barriers are initialised before any remote arrive
  cluster_wait();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  const Part P = load_part(p.sched, part_idx);

  if (warp >= kSoftmaxWarps && warp < kMmaWarp) {
    // ------------------------------------------------------------ producer
    const int ptid = tid - 32 * kSoftmaxWarps;  // 0 .. 32 * kProducerWarps - 1
    const uint64_t pol_q = policy_evict_last();
    // Per key: 16 NoPE chunks of 16 bytes (16 E4M3 codes each) of the rank's
    // two groups, loaded into registers a tile ahead and converted; the two
    // group scales (threads 0-63, one key each), also a tile ahead; on rank
    // 0 the 8 RoPE chunks (8 bf16 each), copied into the stage by cp.async
    // once it is free (they need no conversion).
    const int nope0 = 256 * static_cast<int>(rank);
    constexpr int kPerMax = (kT * 16 + 32 * kProducerWarps - 1) / (32 * kProducerWarps);  // 11
    constexpr int kRopePer = (kT * 8 + 32 * kProducerWarps - 1) / (32 * kProducerWarps);   // 6
    uint32_t t = 0;
    int u = 0;
    bool ok = true;
    uint32_t q_issued = 0;
    for (int b = P.b0; ok && unit_in_part(P, b, p.n_units); ++b) {
      const int L = unit_len(p, b);
      const int nt = num_tiles(sched_len(p, b));
      int lo, hi;
      unit_tiles(P, b, nt, lo, hi);
      if (hi <= lo) continue;
      if (ptid == 0) {
        if (u >= 1) ok = mbar_wait(&bars[Q_EMPTY], (u - 1) & 1, abort_flag, kWaitNs);
        if (ok) {
          mbar_arrive_expect_tx(&bars[Q_FULL], n_boxes * kQBoxBytes);
          const int row0 = b * p.rows + rb * kRowsPerBlock;
          for (int lb = 0; lb < n_boxes; ++lb)
            tma_load_2d(sQ + lb * kQBoxBytes, &q_map, &bars[Q_FULL], box_dim(rank, lb), row0, pol_q);
          ++q_issued;
        }
      }
      if (named_bar_or(kBarProdOr, 32 * kProducerWarps, !ok)) {
        ok = false;
        break;
      }
      // Software pipeline over the unit's tiles: the record loads of tile k+1
      // are issued before tile k is converted, so two tiles' scattered record
      // loads are in flight while one is being written.
      uint4 raw[kPerMax];
      float sc[2];
      // phase 1 for tile tt: its 64 slot entries (loaded earlier, see below)
      // -> record index or -1, and the tile's valid-slot mask for the softmax
      auto publish_indices = [&](int entry, uint32_t tt) {
        named_bar_sync(kBarProdSync, 32 * kProducerWarps);  // the slot's previous tile is no longer read
        if (ptid < kT) {
          const int idx = resolve_slot(p, entry);
          sIdx[(tt & 1) * kT + ptid] = idx;
          const uint32_t half = __ballot_sync(0xffffffffu, idx >= 0);
          if (lane == 0) sVis[(tt & (kVisSlots - 1)) * 2 + (ptid >> 5)] = half;
        }
        named_bar_sync(kBarProdSync, 32 * kProducerWarps);
      };
      // phase 2 for tile tt: the NoPE chunks' loads (a masked slot reads
      // record 0) and, on threads 0-63, the key's two group scales
      auto issue_loads = [&](uint32_t tt, uint4 (&rr)[kPerMax], float (&ss)[2]) {
        const int* idx_t = sIdx + (tt & 1) * kT;
#pragma unroll
        for (int i = 0; i < kPerMax; ++i) {
          const int qq = min(ptid + 32 * kProducerWarps * i, kT * 16 - 1);
          const int idx = idx_t[qq >> 4];
          const uint8_t* rec = p.kv8 + static_cast<size_t>(max(idx, 0)) * MLA_RECORD_BYTES;
          rr[i] = __ldg(reinterpret_cast<const uint4*>(rec + nope0 + 16 * (qq & 15)));
        }
        if (ptid < kT) {
          const uint8_t* rec = p.kv8 + static_cast<size_t>(max(idx_t[ptid], 0)) * MLA_RECORD_BYTES;
          const float2 f = __ldg(reinterpret_cast<const float2*>(rec + 512 + 8 * static_cast<int>(rank)));
          ss[0] = f.x;
          ss[1] = f.y;
        }
      };
      // slot entries are loaded two tiles ahead of their records, so that no
      // tile waits for an index load
      int entry = ptid < kT ? load_slot(p, b, lo * kT + ptid, L) : -1;
      int entry_n = (ptid < kT && lo + 1 < hi) ? load_slot(p, b, (lo + 1) * kT + ptid, L) : -1;
      publish_indices(entry, t);
      issue_loads(t, raw, sc);
      for (int k = lo; ok && k < hi; ++k, ++t) {
        const int st = t & 1;
        uint4 raw_n[kPerMax];
        float sc_n[2];
        if (k + 1 < hi) {
          publish_indices(entry_n, t + 1);
          entry_n = (ptid < kT && k + 2 < hi) ? load_slot(p, b, (k + 2) * kT + ptid, L) : -1;
          issue_loads(t + 1, raw_n, sc_n);
        }
        bool failed = false;
        if (t >= 2) failed = !mbar_wait(&bars[KV_EMPTY + st], ((t - 2) >> 1) & 1, abort_flag, kWaitNs);
        // one decision for the whole producer group: its named barriers need every thread
        if (named_bar_or(kBarProdOr, 32 * kProducerWarps, failed)) {
          ok = false;
          break;
        }
        if (ptid == 0) MLA_TRACE(0, t);
        const int* idx_t = sIdx + (t & 1) * kT;
        uint8_t* stage = sKV + st * kStageBytes;
        float* scale_st = sScale + st * (2 * kT);
        if (rank == 0) {
          // RoPE: straight into the stage's fifth box (zero for a masked slot)
#pragma unroll
          for (int j = 0; j < kRopePer; ++j) {
            const int qq = ptid + 32 * kProducerWarps * j;
            if (qq < kT * 8) {
              const int key = qq >> 3, c = qq & 7;
              const int idx = idx_t[key];
              uint8_t* dst = stage + 4 * kBoxBytes + key * 128 + ((static_cast<uint32_t>(c) ^ (key & 7)) << 4);
              if (idx >= 0)
                cp_async16(smem_u32(dst), p.kv8 + static_cast<size_t>(idx) * MLA_RECORD_BYTES + 528 + 16 * c);
              else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        if (ptid < kT) {
          // a masked slot, and a scale below the smallest normal fp32 (its
          // products with the codes are below 2^-117 and are lost in fp32
          // rounding of any score or value that matters), count as 0; the
          // weights' rounding correction then needs no guard for them
          const bool live = idx_t[ptid] >= 0;
          scale_st[ptid] = live && fabsf(sc[0]) >= 1.17549435e-38f ? sc[0] : 0.f;
          scale_st[kT + ptid] = live && fabsf(sc[1]) >= 1.17549435e-38f ? sc[1] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kPerMax; ++i) {
          const int qq = ptid + 32 * kProducerWarps * i;
          if (qq < kT * 16) {
            const int key = qq >> 4, c = qq & 15;
            const uint4 w = idx_t[key] >= 0 ? raw[i] : make_uint4(0u, 0u, 0u, 0u);
            // 16 codes -> 16 bf16: two 16-byte pieces of box c/4, columns 2(c%4), 2(c%4)+1
            uint8_t* box = stage + (c >> 2) * kBoxBytes + key * 128;
            const uint32_t swz = static_cast<uint32_t>(key & 7);
            const uint32_t cc = 2u * static_cast<uint32_t>(c & 3);
            *reinterpret_cast<uint4*>(box + ((cc ^ swz) << 4)) = codes_to_bf16(make_uint2(w.x, w.y));
            *reinterpret_cast<uint4*>(box + (((cc + 1u) ^ swz) << 4)) = codes_to_bf16(make_uint2(w.z, w.w));
          }
        }
        if (rank == 0) cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&bars[KV_FULL + st]);
        if (ptid == 0) MLA_TRACE(1, t);
#pragma unroll
        for (int i = 0; i < kPerMax; ++i) raw[i] = raw_n[i];
        sc[0] = sc_n[0];
        sc[1] = sc_n[1];
      }
      ++u;
    }
    if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
    // no TMA write may land after this CTA exits
    if (ptid == 0 && q_issued > 0) mbar_wait(&bars[Q_FULL], (q_issued - 1) & 1, nullptr, kWaitNs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kT, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, true);
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kv_desc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(sKV), kBoxBytes, 1024);
      const uint64_t p_desc0 = sdesc_sw128(smem_u32(sP), 16, 1024);
      // Two cursors over the partition's (unit, tile) sequence: QK of tile t
      // needs the single S buffer back from the softmax of tile t-1; PV of
      // tile t needs P of tile t.  Whichever is ready is issued, PV first.
      Cursor cq, cv;
      cursor_init(p, P, cq);
      cursor_init(p, P, cv);
      bool ok = true;
      uint64_t t_last = globaltimer_ns();
      while (cv.valid) {
        bool progressed = false;
        if (cv.t < cq.t) {
          bool ready = mbar_test_wait(&bars[P_FULL], cv.t & 1);
          const bool first = cv.k == cv.lo, last = cv.k == cv.hi - 1;
          if (ready && first && cv.u >= 1) ready = mbar_test_wait(&bars[O_FREE], (cv.u - 1) & 1);
          if (ready) {
            tc_fence_after();
            const int st = cv.t & 1;
            MLA_TRACE(2, cv.t);
            issue_pv(tmem, p_desc0, v_desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4), idesc_pv, first);
            umma_commit(&bars[P_FREE]);
            umma_commit(&bars[KV_EMPTY + st]);
            if (last) umma_commit(&bars[O_FULL]);
            cursor_next(p, P, cv);
            progressed = true;
          }
        }
        if (cq.valid) {
          const int st = cq.t & 1;
          bool ready = true;
          if (cq.k == cq.lo) ready = mbar_test_wait(&bars[Q_FULL], cq.u & 1);
          ready = ready && mbar_test_wait(&bars[KV_FULL + st], (cq.t >> 1) & 1);
          if (ready && cq.t >= 1) ready = mbar_test_wait(&bars[S_FREE], (cq.t - 1) & 1);
          if (ready) {
            tc_fence_after();
            MLA_TRACE(3, cq.t);
            const uint64_t kvs = kv_desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
            // the stall-test instance never computes its first tile's scores
            // (the softmax's wait for them runs out)
            if (!(kStall && cq.t == 0)) {
              if (rank == 0)
                issue_qk<3>(tmem, q_desc0, kvs, idesc_qk);
              else
                issue_qk<2>(tmem, q_desc0, kvs, idesc_qk);
              umma_commit(&bars[S_FULL]);
            }
            if (cq.k == cq.hi - 1) umma_commit(&bars[Q_EMPTY]);
            cursor_next(p, P, cq);
            progressed = true;
          }
        }
        if (progressed) {
          t_last = globaltimer_ns();
        } else {
          if (*abort_flag || globaltimer_ns() - t_last > kWaitNs) {
            ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // every MMA has completed before TMEM is released
      umma_commit(&bars[DRAIN]);
      mbar_wait(&bars[DRAIN], 0, nullptr, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Eight warps: warp w takes the rows of TMEM lane quarter q = w % 4
    // (rows 32q .. 32q+31, one per thread) and scores 32h .. 32h+31 (h = w / 4)
    // of every tile; for O (rescale, epilogue) it takes columns 128h .. 128h+127
    // of the rank's half.  The two warps of a quarter meet at a named barrier
    // (bar.red.or, so that they leave the loop together) to send the
    // quarter's partial scores, to combine the row maxima and the row sums.
    const int q = warp & 3, h = warp >> 2;
    const int r = 32 * q + lane;  // row of the block == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t pair_bar = 1 + q, pair_n = 64;
    const bool sender = h == 0 && lane == 0;  // sends, re-arms and frees the quarter's mailbox
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    // A row's 64 partial scores travel in the row's P footprint (two groups x
    // 128 bytes, 16-byte chunks c at position c ^ (r & 7)): scores
    // 32h + 4k .. 32h + 4k + 3 (k = 0..7) sit in group k >> 2, chunk
    // 4h + (k & 3), exactly where this thread later writes its P.  The peer's
    // mailbox sX has the same layout, so a quarter's partials are two 4 KB
    // pieces (group 0 rows, group 1 rows) on both sides.
    auto chunk_off = [&](int k) -> uint32_t {
      return static_cast<uint32_t>(k >> 2) * kPGroupBytes + r * 128u +
             (((4u * h + static_cast<uint32_t>(k & 3)) ^ swz) << 4);
    };
    const uint32_t x_local = smem_u32(sX), x_stage = smem_u32(sP);
    const uint32_t q_off = static_cast<uint32_t>(32 * q) * 128u;
    const uint32_t x_remote_q = mapa_shared(smem_u32(sX) + q_off, peer);
    const uint32_t xfull_remote = mapa_shared(smem_u32(&bars[X_FULL + q]), peer);
    const uint32_t xfree_remote = mapa_shared(smem_u32(&bars[X_FREE + q]), peer);
    const int n_acc = rank == 0 ? 3 : 2;
    uint32_t t = 0;
    int u = 0;
    bool ok = true;
    for (int b = P.b0; ok && unit_in_part(P, b, p.n_units); ++b) {
      const int L = unit_len(p, b);
      const int nt = num_tiles(sched_len(p, b));
      int lo, hi;
      unit_tiles(P, b, nt, lo, hi);
      if (hi <= lo) continue;
      const int row = rb * kRowsPerBlock + r;
      const bool row_ok = row < p.rows;
      // last key this row sees: with the causal mask, query token i of a
      // request with L keys ends at key L - s_q + i (rows are token-major)
      const int row_last = p.causal ? L - p.s_q + row / p.h_q : L - 1;
      // running max (log2 units), the same in both threads of a row, and
      // this thread's part of the fp32 row sum
      float m_used = -INFINITY, l_part = 0.f;
      // per group of this rank, the P V weights' rounding: sum over this
      // thread's keys of (bf16(p * scale) - p * scale) / scale, so that each
      // group's O columns are divided by the weights the MMA actually used
      float corr0 = 0.f, corr1 = 0.f;
      for (int k = lo; k < hi; ++k, ++t) {
        const int st = t & 1;
        // ---- phase 1: this thread's 32 partial scores, staged for the peer
        if (ok) ok = warp_wait(&bars[KV_FULL + st], (t >> 1) & 1, abort_flag, kWaitNs);
        // which of this thread's 32 slots are valid and visible to the row
        const int lim = row_last - k * kT - 32 * h;
        const uint32_t vis = (ok ? sVis[(t & (kVisSlots - 1)) * 2 + h] : 0u) &
                             (lim >= 31 ? 0xffffffffu : (lim < 0 ? 0u : (0xffffffffu >> (31 - lim))));
        if (ok) ok = warp_wait(&bars[S_FULL], t & 1, abort_flag, kWaitNs);
        // scores 2k, 2k + 1 of this thread's 32 as a pair: the elementwise
        // steps run as packed f32x2 instructions (the same IEEE operations)
        float2 s2[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) s2[k] = make_float2(0.f, 0.f);
        if (ok) {
          if (tid == 0) MLA_TRACE(4, t);
          tc_fence_after();
          const uint32_t sc_base = smem_u32(sScale + st * (2 * kT)) + 128u * h;
#pragma unroll 1
          for (int a = 0; a < n_acc; ++a) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kTmemS + 64u * a + 32u * h, v);
            tmem_wait_ld();
            if (a < 2) {
#pragma unroll
              for (int j4 = 0; j4 < 8; ++j4) {
                const float4 sc = ld_shared_v4(sc_base + (a * kT + 4 * j4) * 4);
                s2[2 * j4] = __ffma2_rn(make_float2(sc.x, sc.y),
                                        make_float2(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1])),
                                        s2[2 * j4]);
                s2[2 * j4 + 1] = __ffma2_rn(make_float2(sc.z, sc.w),
                                            make_float2(__uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3])),
                                            s2[2 * j4 + 1]);
              }
            } else {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                s2[k] = __fadd2_rn(s2[k], make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])));
            }
          }
          tc_fence_before();
          mbar_arrive(&bars[S_FREE]);
          // the P buffer is free once P V of the previous tile is done
          if (t >= 1) ok = warp_wait(&bars[P_FREE], (t - 1) & 1, abort_flag, kWaitNs);
        }
        if (ok) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(x_stage + chunk_off(c), s2[2 * c].x, s2[2 * c].y, s2[2 * c + 1].x, s2[2 * c + 1].y);
          fence_proxy_async_smem();
        }
        if (named_bar_or(pair_bar, pair_n, !ok)) {
          ok = false;
          break;
        }
        // ---- phase 2: send the quarter's partials, receive the peer's, row max
        if (sender) {
          // the peer has read our previous partials (so that copy is complete)
          bool sent = t == 0 || mbar_wait<true>(&bars[X_FREE + q], (t - 1) & 1, abort_flag, kWaitNs);
          if (sent) {
            bulk_copy_to_cluster(x_remote_q, x_stage + q_off, 32 * 128, xfull_remote);
            bulk_copy_to_cluster(x_remote_q + kPGroupBytes, x_stage + kPGroupBytes + q_off, 32 * 128, xfull_remote);
          } else {
            set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
          }
        }
        if (tid == 0) MLA_TRACE(5, t);
        ok = warp_wait_cluster(&bars[X_FULL + q], t & 1, abort_flag, kWaitNs);
        float mt = -INFINITY;
        if (ok) {
          if (tid == 0) MLA_TRACE(6, t);
          // full score = own partial + peer's partial (one fp32 add: the same bits on both ranks)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 o = ld_shared_v4(x_local + chunk_off(c));
            s2[2 * c] = __fadd2_rn(s2[2 * c], make_float2(o.x, o.y));
            s2[2 * c + 1] = __fadd2_rn(s2[2 * c + 1], make_float2(o.z, o.w));
          }
          // mask, scale into the log2 domain, maximum of this thread's 32
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 x = __fmul2_rn(s2[k], sl2);
            s2[k].x = ((vis >> (2 * k)) & 1u) ? x.x : -INFINITY;
            s2[k].y = ((vis >> (2 * k + 1)) & 1u) ? x.y : -INFINITY;
            m4[(2 * k) & 3] = fmaxf(m4[(2 * k) & 3], s2[k].x);
            m4[(2 * k + 1) & 3] = fmaxf(m4[(2 * k + 1) & 3], s2[k].y);
          }
          mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          tmem_st1(tmem + lane_base + kTmemX + h, __float_as_uint(mt));
          tmem_wait_st();
        }
        tc_fence_before();
        if (named_bar_or(pair_bar, pair_n, !ok)) {
          ok = false;
          break;
        }
        // both warps have read the mailbox: arm it for the next tile, free it for the peer
        if (sender) {
          mbar_arrive_expect_tx(&bars[X_FULL + q], 2 * 32 * 128);
          mbar_arrive_remote(xfree_remote);
        }
        // ---- phase 3: the row's tile max, reference, exponentials, P
        tc_fence_after();
        mt = fmaxf(mt, __uint_as_float(tmem_ld1(tmem + lane_base + kTmemX + 1 - h)));
        tmem_wait_ld();
        bool rescale = false;
        float alpha = 1.f;
        if (mt > m_used + kTau) {
          alpha = ex2(m_used - mt);  // 0 when m_used == -inf
          rescale = k > lo;
          l_part *= alpha;
          corr0 *= alpha;
          corr1 *= alpha;
          m_used = mt;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        // ls2[0] = (sum of keys 0 mod 4, 1 mod 4), ls2[1] = (2 mod 4, 3 mod 4)
        float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const float2 nref2 = make_float2(-mref, -mref);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 d = __fadd2_rn(s2[k], nref2);
          s2[k] = make_float2(ex2(d.x), ex2(d.y));
          ls2[k & 1] = __fadd2_rn(ls2[k & 1], s2[k]);
        }
        l_part += (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
        // our partials have left the P buffer (the peer has read them) before P is written there
        ok = warp_wait_cluster(&bars[X_FREE + q], t & 1, abort_flag, kWaitNs);
        if (!ok) {
          set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
          continue;  // the next pair barrier takes both warps out
        }
        if (__any_sync(0xffffffffu, rescale)) {
          tc_fence_after();
#pragma unroll 1
          for (uint32_t c0 = 0; c0 < 128; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_base + kTmemO + 128u * h + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st16(tmem + lane_base + kTmemO + 128u * h + c0, v);
          }
          tmem_wait_st();
        }
        // P_g[j] = p[j] * scale_g[j] for the rank's two groups, bf16, swizzled rows
        const uint32_t sc_base = smem_u32(sScale + st * (2 * kT)) + 128u * h;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float2 corr2 = make_float2(0.f, 0.f);  // (even keys, odd keys)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 sa = ld_shared_v4(sc_base + (g * kT + 8 * c) * 4);
            const float4 sb = ld_shared_v4(sc_base + (g * kT + 8 * c + 4) * 4);
            const float2 w2[4] = {__fmul2_rn(s2[4 * c], make_float2(sa.x, sa.y)),
                                  __fmul2_rn(s2[4 * c + 1], make_float2(sa.z, sa.w)),
                                  __fmul2_rn(s2[4 * c + 2], make_float2(sb.x, sb.y)),
                                  __fmul2_rn(s2[4 * c + 3], make_float2(sb.z, sb.w))};
            const float2 inv2[4] = {make_float2(approx_inv(sa.x), approx_inv(sa.y)),
                                    make_float2(approx_inv(sa.z), approx_inv(sa.w)),
                                    make_float2(approx_inv(sb.x), approx_inv(sb.y)),
                                    make_float2(approx_inv(sb.z), approx_inv(sb.w))};
            uint32_t pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __nv_bfloat162 hv = __floats2bfloat162_rn(w2[i].x, w2[i].y);
              pk[i] = *reinterpret_cast<const uint32_t*>(&hv);
              // the rounding of each weight (an exact difference), in units of
              // p: divided by the key's scale through an approximate inverse
              const float2 rnd = __fadd2_rn(make_float2(__uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xffff0000u)),
                                            make_float2(-w2[i].x, -w2[i].y));
              corr2 = __ffma2_rn(rnd, inv2[i], corr2);
            }
            *reinterpret_cast<uint4*>(sP + g * kPGroupBytes + r * 128 + (((4u * h + c) ^ swz) << 4)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          if (g == 0)
            corr0 += corr2.x + corr2.y;
          else
            corr1 += corr2.x + corr2.y;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[P_FULL]);
        if (tid == 0) MLA_TRACE(7, t);
      }
      if (named_bar_or(pair_bar, pair_n, !ok)) {
        ok = false;
        break;
      }
      // ---- epilogue of this (unit, split): the row sum of both threads
      tmem_st1(tmem + lane_base + kTmemX + 2 + h, __float_as_uint(l_part));
      // the other thread of the row needs this thread's correction of its group (1 - h)
      tmem_st1(tmem + lane_base + kTmemX + 4 + h, __float_as_uint(h == 0 ? corr1 : corr0));
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(pair_bar, pair_n);
      tc_fence_after();
      const uint32_t l_other = tmem_ld1(tmem + lane_base + kTmemX + 3 - h);
      tmem_wait_ld();
      const uint32_t c_other = tmem_ld1(tmem + lane_base + kTmemX + 5 - h);
      tmem_wait_ld();
      const float l_sum = l_part + __uint_as_float(l_other);
      // this thread's O columns are group h's: divided by the sum of the
      // weights that multiplied them (the LSE keeps the exact sum)
      const float l_norm = l_sum + ((h == 0 ? corr0 : corr1) + __uint_as_float(c_other));
      ok = warp_wait(&bars[O_FULL], u & 1, abort_flag, kWaitNs);
      if (named_bar_or(pair_bar, pair_n, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int s_begin = p.split_offset[b];
      const int nsplit = p.split_offset[b + 1] - s_begin;
      const int slot = s_begin + ((b == P.b0) ? P.s0 : 0);
      const float inv_l = l_sum > 0.f ? 1.f / l_norm : 0.f;
      const size_t orow = static_cast<size_t>(b) * p.rows + row;
      const size_t arow = static_cast<size_t>(slot) * p.rows + row;
      const bool direct = (nsplit == 1);
      const bool out16 = direct && p.out_type != MLA_DTYPE_FP32;
      const bool half = p.out_type == MLA_DTYPE_FP16;
      // Through a 4 KB stage per warp (its own rows' bytes of the P buffer,
      // free once the last P V is done): each thread writes its row's 32
      // values, then the warp stores whole row segments, so that a store
      // instruction covers four (fp32) or eight (16-bit) rows' contiguous
      // bytes instead of 32 rows' 16 bytes each.
      uint8_t* stage = sP + warp * (32 * 128);
      const int row_base = rb * kRowsPerBlock + 32 * q;  // the warp's first row
#pragma unroll 1
      for (uint32_t c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kTmemO + 128u * h + c0, v);
        tmem_wait_ld();
        uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
        if (out16) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float x0 = __uint_as_float(v[8 * c + 2 * i]) * inv_l;
              const float x1 = __uint_as_float(v[8 * c + 2 * i + 1]) * inv_l;
              if (half) {
                const __half2 hh = __floats2half2_rn(x0, x1);
                w[i] = *reinterpret_cast<const uint32_t*>(&hh);
              } else {
                const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
                w[i] = *reinterpret_cast<const uint32_t*>(&hh);
              }
            }
            srow[c ^ (lane & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            srow[c ^ (lane & 7)] =
                make_uint4(__float_as_uint(__uint_as_float(v[4 * c]) * inv_l),
                           __float_as_uint(__uint_as_float(v[4 * c + 1]) * inv_l),
                           __float_as_uint(__uint_as_float(v[4 * c + 2]) * inv_l),
                           __float_as_uint(__uint_as_float(v[4 * c + 3]) * inv_l));
        }
        __syncwarp();
        // 16-byte pieces per row: 4 (16-bit output) or 8 (fp32)
        const int pieces = out16 ? 4 : 8;
        const size_t col = 256u * rank + 128u * h + c0;
#pragma unroll 1
        for (int i = lane; i < 32 * pieces; i += 32) {
          const int rl = i / pieces, pc = i - rl * pieces;
          const int row_g = row_base + rl;
          if (row_g < p.rows) {
            const uint4 val = reinterpret_cast<const uint4*>(stage + rl * 128)[pc ^ (rl & 7)];
            if (out16) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                    (static_cast<size_t>(b) * p.rows + row_g) * kDv + col);
              dst[pc] = val;
            } else {
              float* base = direct ? static_cast<float*>(p.out) + (static_cast<size_t>(b) * p.rows + row_g) * kDv
                                   : p.o_accum + (static_cast<size_t>(slot) * p.rows + row_g) * kDv;
              reinterpret_cast<uint4*>(base + col)[pc] = val;
            }
          }
        }
        __syncwarp();
      }
      // the other warp of the pair has read its stage too before either writes
      // the next unit's partial scores into these bytes
      named_bar_sync(pair_bar, pair_n);
      tc_fence_before();
      mbar_arrive(&bars[O_FREE]);
      if (rank == 0 && h == 0 && row_ok) {
        const float lse = l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
        if (direct)
          p.lse[orow] = lse;
        else
          p.lse_accum[arow] = lse;
      }
      ++u;
    }
    if (!ok && sender) {
      set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // partial scores the peer already sent may still be landing here
      mbar_wait<true>(&bars[X_FULL + q], t & 1, nullptr, kWaitNs);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_arrive();  // the peer no longer touches this CTA's shared memory
  cluster_wait();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Selected-record packing (FlashMLA PR #200, "[SM90] Add packed selected-KV
// sparse decode", sections Motivation and "SM90 packing kernel": the selected
// records are copied byte for byte into a tile-major workspace ahead of the
// attention, so that no index translation sits on its critical path).  One
// block per (tile of 64 slots, unit): slot t < topk_length with a valid index
// gets its 656-byte record, every other slot 656 zero bytes; the tile's
// 64-bit valid mask goes to `masks`.  An index outside [-1, pool) is reported
// (MLA_ERR_BAD_INDEX) and packed as masked.
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is signalled as
// transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_smem),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Bulk copy of `bytes` (multiple of 16, 16-byte aligned) from this CTA's shared
// memory to global memory, in the thread's current bulk async-group.
__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(src_smem), "r"(bytes)
               : "memory");
}

// Close the thread's bulk async-group, then wait until all its groups have
// completed (the writes are done).
__device__ __forceinline__ void bulk_commit_and_wait_all() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Wait budget of the stall-test instance (below): short, so that the test
// ends quickly; the real instance keeps the 2 s budget of every other wait.
constexpr uint64_t kStallTestWaitNs = 200000;  // 200 us

// kStallTest: the test instance of the timeout path.  Thread 0 withholds the
// arrival (with the transaction count) that completes its tile's bulk-copy
// barrier, so its bounded wait runs out as if a copy had never landed; it
// reports MLA_ERR_TIMEOUT, zeroes the tile's mask, then makes the arrival
// after all, waits (bounded) until its copies have landed, and leaves without
// storing.  (A barrier's transaction count may go below zero before the
// arrival that raises it: the copies' completions are simply counted first.)
template <bool kStallTest>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t* __restrict__ kv8, int num_pages,
                                                   const int32_t* __restrict__ indices, int topk,
                                                   const int32_t* __restrict__ topk_length, uint8_t* __restrict__ packed,
                                                   uint64_t* __restrict__ masks, int32_t* status) {
  // The tile's 64 records are staged in shared memory: each valid one comes
  // in by one bulk copy (656 bytes, 16-byte aligned at both ends), the others
  // are zero-filled there, and the whole tile (41 984 contiguous bytes) goes
  // out by one bulk store.
  constexpr int kTileBytes = kT * MLA_RECORD_BYTES;
  __shared__ __align__(128) uint8_t s_rec[kTileBytes];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_idx[kT];
  __shared__ uint32_t s_half[2];
  const int tiles = gridDim.x, tile = blockIdx.x, unit = blockIdx.y;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init_cluster();
  }
  if (tid < kT) {
    const int t = tile * kT + tid;
    const int L = topk_length != nullptr ? max(min(topk_length[unit], topk), 0) : topk;
    int idx = -1;
    if (t < L) {
      idx = indices[static_cast<size_t>(unit) * topk + t];
      if (idx != -1 && (idx < 0 || idx >= num_pages * kT)) {
        report(status, MLA_ERR_BAD_INDEX);
        idx = -1;
      }
    }
    s_idx[tid] = idx;
    const uint32_t half = __ballot_sync(0xffffffffu, idx >= 0);
    if ((tid & 31) == 0) s_half[tid >> 5] = half;
  }
  __syncthreads();
  const uint64_t valid = s_half[0] | (static_cast<uint64_t>(s_half[1]) << 32);
  if (tid == 0) masks[static_cast<size_t>(unit) * tiles + tile] = valid;
  const uint32_t n_valid = static_cast<uint32_t>(__popcll(valid));
  if (tid < 32) {
    // warp 0: the transaction count first, then the copies (lanes k and k + 32)
    if (tid == 0 && !kStallTest) mbar_arrive_expect_tx(&s_bar, n_valid * MLA_RECORD_BYTES);
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int k = tid + 32 * h;
      const int idx = s_idx[k];
      if (idx >= 0)
        bulk_load_g2s(smem_u32(s_rec + k * MLA_RECORD_BYTES), kv8 + static_cast<size_t>(idx) * MLA_RECORD_BYTES,
                      MLA_RECORD_BYTES, &s_bar);
    }
  }
  // the unused slots' records are zeros (16-byte pieces, generic proxy)
  for (int c = tid; c < kT * (MLA_RECORD_BYTES / 16); c += 256) {
    const int key = c / (MLA_RECORD_BYTES / 16);
    if (s_idx[key] < 0) reinterpret_cast<uint4*>(s_rec)[c] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();  // the zeros are visible to the bulk store
  __syncthreads();
  if (tid == 0) {
    if (mbar_wait(&s_bar, 0, nullptr, kStallTest ? kStallTestWaitNs : MLA_WAIT_LIMIT_NS)) {
      bulk_store_s2g(packed + (static_cast<size_t>(unit) * tiles + tile) * kTileBytes, smem_u32(s_rec), kTileBytes);
      bulk_commit_and_wait_all();
    } else {
      // the tile's records are not stored: its mask says no slot is valid, so
      // the attention ignores whatever the workspace holds there
      report(status, MLA_ERR_TIMEOUT);
      masks[static_cast<size_t>(unit) * tiles + tile] = 0ull;
      if (kStallTest) mbar_arrive_expect_tx(&s_bar, n_valid * MLA_RECORD_BYTES);  // the withheld arrival
      mbar_wait(&s_bar, 0, nullptr);  // no copy may still be landing when the block exits
    }
  }
}

// Bit-exact record unpack: one thread per (record, 8-dim chunk).
__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ kv8, int num_pages,
                                                     const int32_t* __restrict__ indices, int n,
                                                     float* __restrict__ k_out, int32_t* status) {
  const long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= static_cast<long long>(n) * 72) return;
  const int rec_i = static_cast<int>(g / 72), c = static_cast<int>(g % 72);
  const int idx = indices[rec_i];
  float4* dst = reinterpret_cast<float4*>(k_out + static_cast<size_t>(rec_i) * kDqk + 8 * c);
  if (idx < 0 || idx >= num_pages * kTile) {
    if (idx != -1 && c == 0) report(status, MLA_ERR_BAD_INDEX);
    dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const uint8_t* rec = kv8 + static_cast<size_t>(idx) * MLA_RECORD_BYTES;
  float f[8];
  if (c < 64) {
    const uint2 codes = *reinterpret_cast<const uint2*>(rec + 8 * c);
    const float scale = reinterpret_cast<const float*>(rec + 512)[c >> 4];
    const uint4 b = codes_to_bf16(codes);
    const uint32_t ws[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __fmul_rn(__uint_as_float(ws[i] << 16), scale);
      f[2 * i + 1] = __fmul_rn(__uint_as_float(ws[i] & 0xFFFF0000u), scale);
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(rec + 528 + 16 * (c - 64));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(ws[i] << 16);
      f[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
    }
  }
  dst[0] = make_float4(f[0], f[1], f[2], f[3]);
  dst[1] = make_float4(f[4], f[5], f[6], f[7]);
}

}  // namespace sp

int sparse_smem_bytes() { return sp::kSmemBytes; }
int sparse_threads() { return sp::kThreads; }
// stall 1: the test instance whose first tile's scores are never computed
const void* sparse_kernel_ptr(int stall) {
  return stall ? reinterpret_cast<const void*>(&sp::sparse_decode_kernel<true>)
               : reinterpret_cast<const void*>(&sp::sparse_decode_kernel<false>);
}

cudaError_t launch_sparse(const CUtensorMap& q_map, const DecodeParams& p, int num_parts, int stall,
                          cudaStream_t stream) {
  const dim3 grid(2 * num_parts * p.row_blocks);
  if (stall)
    sp::sparse_decode_kernel<true><<<grid, sp::kThreads, sp::kSmemBytes, stream>>>(q_map, p);
  else
    sp::sparse_decode_kernel<false><<<grid, sp::kThreads, sp::kSmemBytes, stream>>>(q_map, p);
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* kv8, int num_pages, const int32_t* indices, int topk,
                        const int32_t* topk_length, int n_units, uint8_t* packed, uint64_t* masks, int32_t* status,
                        int stall_test, cudaStream_t stream) {
  const dim3 grid((topk + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE, n_units);
  if (stall_test)
    sp::pack_kernel<true><<<grid, 256, 0, stream>>>(kv8, num_pages, indices, topk, topk_length, packed, masks,
                                                    status);
  else
    sp::pack_kernel<false><<<grid, 256, 0, stream>>>(kv8, num_pages, indices, topk, topk_length, packed, masks,
                                                     status);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* kv8, int num_pages, const int32_t* indices, int n, float* k_out,
                          int32_t* status, cudaStream_t stream) {
  const long long threads = static_cast<long long>(n) * 72;
  const int blocks = static_cast<int>((threads + 255) / 256);
  sp::unpack_kernel<<<blocks, 256, 0, stream>>>(kv8, num_pages, indices, n, k_out, status);
  return cudaGetLastError();
}

}  // namespace mla
