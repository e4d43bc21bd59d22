// MLA split-KV decode kernels for sm_103a (tcgen05 + TMEM + TMA), dense bf16
// and sparse FP8.
//
// What they compute (FlashMLA PR #183, "Add SM80 (Ampere/A100) dense MLA
// decode kernel", section Design; FlashMLA PR #200, "[SM90] Add packed
// selected-KV sparse decode", sections Motivation and "SM90 packing
// kernel"): for the 128 query rows of one row block of a unit (all heads
// share one latent KV head), over the keys of one split: S = Q K^T on 576
// dims, online softmax, O = P V with V = the first 512 dims of the same
// latent rows; then O / l and the split's LSE.  Dense keys come from 64-token
// bf16 pages through the block table; sparse keys are 656-byte FP8 records
// picked by physical slot index and dequantised in the kernel.
//
// How (GB300 design, not the pages' SM80/SM90 ones):
//  * One 2-CTA cluster per (partition, row block).  TMEM holds 512 fp32
//    columns per SM, exactly one 128 x 512 accumulator, so the two CTAs
//    split the value dims: rank c accumulates O[:, 256c : 256c+256).  To
//    avoid computing Q K^T twice they also split the score dims: rank 0 sums
//    dims [0, 288), rank 1 dims [288, 576), and the two partial score tiles
//    are exchanged through distributed shared memory.  Both ranks then run
//    the same softmax on the same sums, so P is identical on both.
//  * Each CTA stages the 64-column boxes it needs: rank c boxes 4c .. 4c+4
//    (320 dims: its score dims plus its value dims) of Q (once per unit) and
//    of every 64-key tile, in a 2-stage mbarrier ring.  Dense: one TMA per
//    box, 128-byte swizzle, page from the block table.  Sparse: a producer
//    warpgroup gathers the records, dequantises E4M3 x fp32 scale to bf16
//    and writes the same swizzled layout.
//  * tcgen05.mma M=128: S (N=64) and O (N=256) accumulate in TMEM.  P is
//    written as bf16 by the softmax threads into swizzled shared memory.
//  * Online softmax in the log2 domain with a lazy rescale: O is rescaled
//    only when the running max grows by more than 2^8.
// Roles: warps 0-3 softmax + epilogue (thread = row = TMEM lane),
//        then the producer warp(s), then one MMA warp that owns TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {
namespace dec {

constexpr int kBoxes = 5;
constexpr int kQBoxBytes = kRowsPerBlock * 128;  // 128 rows x 64 bf16
constexpr int kKVBoxBytes = kTile * 128;         // 64 keys x 64 bf16
constexpr int kStages = 2;
constexpr int kStageBytes = kBoxes * kKVBoxBytes;
constexpr int kXBytes = kRowsPerBlock * kTile * 4;  // peer's partial scores
constexpr int kPBytes = kRowsPerBlock * kTile * 2;  // P tile, bf16

constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kBoxes * kQBoxBytes;
constexpr int kOffX = kOffKV + kStages * kStageBytes;
constexpr int kOffP = kOffX + kXBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kNumBars = 26;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // S buffers: [256, 320) and [320, 384)

enum : int {
  Q_FULL = 0,
  Q_EMPTY = 1,
  KV_FULL = 2,   // +stage
  KV_EMPTY = 4,  // +stage
  S_FULL = 6,    // +buffer
  S_FREE = 8,    // +buffer
  P_FULL = 10,   // +buffer
  P_FREE = 12,   // +buffer
  O_FULL = 14,
  O_FREE = 15,
  X_FULL = 16,   // +warp
  X_FREE = 20,   // +warp
  DRAIN = 24,
};

constexpr float kTau = 8.0f;  // lazy-rescale threshold (log2 units)
constexpr float kLn2 = 0.69314718055994530942f;

template <bool kSparse>
struct Roles {
  static constexpr int kProducerWarps = kSparse ? 4 : 1;
  static constexpr int kMmaWarp = 4 + kProducerWarps;
  static constexpr int kThreads = 32 * (kMmaWarp + 1);
};

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

struct Part {
  int b0, t0, b1, t1, s0;
};

__device__ __forceinline__ Part load_part(const int32_t* sched, int idx) {
  const int32_t* e = sched + idx * MLA_SCHED_INTS;
  return Part{e[0], e[1], e[2], e[3], e[4]};
}

// Keys of unit b (sparse lengths are clamped to topk).
__device__ __forceinline__ int unit_len(const DecodeParams& p, int b) {
  int L = p.lengths != nullptr ? p.lengths[b] : p.default_length;
  if (p.indices != nullptr) L = min(L, p.topk);
  return max(L, 0);
}

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
    unit_tiles(P, b, num_tiles(unit_len(p, b)), lo, hi);
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

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait<true>(bar, parity, abort_flag));
}

// 8 E4M3 codes times one fp32 scale -> 8 bf16 (fp32 product rounded once to bf16).
__device__ __forceinline__ uint4 dequant8(uint2 codes, float scale) {
  uint32_t w[4];
  const uint32_t src[2] = {codes.x, codes.y};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const __nv_fp8x2_storage_t two = static_cast<__nv_fp8x2_storage_t>((src[h] >> (16 * q)) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
      w[2 * h + q] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Validity of sparse selection entry t of unit b (as the oracle defines it).
__device__ __forceinline__ bool sparse_valid(const DecodeParams& p, int b, int t, int L, int& idx) {
  idx = -1;
  if (t >= L) return false;
  idx = p.indices[static_cast<size_t>(b) * p.topk + t];
  if (idx == -1) return false;
  if (idx < 0 || idx >= p.num_pages * kTile) {
    report(p.status, MLA_ERR_BAD_INDEX);
    idx = -1;
    return false;
  }
  return true;
}

template <bool kSparse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Roles<kSparse>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kv_map,
                      const DecodeParams p) {
  using R = Roles<kSparse>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKV = smem + kOffKV;
  uint8_t* sX = smem + kOffX;
  uint8_t* sP = smem + kOffP;
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

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bars[Q_FULL], 1);
    mbar_init(&bars[Q_EMPTY], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[KV_FULL + i], kSparse ? 32 * R::kProducerWarps : 1);
      mbar_init(&bars[KV_EMPTY + i], 1);
      mbar_init(&bars[S_FULL + i], 1);
      mbar_init(&bars[S_FREE + i], 128);
      mbar_init(&bars[P_FULL + i], 128);
      mbar_init(&bars[P_FREE + i], 1);
    }
    mbar_init(&bars[O_FULL], 1);
    mbar_init(&bars[O_FREE], 128);
    for (int w = 0; w < 4; ++w) {
      mbar_init(&bars[X_FULL + w], 32);
      mbar_init(&bars[X_FREE + w], 32);
    }
    mbar_init(&bars[DRAIN], 1);
    fence_mbar_init_cluster();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&q_map);
    if (!kSparse) prefetch_tmap(&kv_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // the peer's barriers are initialised before any remote arrive
  cluster_wait();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  const Part P = load_part(p.sched, part_idx);

  if (warp >= 4 && warp < R::kMmaWarp) {
    // ------------------------------------------------------------ producer
    const int ptid = tid - 128;  // 0 .. 32*kProducerWarps-1
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    uint32_t t = 0;
    int u = 0;
    bool ok = true;
    uint32_t issued[2] = {0u, 0u};
    uint32_t q_issued = 0;
    for (int b = P.b0; ok && unit_in_part(P, b, p.n_units); ++b) {
      const int L = unit_len(p, b);
      const int nt = num_tiles(L);
      int lo, hi;
      unit_tiles(P, b, nt, lo, hi);
      if (hi <= lo) continue;
      if (ptid == 0) {
        if (u >= 1) ok = mbar_wait(&bars[Q_EMPTY], (u - 1) & 1, abort_flag);
        if (ok) {
          mbar_arrive_expect_tx(&bars[Q_FULL], kBoxes * kQBoxBytes);
          const int row0 = b * p.rows + rb * kRowsPerBlock;
#pragma unroll
          for (int lb = 0; lb < kBoxes; ++lb)
            tma_load_2d(sQ + lb * kQBoxBytes, &q_map, &bars[Q_FULL], 64 * (4 * static_cast<int>(rank) + lb), row0,
                        pol_q);
          ++q_issued;
        }
      }
      if constexpr (!kSparse) {
        ok = __shfl_sync(0xffffffffu, ok, 0);
        int page_reg = 0;
        for (int k = lo; ok && k < hi; ++k, ++t) {
          if (((k - lo) & 31) == 0) {
            const int kk = k + lane;
            int pg = 0;
            if (kk < hi) {
              pg = kk < p.max_pages ? p.block_table[static_cast<size_t>(b) * p.max_pages + kk] : -1;
              if (pg < 0 || pg >= p.num_pages) {
                report(p.status, MLA_ERR_BAD_INDEX);
                pg = 0;
              }
            }
            page_reg = pg;
          }
          const int page = __shfl_sync(0xffffffffu, page_reg, (k - lo) & 31);
          const int st = t & 1;
          if (lane == 0) {
            if (t >= 2) ok = mbar_wait(&bars[KV_EMPTY + st], ((t - 2) >> 1) & 1, abort_flag);
            if (ok) {
              mbar_arrive_expect_tx(&bars[KV_FULL + st], kStageBytes);
#pragma unroll
              for (int lb = 0; lb < kBoxes; ++lb)
                tma_load_3d(sKV + st * kStageBytes + lb * kKVBoxBytes, &kv_map, &bars[KV_FULL + st],
                            64 * (4 * static_cast<int>(rank) + lb), 0, page, pol_kv);
              ++issued[st];
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      } else {
        // gather + dequant: 64 keys x 40 chunks of 8 dims (dims 256*rank + 8c)
        constexpr int kChunks = kTile * 40;
        constexpr int kPer = kChunks / (32 * R::kProducerWarps);
        static_assert(kChunks % (32 * R::kProducerWarps) == 0, "chunk split");
        const int dim0 = 256 * static_cast<int>(rank);
        for (int k = lo; ok && k < hi; ++k, ++t) {
          const int st = t & 1;
          if (t >= 2) ok = mbar_wait(&bars[KV_EMPTY + st], ((t - 2) >> 1) & 1, abort_flag);
          if (!ok) break;
          uint4 raw[kPer];
          float sc[kPer];
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int q = ptid + 32 * R::kProducerWarps * i;
            const int key = q / 40, c = q - 40 * (q / 40);
            const int d = dim0 + 8 * c;
            int idx;
            raw[i] = make_uint4(0u, 0u, 0u, 0u);
            sc[i] = 0.f;
            if (sparse_valid(p, b, k * kTile + key, L, idx)) {
              const uint8_t* rec = p.kv8 + static_cast<size_t>(idx) * MLA_RECORD_BYTES;
              if (d < 512) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(rec + d));
                raw[i] = make_uint4(v.x, v.y, 0u, 0u);
                sc[i] = __ldg(reinterpret_cast<const float*>(rec + 512) + (d >> 7));
              } else {
                raw[i] = __ldg(reinterpret_cast<const uint4*>(rec + 528 + 2 * (d - 512)));
                sc[i] = 1.f;
              }
            }
          }
          uint8_t* stage = sKV + st * kStageBytes;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int q = ptid + 32 * R::kProducerWarps * i;
            const int key = q / 40, c = q - 40 * (q / 40);
            const int d = dim0 + 8 * c;
            const uint4 outv = (d < 512) ? dequant8(make_uint2(raw[i].x, raw[i].y), sc[i]) : raw[i];
            const int lb = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4*>(stage + lb * kKVBoxBytes + key * 128 + ((cc ^ (key & 7)) << 4)) = outv;
          }
          fence_proxy_async_smem();
          mbar_arrive(&bars[KV_FULL + st]);
        }
      }
      ++u;
    }
    if (ptid == 0) {
      if (!ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
      // no TMA write may land after this CTA exits
      if (!kSparse)
        for (int st = 0; st < 2; ++st)
          if (issued[st] > 0) mbar_wait(&bars[KV_FULL + st], (issued[st] - 1) & 1, nullptr);
      if (q_issued > 0) mbar_wait(&bars[Q_FULL], (q_issued - 1) & 1, nullptr);
    }
    if (kSparse && !ok) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
  } else if (warp == R::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, kTile, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, 256, true);
      const int ks0 = rank == 0 ? 0 : 18;
      const int ks1 = ks0 + 18;
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kv_desc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(sKV), kKVBoxBytes, 1024);
      const uint64_t p_desc0 = sdesc_sw128(smem_u32(sP), 16, 1024);
      // Two cursors over the partition's (unit, tile) sequence: QK runs ahead of
      // PV by at most the two S/KV buffers.  Whichever is ready is issued, PV
      // first, so a KV stage is released as soon as its PV is issued.
      Cursor cq, cv;
      cursor_init(p, P, cq);
      cursor_init(p, P, cv);
      bool ok = true;
      uint64_t t_last = globaltimer_ns();
      while (cv.valid) {
        bool progressed = false;
        if (cv.t < cq.t) {
          const int pb = cv.t & 1;
          bool ready = mbar_test_wait(&bars[P_FULL + pb], (cv.t >> 1) & 1);
          const bool first = cv.k == cv.lo, last = cv.k == cv.hi - 1;
          if (ready && first && cv.u >= 1) ready = mbar_test_wait(&bars[O_FREE], (cv.u - 1) & 1);
          if (ready) {
            tc_fence_after();
            const uint64_t a0 = p_desc0 + static_cast<uint64_t>((pb * kPBytes) >> 4);
            const uint64_t b0 = v_desc0 + static_cast<uint64_t>((pb * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_f16(tmem + kTmemO, a0 + static_cast<uint64_t>((kk * 32) >> 4),
                       b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (first && kk == 0) ? 0u : 1u);
            umma_commit(&bars[P_FREE + pb]);
            umma_commit(&bars[KV_EMPTY + pb]);
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
          if (ready && cq.t >= 2) ready = mbar_test_wait(&bars[S_FREE + st], ((cq.t - 2) >> 1) & 1);
          if (ready) {
            tc_fence_after();
            const uint64_t kvs = kv_desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
            for (int ks = ks0; ks < ks1; ++ks) {
              const int lb = (ks >> 2) - 4 * static_cast<int>(rank);
              const uint32_t off_q = lb * kQBoxBytes + (ks & 3) * 32;
              const uint32_t off_k = lb * kKVBoxBytes + (ks & 3) * 32;
              umma_f16(tmem + kTmemS + 64u * st, q_desc0 + (off_q >> 4), kvs + (off_k >> 4), idesc_qk,
                       ks > ks0 ? 1u : 0u);
            }
            umma_commit(&bars[S_FULL + st]);
            if (cq.k == cq.hi - 1) umma_commit(&bars[Q_EMPTY]);
            cursor_next(p, P, cq);
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
          __nanosleep(32);
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
    const uint32_t x_local = smem_u32(sX) + r * 256;
    const uint32_t x_remote = mapa_shared(x_local, peer);
    const uint32_t xfull_remote = mapa_shared(smem_u32(&bars[X_FULL + warp]), peer);
    const uint32_t xfree_remote = mapa_shared(smem_u32(&bars[X_FREE + warp]), peer);
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    uint32_t t = 0;
    int u = 0;
    bool ok = true;
    for (int b = P.b0; ok && unit_in_part(P, b, p.n_units); ++b) {
      const int L = unit_len(p, b);
      const int nt = num_tiles(L);
      int lo, hi;
      unit_tiles(P, b, nt, lo, hi);
      if (hi <= lo) continue;
      const int row = rb * kRowsPerBlock + r;
      const bool row_ok = row < p.rows;
      const int tok = row_ok ? row / p.h_q : 0;
      const int jmax = p.causal ? (L - p.s_q + tok) : (L - 1);  // dense: last visible key
      // l_sum: fp32 sum of the unrounded weights (gives the LSE);
      // l_used: sum of the bf16 weights the tensor core multiplies (normalises O)
      float m_used = -INFINITY, l_sum = 0.f, l_used = 0.f;
      for (int k = lo; ok && k < hi; ++k, ++t) {
        // which of the tile's 64 keys this row may see
        uint64_t vis_mask;
        if constexpr (kSparse) {
          int idx;
          const bool v0 = sparse_valid(p, b, k * kTile + lane, L, idx);
          const bool v1 = sparse_valid(p, b, k * kTile + 32 + lane, L, idx);
          vis_mask = static_cast<uint64_t>(__ballot_sync(0xffffffffu, v0)) |
                     (static_cast<uint64_t>(__ballot_sync(0xffffffffu, v1)) << 32);
        } else {
          const int vis = jmax - k * kTile;  // keys 0..vis of this tile are visible
          vis_mask = vis >= 63 ? ~0ull : (vis < 0 ? 0ull : ((2ull << vis) - 1ull));
        }
        const int sb = t & 1;
        ok = warp_wait(&bars[S_FULL + sb], (t >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[64];
        {
          uint32_t (&lo32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          uint32_t (&hi32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
          tmem_ld32(tmem + lane_base + kTmemS + 64u * sb, lo32);
          tmem_ld32(tmem + lane_base + kTmemS + 64u * sb + 32u, hi32);
          tmem_wait_ld();
        }
        tc_fence_before();
        mbar_arrive(&bars[S_FREE + sb]);
        // swap partial scores with the peer CTA
        if (t >= 1) {
          ok = warp_wait_cluster(&bars[X_FREE + warp], (t - 1) & 1, abort_flag);
          if (!ok) break;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_cluster_v4(x_remote + ((static_cast<uint32_t>(c) ^ swz) << 4), __uint_as_float(sr[4 * c]),
                        __uint_as_float(sr[4 * c + 1]), __uint_as_float(sr[4 * c + 2]),
                        __uint_as_float(sr[4 * c + 3]));
        mbar_arrive_remote(xfull_remote);
        ok = warp_wait_cluster(&bars[X_FULL + warp], t & 1, abort_flag);
        if (!ok) break;
        float s[64];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 o = ld_shared_v4(x_local + ((static_cast<uint32_t>(c) ^ swz) << 4));
          s[4 * c + 0] = __uint_as_float(sr[4 * c + 0]) + o.x;
          s[4 * c + 1] = __uint_as_float(sr[4 * c + 1]) + o.y;
          s[4 * c + 2] = __uint_as_float(sr[4 * c + 2]) + o.z;
          s[4 * c + 3] = __uint_as_float(sr[4 * c + 3]) + o.w;
        }
        mbar_arrive_remote(xfree_remote);
        // mask, scale into the log2 domain, tile max
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          s[j] = ((vis_mask >> j) & 1ull) ? s[j] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[j]);
        }
        bool rescale = false;
        float alpha = 1.f;
        if (mt > m_used + kTau) {
          alpha = ex2(m_used - mt);  // 0 when m_used == -inf
          rescale = k > lo;
          l_sum *= alpha;
          l_used *= alpha;
          m_used = mt;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        uint32_t pk[32];
        float psum = 0.f, pused = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2(s[2 * i] - mref), p1 = ex2(s[2 * i + 1] - mref);
          const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
          const float2 back = __bfloat1622float2(h);
          psum += p0 + p1;
          pused += back.x + back.y;
          pk[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        l_sum += psum;
        l_used += pused;
        const int pb = t & 1;
        if (t >= 2) {
          ok = warp_wait(&bars[P_FREE + pb], ((t - 2) >> 1) & 1, abort_flag);
          if (!ok) break;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O accumulated so far (through PV of the previous tile) times alpha
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
        uint8_t* prow = sP + pb * kPBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((static_cast<uint32_t>(c) ^ swz) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[P_FULL + pb]);
      }
      if (!ok) break;
      // ---- epilogue of this (unit, split)
      ok = warp_wait(&bars[O_FULL], u & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int s_begin = p.split_offset[b];
      const int nsplit = p.split_offset[b + 1] - s_begin;
      const int slot = s_begin + ((b == P.b0) ? P.s0 : 0);
      const float inv_l = l_used > 0.f ? 1.f / l_used : 0.f;
      const size_t orow = static_cast<size_t>(b) * p.rows + row;
      const size_t arow = static_cast<size_t>(slot) * p.rows + row;
      const bool direct = (nsplit == 1);
#pragma unroll 1
      for (uint32_t c0 = 0; c0 < 256; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kTmemO + c0, v);
        tmem_wait_ld();
        if (!row_ok) continue;
        const size_t col = 256u * rank + c0;
        if (direct && !p.out_fp32) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow * kDv + col);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[8 * c + 2 * i]) * inv_l,
                                                             __uint_as_float(v[8 * c + 2 * i + 1]) * inv_l);
              w[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float* dst = direct ? static_cast<float*>(p.out) + orow * kDv + col : p.o_accum + arow * kDv + col;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            reinterpret_cast<float4*>(dst)[c] =
                make_float4(__uint_as_float(v[4 * c]) * inv_l, __uint_as_float(v[4 * c + 1]) * inv_l,
                            __uint_as_float(v[4 * c + 2]) * inv_l, __uint_as_float(v[4 * c + 3]) * inv_l);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[O_FREE]);
      if (rank == 0 && row_ok) {
        const float lse = l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
        if (direct)
          p.lse[orow] = lse;
        else
          p.lse_accum[arow] = lse;
      }
      ++u;
    }
    if (!ok && lane == 0) set_abort(abort_flag, p.status, MLA_ERR_TIMEOUT);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_arrive();  // the peer no longer touches this CTA's shared memory
  cluster_wait();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
    const uint32_t src[2] = {codes.x, codes.y};
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const __nv_fp8x2_storage_t two = static_cast<__nv_fp8x2_storage_t>((src[h] >> (16 * q)) & 0xFFFFu);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        f[4 * h + 2 * q] = __fmul_rn(v.x, scale);
        f[4 * h + 2 * q + 1] = __fmul_rn(v.y, scale);
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

}  // namespace dec

int sparse_smem_bytes() { return dec::kSmemBytes; }
int sparse_threads() { return dec::Roles<true>::kThreads; }
const void* sparse_kernel_ptr() { return reinterpret_cast<const void*>(&dec::mla_decode_kernel<true>); }

cudaError_t launch_sparse(const CUtensorMap& q_map, const DecodeParams& p, int num_parts, cudaStream_t stream) {
  const dim3 grid(2 * num_parts * p.row_blocks);
  // the KV map is unused by the sparse kernel; pass the Q map in its place
  dec::mla_decode_kernel<true><<<grid, dec::Roles<true>::kThreads, dec::kSmemBytes, stream>>>(q_map, q_map, p);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* kv8, int num_pages, const int32_t* indices, int n, float* k_out,
                          int32_t* status, cudaStream_t stream) {
  const long long threads = static_cast<long long>(n) * 72;
  const int blocks = static_cast<int>((threads + 255) / 256);
  dec::unpack_kernel<<<blocks, 256, 0, stream>>>(kv8, num_pages, indices, n, k_out, status);
  return cudaGetLastError();
}

}  // namespace mla
