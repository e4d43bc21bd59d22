// LSE-weighted combine of split-KV partials.
//
// FlashMLA PR #183 (Summary; "Modifications outside csrc/sm80/") merges the
// per-split partial outputs with a combine kernel and bounds the split count
// by a compile-time ladder.  Here the split count is a runtime loop bound, so
// any number of splits is merged.  Per output row:
//   m = max_s lse_s,  w_s = exp(lse_s - m),  Z = sum_s w_s,
//   out = sum_s (w_s / Z) O_s,  lse = m + ln Z
// with -inf splits weighing 0 and an all-empty row giving out 0, lse -inf.
// Memory bound: every partial is read once, by 32 KB bulk copies (16 rows of
// one split) or, for long-context units, as 512-byte coalesced row quarters.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kCombineWarps = 4;

__device__ __forceinline__ void store_row4(void* out, int out_type, size_t elem, float a, float b, float c,
                                           float d) {
  if (out_type == MLA_DTYPE_FP32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + elem) = make_float4(a, b, c, d);
  } else if (out_type == MLA_DTYPE_FP16) {
    __half2 lo = __floats2half2_rn(a, b);
    __half2 hi = __floats2half2_rn(c, d);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__half*>(out) + elem) = v;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
    __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + elem) = v;
  }
}

__device__ __forceinline__ void acc4(float4& a, float w, const float4& v) {
  if (w != 0.f) {  // a -inf split weighs exactly 0 whatever its partial holds
    a.x = fmaf(w, v.x, a.x);
    a.y = fmaf(w, v.y, a.y);
    a.z = fmaf(w, v.z, a.z);
    a.w = fmaf(w, v.w, a.w);
  }
}

// Many rows (enough to fill the GPU several times over), few splits each:
// a warp merges a whole 512-column row (kVec = 4 float4 per lane per split;
// a block = 4 rows).  Its blocks hold no shared memory, so they stay
// resident beside the attention kernel's CTAs and start the moment it ends.
// Latency: split_offset comes from the plan (complete before the attention
// grid started), so it is read before waiting for that grid.  After the wait
// the split LSEs are loaded with the lanes spread over the splits, and in the
// same round trip the partial rows of the first kPre = 2 splits (the count
// most units have when partitions slightly outnumber requests; a batch of 4
// is 16 float4 a lane, and its registers cost more occupancy than the round
// trip saves).
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_rows_kernel(const float* __restrict__ o_accum, const float* __restrict__ lse_accum,
                        const int32_t* __restrict__ split_offset, int rows, void* __restrict__ out, int out_type,
                        float* __restrict__ lse) {
  constexpr int kVec = 4;
  constexpr int kBatch = 4;
  constexpr int kPre = 2;  // partial rows loaded with the LSEs
  const int unit = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineWarps + warp;
  if (row >= rows) return;
  const int s0 = split_offset[unit];
  const int n = split_offset[unit + 1] - s0;
  if (n == 1) return;  // written directly by the attention kernel
  pdl_wait_prior_grid();
  const size_t orow = static_cast<size_t>(unit) * rows + row;
  const size_t col = lane * 4;
  const bool writes_lse = lane == 0;
  const size_t split_stride = static_cast<size_t>(rows) * kDv / 4;  // float4 between consecutive splits
  const float4* src0 = reinterpret_cast<const float4*>(o_accum + (static_cast<size_t>(s0) * rows + row) * kDv + col);

  // the first 32 LSEs (and the first kPre splits' rows), all in flight at once
  const float l0 = lane < n ? lse_accum[static_cast<size_t>(s0 + lane) * rows + row] : -INFINITY;
  const int first = min(n, kPre);
  float4 v0[kPre][kVec];
#pragma unroll
  for (int i = 0; i < kPre; ++i)
#pragma unroll
    for (int k = 0; k < kVec; ++k)
      v0[i][k] = i < first ? __ldg(src0 + static_cast<size_t>(i) * split_stride + 32 * k)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
  float m = l0;
  for (int s = 32 + lane; s < n; s += 32) m = fmaxf(m, lse_accum[static_cast<size_t>(s0 + s) * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (n <= 0 || m == -INFINITY) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) store_row4(out, out_type, orow * kDv + col + 128 * k, 0.f, 0.f, 0.f, 0.f);
    if (writes_lse) lse[orow] = -INFINITY;
    return;
  }
  float z = (l0 == -INFINITY) ? 0.f : expf(l0 - m);
  for (int s = 32 + lane; s < n; s += 32) {
    const float l = lse_accum[static_cast<size_t>(s0 + s) * rows + row];
    z += (l == -INFINITY) ? 0.f : expf(l - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float inv_z = 1.f / z;

  float4 acc[kVec];
#pragma unroll
  for (int k = 0; k < kVec; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  {
    const float w = (l0 == -INFINITY) ? 0.f : expf(l0 - m) * inv_z;
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const float wj = __shfl_sync(0xffffffffu, w, i);
      if (i < first)
#pragma unroll
        for (int k = 0; k < kVec; ++k) acc4(acc[k], wj, v0[i][k]);
    }
  }
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int cnt = min(32, n - c0);
    const float l = lane < cnt ? lse_accum[static_cast<size_t>(s0 + c0 + lane) * rows + row] : -INFINITY;
    const float w = (l == -INFINITY) ? 0.f : expf(l - m) * inv_z;
    const float4* src = src0 + static_cast<size_t>(c0) * split_stride;
    int j = c0 == 0 ? first : 0;  // the first batch is already summed
    for (; j + kBatch <= cnt; j += kBatch) {
      float4 v[kBatch][kVec];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
#pragma unroll
        for (int k = 0; k < kVec; ++k) v[i][k] = __ldg(src + static_cast<size_t>(j + i) * split_stride + 32 * k);
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const float wj = __shfl_sync(0xffffffffu, w, j + i);
#pragma unroll
        for (int k = 0; k < kVec; ++k) acc4(acc[k], wj, v[i][k]);
      }
    }
    for (; j < cnt; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
      for (int k = 0; k < kVec; ++k) acc4(acc[k], wj, __ldg(src + static_cast<size_t>(j) * split_stride + 32 * k));
    }
  }
#pragma unroll
  for (int k = 0; k < kVec; ++k)
    store_row4(out, out_type, orow * kDv + col + 128 * k, acc[k].x, acc[k].y, acc[k].z, acc[k].w);
  if (writes_lse) lse[orow] = m + logf(z);
}

// Few rows, many splits (long context: one unit, dozens of splits): one
// block per (row, 128-column quarter); its kSubsets warps take every
// kSubsets-th split each.  A warp loads the LSEs and partial rows of up to
// kBatch of its splits in one round of loads and merges them into its own
// (max, sum, weighted row) with the LSE rule, rescaling what it has when a
// later round raises its max; the warps' triples are then merged the same
// way through shared memory.  So the whole combine is one round of global
// latency for up to kSubsets * kBatch splits, instead of one round for the
// maximum, one for the sum and one per batch of rows.
constexpr int kSubsets = 8;

__global__ void __launch_bounds__(kSubsets * 32)
    combine_split_kernel(const float* __restrict__ o_accum, const float* __restrict__ lse_accum,
                         const int32_t* __restrict__ split_offset, int rows, void* __restrict__ out, int out_type,
                         float* __restrict__ lse) {
  constexpr int kBatch = 12;
  __shared__ float4 part[kSubsets][32];
  __shared__ float part_m[kSubsets], part_z[kSubsets];
  const int unit = blockIdx.y;
  const int row = blockIdx.x >> 2, quarter = blockIdx.x & 3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (row >= rows) return;  // uniform over the block
  const int s0 = split_offset[unit];  // from the plan: read before the wait
  const int n = split_offset[unit + 1] - s0;
  if (n == 1) return;  // written directly by the attention kernel
  pdl_wait_prior_grid();
  const size_t orow = static_cast<size_t>(unit) * rows + row;
  const size_t col = static_cast<size_t>(quarter) * 128 + lane * 4;
  const size_t split_stride = static_cast<size_t>(rows) * kDv / 4;  // float4 between consecutive splits
  const float4* src = reinterpret_cast<const float4*>(o_accum + (static_cast<size_t>(s0) * rows + row) * kDv + col);

  // this warp's splits: max m, sum z of exp(lse - m), row acc of exp(lse - m) * O
  float m = -INFINITY, z = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = warp; s < n; s += kSubsets * kBatch) {
    float4 v[kBatch];
    float l[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int si = s + i * kSubsets;
      l[i] = si < n ? lse_accum[static_cast<size_t>(s0 + si) * rows + row] : -INFINITY;
      v[i] = si < n ? __ldg(src + static_cast<size_t>(si) * split_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mb = m;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) mb = fmaxf(mb, l[i]);
    if (mb == -INFINITY) continue;  // nothing but empty splits so far
    const float r = (m == -INFINITY) ? 0.f : expf(m - mb);
    z *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
    m = mb;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const float w = (l[i] == -INFINITY) ? 0.f : expf(l[i] - m);
      z += w;
      acc4(acc, w, v[i]);
    }
  }
  part[warp][lane] = acc;
  if (lane == 0) {
    part_m[warp] = m;
    part_z[warp] = z;
  }
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kSubsets; ++k) M = fmaxf(M, part_m[k]);
    if (M == -INFINITY) {  // every split empty
      store_row4(out, out_type, orow * kDv + col, 0.f, 0.f, 0.f, 0.f);
      if (quarter == 0 && lane == 0) lse[orow] = -INFINITY;
      return;
    }
    float Z = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kSubsets; ++k) {
      const float mk = part_m[k];
      const float r = (mk == -INFINITY) ? 0.f : expf(mk - M);
      Z = fmaf(part_z[k], r, Z);
      acc4(t, r, part[k][lane]);
    }
    const float inv_z = 1.f / Z;
    store_row4(out, out_type, orow * kDv + col, t.x * inv_z, t.y * inv_z, t.z * inv_z, t.w * inv_z);
    if (quarter == 0 && lane == 0) lse[orow] = M + logf(Z);
  }
}

// Units with a few splits each (the common case: partitions slightly
// outnumber requests): one persistent block per SM streams the partial rows
// through shared memory by bulk copies, so that the loads of several items
// are in flight at once without holding registers, and no item waits a
// whole round trip for its rows.  An item is 16 consecutive rows of one
// unit; one split's partials for it are 16 x 512 contiguous fp32 (32 KB),
// one cp.async.bulk.  A producer thread runs up to kCsStages such copies
// ahead, through the items this block takes (blockIdx.x, + gridDim.x, ...);
// consumer warp w merges row w of each item: the maximum of the split LSEs,
// their sum of exp(lse - m), the weights exp(lse_s - m) / Z, then the rows
// accumulated in split order by fmaf (a -inf split adds nothing).  The
// split LSEs of the next item are loaded while the current one is merged.
constexpr int kCsRows = 16;                      // rows per item
constexpr int kCsChunkBytes = kCsRows * kDv * 4;  // one split's rows of an item
constexpr int kCsStages = 6;
constexpr int kCsWarps = kCsRows;                // consumer warp w <-> row w of the item
constexpr int kCsThreads = 32 * (kCsWarps + 1);   // + the producer warp
constexpr int kCsSmemBytes = kCsStages * kCsChunkBytes + 2 * kCsStages * 8 + 16;

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing as
// transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_smem),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool warp_all_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

// Item k of this block is blockIdx.x + k * gridDim.x (a fixed sequence, so
// that the split offsets of later items can be loaded ahead without waiting
// for them): unit u, its rows r0 .. r0 + 15, its splits s0 .. s0 + n - 1.
struct CsItem {
  int u, r0, s0, n;  // u = -1: past the block's last item
};

__device__ __forceinline__ CsItem cs_load(const int32_t* split_offset, int k, int items, int chunks) {
  const int it = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
  if (it >= items) return CsItem{-1, 0, 0, 0};
  const int u = it / chunks;
  return CsItem{u, (it - u * chunks) * kCsRows, split_offset[u], split_offset[u + 1]};  // n: see cs_fix
}

// cs_load leaves the end offset in n so that nothing waits for the loads
// until the item is used.
__device__ __forceinline__ CsItem cs_fix(CsItem x) {
  x.n -= x.s0;
  return x;
}

__global__ void __launch_bounds__(kCsThreads, 1)
    combine_stream_kernel(const float* __restrict__ o_accum, const float* __restrict__ lse_accum,
                          const int32_t* __restrict__ split_offset, int n_units, int rows, void* __restrict__ out,
                          int out_type, float* __restrict__ lse, int32_t* status) {
  extern __shared__ __align__(128) uint8_t cs_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(cs_smem + kCsStages * kCsChunkBytes);
  uint64_t* empty = full + kCsStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCsStages);
  int* issued = reinterpret_cast<int*>(empty + kCsStages) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunks = ceil_div_i(rows, kCsRows);
  const int items = n_units * chunks;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *issued = 0;
    for (int i = 0; i < kCsStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCsWarps);
    }
    fence_mbar_init_cluster();
  }
  __syncthreads();
  // split_offset is the plan's (complete before the grid before): read it before the wait
  CsItem nx = cs_load(split_offset, 0, items, chunks);
  pdl_wait_prior_grid();  // the partials and their LSEs come from the grid before

  if (warp == kCsWarps) {
    // ---- producer: one copy of up to 32 KB per (item, split), kCsStages ahead
    if (lane == 0) {
      uint32_t j = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const CsItem x = cs_fix(nx);
        if (x.u < 0) break;
        nx = cs_load(split_offset, k + 1, items, chunks);
        if (x.n == 1) continue;  // written directly by the attention kernel
        const uint32_t bytes = static_cast<uint32_t>(min(kCsRows, rows - x.r0)) * kDv * 4;
        for (int s = 0; s < x.n; ++s, ++j) {
          const uint32_t st = j % kCsStages;
          if (j >= kCsStages && !mbar_wait(&empty[st], (j / kCsStages - 1) & 1, abort_flag)) {
            report(status, MLA_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], bytes);
          bulk_g2s(smem_u32(cs_smem + st * kCsChunkBytes),
                   o_accum + (static_cast<size_t>(x.s0 + s) * rows + x.r0) * kDv, bytes, &full[st]);
        }
      }
      *issued = static_cast<int>(j);
    }
    __syncwarp();
  } else {
    // ---- consumers: warp w merges row r0 + w of every item
    const int w = warp;
    CsItem cur = cs_fix(nx);
    nx = cs_load(split_offset, 1, items, chunks);
    // the first 32 split LSEs of the current item's row
    auto load_l = [&](const CsItem& x) -> float {
      return (x.u >= 0 && x.n != 1 && lane < x.n && x.r0 + w < rows)
                 ? lse_accum[static_cast<size_t>(x.s0 + lane) * rows + x.r0 + w]
                 : -INFINITY;
    };
    float l_next = load_l(cur);
    uint32_t j = 0;
    bool ok = true;
    for (int k = 0; ok && cur.u >= 0; ++k) {
      const CsItem x = cur;
      const float l0 = l_next;
      // the next item's LSEs (its offsets came an item ago) and the offsets of
      // the one after, both in flight while this item is merged
      cur = cs_fix(nx);
      nx = cs_load(split_offset, k + 2, items, chunks);
      l_next = load_l(cur);
      if (x.n == 1) continue;
      const int row = x.r0 + w;
      const bool live = row < rows;  // a last, partial item: its extra warps only pace the stages
      const int n = x.n;
      float m = live ? l0 : -INFINITY;
      if (live)
        for (int s = 32 + lane; s < n; s += 32) m = fmaxf(m, lse_accum[static_cast<size_t>(x.s0 + s) * rows + row]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float z = (l0 == -INFINITY || !live) ? 0.f : expf(l0 - m);
      if (live && m != -INFINITY)
        for (int s = 32 + lane; s < n; s += 32) {
          const float l = lse_accum[static_cast<size_t>(x.s0 + s) * rows + row];
          z += (l == -INFINITY) ? 0.f : expf(l - m);
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const bool empty_row = m == -INFINITY;  // every split empty, no split, or not a row
      const float inv_z = empty_row ? 0.f : 1.f / z;
      float4 acc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c0 = 0; ok && c0 < n; c0 += 32) {
        const int cnt = min(32, n - c0);
        float l = c0 == 0 ? l0 : -INFINITY;
        if (c0 > 0 && live && lane < cnt) l = lse_accum[static_cast<size_t>(x.s0 + c0 + lane) * rows + row];
        const float wl = (empty_row || l == -INFINITY) ? 0.f : expf(l - m) * inv_z;
        for (int i = 0; i < cnt; ++i, ++j) {
          const uint32_t st = j % kCsStages;
          if (!warp_all_wait(&full[st], (j / kCsStages) & 1, abort_flag)) {
            if (lane == 0) {
              report(status, MLA_ERR_TIMEOUT);
              *abort_flag = 1;
            }
            ok = false;
            break;
          }
          const float wj = __shfl_sync(0xffffffffu, wl, i);
          if (live) {
            const float4* src = reinterpret_cast<const float4*>(cs_smem + st * kCsChunkBytes + w * (kDv * 4)) + lane;
#pragma unroll
            for (int q = 0; q < 4; ++q) acc4(acc[q], wj, src[32 * q]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
      }
      if (!ok || !live) continue;
      const size_t orow = static_cast<size_t>(x.u) * rows + row;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        store_row4(out, out_type, orow * kDv + lane * 4 + 128 * q, acc[q].x, acc[q].y, acc[q].z, acc[q].w);
      if (lane == 0) lse[orow] = empty_row ? -INFINITY : m + logf(z);
    }
  }
  __syncthreads();
  // after a timeout: copies still in flight land before the block's shared memory is released
  if (threadIdx.x == 0 && *abort_flag) {
    const int nj = *issued;
    for (int j = max(0, nj - kCsStages); j < nj; ++j)
      mbar_wait(&full[j % kCsStages], (j / kCsStages) & 1, nullptr);
  }
}

const void* combine_stream_kernel_ptr() { return reinterpret_cast<const void*>(combine_stream_kernel); }
int combine_stream_smem_bytes() { return kCsSmemBytes; }

cudaError_t launch_combine(const float* o_accum, const float* lse_accum, const int32_t* split_offset, int n_units,
                           int rows, int num_parts, void* out, int out_type, float* lse, int32_t* status, int sms,
                           cudaStream_t stream) {
  // whole-row warps once there are rows enough to fill the GPU several times
  // over; else split-parallel blocks when the units average 8 or more splits
  // (long context); else the streaming kernel, one block per SM
  const bool whole_rows = static_cast<long long>(n_units) * rows >= 8192;
  const bool split_par = !whole_rows && num_parts >= 8 * n_units;
  const bool stream_k = !whole_rows && !split_par;
  const int items = n_units * ceil_div_i(rows, kCsRows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = whole_rows ? dim3(ceil_div_i(rows, kCombineWarps), n_units, 1)
                : split_par ? dim3(4 * rows, n_units, 1)
                            : dim3(std::min(items, std::max(sms, 1)), 1, 1);
  cfg.blockDim = dim3((whole_rows ? kCombineWarps : split_par ? kSubsets : kCsWarps + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = stream_k ? kCsSmemBytes : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (whole_rows)
    return cudaLaunchKernelEx(&cfg, combine_rows_kernel, o_accum, lse_accum, split_offset, rows, out, out_type, lse);
  if (split_par)
    return cudaLaunchKernelEx(&cfg, combine_split_kernel, o_accum, lse_accum, split_offset, rows, out, out_type, lse);
  return cudaLaunchKernelEx(&cfg, combine_stream_kernel, o_accum, lse_accum, split_offset, n_units, rows, out,
                            out_type, lse, status);
}

}  // namespace mla
