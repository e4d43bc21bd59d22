// LSE-weighted combine of split-KV partials.
//
// FlashMLA PR #183 (Summary; "Modifications outside csrc/sm80/") merges the
// per-split partial outputs with a combine kernel and bounds the split count
// by a compile-time ladder.  Here the split count is a runtime loop bound, so
// any number of splits is merged.  Per output row:
//   m = max_s lse_s,  w_s = exp(lse_s - m),  Z = sum_s w_s,
//   out = sum_s (w_s / Z) O_s,  lse = m + ln Z
// with -inf splits weighing 0 and an all-empty row giving out 0, lse -inf.
// Memory bound: every partial is read once with 512-byte coalesced rows.
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

// kVec = float4 per lane per split: 4 -> a warp covers a whole 512-column
// row (a block = 4 rows), used when there are rows enough to fill the GPU
// several times over; 1 -> a warp covers a 128-column quarter (a block = 1
// row), 4x the warps for fewer rows.  Few rows with many splits per unit
// (long context) go to combine_split_kernel instead.
// Latency: split_offset comes from the plan (complete before the attention
// grid started), so it is read before waiting for that grid.  After the wait
// the split LSEs are loaded with the lanes spread over the splits, and in the
// same round trip the partial rows of the first kPre splits: kBatch for
// quarter-row warps (kVec = 1), 2 for whole-row warps (the count most units
// have when partitions slightly outnumber requests; a batch of 4 is 16 float4
// a lane, and its registers cost more occupancy than the round trip saves).
template <int kVec>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const float* __restrict__ o_accum, const float* __restrict__ lse_accum,
                   const int32_t* __restrict__ split_offset, int rows, void* __restrict__ out, int out_type,
                   float* __restrict__ lse) {
  constexpr int kBatch = kVec == 4 ? 4 : 8;
  constexpr int kPre = kVec == 1 ? kBatch : 2;  // partial rows loaded with the LSEs
  const int unit = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = kVec == 4 ? blockIdx.x * kCombineWarps + warp : blockIdx.x;
  if (row >= rows) return;
  const int s0 = split_offset[unit];
  const int n = split_offset[unit + 1] - s0;
  if (n == 1) return;  // written directly by the attention kernel
  pdl_wait_prior_grid();
  const size_t orow = static_cast<size_t>(unit) * rows + row;
  const size_t col = (kVec == 4 ? 0 : static_cast<size_t>(warp) * 128) + lane * 4;
  const bool writes_lse = kVec == 4 ? lane == 0 : (warp == 0 && lane == 0);
  const size_t split_stride = static_cast<size_t>(rows) * kDv / 4;  // float4 between consecutive splits
  const float4* src0 = reinterpret_cast<const float4*>(o_accum + (static_cast<size_t>(s0) * rows + row) * kDv + col);

  // the first 32 LSEs (and the first kPre splits' rows), all in flight at once
  const float l0 = lane < n ? lse_accum[static_cast<size_t>(s0 + lane) * rows + row] : -INFINITY;
  const int first = min(n, kPre);
  float4 v0[kPre > 0 ? kPre : 1][kVec];
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

cudaError_t launch_combine(const float* o_accum, const float* lse_accum, const int32_t* split_offset, int n_units,
                           int rows, int num_parts, void* out, int out_type, float* lse, cudaStream_t stream) {
  // whole-row warps once there are enough rows to fill the GPU several times
  // over; else split-parallel blocks when the units average 8 or more splits
  const bool whole_rows = static_cast<long long>(n_units) * rows >= 8192;
  const bool split_par = !whole_rows && num_parts >= 8 * n_units;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = whole_rows ? dim3(ceil_div_i(rows, kCombineWarps), n_units, 1)
                           : dim3(split_par ? 4 * rows : rows, n_units, 1);
  cfg.blockDim = dim3((split_par ? kSubsets : kCombineWarps) * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (whole_rows)
    return cudaLaunchKernelEx(&cfg, combine_kernel<4>, o_accum, lse_accum, split_offset, rows, out, out_type, lse);
  if (split_par)
    return cudaLaunchKernelEx(&cfg, combine_split_kernel, o_accum, lse_accum, split_offset, rows, out, out_type, lse);
  return cudaLaunchKernelEx(&cfg, combine_kernel<1>, o_accum, lse_accum, split_offset, rows, out, out_type, lse);
}

}  // namespace mla
