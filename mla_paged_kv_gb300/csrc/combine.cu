// LSE-weighted combine of split-KV partials.
//
// FlashMLA PR #183 (Summary; "Modifications outside csrc/sm80/") merges the
// per-split partial outputs with a combine kernel and bounds the split count
// by a compile-time ladder.  Here the split count is a runtime loop bound, so
// any number of splits is merged.  One warp per output row:
//   m = max_s lse_s,  w_s = exp(lse_s - m),  Z = sum_s w_s,
//   out = sum_s (w_s / Z) O_s,  lse = m + ln Z
// with -inf splits weighing 0 and an all-empty row giving out 0, lse -inf.
// Memory bound: every partial is read once with 512-byte coalesced rows.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kCombineWarps = 4;

__device__ __forceinline__ void store_row4(void* out, int out_fp32, size_t elem, float a, float b, float c,
                                           float d) {
  if (out_fp32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + elem) = make_float4(a, b, c, d);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
    __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + elem) = v;
  }
}

__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const float* __restrict__ o_accum, const float* __restrict__ lse_accum,
                   const int32_t* __restrict__ split_offset, int rows, void* __restrict__ out, int out_fp32,
                   float* __restrict__ lse) {
  pdl_wait_prior_grid();
  const int unit = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineWarps + warp;
  if (row >= rows) return;
  const int s0 = split_offset[unit];
  const int n = split_offset[unit + 1] - s0;
  if (n == 1) return;  // written directly by the attention kernel
  const size_t orow = static_cast<size_t>(unit) * rows + row;

  float m = -INFINITY;
  for (int s = lane; s < n; s += 32) m = fmaxf(m, lse_accum[static_cast<size_t>(s0 + s) * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (n == 0 || m == -INFINITY) {
#pragma unroll
    for (int k = 0; k < 4; ++k) store_row4(out, out_fp32, orow * kDv + lane * 4 + 128 * k, 0.f, 0.f, 0.f, 0.f);
    if (lane == 0) lse[orow] = -INFINITY;
    return;
  }
  float z = 0.f;
  for (int s = lane; s < n; s += 32) {
    const float l = lse_accum[static_cast<size_t>(s0 + s) * rows + row];
    z += (l == -INFINITY) ? 0.f : expf(l - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float inv_z = 1.f / z;

  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
  for (int s = 0; s < n; ++s) {
    const size_t slot_row = static_cast<size_t>(s0 + s) * rows + row;
    const float l = lse_accum[slot_row];
    if (l == -INFINITY) continue;
    const float w = expf(l - m) * inv_z;
    const float4* src = reinterpret_cast<const float4*>(o_accum + slot_row * kDv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = src[lane + 32 * k];
      acc[k].x = fmaf(w, v.x, acc[k].x);
      acc[k].y = fmaf(w, v.y, acc[k].y);
      acc[k].z = fmaf(w, v.z, acc[k].z);
      acc[k].w = fmaf(w, v.w, acc[k].w);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    store_row4(out, out_fp32, orow * kDv + lane * 4 + 128 * k, acc[k].x, acc[k].y, acc[k].z, acc[k].w);
  if (lane == 0) lse[orow] = m + logf(z);
}

cudaError_t launch_combine(const float* o_accum, const float* lse_accum, const int32_t* split_offset, int n_units,
                           int rows, void* out, int out_fp32, float* lse, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div_i(rows, kCombineWarps), n_units, 1);
  cfg.blockDim = dim3(kCombineWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, o_accum, lse_accum, split_offset, rows, out, out_fp32, lse);
}

}  // namespace mla
