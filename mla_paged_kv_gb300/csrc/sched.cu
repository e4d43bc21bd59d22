// Split-KV scheduler kernel.
//
// FlashMLA PR #183 ("Add SM80 (Ampere/A100) dense MLA decode kernel",
// section "How the occupancy work went") computes the partition of the KV
// work on the device from the sequence lengths, once per batch, and sizes
// the number of partitions by the CTAs that fit; every extra partition costs
// a Q reload, a prologue/epilogue and a combine row.  This kernel implements
// this library's plan (documented in include/mla_paged_kv.h):
//   cost(unit) = tiles(unit) + F,  cap = ceil(sum cost / P) + F,
// partitions take consecutive (unit, tile) ranges within their cap, the last
// partition takes what is left.  The walk is inherently sequential and tiny
// (n_units + num_parts steps), so one thread runs it; a block of threads
// first turns the lengths into tile counts in shared memory when they fit.
#include "common.cuh"

namespace mla {

constexpr int kSchedMaxSmemUnits = 4096;

__global__ void __launch_bounds__(256) sched_kernel(const int32_t* __restrict__ lengths, int default_length,
                                                     int n_units, int num_parts, int fixed_cost,
                                                     int32_t* __restrict__ sched, int32_t* __restrict__ split_offset) {
  // tile counts and per-unit split counters live in shared memory when they
  // fit, so the sequential walk below touches no global memory
  __shared__ int s_nt[kSchedMaxSmemUnits];
  __shared__ int s_touch[kSchedMaxSmemUnits];
  __shared__ long long s_total;
  const bool in_smem = n_units <= kSchedMaxSmemUnits;
  if (threadIdx.x == 0) s_total = 0;
  __syncthreads();
  long long part = 0;
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    const int len = lengths != nullptr ? lengths[u] : default_length;
    const int nt = num_tiles(len);
    if (in_smem) {
      s_nt[u] = nt;
      s_touch[u] = 0;
    } else {
      split_offset[u] = 0;
    }
    if (nt > 0) part += nt + fixed_cost;
  }
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), static_cast<unsigned long long>(part));
  __syncthreads();
  if (threadIdx.x == 0) {
    auto nt_of = [&](int u) -> int {
      if (in_smem) return s_nt[u];
      const int len = lengths != nullptr ? lengths[u] : default_length;
      return num_tiles(len);
    };
    // per-unit "touched" counter: shared memory, or split_offset itself when too many units
    int* touch = in_smem ? s_touch : reinterpret_cast<int*>(split_offset);
    const long long total = s_total;
    const long long cap = total > 0 ? (total + num_parts - 1) / num_parts + fixed_cost : 0;
    int b = 0, t = 0;
    for (int p = 0; p < num_parts; ++p) {
      while (b < n_units && nt_of(b) == 0) {
        ++b;
        t = 0;
      }
      const int begin_b = b, begin_t = t;
      const int begin_split = b < n_units ? touch[b] : 0;
      if (p == num_parts - 1) {
        b = n_units;
        t = 0;
      } else {
        long long budget = cap;
        while (b < n_units) {
          const int nt = nt_of(b);
          if (nt == 0) {
            ++b;
            t = 0;
            continue;
          }
          const long long rem = nt - t;
          if (rem + fixed_cost <= budget) {
            budget -= rem + fixed_cost;
            ++b;
            t = 0;
          } else {
            const long long take = budget - fixed_cost;
            if (take > 0) t += static_cast<int>(take);
            break;
          }
        }
      }
      const int end_b = b, end_t = t;
      if (begin_b != end_b || begin_t != end_t) {
        const int last = end_t > 0 ? end_b : end_b - 1;
        for (int bb = begin_b; bb <= last && bb < n_units; ++bb)
          if (nt_of(bb) > 0) touch[bb] += 1;
      }
      int4* e = reinterpret_cast<int4*>(sched + p * MLA_SCHED_INTS);
      e[0] = make_int4(begin_b, begin_t, end_b, end_t);
      e[1] = make_int4(begin_split, 0, 0, 0);
    }
    if (in_smem) {
      for (int u = 0; u < n_units; ++u) split_offset[u] = s_touch[u];
    }
  }
  __syncthreads();
  // exclusive prefix sum of the counts (one warp; n_units is small)
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base < n_units; base += 32) {
      const int u = base + threadIdx.x;
      const int c = u < n_units ? (in_smem ? s_touch[u] : split_offset[u]) : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (threadIdx.x >= o) x += y;
      }
      __syncwarp();
      if (u < n_units) split_offset[u] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
      __syncwarp();
    }
    if (threadIdx.x == 0) split_offset[n_units] = carry;
  }
}

cudaError_t launch_sched(const int32_t* lengths, int default_length, int n_units, int num_parts,
                         int32_t* sched, int32_t* split_offset, cudaStream_t stream) {
  sched_kernel<<<1, 256, 0, stream>>>(lengths, default_length, n_units, num_parts, MLA_SPLIT_FIXED_COST, sched,
                                      split_offset);
  return cudaGetLastError();
}

}  // namespace mla
