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

constexpr int kSchedMaxSmemUnits = 8192;

__global__ void __launch_bounds__(256) sched_kernel(const int32_t* __restrict__ lengths, int default_length,
                                                     int n_units, int num_parts, int fixed_cost,
                                                     int32_t* __restrict__ sched, int32_t* __restrict__ split_offset) {
  __shared__ int s_nt[kSchedMaxSmemUnits];
  __shared__ long long s_total;
  const bool in_smem = n_units <= kSchedMaxSmemUnits;
  if (threadIdx.x == 0) s_total = 0;
  __syncthreads();
  long long part = 0;
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    const int len = lengths != nullptr ? lengths[u] : default_length;
    const int nt = num_tiles(len);
    if (in_smem) s_nt[u] = nt;
    if (nt > 0) part += nt + fixed_cost;
  }
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), static_cast<unsigned long long>(part));
  __syncthreads();
  if (threadIdx.x != 0) return;

  auto nt_of = [&](int u) -> int {
    if (in_smem) return s_nt[u];
    const int len = lengths != nullptr ? lengths[u] : default_length;
    return num_tiles(len);
  };
  const long long total = s_total;
  const long long cap = total > 0 ? (total + num_parts - 1) / num_parts + fixed_cost : 0;
  // split_offset doubles as the per-unit "touched" counter until the final scan
  for (int u = 0; u <= n_units; ++u) split_offset[u] = 0;
  int b = 0, t = 0;
  for (int p = 0; p < num_parts; ++p) {
    while (b < n_units && nt_of(b) == 0) {
      ++b;
      t = 0;
    }
    const int begin_b = b, begin_t = t;
    const int begin_split = b < n_units ? split_offset[b] : 0;
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
        if (nt_of(bb) > 0) split_offset[bb] += 1;
    }
    int32_t* e = sched + p * MLA_SCHED_INTS;
    e[0] = begin_b;
    e[1] = begin_t;
    e[2] = end_b;
    e[3] = end_t;
    e[4] = begin_split;
    e[5] = 0;
    e[6] = 0;
    e[7] = 0;
  }
  int run = 0;
  for (int u = 0; u < n_units; ++u) {
    const int c = split_offset[u];
    split_offset[u] = run;
    run += c;
  }
  split_offset[n_units] = run;
}

cudaError_t launch_sched(const int32_t* lengths, int default_length, int n_units, int num_parts,
                         int32_t* sched, int32_t* split_offset, cudaStream_t stream) {
  sched_kernel<<<1, 256, 0, stream>>>(lengths, default_length, n_units, num_parts, MLA_SPLIT_FIXED_COST, sched,
                                      split_offset);
  return cudaGetLastError();
}

}  // namespace mla
