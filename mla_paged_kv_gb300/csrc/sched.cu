// Split-KV scheduler kernel.
//
// FlashMLA PR #183 ("Add SM80 (Ampere/A100) dense MLA decode kernel",
// section "How the occupancy work went") computes the partition of the KV
// work on the device from the sequence lengths, once per batch, and sizes
// the number of partitions by the CTAs that fit; every extra partition costs
// a Q reload, a prologue/epilogue and a combine row.  This kernel implements
// this library's plan (documented in include/mla_paged_kv.h):
//   cost(unit) = tiles(unit) + F,  c0 = ceil(sum cost / P),
// partitions take consecutive (unit, tile) ranges within their cap, the last
// partition takes what is left; cap is the smallest value in c0 .. c0 + F
// whose walk leaves the last partition at most cap (c0 + F if none does, or
// for more than kSchedMaxSmemUnits units or kSchedSearchParts partitions).  c0 + F alone often finishes the
// walk early and leaves the last partitions without work.
//
// One block.  The tile counts and the total cost come from all threads; each
// candidate cap's greedy walk is sequential (one thread per candidate, one
// step per unit with a closed form for the partitions a unit spans, shared
// memory only); the metadata is then filled in parallel from the chosen
// walk's partition ends, the per-unit split counts come from a difference
// array, and both prefix sums (counts, then split offsets) are block-wide
// scans.
#include "common.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kSchedThreads = 256;
constexpr int kSchedMaxSmemUnits = 4096;
constexpr int kSchedSearchParts = 128;  // partitions the cap search handles (more: no search)
constexpr int kSchedSearchCaps = MLA_SPLIT_FIXED_COST + 1;  // candidate caps c0 .. c0 + F, one warp each
static_assert(kSchedSearchCaps <= kSchedThreads / 32, "one warp per candidate cap");

// Shared memory of the cap search: each candidate's partition ends, the
// chosen one's begins and last units, and each candidate's leftover cost.
struct SchedSearch {
  int2 end[kSchedSearchCaps * kSchedSearchParts];
  int2 begin[kSchedSearchParts];
  int last[kSchedSearchParts];
  long long left[kSchedSearchCaps];
};

// Exclusive scan of one int per thread over the block; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSchedThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSchedThreads / 32) s_warp[lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  const int base = warp > 0 ? s_warp[warp - 1] : 0;
  *total = s_warp[kSchedThreads / 32 - 1];
  __syncthreads();
  return base + x - v;
}

// The greedy walk over the partitions (one thread).  NtOf is the tile count
// of a unit (shared-memory array or a functor), Int the budget arithmetic
// (32-bit when every budget fits).  Writes the partition table and the
// difference array of the per-unit split counts.
template <typename Int, typename NtOf>
__device__ __forceinline__ void sched_walk(NtOf nt_of, int* diff, int n_units, int num_parts, int fixed_cost,
                                           Int cap, int32_t* sched) {
  int b = 0, t = 0;
  // the last unit touched by an earlier partition, and by how many of them
  int touch_unit = -1, touch_count = 0;
  for (int p = 0; p < num_parts; ++p) {
    while (b < n_units && nt_of[b] == 0) {
      ++b;
      t = 0;
    }
    const int begin_b = b, begin_t = t;
    const int begin_split = (b < n_units && b == touch_unit) ? touch_count : 0;
    if (p == num_parts - 1) {
      b = n_units;
      t = 0;
    } else {
      Int budget = cap;
      while (b < n_units) {
        const int nt = nt_of[b];
        if (nt == 0) {
          ++b;
          t = 0;
          continue;
        }
        const Int rem = static_cast<Int>(nt - t);
        if (rem + fixed_cost <= budget) {
          budget -= rem + fixed_cost;
          ++b;
          t = 0;
        } else {
          const Int take = budget - fixed_cost;
          if (take > 0) t += static_cast<int>(take);
          break;
        }
      }
    }
    const int end_b = b, end_t = t;
    if (begin_b != end_b || begin_t != end_t) {
      const int last = min(end_t > 0 ? end_b : end_b - 1, n_units - 1);
      diff[begin_b] += 1;
      diff[last + 1] -= 1;
      touch_count = (last == begin_b) ? begin_split + 1 : 1;
      touch_unit = last;
    }
    int4* e = reinterpret_cast<int4*>(sched + p * MLA_SCHED_INTS);
    e[0] = make_int4(begin_b, begin_t, end_b, end_t);
    e[1] = make_int4(begin_split, 0, 0, 0);
  }
}

// The greedy walk with budget cap, recording where each partition ends,
// (unit, tile), in end[p].  The same partitions as sched_walk, reached one
// unit at a time instead of one partition at a time: a unit that fits the
// budget left is taken whole; otherwise the current partition takes
// budget - F of its tiles (none if that is not positive) and ends, the
// following partitions take full chunks of w = cap - F tiles while the rest
// does not fit with its F, and the rest opens the next partition with
// cap - rest - F left.  Partitions that never end inside a unit end past the
// last one.  The last partition takes everything left; returns its cost.
// One warp, every lane running the same walk (lane 0 stores): the tile counts
// come 32 at a time, one per lane, by shuffle.  Each step is selects on the
// budget and the partition index (a branch per step stalled the warp ~400
// cycles a unit); the chunk count is a division by the constant w done as a
// 64-bit multiply and one correction.  Once the last partition is reached the
// rest of the units' cost is a warp sum.
__device__ __forceinline__ long long sched_walk_record(const int* nt_of, int n_units, int num_parts, int fixed_cost,
                                                       int cap, int2* end) {
  const int lane = threadIdx.x & 31;
  const int last_p = num_parts - 1;
  const int w = cap - fixed_cost;  // tiles a partition takes from a unit it starts on and cannot finish
  const int wc = max(w, 0);
  const unsigned long long inv_w = w > 0 ? (1ull << 32) / static_cast<unsigned long long>(w) + 1ull : 0ull;
  int p = 0, budget = cap;
  int u_stop = n_units;  // the unit in which the last partition begins (its rest is in `left`)
  long long left = 0;
  for (int base = 0; base < n_units && p < last_p; base += 32) {
    const int mine = base + lane < n_units ? nt_of[base + lane] : 0;
    const int cnt = min(32, n_units - base);
    for (int j = 0; j < cnt && p < last_p; ++j) {
      const int x = __shfl_sync(0xffffffffu, mine, j);
      const bool fits = x + fixed_cost <= budget;
      const int t = max(budget - fixed_cost, 0);
      const int r = x - t;  // >= 1 when the unit does not fit
      // full chunks while the rest does not fit: (r - 1) / w (w > 0), else every partition
      const unsigned int n1 = static_cast<unsigned int>(max(r - 1, 0));
      int q = static_cast<int>((static_cast<unsigned long long>(n1) * inv_w) >> 32);
      q -= (static_cast<long long>(q) * w > n1) ? 1 : 0;
      q += (static_cast<long long>(q + 1) * w <= n1) ? 1 : 0;
      const int k = (r + fixed_cost > cap) ? (w > 0 ? q : last_p) : 0;
      const int kk = min(k, last_p - p - 1);  // chunk partitions before the last one
      const bool split = !fits && x > 0;
      if (split && lane == 0) {
        end[p] = make_int2(base + j, t);
        for (int i = 1; i <= kk; ++i) end[p + i] = make_int2(base + j, t + i * wc);
      }
      const int rem = r - kk * wc;
      const int p_new = split ? p + 1 + kk : p;
      if (split && p_new == last_p) {
        left = rem + fixed_cost;
        u_stop = base + j;
      }
      budget = split ? cap - rem - fixed_cost : (x > 0 ? budget - x - fixed_cost : budget);
      p = p_new;
    }
  }
  if (p == last_p && u_stop == n_units) u_stop = -1;  // one partition: it takes every unit
  // the units after u_stop go to the last partition whole
  long long rest = 0;
  for (int u = u_stop + 1 + lane; u < n_units; u += 32) {
    const int x = nt_of[u];
    if (x > 0) rest += x + fixed_cost;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rest += __shfl_xor_sync(0xffffffffu, rest, o);
  if (lane == 0)
    for (int q2 = p; q2 < num_parts; ++q2) end[q2] = make_int2(n_units, 0);
  return left + rest;
}

// Tile count of unit u straight from the lengths (for the many-units path).
struct NtFromLengths {
  const int32_t* lengths;
  int default_length;
  __device__ __forceinline__ int operator[](int u) const {
    return num_tiles(lengths != nullptr ? lengths[u] : default_length);
  }
};

// The native plan (see the file comment); n_units <= kSchedMaxSmemUnits keeps
// the tile counts and the split-count difference array in shared memory.
__device__ void plan_native(const int32_t* __restrict__ lengths, int default_length, int n_units, int num_parts,
                            int fixed_cost, int32_t* __restrict__ sched, int32_t* __restrict__ split_offset,
                            int* s_nt, int* s_diff, long long* s_warp_cost, int* s_warp, SchedSearch* s) {
  const bool in_smem = n_units <= kSchedMaxSmemUnits;
  // difference array of the per-unit split counts: shared memory, or the
  // output array itself when there are too many units
  int* diff = in_smem ? s_diff : reinterpret_cast<int*>(split_offset);
  const NtFromLengths nt_of{lengths, default_length};

  long long part = 0;
  for (int u = threadIdx.x; u < n_units; u += kSchedThreads) {
    const int nt = num_tiles(lengths != nullptr ? lengths[u] : default_length);
    if (in_smem) s_nt[u] = nt;
    diff[u] = 0;
    if (nt > 0) part += nt + fixed_cost;
  }
  if (threadIdx.x == 0) diff[n_units] = 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((threadIdx.x & 31) == 0) s_warp_cost[threadIdx.x >> 5] = part;
  __syncthreads();

  long long total_cost = 0;
  for (int w = 0; w < kSchedThreads / 32; ++w) total_cost += s_warp_cost[w];
  const long long c0 = total_cost > 0 ? (total_cost + num_parts - 1) / num_parts : 0;
  // Cap search: candidate caps c0 .. c0 + F walk at once, one per warp, each
  // recording its partition bounds; the smallest cap that leaves the last
  // partition at most itself wins (else c0 + F), and the metadata is then
  // filled in parallel from its bounds.  Needs the tile counts in shared
  // memory, at most kSchedSearchParts partitions and F <= MLA_SPLIT_FIXED_COST.
  const bool search = in_smem && total_cost > 0 && c0 + fixed_cost < (1LL << 30) && num_parts <= kSchedSearchParts &&
                      fixed_cost + 1 <= kSchedSearchCaps;
  if (!search) {
    if (threadIdx.x == 0) {
      const long long cap = total_cost > 0 ? c0 + fixed_cost : 0;
      if (in_smem && cap < (1LL << 30))
        sched_walk<int, int*>(s_nt, s_diff, n_units, num_parts, fixed_cost, static_cast<int>(cap), sched);
      else
        sched_walk<long long>(nt_of, diff, n_units, num_parts, fixed_cost, cap, sched);
    }
    __syncthreads();
  } else {
    const int warp = threadIdx.x >> 5;
    if (warp <= fixed_cost) {
      const long long left = sched_walk_record(s_nt, n_units, num_parts, fixed_cost, static_cast<int>(c0) + warp,
                                               s->end + warp * kSchedSearchParts);
      if ((threadIdx.x & 31) == 0) s->left[warp] = left;
    }
    __syncthreads();
    int w = fixed_cost;
    for (int k = 0; k < fixed_cost; ++k)
      if (s->left[k] <= c0 + k) {
        w = k;
        break;
      }
    const int2* end = s->end + w * kSchedSearchParts;
    // each partition's begin and last unit (-1 when it is empty)
    for (int p = threadIdx.x; p < num_parts; p += kSchedThreads) {
      int b = p == 0 ? 0 : end[p - 1].x, t = p == 0 ? 0 : end[p - 1].y;
      while (b < n_units && s_nt[b] == 0) {
        ++b;
        t = 0;
      }
      const int2 e = end[p];
      s->begin[p] = make_int2(b, t);
      s->last[p] = (b == e.x && t == e.y) ? -1 : min(e.y > 0 ? e.x : e.x - 1, n_units - 1);
    }
    __syncthreads();
    for (int p = threadIdx.x; p < num_parts; p += kSchedThreads) {
      const int2 bg = s->begin[p], e = end[p];
      // earlier non-empty partitions ending in this one's first unit
      int begin_split = 0;
      if (bg.x < n_units)
        for (int q = 0; q < p; ++q) begin_split += s->last[q] == bg.x;
      int4* out = reinterpret_cast<int4*>(sched + p * MLA_SCHED_INTS);
      out[0] = make_int4(bg.x, bg.y, e.x, e.y);
      out[1] = make_int4(begin_split, 0, 0, 0);
      if (s->last[p] >= 0) {
        atomicAdd(&diff[bg.x], 1);
        atomicAdd(&diff[s->last[p] + 1], -1);
      }
    }
    __syncthreads();
  }

  // each thread scans a contiguous chunk of units
  const int chunk = (n_units + kSchedThreads - 1) / kSchedThreads;
  const int u0 = min(static_cast<int>(threadIdx.x) * chunk, n_units);
  const int u1 = min(u0 + chunk, n_units);
  int total = 0;
  // pass 1: split count of unit u = (prefix sum of diff)[u], for units with tiles
  int local = 0;
  for (int u = u0; u < u1; ++u) local += diff[u];
  int run = block_exclusive_scan(local, s_warp, &total);
  int csum = 0;
  for (int u = u0; u < u1; ++u) {
    run += diff[u];
    const int count = (in_smem ? s_nt[u] : nt_of[u]) > 0 ? run : 0;
    diff[u] = count;
    csum += count;
  }
  __syncthreads();
  // pass 2: split_offset = exclusive prefix sum of the counts
  int off = block_exclusive_scan(csum, s_warp, &total);
  for (int u = u0; u < u1; ++u) {
    const int count = diff[u];
    split_offset[u] = off;
    off += count;
  }
  if (threadIdx.x == 0) split_offset[n_units] = total;
}

__global__ void __launch_bounds__(kSchedThreads) sched_kernel(const int32_t* __restrict__ lengths,
                                                               int default_length, int n_units, int num_parts,
                                                               int fixed_cost, int32_t* __restrict__ sched,
                                                               int32_t* __restrict__ split_offset) {
  __shared__ int s_nt[kSchedMaxSmemUnits];
  __shared__ int s_diff[kSchedMaxSmemUnits + 1];
  __shared__ long long s_warp_cost[kSchedThreads / 32];
  __shared__ int s_warp[kSchedThreads / 32];
  __shared__ SchedSearch s_search;
  pdl_wait_prior_grid();  // launched early (programmatic dependent launch): the lengths may come from the grid before
  plan_native(lengths, default_length, n_units, num_parts, fixed_cost, sched, split_offset, s_nt, s_diff,
              s_warp_cost, s_warp, &s_search);
}

// Request-local plan (FlashMLA PR #200, section "Scheduler policy", names a
// request-local scheduler for its H=64 path without defining it; this is the
// library's reading): no part spans two units.  Each unit with tiles gets one
// part; the other parts go out in proportion to the tile counts, by largest
// remainder (ties to the lower unit); a unit gets at most one part per tile;
// unit b's k-th of s parts covers tiles [k*n/s, (k+1)*n/s).  Parts are in unit
// order, unused ones empty.  With no tiles, more units with tiles than parts,
// or more than kSchedLocalMaxUnits units, the native plan is used.
constexpr int kSchedLocalMaxUnits = 1024;

__global__ void __launch_bounds__(kSchedThreads) sched_local_kernel(const int32_t* __restrict__ lengths,
                                                                     int default_length, int n_units, int num_parts,
                                                                     int fixed_cost, int32_t* __restrict__ sched,
                                                                     int32_t* __restrict__ split_offset) {
  __shared__ int s_nt[kSchedMaxSmemUnits];
  __shared__ int s_diff[kSchedMaxSmemUnits + 1];
  __shared__ long long s_warp_cost[kSchedThreads / 32];
  __shared__ int s_warp[kSchedThreads / 32];
  __shared__ long long s_rem[kSchedLocalMaxUnits];
  __shared__ long long s_sum[2];  // total tiles, parts given by the quotas
  __shared__ int s_active;
  __shared__ SchedSearch s_search;
  pdl_wait_prior_grid();  // launched early (programmatic dependent launch): the lengths may come from the grid before
  if (n_units <= kSchedLocalMaxUnits) {
    long long tiles = 0;
    int act = 0;
    for (int u = threadIdx.x; u < n_units; u += kSchedThreads) {
      const int nt = num_tiles(lengths != nullptr ? lengths[u] : default_length);
      s_nt[u] = nt;
      tiles += nt;
      act += nt > 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
      act += __shfl_xor_sync(0xffffffffu, act, o);
    }
    if ((threadIdx.x & 31) == 0) {
      s_warp_cost[threadIdx.x >> 5] = tiles;
      s_warp[threadIdx.x >> 5] = act;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      long long t = 0;
      int a = 0;
      for (int w = 0; w < kSchedThreads / 32; ++w) {
        t += s_warp_cost[w];
        a += s_warp[w];
      }
      s_sum[0] = t;
      s_active = a;
    }
    __syncthreads();
  }
  const int active = n_units <= kSchedLocalMaxUnits ? s_active : 0;
  if (active == 0 || active > num_parts) {
    __syncthreads();
    plan_native(lengths, default_length, n_units, num_parts, fixed_cost, sched, split_offset, s_nt, s_diff,
                s_warp_cost, s_warp, &s_search);
    return;
  }
  const long long total = s_sum[0];
  const long long spare = num_parts - active;
  // quotas: one part each, plus floor(n * spare / total); remainders kept for the ranking
  long long given = 0;
  for (int u = threadIdx.x; u < n_units; u += kSchedThreads) {
    const long long x = static_cast<long long>(s_nt[u]) * spare;
    const long long q = s_nt[u] > 0 ? x / total : 0;
    s_diff[u] = s_nt[u] > 0 ? 1 + static_cast<int>(q) : 0;
    s_rem[u] = s_nt[u] > 0 ? x - q * total : -1;
    given += q;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) given += __shfl_xor_sync(0xffffffffu, given, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_warp_cost[threadIdx.x >> 5] = given;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long g = 0;
    for (int w = 0; w < kSchedThreads / 32; ++w) g += s_warp_cost[w];
    s_sum[1] = g;
  }
  __syncthreads();
  const long long extra = spare - s_sum[1];
  // the `extra` largest remainders (ties: lower unit) get one more part
  for (int u = threadIdx.x; u < n_units; u += kSchedThreads) {
    if (s_nt[u] == 0) continue;
    const long long r = s_rem[u];
    int rank = 0;
    for (int v = 0; v < n_units; ++v) rank += (s_rem[v] > r) || (s_rem[v] == r && v < u);
    int seats = s_diff[u] + (rank < extra ? 1 : 0);
    s_diff[u] = min(seats, s_nt[u]);
  }
  __syncthreads();
  // split offsets = exclusive prefix sum of the part counts (contiguous chunk per thread)
  const int chunk = (n_units + kSchedThreads - 1) / kSchedThreads;
  const int u0 = min(static_cast<int>(threadIdx.x) * chunk, n_units);
  const int u1 = min(u0 + chunk, n_units);
  int csum = 0;
  for (int u = u0; u < u1; ++u) csum += s_diff[u];
  int used = 0;
  int off = block_exclusive_scan(csum, s_warp, &used);
  for (int u = u0; u < u1; ++u) {
    split_offset[u] = off;
    const int n = s_nt[u], parts = s_diff[u];
    for (int k = 0; k < parts; ++k) {
      const int lo = static_cast<int>(static_cast<long long>(k) * n / parts);
      const int hi = static_cast<int>(static_cast<long long>(k + 1) * n / parts);
      int4* e = reinterpret_cast<int4*>(sched + (off + k) * MLA_SCHED_INTS);
      e[0] = hi < n ? make_int4(u, lo, u, hi) : make_int4(u, lo, u + 1, 0);
      e[1] = make_int4(k, 0, 0, 0);
    }
    off += parts;
  }
  if (threadIdx.x == 0) split_offset[n_units] = used;
  for (int p = used + static_cast<int>(threadIdx.x); p < num_parts; p += kSchedThreads) {
    int4* e = reinterpret_cast<int4*>(sched + p * MLA_SCHED_INTS);
    e[0] = make_int4(n_units, 0, n_units, 0);
    e[1] = make_int4(0, 0, 0, 0);
  }
}

cudaError_t launch_sched(const int32_t* lengths, int default_length, int n_units, int num_parts,
                         int32_t* sched, int32_t* split_offset, int request_local, cudaStream_t stream) {
  // A programmatic dependent of whatever runs before it on the stream: the
  // block starts while that grid drains and waits for it on the device
  // (griddepcontrol.wait) before it reads the lengths.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kSchedThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (request_local)
    return cudaLaunchKernelEx(&cfg, sched_local_kernel, lengths, default_length, n_units, num_parts,
                              static_cast<int>(MLA_SPLIT_FIXED_COST), sched, split_offset);
  return cudaLaunchKernelEx(&cfg, sched_kernel, lengths, default_length, n_units, num_parts,
                            static_cast<int>(MLA_SPLIT_FIXED_COST), sched, split_offset);
}

}  // namespace mla
