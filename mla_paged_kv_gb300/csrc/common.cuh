// Shared definitions of the MLA decode kernels (device side).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mla_paged_kv.h"

namespace mla {

constexpr int kTile = MLA_PAGE_SIZE;        // keys per pipeline tile = one page
constexpr int kRowsPerBlock = MLA_ROWS_PER_BLOCK;
constexpr int kDqk = MLA_D_QK;
constexpr int kDv = MLA_D_V;

// First error wins; later ones are dropped so the caller sees the root cause.
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

__host__ __device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int num_tiles(int len) { return len > 0 ? ceil_div_i(len, kTile) : 0; }

// Everything the split-KV attention kernels read besides the tensor maps.
struct DecodeParams {
  // keys per unit (dense: cache_seqlens, sparse: topk_length or NULL)
  const int32_t* lengths;
  int default_length;       // used when lengths == NULL
  int n_units;              // dense: batch; sparse: batch * s_q
  int rows;                 // query rows per unit (dense s_q*h_q, sparse h_q)
  int row_blocks;           // CTA pairs per partition: h_kv * blocks_per_group
  int h_q;
  // dense: latent KV heads.  Query head h reads KV head h / group_heads.  With
  // h_kv = 1 a row block is 128 consecutive rows (token-major) of the unit;
  // with h_kv > 1 it is block_tokens whole tokens of one head group.
  int h_kv;
  int group_heads;          // h_q / h_kv
  int block_tokens;         // h_kv > 1: tokens per row block (group_heads * block_tokens <= 128)
  int blocks_per_group;     // row blocks per head group
  int s_q;                  // query tokens per request (causal alignment)
  int causal;
  float scale_log2;         // softmax_scale * log2(e)
  // dense
  int q_vring;              // host: 1 selects the kernel instance that stages the first unit's Q in the V ring
  const int32_t* block_table;
  int max_pages;
  int num_pages;
  // sparse
  const int32_t* indices;   // [n_units, topk] (native selection), or NULL when packed
  int topk;
  const uint8_t* kv8;       // [num_pages, 64, 656]; packed: the packed records
  const uint64_t* packed_mask;  // packed: [n_units, ceil(topk/64)] valid-slot bits, else NULL
  // sparse kernel over a dense FP8 cache (block_table set): unit b reads
  // block-table row b / unit_request_div (s_q when a unit is one query token
  // of a request, 1 when it is the whole request)
  int unit_request_div;
  // schedule
  const int32_t* sched;
  const int32_t* split_offset;
  int num_parts;
  // outputs
  float* o_accum;           // [slots, rows, 512]
  float* lse_accum;         // [slots, rows]
  void* out;                // [n_units, rows, 512]
  int out_type;             // MLA_DTYPE_BF16, MLA_DTYPE_FP32 or MLA_DTYPE_FP16
  float* lse;               // [n_units, rows]
  int32_t* status;
};

}  // namespace mla
