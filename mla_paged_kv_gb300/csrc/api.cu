// C ABI of the MLA paged-KV decode library: argument checks, tensor maps,
// partition counts and launches.  No device memory is allocated here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_paged_kv.h"
#include "common.cuh"

namespace mla {
cudaError_t launch_sched(const int32_t*, int, int, int, int32_t*, int32_t*, int, cudaStream_t);
cudaError_t launch_combine(const float*, const float*, const int32_t*, int, int, int, void*, int, float*, int32_t*, int,
                           cudaStream_t);
const void* combine_stream_kernel_ptr();
int combine_stream_smem_bytes();
cudaError_t launch_dense(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                         const DecodeParams&, int, int, cudaStream_t);
int dense_smem_bytes();
int dense_threads(int kind);
const void* dense_kernel_ptr(int kind);
cudaError_t launch_sparse(const CUtensorMap&, const DecodeParams&, int, int, cudaStream_t);
int sparse_smem_bytes();
int sparse_threads();
const void* sparse_kernel_ptr(int stall);
cudaError_t launch_unpack(const uint8_t*, int, const int32_t*, int, float*, int32_t*, cudaStream_t);
cudaError_t launch_pack(const uint8_t*, int, const int32_t*, int, const int32_t*, int, uint8_t*, uint64_t*,
                        int32_t*, int, cudaStream_t);
}  // namespace mla

using namespace mla;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int status = MLA_OK;
  int dense_clusters = 0;
  int sparse_clusters = 0;
  int sms = 0;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int max_clusters(const void* kernel, int threads, int smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return -1;
  return n;
}

// Per-device one-time setup: shared-memory opt-in and co-resident cluster counts.
const DeviceInfo& device_info() {
  int dev = 0;
  static DeviceInfo bad;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    bad.status = MLA_ERR_CUDA;
    return bad;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.ready) return d;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    d.status = MLA_ERR_UNSUPPORTED;  // built for sm_103a only
    d.ready = true;
    return d;
  }
  bool attr_ok = true;
  for (int stall = 0; stall < 2; ++stall)
    attr_ok = attr_ok && cudaFuncSetAttribute(sparse_kernel_ptr(stall), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              sparse_smem_bytes()) == cudaSuccess;
  for (int kind = 0; kind < 5; ++kind)
    attr_ok = attr_ok && cudaFuncSetAttribute(dense_kernel_ptr(kind), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              dense_smem_bytes()) == cudaSuccess;
  attr_ok = attr_ok && cudaFuncSetAttribute(combine_stream_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            combine_stream_smem_bytes()) == cudaSuccess;
  if (!attr_ok) {
    cudaGetLastError();
    d.status = MLA_ERR_CUDA;
    d.ready = true;
    return d;
  }
  // the dense plan also sizes the FP8-record calls, which run the sparse kernel
  d.dense_clusters = std::min(max_clusters(dense_kernel_ptr(0), dense_threads(0), dense_smem_bytes()),
                              max_clusters(sparse_kernel_ptr(0), sparse_threads(), sparse_smem_bytes()));
  d.sparse_clusters = max_clusters(sparse_kernel_ptr(0), sparse_threads(), sparse_smem_bytes());
  cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (d.dense_clusters <= 0 || d.sparse_clusters <= 0 || d.sms <= 0) {
    cudaGetLastError();
    d.status = MLA_ERR_CUDA;
  }
  d.ready = true;
  return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WorkspaceLayout {
  size_t o_bytes, lse_off, total;
};

WorkspaceLayout ws_layout(int n_units, int rows, int num_parts) {
  const size_t slots = static_cast<size_t>(n_units) + static_cast<size_t>(num_parts);
  WorkspaceLayout w;
  w.o_bytes = slots * rows * MLA_D_V * sizeof(float);
  w.lse_off = align_up(w.o_bytes, 256);
  w.total = align_up(w.lse_off + slots * rows * sizeof(float), 256);
  return w;
}

int encode_q_map(CUtensorMap* m, const void* q, long long rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return MLA_ERR_CUDA;
  cuuint64_t dims[2] = {MLA_D_QK, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {MLA_D_QK * 2};
  cuuint32_t box[2] = {64, MLA_ROWS_PER_BLOCK};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// Dense KV pool as [num_pages][64][h_kv][576] (16-bit elements), viewed as
// five dims, innermost first: (64 dims of a slice, 64 tokens, 9 slices of 64
// dims, h_kv, num_pages).  One box = `slices` consecutive 64-dim slices of
// the 64 tokens of one page and one KV head; it lands as `slices` 8 KB
// 128-byte-swizzled boxes of 64 tokens x 64 dims one after another, the
// layout the MMA descriptors read, in one TMA instruction (the TMA engine's
// time goes mostly per instruction, so whole slice ranges per instruction
// move several times the bytes per second of one 8 KB box each).
int encode_kv_map(CUtensorMap* m, const void* kv, int num_pages, int h_kv, int slices) {
  auto fn = encode_fn();
  if (fn == nullptr) return MLA_ERR_CUDA;
  const cuuint64_t row = static_cast<cuuint64_t>(MLA_D_QK) * 2;
  cuuint64_t dims[5] = {64, MLA_PAGE_SIZE, MLA_D_QK / 64, static_cast<cuuint64_t>(h_kv),
                        static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[4] = {row * h_kv, 128, row, row * h_kv * MLA_PAGE_SIZE};
  cuuint32_t box[5] = {64, MLA_PAGE_SIZE, static_cast<cuuint32_t>(slices), 1, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(kv), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// Dense Q with h_kv > 1 as [tokens = batch*s_q][h_kv][group_heads][576], dims
// innermost first: (576, group_heads, h_kv, tokens).  One box = 64 dims x
// group_heads heads x block_tokens tokens of one head group.
int encode_q_map_groups(CUtensorMap* m, const void* q, long long tokens, int h_kv, int group_heads,
                        int block_tokens) {
  auto fn = encode_fn();
  if (fn == nullptr) return MLA_ERR_CUDA;
  const cuuint64_t row = static_cast<cuuint64_t>(MLA_D_QK) * 2;
  cuuint64_t dims[4] = {MLA_D_QK, static_cast<cuuint64_t>(group_heads), static_cast<cuuint64_t>(h_kv),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[3] = {row, row * group_heads, row * group_heads * h_kv};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(group_heads), 1, static_cast<cuuint32_t>(block_tokens)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(q), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

int dense_prepare(const void* q, const void* kv, const int32_t* block_table, int max_pages, int num_pages,
                  const int32_t* seqlens, int batch, int s_q, int h_q, int h_kv, int dtype, int causal, float scale,
                  const int32_t* sched, const int32_t* split_offset, int num_parts, void* workspace,
                  size_t workspace_bytes, void* out, int out_type, float* lse, int32_t* status, DecodeParams* p,
                  CUtensorMap* q_map, CUtensorMap* kv_map, CUtensorMap* sc_map, CUtensorMap* rope_map) {
  if (!q || !kv || !block_table || !seqlens || !sched || !split_offset || !workspace || !out || !lse || !status)
    return MLA_ERR_INVALID_ARG;
  if (batch < 1 || s_q < 1 || h_q < 1 || h_kv < 1 || max_pages < 1 || num_pages < 1 || num_parts < 1)
    return MLA_ERR_INVALID_ARG;
  if (h_q % h_kv != 0) return MLA_ERR_INVALID_ARG;
  if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_FP16) return MLA_ERR_INVALID_ARG;
  if (out_type != MLA_DTYPE_BF16 && out_type != MLA_DTYPE_FP32 && out_type != MLA_DTYPE_FP16)
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return MLA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(s_q) * h_q;
  if (rows > (1 << 20) || static_cast<long long>(batch) * rows > (1LL << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * MLA_PAGE_SIZE * h_kv > (1LL << 31)) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(workspace) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  const WorkspaceLayout w = ws_layout(batch, static_cast<int>(rows), num_parts);
  if (workspace_bytes < w.total) return MLA_ERR_INVALID_ARG;
  const int group_heads = h_q / h_kv;
  int block_tokens = 0, blocks_per_group = 0;
  if (h_kv == 1) {
    blocks_per_group = static_cast<int>((rows + MLA_ROWS_PER_BLOCK - 1) / MLA_ROWS_PER_BLOCK);
  } else {
    if (group_heads > MLA_ROWS_PER_BLOCK) return MLA_ERR_UNSUPPORTED;
    block_tokens = std::min(s_q, MLA_ROWS_PER_BLOCK / group_heads);
    blocks_per_group = (s_q + block_tokens - 1) / block_tokens;
  }
  const long long row_blocks = static_cast<long long>(h_kv) * blocks_per_group;
  if (2LL * num_parts * row_blocks > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo& d = device_info();
  if (d.status != MLA_OK) return d.status;
  int rc = h_kv == 1 ? encode_q_map(q_map, q, static_cast<long long>(batch) * rows)
                     : encode_q_map_groups(q_map, q, static_cast<long long>(batch) * s_q, h_kv, group_heads,
                                           block_tokens);
  if (rc != MLA_OK) return rc;
  // the three box widths the producers load (a value half: 4 slices; rank
  // 0's K slot: slices 4-8; rank 1's RoPE slice), passed in the kernel's kv /
  // sc / rope map parameters
  rc = encode_kv_map(kv_map, kv, num_pages, h_kv, 4);
  if (rc == MLA_OK) rc = encode_kv_map(sc_map, kv, num_pages, h_kv, 5);
  if (rc == MLA_OK) rc = encode_kv_map(rope_map, kv, num_pages, h_kv, 1);
  if (rc != MLA_OK) return rc;
  *p = DecodeParams{};
  p->lengths = seqlens;
  p->default_length = 0;
  p->n_units = batch;
  p->rows = static_cast<int>(rows);
  p->row_blocks = static_cast<int>(row_blocks);
  p->h_q = h_q;
  p->s_q = s_q;
  p->h_kv = h_kv;
  p->group_heads = group_heads;
  p->block_tokens = block_tokens;
  p->blocks_per_group = blocks_per_group;
  p->causal = causal ? 1 : 0;
  p->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  // with many partitions per request their CTAs read the same Q, which is
  // then an L2 hit: all nine boxes at once (staged in the empty V ring) beat
  // streaming them through three slots; with one or two partitions per
  // request the burst crowds the TMA queue and the streamed path wins
  p->q_vring = num_parts >= 4 * batch ? 1 : 0;
  p->block_table = block_table;
  p->max_pages = max_pages;
  p->num_pages = num_pages;
  p->sched = sched;
  p->split_offset = split_offset;
  p->num_parts = num_parts;
  p->o_accum = static_cast<float*>(workspace);
  p->lse_accum = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.lse_off);
  p->out = out;
  p->out_type = out_type;
  p->lse = lse;
  p->status = status;
  return MLA_OK;
}

// How a unit's slots address the record pool: an index list (native
// sparse), per-tile masks over packed records, or a block table (dense FP8).
struct SlotSource {
  const int32_t* indices = nullptr;
  const uint64_t* masks = nullptr;
  const int32_t* block_table = nullptr;
  int max_pages = 0;
};

// One launch of the sparse kernel over a record pool, and its combine.  A
// unit is one query token (native and packed selections: rows = h_q <= 128)
// or one request (a dense FP8 cache under the dense plan: rows = s_q * h_q
// in row blocks of 128, token-major, with the causal alignment per row).
struct SparseCall {
  const void* q = nullptr;
  const uint8_t* kv8 = nullptr;
  int num_pages = 0;
  SlotSource src;
  int topk = 0;                      // slots per unit that may exist
  const int32_t* lengths = nullptr;  // keys (slots) per unit, or NULL: topk
  int n_units = 0, rows = 0, s_q = 1, h_q = 0, causal = 0, unit_request_div = 1;
  float scale = 0.f;
  const int32_t* sched = nullptr;
  const int32_t* split_offset = nullptr;
  int num_parts = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* out = nullptr;
  int out_type = MLA_DTYPE_BF16;
  float* lse = nullptr;
  int32_t* status = nullptr;
  mla_stream_t stream = nullptr;
  int stall = 0;  // 1: the kernel's stall-test instance (mla_test_decode_timeout)
};

int sparse_run(const SparseCall& c, bool combine) {
  if (!c.q || !c.kv8 || (!c.src.indices && !c.src.masks && !c.src.block_table) || !c.sched || !c.split_offset ||
      !c.ws || !c.out || !c.lse || !c.status)
    return MLA_ERR_INVALID_ARG;
  if (c.n_units < 1 || c.rows < 1 || c.h_q < 1 || c.num_pages < 1 || c.topk < 1 || c.num_parts < 1)
    return MLA_ERR_INVALID_ARG;
  if (c.out_type != MLA_DTYPE_BF16 && c.out_type != MLA_DTYPE_FP32 && c.out_type != MLA_DTYPE_FP16)
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(c.scale) || !(c.scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (c.n_units > 65535) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(c.n_units) * c.rows > (1LL << 31) - 1) return MLA_ERR_UNSUPPORTED;
  // record ordinals are 32-bit
  if (static_cast<long long>(c.num_pages) * MLA_PAGE_SIZE > (1LL << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(c.q) || !aligned16(c.kv8) || !aligned16(c.ws) || !aligned16(c.out)) return MLA_ERR_INVALID_ARG;
  const WorkspaceLayout w = ws_layout(c.n_units, c.rows, c.num_parts);
  if (c.ws_bytes < w.total) return MLA_ERR_INVALID_ARG;
  const int row_blocks = (c.rows + MLA_ROWS_PER_BLOCK - 1) / MLA_ROWS_PER_BLOCK;
  if (2LL * c.num_parts * row_blocks > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo& d = device_info();
  if (d.status != MLA_OK) return d.status;
  DecodeParams p{};
  p.lengths = c.lengths;
  p.default_length = c.topk;
  p.n_units = c.n_units;
  p.rows = c.rows;
  p.row_blocks = row_blocks;
  p.h_q = c.h_q;
  p.s_q = c.s_q;
  p.h_kv = 1;
  p.causal = c.causal;
  p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634);
  p.num_pages = c.num_pages;
  p.indices = c.src.indices;
  p.packed_mask = c.src.masks;
  p.block_table = c.src.block_table;
  p.max_pages = c.src.max_pages;
  p.unit_request_div = c.unit_request_div;
  p.topk = c.topk;
  p.kv8 = c.kv8;
  p.sched = c.sched;
  p.split_offset = c.split_offset;
  p.num_parts = c.num_parts;
  p.o_accum = static_cast<float*>(c.ws);
  p.lse_accum = reinterpret_cast<float*>(static_cast<char*>(c.ws) + w.lse_off);
  p.out = c.out;
  p.out_type = c.out_type;
  p.lse = c.lse;
  p.status = c.status;
  CUtensorMap qm;
  const int rc = encode_q_map(&qm, c.q, static_cast<long long>(c.n_units) * c.rows);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(c.stream);
  if (launch_sparse(qm, p, c.num_parts, c.stall, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (!combine) return MLA_OK;
  return mla_combine(c.ws, c.ws_bytes, c.split_offset, c.n_units, c.rows, c.num_parts, c.out, c.out_type, c.lse,
                     c.status, c.stream);
}

// A cache of FP8 records runs the sparse kernel (exact scores in codes and
// scales) with the block table as the slot source and a whole request as
// the unit, under the same plan as the 16-bit caches.
int fp8_record_splits(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages, int num_pages,
                      const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv, int causal,
                      float softmax_scale, const int32_t* d_sched, const int32_t* d_split_offset, int num_parts,
                      void* d_workspace, size_t workspace_bytes, void* d_out, int out_type, float* d_lse,
                      int32_t* d_status, mla_stream_t stream, int stall) {
  if (!d_block_table || !d_cache_seqlens || max_pages < 1 || batch < 1 || s_q < 1 || h_q < 1)
    return MLA_ERR_INVALID_ARG;
  if (h_kv != 1) return MLA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(s_q) * h_q;
  if (rows > (1 << 20) || static_cast<long long>(max_pages) * MLA_PAGE_SIZE > (1LL << 31) - 1)
    return MLA_ERR_UNSUPPORTED;
  SparseCall c;
  c.q = d_q;
  c.kv8 = static_cast<const uint8_t*>(d_kv);
  c.num_pages = num_pages;
  c.src.block_table = d_block_table;
  c.src.max_pages = max_pages;
  c.topk = max_pages * MLA_PAGE_SIZE;
  c.lengths = d_cache_seqlens;
  c.n_units = batch;
  c.rows = static_cast<int>(rows);
  c.s_q = s_q;
  c.h_q = h_q;
  c.causal = causal ? 1 : 0;
  c.unit_request_div = 1;
  c.scale = softmax_scale;
  c.sched = d_sched;
  c.split_offset = d_split_offset;
  c.num_parts = num_parts;
  c.ws = d_workspace;
  c.ws_bytes = workspace_bytes;
  c.out = d_out;
  c.out_type = out_type;
  c.lse = d_lse;
  c.status = d_status;
  c.stream = stream;
  c.stall = stall;
  return sparse_run(c, false);
}

}  // namespace

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null pointer, bad size, misalignment or small workspace";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape or device not supported by this sm_103a build";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA runtime call failed";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a device pipeline wait ran out of time";
    case MLA_ERR_BAD_INDEX: return "MLA_ERR_BAD_INDEX: block-table entry or sparse index outside the pool";
    default: return "unknown mla status";
  }
}

int mla_num_parts(int rows_per_unit, int is_sparse_fp8) {
  if (rows_per_unit < 1 || (is_sparse_fp8 != 0 && is_sparse_fp8 != 1)) return -MLA_ERR_INVALID_ARG;
  const DeviceInfo& d = device_info();
  if (d.status != MLA_OK) return -d.status;
  const int clusters = is_sparse_fp8 ? d.sparse_clusters : d.dense_clusters;
  const int row_blocks = (rows_per_unit + MLA_ROWS_PER_BLOCK - 1) / MLA_ROWS_PER_BLOCK;
  const int parts = clusters / row_blocks;
  return parts > 0 ? parts : 1;
}

int mla_num_parts_dense(int s_q, int h_q, int h_kv) {
  if (s_q < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0) return -MLA_ERR_INVALID_ARG;
  const int group_heads = h_q / h_kv;
  if (h_kv > 1 && group_heads > MLA_ROWS_PER_BLOCK) return -MLA_ERR_UNSUPPORTED;
  const DeviceInfo& d = device_info();
  if (d.status != MLA_OK) return -d.status;
  long long row_blocks;
  if (h_kv == 1) {
    row_blocks = (static_cast<long long>(s_q) * h_q + MLA_ROWS_PER_BLOCK - 1) / MLA_ROWS_PER_BLOCK;
  } else {
    const int block_tokens = std::min(s_q, MLA_ROWS_PER_BLOCK / group_heads);
    row_blocks = static_cast<long long>(h_kv) * ((s_q + block_tokens - 1) / block_tokens);
  }
  const long long parts = d.dense_clusters / row_blocks;
  return parts > 0 ? static_cast<int>(parts) : 1;
}

size_t mla_workspace_bytes(int n_units, int rows_per_unit, int num_parts) {
  if (n_units < 0 || rows_per_unit < 1 || num_parts < 1) return 0;
  return ws_layout(n_units, rows_per_unit, num_parts).total;
}

namespace {

int get_metadata(const int32_t* d_lengths, int default_length, int n_units, int num_parts, int32_t* d_sched,
                 int32_t* d_split_offset, int request_local, mla_stream_t stream) {
  if (n_units < 1 || num_parts < 1 || !d_sched || !d_split_offset) return MLA_ERR_INVALID_ARG;
  if (d_lengths == nullptr && default_length < 0) return MLA_ERR_INVALID_ARG;
  return launch_sched(d_lengths, default_length, n_units, num_parts, d_sched, d_split_offset, request_local,
                      reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace

int mla_get_metadata(const int32_t* d_lengths, int default_length, int n_units, int num_parts, int32_t* d_sched,
                     int32_t* d_split_offset, mla_stream_t stream) {
  return get_metadata(d_lengths, default_length, n_units, num_parts, d_sched, d_split_offset, 0, stream);
}

int mla_get_metadata_request_local(const int32_t* d_lengths, int default_length, int n_units, int num_parts,
                                   int32_t* d_sched, int32_t* d_split_offset, mla_stream_t stream) {
  return get_metadata(d_lengths, default_length, n_units, num_parts, d_sched, d_split_offset, 1, stream);
}

int mla_decode_splits(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages,
                      int num_pages, const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                      int dtype, int causal, float softmax_scale, const int32_t* d_sched,
                      const int32_t* d_split_offset, int num_parts, void* d_workspace, size_t workspace_bytes,
                      void* d_out, int out_type, float* d_lse, int32_t* d_status, mla_stream_t stream) {
  if (dtype == MLA_DTYPE_FP8_RECORD)
    return fp8_record_splits(d_q, d_kv, d_block_table, max_pages, num_pages, d_cache_seqlens, batch, s_q, h_q, h_kv,
                             causal, softmax_scale, d_sched, d_split_offset, num_parts, d_workspace, workspace_bytes,
                             d_out, out_type, d_lse, d_status, stream, 0);
  DecodeParams p;
  CUtensorMap qm, km, sm, rm;
  const int rc = dense_prepare(d_q, d_kv, d_block_table, max_pages, num_pages, d_cache_seqlens, batch, s_q, h_q,
                               h_kv, dtype, causal, softmax_scale, d_sched, d_split_offset, num_parts, d_workspace,
                               workspace_bytes, d_out, out_type, d_lse, d_status, &p, &qm, &km, &sm, &rm);
  if (rc != MLA_OK) return rc;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int kind = (dtype == MLA_DTYPE_FP16 ? 1 : 0) + (p.q_vring ? 2 : 0);
  return launch_dense(qm, km, sm, rm, p, num_parts, kind, cs) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_combine(const void* d_workspace, size_t workspace_bytes, const int32_t* d_split_offset, int n_units,
                int rows_per_unit, int num_parts, void* d_out, int out_type, float* d_lse, int32_t* d_status,
                mla_stream_t stream) {
  if (!d_workspace || !d_split_offset || !d_out || !d_lse) return MLA_ERR_INVALID_ARG;
  if (n_units < 1 || n_units > 65535 || rows_per_unit < 1 || num_parts < 1) return MLA_ERR_INVALID_ARG;
  if (out_type != MLA_DTYPE_BF16 && out_type != MLA_DTYPE_FP32 && out_type != MLA_DTYPE_FP16)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(d_workspace) || !aligned16(d_out)) return MLA_ERR_INVALID_ARG;
  const WorkspaceLayout w = ws_layout(n_units, rows_per_unit, num_parts);
  if (workspace_bytes < w.total) return MLA_ERR_INVALID_ARG;
  const DeviceInfo& d = device_info();
  if (d.status != MLA_OK) return d.status;
  const float* o = static_cast<const float*>(d_workspace);
  const float* l = reinterpret_cast<const float*>(static_cast<const char*>(d_workspace) + w.lse_off);
  return launch_combine(o, l, d_split_offset, n_units, rows_per_unit, num_parts, d_out, out_type, d_lse, d_status,
                        d.sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_decode_fwd(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages, int num_pages,
                   const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv, int dtype, int causal,
                   float softmax_scale, const int32_t* d_sched, const int32_t* d_split_offset, int num_parts,
                   void* d_workspace, size_t workspace_bytes, void* d_out, int out_type, float* d_lse,
                   int32_t* d_status, mla_stream_t stream) {
  if (batch > 65535) return MLA_ERR_UNSUPPORTED;
  int rc = mla_decode_splits(d_q, d_kv, d_block_table, max_pages, num_pages, d_cache_seqlens, batch, s_q, h_q, h_kv,
                             dtype, causal, softmax_scale, d_sched, d_split_offset, num_parts, d_workspace,
                             workspace_bytes, d_out, out_type, d_lse, d_status, stream);
  if (rc != MLA_OK) return rc;
  return mla_combine(d_workspace, workspace_bytes, d_split_offset, batch, s_q * h_q, num_parts, d_out, out_type,
                     d_lse, d_status, stream);
}

namespace {

// A selection (native or packed): one unit per query token, h_q <= 128 rows.
int sparse_decode(const void* d_q, const uint8_t* d_kv8, int num_pages, SlotSource src, int topk,
                  const int32_t* d_topk_length, int batch, int s_q, int h_q, float softmax_scale,
                  const int32_t* d_sched, const int32_t* d_split_offset, int num_parts, void* d_workspace,
                  size_t workspace_bytes, void* d_out, float* d_lse, int32_t* d_status, mla_stream_t stream) {
  if (batch < 1 || s_q < 1 || h_q < 1) return MLA_ERR_INVALID_ARG;
  if (h_q > MLA_ROWS_PER_BLOCK) return MLA_ERR_UNSUPPORTED;
  const long long units = static_cast<long long>(batch) * s_q;
  if (units > 65535) return MLA_ERR_UNSUPPORTED;
  SparseCall c;
  c.q = d_q;
  c.kv8 = d_kv8;
  c.num_pages = num_pages;
  c.src = src;
  c.topk = topk;
  c.lengths = d_topk_length;
  c.n_units = static_cast<int>(units);
  c.rows = h_q;
  c.h_q = h_q;
  c.scale = softmax_scale;
  c.sched = d_sched;
  c.split_offset = d_split_offset;
  c.num_parts = num_parts;
  c.ws = d_workspace;
  c.ws_bytes = workspace_bytes;
  c.out = d_out;
  c.lse = d_lse;
  c.status = d_status;
  c.stream = stream;
  return sparse_run(c, true);
}

// Packed workspace layout: records, then one 64-bit mask per (unit, tile).
struct PackedLayout {
  long long tiles, records_bytes, total;
};

PackedLayout packed_layout(long long n_units, int topk) {
  PackedLayout l;
  l.tiles = (topk + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
  l.records_bytes = n_units * l.tiles * MLA_PAGE_SIZE * MLA_RECORD_BYTES;
  l.total = l.records_bytes + n_units * l.tiles * static_cast<long long>(sizeof(uint64_t));
  return l;
}

}  // namespace

int mla_sparse_fp8_decode_fwd(const void* d_q, const uint8_t* d_kv8, int num_pages, const int32_t* d_indices,
                              int topk, const int32_t* d_topk_length, int batch, int s_q, int h_q,
                              float softmax_scale, const int32_t* d_sched, const int32_t* d_split_offset,
                              int num_parts, void* d_workspace, size_t workspace_bytes, void* d_out, float* d_lse,
                              int32_t* d_status, mla_stream_t stream) {
  if (!d_indices) return MLA_ERR_INVALID_ARG;
  SlotSource src;
  src.indices = d_indices;
  return sparse_decode(d_q, d_kv8, num_pages, src, topk, d_topk_length, batch, s_q, h_q, softmax_scale, d_sched,
                       d_split_offset, num_parts, d_workspace, workspace_bytes, d_out, d_lse, d_status, stream);
}

size_t mla_packed_kv_workspace_bytes(int n_units, int topk) {
  if (n_units < 0 || topk < 1) return 0;
  return static_cast<size_t>(packed_layout(n_units, topk).total);
}

namespace {

int pack_selected(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int topk,
                  const int32_t* d_topk_length, int n_units, void* d_packed, size_t packed_bytes, int32_t* d_status,
                  int stall_test, mla_stream_t stream) {
  if (!d_kv8 || !d_indices || !d_packed || !d_status) return MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || topk < 1 || n_units < 0) return MLA_ERR_INVALID_ARG;
  if (n_units > 65535) return MLA_ERR_UNSUPPORTED;
  // slot indices are 32-bit: the pool's slots must fit
  if (static_cast<long long>(num_pages) * MLA_PAGE_SIZE > (1LL << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(d_kv8) || !aligned16(d_packed)) return MLA_ERR_INVALID_ARG;
  const PackedLayout l = packed_layout(n_units, topk);
  if (packed_bytes < static_cast<size_t>(l.total)) return MLA_ERR_INVALID_ARG;
  if (n_units == 0) return MLA_OK;
  uint8_t* records = static_cast<uint8_t*>(d_packed);
  uint64_t* masks = reinterpret_cast<uint64_t*>(records + l.records_bytes);
  return launch_pack(d_kv8, num_pages, d_indices, topk, d_topk_length, n_units, records, masks, d_status,
                     stall_test, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace

int mla_pack_selected_kv(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int topk,
                         const int32_t* d_topk_length, int n_units, void* d_packed, size_t packed_bytes,
                         int32_t* d_status, mla_stream_t stream) {
  return pack_selected(d_kv8, num_pages, d_indices, topk, d_topk_length, n_units, d_packed, packed_bytes, d_status,
                       0, stream);
}

int mla_test_decode_timeout(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages,
                            int num_pages, const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                            int dtype, int causal, float softmax_scale, const int32_t* d_sched,
                            const int32_t* d_split_offset, int num_parts, void* d_workspace, size_t workspace_bytes,
                            void* d_out, int out_type, float* d_lse, int32_t* d_status, mla_stream_t stream) {
  if (dtype == MLA_DTYPE_FP8_RECORD)
    return fp8_record_splits(d_q, d_kv, d_block_table, max_pages, num_pages, d_cache_seqlens, batch, s_q, h_q, h_kv,
                             causal, softmax_scale, d_sched, d_split_offset, num_parts, d_workspace, workspace_bytes,
                             d_out, out_type, d_lse, d_status, stream, 1);
  if (dtype != MLA_DTYPE_BF16) return MLA_ERR_UNSUPPORTED;
  DecodeParams p;
  CUtensorMap qm, km, sm, rm;
  const int rc = dense_prepare(d_q, d_kv, d_block_table, max_pages, num_pages, d_cache_seqlens, batch, s_q, h_q,
                               h_kv, dtype, causal, softmax_scale, d_sched, d_split_offset, num_parts, d_workspace,
                               workspace_bytes, d_out, out_type, d_lse, d_status, &p, &qm, &km, &sm, &rm);
  if (rc != MLA_OK) return rc;
  return launch_dense(qm, km, sm, rm, p, num_parts, 4, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_test_pack_timeout(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int topk,
                          const int32_t* d_topk_length, int n_units, void* d_packed, size_t packed_bytes,
                          int32_t* d_status, mla_stream_t stream) {
  return pack_selected(d_kv8, num_pages, d_indices, topk, d_topk_length, n_units, d_packed, packed_bytes, d_status,
                       1, stream);
}

int mla_sparse_fp8_packed_decode_fwd(const void* d_q, const void* d_packed, size_t packed_bytes, int topk,
                                     const int32_t* d_topk_length, int batch, int s_q, int h_q, float softmax_scale,
                                     const int32_t* d_sched, const int32_t* d_split_offset, int num_parts,
                                     void* d_workspace, size_t workspace_bytes, void* d_out, float* d_lse,
                                     int32_t* d_status, mla_stream_t stream) {
  if (!d_packed || topk < 1 || batch < 1 || s_q < 1) return MLA_ERR_INVALID_ARG;
  const long long units = static_cast<long long>(batch) * s_q;
  if (units > 65535) return MLA_ERR_UNSUPPORTED;
  const PackedLayout l = packed_layout(units, topk);
  if (packed_bytes < static_cast<size_t>(l.total)) return MLA_ERR_INVALID_ARG;
  const uint8_t* records = static_cast<const uint8_t*>(d_packed);
  // the packed records form a pool of units * tiles pages of 64 records,
  // unit u's tiles being pages u * tiles .. u * tiles + tiles - 1; slot t of
  // unit u is record u * tiles * 64 + t, live when its mask bit is set
  const long long pool_pages = units * l.tiles;
  if (pool_pages * MLA_PAGE_SIZE > (1LL << 31) - 1) return MLA_ERR_UNSUPPORTED;
  SlotSource src;
  src.masks = reinterpret_cast<const uint64_t*>(records + l.records_bytes);
  return sparse_decode(d_q, records, static_cast<int>(pool_pages), src, topk, d_topk_length, batch, s_q, h_q,
                       softmax_scale, d_sched, d_split_offset, num_parts, d_workspace, workspace_bytes, d_out, d_lse,
                       d_status, stream);
}


int mla_sparse_fp8_unpack(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int n, float* d_k_out,
                          int32_t* d_status, mla_stream_t stream) {
  if (!d_kv8 || !d_indices || !d_k_out || !d_status || num_pages < 1 || n < 0) return MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * MLA_PAGE_SIZE > (1LL << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(d_kv8) || !aligned16(d_k_out)) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  return launch_unpack(d_kv8, num_pages, d_indices, n, d_k_out, d_status, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // extern "C"
