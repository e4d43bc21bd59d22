// Dense decode with the split workspace in a file-scope device array, for
// callers that cannot hand the library any device scratch of their own.
//
// Who needs it: a host program written in plain C that links only this
// library and has no device allocator to draw a workspace from, and a serving
// runtime that reserves almost all of HBM for its KV pool when it starts and
// allows no allocation on the decode path afterwards (a cudaMalloc there can
// fail once the pool is reserved, and it synchronises the device, which
// stalls every stream of the process).  Such a caller passes its inputs and
// outputs as usual and the partial outputs go to the array below, which is
// sized once, at load time, and never grows.
//
// The array is ordinary module memory: every GPU on which the library's
// device code is loaded holds its MLA_STATIC_WORKSPACE_BYTES until the
// process exits.  Nothing here calls cudaMalloc, cudaFree or any routine
// that allocates device memory.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "mla_paged_kv.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MLA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// In host code `g_static_workspace` names a host-side stand-in that the
// runtime maps to the array, not a device address; the address a kernel may
// use comes from cudaGetSymbolAddress, once per device, with that device
// current.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

void* g_ws_ptr[kMaxDevices] = {};
std::mutex g_ws_mu;

// Device address of the array on the current device.  The first call on a
// device looks it up (which also makes the runtime load this module there)
// and caches it.
int static_workspace(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  if (g_ws_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_ws_ptr[dev] = p;
  }
  *ptr = g_ws_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_fwd_static_ws(const void* d_q, const void* d_kv, const int32_t* d_block_table,
                                        int max_pages, int num_pages, const int32_t* d_cache_seqlens, int batch,
                                        int s_q, int h_q, int h_kv, int dtype, int causal, float softmax_scale,
                                        const int32_t* d_sched, const int32_t* d_split_offset, int num_parts,
                                        void* d_out, int out_type, float* d_lse, int32_t* d_status,
                                        mla_stream_t stream) {
  if (batch < 1 || s_q < 1 || h_q < 1 || num_parts < 1) return MLA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(s_q) * h_q;
  if (rows > (1 << 20)) return MLA_ERR_UNSUPPORTED;
  // Size check before anything touches the device: a problem whose partials
  // do not fit the fixed array is refused, never truncated.
  const size_t need = mla_workspace_bytes(batch, static_cast<int>(rows), num_parts);
  if (need == 0 || need > kStaticWorkspaceBytes) return MLA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  const int rc = static_workspace(&ws);
  if (rc != MLA_OK) return rc;
  // No part of the array needs clearing: in one call the decode kernel writes
  // every partial output and LSE that the combine then reads.
  return mla_decode_fwd(d_q, d_kv, d_block_table, max_pages, num_pages, d_cache_seqlens, batch, s_q, h_q, h_kv,
                        dtype, causal, softmax_scale, d_sched, d_split_offset, num_parts, ws, kStaticWorkspaceBytes,
                        d_out, out_type, d_lse, d_status, stream);
}
