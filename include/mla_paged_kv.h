/*
 * mla_paged_kv.h -- C ABI of the GB300 (sm_103a) MLA paged-KV decode library.
 *
 * Multi-head latent attention decode: every query token has h_q heads that
 * all attend to ONE latent KV head of 576 entries (512 "NoPE" + 64 "RoPE").
 * The score is the dot product over all 576 entries; the value is the first
 * 512 entries of the same row (FlashMLA PR #183 "Add SM80 (Ampere/A100)
 * dense MLA decode kernel", section Design).  Keys live in a paged cache of
 * 64-token pages addressed through a per-request block table (same page,
 * section "How the occupancy work went").  Work is split along the keys
 * (split-KV); every split writes a partial output and its log-sum-exp, and a
 * combine kernel merges them (same page, Summary and "Modifications outside
 * csrc/sm80/").  The sparse variant attends over top-k selected 656-byte FP8
 * records addressed by physical slot index (FlashMLA PR #200 "[SM90] Add
 * packed selected-KV sparse decode", sections Motivation and "SM90 packing
 * kernel").
 *
 * Conventions for every entry point:
 *  - All pointers named d_* are DEVICE pointers owned by the caller.  The
 *    library never allocates or frees device memory and keeps no state
 *    besides a per-device cache of kernel attributes (and, for
 *    mla_decode_fwd_static_ws only, one fixed device array and its address).
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  No call synchronises with the host.
 *  - Host-detectable errors are returned BEFORE anything is launched.
 *  - Errors found on the device (bad block-table entry, bad sparse index,
 *    a pipeline wait that timed out) are written to *d_status (int32, must
 *    be zeroed by the caller before the call; the first error wins).  A
 *    block-table entry or sparse index outside the pool masks the keys it
 *    names (weight 0, as if absent) and the rest of the call is exact.
 *    After MLA_ERR_TIMEOUT the kernel has given up part of its work: the
 *    results of that call are unspecified and must not be used (the context
 *    and the stream stay usable for later calls).
 *  - Layouts are row-major and contiguous.  A query "row" of request b is
 *    r = i * h_q + h for query token i < s_q and head h < h_q.
 *  - Every d_* pointer must be 16-byte aligned.
 */
#ifndef MLA_PAGED_KV_H_
#define MLA_PAGED_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* same type as cudaStream_t */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, workspace too small */
  MLA_ERR_UNSUPPORTED = 2, /* shape this build does not handle, or no sm_103a device */
  MLA_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, attribute query) */
  MLA_ERR_TIMEOUT = 4,     /* device: a pipeline wait exceeded its time budget */
  MLA_ERR_BAD_INDEX = 5    /* device: block-table entry or sparse index outside the pool */
} mla_status_t;

/* Element types of query, cache and output tensors.  The values keep the
 * meaning of an older 0/1 "fp32 output" flag: 0 = bf16, 1 = fp32. */
typedef enum {
  MLA_DTYPE_BF16 = 0,
  MLA_DTYPE_FP32 = 1, /* outputs only */
  MLA_DTYPE_FP16 = 2,
  MLA_DTYPE_FP8_RECORD = 3 /* KV only: the pool of 656-byte FP8 records, bf16 Q */
} mla_dtype_t;

/* Fixed geometry (FlashMLA PR #183 Design; PR #200 "SM90 packing kernel"). */
#define MLA_PAGE_SIZE 64      /* tokens per page */
#define MLA_D_QK 576          /* latent row: 512 NoPE + 64 RoPE */
#define MLA_D_V 512           /* value = first 512 entries of the row */
#define MLA_RECORD_BYTES 656  /* FP8 record: 512 E4M3 + 4 fp32 scales + 64 bf16 */
#define MLA_ROWS_PER_BLOCK 128 /* query rows handled by one CTA pair */
#define MLA_SCHED_INTS 8      /* int32 per partition in the scheduler metadata */
#define MLA_SPLIT_FIXED_COST 4 /* per-split fixed cost, in 64-key tiles, used by the scheduler */

/* Human-readable name of a status code.  Never returns NULL. */
const char* mla_status_string(int status);

/* Number of key partitions (CTA pairs per row block) the decode kernels run,
 * derived from how many 2-CTA clusters of the kernel fit on the current
 * device at once (FlashMLA PR #183, "How the occupancy work went": the
 * split count follows the CTAs that actually fit).
 *   rows_per_unit: query rows sharing one key set (dense: s_q*h_q;
 *                  sparse: h_q), >= 1.
 *   is_sparse_fp8: 0 for the dense bf16 kernel, 1 for the sparse FP8 one.
 * Returns >= 1, or a negative mla_status_t on error. */
int mla_num_parts(int rows_per_unit, int is_sparse_fp8);

/* The same for the dense kernel with h_kv latent KV heads: one partition
 * runs h_kv * (row blocks per head group) CTA pairs, counted exactly as
 * mla_decode_fwd counts them.  For h_kv = 1 it equals
 * mla_num_parts(s_q * h_q, 0).  Returns >= 1, or a negative mla_status_t. */
int mla_num_parts_dense(int s_q, int h_q, int h_kv);

/* Bytes of split workspace needed: (n_units + num_parts) split slots, each
 * rows_per_unit x 512 fp32 partial outputs plus rows_per_unit fp32 LSEs,
 * then n_units x rows_per_unit x 576 fp16 values (the fp16 copy of Q that
 * the FP8-record calls make once per call; other calls leave it unused),
 * each region starting on a 256-byte boundary.
 * n_units: dense = batch, sparse = batch*s_q. */
size_t mla_workspace_bytes(int n_units, int rows_per_unit, int num_parts);

/* Split-KV scheduler (FlashMLA PR #183: computed once per batch on device
 * from the sequence lengths and reused by every layer).
 *   d_lengths   int32 [n_units]: keys per unit (dense: cache_seqlens; sparse:
 *               topk_length flattened over (b, i)).  May be NULL only when
 *               default_length >= 0, in which case every unit has that many.
 *   num_parts   from mla_num_parts().
 *   d_sched     int32 [num_parts * MLA_SCHED_INTS] out: per partition
 *               (begin_unit, begin_tile, end_unit, end_tile, begin_split, 0,0,0)
 *               over 64-key tiles.
 *   d_split_offset int32 [n_units + 1] out: prefix sum of splits per unit.
 * The plan: cost(unit) = tiles + F (F = MLA_SPLIT_FIXED_COST); partitions
 * take consecutive (unit, tile) ranges of at most `cap` cost (whole units
 * while remaining + F fits, then budget - F tiles of the next one); the last
 * one takes the rest.  With c0 = ceil(total cost / num_parts), cap is the
 * smallest value in c0 .. c0 + F that leaves the last partition at most cap;
 * c0 + F if none does, or when n_units > 4096 or num_parts > 128 (the
 * candidates walk at once, one warp each).  One thread block. */
int mla_get_metadata(const int32_t* d_lengths, int default_length, int n_units, int num_parts,
                     int32_t* d_sched, int32_t* d_split_offset, mla_stream_t stream);

/* Request-local split plan, in the same metadata format (FlashMLA PR #200,
 * section "Scheduler policy", names a request-local scheduler for its H=64
 * sparse path without defining it; this is the library's reading of it).
 * No partition spans two units.  Each unit with tiles gets one partition; the
 * other num_parts - (units with tiles) partitions are shared out in proportion
 * to the tile counts, by largest remainder of tiles * spare / total tiles (ties
 * to the lower unit), and a unit gets at most one partition per tile.  Unit
 * u's k-th of s partitions covers tiles [k*n/s, (k+1)*n/s); partitions are
 * numbered in unit order and unused ones are empty.  Falls back to
 * mla_get_metadata's plan when no unit has tiles, when more units have tiles
 * than there are partitions, or above 1024 units.  Arguments as for
 * mla_get_metadata; both decode entry points accept either plan. */
int mla_get_metadata_request_local(const int32_t* d_lengths, int default_length, int n_units, int num_parts,
                                   int32_t* d_sched, int32_t* d_split_offset, mla_stream_t stream);

/* Dense MLA decode: split-KV attention kernel, then the combine kernel
 * (chained with programmatic dependent launch).  FlashMLA PR #183 (Summary,
 * Test plan) checks bf16 and fp16 and 1 to 4 KV heads; both are here.
 *   d_q            [batch, s_q, h_q, 576], element type `dtype`
 *   d_kv           [num_pages, 64, h_kv, 576] paged latent cache, type `dtype`
 *                  (h_kv = 1: [num_pages, 64, 576])
 *   d_block_table  int32 [batch, max_pages]: logical page -> physical page.
 *                  An entry outside [0, num_pages) at a position the request
 *                  reads masks that page's 64 keys and is reported
 *                  (MLA_ERR_BAD_INDEX).
 *   d_cache_seqlens int32 [batch]: keys of request b, including its s_q new
 *                  tokens.  Key j of request b is row j%64 of page
 *                  block_table[b][j/64].
 *   h_kv           latent KV heads, dividing h_q; query head h reads KV head
 *                  h / (h_q / h_kv).  h_q / h_kv <= 128 when h_kv > 1.
 *   dtype          MLA_DTYPE_BF16 or MLA_DTYPE_FP16 (q and kv alike; P is
 *                  rounded to the same type before the P V product), or
 *                  MLA_DTYPE_FP8_RECORD: d_kv is a paged cache of FP8 records
 *                  [num_pages, 64, 656] (FlashMLA PR #200, "FP8 KV cache
 *                  format": 512 E4M3 NoPE codes, four fp32 scales, one per
 *                  128 dims, 64 bf16 RoPE dims), q is bf16, h_kv must be 1.
 *                  Token j of request b is record j%64 of page
 *                  block_table[b][j/64], decoded as for
 *                  mla_sparse_fp8_decode_fwd (FlashMLA PR #183, "Limitations
 *                  / future work", names an FP8 cache as missing from its
 *                  dense kernel without giving a format; PR #200's record is
 *                  the FP8 format the pages define).  This dtype runs the
 *                  sparse kernel with the block table as its slot source and
 *                  a whole request as its unit, under the same plan and
 *                  workspace as the 16-bit caches: the scores stay exact in
 *                  codes and scales (a per-group fp32 accumulator each, the
 *                  scales applied in fp32), the value scale is folded into
 *                  P (rounded to bf16).
 *   causal         1: query token i sees keys j <= L_b - s_q + i.
 *   softmax_scale  multiplies q.k (e.g. 1/sqrt(576)); must be finite and > 0.
 *   d_sched, d_split_offset, num_parts: from mla_get_metadata (or its
 *                  request-local form) with d_lengths = d_cache_seqlens,
 *                  n_units = batch.
 *   d_workspace    >= mla_workspace_bytes(batch, s_q*h_q, num_parts) bytes.
 *   d_out          [batch, s_q, h_q, 512] of out_type: MLA_DTYPE_BF16,
 *                  MLA_DTYPE_FP16 or MLA_DTYPE_FP32 (0, 2, 1)
 *   d_lse          fp32 [batch, s_q, h_q]: natural-log LSE of the scaled
 *                  scores; -inf (and out = 0) for a row that sees no key.
 *   d_status       int32, caller-zeroed; see conventions above. */
int mla_decode_fwd(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages,
                   int num_pages, const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                   int dtype, int causal, float softmax_scale, const int32_t* d_sched,
                   const int32_t* d_split_offset, int num_parts, void* d_workspace, size_t workspace_bytes,
                   void* d_out, int out_type, float* d_lse, int32_t* d_status, mla_stream_t stream);

/* The first half of mla_decode_fwd alone: the split-KV attention kernel.
 * Units with exactly one split are written straight to d_out/d_lse; the
 * others leave their partials in d_workspace for mla_combine (or for an
 * exchange step before it).  Same arguments as mla_decode_fwd. */
int mla_decode_splits(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages,
                      int num_pages, const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                      int dtype, int causal, float softmax_scale, const int32_t* d_sched,
                      const int32_t* d_split_offset, int num_parts, void* d_workspace, size_t workspace_bytes,
                      void* d_out, int out_type, float* d_lse, int32_t* d_status, mla_stream_t stream);

/* Size of the device array mla_decode_fwd_static_ws keeps its split
 * workspace in: 64 MiB on every GPU that loads the library. */
#define MLA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)

/* mla_decode_fwd for callers that cannot provide device scratch.  Neither
 * FlashMLA page has a counterpart: it is this library's own addition.  Some
 * callers have no workspace to give: a plain C host program linked only
 * against this library has no device allocator at hand, and a serving
 * runtime that reserves nearly all of HBM for its KV pool at start-up may
 * forbid allocation on the decode path, where a cudaMalloc could fail and
 * would synchronise the device.  This call takes the same inputs and outputs
 * as mla_decode_fwd minus d_workspace/workspace_bytes, allocates nothing,
 * and keeps the partials in a file-scope device array of
 * MLA_STATIC_WORKSPACE_BYTES, which every GPU that loads the library holds
 * until the process exits.
 *  - Returns MLA_ERR_UNSUPPORTED, before any launch, when
 *    mla_workspace_bytes(batch, s_q*h_q, num_parts) exceeds
 *    MLA_STATIC_WORKSPACE_BYTES (64 requests x 128 heads with 76 parts need
 *    46.2 MB and fit).
 *  - The first call on a device looks up the array's device address there
 *    (cudaGetSymbolAddress with that device current) and caches it; make
 *    that first call on each device before beginning any stream capture.
 *  - All calls on a device share the one array, and it keeps what the last
 *    call left.  Nothing in it needs to start at zero (the decode kernel
 *    writes every partial the combine reads in the same call), but calls
 *    that can overlap on the GPU (unordered streams) race on it and corrupt
 *    each other's results: order them on one stream or with events. */
int mla_decode_fwd_static_ws(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages,
                             int num_pages, const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                             int dtype, int causal, float softmax_scale, const int32_t* d_sched,
                             const int32_t* d_split_offset, int num_parts, void* d_out, int out_type, float* d_lse,
                             int32_t* d_status, mla_stream_t stream);

/* LSE-weighted combine of split partials (FlashMLA PR #183 Summary: the
 * combine kernel merges the splits).  For every unit with != 1 split and
 * every row r < rows_per_unit:
 *   L = ln sum_s exp(lse_s);  out = sum_s exp(lse_s - L) * O_s;  lse = L,
 * where splits with lse_s = -inf weigh 0; a unit with 0 splits, or whose
 * splits are all -inf, gets out = 0, lse = -inf.  Units with exactly one
 * split are left alone (the decode kernel wrote them).
 *   d_workspace as filled by mla_decode_splits / the sparse kernel.
 *   d_out [n_units, rows_per_unit, 512] of out_type (MLA_DTYPE_BF16, _FP32 or
 *   _FP16), d_lse [n_units, rows].
 *   d_status      int32 (may be NULL): MLA_ERR_TIMEOUT if a wait of the
 *                 kernel for its own bulk copies ran out (the rows it had
 *                 not finished are then unspecified).
 * Launched with programmatic dependent launch: it may start before the
 * previous kernel on the stream ends and waits for it on the device before
 * reading the workspace; d_split_offset it reads before that wait, so it
 * must not be written by the kernel launched just before this call (the
 * plan from mla_get_metadata is ready long before). */
int mla_combine(const void* d_workspace, size_t workspace_bytes, const int32_t* d_split_offset, int n_units,
                int rows_per_unit, int num_parts, void* d_out, int out_type, float* d_lse, int32_t* d_status,
                mla_stream_t stream);

/* Sparse FP8 MLA decode (FlashMLA PR #200).  Query token (b, i) attends to
 * the records selected by d_indices[b][i][0 .. topk_length[b][i]); entry t
 * is a physical slot: page idx/64, row idx%64 of d_kv8.  -1 anywhere is
 * masked; a duplicated index counts twice; an index outside
 * [0, num_pages*64) is masked and reported as MLA_ERR_BAD_INDEX.
 * Record layout (656 B): [0,512) E4M3 codes, [512,528) four fp32 scales,
 * [528,656) 64 bf16 RoPE values; key[d] = e4m3[d] * scale[d/128] (d < 512),
 * key[512+e] = rope[e]; value = key[0..512).  In the kernel the scores are
 * exact in codes and scales: each 128-dim group's codes (exact in bf16) meet
 * Q on the tensor cores with fp32 accumulation, and the group's scale
 * multiplies that product in fp32; for the values, the softmax weight times
 * the group's scale is rounded to bf16 and meets the unscaled codes, and each
 * group's output is divided by the sum of the weights so rounded (the LSE
 * keeps the exact sum), so that a row with one or a few dominant keys
 * carries no rounding of its scales into the output.  A scale below the
 * smallest normal fp32 counts as 0.
 *   d_q           bf16 [batch, s_q, h_q, 576]
 *   d_kv8         uint8 [num_pages, 64, 656]
 *   d_indices     int32 [batch, s_q, topk]
 *   d_topk_length int32 [batch, s_q] or NULL (= topk)
 *   d_sched, d_split_offset, num_parts: from mla_get_metadata with
 *                 d_lengths = d_topk_length (or NULL with default topk),
 *                 n_units = batch*s_q, and mla_num_parts(h_q, 1).
 *   d_workspace   >= mla_workspace_bytes(batch*s_q, h_q, num_parts)
 *   d_out bf16 [batch, s_q, h_q, 512], d_lse fp32 [batch, s_q, h_q]. */
int mla_sparse_fp8_decode_fwd(const void* d_q, const uint8_t* d_kv8, int num_pages, const int32_t* d_indices,
                              int topk, const int32_t* d_topk_length, int batch, int s_q, int h_q,
                              float softmax_scale, const int32_t* d_sched, const int32_t* d_split_offset,
                              int num_parts, void* d_workspace, size_t workspace_bytes, void* d_out,
                              float* d_lse, int32_t* d_status, mla_stream_t stream);

/* Packed selected-KV path (FlashMLA PR #200, "[SM90] Add packed selected-KV
 * sparse decode": Summary, Motivation, "SM90 packing kernel", "Packed
 * attention specialization").  The selection is resolved once, ahead of the
 * attention, by mla_pack_selected_kv, which copies every selected record
 * byte for byte into a caller-owned workspace; the packed attention then
 * reads records at fixed positions, with no index load, check or page
 * translation.  The two calls are separate so a caller can run the pack on
 * another stream, overlapped with earlier work, and order it before the
 * attention with an event.
 *
 * Packed workspace (opaque to callers; fixed here so tests can check it):
 *   tiles = ceil(topk / 64), n_units = batch * s_q.
 *   records: uint8 [n_units, tiles, 64, 656]; slot t of unit u at record
 *            u * tiles * 64 + t.  Valid slots hold the selected record's 656
 *            bytes, every other slot (past topk_length, index -1, a bad
 *            index, the padding up to tiles * 64) holds 656 zero bytes.
 *   masks:   uint64 [n_units, tiles], right after the records; bit j of
 *            mask [u][k] is set iff slot 64k + j of unit u is valid.
 * The pages pack a valid prefix and zero-fill its suffix; the per-tile masks
 * here also carry -1 entries inside the prefix, so the packed result equals
 * the native sparse result for every selection the native call accepts. */
size_t mla_packed_kv_workspace_bytes(int n_units, int topk);

/* Pack the selection of every query token into the packed workspace.
 *   d_kv8, num_pages, d_indices, topk, d_topk_length: as for
 *                 mla_sparse_fp8_decode_fwd; n_units = batch * s_q.
 *   d_packed      16-byte aligned, >= mla_packed_kv_workspace_bytes(n_units,
 *                 topk) bytes; every byte of that size is written.
 * An index outside [-1, num_pages*64) is packed as masked and reported in
 * *d_status as MLA_ERR_BAD_INDEX (stream-ordered).  A tile whose record
 * copies do not land within the wait budget is reported as MLA_ERR_TIMEOUT
 * and gets a zero mask (its records are not written); the results of a call
 * that reports it must not be used.
 * MLA_ERR_UNSUPPORTED (before any launch) when num_pages * 64 exceeds
 * 2^31 - 1 (slot indices are int32). */
int mla_pack_selected_kv(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int topk,
                         const int32_t* d_topk_length, int n_units, void* d_packed, size_t packed_bytes,
                         int32_t* d_status, mla_stream_t stream);

/* Test hook for the device timeout path (no counterpart on the pages: it
 * exists so that a test can make a bounded wait run out on a real GPU
 * without faulting or hanging it).  Same arguments and checks as
 * mla_pack_selected_kv, but every block of its pack kernel withholds the
 * arrival that completes its bulk-copy barrier: the block's 200 us bounded
 * wait runs out, it writes MLA_ERR_TIMEOUT to *d_status and a zero mask for
 * its tile, then makes the withheld arrival, waits (bounded) until its own
 * copies have landed and exits without storing records.  The context and
 * the stream stay usable; the records region is left as it was. */
int mla_test_pack_timeout(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int topk,
                          const int32_t* d_topk_length, int n_units, void* d_packed, size_t packed_bytes,
                          int32_t* d_status, mla_stream_t stream);

/* Test hook for the dense decode kernel's timeout and unwind path (no
 * counterpart on the pages).  Same arguments and checks as
 * mla_decode_splits, for a bf16 cache or a cache of FP8 records (else
 * MLA_ERR_UNSUPPORTED before any launch).  bf16: an instance of the dense
 * kernel whose K producer never loads the first own tile of each CTA and
 * whose waits have a 200 us budget: the Q K^T thread's wait for that tile
 * runs out, the CTA writes MLA_ERR_TIMEOUT to *d_status and unwinds (every
 * role leaves its loop, the copies it issued land, the MMAs it issued
 * complete, TMEM is released), its peer CTA's waits for messages that never
 * come run out the same way, and the grid ends.  FP8 records: an instance
 * of the sparse kernel (the one such a cache runs) that never computes the
 * first tile's scores, with the same 200 us budgets and the same unwinding.
 * The context and the stream stay usable; out, lse and the workspace are
 * unspecified. */
int mla_test_decode_timeout(const void* d_q, const void* d_kv, const int32_t* d_block_table, int max_pages,
                            int num_pages, const int32_t* d_cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                            int dtype, int causal, float softmax_scale, const int32_t* d_sched,
                            const int32_t* d_split_offset, int num_parts, void* d_workspace, size_t workspace_bytes,
                            void* d_out, int out_type, float* d_lse, int32_t* d_status, mla_stream_t stream);

/* Sparse FP8 decode over a packed workspace (FlashMLA PR #200, "Packed
 * attention specialization": the packed attention reuses the native
 * dequantisation, softmax, split and combine pipeline and only replaces the
 * index/page/gather loader with direct loads of the packed tiles).  The same
 * kernel as mla_sparse_fp8_decode_fwd runs with slot t of unit u read from
 * packed record u * tiles * 64 + t and masked by its mask bit: the scores stay
 * exact in codes and scales, and under the same plan the result equals the
 * native call's on the same selection bit for bit.  d_topk_length must be
 * the one given to the pack (the plan counts each unit's tiles from it;
 * entries above topk are allowed, only the first topk slots exist); the plan
 * comes from mla_get_metadata exactly as for the native call (the pages'
 * H=128 packed path keeps the native scheduler).  h_q <= 128.  A bad index
 * was reported by the pack; this call reports none.  Other arguments as for
 * mla_sparse_fp8_decode_fwd. */
int mla_sparse_fp8_packed_decode_fwd(const void* d_q, const void* d_packed, size_t packed_bytes, int topk,
                                     const int32_t* d_topk_length, int batch, int s_q, int h_q, float softmax_scale,
                                     const int32_t* d_sched, const int32_t* d_split_offset, int num_parts,
                                     void* d_workspace, size_t workspace_bytes, void* d_out, float* d_lse,
                                     int32_t* d_status, mla_stream_t stream);

/* Gather + unpack of selected records to fp32 key rows, bit-exact:
 * k[d] = fp32(e4m3[d]) * scale[d/128] as one fp32 round-to-nearest-even
 * multiply (d < 512), k[512+e] = fp32(bf16 rope[e]).  Index -1 or an index
 * outside the pool gives a zero row (the latter also MLA_ERR_BAD_INDEX).
 *   d_indices int32 [n], d_k_out fp32 [n, 576].
 * MLA_ERR_UNSUPPORTED (before any launch) when num_pages * 64 exceeds
 * 2^31 - 1. */
int mla_sparse_fp8_unpack(const uint8_t* d_kv8, int num_pages, const int32_t* d_indices, int n, float* d_k_out,
                          int32_t* d_status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PAGED_KV_H_ */
