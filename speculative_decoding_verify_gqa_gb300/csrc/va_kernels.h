// Kernel parameter blocks and host-side launchers (internal to
// libverify_attn.so).  Every pointer is a device pointer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "va_internal.h"

namespace va {

// RoPE frequencies theta^(-2i/d) / rope_scale, i < d/2, as float pairs hi + lo
// (computed in double on the host), so that position * frequency keeps ~46
// bits before the angle is reduced.
struct RopeFreq {
  float hi[64], lo[64];
};

struct PartialParams {
  const void* q;              // [total_qo, h_q, D] bf16
  const void* k_cache;        // [num_pages, h_kv, P, D] bf16 / fp8
  const void* v_cache;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_len;
  const int32_t* qo_indptr;
  const uint8_t* mask;        // nullable: causal drafts
  const int32_t* mask_indptr;
  void* out;                  // [total_qo, h_q, D] bf16
  float* lse;                 // nullable
  const WorkItem* items;
  float* part_out;            // [part_rows, D]
  float* part_lse;            // [part_rows]
  int* status;                // device status word
  int batch;                  // requests in the plan: a work item's b must be below it
  int64_t part_rows;          // partial rows in the workspace: a split item's rows lie below
  int h_q, h_kv, group, page_size, log2_page, num_pages;
  float scale_log2;           // sm_scale * k_scale * log2(e)
  float scale_nat;            // sm_scale * k_scale
  float v_scale;
  int n_items;                // work items in `items`
  int n_ctas;                 // persistent tcgen05 variants: item chains (see WorkItem::next)
  int mask_full;              // mask rows hold kv_len bits, prefix included
  int nhd;                    // cache layout [pages, P, h_kv, d]
  const int32_t* q_position;  // nullable: RoPE position of each query token
  int early_inputs;           // 1: q, the tables and the prefix pages may be read before the
                              // wait for the previous grid (this library's append, released
                              // once q's producer is done, or a caller's early-reads promise)
  RopeFreq rope;              // frequencies when q_position is set
  int drafts_new;             // tcgen05 variants: an item of drafts only (kv_lo >= prefix)
                              // reads its keys and values from the new rows (TcMaps kn / vn,
                              // [total_qo, h_kv, D] in the cache dtype) instead of the pages
  int total_qo;               // rows of q (and of the new K / V)
};

struct MergeParams {
  const MergeItem* items;
  const float* part_out;
  const float* part_lse;
  const int32_t* qo_indptr;
  void* out;
  float* lse;                 // nullable
  int64_t part_rows;          // partial rows in the workspace
  int batch, h_q, h_kv, group;
  int early_inputs;           // 1: the merge list and qo_indptr may be read before the wait
};

struct AppendParams {
  const void* k_new;
  const void* v_new;
  const int32_t* append_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_len;
  void* k_cache;
  void* v_cache;
  int* status;                // nullable
  const int32_t* positions;   // nullable: RoPE position of each new token's key
  int batch, h_kv, page_size, log2_page, num_pages;
  int row_chunks;             // threads per (token, head): max(k_chunks, v_chunks)
  int k_chunks, v_chunks;     // 16-byte chunks of a K / V cache row
  int head_dim, head_dim_v;   // elements of a K / V row
  int cache_fp8;              // cache dtype e4m3 (else bf16)
  int quant;                  // bf16 source rows into an e4m3 cache
  int nhd;                    // cache layout [pages, P, h_kv, d] (else [pages, h_kv, P, d])
  int early;                  // 1: release the next kernel at once and read the tables before
                              // the wait (they do not depend on the previous kernel)
  float k_scale, v_scale;     // quantising append: stored = e4m3(x / scale)
  int64_t total_new;
  RopeFreq rope;
};

// Greedy acceptance (see k_accept.cu).
struct AcceptParams {
  const void* logits;         // [total, row_stride] bf16 or fp32
  const int32_t* qo_indptr;   // [batch + 1] rows of each request
  const int32_t* draft_tokens;  // [total]
  const int32_t* parents;     // [total] local parent index, -1 for the root
  int32_t* accept_len;        // [batch]
  int32_t* path;              // [total]: request b's accepted path at qo_indptr[b] ..
  int32_t* bonus;             // [batch]
  int32_t* argmax_out;        // nullable [total]
  int* status;                // nullable
  uint64_t* keys;             // workspace [total, chunks]
  int32_t* node_am;           // workspace [total]
  int32_t* node_state;        // workspace [total]
  int64_t row_stride;         // elements between rows
  int total, vocab, batch, chunks;
  int64_t chunk_elems;
};
cudaError_t launch_accept(const AcceptParams& p, bool bf16, cudaStream_t stream);

// Launch `func` with void** args; pdl = true lets the grid be scheduled
// before the previous kernel in the stream finishes (programmatic dependent
// launch); such kernels call grid_dependency_wait() before touching memory.
inline cudaError_t launch_kernel(const void* func, dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, void** args, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, func, args);
}

// Launchers: return the launch's cudaError_t (cudaErrorInvalidValue for a
// variant that is not compiled).
cudaError_t launch_partial_mma(const PartialParams& p, int kernel, int head_dim, int head_dim_v,
                               bool kv_fp8, int n_items, cudaStream_t stream);

// TMA descriptors of the tensor-core variant: q as [total_qo, h_q, 128] bf16
// with 64 x G x (128 / G) boxes, 128-byte swizzle.  A bf16 cache
// [num_pages, h_kv, P, 128] is viewed as the 5-D tensor
// [num_pages * h_kv][P / 8][2][8][64] (page-and-head, 8-slot group, 64-column
// half, slot in group, column; the half stride, 128 bytes, is below the slot
// stride) with 64 x 8 x 2 x 2 x 1 boxes and 128-byte swizzle: one box per 16
// keys lands as [8-key group][half][8 keys][128 bytes], 8-key groups 2048
// bytes apart and halves 1024 -- a uniform layout that both MMAs read (K
// K-major, V MN-major), in one 4 KB copy per 16 keys.  An fp8 cache keeps the
// 4-D view [num_pages, h_kv, P, 128] with 128 x 16 x 1 x 1 boxes (no swizzle).
// Zero fill out of bounds.  With e4m3 MMAs (plan option q_fp8) the fp8
// boxes land with 128-byte swizzle, as the MMA operands.
//
// kn / vn (drafts_new): the new K / V rows [total_qo, h_kv, D].  bf16: 4-D
// [total_qo][half][h_kv] x 64 with 64 x 8 x 2 x 1 boxes and 128-byte swizzle,
// one box per 8 tokens landing as one 8-key group [half][8][128 bytes] of the
// page tiles' layout; fp8: 3-D [total_qo][h_kv] x 128 with 128 x 16 x 1
// boxes, one per 16 tokens, swizzled as the fp8 page boxes.
struct TcMaps {
  CUtensorMap q, k, v, kn, vn;
};
cudaError_t launch_partial_tc(const PartialParams& p, const TcMaps& maps, bool kv_fp8,
                              int block_rows, int n_items, bool f8mma, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, int head_dim, int n_merge, int block_rows,
                         int max_nsplit, cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

}  // namespace va
