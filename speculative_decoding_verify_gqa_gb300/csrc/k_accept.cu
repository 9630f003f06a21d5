// Greedy acceptance of speculative draft trees against the target model's
// logits: the step after verification (FlashInfer issue #152: Medusa / EAGLE
// trees are verified against the target model's outputs).  Request b's nodes
// are logits rows qo_indptr[b] .. qo_indptr[b+1]; node 0 is the root (the
// last accepted token), parents[i] < i, draft_tokens[i] the token node i
// proposes.  The root is accepted; node i is accepted iff its parent is and
// the argmax of the parent's row (first index among equal maxima) equals
// draft_tokens[i].  The accepted path ends at the deepest accepted node (the
// smallest index among equally deep ones) and the bonus token is the argmax
// of that node's row.
//
// Two kernels: the argmax of every row, each row cut into chunks over
// several CTAs (16-byte loads; each chunk's winner kept as a 64-bit key, the
// order-preserving image of the value above the complement of the index, so
// the largest key is the largest value at the smallest index), then one warp
// per request reduces its rows' chunk keys and walks the tree.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/verify_attn.h"
#include "va_device.cuh"
#include "va_kernels.h"

namespace va {
namespace {

// Order-preserving map of an fp32 bit pattern to uint32 (total order of the
// real values; -0 below +0).
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t argmax_key(float v, uint32_t idx) {
  return ((uint64_t)ordered_bits(v) << 32) | (uint64_t)(0xffffffffu - idx);
}
__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

template <bool BF16>
__global__ void __launch_bounds__(256) accept_argmax_kernel(const AcceptParams p) {
  const int row = blockIdx.y, chunk = blockIdx.x;
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t c0 = (int64_t)chunk * p.chunk_elems;
  const int64_t c1 = min((int64_t)p.vocab, c0 + p.chunk_elems);
  uint64_t best = 0;  // below every key of a real value
  if (row < p.total) {
    const uint8_t* base = static_cast<const uint8_t*>(p.logits) + (size_t)row * p.row_stride * (BF16 ? 2 : 4);
    constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte load
    // 16-byte loads over the aligned middle of [c0, c1), single elements at the ends
    const uintptr_t addr0 = reinterpret_cast<uintptr_t>(base) + (uintptr_t)c0 * (BF16 ? 2 : 4);
    int64_t head = (int64_t)(((16 - (addr0 & 15)) & 15) / (BF16 ? 2 : 4));
    if (((addr0 & 15) % (BF16 ? 2 : 4)) != 0) head = c1 - c0;   // not element-aligned to 16: all scalar
    head = min(head, c1 - c0);
    const int64_t nvec = (c1 - c0 - head) / EPV;
    const int64_t v0 = c0 + head, v1 = v0 + nvec * EPV;
    auto scalar = [&](int64_t e) {
      const float v = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(base)[e] << 16)
                           : reinterpret_cast<const float*>(base)[e];
      best = umax64(best, argmax_key(v, (uint32_t)e));
    };
    for (int64_t e = c0 + threadIdx.x; e < v0; e += blockDim.x) scalar(e);
    for (int64_t e = v1 + threadIdx.x; e < c1; e += blockDim.x) scalar(e);
    const uint4* vp = reinterpret_cast<const uint4*>(base + (size_t)v0 * (BF16 ? 2 : 4));
#pragma unroll 4
    for (int64_t k = threadIdx.x; k < nvec; k += blockDim.x) {
      const uint4 w = __ldg(vp + k);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
      const uint32_t e = (uint32_t)(v0 + k * EPV);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (BF16) {
          best = umax64(best, argmax_key(__uint_as_float(u[q] << 16), e + 2 * q));
          best = umax64(best, argmax_key(__uint_as_float(u[q] & 0xffff0000u), e + 2 * q + 1));
        } else {
          best = umax64(best, argmax_key(__uint_as_float(u[q]), e + q));
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, off));
  __shared__ uint64_t warp_best[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) warp_best[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0 && row < p.total) {
    uint64_t b = warp_best[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) b = umax64(b, warp_best[w]);
    p.keys[(size_t)row * p.chunks + chunk] = b;
  }
}

// One warp per request: reduce each node's chunk keys to its argmax, then
// lane 0 walks the nodes in index order (parents come first).
__global__ void __launch_bounds__(128) accept_walk_kernel(const AcceptParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * 4 + warp;
  if (b >= p.batch) return;
  const int o = p.qo_indptr[b];
  const int L = p.qo_indptr[b + 1] - o;
  if (L < 0 || o < 0 || (int64_t)o + L > p.total) {
    if (lane == 0) {
      p.accept_len[b] = 0;
      p.bonus[b] = -1;
      if (p.status) atomicOr(p.status, VA_DEV_BAD_TABLE);
    }
    return;
  }
  for (int i = lane; i < L; i += 32) {
    const uint64_t* k = p.keys + (size_t)(o + i) * p.chunks;
    uint64_t best = 0;
    for (int c = 0; c < p.chunks; ++c) best = umax64(best, k[c]);
    const int am = (int)(0xffffffffu - (uint32_t)best);
    p.node_am[o + i] = am;
    if (p.argmax_out) p.argmax_out[o + i] = am;
  }
  __syncwarp();
  if (lane != 0) return;
  if (L == 0) {
    p.accept_len[b] = 0;
    p.bonus[b] = -1;
    return;
  }
  // node_state[o + i]: depth if accepted, -1 if not
  int best = -1, best_depth = -1;
  bool ok = true;
  for (int i = 0; i < L; ++i) {
    const int par = p.parents[o + i];
    int d = -1;
    if (i == 0) {
      ok = ok && par < 0;
      d = 0;
    } else if (par < 0 || par >= i) {
      ok = false;
    } else {
      const int dp = p.node_state[o + par];
      if (dp >= 0 && p.node_am[o + par] == p.draft_tokens[o + i]) d = dp + 1;
    }
    p.node_state[o + i] = d;
    if (d > best_depth) {
      best_depth = d;
      best = i;
    }
  }
  if (!ok) {
    p.accept_len[b] = 0;
    p.bonus[b] = -1;
    if (p.status) atomicOr(p.status, VA_DEV_BAD_TABLE);
    return;
  }
  p.accept_len[b] = best_depth + 1;
  p.bonus[b] = p.node_am[o + best];
  for (int j = best, k = best_depth; j >= 0 && k >= 0; j = p.parents[o + j], --k) p.path[o + k] = j;
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, bool bf16, cudaStream_t stream) {
  if (p.total > 0) {
    dim3 grid((unsigned)p.chunks, (unsigned)p.total);
    void* args[] = {const_cast<AcceptParams*>(&p)};
    const void* k = bf16 ? reinterpret_cast<const void*>(accept_argmax_kernel<true>)
                         : reinterpret_cast<const void*>(accept_argmax_kernel<false>);
    cudaError_t e = launch_kernel(k, grid, dim3(256), 0, stream, args, /*pdl=*/true);
    if (e != cudaSuccess) return e;
  }
  if (p.batch <= 0) return cudaSuccess;
  void* args[] = {const_cast<AcceptParams*>(&p)};
  return launch_kernel(reinterpret_cast<const void*>(accept_walk_kernel), dim3((p.batch + 3) / 4),
                       dim3(128), 0, stream, args, /*pdl=*/true);
}

}  // namespace va
