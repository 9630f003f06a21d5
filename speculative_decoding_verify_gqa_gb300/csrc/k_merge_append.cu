// LSE merge of split partials, and the paged K/V append.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/verify_attn.h"
#include "va_device.cuh"
#include "va_kernels.h"

namespace va {
namespace {

// Merge ("flashmap 0.1.0 -- flashmap/sglang/verify_attention.py", merge
// kernel): for each row, m = max_s lse_s, w_s = e^(lse_s - m), out =
// sum_s w_s out_s / sum_s w_s, lse = m + ln sum_s w_s; splits with lse = -inf
// carry no mass, and a row with no mass at all gets out = 0, lse = -inf.
// One warp per row; each lane owns D / 32 consecutive output elements.  The
// splits are read CH at a time, LSE and partial output together, with a
// running max (sums rescaled when it rises), so a row of up to CH splits costs
// one round trip to memory.
// CH: splits whose loads are issued together, chosen from the plan's largest
// split count -- enough to merge a row in one round trip, and no more, since
// the loaded rows live in registers and the registers bound how many rows
// are in flight.
template <int D, int CH>
__global__ void __launch_bounds__(128) verify_merge_kernel(const MergeParams p) {
  constexpr int V = D / 32;
  // After this library's split kernel in an append-and-run call, the merge
  // list (uploaded with the plan) and qo_indptr are read before the wait for
  // it: no kernel of the step writes them.  A call of its own waits first.
  grid_dependents_launch();  // the next kernel may be scheduled; it waits for our completion
  if (!p.early_inputs) grid_dependency_wait();
  const MergeItem it = p.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 4 + warp;
  // a merge list left in the workspace by another plan: nothing outside this
  // call's tables and partial rows is read or written
  const bool item_ok = it.b >= 0 && it.b < p.batch && it.h >= 0 && it.h < p.h_kv &&
                       it.part_row0 >= 0 && it.nsplit >= 1 && it.row0 >= 0 &&
                       (long long)it.part_row0 + (long long)it.nsplit * it.nrows <= p.part_rows;
  const int qo0 = item_ok ? p.qo_indptr[it.b] : 0;
  const bool row_ok = item_ok && r < it.nrows &&
                      (it.row0 + r) / p.group < p.qo_indptr[it.b + 1] - qo0;
  // the partials come from the preceding split kernel; every thread waits,
  // so that this grid's completion implies that kernel's
  grid_dependency_wait();
  if (!row_ok) return;
  const float* lse_base = p.part_lse + it.part_row0 + r;
  float m = -INFINITY, den = 0.f;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < it.nsplit; s0 += CH) {
    float ls[CH];
    float x[CH][V];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int s = s0 + c;
      ls[c] = -INFINITY;
#pragma unroll
      for (int i = 0; i < V; ++i) x[c][i] = 0.f;
      if (s < it.nsplit) {
        ls[c] = lse_base[(size_t)s * it.nrows];
        const float* src = p.part_out + ((size_t)it.part_row0 + (size_t)s * it.nrows + r) * D + lane * V;
        if constexpr (V == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          x[c][0] = v.x; x[c][1] = v.y; x[c][2] = v.z; x[c][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          x[c][0] = v.x; x[c][1] = v.y;
        }
      }
    }
    float cm = -INFINITY;
#pragma unroll
    for (int c = 0; c < CH; ++c) cm = fmaxf(cm, ls[c]);
    if (cm == -INFINITY) continue;  // no split of this chunk carries mass
    if (cm > m) {
      const float sc = ex2((m - cm) * kLog2e);  // 0 while m = -inf
      den *= sc;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] *= sc;
      m = cm;
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (ls[c] == -INFINITY) continue;  // an empty split carries no mass
      const float w = ex2((ls[c] - m) * kLog2e);
      den += w;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += w * x[c][i];
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const int rr = it.row0 + r;
  const int t = rr / p.group, g = rr - t * p.group;
  const size_t orow = (size_t)(qo0 + t) * p.h_q + (size_t)it.h * p.group + g;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + orow * D + lane * V;
  if constexpr (V == 4) {
    uint2 v;
    v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = v;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (p.lse && lane == 0) p.lse[orow] = den > 0.f ? m + logf(den) : -INFINITY;
}

// Paged append (vLLM PR #1679: every draft's K/V is cached before attention;
// FlashInfer PR #286's page table).  One thread per 16-byte chunk of one
// (token, KV head) cache row, for K and V: slot pos % P of page
// kv_indices[kv_indptr[b] + pos / P], pos = kv_len_b - n_b + i, in the HND
// ([page][head][slot]) or NHD ([page][slot][head]) layout.  A plain append is
// a bit-exact copy.  A quantising append (FlashInfer PR #286's fp8 cache with
// a per-tensor scale) reads bf16 rows and stores e4m3(x / scale): the
// correctly rounded binary32 quotient converted with round-to-nearest-even
// and saturation to +-448.  With positions, K rows are rotated first (RoPE,
// LLaMA's rotate-half pairing (i, i + d/2) at angle position * theta^(-2i/d)
// / rope_scale, FlashInfer PR #286's ROPE_LLAMA, at the tree positions
// FlashInfer issue #152 asks for), in fp32, then rounded to the cache dtype.
__device__ __forceinline__ void load_f32(const uint8_t* row, int bf16_src, int e0, int n, float* x) {
  if (bf16_src) {
    const uint4* s4 = reinterpret_cast<const uint4*>(row + 2 * e0);
    for (int c = 0; c < n / 8; ++c) {
      const uint4 w = s4[c];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[8 * c + 2 * k] = __uint_as_float(u[k] << 16);
        x[8 * c + 2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
      }
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(row + e0);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t hv = e4m3x2_to_f16x2((uint16_t)(u[k] >> (16 * j)));
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hv));
        x[4 * k + 2 * j] = f.x;
        x[4 * k + 2 * j + 1] = f.y;
      }
    }
  }
}

__global__ void __launch_bounds__(256) paged_kv_append_kernel(const AppendParams p) {
  // Launched with programmatic serialization: nothing the kernel before this
  // one may produce (the new rows, q, the tables) is read before it has
  // completed, and the attention kernel after this one is released right
  // then: it may read q and the prefix pages at once, and waits for our
  // completion before it reads a draft's slot.  When the caller promises
  // that the step's inputs (q, the new rows, the tables) were complete
  // before that kernel started (early), the next kernel is released at once
  // and the tables and new rows are read before the wait; the slots are
  // still written after it.
  if (!p.early) grid_dependency_wait();
  grid_dependents_launch();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per_tok = (long long)p.h_kv * p.row_chunks;
  if (idx >= p.total_new * per_tok) return;
  const int i = (int)(idx / per_tok);
  const int rem = (int)(idx - (long long)i * per_tok);
  const int h = rem / p.row_chunks, ch = rem - h * p.row_chunks;
  // request of token i: the last b with append_indptr[b] <= i
  int lo = 0, hi = p.batch;  // invariant: append_indptr[lo] <= i < append_indptr[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.append_indptr + mid) <= i) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int a0 = __ldg(p.append_indptr + b);
  const int n = __ldg(p.append_indptr + b + 1) - a0;
  const int pg0 = __ldg(p.kv_indptr + b);
  const int npg = __ldg(p.kv_indptr + b + 1) - pg0;
  const int lpl = npg > 0 ? __ldg(p.last_page_len + b) : 0;
  const long long kv_len = npg > 0 ? (long long)(npg - 1) * p.page_size + lpl : 0;
  const long long pos = kv_len - n + (i - a0);
  const bool pos_ok = !(i < a0 || i - a0 >= n || pos < 0 || (npg > 0 && (lpl < 1 || lpl > p.page_size)) ||
                        (pos >> p.log2_page) >= npg);
  const int page = pos_ok ? __ldg(p.kv_indices + pg0 + (int)(pos >> p.log2_page)) : -1;
  if (!pos_ok || (unsigned)page >= (unsigned)p.num_pages) {
    if (p.early) grid_dependency_wait();
    if (p.status) atomicOr(p.status, pos_ok ? VA_DEV_BAD_PAGE : VA_DEV_BAD_APPEND);
    return;
  }
  // K rows hold head_dim elements, V rows head_dim_v: this thread's chunk
  // ch of each row that has one
  const bool do_k = ch < p.k_chunks, do_v = ch < p.v_chunks;
  const size_t slot = (size_t)(pos & (p.page_size - 1));
  const size_t row = p.nhd ? ((size_t)page * p.page_size + slot) * p.h_kv + h
                           : ((size_t)page * p.h_kv + h) * p.page_size + slot;
  uint8_t* kd = static_cast<uint8_t*>(p.k_cache) + row * (size_t)p.k_chunks * 16 + (size_t)ch * 16;
  uint8_t* vd = static_cast<uint8_t*>(p.v_cache) + row * (size_t)p.v_chunks * 16 + (size_t)ch * 16;
  const int D = p.head_dim;
  const bool bf16_src = p.quant || !p.cache_fp8;
  const size_t src_es = bf16_src ? 2 : 1;
  const uint8_t* ks = static_cast<const uint8_t*>(p.k_new) + ((size_t)i * p.h_kv + h) * (size_t)D * src_es;
  const uint8_t* vs = static_cast<const uint8_t*>(p.v_new) +
                      ((size_t)i * p.h_kv + h) * (size_t)p.head_dim_v * src_es;
  if (!p.quant && !p.positions) {  // a bit-exact copy
    const uint4 kq = do_k ? *reinterpret_cast<const uint4*>(ks + (size_t)ch * 16) : make_uint4(0, 0, 0, 0);
    const uint4 vq = do_v ? *reinterpret_cast<const uint4*>(vs + (size_t)ch * 16) : make_uint4(0, 0, 0, 0);
    if (p.early) grid_dependency_wait();   // the slots may still be read before it
    if (do_k) *reinterpret_cast<uint4*>(kd) = kq;
    if (do_v) *reinterpret_cast<uint4*>(vd) = vq;
    return;
  }
  // elements e0 .. e0 + E - 1 of the row: 8 for a bf16 cache, 16 for fp8
  const int E = p.cache_fp8 ? 16 : 8;
  const int e0 = ch * E;
  float xk[16] = {}, xv[16] = {};
  if (do_k) load_f32(ks, bf16_src, e0, E, xk);
  if (do_v) load_f32(vs, bf16_src, e0, E, xv);
  if (p.positions && do_k) {
    const int half = D / 2;
    const int partner = e0 < half ? e0 + half : e0 - half;
    float yk[16];
    load_f32(ks, bf16_src, partner, E, yk);
    const int kpos = __ldg(p.positions + i);
    const float sgn = e0 < half ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (e >= E) break;
      const int j = (e0 + e) & (half - 1);
      float c, s;
      rope_cos_sin(kpos, p.rope.hi[j], p.rope.lo[j], &c, &s);
      xk[e] = fmaf(xk[e], c, sgn * yk[e] * s);
    }
  }
  if (p.early) grid_dependency_wait();   // the slots may still be read before it
  if (!p.cache_fp8) {
    uint4 wk, wv;
    wk.x = pack_bf16x2(xk[0], xk[1]); wk.y = pack_bf16x2(xk[2], xk[3]);
    wk.z = pack_bf16x2(xk[4], xk[5]); wk.w = pack_bf16x2(xk[6], xk[7]);
    wv.x = pack_bf16x2(xv[0], xv[1]); wv.y = pack_bf16x2(xv[2], xv[3]);
    wv.z = pack_bf16x2(xv[4], xv[5]); wv.w = pack_bf16x2(xv[6], xv[7]);
    if (do_k) *reinterpret_cast<uint4*>(kd) = wk;
    if (do_v) *reinterpret_cast<uint4*>(vd) = wv;
    return;
  }
  // e4m3 codes: quantising appends divide by the per-tensor scale first (a
  // copy of fp8 rows that were only rotated keeps their scale)
  const float ksc = p.quant ? p.k_scale : 1.f, vsc = p.quant ? p.v_scale : 1.f;
  uint32_t ck[4], cv[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ck[k] = e4m3x4_rn_satfinite(__fdiv_rn(xk[4 * k], ksc), __fdiv_rn(xk[4 * k + 1], ksc),
                                __fdiv_rn(xk[4 * k + 2], ksc), __fdiv_rn(xk[4 * k + 3], ksc));
    cv[k] = e4m3x4_rn_satfinite(__fdiv_rn(xv[4 * k], vsc), __fdiv_rn(xv[4 * k + 1], vsc),
                                __fdiv_rn(xv[4 * k + 2], vsc), __fdiv_rn(xv[4 * k + 3], vsc));
  }
  if (do_k) *reinterpret_cast<uint4*>(kd) = make_uint4(ck[0], ck[1], ck[2], ck[3]);
  if (do_v) *reinterpret_cast<uint4*>(vd) = make_uint4(cv[0], cv[1], cv[2], cv[3]);
}

}  // namespace

template <int D>
static cudaError_t launch_merge_d(const MergeParams& p, int n_merge, int block_rows,
                                  int max_nsplit, cudaStream_t stream) {
  dim3 grid(n_merge, (block_rows + 3) / 4);
  void* args[] = {const_cast<MergeParams*>(&p)};
  const void* k = max_nsplit <= 4   ? reinterpret_cast<const void*>(verify_merge_kernel<D, 4>)
                  : max_nsplit <= 8 ? reinterpret_cast<const void*>(verify_merge_kernel<D, 8>)
                                    : reinterpret_cast<const void*>(verify_merge_kernel<D, 24>);
  return launch_kernel(k, grid, dim3(128), 0, stream, args, /*pdl=*/true);
}

cudaError_t launch_merge(const MergeParams& p, int head_dim, int n_merge, int block_rows,
                         int max_nsplit, cudaStream_t stream) {
  if (n_merge <= 0) return cudaSuccess;
  if (head_dim == 128) return launch_merge_d<128>(p, n_merge, block_rows, max_nsplit, stream);
  if (head_dim == 64) return launch_merge_d<64>(p, n_merge, block_rows, max_nsplit, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const long long threads = p.total_new * (long long)p.h_kv * p.row_chunks;
  if (threads <= 0) return cudaSuccess;
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  void* args[] = {const_cast<AppendParams*>(&p)};
  return launch_kernel(reinterpret_cast<const void*>(paged_kv_append_kernel),
                       dim3((unsigned)blocks), dim3(256), 0, stream, args, /*pdl=*/true);
}

}  // namespace va
