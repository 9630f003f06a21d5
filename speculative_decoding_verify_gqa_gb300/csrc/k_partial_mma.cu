// Split-KV verify attention over a paged KV cache: warp-level tensor-core
// variant (mma.sync m16n8k16 bf16 -> fp32).
//
// Algorithm ("flashmap 0.1.0 -- flashmap/sglang/verify_attention.py", partial
// kernel): one CTA per work item (request b, KV head h, block of rows, kv
// chunk [lo, hi)).  The block's rows are every query head h*G .. h*G+G-1 of
// the request's draft tokens, so each key / value row fetched from HBM serves
// all G heads (GQA, vLLM PR #2401).  The chunk is walked in tiles of 64 keys:
// S = Q K^T, mask, online softmax in fp32 (running max m and sum l, rescaled
// accumulator), acc += P V.  The chunk's result is written either as the final
// bf16 output and natural-log LSE (unsplit item) or as an fp32 normalised
// partial plus its LSE for the merge kernel.
//
// GB300 design: rows are token-major (row r = token r / G, head r % G) so a
// block's Q rows are G contiguous head vectors per token; page rows are
// gathered with 16-byte cp.async into a 3-stage shared-memory ring
// (XOR-swizzled for conflict-free ldmatrix), zero-filled past the chunk end
// (so stale or NaN page slots never reach the tensor cores); each warp owns 16
// rows and keeps Q, S and the output accumulator in registers; fp8-e4m3 pages
// are widened to bf16 in shared memory once per tile (exact), with k_scale
// folded into the logit scale and v_scale into the final normalisation.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/verify_attn.h"
#include "va_device.cuh"
#include "va_kernels.h"

namespace va {
namespace {

// D: elements of a query / key row; DV: of a value / output row (sglang's
// value head size, which may differ).
template <int D, int DV, bool FP8, int NW, int STAGES>
struct MmaCfg {
  static constexpr int BN = kTileKeys;            // keys per tile
  static constexpr int BM = 16 * NW;              // rows per CTA
  static constexpr int NT = 32 * NW;              // threads
  static constexpr int QROW = D * 2;              // bytes per bf16 Q / K row
  static constexpr int VROW = DV * 2;             // bytes per bf16 V row
  static constexpr int KVROW = FP8 ? D : 2 * D;   // bytes per K cache row
  static constexpr int VVROW = FP8 ? DV : 2 * DV; // bytes per V cache row
  static constexpr int KV_CH = KVROW / 16;        // 16-byte chunks per K cache row
  static constexpr int V_CH = VVROW / 16;         // 16-byte chunks per V cache row
  static constexpr int Q_CH = QROW / 16;
  static constexpr int Q_BYTES = BM * QROW;
  static constexpr int TILE_BYTES = BN * KVROW;   // one K tile in cache format
  static constexpr int VTILE_BYTES = BN * VVROW;  // one V tile in cache format
  static constexpr int STAGE_BYTES = TILE_BYTES + VTILE_BYTES;
  static constexpr int CONV_BYTES = FP8 ? BN * (QROW + VROW) : 0;
  static constexpr int RING_BYTES = STAGES * BN * 4;  // page id of every key of the tiles in flight
  static constexpr int SMEM = Q_BYTES + STAGES * STAGE_BYTES + CONV_BYTES + RING_BYTES;
  static_assert(BN == 64, "tile loop assumes 64 keys");
  static_assert(NT >= BN, "one thread per key fetches page ids");
};

template <int D, int DV, bool FP8, int NW, int STAGES>
__global__ void __launch_bounds__(32 * NW, NW == 4 ? 2 : 1)
    verify_partial_mma_kernel(const PartialParams p) {
  using C = MmaCfg<D, DV, FP8, NW, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sStage = smem + C::Q_BYTES;
  uint8_t* sConv = sStage + STAGES * C::STAGE_BYTES;
  int* sPage = reinterpret_cast<int*>(sConv + C::CONV_BYTES);  // [STAGES][BN]

  // Inputs (pages appended by the previous kernel, q, tables) may come from
  // the grid before this one in the stream.
  grid_dependency_wait();
  const WorkItem it = p.items[blockIdx.x];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = it.b, h = it.h;
  const int G = p.group;

  // Request geometry, from the device tables the caller passed (nothing is
  // read for a work item that names a request or head outside this call's
  // tables, as one left in the workspace by another plan may).
  const bool idx_ok = b >= 0 && b < p.batch && h >= 0 && h < p.h_kv;
  const int qo0 = idx_ok ? p.qo_indptr[b] : 0;
  const int L = idx_ok ? p.qo_indptr[b + 1] - qo0 : -1;
  const int pg0 = idx_ok ? p.kv_indptr[b] : 0;
  const int npg = idx_ok ? p.kv_indptr[b + 1] - pg0 : -1;
  const int lpl = npg > 0 ? p.last_page_len[b] : 1;
  const long long kv_len_ll = npg > 0 ? (long long)(npg - 1) * p.page_size + lpl : 0;
  const int kv_len = (int)kv_len_ll;
  const int prefix = kv_len - L;
  const bool ok = L >= 0 && npg >= 0 && lpl >= 1 && lpl <= p.page_size && prefix >= 0 &&
                  it.row0 >= 0 && it.nrows > 0 && it.nrows <= C::BM &&
                  (long long)it.row0 + it.nrows <= (long long)G * L && it.kv_lo >= 0 &&
                  it.kv_lo < it.kv_hi && it.kv_hi <= kv_len && kv_len_ll <= 0x7fffffffLL &&
                  (it.part_row < 0 || (long long)it.part_row + it.nrows <= p.part_rows);
  if (!ok) {
    if (tid == 0) atomicOr(p.status, VA_DEV_BAD_TABLE);
    return;
  }

  const int nrows = it.nrows, row0 = it.row0;
  const int lo = it.kv_lo, hi = it.kv_hi;
  const int n_tiles = (hi - lo + C::BN - 1) / C::BN;
  // HND [page][head][slot][d] or NHD [page][slot][head][d]
  // (element strides are the same for K and V; the row widths differ)
  const size_t slot_rows = p.nhd ? (size_t)p.h_kv : 1;
  const size_t head_rows = p.nhd ? (size_t)h : (size_t)h * p.page_size;
  const size_t page_rows = (size_t)p.h_kv * p.page_size;
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k_cache) + head_rows * C::KVROW;
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v_cache) + head_rows * C::VVROW;
  const int pmask = p.page_size - 1;
  int bad_page = 0;

  // Q rows of the block -> shared memory (zero past nrows).
  for (int c = tid; c < C::BM * C::Q_CH; c += C::NT) {
    const int r = c / C::Q_CH, ch = c % C::Q_CH;
    const uint8_t* src = static_cast<const uint8_t*>(p.q);
    int bytes = 0;
    if (r < nrows) {
      const int rr = row0 + r;
      const int t = rr / G, g = rr - t * G;
      src += (((size_t)(qo0 + t) * p.h_q + (size_t)h * G + g) * D) * 2 + ch * 16;
      bytes = 16;
    }
    cp_async_16(smem_u32(sQ + swz(r, ch, C::QROW)), src, bytes);
  }
  cp_async_commit();

  // Page id of one key of a tile (-1 past the chunk end).
  auto page_of = [&](int tile, int r) -> int {
    const int key = lo + tile * C::BN + r;
    return (tile < n_tiles && key < hi) ? __ldg(p.kv_indices + pg0 + (key >> p.log2_page)) : -1;
  };
  // Issue the K and V rows of a tile from the page ids in its ring slot.
  auto issue_tile = [&](int tile, int stage) {
    const int k0 = lo + tile * C::BN;
    const int* pages = sPage + (tile % STAGES) * C::BN;
    uint8_t* sK = sStage + stage * C::STAGE_BYTES;
    uint8_t* sV = sK + C::TILE_BYTES;
    constexpr int CH = C::KV_CH > C::V_CH ? C::KV_CH : C::V_CH;  // chunks of the wider row
#pragma unroll 4
    for (int c = tid; c < C::BN * CH; c += C::NT) {
      const int r = c / CH, ch = c % CH;
      const int key = k0 + r;
      size_t row = 0;
      int bytes = 0;
      if (key < hi) {
        const int page = pages[r];
        if ((unsigned)page < (unsigned)p.num_pages) {
          row = (size_t)page * page_rows + (size_t)(key & pmask) * slot_rows;
          bytes = 16;
        } else {
          bad_page = 1;
        }
      }
      if (C::KV_CH == CH || ch < C::KV_CH) {
        const uint32_t doff = FP8 ? (uint32_t)(r * C::KVROW + ch * 16) : swz(r, ch, C::QROW);
        cp_async_16(smem_u32(sK + doff), bytes ? kbase + row * C::KVROW + ch * 16 : kbase, bytes);
      }
      if (C::V_CH == CH || ch < C::V_CH) {
        const uint32_t doff = FP8 ? (uint32_t)(r * C::VVROW + ch * 16) : swz(r, ch, C::VROW);
        cp_async_16(smem_u32(sV + doff), bytes ? vbase + row * C::VVROW + ch * 16 : vbase, bytes);
      }
    }
  };

  // Page ids of the first STAGES tiles, then the first STAGES-1 tiles' rows.
  for (int i = tid; i < STAGES * C::BN; i += C::NT) sPage[i] = page_of(i / C::BN, i % C::BN);
  __syncthreads();
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < n_tiles) issue_tile(s, s);
    cp_async_commit();
  }

  // RoPE: once Q has landed, each thread rotates (row, chunk) pairs of its
  // rows in place -- element i with element i + D/2, i.e. chunk ch with
  // chunk ch + D/16 -- at the row's position, rounding to bf16.
  if (p.q_position) {
    cp_async_wait<STAGES - 1>();   // the Q group (committed first) is complete
    __syncthreads();
    constexpr int HC = D / 16;     // chunks per half row
    for (int c = tid; c < C::BM * HC; c += C::NT) {
      const int r = c / HC, ch = c % HC;
      if (r >= nrows) continue;
      const int qpos = __ldg(p.q_position + qo0 + (row0 + r) / G);
      uint4* pa = reinterpret_cast<uint4*>(sQ + swz(r, ch, C::QROW));
      uint4* pb = reinterpret_cast<uint4*>(sQ + swz(r, ch + HC, C::QROW));
      uint4 a = *pa, bq = *pb;
      uint32_t* wa = reinterpret_cast<uint32_t*>(&a);
      uint32_t* wb = reinterpret_cast<uint32_t*>(&bq);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ch * 8 + 2 * k;
        float c0, s0, c1, s1;
        rope_cos_sin(qpos, p.rope.hi[i], p.rope.lo[i], &c0, &s0);
        rope_cos_sin(qpos, p.rope.hi[i + 1], p.rope.lo[i + 1], &c1, &s1);
        const float a0 = __uint_as_float(wa[k] << 16), a1 = __uint_as_float(wa[k] & 0xffff0000u);
        const float b0 = __uint_as_float(wb[k] << 16), b1 = __uint_as_float(wb[k] & 0xffff0000u);
        wa[k] = pack_bf16x2(fmaf(a0, c0, -b0 * s0), fmaf(a1, c1, -b1 * s1));
        wb[k] = pack_bf16x2(fmaf(b0, c0, a0 * s0), fmaf(b1, c1, a1 * s1));
      }
      *pa = a;
      *pb = bq;
    }
    __syncthreads();
  }

  // This warp's rows: local rows wrow + g and wrow + g + 8 (g = lane / 4).
  const int wrow = warp * 16;
  const bool warp_active = wrow < nrows;
  const int g4 = lane >> 2, tq = lane & 3;
  const int t_lo = (row0 + wrow + g4) / G;
  const int t_hi = (row0 + wrow + g4 + 8) / G;
  const int w_last = min(wrow + 15, nrows - 1);
  // keys past it are masked for every row of the warp (causal drafts only: a
  // custom mask may open later drafts)
  const int warp_kv_end = p.mask ? kv_len : prefix + (row0 + w_last) / G + 1;
  const int moff = p.mask ? p.mask_indptr[b] : 0;
  const float sl2 = p.scale_log2;

  uint32_t qa[D / 16][4];
  float o[DV / 8][4];
#pragma unroll
  for (int j = 0; j < DV / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  for (int tile = 0; tile < n_tiles; ++tile) {
    // page ids of tile + STAGES, stored after this tile's compute (ring slot
    // tile % STAGES, whose ids were last read when this tile was issued)
    const int next_page = tid < C::BN ? page_of(tile + STAGES, tid) : -1;
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const int stage = tile % STAGES;
    if (tile + STAGES - 1 < n_tiles) issue_tile(tile + STAGES - 1, (tile + STAGES - 1) % STAGES);
    cp_async_commit();

    if (tile == 0 && warp_active) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(smem_u32(sQ + swz(wrow + (lane & 15), 2 * kk + (lane >> 4), C::QROW)), qa[kk][0],
                qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    const uint8_t* sK;
    const uint8_t* sV;
    if constexpr (FP8) {
      const uint8_t* raw = sStage + stage * C::STAGE_BYTES;
      // K's 16-byte chunks, then V's (rows of D and DV codes)
      for (int c = tid; c < C::BN * (C::KV_CH + C::V_CH); c += C::NT) {
        const int which = c < C::BN * C::KV_CH ? 0 : 1;
        const int nch = which ? C::V_CH : C::KV_CH;
        const int cc = c - which * (C::BN * C::KV_CH);
        const int r = cc / nch, ch = cc % nch;
        const uint4 w = *reinterpret_cast<const uint4*>(raw + which * C::TILE_BYTES +
                                                        r * (which ? C::VVROW : C::KVROW) + ch * 16);
        uint4 a, bq;
        a.x = e4m3x2_to_bf16x2((uint16_t)(w.x & 0xffff));
        a.y = e4m3x2_to_bf16x2((uint16_t)(w.x >> 16));
        a.z = e4m3x2_to_bf16x2((uint16_t)(w.y & 0xffff));
        a.w = e4m3x2_to_bf16x2((uint16_t)(w.y >> 16));
        bq.x = e4m3x2_to_bf16x2((uint16_t)(w.z & 0xffff));
        bq.y = e4m3x2_to_bf16x2((uint16_t)(w.z >> 16));
        bq.z = e4m3x2_to_bf16x2((uint16_t)(w.w & 0xffff));
        bq.w = e4m3x2_to_bf16x2((uint16_t)(w.w >> 16));
        uint8_t* dst = sConv + which * (C::BN * C::QROW);
        const int rb = which ? C::VROW : C::QROW;
        *reinterpret_cast<uint4*>(dst + swz(r, 2 * ch, rb)) = a;
        *reinterpret_cast<uint4*>(dst + swz(r, 2 * ch + 1, rb)) = bq;
      }
      __syncthreads();
      sK = sConv;
      sV = sConv + C::BN * C::QROW;
    } else {
      sK = sStage + stage * C::STAGE_BYTES;
      sV = sK + C::TILE_BYTES;
    }

    const int k0 = lo + tile * C::BN;
    if (warp_active && k0 < warp_kv_end) {
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b0, b1, b2, b3;
          const int key = j * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int ch = 2 * kk + ((lane >> 3) & 1);
          ldsm_x4(smem_u32(sK + swz(key, ch, C::QROW)), b0, b1, b2, b3);
          mma_bf16_16816(s[2 * j], qa[kk], b0, b1);
          mma_bf16_16816(s[2 * j + 1], qa[kk], b2, b3);
        }
      }
      // Visibility: keys < prefix always; draft key prefix + u when the mask
      // bit (t, u) is set (or u <= t without a mask); nothing at or past hi.
      if (p.mask_full) {
        // one row of kv_len bits per token, prefix included
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = k0 + j * 8 + 2 * tq + (e & 1);
            const int t = e < 2 ? t_lo : t_hi;
            bool vis = key < hi && t < L;
            if (vis) {
              const long long bit = (long long)moff + (long long)t * kv_len + key;
              vis = (__ldg(p.mask + (bit >> 3)) >> (bit & 7)) & 1;
            }
            if (!vis) s[j][e] = -INFINITY;
          }
        }
      } else if (!p.mask && (k0 + C::BN > prefix || k0 + C::BN > hi)) {
        // causal drafts: a row sees keys below min(hi, prefix + t + 1)
        const int lim_lo = min(hi, prefix + t_lo + 1) - k0;
        const int lim_hi = min(hi, prefix + t_hi + 1) - k0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kc = j * 8 + 2 * tq + (e & 1);
            if (kc >= (e < 2 ? lim_lo : lim_hi)) s[j][e] = -INFINITY;
          }
        }
      } else if (k0 + C::BN > prefix || k0 + C::BN > hi) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = k0 + j * 8 + 2 * tq + (e & 1);
            const int t = e < 2 ? t_lo : t_hi;
            bool vis = key < hi;
            if (vis && key >= prefix) {
              const int u = key - prefix;
              if (p.mask) {
                const long long bit = (long long)moff + (long long)t * L + u;
                vis = t < L && ((__ldg(p.mask + (bit >> 3)) >> (bit & 7)) & 1);
              } else {
                vis = u <= t;
              }
            }
            if (!vis) s[j][e] = -INFINITY;
          }
        }
      }
      // Online softmax (log2 domain, scale folded into one FFMA per logit).
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mx_lo = fmaxf(mx_lo, fmaxf(s[j][0], s[j][1]));
        mx_hi = fmaxf(mx_hi, fmaxf(s[j][2], s[j][3]));
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo * sl2;
      const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi * sl2;
      const float a_lo = ex2(m_lo * sl2 - base_lo);
      const float a_hi = ex2(m_hi * sl2 - base_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s[j][0] = ex2(fmaf(s[j][0], sl2, -base_lo));
        s[j][1] = ex2(fmaf(s[j][1], sl2, -base_lo));
        s[j][2] = ex2(fmaf(s[j][2], sl2, -base_hi));
        s[j][3] = ex2(fmaf(s[j][3], sl2, -base_hi));
        sum_lo += s[j][0] + s[j][1];
        sum_hi += s[j][2] + s[j][3];
      }
      l_lo = l_lo * a_lo + sum_lo;
      l_hi = l_hi * a_hi + sum_hi;
#pragma unroll
      for (int j = 0; j < DV / 8; ++j) {
        o[j][0] *= a_lo;
        o[j][1] *= a_lo;
        o[j][2] *= a_hi;
        o[j][3] *= a_hi;
      }
      // acc += P V  (P from the S registers, bf16)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dj = 0; dj < DV / 16; ++dj) {
          uint32_t b0, b1, b2, b3;
          const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = 2 * dj + (lane >> 4);
          ldsm_x4_t(smem_u32(sV + swz(key, ch, C::VROW)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * dj], pa, b0, b1);
          mma_bf16_16816(o[2 * dj + 1], pa, b2, b3);
        }
      }
    }
    if (tid < C::BN) sPage[(tile % STAGES) * C::BN + tid] = next_page;
  }
  cp_async_wait<0>();
  grid_dependents_launch();
  if (bad_page) atomicOr(p.status, VA_DEV_BAD_PAGE);

  if (!warp_active) return;

  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);

#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int rl = wrow + g4 + half * 8;
    if (rl >= nrows) continue;
    const float m = half ? m_hi : m_lo;
    const float l = half ? l_hi : l_lo;
    const float lse = l > 0.f ? m * p.scale_nat + logf(l) : -INFINITY;
    const float inv = l > 0.f ? p.v_scale / l : 0.f;
    if (it.part_row < 0) {
      const int rr = row0 + rl;
      const int t = rr / G, g = rr - t * G;
      const size_t orow = (size_t)(qo0 + t) * p.h_q + (size_t)h * G + g;
      uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + orow * DV);
#pragma unroll
      for (int j = 0; j < DV / 8; ++j)
        dst[j * 4 + tq] = pack_bf16x2(o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
      if (p.lse && tq == 0) p.lse[orow] = lse;
    } else {
      const size_t prow = (size_t)it.part_row + rl;
      float2* dst = reinterpret_cast<float2*>(p.part_out + prow * DV);
#pragma unroll
      for (int j = 0; j < DV / 8; ++j)
        dst[j * 4 + tq] = make_float2(o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
      if (tq == 0) p.part_lse[prow] = lse;
    }
  }
}

template <int D, int DV, bool FP8, int NW>
cudaError_t launch_variant(const PartialParams& p, int n_items, cudaStream_t stream) {
  // 8 warps: one CTA per SM, 4 tiles in flight; 4 warps: two CTAs per SM, 3 each.
  constexpr int STAGES = NW == 8 ? 4 : 3;
  using C = MmaCfg<D, DV, FP8, NW, STAGES>;
  static_assert(C::SMEM <= (NW == 8 ? 227 * 1024 : 113 * 1024), "shared memory budget");
  auto kern = verify_partial_mma_kernel<D, DV, FP8, NW, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<PartialParams*>(&p)};
  return launch_kernel(reinterpret_cast<const void*>(kern), dim3(n_items), dim3(C::NT), C::SMEM,
                       stream, args, /*pdl=*/true);
}

}  // namespace

template <int D, int DV>
static cudaError_t launch_shape(const PartialParams& p, bool w4, bool kv_fp8, int n_items,
                         cudaStream_t stream) {
  if (kv_fp8) return w4 ? launch_variant<D, DV, true, 4>(p, n_items, stream)
                        : launch_variant<D, DV, true, 8>(p, n_items, stream);
  return w4 ? launch_variant<D, DV, false, 4>(p, n_items, stream)
            : launch_variant<D, DV, false, 8>(p, n_items, stream);
}

cudaError_t launch_partial_mma(const PartialParams& p, int kernel, int head_dim, int head_dim_v,
                               bool kv_fp8, int n_items, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  const bool w4 = kernel == kKernelMma64;
  if (head_dim == 128 && head_dim_v == 128) return launch_shape<128, 128>(p, w4, kv_fp8, n_items, stream);
  if (head_dim == 64 && head_dim_v == 64) return launch_shape<64, 64>(p, w4, kv_fp8, n_items, stream);
  if (head_dim == 128 && head_dim_v == 64) return launch_shape<128, 64>(p, w4, kv_fp8, n_items, stream);
  if (head_dim == 64 && head_dim_v == 128) return launch_shape<64, 128>(p, w4, kv_fp8, n_items, stream);
  return cudaErrorInvalidValue;
}

}  // namespace va
