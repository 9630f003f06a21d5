// Split-KV verify attention on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA page gather) for blocks of 128 query rows.
//
// Same algorithm as the warp-level variant ("flashmap 0.1.0 --
// flashmap/sglang/verify_attention.py", partial kernel: one CTA per request,
// KV head, row block and kv chunk; online softmax; normalised output or fp32
// partial + LSE), laid out for sm_103a:
//  * warp 0, one thread: TMA producer.  Q arrives as one 3-D box per 64-column
//    half (G heads x 128/G tokens: the block's token-major rows); each key tile
//    arrives as 16-row page boxes of the 4-D cache [page, head, slot, dim]
//    (page ids read from the page table; boxes past the chunk point outside
//    the pool, so TMA zero-fills them) into a ring of mbarrier-tracked stages.
//  * warp 1, one thread: tcgen05.mma issuer.  S_j = Q K_j^T (M 128, N = tile
//    keys, K 128) into one of two TMEM S buffers while the softmax works on the
//    other; O += P_{j-1} V_{j-1} (V read MN-major) into a TMEM O accumulator.
//    tcgen05.commit signals S-ready, O-ready and buffer-free mbarriers.
//  * warps 4-7: one thread per query row (= TMEM lane).  Loads its S row,
//    masks it, keeps a running max m and sum l in fp32, writes P = 2^(s c - m)
//    for the next PV MMA.  The max used for P is only raised when a logit
//    exceeds it by more than 2^8 (then O and l are rescaled in TMEM); O / l is
//    exact either way.
//  * bf16 caches: 128-key tiles, bf16 MMAs, 128-byte-swizzled TMA boxes that
//    are the MMA operands as they land.
//  * fp8-e4m3 caches: 64-key tiles land unswizzled; warps 2-3 widen each tile
//    to f16 (cvt.rn.f16x2.e4m3x2, exact) into a double-buffered swizzled
//    operand, zeroing rows past the chunk; the MMAs run on f16 (Q converted
//    once per CTA, P packed as f16); k_scale / v_scale stay in the softmax
//    scale and the final normalisation.
// All mbarrier waits are bounded; on expiry the CTA raises VA_DEV_TIMEOUT,
// stops issuing work, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/verify_attn.h"
#include "va_device.cuh"
#include "va_kernels.h"
#include "va_tc.cuh"

namespace va {
namespace {

// NQ = 1: one 128-row Q tile per CTA.  NQ = 2: two Q tiles (256 rows) share
// every K/V tile, each with its own softmax warpgroup, TMEM S buffers and O
// accumulator, so K/V bytes, TMA traffic and fp8 widening per row halve and
// one warpgroup's softmax overlaps the other's MMAs.
template <bool FP8, int NQ>
struct TcCfg {
  static constexpr int ROWS = 128, D = 128;              // rows per Q tile = TMEM lanes
  static constexpr int BLOCK_ROWS = NQ * ROWS;
  static constexpr int THREADS = 128 + 128 * NQ;         // 4 role warps + 4 softmax warps per Q tile
  static constexpr int KEYS = 64;                        // keys per tile
  static constexpr int STAGES = NQ == 2 ? 4 : (FP8 ? 3 : 2);  // TMA stages (raw fp8, or bf16 operands)
  static constexpr int CTAS_PER_SM = (NQ == 1 && !FP8) ? 2 : 1;  // two small CTAs hide each other's waits
  static constexpr int QT_BYTES = ROWS * D * 2;          // one Q tile: [2 halves][128 rows][128 B]
  static constexpr int Q_BYTES = NQ * QT_BYTES;
  static constexpr int OP_BYTES = KEYS * D * 2;          // 16-bit K (or V) operand tile
  static constexpr int RAW_BYTES = KEYS * D;             // fp8 K (or V) tile [keys][128 B]
  static constexpr int STAGE_BYTES = FP8 ? 2 * RAW_BYTES : 2 * OP_BYTES;
  static constexpr int CONV_BUFS = FP8 ? 2 : 0;          // widened K+V operand buffers
  static constexpr int PT_BYTES = ROWS * KEYS * 2;       // one P tile: [key blocks][128 rows][128 B]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + Q_BYTES;
  static constexpr int OFF_CONV = OFF_KV + STAGES * STAGE_BYTES;
  static constexpr int OFF_P = OFF_CONV + CONV_BUFS * 2 * OP_BYTES;
  static constexpr int OFF_BAR = OFF_P + NQ * PT_BYTES;
  static constexpr int SMEM = OFF_BAR + 256;              // + barriers, TMEM address, abort flag
  static constexpr uint32_t QT_COLS = 256;               // per Q tile: S0 | S1 | O (64 + 64 + 128)
  static constexpr uint32_t TMEM_COLS = NQ * QT_COLS;
  static constexpr uint32_t COL_O = 2 * KEYS;
  static constexpr int CONV_WARPS = 2;                    // warps 2-3 (fp8 only)
  // 228 KB per SM, 1 KB reserved per CTA; at most 227 KB for one CTA
  static_assert(CTAS_PER_SM * (SMEM + 1024) <= 228 * 1024, "shared memory budget");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(CTAS_PER_SM * TMEM_COLS <= 512, "tensor memory budget");
  static_assert(STAGES <= 4, "barrier slots");
};

constexpr float kLn2 = 0.6931471805599453f;

// barrier slots (per-Q-tile barriers at base + qt, or base + 2 qt + buffer)
enum { B_Q = 0, B_Q_READY = 1, B_KV_FULL = 2, B_KV_EMPTY = 6, B_CONV_FULL = 10, B_CONV_FREE = 12,
       B_S_FULL = 14, B_S_FREE = 18, B_P_FULL = 22, B_O_DONE = 24, B_COUNT = 26 };
static_assert(8 * B_COUNT + 16 <= 256, "barrier area");

// Instruction descriptor, kind::f16 with f16 A and B (fp32 accumulator).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

template <bool FP8, int NQ>
__global__ void __launch_bounds__(TcCfg<FP8, NQ>::THREADS, TcCfg<FP8, NQ>::CTAS_PER_SM)
    verify_partial_tc_kernel(const PartialParams p, const __grid_constant__ TcMaps maps) {
  using C = TcCfg<FP8, NQ>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled operand tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.status, VA_DEV_BAD_TABLE);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * B_COUNT + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dependency_wait();
  const WorkItem it = p.items[blockIdx.x];
  const int b = it.b, h = it.h, G = p.group;
  const int qo0 = p.qo_indptr[b];
  const int L = p.qo_indptr[b + 1] - qo0;
  const int pg0 = p.kv_indptr[b];
  const int npg = p.kv_indptr[b + 1] - pg0;
  const int lpl = npg > 0 ? p.last_page_len[b] : 1;
  const long long kv_len_ll = npg > 0 ? (long long)(npg - 1) * p.page_size + lpl : 0;
  const int kv_len = (int)kv_len_ll;
  const int prefix = kv_len - L;
  const bool ok = L >= 0 && npg >= 0 && lpl >= 1 && lpl <= p.page_size && prefix >= 0 &&
                  it.row0 >= 0 && it.nrows > 0 && it.nrows <= C::BLOCK_ROWS &&
                  it.row0 % C::BLOCK_ROWS == 0 &&
                  (long long)it.row0 + it.nrows <= (long long)G * L && it.kv_lo >= 0 &&
                  it.kv_lo % 16 == 0 && it.kv_lo < it.kv_hi && it.kv_hi <= kv_len &&
                  kv_len_ll <= 0x7fffffffLL;
  if (!ok) {
    if (tid == 0) atomicOr(p.status, VA_DEV_BAD_TABLE);
    return;
  }
  const int nrows = it.nrows, row0 = it.row0, lo = it.kv_lo, hi = it.kv_hi;
  const int n_tiles = (hi - lo + C::KEYS - 1) / C::KEYS;
  const int nq = (nrows + C::ROWS - 1) / C::ROWS;  // live Q tiles (1 .. NQ)

  if (tid == 0) {
    mbar_init(bar(B_Q), 1);
    mbar_init(bar(B_Q_READY), 4 * nq);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), FP8 ? C::CONV_WARPS : 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_CONV_FULL + s), C::CONV_WARPS);
      mbar_init(bar(B_CONV_FREE + s), 1);
    }
    for (int qt = 0; qt < NQ; ++qt) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(bar(B_S_FULL + 2 * qt + s), 1);
        mbar_init(bar(B_S_FREE + 2 * qt + s), 4);
      }
      mbar_init(bar(B_P_FULL + qt), 4);
      mbar_init(bar(B_O_DONE + qt), 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      mbar_expect_tx(bar(B_Q), nq * C::QT_BYTES);
      const int tok0 = qo0 + row0 / G;
      for (int qt = 0; qt < nq; ++qt)
        for (int half = 0; half < 2; ++half)
          tma_load_3d(sbase + C::OFF_Q + qt * C::QT_BYTES + half * (C::QT_BYTES / 2), &maps.q,
                      half * 64, h * G, tok0 + qt * (C::ROWS / G), bar(B_Q));
      int bad = 0;
      // Page ids of a tile's 16-key boxes (-1 past the chunk), loaded one tile
      // ahead so their latency hides behind the previous tile's wait.
      constexpr int NG = C::KEYS / 16;
      int cur[NG], nxt[NG];
      auto load_pages = [&](int j, int* pg) {
        const int k0 = lo + j * C::KEYS;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const int key = k0 + 16 * g;
          pg[g] = (j < n_tiles && key < hi) ? __ldg(p.kv_indices + pg0 + (key >> p.log2_page)) : -1;
        }
      };
      load_pages(0, cur);
      for (int j = 0; j < n_tiles; ++j) {
        load_pages(j + 1, nxt);
        const int s = j % C::STAGES;
        if (j >= C::STAGES &&
            !mbar_wait(bar(B_KV_EMPTY + s), ((j / C::STAGES) - 1) & 1, abort_flag))
          break;
        mbar_expect_tx(bar(B_KV_FULL + s), C::STAGE_BYTES);
        const uint32_t kdst = sbase + C::OFF_KV + s * C::STAGE_BYTES;
        const uint32_t vdst = kdst + C::STAGE_BYTES / 2;
        const int k0 = lo + j * C::KEYS;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const int key = k0 + 16 * g;
          int page = p.num_pages;  // outside the pool: zero fill
          int slot = 0;
          if (key < hi) {
            const int pid = cur[g];
            if ((unsigned)pid < (unsigned)p.num_pages) {
              page = pid;
              slot = key & (p.page_size - 1);
            } else {
              bad = 1;
            }
          }
          if constexpr (FP8) {
            tma_load_4d(kdst + g * 2048, &maps.k, 0, slot, h, page, bar(B_KV_FULL + s));
            tma_load_4d(vdst + g * 2048, &maps.v, 0, slot, h, page, bar(B_KV_FULL + s));
          } else {
            for (int half = 0; half < 2; ++half) {
              const uint32_t off = half * (C::KEYS * 128) + g * 2048;
              tma_load_4d(kdst + off, &maps.k, half * 64, slot, h, page, bar(B_KV_FULL + s));
              tma_load_4d(vdst + off, &maps.v, half * 64, slot, h, page, bar(B_KV_FULL + s));
            }
          }
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) cur[g] = nxt[g];
      }
      if (bad) atomicOr(p.status, VA_DEV_BAD_PAGE);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t id_s = FP8 ? idesc_f16(C::ROWS, C::KEYS, false)
                                    : idesc_bf16(C::ROWS, C::KEYS, false);
      constexpr uint32_t id_o = FP8 ? idesc_f16(C::ROWS, C::D, true) : idesc_bf16(C::ROWS, C::D, true);
      auto kop = [&](int j) {  // K operand of tile j
        return FP8 ? sbase + C::OFF_CONV + (j & 1) * 2 * C::OP_BYTES
                   : sbase + C::OFF_KV + (j % C::STAGES) * C::STAGE_BYTES;
      };
      auto free_bar = [&](int j) {  // released once tile j's last MMA is done
        return FP8 ? bar(B_CONV_FREE + (j & 1)) : bar(B_KV_EMPTY + j % C::STAGES);
      };
      auto pv = [&](int qt, int j) {  // O_qt (+)= P_qt V_j
        const uint32_t vaddr = kop(j) + C::OP_BYTES;
        const uint32_t paddr = sbase + C::OFF_P + qt * C::PT_BYTES;
        for (int kk = 0; kk < C::KEYS / 16; ++kk) {
          const uint64_t a = smem_desc_sw128(paddr + (kk >> 2) * (C::ROWS * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(vaddr + kk * 16 * 128, C::KEYS * 128, 1024);
          umma_bf16(tmem + qt * C::QT_COLS + C::COL_O, a, bd, id_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_O_DONE + qt));
      };
      // all live Q tiles' P_{j} -> PV, then release tile j's operands
      auto pv_all = [&](int j) {
        for (int qt = 0; qt < nq; ++qt) {
          if (!mbar_wait(bar(B_P_FULL + qt), j & 1, abort_flag)) return false;
          tc_fence_after();
          pv(qt, j);
        }
        umma_commit(free_bar(j));
        return true;
      };
      bool live = mbar_wait(bar(FP8 ? B_Q_READY : B_Q), 0, abort_flag);
      int issued_pv = 0;
      for (int j = 0; live && j < n_tiles; ++j) {
        const int sb = j & 1;
        if (FP8) {
          if (!mbar_wait(bar(B_CONV_FULL + sb), (j >> 1) & 1, abort_flag)) break;
        } else {
          if (!mbar_wait(bar(B_KV_FULL + j % C::STAGES), (j / C::STAGES) & 1, abort_flag)) break;
        }
        const uint32_t kaddr = kop(j);
        for (int qt = 0; qt < nq; ++qt) {
          if (j >= 2 && !mbar_wait(bar(B_S_FREE + 2 * qt + sb), ((j >> 1) - 1) & 1, abort_flag)) {
            live = false;
            break;
          }
          tc_fence_after();
          const uint32_t qaddr = sbase + C::OFF_Q + qt * C::QT_BYTES;
          for (int kk = 0; kk < C::D / 16; ++kk) {
            const uint64_t a = smem_desc_sw128(qaddr + (kk >> 2) * (C::ROWS * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(kaddr + (kk >> 2) * (C::KEYS * 128) + (kk & 3) * 32, 16, 1024);
            umma_bf16(tmem + qt * C::QT_COLS + sb * C::KEYS, a, bd, id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(B_S_FULL + 2 * qt + sb));
        }
        if (!live) break;
        if (j >= 1) {
          if (!pv_all(j - 1)) break;
          issued_pv = j;
        }
      }
      if (!*abort_flag && issued_pv == n_tiles - 1) {
        const int j = n_tiles - 1;
        // the last buffer release lands before the CTA's shared memory goes away
        if (pv_all(j)) {
          if (FP8)
            mbar_wait(bar(B_CONV_FREE + (j & 1)), (j >> 1) & 1, abort_flag);
          else
            mbar_wait(bar(B_KV_EMPTY + j % C::STAGES), (j / C::STAGES) & 1, abort_flag);
        }
      }
    }
  } else if (warp < 4) {
    if constexpr (FP8) {
      // ---------------- fp8 -> f16 widening (warps 2-3) ----------------
      const int ct = tid - 64;                      // 0 .. 63
      constexpr int CH = C::KEYS * 8;               // 16-byte raw chunks per K (or V) tile
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % C::STAGES, cb = j & 1;
        if (!mbar_wait(bar(B_KV_FULL + s), (j / C::STAGES) & 1, abort_flag)) break;
        if (j >= 2 && !mbar_wait(bar(B_CONV_FREE + cb), ((j >> 1) - 1) & 1, abort_flag)) break;
        const uint8_t* raw = smem + C::OFF_KV + s * C::STAGE_BYTES;
        uint8_t* dst = smem + C::OFF_CONV + cb * 2 * C::OP_BYTES;
        const int k0 = lo + j * C::KEYS;
#pragma unroll 4
        for (int c = ct; c < 2 * CH; c += 64) {
          const int which = c / CH, cc = c - which * CH;
          const int r = cc >> 3, ch = cc & 7;       // key row, 16-element column group
          uint4 a = make_uint4(0u, 0u, 0u, 0u), bq = a;
          if (k0 + r < hi) {
            const uint4 w = *reinterpret_cast<const uint4*>(raw + which * C::RAW_BYTES + r * 128 + ch * 16);
            a.x = e4m3x2_to_f16x2((uint16_t)(w.x & 0xffff));
            a.y = e4m3x2_to_f16x2((uint16_t)(w.x >> 16));
            a.z = e4m3x2_to_f16x2((uint16_t)(w.y & 0xffff));
            a.w = e4m3x2_to_f16x2((uint16_t)(w.y >> 16));
            bq.x = e4m3x2_to_f16x2((uint16_t)(w.z & 0xffff));
            bq.y = e4m3x2_to_f16x2((uint16_t)(w.z >> 16));
            bq.z = e4m3x2_to_f16x2((uint16_t)(w.w & 0xffff));
            bq.w = e4m3x2_to_f16x2((uint16_t)(w.w >> 16));
          }
          // 16 f16 = 2 chunks of the swizzled operand row (half = ch / 4)
          uint8_t* row = dst + which * C::OP_BYTES + (ch >> 2) * (C::KEYS * 128) + r * 128;
          const int c0 = (ch & 3) * 2;
          *reinterpret_cast<uint4*>(row + (((c0) ^ (r & 7)) << 4)) = a;
          *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = bq;
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_CONV_FULL + cb));
          mbar_arrive(bar(B_KV_EMPTY + s));
        }
      }
    }
  } else if ((warp - 4) / 4 < nq) {
    // ---------------- softmax / epilogue: one thread per row, 4 warps per Q tile ----------------
    const int qt = (warp - 4) >> 2;                 // Q tile of this warpgroup
    const int quad = warp & 3;                      // TMEM lane quarter this warp may access
    const int r = quad * 32 + lane;                 // row of the Q tile = TMEM lane
    const int br = qt * C::ROWS + r;                // row of the block
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16) + qt * C::QT_COLS;
    const bool row_ok = br < nrows;
    const int t = (row0 + br) / G;                  // draft token of the row
    const int moff = p.mask ? p.mask_indptr[b] : 0;
    const float c = p.scale_log2;
    const uint32_t b_s_full = bar(B_S_FULL + 2 * qt), b_s_free = bar(B_S_FREE + 2 * qt);
    const uint32_t b_p_full = bar(B_P_FULL + qt), b_o_done = bar(B_O_DONE + qt);
    uint8_t* const ptile = smem + C::OFF_P + qt * C::PT_BYTES;
    float m_used = -INFINITY;                       // in units of s * c (log2 domain)
    float l = 0.f;
    float s[C::KEYS];
    uint32_t pk[C::KEYS / 2];
    bool live = true;
    if (FP8) {
      // Q to f16, in place (each thread its own row)
      if (!mbar_wait(bar(B_Q), 0, abort_flag)) live = false;
      if (live) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint4* q4 = reinterpret_cast<uint4*>(smem + C::OFF_Q + qt * C::QT_BYTES +
                                               half * (C::QT_BYTES / 2) + r * 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint4 v = q4[ch];
            v.x = bf16x2_to_f16x2(v.x);
            v.y = bf16x2_to_f16x2(v.y);
            v.z = bf16x2_to_f16x2(v.z);
            v.w = bf16x2_to_f16x2(v.w);
            q4[ch] = v;
          }
        }
        fence_proxy_async();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_Q_READY));
    }
    for (int j = 0; live && j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(b_s_full + 8 * sb, (j >> 1) & 1, abort_flag)) { live = false; break; }
      tc_fence_after();
      {
        uint32_t raw[C::KEYS];
#pragma unroll
        for (int q = 0; q < C::KEYS / 32; ++q) tmem_ld32(lane_addr + sb * C::KEYS + q * 32, raw + q * 32);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < C::KEYS; ++e) s[e] = __uint_as_float(raw[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_s_free + 8 * sb);

      const int k0 = lo + j * C::KEYS;
      if (k0 + C::KEYS > prefix || k0 + C::KEYS > hi) {
        if (!p.mask) {
          // causal drafts: this row sees keys below min(hi, prefix + t + 1)
          const int lim = min(hi, prefix + t + 1) - k0;
#pragma unroll
          for (int cc = 0; cc < C::KEYS; ++cc) s[cc] = cc < lim ? s[cc] : -INFINITY;
        } else {
          // per 32-key group: visibility bits (prefix 1, drafts from the
          // row's mask bits, nothing at or past hi), then one select per key
#pragma unroll
          for (int q = 0; q < C::KEYS / 32; ++q) {
            const int g0 = k0 + 32 * q;
            uint32_t vis = 0;
            if (g0 < hi) {
              const int below_prefix = min(max(prefix - g0, 0), 32);
              vis = below_prefix == 32 ? 0xffffffffu : ((1u << below_prefix) - 1u);
              if (below_prefix < 32 && t < L) {
                // draft columns u = g0 + i - prefix for i >= below_prefix
                const int u0 = g0 + below_prefix - prefix;
                const long long bit0 = (long long)moff + (long long)t * L + u0;
                const int nbits = min(32 - below_prefix, L - u0);
                if (nbits > 0) {
                  uint64_t w = 0;
                  const int nbytes = (int)((((bit0 & 7) + nbits) + 7) >> 3);
                  for (int k = 0; k < nbytes; ++k)
                    w |= (uint64_t)__ldg(p.mask + (bit0 >> 3) + k) << (8 * k);
                  w >>= (bit0 & 7);
                  const uint32_t dbits =
                      (uint32_t)(w & (nbits >= 32 ? 0xffffffffull : ((1ull << nbits) - 1ull)));
                  vis |= dbits << below_prefix;
                }
              }
              const int in_range = min(hi - g0, 32);
              if (in_range < 32) vis &= (1u << in_range) - 1u;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)
              s[32 * q + i] = ((vis >> i) & 1u) ? s[32 * q + i] : -INFINITY;
          }
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < C::KEYS; ++cc) mx = fmaxf(mx, s[cc]);
      mx *= c;  // c > 0
      float m_new = m_used;
      if (mx > m_used + 8.f) m_new = mx;   // also taken when m_used = -inf and mx is finite
      const float alpha = (m_new == m_used) ? 1.f : ex2(m_used - m_new);
      const float base = m_new == -INFINITY ? 0.f : m_new;
      float sum = 0.f;
#pragma unroll
      for (int cc = 0; cc < C::KEYS; cc += 2) {
        const float p0 = ex2(fmaf(s[cc], c, -base));
        const float p1 = ex2(fmaf(s[cc + 1], c, -base));
        sum += p0 + p1;
        pk[cc / 2] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
      }
      l = l * alpha + sum;
      // P buffer and O are free once the previous PV has completed.
      if (j >= 1) {
        if (!mbar_wait(b_o_done, (j - 1) & 1, abort_flag)) { live = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          for (int q = 0; q < C::D / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(lane_addr + C::COL_O + q * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(lane_addr + C::COL_O + q * 32, ov);
          }
          tmem_wait_st();
        }
      }
      if constexpr (!FP8) {
        // Rows of V past the chunk end inside the last 16-key box may hold
        // stale (even NaN) slots: zero them, since 0 * NaN would poison O.
        // Q tile 0's warps do it; the MMAs of every Q tile's PV wait for them.
        const int tail = hi - k0;
        if (qt == 0 && tail < C::KEYS && (tail & 15)) {
          const int zlo = tail, zhi = (tail + 15) & ~15;
          uint8_t* vt = smem + C::OFF_KV + (j % C::STAGES) * C::STAGE_BYTES + C::OP_BYTES;
          for (int z = r; z < (zhi - zlo) * 16; z += C::ROWS) {
            const int row = zlo + z / 16, half = (z / 8) & 1, ch = z & 7;
            *reinterpret_cast<uint4*>(vt + half * (C::KEYS * 128) + row * 128 + (ch << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      // P row -> shared memory, K-major 128-byte-swizzled [key block][row][128 B]
#pragma unroll
      for (int ch = 0; ch < C::KEYS / 8; ++ch) {
        const int kb = ch >> 3, c8 = ch & 7;
        *reinterpret_cast<uint4*>(ptile + kb * (C::ROWS * 128) + r * 128 + ((c8 ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p_full);
      m_used = m_new;
    }
    // epilogue
    if (live && mbar_wait(b_o_done, (n_tiles - 1) & 1, abort_flag)) {
      tc_fence_after();
      const float lse = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      const float inv = l > 0.f ? p.v_scale / l : 0.f;
      size_t orow = 0;
      if (row_ok) {
        const int g = (row0 + br) - t * G;
        orow = (size_t)(qo0 + t) * p.h_q + (size_t)h * G + g;
      }
      for (int q = 0; q < C::D / 32; ++q) {
        uint32_t ov[32];
        tmem_ld32(lane_addr + C::COL_O + q * 32, ov);
        tmem_wait_ld();
        if (!row_ok) continue;
        if (it.part_row < 0) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow * C::D + q * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
            dst[e] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.part_out + ((size_t)it.part_row + br) * C::D + q * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(ov[4 * e]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                                 __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv);
        }
      }
      if (row_ok) {
        if (it.part_row < 0) {
          if (p.lse) p.lse[orow] = lse;
        } else {
          p.part_lse[(size_t)it.part_row + br] = lse;
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  grid_dependents_launch();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) atomicOr(p.status, VA_DEV_TIMEOUT);
}

template <bool FP8, int NQ>
cudaError_t launch_tc(const PartialParams& p, const TcMaps& maps, int n_items,
                      cudaStream_t stream) {
  using C = TcCfg<FP8, NQ>;
  auto kern = verify_partial_tc_kernel<FP8, NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<PartialParams*>(&p), const_cast<TcMaps*>(&maps)};
  return launch_kernel(reinterpret_cast<const void*>(kern), dim3(n_items), dim3(C::THREADS),
                       C::SMEM, stream, args, /*pdl=*/true);
}

}  // namespace

cudaError_t launch_partial_tc(const PartialParams& p, const TcMaps& maps, bool kv_fp8,
                              int block_rows, int n_items, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (block_rows == 256)
    return kv_fp8 ? launch_tc<true, 2>(p, maps, n_items, stream)
                  : launch_tc<false, 2>(p, maps, n_items, stream);
  return kv_fp8 ? launch_tc<true, 1>(p, maps, n_items, stream)
                : launch_tc<false, 1>(p, maps, n_items, stream);
}

}  // namespace va
