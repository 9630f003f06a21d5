// Split-KV verify attention on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA page gather) for blocks of one or two 128-row Q tiles,
// one persistent CTA per SM.
//
// Same algorithm as the warp-level variant ("flashmap 0.1.0 --
// flashmap/sglang/verify_attention.py", partial kernel: one CTA per request,
// KV head, row block and kv chunk; online softmax; normalised output or fp32
// partial + LSE), laid out for sm_103a:
//  * warp 0, one thread: TMA producer.  Q arrives as one 3-D box per 64-column
//    half and Q tile (G heads x 128/G tokens: the tile's token-major rows);
//    key tiles of 128 keys arrive as one 4 KB box per 16 keys of a page
//    (bf16: the cache viewed as [page * h_kv + head][slot / 8][half][slot % 8]
//    [64], which lands in the MMAs' swizzled operand layout; fp8: 2 KB raw
//    boxes) -- page ids read two tiles ahead; boxes past the chunk point
//    outside the pool, so TMA zero-fills them -- into one ring of
//    mbarrier-tracked slots holding K_0, V_0, K_1, V_1, ...
//  * warp 1, one thread: tcgen05.mma issuer.  Per Q tile and key tile j it
//    issues O += P_{j-1} V_{j-1} (P read from tensor memory, V MN-major from
//    shared memory), then S_j = Q K_j^T (M 128, N 128, K 128) into the same
//    TMEM columns, so P and S share them; the two Q tiles alternate, and one
//    tile's softmax runs while the tensor core works on the other's MMAs.
//    tcgen05.commit signals S-ready, O-done and slot-free mbarriers.
//  * softmax warps, four per Q tile: one thread per query row (= TMEM lane).
//    Loads its S row, masks it, keeps a running max m and sum l in fp32, and
//    writes P = 2^(s c - m) back into tensor memory over S.  The max used for
//    P is only raised when a logit exceeds it by more than 2^8 (then O and l
//    are rescaled; O is idle at that point); O / l is exact either way.
//  * bf16 caches: the TMA boxes land in the MMA's 128-byte-swizzled operand
//    layout; rows of V past the chunk end are zeroed before the PV MMA reads
//    them (stale slots may hold NaN).
//  * fp8-e4m3 caches: raw tiles land unswizzled; six converter warps widen
//    them into swizzled f16 operand buffers (cvt.rn.f16x2.e4m3x2: every e4m3
//    value, subnormals included, is an f16 value) and zero rows past the
//    chunk; k_scale / v_scale stay in the softmax scale and the final
//    normalisation.  The MMAs run on f16 (Q converted once per item, P packed
//    as f16).
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

// FP8: the cache is fp8-e4m3.  F8MMA (fp8 caches only): the MMAs run on
// e4m3 operands (kind::f8f6f4: Q quantised per row, P as e4m3, K / V as
// stored) instead of widening K / V to f16 (kind::f16).
template <bool FP8, int NQ, bool F8MMA = false>
struct TcCfg {
  static constexpr int ROWS = 128, D = 128;              // rows per Q tile = TMEM lanes
  static constexpr int KEYS = 128;                       // keys per tile (MMA N of S, K of PV)
  static constexpr int BLOCK_ROWS = NQ * ROWS;
  static constexpr int CONV_WARP0 = 4 + 4 * NQ;          // after producer, MMA, 2 spare, softmax
  // fp8 widening: warps 2, 3 and CONV_WARP0 .. CONV_WARP0 + 3.  Four of them
  // sit on the SM sub-partitions 2 and 3 (warp % 4), two share the
  // producer's and the MMA issuer's; six measured faster than those four
  // alone (fp8 wide tree 306.5 -> 297.7 us): the widening of V_{j-1} is on
  // the path from PV_{j-2} to PV_{j-1}.
  static constexpr bool WIDEN = FP8 && !F8MMA;           // fp8 widened to f16 by converter warps
  static constexpr int CONV_WARPS = WIDEN ? 6 : 0;
  static constexpr int THREADS = 32 * (CONV_WARP0 + (WIDEN ? 4 : 0));  // fp8: 4 warps past the softmax
  static constexpr int QT_BYTES = ROWS * D * 2;          // one Q tile: [2 halves][128 rows][128 B]
  static constexpr int Q_BYTES = NQ * QT_BYTES;
  static constexpr int OP_BYTES = KEYS * D * 2;          // 16-bit K (or V) operand tile
  static constexpr int RAW_BYTES = KEYS * D;             // fp8 K (or V) tile [keys][128 B]
  static constexpr int SLOT_BYTES = FP8 ? RAW_BYTES : OP_BYTES;
  static constexpr int CONV_BYTES = WIDEN ? 3 * OP_BYTES : 0;  // widened K (two) and V (one)
  static constexpr int BAR_BYTES = 1024;                 // barriers, TMEM address, item queue
  static constexpr int RING_AVAIL = 227 * 1024 - BAR_BYTES - Q_BYTES - CONV_BYTES;
  static constexpr int NSLOT = RING_AVAIL / SLOT_BYTES > 8 ? 8 : RING_AVAIL / SLOT_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_CONV = OFF_Q + Q_BYTES;
  static constexpr int OFF_RING = OFF_CONV + CONV_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * SLOT_BYTES;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES;
  // S / P buffers per Q tile: one Q tile double-buffers S, so S_{j+1} is
  // computed while the softmax works on S_j; two Q tiles fill tensor memory
  // with one buffer each and alternate instead.
  static constexpr int SBUF = NQ == 1 ? 2 : 1;
  static constexpr uint32_t QT_COLS = 128 * (SBUF + 1);  // per Q tile: S / P (128 each) | O (128)
  static constexpr uint32_t COL_O = 128 * SBUF;
  static constexpr uint32_t TMEM_COLS = 512;             // NQ * QT_COLS, as a power of two
  static_assert(NSLOT >= 3, "ring depth");
  static_assert(!WIDEN || THREADS == 32 * (CONV_WARP0 + 4), "converter warps: 2, 3, CONV_WARP0 .. + 3");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(NQ * QT_COLS <= TMEM_COLS, "tensor memory budget");
};

constexpr float kLn2 = 0.6931471805599453f;

// barrier slots (per-Q-tile barriers at base + qt; S_FULL / P_FULL at base +
// buffer when one Q tile double-buffers S)
enum { B_Q = 0, B_Q_READY = 1, B_Q_FREE = 2, B_FULL = 3, B_EMPTY = 11, B_CK_FULL = 19,
       B_CK_FREE = 21, B_CV_FULL = 23, B_CV_FREE = 24, B_S_FULL = 25, B_P_FULL = 27, B_O_DONE = 29,
       B_O_FREE = 31, B_PV_DONE = 33, B_GQ_FULL = 34, B_GQ_FREE = 38, B_COUNT = 42 };
constexpr int kGeoQueue = 4;  // entries of the shared item-geometry queue (B_GQ_FULL / B_GQ_FREE + e)

// Instruction descriptor, kind::f16 with f16 A and B (fp32 accumulator).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// TMEM column (relative to the Q tile's S / P columns) of P's keys
// 16 kk .. 16 kk + 15, packed two per column: the P of logits 32 q .. 32 q + 31
// sits in the first half of their own S columns, 32 q .. 32 q + 15, so the
// softmax may write it as soon as it has read that chunk of S.
__host__ __device__ constexpr uint32_t p_col(int kk) { return 32u * (kk >> 1) + 8u * (kk & 1); }

// max(a, b, c) in one instruction (three-input form of sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

// One work item's geometry, as every role of the CTA decodes it.
// lov: the item's first key; lo: its tile grid's start, lov rounded down to
// 16 keys (keys lo .. lov - 1 are loaded and masked: a draft item starts at
// the prefix length, mid-page).
struct ItemGeo {
  int b, h, row0, nrows, lo, lov, hi, part_row, qo0, L, pg0, prefix, n_tiles, nq, moff;
  bool ok;
};
// One entry of the item-geometry queue: the producer decodes each item of the
// CTA's chain once and posts it; end marks the end of the chain.
struct GeoSlot {
  ItemGeo g;
  int end;
};
static_assert(8 * B_COUNT + 16 + kGeoQueue * sizeof(GeoSlot) <= 1024, "barrier area");

template <int BLOCK_ROWS, int ROWS, int KEYS>
__device__ __forceinline__ ItemGeo decode_item(const PartialParams& p, int i) {
  const WorkItem it = p.items[i];
  ItemGeo g;
  g.b = it.b;
  g.h = it.h;
  g.row0 = it.row0;
  g.nrows = it.nrows;
  g.lov = it.kv_lo;
  g.lo = it.kv_lo & ~15;
  g.hi = it.kv_hi;
  g.part_row = it.part_row;
  // a work list left in the workspace by another plan may name requests
  // past this call's tables: nothing is read for those
  const bool idx_ok = g.b >= 0 && g.b < p.batch && g.h >= 0 && g.h < p.h_kv;
  g.qo0 = idx_ok ? p.qo_indptr[g.b] : 0;
  g.L = idx_ok ? p.qo_indptr[g.b + 1] - g.qo0 : -1;
  g.pg0 = idx_ok ? p.kv_indptr[g.b] : 0;
  const int npg = idx_ok ? p.kv_indptr[g.b + 1] - g.pg0 : -1;
  const int lpl = npg > 0 ? p.last_page_len[g.b] : 1;
  const long long kv_len = npg > 0 ? (long long)(npg - 1) * p.page_size + lpl : 0;
  g.prefix = (int)kv_len - g.L;
  g.ok = g.L >= 0 && npg >= 0 && lpl >= 1 && lpl <= p.page_size && kv_len <= 0x7fffffffLL &&
         g.prefix >= 0 && g.row0 >= 0 && g.nrows > 0 && g.nrows <= BLOCK_ROWS &&
         g.row0 % BLOCK_ROWS == 0 && (long long)g.row0 + g.nrows <= (long long)p.group * g.L &&
         g.lov >= 0 && g.lov < g.hi && g.hi <= kv_len &&
         (g.part_row < 0 || (long long)g.part_row + g.nrows <= p.part_rows);
  g.n_tiles = g.ok ? (g.hi - g.lo + KEYS - 1) / KEYS : 0;
  g.moff = g.ok && p.mask ? p.mask_indptr[g.b] : 0;
  g.nq = (g.nrows + ROWS - 1) / ROWS;  // live Q tiles (1 .. NQ)
  return g;
}

// Persistent: one CTA per SM walks its chain of work items (dealt by the
// planner longest-first onto the least-loaded CTA), and every role streams
// from one item into the next.  The producer loads item k + 1's Q as soon as
// item k's last S MMA has read Q, and its keys into the same slot ring; the
// MMA issuer starts item k + 1's S MMAs while the softmax warps still write
// item k's output, and its first PV once that output has left O.
template <bool FP8, int NQ, bool F8MMA>
__global__ void __launch_bounds__(TcCfg<FP8, NQ, F8MMA>::THREADS, 1)
    verify_partial_tc_kernel(const PartialParams p, const __grid_constant__ TcMaps maps) {
  using C = TcCfg<FP8, NQ, F8MMA>;
  constexpr bool WIDEN = C::WIDEN;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled operand tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.status, VA_DEV_BAD_TABLE);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * B_COUNT + 4);
  GeoSlot* geoq = reinterpret_cast<GeoSlot*>(smem + C::OFF_BAR + 8 * B_COUNT + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  // Q is rewritten in shared memory by the softmax warps before the first S
  // MMA reads it: to f16 for an fp8 cache, rotated at its positions for RoPE
  const bool q_pass = FP8 || p.q_position != nullptr;   // f16 widening or e4m3 quantisation
  // This CTA's items: chain blockIdx.x (then blockIdx.x + gridDim.x, ... if
  // the grid is smaller than the plan's chain count), linked through next; a
  // malformed link ends its chain.
  auto first_item = [&](int slot) -> int { return slot < p.n_ctas && slot < p.n_items ? slot : -1; };
  auto next_item = [&](int i, int& slot, int& steps) -> int {
    int n = p.items[i].next;
    if (++steps > p.n_items || n >= p.n_items) n = -1;
    if (n >= 0) return n;
    slot += (int)gridDim.x;
    return first_item(slot);
  };
  auto decode = [&](int i) { return decode_item<C::BLOCK_ROWS, C::ROWS, C::KEYS>(p, i); };
  // The producer walks the chain and decodes each item (a few dependent
  // global loads) once; the MMA issuer, the softmax and converter warps read
  // the decoded geometry from a small shared queue, so none of them stalls
  // on those loads between items.
  constexpr int GQ_USERS = 1 + 4 * NQ + C::CONV_WARPS;
  auto take_geo_thread = [&](int k, ItemGeo& g) -> bool {  // false: end of chain (or timeout)
    const int e = k % kGeoQueue;
    if (!mbar_wait(bar(B_GQ_FULL + e), (k / kGeoQueue) & 1, abort_flag)) return false;
    g = geoq[e].g;
    const int end = geoq[e].end;
    mbar_arrive(bar(B_GQ_FREE + e));
    return !end;
  };
  auto take_geo_warp = [&](int k, ItemGeo& g) -> bool {
    const int e = k % kGeoQueue;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(B_GQ_FULL + e), (k / kGeoQueue) & 1, abort_flag))) return false;
    g = geoq[e].g;
    const int end = geoq[e].end;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_GQ_FREE + e));
    return !end;
  };

  // While the previous kernel may still run: fetch the three TMA descriptors
  // (kernel parameters) and this CTA's first work item (uploaded with the
  // plan, never written by a kernel) towards the SM, so the first loads after
  // the dependency wait do not each pay a round trip to memory.
  if (tid == 0) {
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
    if (p.drafts_new) {
      tma_prefetch_desc(&maps.kn);
      tma_prefetch_desc(&maps.vn);
    }
    if ((int)blockIdx.x < p.n_items) prefetch_l1(p.items + blockIdx.x);
  }
  if (tid == 0) {
    mbar_init(bar(B_Q), 1);
    mbar_init(bar(B_Q_READY), 4 * NQ);
    mbar_init(bar(B_Q_FREE), 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), WIDEN ? C::CONV_WARPS : 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_CK_FULL + s), C::CONV_WARPS > 0 ? C::CONV_WARPS : 1);
      mbar_init(bar(B_CK_FREE + s), 1);
    }
    mbar_init(bar(B_CV_FULL), C::CONV_WARPS > 0 ? C::CONV_WARPS : 1);
    mbar_init(bar(B_CV_FREE), 1);
    for (int s = 0; s < NQ * C::SBUF; ++s) {
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_P_FULL + s), 4);
    }
    for (int qt = 0; qt < NQ; ++qt) {
      mbar_init(bar(B_O_DONE + qt), 1);
      mbar_init(bar(B_O_FREE + qt), 4);
    }
    mbar_init(bar(B_PV_DONE), 1);
    for (int e = 0; e < kGeoQueue; ++e) {
      mbar_init(bar(B_GQ_FULL + e), 1);
      mbar_init(bar(B_GQ_FREE + e), GQ_USERS);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA of this persistent grid is resident, so the next kernel (the
  // merge) may be scheduled now: it waits for our completion before reading
  // anything.  The wait for the grid before this one in the stream (which
  // may still be writing the drafts' pages) is the producer's alone: it is
  // taken before the first load of a key tile holding draft keys, and every
  // role that writes memory does so after consuming such loads or q, so its
  // writes follow the previous grid's completion.
  grid_dependents_launch();

  // Operand u = 2 j (K_j) or 2 j + 1 (V_j) of the CTA's running tile count j
  // sits in ring slot u % NSLOT, on its (u / NSLOT)-th use of that slot.
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int bad = 0, bad_item = 0, nit = 0;
      int u = 0;
      bool live = true;
      constexpr int NG = C::KEYS / 16;
      int k = 0;
      auto post = [&](const ItemGeo& g, int end) -> bool {
        const int e = k % kGeoQueue;
        if (k >= kGeoQueue && !mbar_wait(bar(B_GQ_FREE + e), ((k / kGeoQueue) - 1) & 1, abort_flag))
          return false;
        geoq[e].g = g;
        geoq[e].end = end;
        mbar_arrive(bar(B_GQ_FULL + e));  // release: the entry is visible to the waiters
        ++k;
        return true;
      };
      int slot = blockIdx.x, steps = 0;
      bool waited = false;  // the dependency on the previous grid has been waited for
      if (!p.early_inputs) {
        // a call of its own: nothing is read before the previous grid is done
        grid_dependency_wait();
        waited = true;
      }
      const bool nhd = p.nhd != 0;
      const int ps8 = p.page_size >> 3;
      for (int i = first_item(slot); live && i >= 0; i = next_item(i, slot, steps)) {
        const ItemGeo g = decode(i);
        if (!post(g, 0)) {
          live = false;
          break;
        }
        if (!g.ok) {
          bad_item = 1;
          continue;
        }
        // Page ids of a tile's 16-key boxes (-1 past the chunk), loaded two
        // tiles ahead so their latency hides behind the previous tiles' waits
        // (and an item's first two tiles wait for one round trip, not two).
        int cur[NG], nxt[NG], nx2[NG];
        auto load_pages = [&](int j, int* pg) {
          const int k0 = g.lo + j * C::KEYS;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            const int key = k0 + 16 * q;
            pg[q] = (j < g.n_tiles && key < g.hi) ? __ldg(p.kv_indices + g.pg0 + (key >> p.log2_page)) : -1;
          }
        };
        // Q of this item once the previous item's S MMAs are done with Q
        auto issue_q = [&]() -> bool {
          if (nit >= 1 && !mbar_wait(bar(B_Q_FREE), (nit - 1) & 1, abort_flag)) return false;
          mbar_expect_tx(bar(B_Q), g.nq * C::QT_BYTES);
          const int tok0 = g.qo0 + g.row0 / G;
          for (int qt = 0; qt < g.nq; ++qt)
            for (int half = 0; half < 2; ++half)
              tma_load_3d(sbase + C::OFF_Q + qt * C::QT_BYTES + half * (C::QT_BYTES / 2), &maps.q,
                          half * 64, g.h * G, tok0 + qt * (C::ROWS / G), bar(B_Q));
          return true;
        };
        load_pages(0, cur);
        load_pages(1, nxt);
        // With early inputs (after this library's append, or on the caller's
        // promise) q and the key tiles that hold prefix keys only are issued
        // before the dependency wait: the previous grid writes none of them
        // (the append writes only the drafts' slots, and releases this kernel
        // only after its own predecessor -- the producer of q -- has
        // completed), so they stream in while it finishes.  A tile with draft
        // keys read from the pages waits for it; an item of drafts only,
        // read from the new rows, does not.
        const bool from_new = p.drafts_new && g.lov >= g.prefix;
        if (!issue_q()) break;
        for (int j = 0; live && j < g.n_tiles; ++j) {
          if (!waited && !from_new && min(g.lo + (j + 1) * C::KEYS, g.hi) > g.prefix) {
            grid_dependency_wait();
            waited = true;
          }
          load_pages(j + 2, nx2);
          const int k0 = g.lo + j * C::KEYS;
          for (int v = 0; v < 2; ++v, ++u) {
            const int s = u % C::NSLOT, n = u / C::NSLOT;
            if (n >= 1 && !mbar_wait(bar(B_EMPTY + s), (n - 1) & 1, abort_flag)) {
              live = false;
              break;
            }
            mbar_expect_tx(bar(B_FULL + s), C::SLOT_BYTES);
            const uint32_t dst = sbase + C::OFF_RING + s * C::SLOT_BYTES;
            if (from_new) {
              // key k >= prefix is new row qo0 + k - prefix; rows past the item
              // (a later request's, or past the end: zero fill) are masked, and
              // V rows past the chunk end are zeroed like a page tile's
              const void* nmap = v ? static_cast<const void*>(&maps.vn) : static_cast<const void*>(&maps.kn);
              if constexpr (FP8) {
#pragma unroll
                for (int q = 0; q < NG; ++q) {
                  const int key = k0 + 16 * q;
                  const int tok = key < g.hi ? g.qo0 + key - g.prefix : p.total_qo;
                  tma_load_3d(dst + q * 2048, nmap, 0, tok, g.h, bar(B_FULL + s));
                }
              } else {
#pragma unroll
                for (int q = 0; q < 2 * NG; ++q) {
                  const int key = k0 + 8 * q;
                  const int tok = key < g.hi ? g.qo0 + key - g.prefix : p.total_qo;
                  tma_load_4d(dst + q * 2048, nmap, 0, tok, 0, g.h, bar(B_FULL + s));
                }
              }
              continue;
            }
            const void* map = v ? static_cast<const void*>(&maps.v) : static_cast<const void*>(&maps.k);
#pragma unroll
            for (int q = 0; q < NG; ++q) {
              const int key = k0 + 16 * q;
              int page = p.num_pages;  // outside the pool: zero fill
              int slot = 0;
              if (key < g.hi) {
                const int pid = cur[q];
                if ((unsigned)pid < (unsigned)p.num_pages) {
                  page = pid;
                  slot = key & (p.page_size - 1);
                } else {
                  bad = 1;
                }
              }
              if constexpr (FP8) {
                tma_load_4d(dst + q * 2048, map, 0, slot, g.h, page, bar(B_FULL + s));
              } else {
                // HND view [page * h_kv + head][slot / 8]...; NHD view
                // [page * P / 8 + slot / 8][head]...
                const int c3 = nhd ? g.h : (slot >> 3);
                const int c4 = nhd ? page * ps8 + (slot >> 3) : page * p.h_kv + g.h;
                tma_load_5d(dst + q * 4096, map, 0, 0, 0, c3, c4, bar(B_FULL + s));
              }
            }
          }
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            cur[q] = nxt[q];
            nxt[q] = nx2[q];
          }
        }
        if (!live) break;
        ++nit;
      }
      // A CTA that met no valid item still waits once, so that this grid's
      // completion implies the previous grid's (the next kernel relies on it)
      if (!waited) grid_dependency_wait();
      if (live) post(ItemGeo{}, 1);  // end of the chain
      if (bad) atomicOr(p.status, VA_DEV_BAD_PAGE);
      if (bad_item) atomicOr(p.status, VA_DEV_BAD_TABLE);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t id_s = FP8 ? idesc_f16(C::ROWS, C::KEYS, false)
                                    : idesc_bf16(C::ROWS, C::KEYS, false);
      constexpr uint32_t id_o = FP8 ? idesc_f16(C::ROWS, C::D, true) : idesc_bf16(C::ROWS, C::D, true);
      // K / V operand layouts: widened fp8 in 64-column halves [half][keys][64]
      // (halves KEYS * 128 bytes apart, 8-key groups 1024); bf16 as the TMA
      // boxes land, [8-key group][half][8][64] (groups 2048 apart, halves 1024)
      // e4m3 operands (F8MMA) as they land: [keys][128 B], 8-key groups 1024
      // apart, one 128-byte swizzle atom across the whole head dimension
      constexpr uint32_t KV_SBO = FP8 ? 1024 : 2048;            // 8-key group stride
      constexpr uint32_t KV_HALF = WIDEN ? C::KEYS * 128 : (F8MMA ? 0 : 1024);  // 64-column half stride
      constexpr uint32_t V_LBO = F8MMA ? 8192 : KV_HALF;      // F8MMA: one atom across d (unused)
      constexpr uint32_t V_KK = (F8MMA ? 4 : 2) * KV_SBO;     // PV: 16 (f16) or 32 (e4m3) keys per MMA
      // tcgen05.mma issue is close to synchronous: whatever this thread runs
      // between two MMAs (an mbarrier poll costs about as much as an N = 128
      // MMA) leaves the tensor core idle, and the thread shares its
      // sub-partition with two softmax warps.  So the loop keeps its
      // bookkeeping small: Q descriptors are built once, ring slots and
      // phases advance incrementally, and each batch of MMAs is issued from
      // one asm block with its descriptors already in registers.  The
      // descriptor of an operand at shared address x is the base descriptor
      // + (x >> 4) (every operand lies below 256 KB: the address field never
      // carries).
      const uint64_t KD0 = smem_desc_sw128(0, 16, KV_SBO), VD0 = smem_desc_sw128(0, V_LBO, KV_SBO);
      uint64_t dq[NQ][8];
#pragma unroll
      for (int qt = 0; qt < NQ; ++qt)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          // 16-bit Q: [half][128 rows][128 B], 8 steps of 16 elements; e4m3
          // Q (F8MMA): [128 rows][128 B] in the first half, 4 steps of 32
          dq[qt][kk] = F8MMA ? smem_desc_sw128(sbase + C::OFF_Q + qt * C::QT_BYTES + (kk & 3) * 32, 16, 1024)
                             : smem_desc_sw128(sbase + C::OFF_Q + qt * C::QT_BYTES + (kk >> 2) * (C::ROWS * 128) + (kk & 3) * 32,
                                               16, 1024);
      // S = Q_qt K^T into TMEM column d (K at shared address kx)
      auto s_batch = [&](uint32_t d, const uint64_t (&aq)[8], uint32_t kx) {
        const uint64_t dk = KD0 + (uint64_t)(kx >> 4);
        if constexpr (F8MMA) {
          uint64_t a4[4], bk[4];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            a4[kk] = aq[kk];
            bk[kk] = dk + (uint64_t)((kk * 32) >> 4);
          }
          umma_ss_x4_f8(d, a4, bk, id_s);
        } else {
          uint64_t bk[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) bk[kk] = dk + (uint64_t)(((kk >> 2) * KV_HALF + (kk & 3) * 32) >> 4);
          umma_ss_x8(d, aq, bk, id_s);
        }
      };
      // O (+)= P V: O at TMEM column d, P at column pc, V at shared address vx
      auto pv_batch = [&](uint32_t d, uint32_t pc, uint32_t vx, uint32_t acc0) {
        const uint64_t dv = VD0 + (uint64_t)(vx >> 4);
        uint64_t bv[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) bv[kk] = dv + (uint64_t)((kk * V_KK) >> 4);
        if constexpr (F8MMA) {
          umma_ts_x4_f8(d, pc, bv, id_o, acc0);   // P of keys 32 q at column 32 q
        } else {
          umma_ts_x4(d, pc + p_col(0), bv, id_o, acc0);
          umma_ts_x4(d, pc + p_col(4), bv + 4, id_o, 1u);
        }
      };
      // Ring cursors of the next K and V operands: bf16 operand u = 2 t (K_t)
      // or 2 t + 1 (V_t) of the running key tile count t sits in slot u % NSLOT,
      // FULL / EMPTY parity (u / NSLOT) & 1; fp8 K_t in widened buffer t % 2
      // (parity (t / 2) & 1), V_t in the one V buffer (parity t & 1).
      struct Cur {
        int slot;
        uint32_t par;
        int t;
      };
      Cur kc{0, 0u, 0}, vc{1, 0u, 0};  // K_0: operand 0, V_0: operand 1 (NSLOT >= 3)
      auto advance = [&](Cur& cu) {
        cu.slot += 2;
        if (cu.slot >= C::NSLOT) {
          cu.slot -= C::NSLOT;
          cu.par ^= 1u;
        }
        ++cu.t;
      };
      auto k_full = [&](const Cur& cu) { return WIDEN ? bar(B_CK_FULL + (cu.t & 1)) : bar(B_FULL + cu.slot); };
      auto k_par = [&](const Cur& cu) -> uint32_t { return WIDEN ? (uint32_t)(cu.t >> 1) & 1u : cu.par; };
      auto k_free = [&](const Cur& cu) { return WIDEN ? bar(B_CK_FREE + (cu.t & 1)) : bar(B_EMPTY + cu.slot); };
      auto k_base = [&](const Cur& cu) -> uint32_t {
        return WIDEN ? sbase + C::OFF_CONV + (cu.t & 1) * C::OP_BYTES : sbase + C::OFF_RING + cu.slot * C::SLOT_BYTES;
      };
      auto v_full = [&](const Cur& cu) { return WIDEN ? bar(B_CV_FULL) : bar(B_FULL + cu.slot); };
      auto v_par = [&](const Cur& cu) -> uint32_t { return WIDEN ? (uint32_t)cu.t & 1u : cu.par; };
      auto v_free = [&](const Cur& cu) { return WIDEN ? bar(B_CV_FREE) : bar(B_EMPTY + cu.slot); };
      auto v_base = [&](const Cur& cu) -> uint32_t {
        return WIDEN ? sbase + C::OFF_CONV + 2 * C::OP_BYTES : sbase + C::OFF_RING + cu.slot * C::SLOT_BYTES;
      };
      // releases of the last K / V operand (the exit waits for them)
      uint32_t last_k = 0, last_kp = 0, last_v = 0, last_vp = 0;
      auto free_k = [&]() {
        umma_commit(k_free(kc));
        last_k = k_free(kc);
        last_kp = k_par(kc);
        advance(kc);
      };
      auto free_v = [&]() {
        umma_commit(v_free(vc));
        last_v = v_free(vc);
        last_vp = v_par(vc);
        advance(vc);
      };
      // items (nit); per Q tile the S tiles issued (ns) and items completed
      // (no); PVs issued (npv, one Q tile with double-buffered S)
      int nit = 0, npv = 0;
      int ns[NQ], no[NQ];
#pragma unroll
      for (int qt = 0; qt < NQ; ++qt) ns[qt] = no[qt] = 0;
      bool live = true;
      ItemGeo g;
      for (int k = 0; live && take_geo_thread(k, g); ++k) {
        if (!g.ok) continue;
        if (!mbar_wait(bar(q_pass ? B_Q_READY : B_Q), nit & 1, abort_flag)) break;
        if constexpr (C::SBUF == 2) {
          // One Q tile, S double-buffered: step j issues S_j into buffer
          // (S count) % 2 before it waits for P_{j-1}, so the tensor core
          // computes S_j while the softmax still works on S_{j-1}.  S_j
          // overwrites P_{j-2}, whose PV was issued one step earlier (the MMAs
          // of this thread run in issue order).
          for (int j = 0; live && j <= g.n_tiles; ++j) {
            if (j < g.n_tiles) {
              if (!mbar_wait(k_full(kc), k_par(kc), abort_flag)) { live = false; break; }
              const int b = ns[0] & 1;
              s_batch(tmem + b * 128, dq[0], k_base(kc));
              umma_commit(bar(B_S_FULL + b));
              ++ns[0];
              if (j == g.n_tiles - 1) umma_commit(bar(B_Q_FREE));  // Q read by this item's last S
              free_k();
            }
            if (j >= 1) {
              if (!mbar_wait(v_full(vc), v_par(vc), abort_flag)) { live = false; break; }
              // the first PV of an item overwrites O: the previous item's
              // epilogue must have read it out
              if (j == 1 && no[0] >= 1 && !mbar_wait(bar(B_O_FREE), (no[0] - 1) & 1, abort_flag)) {
                live = false;
                break;
              }
              const int b = npv & 1;  // buffer of S_{j-1} / P_{j-1}
              if (!mbar_wait(bar(B_P_FULL + b), (npv >> 1) & 1, abort_flag)) { live = false; break; }
              tc_fence_after();
              pv_batch(tmem + C::COL_O, tmem + b * 128, v_base(vc), j > 1 ? 1u : 0u);
              umma_commit(bar(B_PV_DONE));
              if (j == g.n_tiles) umma_commit(bar(B_O_DONE));
              free_v();
              ++npv;
            }
          }
        } else {
          for (int j = 0; live && j <= g.n_tiles; ++j) {
            // step j: PV of tile j - 1 and S of tile j, Q tile by Q tile
            if (j < g.n_tiles && !mbar_wait(k_full(kc), k_par(kc), abort_flag)) { live = false; break; }
            if (j >= 1 && !mbar_wait(v_full(vc), v_par(vc), abort_flag)) { live = false; break; }
            const uint32_t kx = k_base(kc), vx = v_base(vc);
#pragma unroll
            for (int qt = 0; qt < NQ; ++qt) {
              if (qt >= g.nq) break;
              const uint32_t ts = tmem + qt * C::QT_COLS;  // S_qt / P_qt columns
              if (j >= 1) {
                // the first PV of an item overwrites O: the previous item's
                // epilogue must have read it out
                if (j == 1 && no[qt] >= 1 &&
                    !mbar_wait(bar(B_O_FREE + qt), (no[qt] - 1) & 1, abort_flag)) {
                  live = false;
                  break;
                }
                if (!mbar_wait(bar(B_P_FULL + qt), (ns[qt] - 1) & 1, abort_flag)) {
                  live = false;
                  break;
                }
                tc_fence_after();
                pv_batch(ts + C::COL_O, ts, vx, j > 1 ? 1u : 0u);
                if (j == g.n_tiles) umma_commit(bar(B_O_DONE + qt));
              }
              if (j < g.n_tiles) {
                s_batch(ts, dq[qt], kx);
                umma_commit(bar(B_S_FULL + qt));
                ++ns[qt];
              }
            }
            if (!live) break;
            if (j == g.n_tiles - 1) umma_commit(bar(B_Q_FREE));  // Q read by this item's last S
            if (j >= 1) free_v();
            if (j < g.n_tiles) free_k();
          }
        }
        if (!live) break;
#pragma unroll
        for (int qt = 0; qt < NQ; ++qt)
          if (qt < g.nq) ++no[qt];
        ++nit;
      }
      // the last slot releases land before the CTA's shared memory goes away
      if (live && !*abort_flag && kc.t >= 1) {
        mbar_wait(last_v, last_vp, abort_flag);
        mbar_wait(last_k, last_kp, abort_flag);
      }
    }
  } else if (WIDEN && (warp == 2 || warp == 3 || warp >= C::CONV_WARP0)) {
    // ---------------- fp8 -> scaled f16 widening ----------------
    // Step i of an item widens K_i, then V_{i-1}: K runs a tile ahead, since
    // S_i needs only K_i while V's single buffer frees up one PV later.
    const int ct = (warp < 4 ? warp - 2 : warp - C::CONV_WARP0 + 2) * 32 + lane;  // 0 .. 191
    constexpr int NCT = 32 * C::CONV_WARPS;
    int u0 = 0, t0 = 0;
    bool go = true;
    ItemGeo g;
    for (int k = 0; go && take_geo_warp(k, g); ++k) {
      if (!g.ok) continue;
      for (int i = 0; go && i <= g.n_tiles; ++i) {
        for (int v = 0; v < 2; ++v) {
          const int j = i - v;                            // tile of this operand
          if (j < 0 || j >= g.n_tiles) continue;
          const int u = u0 + 2 * j + v, s = u % C::NSLOT, n = u / C::NSLOT;
          const int tj = t0 + j;                          // running tile count
          if (!mbar_wait(bar(B_FULL + s), n & 1, abort_flag)) { go = false; break; }
          if (v == 0 && tj >= 2 && !mbar_wait(bar(B_CK_FREE + (tj & 1)), ((tj >> 1) - 1) & 1, abort_flag)) {
            go = false;
            break;
          }
          if (v == 1 && tj >= 1 && !mbar_wait(bar(B_CV_FREE), (tj - 1) & 1, abort_flag)) {
            go = false;
            break;
          }
          const int k0 = g.lo + j * C::KEYS;
          const uint8_t* raw = smem + C::OFF_RING + s * C::SLOT_BYTES;
          uint8_t* dst = smem + C::OFF_CONV + (v ? 2 : (tj & 1)) * C::OP_BYTES;
#pragma unroll  // all of a thread's chunks in flight at once (5-6 of them)
          for (int c = ct; c < C::KEYS * 8; c += NCT) {
            const int r = c >> 3, ch = c & 7;         // key row, 16-code group
            uint4 a = make_uint4(0u, 0u, 0u, 0u), bq = a;
            if (k0 + r < g.hi) {
              const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 128 + ch * 16);
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
            uint8_t* row = dst + (ch >> 2) * (C::KEYS * 128) + r * 128;
            const int c0 = (ch & 3) * 2;
            *reinterpret_cast<uint4*>(row + (((c0) ^ (r & 7)) << 4)) = a;
            *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = bq;
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(v ? B_CV_FULL : B_CK_FULL + (tj & 1)));
            mbar_arrive(bar(B_EMPTY + s));
          }
        }
      }
      u0 += 2 * g.n_tiles;
      t0 += g.n_tiles;
    }
  } else if (warp >= 4 && warp < 4 + 4 * NQ) {
    // ---------------- softmax / epilogue: one thread per row, 4 warps per Q tile ----------------
    const int qt = (warp - 4) >> 2;                 // Q tile of this warpgroup
    const int quad = warp & 3;                      // TMEM lane quarter this warp may access
    const int r = quad * 32 + lane;                 // row of the Q tile = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16) + qt * C::QT_COLS;
    float c = p.scale_log2;                         // logit scale (log2 units), per row for F8MMA
    float qsc = 1.f;                                // F8MMA: this row's query scale
    int ns = 0, no = 0, nit = 0, u0 = 0;            // S tiles seen, items done, items, ring base
    bool live = true;
    bool dep_waited = false;                        // this thread has waited for the previous grid
    ItemGeo g;
    for (int k = 0; live && take_geo_warp(k, g); ++k) {
      if (!g.ok) continue;
      const bool mine = qt < g.nq;
      if (q_pass) {
        // Q in place, each thread its own row of its Q tile: rotated at the
        // row's position (RoPE: element i with i + 64, i.e. chunk j of the
        // first 64-column half with chunk j of the second, the same swizzled
        // slot) and rounded to bf16, then widened to f16 for an fp8 cache.  A Q tile the item does not use still counts its arrival.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_Q), nit & 1, abort_flag))) { live = false; break; }
        if (mine) {
          const int brq = qt * C::ROWS + r;
          const bool rot = p.q_position != nullptr && brq < g.nrows;
          const int qpos = rot ? __ldg(p.q_position + g.qo0 + (g.row0 + brq) / G) : 0;
          uint8_t* h0 = smem + C::OFF_Q + qt * C::QT_BYTES + r * 128;
          uint8_t* h1 = h0 + C::QT_BYTES / 2;
          if (rot) {
#pragma unroll 1
            for (int jp = 0; jp < 8; ++jp) {
              uint4 a = *reinterpret_cast<uint4*>(h0 + jp * 16);
              uint4 b = *reinterpret_cast<uint4*>(h1 + jp * 16);
              const int i0 = (jp ^ (r & 7)) << 3;   // frequency index of the chunk's first element
              uint32_t* wa = reinterpret_cast<uint32_t*>(&a);
              uint32_t* wb = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float c0, s0, c1, s1;
                rope_cos_sin(qpos, p.rope.hi[i0 + 2 * k], p.rope.lo[i0 + 2 * k], &c0, &s0);
                rope_cos_sin(qpos, p.rope.hi[i0 + 2 * k + 1], p.rope.lo[i0 + 2 * k + 1], &c1, &s1);
                const float a0 = __uint_as_float(wa[k] << 16), a1 = __uint_as_float(wa[k] & 0xffff0000u);
                const float b0 = __uint_as_float(wb[k] << 16), b1 = __uint_as_float(wb[k] & 0xffff0000u);
                const float ya0 = fmaf(a0, c0, -b0 * s0), ya1 = fmaf(a1, c1, -b1 * s1);
                const float yb0 = fmaf(b0, c0, a0 * s0), yb1 = fmaf(b1, c1, a1 * s1);
                // the rotated query is a bf16 tensor; an fp8 cache's f16
                // MMAs take it widened (exactly) to f16
                wa[k] = pack_bf16x2(ya0, ya1);
                wb[k] = pack_bf16x2(yb0, yb1);
                if (WIDEN) {
                  wa[k] = bf16x2_to_f16x2(wa[k]);
                  wb[k] = bf16x2_to_f16x2(wb[k]);
                }
              }
              *reinterpret_cast<uint4*>(h0 + jp * 16) = a;
              *reinterpret_cast<uint4*>(h1 + jp * 16) = b;
            }
          } else if (WIDEN) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint4* q4 = reinterpret_cast<uint4*>(half ? h1 : h0);
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
          }
          if constexpr (F8MMA) {
            // e4m3 row with its own scale: q = q8 * qsc, qsc = amax |q| / 448;
            // the row (bf16, rotated if RoPE) is read whole before the e4m3
            // bytes overwrite its first half (the row's first 128 bytes hold
            // [128 elements] e4m3 in the same 128-byte swizzle)
            uint4 lo8[8];
            float amax = 0.f;
#pragma unroll
            for (int jp = 0; jp < 8; ++jp) {
              lo8[jp] = *reinterpret_cast<const uint4*>(h0 + jp * 16);
              const uint4 hb = *reinterpret_cast<const uint4*>(h1 + jp * 16);
              const uint32_t wa4[4] = {lo8[jp].x, lo8[jp].y, lo8[jp].z, lo8[jp].w};
              const uint32_t wb4[4] = {hb.x, hb.y, hb.z, hb.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                amax = fmax3(amax, fabsf(__uint_as_float(wa4[k] << 16)), fabsf(__uint_as_float(wa4[k] & 0xffff0000u)));
                amax = fmax3(amax, fabsf(__uint_as_float(wb4[k] << 16)), fabsf(__uint_as_float(wb4[k] & 0xffff0000u)));
              }
            }
            const float inv = amax > 0.f ? 448.f / amax : 1.f;
            qsc = amax > 0.f ? amax / 448.f : 1.f;
            const int x = r & 7;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int jp = 0; jp < 8; ++jp) {
                const uint4 w = half ? *reinterpret_cast<const uint4*>(h1 + jp * 16) : lo8[jp];
                const int e0 = 64 * half + 8 * (jp ^ x);       // first element of the chunk
                const uint32_t b0 = e4m3x4_rn_satfinite(
                    __uint_as_float(w.x << 16) * inv, __uint_as_float(w.x & 0xffff0000u) * inv,
                    __uint_as_float(w.y << 16) * inv, __uint_as_float(w.y & 0xffff0000u) * inv);
                const uint32_t b1 = e4m3x4_rn_satfinite(
                    __uint_as_float(w.z << 16) * inv, __uint_as_float(w.z & 0xffff0000u) * inv,
                    __uint_as_float(w.w << 16) * inv, __uint_as_float(w.w & 0xffff0000u) * inv);
                *reinterpret_cast<uint2*>(h0 + (((e0 >> 4) ^ x) << 4) + (e0 & 15)) = make_uint2(b0, b1);
              }
            }
          }
          fence_proxy_async();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_Q_READY));
      }
      ++nit;
      if constexpr (F8MMA) c = p.scale_log2 * qsc;
      if (!mine) {
        u0 += 2 * g.n_tiles;
        continue;
      }
      const int br = qt * C::ROWS + r;              // row of the block
      const bool row_ok = br < g.nrows;
      const int t = (g.row0 + br) / G;              // draft token of the row
      const int moff = g.moff;
      const int L = g.L, prefix = g.prefix, hi = g.hi;
      // A draft-block mask row of at most 64 bits is fetched once, here, so
      // its loads overlap the item's prefix tiles instead of stalling the
      // tile that holds the drafts.
      const bool row_bits_pre = p.mask && !p.mask_full && L <= 64 && hi > prefix;
      uint64_t row_bits = 0;
      if (row_bits_pre && t < L) {
        const long long bit0 = (long long)moff + (long long)t * L;
        const int sh = (int)(bit0 & 7);
        const int nbytes = (sh + L + 7) >> 3;        // <= 9
        uint64_t w = 0;
        uint32_t top = 0;
        for (int k = 0; k < nbytes; ++k) {
          const uint32_t byte = __ldg(p.mask + (bit0 >> 3) + k);
          if (k < 8) w |= (uint64_t)byte << (8 * k);
          else top = byte;
        }
        row_bits = (w >> sh) | (sh ? (uint64_t)top << (64 - sh) : 0ull);
        if (L < 64) row_bits &= (1ull << L) - 1ull;
      }
      float m_used = -INFINITY;                     // in units of s * c (log2 domain)
      float l = 0.f;
      for (int j = 0; live && j < g.n_tiles; ++j) {
        const int k0 = g.lo + j * C::KEYS;
        if constexpr (F8MMA) {
          // Rows of V_j past the chunk end inside the last 16-key box may hold
          // stale (even NaN) slots: zero them, since 0 * NaN would poison O
          // (e4m3 V as it landed: [keys][128 B])
          const int tail = hi - k0;
          if (qt == 0 && tail < C::KEYS && (tail & 15)) {
            const int u = u0 + 2 * j + 1, s = u % C::NSLOT;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_FULL + s), (u / C::NSLOT) & 1, abort_flag))) {
              live = false;
              break;
            }
            const int zlo = tail, zhi = (tail + 15) & ~15;
            uint8_t* vt = smem + C::OFF_RING + s * C::SLOT_BYTES;
            for (int z = r; z < (zhi - zlo) * 8; z += C::ROWS)
              *reinterpret_cast<uint4*>(vt + (zlo + z / 8) * 128 + ((z & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async();
          }
        }
        if constexpr (!FP8) {
          // Rows of V_j past the chunk end inside the last 16-key box may hold
          // stale (even NaN) slots: zero them, since 0 * NaN would poison O.
          // Q tile 0's warps do it before their P_j is posted; PV_j of every Q
          // tile is issued after that.
          const int tail = hi - k0;
          if (qt == 0 && tail < C::KEYS && (tail & 15)) {
            const int u = u0 + 2 * j + 1, s = u % C::NSLOT;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_FULL + s), (u / C::NSLOT) & 1, abort_flag))) {
              live = false;
              break;
            }
            const int zlo = tail, zhi = (tail + 15) & ~15;
            uint8_t* vt = smem + C::OFF_RING + s * C::SLOT_BYTES;
            for (int z = r; z < (zhi - zlo) * 16; z += C::ROWS) {
              const int row = zlo + z / 16, half = (z / 8) & 1, ch = z & 7;
              const int off = (row >> 3) * 2048 + half * 1024 + (row & 7) * 128;
              *reinterpret_cast<uint4*>(vt + off + (ch << 4)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async();
          }
        }
        // S_j: buffer ns % 2 of the one Q tile (double-buffered), else the Q
        // tile's only buffer
        const int sb = C::SBUF == 2 ? (ns & 1) : 0;
        const uint32_t s_addr = lane_addr + sb * 128;
        const uint32_t b_sp = C::SBUF == 2 ? sb : qt;  // S_FULL / P_FULL of this buffer
        const uint32_t s_par = C::SBUF == 2 ? (ns >> 1) & 1 : ns & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S_FULL + b_sp), s_par, abort_flag))) {
          live = false;
          break;
        }
        ++ns;
        tc_fence_after();
        // Visibility of the tile's keys for this row.  Causal drafts: keys below
        // lim = min(hi, prefix + t + 1) - k0.  Custom mask: one word per 32 keys
        // (prefix 1, drafts from the row's mask bits, nothing at or past hi).
        // A tile every row of the warp sees whole skips the per-key selects.
        const int lim = min(hi, prefix + t + 1) - k0;
        // keys of the item's first tile below its first key (0 .. 15 of them)
        const int lowcut = g.lov - k0;
        const uint32_t lowmask = lowcut > 0 ? ~((1u << lowcut) - 1u) : 0xffffffffu;
        uint32_t vis[C::KEYS / 32];
        bool full;
        if (!p.mask) {
          full = __all_sync(0xffffffffu, lim >= C::KEYS);
        } else if (p.mask_full) {
          // one row of kv_len = prefix + L bits per token, prefix included
          uint32_t all = 0xffffffffu;
#pragma unroll
          for (int q = 0; q < C::KEYS / 32; ++q) {
            const int g0 = k0 + 32 * q;
            uint32_t w32 = 0;
            if (g0 < hi && t < L) {
              const int nbits = min(32, hi - g0);
              const long long bit0 = (long long)moff + (long long)t * (prefix + L) + g0;
              const int nbytes = (int)((((bit0 & 7) + nbits) + 7) >> 3);
              uint64_t w = 0;
              for (int k = 0; k < nbytes; ++k) w |= (uint64_t)__ldg(p.mask + (bit0 >> 3) + k) << (8 * k);
              w >>= (bit0 & 7);
              w32 = (uint32_t)(w & (nbits >= 32 ? 0xffffffffull : ((1ull << nbits) - 1ull)));
            }
            vis[q] = w32;
            all &= w32;
          }
          full = __all_sync(0xffffffffu, all == 0xffffffffu);
        } else if (k0 + C::KEYS <= prefix && k0 + C::KEYS <= hi) {
          full = true;
#pragma unroll
          for (int q = 0; q < C::KEYS / 32; ++q) vis[q] = 0xffffffffu;
        } else {
          uint32_t all = 0xffffffffu;
#pragma unroll
          for (int q = 0; q < C::KEYS / 32; ++q) {
            const int g0 = k0 + 32 * q;
            uint32_t w32 = 0;
            if (g0 < hi) {
              const int below_prefix = min(max(prefix - g0, 0), 32);
              w32 = below_prefix == 32 ? 0xffffffffu : ((1u << below_prefix) - 1u);
              if (below_prefix < 32 && t < L) {
                // draft columns d = g0 + i - prefix for i >= below_prefix
                const int d0 = g0 + below_prefix - prefix;
                const long long bit0 = (long long)moff + (long long)t * L + d0;
                const int nbits = min(32 - below_prefix, L - d0);
                if (nbits > 0) {
                  uint64_t w = 0;
                  if (row_bits_pre) {
                    w = row_bits >> d0;
                  } else {
                    const int nbytes = (int)((((bit0 & 7) + nbits) + 7) >> 3);
                    for (int k = 0; k < nbytes; ++k)
                      w |= (uint64_t)__ldg(p.mask + (bit0 >> 3) + k) << (8 * k);
                    w >>= (bit0 & 7);
                  }
                  const uint32_t dbits =
                      (uint32_t)(w & (nbits >= 32 ? 0xffffffffull : ((1ull << nbits) - 1ull)));
                  w32 |= dbits << below_prefix;
                }
              }
              const int in_range = min(hi - g0, 32);
              if (in_range < 32) w32 &= (1u << in_range) - 1u;
            }
            vis[q] = w32;
            all &= w32;
          }
          full = __all_sync(0xffffffffu, all == 0xffffffffu);
        }
        if (lowcut > 0) {  // uniform over the item
          full = false;
          if (p.mask) vis[0] &= lowmask;
        }
        // Keys 32 q .. 32 q + 31 of the tile this row may see, one bit each.
        auto vis_word = [&](int q) -> uint32_t {
          if (!p.mask) {
            const int n = lim - 32 * q;
            const uint32_t w = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
            return q == 0 ? w & lowmask : w;
          }
          return q == 0 ? vis[0] : q == 1 ? vis[1] : q == 2 ? vis[2] : vis[3];
        };
        // One pass over the tile, 32 logits at a time (a rolled loop: a small
        // body keeps every warp's code in the instruction cache).  P is taken
        // against the row's reference max m_used (log2 units); a chunk whose
        // max exceeds it by more than 8 raises it by the least multiple of 8
        // that covers the chunk (the row's first visible chunk sets it to the
        // chunk max), so every P stays <= 2^8 and every rescale factor is an
        // exact power of two: the tile's P chunks written so far, the sums and
        // (once the tile is done) O are multiplied by it.  The scale-and-shift
        // and the sums run two logits per instruction (fp32x2), which leaves
        // more issue slots to the MMA issuer and the converter warps sharing
        // the sub-partitions.  With e4m3 MMAs the reference max is settled for the
        // whole tile first, in a pass of its own over S (read from tensor
        // memory twice): no P chunk is rescaled after it is written.  That
        // measured faster there (fp8 wide tree 198.0 -> 192.2 us) and slower
        // for the 16-bit P of the other variants (prefill 222.3 -> 230.5 us).
        auto mask_chunk = [&](uint32_t* raw, int q) {
          if (!full) {
            const uint32_t vw = vis_word(q);
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = ((vw >> i) & 1u) ? raw[i] : __float_as_uint(-INFINITY);
          }
        };
        float o_scale = 1.f;                   // product of this tile's rescale factors
        if constexpr (F8MMA) {
          float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
          for (int q = 0; q < C::KEYS / 32; ++q) {
            uint32_t raw[32];
            tmem_ld32(s_addr + q * 32, raw);
            tmem_wait_ld();
            mask_chunk(raw, q);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              mxs[i & 3] = fmax3(mxs[i & 3], __uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
          }
          const float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])) * c;  // c > 0
          if (mx > m_used + 8.f) {  // also when m_used = -inf and mx is finite
            if (m_used == -INFINITY) {
              o_scale = 0.f;  // nothing seen yet: l and O are 0
              m_used = mx;
            } else {
              const int k = (int)ceilf((mx - m_used - 8.f) * 0.125f);  // >= 1
              o_scale = k < 15 ? __int_as_float((127 - 8 * k) << 23) : 0.f;   // 2^-8k
              m_used += 8.f * (float)k;
            }
          }
        }
        uint64_t sums2[2] = {0ull, 0ull};      // fp32x2 pairs
#pragma unroll 1
        for (int q = 0; q < C::KEYS / 32; ++q) {
          uint32_t raw[32];
          tmem_ld32(s_addr + q * 32, raw);
          tmem_wait_ld();
          if constexpr (F8MMA) {
            mask_chunk(raw, q);
          } else {
            float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                mxs[i & 3] = fmax3(mxs[i & 3], __uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
            } else {
              const uint32_t vw = vis_word(q);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                raw[2 * i] = ((vw >> (2 * i)) & 1u) ? raw[2 * i] : __float_as_uint(-INFINITY);
                raw[2 * i + 1] = ((vw >> (2 * i + 1)) & 1u) ? raw[2 * i + 1] : __float_as_uint(-INFINITY);
                mxs[i & 3] = fmax3(mxs[i & 3], __uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
              }
            }
            const float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])) * c;  // c > 0
            const bool raise = mx > m_used + 8.f;  // also when m_used = -inf and mx is finite
            if (__any_sync(0xffffffffu, raise)) {
              float a = 1.f;
              if (raise) {
                if (m_used == -INFINITY) {
                  a = 0.f;  // nothing seen yet: every sum so far is 0
                  m_used = mx;
                } else {
                  const int k = (int)ceilf((mx - m_used - 8.f) * 0.125f);  // >= 1
                  a = k < 15 ? __int_as_float((127 - 8 * k) << 23) : 0.f;   // 2^-8k
                  m_used += 8.f * (float)k;
                }
              }
              if (q > 0) {
                // this tile's P chunks 0 .. q-1, already in tensor memory
                tmem_wait_st();
                for (int q2 = 0; q2 < q; ++q2) {
                  uint32_t pk[16];
                  tmem_ld16(s_addr + 32 * q2, pk);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 16; ++i) pk[i] = FP8 ? scale_f16x2(pk[i], a) : scale_bf16x2(pk[i], a);
                  tmem_st16(s_addr + 32 * q2, pk);
                }
              }
#pragma unroll
              for (int i = 0; i < 2; ++i) sums2[i] = f32x2(f32x2_lo(sums2[i]) * a, f32x2_hi(sums2[i]) * a);
              o_scale *= a;
            }
          }
          // P of these 32 logits into columns 32 q .. 32 q + 15
          const float base = m_used == -INFINITY ? 0.f : m_used;
          const uint64_t cc = f32x2(c, c), nb = f32x2(-base, -base);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = fma_f32x2(f32x2(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1])), cc, nb);
            const float p0 = ex2(f32x2_lo(x)), p1 = ex2(f32x2_hi(x));
            sums2[i & 1] = add_f32x2(sums2[i & 1], f32x2(p0, p1));
            if constexpr (F8MMA) {
              raw[2 * i] = __float_as_uint(p0);     // packed four to a column below
              raw[2 * i + 1] = __float_as_uint(p1);
            } else {
              pk[i] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
          }
          if constexpr (F8MMA) {
            // P of the 32 logits as e4m3, four keys to a column, into columns
            // 32 q .. 32 q + 7 (P <= 2^8 < 448 by the lazy reference max)
#pragma unroll
            for (int w = 0; w < 8; ++w)
              pk[w] = e4m3x4_rn_satfinite(__uint_as_float(raw[4 * w]), __uint_as_float(raw[4 * w + 1]),
                                          __uint_as_float(raw[4 * w + 2]), __uint_as_float(raw[4 * w + 3]));
            tmem_st8(s_addr + 32 * q, pk);
          } else {
            tmem_st16(s_addr + 32 * q, pk);
          }
        }
        const float sum = (f32x2_lo(sums2[0]) + f32x2_hi(sums2[0])) + (f32x2_lo(sums2[1]) + f32x2_hi(sums2[1]));
        l = l * o_scale + sum;
        // O holds P_0 V .. P_{j-1} V against the old reference: rescale it once
        // PV_{j-1} is done with it (with a single S buffer it completed before
        // S_j did; a double-buffered S_j may complete first, so wait for it)
        if (j >= 1 && __any_sync(0xffffffffu, o_scale != 1.f)) {
          if (C::SBUF == 2) {
            // PV of the previous S tile (global count ns - 2) has completed
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_PV_DONE), (ns - 2) & 1, abort_flag))) live = false;
            tc_fence_after();
          }
          for (int q = 0; q < C::D / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(lane_addr + C::COL_O + q * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * o_scale);
            tmem_st32(lane_addr + C::COL_O + q * 32, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL + b_sp));
      }
      if (!live) break;
      // epilogue
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_O_DONE + qt), no & 1, abort_flag))) { live = false; break; }
      tc_fence_after();
      const float lse = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      const float inv = l > 0.f ? p.v_scale / l : 0.f;
      // The first write of this thread waits for the previous grid: an item
      // whose tiles all went out before the producer's wait could otherwise
      // finish before it, and that grid may still read the workspace (a
      // merge of the previous call) or the output
      if (!dep_waited) {
        grid_dependency_wait();
        dep_waited = true;
      }
      // Output row of block row br (token-major: token br / G, head h G + br % G).
      auto out_row = [&](int brr) -> size_t {
        const int tt = (g.row0 + brr) / G;
        return (size_t)(g.qo0 + tt) * p.h_q + (size_t)g.h * G + ((g.row0 + brr) - tt * G);
      };
      if (row_ok) {
        if (g.part_row < 0) {
          if (p.lse) p.lse[out_row(br)] = lse;
        } else {
          p.part_lse[(size_t)g.part_row + br] = lse;
        }
      }
      // O read as 16-lane x 256-bit fragments: four neighbouring threads
      // hold eight consecutive columns of one row, so a warp's store covers
      // eight rows in 32-byte (fp32) or 16-byte (bf16) runs instead of 32
      // rows in 16-byte pieces.  Rows ra = 32 quad + 16 hl + lane / 4 and
      // ra + 8; their scale comes from the lanes that own them.
#pragma unroll 1
      for (int hl = 0; hl < 2; ++hl) {
        const int rl = 16 * hl + (lane >> 2);
        const float inv_a = __shfl_sync(0xffffffffu, inv, rl);
        const float inv_b = __shfl_sync(0xffffffffu, inv, rl + 8);
        const int br_a = qt * C::ROWS + quad * 32 + rl, br_b = br_a + 8;
        const bool ok_a = br_a < g.nrows, ok_b = br_b < g.nrows;
        const int c_lo = 2 * (lane & 3);
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t ov[32];
          tmem_ld_16x256b_x8(tmem + ((uint32_t)(quad * 32 + 16 * hl) << 16) + qt * C::QT_COLS + C::COL_O + 64 * cc, ov);
          tmem_wait_ld();
          if (g.part_row < 0) {
            __nv_bfloat16* da = static_cast<__nv_bfloat16*>(p.out) + (ok_a ? out_row(br_a) : 0) * C::D + 64 * cc + c_lo;
            __nv_bfloat16* db = static_cast<__nv_bfloat16*>(p.out) + (ok_b ? out_row(br_b) : 0) * C::D + 64 * cc + c_lo;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (ok_a)
                *reinterpret_cast<uint32_t*>(da + 8 * k) =
                    pack_bf16x2(__uint_as_float(ov[4 * k]) * inv_a, __uint_as_float(ov[4 * k + 1]) * inv_a);
              if (ok_b)
                *reinterpret_cast<uint32_t*>(db + 8 * k) =
                    pack_bf16x2(__uint_as_float(ov[4 * k + 2]) * inv_b, __uint_as_float(ov[4 * k + 3]) * inv_b);
            }
          } else {
            float* da = p.part_out + ((size_t)g.part_row + br_a) * C::D + 64 * cc + c_lo;
            float* db = p.part_out + ((size_t)g.part_row + br_b) * C::D + 64 * cc + c_lo;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (ok_a)
                *reinterpret_cast<float2*>(da + 8 * k) =
                    make_float2(__uint_as_float(ov[4 * k]) * inv_a, __uint_as_float(ov[4 * k + 1]) * inv_a);
              if (ok_b)
                *reinterpret_cast<float2*>(db + 8 * k) =
                    make_float2(__uint_as_float(ov[4 * k + 2]) * inv_b, __uint_as_float(ov[4 * k + 3]) * inv_b);
            }
          }
        }
      }
      // O has been read: the next item's first PV may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_O_FREE + qt));
      ++no;
      u0 += 2 * g.n_tiles;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) atomicOr(p.status, VA_DEV_TIMEOUT);
}

template <bool FP8, int NQ, bool F8MMA = false>
cudaError_t launch_tc(const PartialParams& p, const TcMaps& maps, int n_items,
                      cudaStream_t stream) {
  using C = TcCfg<FP8, NQ, F8MMA>;
  auto kern = verify_partial_tc_kernel<FP8, NQ, F8MMA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<PartialParams*>(&p), const_cast<TcMaps*>(&maps)};
  // persistent: one CTA per item chain of the plan (one per SM)
  (void)n_items;
  if (p.n_ctas <= 0) return cudaSuccess;
  return launch_kernel(reinterpret_cast<const void*>(kern), dim3(p.n_ctas), dim3(C::THREADS),
                       C::SMEM, stream, args, /*pdl=*/true);
}

}  // namespace

cudaError_t launch_partial_tc(const PartialParams& p, const TcMaps& maps, bool kv_fp8,
                              int block_rows, int n_items, bool f8mma, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (f8mma) {
    if (!kv_fp8) return cudaErrorInvalidValue;
    return block_rows == 256 ? launch_tc<true, 2, true>(p, maps, n_items, stream)
                             : launch_tc<true, 1, true>(p, maps, n_items, stream);
  }
  if (block_rows == 256)
    return kv_fp8 ? launch_tc<true, 2>(p, maps, n_items, stream)
                  : launch_tc<false, 2>(p, maps, n_items, stream);
  return kv_fp8 ? launch_tc<true, 1>(p, maps, n_items, stream)
                : launch_tc<false, 1>(p, maps, n_items, stream);
}

}  // namespace va
