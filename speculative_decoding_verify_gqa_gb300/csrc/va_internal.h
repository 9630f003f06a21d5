// Internal definitions shared by the host planner, the C ABI and the kernels
// of libverify_attn.so: the plan's header and work-list records, and the
// workspace layout.  Not part of the public ABI.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace va {

constexpr uint32_t kPlanMagic = 0x31504156u;  // "VAP1"
constexpr uint32_t kPlanVersion = 4;

// Key tile of the partial kernels (keys per pipeline stage).  Split chunks are
// cut on multiples of it, so every tile starts on a page boundary whenever
// page_size <= kTileKeys, and lies inside one page otherwise.
constexpr int kTileKeys = 64;
// Key tile of the tcgen05 variants (the MMA's N for S = Q K^T), and the rows
// of one of their Q tiles.
constexpr int kTcTileKeys = 128;
constexpr int kTcRowsPerTile = 128;

// Kernel variants (values match VA_KERNEL_* in verify_attn.h).
enum Kernel : int32_t {
  kKernelMma64 = 1,   // warp-level mma.sync, 4 warps x 16 rows
  kKernelMma128 = 2,  // warp-level mma.sync, 8 warps x 16 rows
  kKernelTc128 = 3,   // tcgen05 + TMA, 128 rows per CTA
  kKernelTc256 = 4,   // tcgen05 + TMA, two 128-row Q tiles per CTA
};

inline int kernel_rows(int k) { return k == kKernelMma64 ? 64 : k == kKernelTc256 ? 256 : 128; }
inline bool kernel_is_tc(int k) { return k == kKernelTc128 || k == kKernelTc256; }
inline int kernel_threads(int k) { return k == kKernelMma64 ? 128 : 256; }
inline int kernel_ctas_per_sm(int k) { return k == kKernelMma64 ? 2 : 1; }

// One CTA's work: rows [row0, row0 + nrows) of request b's KV head h (row r is
// query head h * G + r % G at draft token r / G: the G heads sharing the KV
// head sit next to each other), against kv positions [kv_lo, kv_hi).
// part_row < 0: the item covers the unit's whole kv range and writes the final
// out / lse; otherwise it writes fp32 partials at rows part_row .. of the
// workspace partial buffers.  next: for the persistent tcgen05 variants, the
// index of the next item of the same CTA (-1 at the end of its chain; chain c
// starts at item c); -1 for the others.
struct WorkItem {
  int32_t b, h, row0, nrows;
  int32_t kv_lo, kv_hi, part_row, next;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// One split unit to merge: nsplit partials of nrows rows each, split s at
// part rows part_row0 + s * nrows.
struct MergeItem {
  int32_t b, h, row0, nrows;
  int32_t part_row0, nsplit, pad0, pad1;
};
static_assert(sizeof(MergeItem) == 32, "MergeItem layout");

// Host plan buffer: PlanHeader, then n_items WorkItems, then n_merge
// MergeItems.  The WorkItems and MergeItems are uploaded verbatim to the
// device workspace at off_items.
// PlanHeader::flags: the call features the plan was made for.
constexpr int64_t kPlanMaskFull = 1;  // mask rows of kv_len bits (prefix included)
constexpr int64_t kPlanNhd = 2;       // cache layout [pages, P, h_kv, d]
constexpr int64_t kPlanRope = 4;      // queries rotated at their positions
constexpr int64_t kPlanF8Mma = 8;     // e4m3 MMAs: queries quantised per row, P as e4m3

struct PlanHeader {
  uint32_t magic, version;
  int32_t batch, h_q, h_kv, head_dim, page_size, q_dtype, kv_dtype, has_mask;
  int32_t group, kernel, block_rows, tile_keys;
  int32_t n_items, n_merge, n_units, num_sms;
  int64_t total_qo, part_rows, chunk;
  uint64_t off_status, off_items, off_merge, off_part_lse, off_part_out, ws_bytes;
  uint64_t plan_bytes;
  int64_t flags;    // feature bits of the call the plan serves (0: none)
  int64_t n_ctas;   // persistent tcgen05 variants: CTAs (item chains); 0 otherwise
  int64_t head_dim_v;  // elements of a value row (v_cache, partials and out)
  int64_t max_nsplit;  // largest split count of a merge item (0: no merges)
};
static_assert(sizeof(PlanHeader) == 184, "PlanHeader layout (read by the Python binding)");

constexpr size_t kWsAlign = 256;
constexpr int kMaxHeadDimV = 128;  // widest value row a plan may have
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace va
