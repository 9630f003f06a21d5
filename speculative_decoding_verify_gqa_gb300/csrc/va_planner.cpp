// Host planner for paged-KV GQA verify attention (no CUDA calls).
//
// Restates the work decomposition of "flashmap 0.1.0 -- flashmap/sglang/
// verify_attention.py" (one program per request, KV head, row block and kv
// split; row blocks of up to 128 rows; splits sized to fill the GPU's SMs for
// a few waves, each holding at least a minimum chunk of keys) and the
// plan-once / run-many split of FlashInfer PR #286 "Separate Q and KV dtypes
// for decode" (begin_forward reads the index arrays on the host, sizes the
// split from the SM count, and caches the result for many forward calls).
//
// Differences from the page's planner, for this GPU: the split count is
// chosen per (request, KV head, row block) from its own kv length rather
// than one power of two for the whole batch, so a batch of very different
// prefix lengths is cut into chunks of near-equal size; the verify tokens are
// not a separate split (they are appended into the pages first and fall in the
// last chunk); and the work list is sorted longest-first so the hardware
// block scheduler packs the SMs evenly.
#include <algorithm>
#include <cstring>
#include <functional>
#include <map>
#include <vector>

#include "../../include/verify_attn.h"
#include "va_internal.h"

namespace va {

namespace {

constexpr int kMaxTargetPerSm = 4;

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Unit {
  int32_t b, row0, nrows, kv_end;
};

}  // namespace

int check_common(int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int q_dtype,
                 int kv_dtype) {
  if (num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0)
    return VA_ERR_INVALID_ARGUMENT;
  if (num_qo_heads % num_kv_heads != 0) return VA_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return VA_ERR_UNSUPPORTED;
  if (!is_pow2(page_size) || page_size > 256) return VA_ERR_UNSUPPORTED;
  if (q_dtype != VA_DTYPE_BF16) return VA_ERR_UNSUPPORTED;
  if (kv_dtype != VA_DTYPE_BF16 && kv_dtype != VA_DTYPE_FP8_E4M3) return VA_ERR_UNSUPPORTED;
  return VA_OK;
}

int plan_bounds(int batch, int64_t total_qo, int num_qo_heads, int num_kv_heads, int head_dim,
                int num_sms, size_t* plan_bytes, size_t* workspace_bytes) {
  if (!plan_bytes || !workspace_bytes || batch < 0 || total_qo < 0 || num_sms <= 0 ||
      num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads || head_dim <= 0)
    return VA_ERR_INVALID_ARGUMENT;
  // Units: a request's G * L_b rows in blocks of >= 64 rows, per KV head.
  int64_t units = ceil_div((int64_t)num_qo_heads * total_qo, 64) + (int64_t)num_kv_heads * batch;
  int64_t target = (int64_t)kMaxTargetPerSm * num_sms;
  // sum_u ceil(kv_end_u / C) <= W / C + units <= target + units, plus at most
  // one draft item per unit.
  int64_t items = target + 2 * units;
  // Split units hold kv_end > C keys, so their split counts total < 2 W / C
  // <= 2 target (3 target with a draft item each: n + 1 <= 1.5 n for n >= 2),
  // each with at most the largest block's rows (256).
  int64_t part_rows = 256 * 3 * target;
  size_t pb = sizeof(PlanHeader) + (size_t)(items + units) * 32;
  size_t ws = kWsAlign + (size_t)(items + units) * 32;
  ws = align_up(ws, kWsAlign) + (size_t)part_rows * 4;
  // partial rows of the widest value row a plan may have (head_dim_v <= 128)
  ws = align_up(ws, kWsAlign) + (size_t)part_rows * std::max(head_dim, kMaxHeadDimV) * 4;
  *plan_bytes = pb;
  *workspace_bytes = align_up(ws, kWsAlign);
  return VA_OK;
}

int plan_host(const int32_t* kv_indptr, const int32_t* qo_indptr, const int32_t* last_page_len,
              const int32_t* mask_indptr, int batch, int num_qo_heads, int num_kv_heads,
              int head_dim, int page_size, int q_dtype, int kv_dtype, int has_mask, int num_sms,
              const va_plan_options_t* opts, void* plan_h, size_t plan_bytes,
              size_t* workspace_bytes) {
  if (!workspace_bytes || !plan_h || batch < 0 || num_sms <= 0) return VA_ERR_INVALID_ARGUMENT;
  if (!kv_indptr || !qo_indptr || (batch > 0 && !last_page_len)) return VA_ERR_INVALID_ARGUMENT;
  if (has_mask && !mask_indptr) return VA_ERR_INVALID_ARGUMENT;
  int rc = check_common(num_qo_heads, num_kv_heads, head_dim, page_size, q_dtype, kv_dtype);
  if (rc) return rc;
  va_plan_options_t o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.max_splits < 0 || o.min_chunk < 0 || o.target_ctas < 0) return VA_ERR_INVALID_ARGUMENT;
  if ((o.mask_layout != VA_MASK_QLEN && o.mask_layout != VA_MASK_FULL) ||
      (o.kv_layout != VA_LAYOUT_HND && o.kv_layout != VA_LAYOUT_NHD) || (o.rope != 0 && o.rope != 1))
    return VA_ERR_INVALID_ARGUMENT;
  const bool full_mask = o.mask_layout == VA_MASK_FULL;
  if (o.q_fp8 != 0 && o.q_fp8 != 1) return VA_ERR_INVALID_ARGUMENT;
  if (o.draft_items < -1 || o.draft_items > 1) return VA_ERR_INVALID_ARGUMENT;
  if (o.head_dim_v < 0) return VA_ERR_INVALID_ARGUMENT;
  const int dv = o.head_dim_v ? o.head_dim_v : head_dim;
  if (dv != 64 && dv != 128) return VA_ERR_UNSUPPORTED;
  if (o.q_fp8 && kv_dtype != VA_DTYPE_FP8_E4M3) return VA_ERR_UNSUPPORTED;
  if (full_mask && !has_mask) return VA_ERR_INVALID_ARGUMENT;
  if (o.kernel != VA_KERNEL_AUTO && o.kernel != VA_KERNEL_MMA_64 && o.kernel != VA_KERNEL_MMA_128 &&
      o.kernel != VA_KERNEL_TC_128 && o.kernel != VA_KERNEL_TC_256)
    return VA_ERR_INVALID_ARGUMENT;

  const int G = num_qo_heads / num_kv_heads;
  if (qo_indptr[0] < 0 || kv_indptr[0] < 0) return VA_ERR_INVALID_ARGUMENT;
  int64_t max_rows = 0;
  std::vector<int64_t> prefix(batch), qlen(batch);
  for (int b = 0; b < batch; ++b) {
    int64_t np = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    int64_t L = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    if (np < 0 || L < 0) return VA_ERR_INVALID_ARGUMENT;
    int64_t kv_len = 0;
    if (np > 0) {
      if (last_page_len[b] < 1 || last_page_len[b] > page_size) return VA_ERR_INVALID_ARGUMENT;
      kv_len = (np - 1) * page_size + last_page_len[b];
    }
    if (kv_len > INT32_MAX) return VA_ERR_UNSUPPORTED;
    if (kv_len < L) return VA_ERR_INVALID_ARGUMENT;
    if (has_mask) {
      const int64_t cols = full_mask ? kv_len : L;
      if (mask_indptr[b] < 0 || (int64_t)mask_indptr[b + 1] - mask_indptr[b] != L * cols)
        return VA_ERR_INVALID_ARGUMENT;
    }
    if ((int64_t)G * L > INT32_MAX) return VA_ERR_UNSUPPORTED;
    prefix[b] = kv_len - L;
    qlen[b] = L;
    max_rows = std::max(max_rows, (int64_t)G * L);
  }

  // The tensor-core variant serves head_dim 128, page sizes that are multiples
  // of its 16-row TMA boxes, and groups that tile its 128 rows.
  const bool tc_ok = head_dim == 128 && dv == head_dim && page_size % 16 == 0 && 128 % G == 0;
  int kernel = o.kernel;
  if ((kernel == VA_KERNEL_TC_128 || kernel == VA_KERNEL_TC_256) && !tc_ok) return VA_ERR_UNSUPPORTED;
  // e4m3 MMAs exist in the tcgen05 variants only
  if (o.q_fp8 && (!tc_ok || kernel == VA_KERNEL_MMA_64 || kernel == VA_KERNEL_MMA_128))
    return VA_ERR_UNSUPPORTED;
  if (kernel == VA_KERNEL_AUTO) {
    // Measured on GB300: the tcgen05 variants beat the warp-level one on every
    // shape they serve (mma.sync runs at a fraction of the tensor-core rate
    // there, so even verify-sized blocks that fill half of the 128-row MMA
    // come out ahead); two Q tiles per CTA once a KV head has > 128 rows.  The
    // warp-level variant keeps head_dim 64, odd page sizes and groups that do
    // not tile 128 rows.
    if (tc_ok) kernel = max_rows > 128 ? kKernelTc256 : kKernelTc128;
    else kernel = max_rows <= 64 ? kKernelMma64 : kKernelMma128;
  }
  const int BM = kernel_rows(kernel);
  // chunks are cut on the key tile of the chosen variant
  const int TK = kernel_is_tc(kernel) ? kTcTileKeys : kTileKeys;

  // Units of work: row blocks of each request (times each KV head).  Without
  // a mask a row block's last visible key is that of its last token, prefix +
  // t_max; a custom mask may let a draft see later drafts, so its rows scan
  // the request's whole kv range.
  std::vector<Unit> units;
  int64_t W = 0;
  int max_unit_rows = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t R = (int64_t)G * qlen[b];
    for (int64_t row0 = 0; row0 < R; row0 += BM) {
      int32_t nrows = (int32_t)std::min<int64_t>(BM, R - row0);
      int64_t tmax = (row0 + nrows - 1) / G;
      int32_t kv_end = (int32_t)(has_mask ? prefix[b] + qlen[b] : prefix[b] + tmax + 1);
      units.push_back({b, (int32_t)row0, nrows, kv_end});
      W += (int64_t)kv_end * num_kv_heads;
      max_unit_rows = std::max(max_unit_rows, (int)nrows);
    }
  }

  // Split size.  A CTA's cost is modelled in bytes: its K/V rows (2 * D * es
  // per key), a fixed prologue / pipeline-fill cost, and for a split item its
  // fp32 partial (written, then read by the merge, mostly inside L2).  The
  // hardware hands the longest-first list to the SMs as they free up, so for
  // a few candidate wave counts the chunk size is derived from the total key
  // count, the list is packed onto the CTA slots longest-first, and the
  // candidate with the smallest estimated finish time wins.
  // the 128-row tensor-core variant fits two CTAs per SM with bf16 caches, one
  // with fp8; the 256-row one fills an SM's tensor memory alone
  const int64_t slots =
      (int64_t)num_sms * (kernel == kKernelTc128 ? (kv_dtype == VA_DTYPE_BF16 ? 2 : 1)
                                                : kernel_ctas_per_sm(kernel));
  const int es = kv_dtype == VA_DTYPE_FP8_E4M3 ? 1 : 2;
  const int64_t key_bytes = (int64_t)(head_dim + dv) * es;
  // fixed cost of a work item (prologue, pipeline fill and drain, epilogue)
  // in K/V-byte equivalents: about one key tile for both variants (the
  // persistent tcgen05 CTAs overlap part of it with the previous item); on
  // GB300 the fp8 wide tree measured 407 us with 7 splits per unit against
  // 447 us with 2, which a larger value would have chosen
  const int64_t fixed_bytes = kernel_is_tc(kernel) ? 64 * 1024 : 48 * 1024;
  const int64_t partial_bytes_per_row = 4LL * dv;
  int64_t min_chunk = o.min_chunk > 0 ? o.min_chunk : 2 * TK;
  min_chunk = ceil_div(min_chunk, TK) * TK;
  auto chunk_for = [&](int64_t target) {
    return std::max<int64_t>(min_chunk,
                             ceil_div(ceil_div(W, std::max<int64_t>(target, 1)), TK) * TK);
  };
  // A unit is cut either into near-equal chunks (equal = true) or into full
  // chunks of the target size plus a shorter remainder; the remainders let
  // the longest-first packing fill SMs that equal cuts would leave idle.
  auto split_of = [&](const Unit& u, int64_t chunk, bool equal, int64_t* cu) {
    int64_t n = ceil_div(u.kv_end, chunk);
    if (o.max_splits > 0) n = std::min<int64_t>(n, o.max_splits);
    n = std::max<int64_t>(n, 1);
    *cu = equal || n * chunk < u.kv_end ? ceil_div(ceil_div(u.kv_end, n), TK) * TK : chunk;
    return ceil_div(u.kv_end, *cu);
  };
  // Latency regime (tcgen05, at most four key tiles of K / V per SM: the
  // verify steps of one or a few requests): spreading the keys over every SM
  // in the shortest chunks costs more than it gains -- each CTA's set-up and
  // epilogue, the later start of CTAs on SMs the previous kernel still holds,
  // a merge over more partials.  On GB300 the Llama-3-8B tree verify step
  // measured 10.7 us with 96 CTAs against 11.6-12.2 us with 136 and 11.3 us
  // with 72, so there the candidates aim at two thirds of the SMs.
  const bool latency = kernel_is_tc(kernel) && W * key_bytes <= 4LL * 64 * 1024 * num_sms;
  const int64_t cand_slots = latency ? std::max<int64_t>(1, 2 * (int64_t)num_sms / 3) : slots;
  int64_t chunk;
  double best_lpt = -1.0;  // the chosen split candidate's estimated finish
  bool equal = true;
  if (o.target_ctas > 0) {
    chunk = chunk_for(std::min<int64_t>(o.target_ctas, kMaxTargetPerSm * num_sms));
  } else {
    chunk = chunk_for(cand_slots);
    double best = -1.0;
    std::vector<std::pair<int64_t, int64_t>> groups;  // (item cost, items)
    std::map<int64_t, int64_t> loads;                  // slot load -> slots
    // candidates: 1-4 waves of CTA slots, equal or full-plus-remainder cuts;
    // for the persistent tcgen05 variants (items dealt onto one chain per
    // SM), when the units alone would leave SMs idle, also the longest unit
    // cut into n equal chunks for the n that make the item count land near a
    // multiple of the SM count, so that the dealing can even the chains out.
    // Chunks at least as long as the longest unit leave every unit whole and
    // are scored once.
    int64_t longest = 0;
    for (const Unit& u : units) longest = std::max<int64_t>(longest, u.kv_end);
    const int64_t whole = std::max<int64_t>(min_chunk, ceil_div(longest, TK) * TK);
    std::vector<std::pair<int64_t, bool>> cands;
    auto add = [&](int64_t c, bool eq) {
      if (c >= whole) {
        c = whole;
        eq = true;
      }
      for (const auto& x : cands)
        if (x.first == c && x.second == eq) return;
      cands.push_back({c, eq});
    };
    for (int cand = 0; cand < 8; ++cand) {
      const int waves = 1 + (cand >> 1);
      const int64_t target = std::min<int64_t>(waves * cand_slots, kMaxTargetPerSm * num_sms);
      add(chunk_for(target), (cand & 1) == 0);
    }
    const int64_t unit_heads = std::max<int64_t>(1, (int64_t)units.size() * num_kv_heads);
    if (kernel_is_tc(kernel) && unit_heads < cand_slots) {
      for (int64_t k = 1; k <= 6; ++k) {
        const int64_t n0 = (k * cand_slots + unit_heads / 2) / unit_heads;
        for (int64_t n = std::max<int64_t>(1, n0 - 1); n <= std::min<int64_t>(32, n0 + 1); ++n)
          add(std::max<int64_t>(min_chunk, ceil_div(ceil_div(longest, n), TK) * TK), true);
      }
    }
    for (const auto& cand : cands) {
      const int64_t c = cand.first;
      const bool eq = cand.second;
      // The candidate's items as (cost, count) groups: a unit's chunks are
      // cu keys long but the last, and each runs on every KV head.
      groups.clear();
      for (const Unit& u : units) {
        int64_t cu;
        const int64_t n = split_of(u, c, eq, &cu);
        const int64_t extra = fixed_bytes + (n > 1 ? (int64_t)u.nrows * partial_bytes_per_row : 0);
        if (n > 1) groups.push_back({extra + cu * key_bytes, (n - 1) * num_kv_heads});
        groups.push_back({extra + (u.kv_end - (n - 1) * cu) * key_bytes, (int64_t)num_kv_heads});
      }
      std::sort(groups.begin(), groups.end(),
                [](const std::pair<int64_t, int64_t>& a, const std::pair<int64_t, int64_t>& b) {
                  return a.first > b.first;
                });
      // Longest first onto the least-loaded slot, a group at a time: the slot
      // loads are kept as (load, number of slots) levels, and the items of a
      // group fill the lowest level one slot each before the next level is
      // reached -- the same loads as placing the items one by one.
      loads.clear();
      loads[0] = cand_slots;
      for (const auto& gr : groups) {
        int64_t cnt = gr.second;
        while (cnt > 0) {
          auto lo = loads.begin();
          const int64_t level = lo->first, take = std::min(cnt, lo->second);
          if ((lo->second -= take) == 0) loads.erase(lo);
          loads[level + gr.first] += take;
          cnt -= take;
        }
      }
      const int64_t finish = loads.rbegin()->first;
      if (best < 0 || (double)finish < best * 0.97) {
        best = (double)finish;
        chunk = c;
        equal = eq;
      }
    }
    best_lpt = best;
  }

  struct Tmp {
    WorkItem it;
    int64_t cost;
  };
  std::vector<Tmp> items;
  std::vector<MergeItem> merges;
  int64_t part_rows = 0;
  std::vector<int64_t> cuts;
  int64_t n_ctas = 0;

  // Stream cut (two-Q-tile persistent kernel): the key tiles of every unit,
  // unit after unit, cut into one run of equal length per CTA; a CTA's run is
  // its chain of items (pieces of the units it crosses), and only the units a
  // run boundary falls inside are merged -- fewer and larger partials than
  // cutting every unit, at the same balance.  Scored with the same cost
  // model as the split candidates and taken when clearly cheaper.
  bool stream = false;
  if (kernel == kKernelTc256 && o.target_ctas == 0 && o.max_splits == 0 && o.draft_items != 1 &&
      best_lpt > 0) {
    int64_t total = 0;
    for (const Unit& u : units) total += ceil_div(u.kv_end, TK) * num_kv_heads;
    const int64_t n = std::min<int64_t>(num_sms, total);
    // run c covers global tiles [run_lo(c), run_lo(c + 1))
    auto run_lo = [&](int64_t c) { return c * total / n; };
    std::vector<int64_t> cost((size_t)n, 0);
    int64_t g = 0, c = 0;
    for (const Unit& u : units) {
      const int64_t T = ceil_div(u.kv_end, TK);
      for (int h = 0; h < num_kv_heads; ++h, g += T) {
        while (run_lo(c + 1) <= g) ++c;
        const bool split = run_lo(c + 1) < g + T;
        for (int64_t cc = c, t = g; t < g + T; ++cc) {
          const int64_t t1 = std::min(g + T, run_lo(cc + 1));
          const int64_t keys = std::min<int64_t>((t1 - g) * TK, u.kv_end) - (t - g) * TK;
          cost[(size_t)cc] += fixed_bytes + keys * key_bytes +
                              (split ? (int64_t)u.nrows * partial_bytes_per_row : 0);
          t = t1;
        }
      }
    }
    const int64_t finish = *std::max_element(cost.begin(), cost.end());
    if ((double)finish < best_lpt * 0.97) {
      stream = true;
      n_ctas = n;
      std::vector<std::vector<Tmp>> runs;  // pieces of each run, in order (one plan's worth)
      runs.resize((size_t)n);
      g = 0;
      c = 0;
      for (const Unit& u : units) {
        const int64_t T = ceil_div(u.kv_end, TK);
        for (int h = 0; h < num_kv_heads; ++h, g += T) {
          while (run_lo(c + 1) <= g) ++c;
          int64_t pieces = 0;
          for (int64_t cc = c, t = g; t < g + T; ++cc, ++pieces) t = std::min(g + T, run_lo(cc + 1));
          int64_t base = -1;
          if (pieces > 1) {
            base = part_rows;
            merges.push_back({u.b, h, u.row0, u.nrows, (int32_t)base, (int32_t)pieces, 0, 0});
            part_rows += pieces * u.nrows;
          }
          int64_t s = 0;
          for (int64_t cc = c, t = g; t < g + T; ++cc, ++s) {
            const int64_t t1 = std::min(g + T, run_lo(cc + 1));
            const int32_t lo = (int32_t)((t - g) * TK);
            const int32_t hi = (int32_t)std::min<int64_t>((t1 - g) * TK, u.kv_end);
            WorkItem w{u.b, h, u.row0, u.nrows, lo, hi,
                       base >= 0 ? (int32_t)(base + s * u.nrows) : -1, -1};
            runs[(size_t)cc].push_back({w, (int64_t)(hi - lo) * (u.nrows + 16)});
            t = t1;
          }
        }
      }
      // chain c's first piece at index c, the rest after all the firsts
      for (int64_t cc = 0; cc < n; ++cc) items.push_back(runs[(size_t)cc].front());
      for (int64_t cc = 0; cc < n; ++cc) {
        int32_t prev = (int32_t)cc;
        for (size_t k = 1; k < runs[(size_t)cc].size(); ++k) {
          items.push_back(runs[(size_t)cc][k]);
          items[(size_t)prev].it.next = (int32_t)(items.size() - 1);
          prev = (int32_t)(items.size() - 1);
        }
        items[(size_t)prev].it.next = -1;
      }
    }
  }

  if (!stream) {
  // Draft items: with few units next to the CTAs (the latency-bound verify
  // shapes, whose units are split many ways), a split unit's drafts -- keys
  // prefix .. kv_end, at most one key tile -- become an item of their own,
  // which the fused append + attention call can serve from the new rows
  // while the append runs.
  const int64_t all_heads = (int64_t)units.size() * num_kv_heads;
  const bool draft_items =
      kernel_is_tc(kernel) && (o.draft_items == 1 || (o.draft_items == 0 && 2 * all_heads <= slots));
  {
    int64_t n_all = 0;  // an upper bound of the items (a draft item adds one per unit)
    for (const Unit& u : units) {
      int64_t cu;
      n_all += (split_of(u, chunk, equal, &cu) + (draft_items ? 1 : 0)) * num_kv_heads;
    }
    items.reserve((size_t)n_all);
  }
  for (const Unit& u : units) {
    int64_t cu;
    int64_t n = split_of(u, chunk, equal, &cu);
    const int64_t pre = prefix[u.b];
    if (draft_items && n > 1 && pre > 0 && u.kv_end > pre && u.kv_end - pre <= TK) {
      // the prefix cut as before (a short last prefix chunk joins the one
      // before it), then the drafts alone
      cuts.assign(1, 0);
      for (int64_t s = 1; s * cu < pre; ++s) cuts.push_back(s * cu);
      if (cuts.size() > 1 && pre - cuts.back() < TK) cuts.pop_back();
      cuts.push_back(pre);
      cuts.push_back(u.kv_end);
      n = (int64_t)cuts.size() - 1;
      for (int h = 0; h < num_kv_heads; ++h) {
        const int64_t base = part_rows;
        merges.push_back({u.b, h, u.row0, u.nrows, (int32_t)base, (int32_t)n, 0, 0});
        part_rows += n * u.nrows;
        for (int64_t s = 0; s < n; ++s) {
          const int64_t lo = cuts[s], hi = cuts[s + 1];
          WorkItem w{u.b, h, u.row0, u.nrows, (int32_t)lo, (int32_t)hi,
                     (int32_t)(base + s * u.nrows), -1};
          items.push_back({w, (hi - lo) * (int64_t)(u.nrows + 16)});
        }
      }
      continue;
    }
    // Chunk boundaries: multiples of the chunk size from the front.  For
    // the tcgen05 kernels a last chunk shorter than one key tile joins the
    // one before it: the tail of a request (its drafts, appended in the same
    // step) then shares a CTA with full prefix tiles that stream in before
    // the append is done, instead of a CTA of its own that would start cold
    // after it (a 17-key chunk of drafts alone was the tree verify's
    // critical path).
    cuts.assign(1, 0);
    for (int64_t s = 1; s < n; ++s) cuts.push_back(s * cu);
    if (kernel_is_tc(kernel) && n > 1 && u.kv_end - cuts.back() < TK) cuts.pop_back();
    cuts.push_back(u.kv_end);
    n = (int64_t)cuts.size() - 1;
    for (int h = 0; h < num_kv_heads; ++h) {
      int64_t base = part_rows;
      if (n > 1) {
        merges.push_back({u.b, h, u.row0, u.nrows, (int32_t)base, (int32_t)n, 0, 0});
        part_rows += n * u.nrows;
      }
      for (int64_t s = 0; s < n; ++s) {
        int64_t lo = cuts[s], hi = cuts[s + 1];
        WorkItem w{u.b, h, u.row0, u.nrows, (int32_t)lo, (int32_t)hi,
                   n > 1 ? (int32_t)(base + s * u.nrows) : -1, -1};
        items.push_back({w, (hi - lo) * (int64_t)(u.nrows + 16)});
      }
    }
  }
  }  // !stream
  if (part_rows > INT32_MAX) return VA_ERR_UNSUPPORTED;
  // Longest first; among equals, row blocks that read the same (request, KV
  // head, kv chunk) sit next to each other so they run together and the
  // later ones find the chunk in L2.  (b, h, kv_lo, row0) identifies an item,
  // so the order is total.
  if (!stream) {
    // sorted as 24-byte keys (cost descending, then b, h, kv_lo, row0, all
    // non-negative here) and the items permuted once
    struct Key {
      uint64_t k0, k1, k2;
      uint32_t idx;
    };
    std::vector<Key> keys(items.size());
    for (size_t i = 0; i < items.size(); ++i) {
      const WorkItem& w = items[i].it;
      keys[i] = {~(uint64_t)items[i].cost, ((uint64_t)(uint32_t)w.b << 32) | (uint32_t)w.h,
                 ((uint64_t)(uint32_t)w.kv_lo << 32) | (uint32_t)w.row0, (uint32_t)i};
    }
    std::sort(keys.begin(), keys.end(), [](const Key& a, const Key& b) {
      if (a.k0 != b.k0) return a.k0 < b.k0;
      if (a.k1 != b.k1) return a.k1 < b.k1;
      return a.k2 < b.k2;
    });
    std::vector<Tmp> sorted(items.size());
    for (size_t i = 0; i < keys.size(); ++i) sorted[i] = items[keys[i].idx];
    items.swap(sorted);
  }

  // Persistent tcgen05 variants: one CTA per SM walks a chain of items.  The
  // longest-first list is dealt onto the CTAs by LPT (each item to the
  // least-loaded CTA, with a per-item overhead of one key tile), chain c's
  // first item is put at index c and the rest follow, linked through next.
  if (!stream && kernel_is_tc(kernel) && !items.empty()) {
    n_ctas = std::min<int64_t>((int64_t)items.size(), num_sms);
    if ((int64_t)items.size() <= n_ctas) {
      // one item per CTA: item c is chain c
      for (auto& t : items) t.it.next = -1;
    } else {
      // LPT: each item (longest first) to the least-loaded chain, the
      // lowest chain index among equal loads; then the items are laid out
      // chain by chain (a counting sort on the owner), chain c's first at
      // index c.  The chain loads are kept as levels (load -> its chains,
      // ascending), and a run of items of equal increment is dealt a level
      // at a time: the lowest level's chains take the next items in index
      // order and move up together -- the same owners as dealing the items
      // one by one from a min-heap of (load, chain).
      // key tiles plus one of overhead; a tile of two Q tiles costs 5/3 of one
      auto inc = [&](const WorkItem& w) -> int64_t {
        return (ceil_div(w.kv_hi - w.kv_lo, TK) + 1) * (w.nrows > kTcRowsPerTile ? 5 : 3);
      };
      std::map<int64_t, std::vector<int32_t>> levels;
      {
        std::vector<int32_t>& all = levels[0];
        all.resize((size_t)n_ctas);
        for (int64_t c = 0; c < n_ctas; ++c) all[(size_t)c] = (int32_t)c;
      }
      std::vector<int32_t> owner(items.size()), moved, merged;
      for (size_t i = 0; i < items.size();) {
        const int64_t x = inc(items[i].it);
        size_t run = 1;
        while (i + run < items.size() && inc(items[i + run].it) == x) ++run;
        while (run > 0) {
          auto lo = levels.begin();
          const int64_t level = lo->first;
          std::vector<int32_t>& ids = lo->second;
          const size_t take = std::min(run, ids.size());
          for (size_t t = 0; t < take; ++t) owner[i++] = ids[t];
          moved.assign(ids.begin(), ids.begin() + (std::ptrdiff_t)take);
          if (take == ids.size()) levels.erase(lo);
          else ids.erase(ids.begin(), ids.begin() + (std::ptrdiff_t)take);
          std::vector<int32_t>& up = levels[level + x];
          if (up.empty()) {
            up.swap(moved);
          } else {
            merged.resize(up.size() + moved.size());
            std::merge(up.begin(), up.end(), moved.begin(), moved.end(), merged.begin());
            up.swap(merged);
          }
          run -= take;
        }
      }
      // chain c: its first item at index c, the rest after all the firsts, in
      // chain order, each linked to the next
      std::vector<int32_t> count((size_t)n_ctas, 0), first((size_t)n_ctas, -1);
      for (size_t i = 0; i < items.size(); ++i) ++count[(size_t)owner[i]];
      std::vector<int64_t> start((size_t)n_ctas + 1, 0);  // of the chains' tails
      for (int64_t c = 0; c < n_ctas; ++c) start[(size_t)c + 1] = start[(size_t)c] + count[(size_t)c] - 1;
      std::vector<Tmp> out(items.size());
      std::vector<int64_t> fill(start.begin(), start.end() - 1);
      std::vector<int32_t> last((size_t)n_ctas, -1);
      for (size_t i = 0; i < items.size(); ++i) {
        const int32_t c = owner[i];
        int64_t pos;
        if (first[(size_t)c] < 0) {
          pos = c;
          first[(size_t)c] = c;
        } else {
          pos = n_ctas + fill[(size_t)c]++;
        }
        out[(size_t)pos] = items[i];
        out[(size_t)pos].it.next = -1;
        if (last[(size_t)c] >= 0) out[(size_t)last[(size_t)c]].it.next = (int32_t)pos;
        last[(size_t)c] = (int32_t)pos;
      }
      items.swap(out);
    }
  }

  size_t need = sizeof(PlanHeader) + items.size() * sizeof(WorkItem) +
                merges.size() * sizeof(MergeItem);
  if (plan_bytes < need) {
    *workspace_bytes = need;
    return VA_ERR_PLAN_BUFFER_TOO_SMALL;
  }
  PlanHeader hd;
  std::memset(&hd, 0, sizeof(hd));
  hd.magic = kPlanMagic;
  hd.version = kPlanVersion;
  hd.batch = batch;
  hd.h_q = num_qo_heads;
  hd.h_kv = num_kv_heads;
  hd.head_dim = head_dim;
  hd.head_dim_v = dv;
  hd.max_nsplit = 0;
  for (const MergeItem& m : merges) hd.max_nsplit = std::max<int64_t>(hd.max_nsplit, m.nsplit);
  hd.page_size = page_size;
  hd.q_dtype = q_dtype;
  hd.kv_dtype = kv_dtype;
  hd.has_mask = has_mask ? 1 : 0;
  hd.group = G;
  hd.kernel = kernel;
  hd.block_rows = BM;
  hd.tile_keys = TK;
  hd.n_items = (int32_t)items.size();
  hd.n_merge = (int32_t)merges.size();
  hd.n_units = (int32_t)units.size();
  hd.num_sms = num_sms;
  hd.total_qo = batch > 0 ? qo_indptr[batch] : 0;
  hd.part_rows = part_rows;
  hd.chunk = chunk;
  hd.off_status = 0;
  hd.off_items = kWsAlign;
  hd.off_merge = hd.off_items + items.size() * sizeof(WorkItem);
  hd.off_part_lse = align_up(hd.off_merge + merges.size() * sizeof(MergeItem), kWsAlign);
  hd.off_part_out = align_up(hd.off_part_lse + (size_t)part_rows * 4, kWsAlign);
  hd.ws_bytes = align_up(hd.off_part_out + (size_t)part_rows * dv * 4, kWsAlign);
  hd.plan_bytes = need;
  hd.n_ctas = n_ctas;
  hd.flags = (full_mask ? kPlanMaskFull : 0) | (o.kv_layout == VA_LAYOUT_NHD ? kPlanNhd : 0) |
             (o.rope ? kPlanRope : 0) | (o.q_fp8 ? kPlanF8Mma : 0);

  char* dst = static_cast<char*>(plan_h);
  std::memcpy(dst, &hd, sizeof(hd));
  WorkItem* wi = reinterpret_cast<WorkItem*>(dst + sizeof(hd));
  for (size_t i = 0; i < items.size(); ++i) wi[i] = items[i].it;
  if (!merges.empty())
    std::memcpy(wi + items.size(), merges.data(), merges.size() * sizeof(MergeItem));
  *workspace_bytes = hd.ws_bytes;
  return VA_OK;
}

}  // namespace va
