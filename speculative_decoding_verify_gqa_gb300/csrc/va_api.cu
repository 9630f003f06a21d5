// C ABI of libverify_attn.so: argument checks, plan upload and kernel
// launches.  See include/verify_attn.h for the contract of every entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/verify_attn.h"
#include "va_internal.h"
#include "va_kernels.h"

namespace va {
int check_common(int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int q_dtype,
                 int kv_dtype);
int plan_bounds(int batch, int64_t total_qo, int num_qo_heads, int num_kv_heads, int head_dim,
                int num_sms, size_t* plan_bytes, size_t* workspace_bytes);
int plan_host(const int32_t* kv_indptr, const int32_t* qo_indptr, const int32_t* last_page_len,
              const int32_t* mask_indptr, int batch, int num_qo_heads, int num_kv_heads,
              int head_dim, int page_size, int q_dtype, int kv_dtype, int has_mask, int num_sms,
              const va_plan_options_t* opts, void* plan_h, size_t plan_bytes,
              size_t* workspace_bytes);
}  // namespace va

using namespace va;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int log2_int(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

int query_sms(int* n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VA_ERR_CUDA;
  if (cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return VA_ERR_CUDA;
  return *n > 0 ? VA_OK : VA_ERR_CUDA;
}

const PlanHeader* plan_header(const void* plan_h) {
  if (!plan_h) return nullptr;
  const PlanHeader* hd = static_cast<const PlanHeader*>(plan_h);
  if (hd->magic != kPlanMagic || hd->version != kPlanVersion) return nullptr;
  if (hd->kernel < kKernelMma64 || hd->kernel > kKernelTc256 ||
      hd->block_rows != kernel_rows(hd->kernel))
    return nullptr;
  return hd;
}

// RoPE frequencies theta^(-2i/d) / scale for i < d/2, in double, each split
// into a float head and the float nearest to the rest.
void rope_frequencies(float theta, float scale, int head_dim, RopeFreq* f) {
  for (int i = 0; i < 64; ++i) {
    f->hi[i] = f->lo[i] = 0.f;
    if (2 * i >= head_dim) continue;
    const double v = pow((double)theta, -2.0 * i / head_dim) / (double)scale;
    f->hi[i] = (float)v;
    f->lo[i] = (float)(v - (double)f->hi[i]);
  }
}

// Shared checks of verify_attn_run / _partial: the plan matches the call.
int check_run(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
              const int32_t* kv_indices, const int32_t* last_page_len, const int32_t* qo_indptr,
              const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads, int num_kv_heads,
              int head_dim, int page_size, float* sm_scale, float k_scale, float v_scale,
              const void* out, const float* lse, int num_pages, const void* plan_h,
              const void* workspace_d, size_t workspace_bytes, const va_run_options_t* o,
              const PlanHeader** hd_out) {
  const PlanHeader* hd = plan_header(plan_h);
  if (!hd) return VA_ERR_INVALID_ARGUMENT;
  if (o) {
    for (int r : o->reserved)
      if (r) return VA_ERR_INVALID_ARGUMENT;
  }
  const bool rope = (hd->flags & kPlanRope) != 0;
  const int32_t* q_position = o ? o->q_position : nullptr;
  if (rope != (q_position != nullptr)) return VA_ERR_PLAN_MISMATCH;
  if (rope) {
    const float sc = o->rope_scale == 0.f ? 1.f : o->rope_scale;
    if (!(isfinite(o->rope_theta) && o->rope_theta > 0.f && isfinite(sc) && sc > 0.f))
      return VA_ERR_INVALID_ARGUMENT;
  }
  if (hd->h_q != num_qo_heads || hd->h_kv != num_kv_heads || hd->head_dim != head_dim ||
      hd->page_size != page_size || hd->has_mask != (mask != nullptr ? 1 : 0))
    return VA_ERR_PLAN_MISMATCH;
  if ((mask != nullptr) != (mask_indptr != nullptr)) return VA_ERR_INVALID_ARGUMENT;
  if (!workspace_d || workspace_bytes < hd->ws_bytes) return VA_ERR_WORKSPACE_TOO_SMALL;
  if (!(isfinite(k_scale) && k_scale > 0.f && isfinite(v_scale) && v_scale > 0.f))
    return VA_ERR_INVALID_ARGUMENT;
  if (!isfinite(*sm_scale)) return VA_ERR_INVALID_ARGUMENT;
  if (*sm_scale <= 0.f) *sm_scale = 1.0f / sqrtf((float)head_dim);
  *hd_out = hd;
  if (hd->n_items == 0) return VA_OK;
  if (!q || !k_cache || !v_cache || !kv_indptr || !kv_indices || !last_page_len || !qo_indptr ||
      !out || num_pages <= 0)
    return VA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace_d))
    return VA_ERR_INVALID_ARGUMENT;
  (void)lse;
  return VA_OK;
}

PartialParams make_partial(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, const int32_t* qo_indptr,
                           const uint8_t* mask, const int32_t* mask_indptr, float sm_scale,
                           float k_scale, float v_scale, void* out, float* lse, int num_pages,
                           const PlanHeader* hd, void* workspace_d, const va_run_options_t* o) {
  char* ws = static_cast<char*>(workspace_d);
  PartialParams p;
  memset(&p, 0, sizeof(p));
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.last_page_len = last_page_len;
  p.qo_indptr = qo_indptr;
  p.mask = mask;
  p.mask_indptr = mask_indptr;
  p.out = out;
  p.lse = lse;
  p.items = reinterpret_cast<const WorkItem*>(ws + hd->off_items);
  p.part_out = reinterpret_cast<float*>(ws + hd->off_part_out);
  p.part_lse = reinterpret_cast<float*>(ws + hd->off_part_lse);
  p.status = reinterpret_cast<int*>(ws + hd->off_status);
  p.batch = hd->batch;
  p.part_rows = hd->part_rows;
  p.h_q = hd->h_q;
  p.h_kv = hd->h_kv;
  p.group = hd->group;
  p.page_size = hd->page_size;
  p.log2_page = log2_int(hd->page_size);
  p.num_pages = num_pages;
  p.scale_nat = sm_scale * k_scale;
  p.scale_log2 = sm_scale * k_scale * 1.4426950408889634f;
  p.v_scale = v_scale;
  p.n_items = hd->n_items;
  p.n_ctas = (int)hd->n_ctas;
  p.mask_full = (hd->flags & kPlanMaskFull) ? 1 : 0;
  p.nhd = (hd->flags & kPlanNhd) ? 1 : 0;
  if ((hd->flags & kPlanRope) && o && o->q_position) {
    p.q_position = o->q_position;
    rope_frequencies(o->rope_theta, o->rope_scale == 0.f ? 1.f : o->rope_scale, hd->head_dim,
                     &p.rope);
  }
  return p;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// TMA descriptors of the tensor-core variant (see TcMaps).
int make_tc_maps(const void* q, int64_t total_qo, const void* k_cache, const void* v_cache,
                 int num_pages, const PlanHeader* hd, const void* k_new, const void* v_new,
                 TcMaps* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return VA_ERR_CUDA;
  const int G = hd->group, D = hd->head_dim, P = hd->page_size;
  if (total_qo <= 0 || num_pages <= 0) return VA_ERR_INVALID_ARGUMENT;
  // the bf16 views index page * h_kv + head, or page * P / 8 + slot / 8 (plus
  // one page past the pool), in int
  if ((int64_t)(num_pages + 1) * hd->h_kv > 0x7fffffffLL ||
      (int64_t)(num_pages + 1) * hd->page_size / 8 > 0x7fffffffLL)
    return VA_ERR_UNSUPPORTED;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hd->h_q, (cuuint64_t)total_qo};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hd->h_q * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    if (enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return VA_ERR_CUDA;
  }
  const bool fp8 = hd->kv_dtype == VA_DTYPE_FP8_E4M3;
  const bool nhd = (hd->flags & kPlanNhd) != 0;
  const cuuint64_t es = fp8 ? 1 : 2;
  const cuuint64_t H = (cuuint64_t)hd->h_kv;
  // element strides of a slot and of a head: HND [page][head][slot][d],
  // NHD [page][slot][head][d]
  const cuuint64_t slot_st = nhd ? H * D : (cuuint64_t)D;
  const cuuint64_t head_st = nhd ? (cuuint64_t)D : (cuuint64_t)P * D;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)P, H, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {slot_st * es, head_st * es, H * P * D * es};
  cuuint32_t box[4] = {fp8 ? 128u : 64u, 16, 1, 1};
  const void* src[2] = {k_cache, v_cache};
  CUtensorMap* dst[2] = {&m->k, &m->v};
  for (int i = 0; i < 2; ++i) {
    if (!fp8) {
      // HND: [page * h_kv + head][slot / 8][half][slot % 8][64]; NHD: [page * P / 8
      // + slot / 8][head][half][slot % 8][64]; one box per 16 keys of one head
      cuuint64_t vd[5], vs[4];
      cuuint32_t vb[5] = {64, 8, 2, 2, 1};
      vd[0] = 64; vd[1] = 8; vd[2] = 2;
      vs[0] = slot_st * 2; vs[1] = 128;
      if (nhd) {
        vd[3] = H; vd[4] = (cuuint64_t)num_pages * P / 8;
        vs[2] = (cuuint64_t)D * 2; vs[3] = 8 * slot_st * 2;
        vb[3] = 1; vb[4] = 2;
      } else {
        vd[3] = (cuuint64_t)P / 8; vd[4] = H * (cuuint64_t)num_pages;
        vs[2] = 8 * slot_st * 2; vs[3] = (cuuint64_t)P * D * 2;
      }
      cuuint32_t ve[5] = {1, 1, 1, 1, 1};
      if (enc(dst[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(src[i]), vd, vs, vb, ve,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return VA_ERR_CUDA;
      continue;
    }
    if (enc(dst[i], fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void*>(src[i]), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            fp8 && !(hd->flags & kPlanF8Mma) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return VA_ERR_CUDA;
  }
  // the new rows [total_qo, h_kv, D] (see TcMaps)
  const void* nsrc[2] = {k_new, v_new};
  CUtensorMap* ndst[2] = {&m->kn, &m->vn};
  for (int i = 0; i < 2; ++i) {
    if (!nsrc[i]) {
      memset(ndst[i], 0, sizeof(CUtensorMap));
      continue;
    }
    CUresult r;
    if (!fp8) {
      cuuint64_t nd[4] = {64, (cuuint64_t)total_qo, 2, H};
      cuuint64_t ns[3] = {H * D * 2, 128, (cuuint64_t)D * 2};
      cuuint32_t nb[4] = {64, 8, 2, 1};
      r = enc(ndst[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(nsrc[i]), nd, ns, nb,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      cuuint64_t nd[3] = {(cuuint64_t)D, (cuuint64_t)total_qo, H};
      cuuint64_t ns[2] = {H * D, (cuuint64_t)D};
      cuuint32_t nb[3] = {128, 16, 1};
      r = enc(ndst[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(nsrc[i]), nd, ns, nb, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              (hd->flags & kPlanF8Mma) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return VA_ERR_CUDA;
  }
  return VA_OK;
}

}  // namespace

static int verify_attn_merge_impl(const int32_t* qo_indptr, int num_qo_heads, int num_kv_heads,
                                  int head_dim, void* out, float* lse, const void* plan_h,
                                  void* workspace_d, size_t workspace_bytes, int early,
                                  void* stream) {
  const PlanHeader* hd = plan_header(plan_h);
  if (!hd) return VA_ERR_INVALID_ARGUMENT;
  if (hd->h_q != num_qo_heads || hd->h_kv != num_kv_heads || hd->head_dim != head_dim)
    return VA_ERR_PLAN_MISMATCH;
  if (hd->n_merge == 0) return VA_OK;
  if (!workspace_d || workspace_bytes < hd->ws_bytes) return VA_ERR_WORKSPACE_TOO_SMALL;
  if (!qo_indptr || !out || !aligned16(out) || !aligned16(workspace_d))
    return VA_ERR_INVALID_ARGUMENT;
  char* ws = static_cast<char*>(workspace_d);
  MergeParams m;
  m.items = reinterpret_cast<const MergeItem*>(ws + hd->off_merge);
  m.part_out = reinterpret_cast<const float*>(ws + hd->off_part_out);
  m.part_lse = reinterpret_cast<const float*>(ws + hd->off_part_lse);
  m.qo_indptr = qo_indptr;
  m.out = out;
  m.lse = lse;
  m.batch = hd->batch;
  m.part_rows = hd->part_rows;
  m.h_q = hd->h_q;
  m.h_kv = hd->h_kv;
  m.group = hd->group;
  m.early_inputs = early;
  cudaError_t e = launch_merge(m, (int)hd->head_dim_v, hd->n_merge, hd->block_rows,
                               (int)hd->max_nsplit,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VA_OK : VA_ERR_CUDA;
}

static int run_partial(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, const int32_t* qo_indptr,
                           const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                           int num_kv_heads, int head_dim, int page_size, float sm_scale,
                           float k_scale, float v_scale, void* out, float* lse, int num_pages,
                           const void* plan_h, void* workspace_d, size_t workspace_bytes,
                           const va_run_options_t* options, int early, void* stream,
                           const void* k_new = nullptr, const void* v_new = nullptr) {
  const PlanHeader* hd = nullptr;
  int rc = check_run(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
                     mask_indptr, num_qo_heads, num_kv_heads, head_dim, page_size, &sm_scale,
                     k_scale, v_scale, out, lse, num_pages, plan_h, workspace_d, workspace_bytes,
                     options, &hd);
  if (rc) return rc;
  if (hd->n_items == 0) return VA_OK;
  PartialParams p = make_partial(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len,
                                 qo_indptr, mask, mask_indptr, sm_scale, k_scale, v_scale, out,
                                 lse, num_pages, hd, workspace_d, options);
  p.early_inputs = early;
  p.total_qo = (int)hd->total_qo;
  cudaError_t e;
  if (kernel_is_tc(hd->kernel)) {
    // draft items read the new rows only when they are given (a plain copy
    // append in the same call) and every split holds them apart
    const bool from_new = k_new && v_new;
    p.drafts_new = from_new ? 1 : 0;
    TcMaps maps;
    rc = make_tc_maps(q, hd->total_qo, k_cache, v_cache, num_pages, hd,
                      from_new ? k_new : nullptr, from_new ? v_new : nullptr, &maps);
    if (rc) return rc;
    e = launch_partial_tc(p, maps, hd->kv_dtype == VA_DTYPE_FP8_E4M3, hd->block_rows, hd->n_items,
                          (hd->flags & kPlanF8Mma) != 0,
                          static_cast<cudaStream_t>(stream));
  } else {
    e = launch_partial_mma(p, hd->kernel, hd->head_dim, (int)hd->head_dim_v,
                           hd->kv_dtype == VA_DTYPE_FP8_E4M3,
                           hd->n_items, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? VA_OK : VA_ERR_CUDA;
}

extern "C" {

const char* verify_attn_status_string(int status) {
  switch (status) {
    case VA_OK: return "ok";
    case VA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case VA_ERR_UNSUPPORTED: return "unsupported configuration";
    case VA_ERR_WORKSPACE_TOO_SMALL: return "device workspace too small";
    case VA_ERR_PLAN_MISMATCH: return "plan does not match the call";
    case VA_ERR_CUDA: return "CUDA runtime error";
    case VA_ERR_DEVICE_CHECK: return "a device-side check failed";
    case VA_ERR_PLAN_BUFFER_TOO_SMALL: return "host plan buffer too small";
    case VA_ERR_STATIC_SCRATCH_TOO_SMALL:
      return "plan needs more scratch than the library's static scratch array holds";
    default: return "unknown status";
  }
}

int verify_attn_num_sms(int* num_sms) {
  if (!num_sms) return VA_ERR_INVALID_ARGUMENT;
  return query_sms(num_sms);
}

int verify_attn_plan_bounds(int batch, int64_t total_qo, int num_qo_heads, int num_kv_heads,
                            int head_dim, int num_sms, size_t* plan_bytes,
                            size_t* workspace_bytes) {
  if (num_sms <= 0) {
    int rc = query_sms(&num_sms);
    if (rc) return rc;
  }
  return plan_bounds(batch, total_qo, num_qo_heads, num_kv_heads, head_dim, num_sms, plan_bytes,
                     workspace_bytes);
}

int verify_attn_workspace_size(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                               int max_qo_len, int num_sms, size_t* bytes) {
  if (!bytes || batch < 0 || max_qo_len < 0) return VA_ERR_INVALID_ARGUMENT;
  size_t plan_bytes = 0;
  return verify_attn_plan_bounds(batch, (int64_t)batch * max_qo_len, num_qo_heads, num_kv_heads,
                                 head_dim, num_sms, &plan_bytes, bytes);
}

int verify_attn_plan_host(const int32_t* kv_indptr_h, const int32_t* qo_indptr_h,
                          const int32_t* last_page_len_h, const int32_t* mask_indptr_h,
                          int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                          int page_size, va_dtype q_dtype, va_dtype kv_dtype, int has_mask,
                          int num_sms, const va_plan_options_t* options, void* plan_h,
                          size_t plan_bytes, size_t* workspace_bytes) {
  if (num_sms <= 0) {
    int rc = query_sms(&num_sms);
    if (rc) return rc;
  }
  return plan_host(kv_indptr_h, qo_indptr_h, last_page_len_h, mask_indptr_h, batch,
                   num_qo_heads, num_kv_heads, head_dim, page_size, q_dtype, kv_dtype, has_mask,
                   num_sms, options, plan_h, plan_bytes, workspace_bytes);
}

int verify_attn_plan(const int32_t* kv_indptr_h, const int32_t* qo_indptr_h,
                     const int32_t* last_page_len_h, const int32_t* mask_indptr_h, int batch,
                     int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                     va_dtype q_dtype, va_dtype kv_dtype, int has_mask, int num_sms,
                     const va_plan_options_t* options, void* plan_h, size_t plan_bytes,
                     void* workspace_d, size_t workspace_bytes, void* stream) {
  size_t need = 0;
  int rc = verify_attn_plan_host(kv_indptr_h, qo_indptr_h, last_page_len_h, mask_indptr_h, batch,
                                 num_qo_heads, num_kv_heads, head_dim, page_size, q_dtype,
                                 kv_dtype, has_mask, num_sms, options, plan_h, plan_bytes, &need);
  if (rc) return rc;
  if (!workspace_d || workspace_bytes < need) return VA_ERR_WORKSPACE_TOO_SMALL;
  return verify_attn_plan_upload(plan_h, workspace_d, workspace_bytes, stream);
}

int verify_attn_plan_upload(const void* plan_h, void* workspace_d, size_t workspace_bytes,
                            void* stream) {
  const PlanHeader* hd = plan_header(plan_h);
  if (!hd) return VA_ERR_INVALID_ARGUMENT;
  if (!workspace_d || workspace_bytes < hd->ws_bytes) return VA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace_d)) return VA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace_d);
  if (cudaMemsetAsync(ws + hd->off_status, 0, sizeof(int), s) != cudaSuccess) return VA_ERR_CUDA;
  size_t list = (size_t)hd->n_items * sizeof(WorkItem) + (size_t)hd->n_merge * sizeof(MergeItem);
  if (list > 0 &&
      cudaMemcpyAsync(ws + hd->off_items, static_cast<const char*>(plan_h) + sizeof(PlanHeader),
                      list, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return VA_ERR_CUDA;
  return VA_OK;
}

int verify_attn_plan_launches(const void* plan_h, int* launches) {
  const PlanHeader* hd = plan_header(plan_h);
  if (!hd || !launches) return VA_ERR_INVALID_ARGUMENT;
  *launches = (hd->n_items > 0 ? 1 : 0) + (hd->n_merge > 0 ? 1 : 0);
  return VA_OK;
}

int verify_attn_partial_ex(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, const int32_t* qo_indptr,
                           const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                           int num_kv_heads, int head_dim, int page_size, float sm_scale,
                           float k_scale, float v_scale, void* out, float* lse, int num_pages,
                           const void* plan_h, void* workspace_d, size_t workspace_bytes,
                           const va_run_options_t* options, void* stream) {
  return run_partial(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
                     mask_indptr, num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale,
                     k_scale, v_scale, out, lse, num_pages, plan_h, workspace_d, workspace_bytes,
                     options, options && options->early_reads ? 1 : 0, stream);
}

int verify_attn_partial(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* kv_indptr, const int32_t* kv_indices,
                        const int32_t* last_page_len, const int32_t* qo_indptr,
                        const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                        int num_kv_heads, int head_dim, int page_size, float sm_scale,
                        float k_scale, float v_scale, void* out, float* lse, int num_pages,
                        const void* plan_h, void* workspace_d, size_t workspace_bytes,
                        void* stream) {
  return verify_attn_partial_ex(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len,
                                qo_indptr, mask, mask_indptr, num_qo_heads, num_kv_heads,
                                head_dim, page_size, sm_scale, k_scale, v_scale, out, lse,
                                num_pages, plan_h, workspace_d, workspace_bytes, nullptr, stream);
}

int verify_attn_merge(const int32_t* qo_indptr, int num_qo_heads, int num_kv_heads, int head_dim,
                      void* out, float* lse, const void* plan_h, void* workspace_d,
                      size_t workspace_bytes, void* stream) {
  return verify_attn_merge_impl(qo_indptr, num_qo_heads, num_kv_heads, head_dim, out, lse, plan_h,
                                workspace_d, workspace_bytes, 0, stream);
}

int verify_attn_run_ex(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, const int32_t* qo_indptr,
                       const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                       int num_kv_heads, int head_dim, int page_size, float sm_scale,
                       float k_scale, float v_scale, void* out, float* lse, int num_pages,
                       const void* plan_h, void* workspace_d, size_t workspace_bytes,
                       const va_run_options_t* options, void* stream) {
  int rc = verify_attn_partial_ex(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len,
                                  qo_indptr, mask, mask_indptr, num_qo_heads, num_kv_heads,
                                  head_dim, page_size, sm_scale, k_scale, v_scale, out, lse,
                                  num_pages, plan_h, workspace_d, workspace_bytes, options,
                                  stream);
  if (rc) return rc;
  return verify_attn_merge_impl(qo_indptr, num_qo_heads, num_kv_heads, head_dim, out, lse, plan_h,
                                workspace_d, workspace_bytes,
                                options && options->early_reads ? 1 : 0, stream);
}

int verify_attn_run(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* kv_indptr, const int32_t* kv_indices,
                    const int32_t* last_page_len, const int32_t* qo_indptr, const uint8_t* mask,
                    const int32_t* mask_indptr, int num_qo_heads, int num_kv_heads, int head_dim,
                    int page_size, float sm_scale, float k_scale, float v_scale, void* out,
                    float* lse, int num_pages, const void* plan_h, void* workspace_d,
                    size_t workspace_bytes, void* stream) {
  return verify_attn_run_ex(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr,
                            mask, mask_indptr, num_qo_heads, num_kv_heads, head_dim, page_size,
                            sm_scale, k_scale, v_scale, out, lse, num_pages, plan_h, workspace_d,
                            workspace_bytes, nullptr, stream);
}

}  // extern "C"

// ---- scratch for callers that cannot allocate ---------------------------------
// One file-scope device array serves every verify_attn_run_static_scratch call
// (work list, split partials, status word).  In host code its name is only a
// host-side stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress, looked up once per CUDA context.
static __device__ __align__(256) unsigned char g_static_scratch[VA_STATIC_SCRATCH_BYTES];

namespace {

// Address of g_static_scratch in the current context.  The symbol's address
// is a property of the context that loaded this library's module (the
// device's primary context, or another driver context made current by the
// caller), and a context destroyed by cudaDeviceReset takes it along, so the
// look-up is cached per context under the driver's unique context id -- not
// per device ordinal -- and made afresh for a context not seen before.  Before
// any context exists the runtime call creates the primary context, and the
// result is not cached that time.
using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name, int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(f);
}

constexpr int kScratchCache = 16;
std::mutex g_scratch_mu;
unsigned long long g_scratch_ctx[kScratchCache] = {};
void* g_scratch_ptr[kScratchCache] = {};
int g_scratch_next = 0;

int static_scratch_address(void** ptr) {
  static const PfnCtxGetCurrent ctx_current = driver_fn<PfnCtxGetCurrent>("cuCtxGetCurrent", 4000);
  static const PfnCtxGetId ctx_id = driver_fn<PfnCtxGetId>("cuCtxGetId", 12000);
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  const bool keyed = ctx_current && ctx_id && ctx_current(&ctx) == CUDA_SUCCESS && ctx &&
                     ctx_id(ctx, &id) == CUDA_SUCCESS;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (keyed)
    for (int i = 0; i < kScratchCache; ++i)
      if (g_scratch_ptr[i] && g_scratch_ctx[i] == id) {
        *ptr = g_scratch_ptr[i];
        return VA_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return VA_ERR_CUDA;
  if (keyed) {
    g_scratch_ctx[g_scratch_next] = id;
    g_scratch_ptr[g_scratch_next] = p;
    g_scratch_next = (g_scratch_next + 1) % kScratchCache;
  }
  *ptr = p;
  return VA_OK;
}

}  // namespace

extern "C" {

int verify_attn_run_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* last_page_len, const int32_t* qo_indptr,
                                   const uint8_t* mask, const int32_t* mask_indptr,
                                   int num_qo_heads, int num_kv_heads, int head_dim,
                                   int page_size, float sm_scale, float k_scale, float v_scale,
                                   void* out, float* lse, int num_pages, const void* plan_h,
                                   void* stream) {
  const PlanHeader* hd = plan_header(plan_h);
  if (!hd) return VA_ERR_INVALID_ARGUMENT;
  if (hd->ws_bytes > VA_STATIC_SCRATCH_BYTES) return VA_ERR_STATIC_SCRATCH_TOO_SMALL;
  void* scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(scratch);
  // the status word starts at zero; the work list comes from this plan
  if (cudaMemsetAsync(ws + hd->off_status, 0, sizeof(int), s) != cudaSuccess) return VA_ERR_CUDA;
  const size_t list =
      (size_t)hd->n_items * sizeof(WorkItem) + (size_t)hd->n_merge * sizeof(MergeItem);
  if (list > 0 &&
      cudaMemcpyAsync(ws + hd->off_items, static_cast<const char*>(plan_h) + sizeof(PlanHeader),
                      list, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return VA_ERR_CUDA;
  return verify_attn_run(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr,
                         mask, mask_indptr, num_qo_heads, num_kv_heads, head_dim, page_size,
                         sm_scale, k_scale, v_scale, out, lse, num_pages, plan_h, scratch,
                         VA_STATIC_SCRATCH_BYTES, stream);
}

int verify_attn_device_status(void* workspace_d, int* bits, void* stream) {
  if (!workspace_d || !bits) return VA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace_d, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return VA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return VA_ERR_CUDA;
  if (cudaMemsetAsync(workspace_d, 0, sizeof(int), s) != cudaSuccess) return VA_ERR_CUDA;
  *bits = v;
  return v ? VA_ERR_DEVICE_CHECK : VA_OK;
}

int verify_attn_static_scratch_status(int* bits, void* stream) {
  if (!bits) return VA_ERR_INVALID_ARGUMENT;
  void* scratch = nullptr;
  const int rc = static_scratch_address(&scratch);
  if (rc) return rc;
  // the status word is the scratch's first word (every plan's off_status)
  return verify_attn_device_status(scratch, bits, stream);
}

static int append_impl(const void* k_new, const void* v_new, const int32_t* append_indptr,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, void* k_cache, void* v_cache, int batch,
                       int num_kv_heads, int head_dim, int page_size, int num_pages,
                       va_dtype kv_dtype, int64_t total_new, const va_append_options_t* options,
                       int* status_d, int early, void* stream) {
  va_append_options_t o;
  memset(&o, 0, sizeof(o));
  if (options) o = *options;
  for (int r : o.reserved)
    if (r) return VA_ERR_INVALID_ARGUMENT;
  if (batch < 0 || total_new < 0 || num_kv_heads <= 0) return VA_ERR_INVALID_ARGUMENT;
  int rc = check_common(num_kv_heads, num_kv_heads, head_dim, page_size, VA_DTYPE_BF16, kv_dtype);
  if (rc) return rc;
  if (o.kv_layout != VA_LAYOUT_HND && o.kv_layout != VA_LAYOUT_NHD) return VA_ERR_INVALID_ARGUMENT;
  if (o.quantize != 0 && o.quantize != 1) return VA_ERR_INVALID_ARGUMENT;
  if (o.head_dim_v < 0) return VA_ERR_INVALID_ARGUMENT;
  const int head_dim_v = o.head_dim_v ? o.head_dim_v : head_dim;
  if (head_dim_v != 64 && head_dim_v != 128) return VA_ERR_UNSUPPORTED;
  if (o.quantize && (kv_dtype != VA_DTYPE_FP8_E4M3 || !(isfinite(o.k_scale) && o.k_scale > 0.f) ||
                     !(isfinite(o.v_scale) && o.v_scale > 0.f)))
    return VA_ERR_INVALID_ARGUMENT;
  float rope_scale = o.rope_scale == 0.f ? 1.f : o.rope_scale;
  if (o.positions && !(isfinite(o.rope_theta) && o.rope_theta > 0.f && isfinite(rope_scale) &&
                       rope_scale > 0.f))
    return VA_ERR_INVALID_ARGUMENT;
  if (total_new == 0) return VA_OK;
  if (batch == 0) return VA_ERR_INVALID_ARGUMENT;
  if (!k_new || !v_new || !append_indptr || !kv_indptr || !kv_indices || !last_page_len ||
      !k_cache || !v_cache || num_pages <= 0)
    return VA_ERR_INVALID_ARGUMENT;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return VA_ERR_INVALID_ARGUMENT;
  if (total_new > 0x7fffffffLL) return VA_ERR_UNSUPPORTED;
  AppendParams p;
  memset(&p, 0, sizeof(p));
  p.k_new = k_new;
  p.v_new = v_new;
  p.append_indptr = append_indptr;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.last_page_len = last_page_len;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.status = status_d;
  p.positions = o.positions;
  p.batch = batch;
  p.h_kv = num_kv_heads;
  p.page_size = page_size;
  p.log2_page = log2_int(page_size);
  p.num_pages = num_pages;
  p.cache_fp8 = kv_dtype == VA_DTYPE_FP8_E4M3;
  p.k_chunks = head_dim * (p.cache_fp8 ? 1 : 2) / 16;
  p.v_chunks = head_dim_v * (p.cache_fp8 ? 1 : 2) / 16;
  p.row_chunks = std::max(p.k_chunks, p.v_chunks);
  p.head_dim = head_dim;
  p.head_dim_v = head_dim_v;
  p.quant = o.quantize;
  p.nhd = o.kv_layout == VA_LAYOUT_NHD;
  p.k_scale = o.k_scale;
  p.v_scale = o.v_scale;
  p.total_new = total_new;
  p.early = early;
  if (o.positions) rope_frequencies(o.rope_theta, rope_scale, head_dim, &p.rope);
  cudaError_t e = launch_append(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VA_OK : VA_ERR_CUDA;
}

int paged_kv_append_ex(const void* k_new, const void* v_new, const int32_t* append_indptr,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, void* k_cache, void* v_cache, int batch,
                       int num_kv_heads, int head_dim, int page_size, int num_pages,
                       va_dtype kv_dtype, int64_t total_new, const va_append_options_t* options,
                       int* status_d, void* stream) {
  return append_impl(k_new, v_new, append_indptr, kv_indptr, kv_indices, last_page_len, k_cache,
                     v_cache, batch, num_kv_heads, head_dim, page_size, num_pages, kv_dtype,
                     total_new, options, status_d, 0, stream);
}

int verify_attn_append_run(const void* k_new, const void* v_new,
                           const va_append_options_t* append_options, const void* q, void* k_cache,
                           void* v_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, const int32_t* qo_indptr,
                           const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                           int num_kv_heads, int head_dim, int page_size, float sm_scale,
                           float k_scale, float v_scale, void* out, float* lse, int num_pages,
                           const void* plan_h, void* workspace_d, size_t workspace_bytes,
                           const va_run_options_t* run_options, void* stream) {
  // every check of the run before anything is enqueued
  const PlanHeader* hd = nullptr;
  float sc = sm_scale;
  int rc = check_run(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
                     mask_indptr, num_qo_heads, num_kv_heads, head_dim, page_size, &sc, k_scale,
                     v_scale, out, lse, num_pages, plan_h, workspace_d, workspace_bytes,
                     run_options, &hd);
  if (rc) return rc;
  const int early = run_options && run_options->early_reads ? 1 : 0;
  const int layout = append_options ? (int)append_options->kv_layout : VA_LAYOUT_HND;
  if (layout != ((hd->flags & kPlanNhd) ? VA_LAYOUT_NHD : VA_LAYOUT_HND)) return VA_ERR_PLAN_MISMATCH;
  // the append's value rows are the plan's
  va_append_options_t ao;
  memset(&ao, 0, sizeof(ao));
  if (append_options) ao = *append_options;
  if (ao.head_dim_v != 0 && ao.head_dim_v != hd->head_dim_v) return VA_ERR_PLAN_MISMATCH;
  ao.head_dim_v = (int)hd->head_dim_v;
  if (hd->total_qo > 0) {
    int* status = reinterpret_cast<int*>(static_cast<char*>(workspace_d) + hd->off_status);
    rc = append_impl(k_new, v_new, qo_indptr, kv_indptr, kv_indices, last_page_len, k_cache,
                     v_cache, hd->batch, num_kv_heads, head_dim, page_size, num_pages,
                     (va_dtype)hd->kv_dtype, hd->total_qo, &ao, status, early, stream);
    if (rc) return rc;
  }
  // A plain copy (no quantisation, no rotation) stores exactly the bytes of
  // k_new / v_new: the attention may read the drafts from there.
  const bool plain = !append_options || (!append_options->quantize && !append_options->positions);
  rc = run_partial(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
                   mask_indptr, num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale, k_scale,
                   v_scale, out, lse, num_pages, plan_h, workspace_d, workspace_bytes, run_options,
                   1, stream, plain ? k_new : nullptr, plain ? v_new : nullptr);
  if (rc) return rc;
  return verify_attn_merge_impl(qo_indptr, num_qo_heads, num_kv_heads, head_dim, out, lse, plan_h,
                                workspace_d, workspace_bytes, 1, stream);
}

// [off, off + bytes) lies inside a buffer of `size` bytes
static bool in_buffer(int64_t off, int64_t bytes, size_t size) {
  return off >= 0 && bytes >= 0 && (uint64_t)off <= size && (uint64_t)bytes <= size - (uint64_t)off;
}

int verify_attn_step_host(const void* staging_h, void* staging_d, size_t staging_bytes,
                          const va_step_offsets_t* offsets, int batch, int num_qo_heads,
                          int num_kv_heads, int head_dim, int page_size, va_dtype kv_dtype,
                          int num_sms, const va_plan_options_t* plan_options, void* plan_h,
                          size_t plan_bytes, void* workspace_d, size_t workspace_bytes,
                          const va_append_options_t* append_options, void* k_cache, void* v_cache,
                          int num_pages, float sm_scale, float k_scale, float v_scale, void* out_d,
                          float* lse_d, void* result_h, size_t result_bytes,
                          const va_run_options_t* run_options, int synchronize, void* stream) {
  if (!staging_h || !staging_d || !offsets || !result_h || !out_d || batch < 0 ||
      num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return VA_ERR_INVALID_ARGUMENT;
  const va_step_offsets_t& o = *offsets;
  const char* h = static_cast<const char*>(staging_h);
  char* d = static_cast<char*>(staging_d);
  const int64_t nb = (int64_t)batch;
  const bool has_mask = o.mask >= 0 || o.mask_indptr >= 0;
  // the tables the host reads, then the arrays they size
  if (!in_buffer(o.qo_indptr, 4 * (nb + 1), staging_bytes) ||
      !in_buffer(o.kv_indptr, 4 * (nb + 1), staging_bytes) ||
      !in_buffer(o.last_page_len, 4 * nb, staging_bytes) ||
      (has_mask && !in_buffer(o.mask_indptr, 4 * (nb + 1), staging_bytes)))
    return VA_ERR_INVALID_ARGUMENT;
  if ((o.qo_indptr | o.kv_indptr | o.last_page_len | (has_mask ? o.mask_indptr : 0)) & 3)
    return VA_ERR_INVALID_ARGUMENT;
  const int32_t* qo_h = reinterpret_cast<const int32_t*>(h + o.qo_indptr);
  const int32_t* kv_h = reinterpret_cast<const int32_t*>(h + o.kv_indptr);
  const int32_t* lpl_h = reinterpret_cast<const int32_t*>(h + o.last_page_len);
  const int32_t* mi_h = has_mask ? reinterpret_cast<const int32_t*>(h + o.mask_indptr) : nullptr;
  const int64_t total_qo = qo_h[batch], n_idx = kv_h[batch];
  if (total_qo < 0 || n_idx < 0 || (has_mask && mi_h[batch] < 0)) return VA_ERR_INVALID_ARGUMENT;
  const int dv = plan_options && plan_options->head_dim_v ? plan_options->head_dim_v : head_dim;
  const bool quantize = append_options && append_options->quantize;
  const int64_t es_kv = kv_dtype == VA_FP8_E4M3 ? 1 : 2, es_new = quantize ? 2 : es_kv;
  const int64_t rows_q = total_qo * num_qo_heads, rows_kv = total_qo * num_kv_heads;
  if (!in_buffer(o.q, rows_q * head_dim * 2, staging_bytes) ||
      !in_buffer(o.k_new, rows_kv * head_dim * es_new, staging_bytes) ||
      !in_buffer(o.v_new, rows_kv * dv * es_new, staging_bytes) ||
      !in_buffer(o.kv_indices, 4 * n_idx, staging_bytes) ||
      (has_mask && !in_buffer(o.mask, ((int64_t)mi_h[batch] + 7) / 8, staging_bytes)))
    return VA_ERR_INVALID_ARGUMENT;
  const int64_t out_bytes = rows_q * dv * 2, lse_off = (out_bytes + 255) / 256 * 256;
  const int64_t res_need = lse_d ? lse_off + rows_q * 4 : out_bytes;
  if ((uint64_t)res_need > result_bytes) return VA_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the host plan (no CUDA call) before anything is enqueued
  size_t ws_need = 0;
  int rc = verify_attn_plan_host(kv_h, qo_h, lpl_h, mi_h, batch, num_qo_heads, num_kv_heads,
                                 head_dim, page_size, VA_BF16, kv_dtype, has_mask ? 1 : 0, num_sms,
                                 plan_options, plan_h, plan_bytes, &ws_need);
  if (rc) return rc;
  if (!workspace_d || workspace_bytes < ws_need) return VA_ERR_WORKSPACE_TOO_SMALL;
  if (staging_bytes > 0 &&
      cudaMemcpyAsync(staging_d, staging_h, staging_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return VA_ERR_CUDA;
  rc = verify_attn_plan_upload(plan_h, workspace_d, workspace_bytes, stream);
  if (rc) return rc;
  auto dev = [&](int64_t off) -> char* { return off >= 0 ? d + off : nullptr; };
  rc = verify_attn_append_run(dev(o.k_new), dev(o.v_new), append_options, dev(o.q), k_cache, v_cache,
                              reinterpret_cast<const int32_t*>(dev(o.kv_indptr)),
                              reinterpret_cast<const int32_t*>(dev(o.kv_indices)),
                              reinterpret_cast<const int32_t*>(dev(o.last_page_len)),
                              reinterpret_cast<const int32_t*>(dev(o.qo_indptr)),
                              has_mask ? reinterpret_cast<const uint8_t*>(dev(o.mask)) : nullptr,
                              has_mask ? reinterpret_cast<const int32_t*>(dev(o.mask_indptr)) : nullptr,
                              num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale, k_scale,
                              v_scale, out_d, lse_d, num_pages, plan_h, workspace_d,
                              workspace_bytes, run_options, stream);
  if (rc) return rc;
  char* res = static_cast<char*>(result_h);
  if (lse_d && reinterpret_cast<char*>(lse_d) == static_cast<char*>(out_d) + lse_off) {
    if (res_need > 0 &&
        cudaMemcpyAsync(res, out_d, res_need, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return VA_ERR_CUDA;
  } else {
    if (out_bytes > 0 &&
        cudaMemcpyAsync(res, out_d, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return VA_ERR_CUDA;
    if (lse_d && rows_q > 0 &&
        cudaMemcpyAsync(res + lse_off, lse_d, rows_q * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return VA_ERR_CUDA;
  }
  if (synchronize && cudaStreamSynchronize(st) != cudaSuccess) return VA_ERR_CUDA;
  return VA_OK;
}

// Chunks per logits row for the argmax kernel: about two CTAs per SM over
// all rows, each chunk at least 4096 elements.
static void accept_chunks(int64_t total_qo, int vocab, int num_sms, int* chunks, int64_t* elems) {
  int64_t c = total_qo > 0 ? (2LL * num_sms + total_qo - 1) / total_qo : 1;
  c = std::max<int64_t>(1, std::min<int64_t>(c, (vocab + 4095) / 4096));
  c = std::min<int64_t>(c, 64);
  int64_t e = (vocab + c - 1) / c;
  e = (e + 7) / 8 * 8;
  *chunks = (int)((vocab + e - 1) / e);
  *elems = e;
}

int verify_accept_workspace_size(int64_t total_qo, int vocab, int num_sms, size_t* bytes) {
  if (!bytes || total_qo < 0 || vocab <= 0) return VA_ERR_INVALID_ARGUMENT;
  if (num_sms <= 0) {
    int rc = query_sms(&num_sms);
    if (rc) return rc;
  }
  int chunks;
  int64_t elems;
  accept_chunks(total_qo, vocab, num_sms, &chunks, &elems);
  size_t ws = align_up((size_t)total_qo * chunks * 8, kWsAlign);
  ws += 2 * align_up((size_t)total_qo * 4, kWsAlign);
  *bytes = std::max<size_t>(ws, kWsAlign);
  return VA_OK;
}

int verify_accept_greedy(const void* logits, va_dtype logits_dtype, int64_t total_qo, int vocab,
                         int64_t row_stride, const int32_t* qo_indptr, int batch,
                         const int32_t* draft_tokens, const int32_t* parents,
                         int32_t* accept_len, int32_t* accepted_nodes, int32_t* bonus_token,
                         int32_t* argmax_out, int* status_d, int num_sms, void* workspace_d,
                         size_t workspace_bytes, void* stream) {
  if (batch < 0 || total_qo < 0 || vocab <= 0 || row_stride < vocab) return VA_ERR_INVALID_ARGUMENT;
  if (logits_dtype != VA_BF16 && logits_dtype != VA_F32) return VA_ERR_UNSUPPORTED;
  if (total_qo > 0x7fffffffLL || total_qo * row_stride > (int64_t)1 << 47) return VA_ERR_UNSUPPORTED;
  if (batch == 0) return VA_OK;
  if (!qo_indptr || !accept_len || !bonus_token || (total_qo > 0 && (!logits || !draft_tokens ||
                                                                      !parents || !accepted_nodes)))
    return VA_ERR_INVALID_ARGUMENT;
  if (num_sms <= 0) {
    int rc = query_sms(&num_sms);
    if (rc) return rc;
  }
  size_t need = 0;
  int rc = verify_accept_workspace_size(total_qo, vocab, num_sms, &need);
  if (rc) return rc;
  if (!workspace_d || workspace_bytes < need) return VA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace_d)) return VA_ERR_INVALID_ARGUMENT;
  AcceptParams p;
  memset(&p, 0, sizeof(p));
  accept_chunks(total_qo, vocab, num_sms, &p.chunks, &p.chunk_elems);
  char* ws = static_cast<char*>(workspace_d);
  p.keys = reinterpret_cast<uint64_t*>(ws);
  ws += align_up((size_t)total_qo * p.chunks * 8, kWsAlign);
  p.node_am = reinterpret_cast<int32_t*>(ws);
  ws += align_up((size_t)total_qo * 4, kWsAlign);
  p.node_state = reinterpret_cast<int32_t*>(ws);
  p.logits = logits;
  p.qo_indptr = qo_indptr;
  p.draft_tokens = draft_tokens;
  p.parents = parents;
  p.accept_len = accept_len;
  p.path = accepted_nodes;
  p.bonus = bonus_token;
  p.argmax_out = argmax_out;
  p.status = status_d;
  p.row_stride = row_stride;
  p.total = (int)total_qo;
  p.vocab = vocab;
  p.batch = batch;
  cudaError_t e = launch_accept(p, logits_dtype == VA_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VA_OK : VA_ERR_CUDA;
}

int paged_kv_append(const void* k_new, const void* v_new, const int32_t* append_indptr,
                    const int32_t* kv_indptr, const int32_t* kv_indices,
                    const int32_t* last_page_len, void* k_cache, void* v_cache, int batch,
                    int num_kv_heads, int head_dim, int page_size, int num_pages,
                    va_dtype kv_dtype, int64_t total_new, int* status_d, void* stream) {
  return append_impl(k_new, v_new, append_indptr, kv_indptr, kv_indices, last_page_len, k_cache,
                     v_cache, batch, num_kv_heads, head_dim, page_size, num_pages, kv_dtype,
                     total_new, nullptr, status_d, 0, stream);
}

}  // extern "C"
