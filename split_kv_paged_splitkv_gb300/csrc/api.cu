// C-ABI layer: argument validation, workspace layout, tensor maps, launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"

namespace splitkv {

namespace {
thread_local char g_err[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map over a GQA K or V page pool (rows of 128 elements) in either
// layout, with coordinates that do not depend on the layout -- (dims, key in
// page, [column half,] KV head, page) -- and the 128-byte swizzle:
//   e4m3: 4-D (128 dims, key, head, page), boxes [hpi heads][16 keys][128];
//   bf16: 5-D (64 dims, key, column half, head, page), boxes
//         [2 halves][16 keys][64] (one 16-key tile of one head; a 128-byte
//         swizzled row holds 64 bf16, so each key row is two 64-wide halves).
// Only the strides tell the layouts apart (HND: key rows of a head adjacent;
// NHD: the heads of a key adjacent); the shared-memory image of a box is the
// same in both.
splitkv_status make_gqa_map(TmaDesc* out, const void* base, bool fp8, int P, int Hkv,
                            int num_pages, int hpi, bool nhd) {
  auto fn = encode_fn();
  if (!fn) return fail(SPLITKV_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t row = fp8 ? 128u : 256u;  // bytes of one 128-element row
  const cuuint64_t key_stride = nhd ? row * Hkv : row;
  const cuuint64_t head_stride = nhd ? row : row * P;
  const cuuint64_t page_stride = row * P * Hkv;
  CUtensorMap m;
  CUresult r;
  if (fp8) {
    cuuint64_t gdim[4] = {128u, cuuint64_t(P), cuuint64_t(Hkv), cuuint64_t(num_pages)};
    cuuint64_t gstride[3] = {key_stride, head_stride, page_stride};
    cuuint32_t box[4] = {128u, 16u, cuuint32_t(hpi), 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), gdim, gstride, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t gdim[5] = {64u, cuuint64_t(P), 2u, cuuint64_t(Hkv), cuuint64_t(num_pages)};
    cuuint64_t gstride[4] = {key_stride, 128u, head_stride, page_stride};
    cuuint32_t box[5] = {64u, 16u, 2u, 1u, 1u};
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), gdim, gstride, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(SPLITKV_ECUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  static_assert(sizeof(CUtensorMap) == sizeof(TmaDesc), "tensor map size");
  std::memcpy(out, &m, sizeof(m));
  return SPLITKV_OK;
}

// 2-D bf16 map over [rows][dim] with boxes of 64 columns x box_rows rows.
splitkv_status make_bf16_map(TmaDesc* out, const void* base, int dim, int64_t rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(SPLITKV_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap m;
  cuuint64_t gdim[2] = {cuuint64_t(dim), cuuint64_t(rows)};
  cuuint64_t gstride[1] = {cuuint64_t(dim) * 2};
  cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPLITKV_ECUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  std::memcpy(out, &m, sizeof(m));
  return SPLITKV_OK;
}

// 2-D uint8 map over [rows][dim] e4m3 codes with unswizzled boxes of 64
// columns x box_rows rows (64-byte rows, the MLA kernel's FP8 staging).
splitkv_status make_u8_map(TmaDesc* out, const void* base, int dim, int64_t rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(SPLITKV_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap m;
  cuuint64_t gdim[2] = {cuuint64_t(dim), cuuint64_t(rows)};
  cuuint64_t gstride[1] = {cuuint64_t(dim)};
  cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPLITKV_ECUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  std::memcpy(out, &m, sizeof(m));
  return SPLITKV_OK;
}

splitkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SPLITKV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

splitkv_status validate_desc(const splitkv_desc_t* d) {
  if (!d) return fail(SPLITKV_EINVAL, "desc is NULL");
  if (d->batch < 1 || d->q_tokens < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1)
    return fail(SPLITKV_EINVAL, "batch, q_tokens and head counts must be >= 1");
  if (d->num_q_heads % d->num_kv_heads)
    return fail(SPLITKV_EINVAL, "num_q_heads (%d) must be a multiple of num_kv_heads (%d)",
                d->num_q_heads, d->num_kv_heads);
  if (d->qk_dim < 1 || d->v_dim < 1) return fail(SPLITKV_EINVAL, "dims must be >= 1");
  if (d->page_size < 16 || d->page_size % 16)
    return fail(SPLITKV_EINVAL, "page_size (%d) must be a positive multiple of 16", d->page_size);
  if (d->max_pages_per_seq < 1 || d->num_pages_total < 1)
    return fail(SPLITKV_EINVAL, "max_pages_per_seq and num_pages_total must be >= 1");
  if (d->kv_dtype != SPLITKV_BF16 && d->kv_dtype != SPLITKV_FP8_E4M3)
    return fail(SPLITKV_EINVAL, "unknown kv_dtype %d", d->kv_dtype);
  if (d->v_shares_k != 0 && d->v_shares_k != 1) return fail(SPLITKV_EINVAL, "v_shares_k must be 0 or 1");
  if (d->v_shares_k && d->v_dim > d->qk_dim)
    return fail(SPLITKV_EINVAL, "v_shares_k needs v_dim <= qk_dim");
  if (d->combine_mode != SPLITKV_COMBINE_FUSED && d->combine_mode != SPLITKV_COMBINE_SEPARATE)
    return fail(SPLITKV_EINVAL, "unknown combine_mode %d", d->combine_mode);
  if (d->kv_layout != SPLITKV_LAYOUT_HND && d->kv_layout != SPLITKV_LAYOUT_NHD)
    return fail(SPLITKV_EINVAL, "unknown kv_layout %d", d->kv_layout);
  if (int64_t(d->num_pages_total) * d->num_kv_heads * d->page_size >= (int64_t(1) << 31))
    return fail(SPLITKV_EINVAL, "num_pages_total * num_kv_heads * page_size must be < 2^31");
  if (family_of(*d) == Family::kNone)
    return fail(SPLITKV_EUNSUPPORTED,
                "no kernel for qk_dim=%d v_dim=%d T=%d G=%d kv_dtype=%d v_shares_k=%d "
                "(GQA: qk_dim=v_dim=128, T*G<=32; MLA: 128 q heads, 1 latent head, "
                "qk_dim=576, v_dim=512, page_size 16, 32 or a multiple of 64, T<=16, "
                "e4m3 only with V in the latent rows)",
                d->qk_dim, d->v_dim, d->q_tokens, d->num_q_heads / d->num_kv_heads, d->kv_dtype,
                d->v_shares_k);
  return SPLITKV_OK;
}

}  // namespace

splitkv_status fail(splitkv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

Family family_of(const splitkv_desc_t& d) {
  const int G = d.num_q_heads / d.num_kv_heads;
  if (d.qk_dim == 128 && d.v_dim == 128 && !d.v_shares_k && d.q_tokens * G <= 32) return Family::kGqa;
  // V either shares the latent rows (their first 512 columns) or is its own
  // tensor.  Keys stream in 64-key blocks: pages of 16 or 32 keys fill a block
  // with 4 or 2 boxes, larger pages (multiples of 64) hold whole blocks.
  // An e4m3 latent cache holds V in its rows (a separate e4m3 V tensor is
  // not served).
  if (d.qk_dim == 576 && d.v_dim == 512 && d.num_kv_heads == 1 && d.num_q_heads == 128 &&
      (d.kv_dtype == SPLITKV_BF16 || d.v_shares_k) && d.q_tokens <= 16 &&
      (64 % d.page_size == 0 || d.page_size % 64 == 0))
    return Family::kMla;
  return Family::kNone;
}

int ctas_per_item(const splitkv_desc_t& d) {
  return family_of(d) == Family::kMla ? 2 * d.q_tokens : 1;
}

int ctas_per_sm(const splitkv_desc_t& d) {
  return family_of(d) == Family::kGqa ? kGqaCtasPerSm : 1;
}

int heads_per_item(const splitkv_desc_t& d) {
  const int rows_per_head = d.q_tokens * (d.num_q_heads / d.num_kv_heads);
  if (family_of(d) != Family::kGqa || d.kv_dtype != SPLITKV_FP8_E4M3 || rows_per_head > 16) return 1;
  // Two heads per item measured best on GB300 (e4m3, 32 query / 4 KV heads,
  // 28k-33k keys: 47.1 us per call against 50.1 with four and 54.9 with one;
  // with two query tokens, 16 rows per head, 60.3 against 69.4 with one).
  // Past 16 rows the two heads' four row groups would need more warps than
  // the two-stage kernel form has threads and registers for.
  return d.num_kv_heads % 2 == 0 ? 2 : 1;
}

}  // namespace splitkv

using namespace splitkv;

extern "C" {

const char* splitkv_last_error(void) { return g_err; }

splitkv_status splitkv_plan(const splitkv_desc_t* desc, const int32_t* seq_lens_host,
                            int32_t num_splits, int32_t num_sms, splitkv_plan_t** plan_out) {
  if (!plan_out) return fail(SPLITKV_EINVAL, "plan_out is NULL");
  *plan_out = nullptr;
  splitkv_status st = validate_desc(desc);
  if (st != SPLITKV_OK) return st;
  if (!seq_lens_host) return fail(SPLITKV_EINVAL, "seq_lens_host is NULL");
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(SPLITKV_EINVAL, "num_splits (%d) must be in [0, %d]", num_splits, kMaxSplits);
  if (num_sms < 0) return fail(SPLITKV_EINVAL, "num_sms must be >= 0");
  const int64_t cap = int64_t(desc->max_pages_per_seq) * desc->page_size;
  for (int b = 0; b < desc->batch; ++b) {
    const int32_t L = seq_lens_host[b];
    if (L < 0 || L > cap)
      return fail(SPLITKV_EINVAL, "seq_lens[%d] = %d outside [0, max_pages_per_seq * page_size = %lld]",
                  b, L, (long long)cap);
    if (L > 0 && L < desc->q_tokens)
      return fail(SPLITKV_EINVAL, "seq_lens[%d] = %d is shorter than q_tokens = %d", b, L,
                  desc->q_tokens);
  }
  if (num_sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "querying the SM count");
  }
  splitkv_plan_s* p = new (std::nothrow) splitkv_plan_s();
  if (!p) return fail(SPLITKV_EINVAL, "out of host memory");
  p->desc = *desc;
  p->num_splits = num_splits;
  p->num_sms = num_sms;
  p->seq_lens.assign(seq_lens_host, seq_lens_host + desc->batch);
  build_plan(p);
  *plan_out = p;
  return SPLITKV_OK;
}

splitkv_status splitkv_plan_fixed(const splitkv_desc_t* desc, int32_t num_splits,
                                  splitkv_plan_t** plan_out) {
  if (!plan_out) return fail(SPLITKV_EINVAL, "plan_out is NULL");
  *plan_out = nullptr;
  splitkv_status st = validate_desc(desc);
  if (st != SPLITKV_OK) return st;
  if (num_splits < 1 || num_splits > kMaxSplits)
    return fail(SPLITKV_EINVAL, "num_splits (%d) must be in [1, %d] for a fixed plan", num_splits,
                kMaxSplits);
  const int64_t items = int64_t(desc->batch) * (desc->num_kv_heads / heads_per_item(*desc)) * num_splits;
  if (items * ctas_per_item(*desc) > (int64_t(1) << 31) - 1)
    return fail(SPLITKV_EINVAL, "too many work items (%lld)", (long long)items);
  splitkv_plan_s* p = new (std::nothrow) splitkv_plan_s();
  if (!p) return fail(SPLITKV_EINVAL, "out of host memory");
  p->desc = *desc;
  p->num_splits = num_splits;
  p->fixed = true;
  build_fixed_plan(p);
  *plan_out = p;
  return SPLITKV_OK;
}

splitkv_status splitkv_plan_refresh(const splitkv_plan_t* plan, void* workspace,
                                    const int32_t* seq_lens, void* stream) {
  if (!plan) return fail(SPLITKV_EINVAL, "plan is NULL");
  if (!plan->fixed) return fail(SPLITKV_EINVAL, "plan was not made by splitkv_plan_fixed");
  if (!workspace) return fail(SPLITKV_EWORKSPACE, "workspace is NULL");
  if (!seq_lens) return fail(SPLITKV_EINVAL, "seq_lens is NULL");
  if (!aligned16(workspace) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(SPLITKV_EINVAL, "workspace must be 16-byte and seq_lens 4-byte aligned");
  cudaError_t e = launch_refresh(*plan, workspace, seq_lens, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the plan refresh kernel");
  return SPLITKV_OK;
}

splitkv_status splitkv_read_items(const splitkv_plan_t* plan, const void* workspace,
                                  int32_t* items_host, int32_t capacity, void* stream) {
  if (!plan || !workspace || !items_host) return fail(SPLITKV_EINVAL, "NULL argument");
  if (capacity < plan->n_items)
    return fail(SPLITKV_EINVAL, "capacity %d < %d items", capacity, plan->n_items);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(items_host, static_cast<const unsigned char*>(workspace) + plan->off_items,
                                  plan->items.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the work list");
  return SPLITKV_OK;
}

void splitkv_plan_destroy(splitkv_plan_t* plan) { delete plan; }

int32_t splitkv_plan_num_items(const splitkv_plan_t* plan) { return plan ? plan->n_items : 0; }

int32_t splitkv_plan_num_ctas(const splitkv_plan_t* plan) { return plan ? plan->n_ctas : 0; }

int32_t splitkv_plan_heads_per_item(const splitkv_plan_t* plan) {
  return plan ? heads_per_item(plan->desc) : 0;
}

int32_t splitkv_plan_launches_per_call(const splitkv_plan_t* plan) {
  if (!plan) return 0;
  if (plan->n_groups == 0) return 1;
  const bool fused = plan->desc.combine_mode == SPLITKV_COMBINE_FUSED &&
                     family_of(plan->desc) == Family::kGqa;
  return fused ? 1 : 2;
}

splitkv_status splitkv_plan_get_items(const splitkv_plan_t* plan, int32_t* items_host,
                                      int32_t capacity, int32_t* n_items) {
  if (!plan || !n_items) return fail(SPLITKV_EINVAL, "plan and n_items must not be NULL");
  *n_items = plan->n_items;
  if (!items_host) return capacity == 0 ? SPLITKV_OK : fail(SPLITKV_EINVAL, "items_host is NULL");
  if (capacity < plan->n_items)
    return fail(SPLITKV_EINVAL, "capacity %d < %d items", capacity, plan->n_items);
  std::memcpy(items_host, plan->items.data(), plan->items.size() * sizeof(int32_t));
  return SPLITKV_OK;
}

splitkv_status splitkv_plan_get_ranges(const splitkv_plan_t* plan, int32_t* ranges_host,
                                       int32_t capacity, int32_t* n_ranges) {
  if (!plan || !n_ranges) return fail(SPLITKV_EINVAL, "plan and n_ranges must not be NULL");
  const int hpi = heads_per_item(plan->desc);
  const int32_t n = plan->n_items * hpi;
  *n_ranges = n;
  if (!ranges_host) return capacity == 0 ? SPLITKV_OK : fail(SPLITKV_EINVAL, "ranges_host is NULL");
  if (capacity < n) return fail(SPLITKV_EINVAL, "capacity %d < %d ranges", capacity, n);
  int32_t* out = ranges_host;
  for (int32_t i = 0; i < plan->n_items; ++i) {
    const int32_t* it = plan->items.data() + size_t(i) * SPLITKV_ITEM_FIELDS;
    for (int hh = 0; hh < hpi; ++hh, out += SPLITKV_RANGE_FIELDS) {
      out[0] = it[SPLITKV_ITEM_B];
      out[1] = it[SPLITKV_ITEM_HKV] + hh;
      out[2] = it[SPLITKV_ITEM_SPLIT];
      out[3] = it[SPLITKV_ITEM_PAGE0];
      out[4] = it[SPLITKV_ITEM_PAGE1];
    }
  }
  return SPLITKV_OK;
}

size_t splitkv_workspace_size(const splitkv_plan_t* plan) { return plan ? plan->total : 0; }

splitkv_status splitkv_plan_upload(const splitkv_plan_t* plan, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!plan) return fail(SPLITKV_EINVAL, "plan is NULL");
  if (!workspace) return fail(SPLITKV_EWORKSPACE, "workspace is NULL");
  if (!aligned16(workspace)) return fail(SPLITKV_EINVAL, "workspace must be 16-byte aligned");
  if (workspace_bytes < plan->total)
    return fail(SPLITKV_EWORKSPACE, "workspace has %zu bytes, plan needs %zu", workspace_bytes,
                plan->total);
  cudaError_t e = cudaMemcpyAsync(workspace, plan->upload.data(), plan->upload_bytes,
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "uploading the plan");
  return SPLITKV_OK;
}

namespace {

// The decode call; k_scale / v_scale (device, [Hkv]) replace kv_scale when
// given.  Without `merge` only the split-KV kernel runs (in SEPARATE form):
// sequences with more than one split leave their partials in the workspace.
splitkv_status decode_impl(const splitkv_plan_t* plan, void* workspace, const void* q,
                           const void* k_pages, const void* v_pages, const int32_t* block_table,
                           const int32_t* seq_lens, int32_t num_splits, float scale,
                           float kv_scale, const float* k_scale, const float* v_scale, void* out,
                           float* lse, void* stream, bool merge = true) {
  if (!plan) return fail(SPLITKV_EINVAL, "plan is NULL");
  const splitkv_desc_t& d = plan->desc;
  if (!workspace) return fail(SPLITKV_EWORKSPACE, "workspace is NULL");
  if (!q || !k_pages || !block_table || !seq_lens || !out)
    return fail(SPLITKV_EINVAL, "q, k_pages, block_table, seq_lens and out must not be NULL");
  if (!d.v_shares_k && !v_pages) return fail(SPLITKV_EINVAL, "v_pages is NULL");
  const void* ptrs[] = {workspace, q, k_pages, out, block_table, seq_lens};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return fail(SPLITKV_EINVAL, "device pointers must be 16-byte aligned");
  if (v_pages && !aligned16(v_pages)) return fail(SPLITKV_EINVAL, "v_pages must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SPLITKV_EINVAL, "lse must be 4-byte aligned");
  if (num_splits != 0 && num_splits != plan->num_splits)
    return fail(SPLITKV_EINVAL, "num_splits %d differs from the plan's %d", num_splits,
                plan->num_splits);
  if (!(scale > 0.f) || !(scale < 1e30f)) return fail(SPLITKV_EINVAL, "scale must be positive and finite");
  const bool fp8 = d.kv_dtype == SPLITKV_FP8_E4M3;
  const bool per_head = k_scale || v_scale;
  if (per_head) {
    if (!k_scale || !v_scale) return fail(SPLITKV_EINVAL, "k_scale and v_scale must both be given");
    if (!fp8 || family_of(d) != Family::kGqa)
      return fail(SPLITKV_EUNSUPPORTED, "per-head K/V scales apply to e4m3 GQA caches only");
    if ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u)
      return fail(SPLITKV_EINVAL, "k_scale and v_scale must be 4-byte aligned");
  } else if (fp8 && (!(kv_scale > 0.f) || !(kv_scale < 1e30f))) {
    return fail(SPLITKV_EINVAL, "kv_scale must be positive and finite");
  }

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  DecodeArgs a{};
  a.items = reinterpret_cast<const int32_t*>(ws + plan->off_items);
  a.groups = reinterpret_cast<const int32_t*>(ws + plan->off_groups);
  a.plan_lens = reinterpret_cast<const int32_t*>(ws + plan->off_seqlens);
  a.tickets = reinterpret_cast<int32_t*>(ws + plan->off_tickets);
  a.cta_log = reinterpret_cast<int32_t*>(ws + plan->off_log);
  a.status = reinterpret_cast<int32_t*>(ws + plan->off_status);
  a.lse_part = reinterpret_cast<float*>(ws + plan->off_lse);
  a.o_part = reinterpret_cast<float*>(ws + plan->off_o);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.q = q;
  a.out = out;
  a.lse = lse;
  a.n_items = plan->n_items;
  a.n_groups = plan->n_groups;
  a.batch = d.batch;
  a.T = d.q_tokens;
  a.Hq = d.num_q_heads;
  a.Hkv = d.num_kv_heads;
  a.G = d.num_q_heads / d.num_kv_heads;
  a.P = d.page_size;
  a.max_pages = d.max_pages_per_seq;
  a.num_pages = d.num_pages_total;
  a.rows = plan->rows;
  a.dv = d.v_dim;
  const float kLog2e = 1.4426950408889634f;
  // FP8 tiles are converted to their e4m3 values; the per-tensor kv_scale is
  // applied once to the scores and once to the output.
  a.qk_scale_log2 = scale * kLog2e * (fp8 && !per_head ? kv_scale : 1.f);
  a.o_scale = fp8 && !per_head ? kv_scale : 1.f;
  a.k_scale = k_scale;  // per-head factors, applied by the kernel per KV head
  a.v_scale = v_scale;
  a.fixed = plan->fixed ? 1 : 0;
  a.max_splits = plan->max_group_splits;
  a.hpi = heads_per_item(d);
  if (plan->fixed) a.fx = fixed_shape(*plan, seq_lens);
  a.fused = merge && d.combine_mode == SPLITKV_COMBINE_FUSED;
  // A grid of at most one CTA per SM takes the four-stage ring.  A capacity
  // plan is made without a device, so its decode reads the SM count of the
  // device it runs on.
  int sms = plan->num_sms;
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "querying the SM count");
  }
  a.deep_ring = plan->n_items <= sms ? 1 : 0;

  const int64_t rows_total = int64_t(d.num_pages_total) * d.num_kv_heads * d.page_size;
  if (family_of(d) == Family::kMla) {
    // Latent cache rows of 576 bf16 (boxes of min(P, 64) rows, one page at
    // most), and with a separate V tensor its rows of 512; the query rows are read by the
    // kernel's threads.  The partials are always merged by the separate
    // combine kernel.
    TmaDesc tk, tv;
    const int box_rows = d.page_size < 64 ? d.page_size : 64;
    splitkv_status st = fp8 ? make_u8_map(&tk, k_pages, d.qk_dim, rows_total, box_rows)
                            : make_bf16_map(&tk, k_pages, d.qk_dim, rows_total, box_rows);
    if (st != SPLITKV_OK) return st;
    if (!d.v_shares_k) {
      st = make_bf16_map(&tv, v_pages, d.v_dim, rows_total, box_rows);
      if (st != SPLITKV_OK) return st;
    }
    a.fused = 0;
    cudaError_t e = launch_mla(a, tk, d.v_shares_k ? nullptr : &tv, fp8, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the MLA split-KV kernel");
    if (merge) {
      e = launch_combine(a, true, stream);
      if (e != cudaSuccess) return cuda_fail(e, "launching the combine kernel");
    }
    return SPLITKV_OK;
  }
  TmaDesc tk, tv;
  const bool nhd = d.kv_layout == SPLITKV_LAYOUT_NHD;
  splitkv_status st =
      make_gqa_map(&tk, k_pages, fp8, d.page_size, d.num_kv_heads, d.num_pages_total, a.hpi, nhd);
  if (st != SPLITKV_OK) return st;
  st = make_gqa_map(&tv, v_pages, fp8, d.page_size, d.num_kv_heads, d.num_pages_total, a.hpi, nhd);
  if (st != SPLITKV_OK) return st;

  cudaError_t e = launch_gqa(a, tk, tv, fp8, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the split-KV kernel");
  if (merge && !a.fused) {
    e = launch_combine(a, true, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the combine kernel");
  }
  return SPLITKV_OK;
}

}  // namespace

splitkv_status splitkv_decode(const splitkv_plan_t* plan, void* workspace, const void* q,
                              const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* seq_lens,
                              int32_t num_splits, float scale, float kv_scale, void* out,
                              float* lse, void* stream) {
  return decode_impl(plan, workspace, q, k_pages, v_pages, block_table, seq_lens, num_splits,
                     scale, kv_scale, nullptr, nullptr, out, lse, stream);
}

splitkv_status splitkv_decode_kv_scales(const splitkv_plan_t* plan, void* workspace,
                                        const void* q, const void* k_pages, const void* v_pages,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int32_t num_splits, float scale, const float* k_scale,
                                        const float* v_scale, void* out, float* lse,
                                        void* stream) {
  if (!k_scale || !v_scale) return fail(SPLITKV_EINVAL, "k_scale and v_scale must not be NULL");
  return decode_impl(plan, workspace, q, k_pages, v_pages, block_table, seq_lens, num_splits,
                     scale, 1.f, k_scale, v_scale, out, lse, stream);
}

splitkv_status splitkv_decode_partials(const splitkv_plan_t* plan, void* workspace,
                                       const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       int32_t num_splits, float scale, float kv_scale, void* out,
                                       float* lse, void* stream) {
  return decode_impl(plan, workspace, q, k_pages, v_pages, block_table, seq_lens, num_splits,
                     scale, kv_scale, nullptr, nullptr, out, lse, stream, false);
}

splitkv_status splitkv_combine_workspace(const splitkv_plan_t* plan, void* workspace, void* out,
                                         float* lse, void* stream) {
  if (!plan) return fail(SPLITKV_EINVAL, "plan is NULL");
  if (!workspace) return fail(SPLITKV_EWORKSPACE, "workspace is NULL");
  if (!out) return fail(SPLITKV_EINVAL, "out must not be NULL");
  if (!aligned16(workspace) || !aligned16(out))
    return fail(SPLITKV_EINVAL, "device pointers must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SPLITKV_EINVAL, "lse must be 4-byte aligned");
  const splitkv_desc_t& d = plan->desc;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  DecodeArgs a{};
  a.groups = reinterpret_cast<const int32_t*>(ws + plan->off_groups);
  a.lse_part = reinterpret_cast<float*>(ws + plan->off_lse);
  a.o_part = reinterpret_cast<float*>(ws + plan->off_o);
  a.out = out;
  a.lse = lse;
  a.n_groups = plan->n_groups;
  a.T = d.q_tokens;
  a.Hq = d.num_q_heads;
  a.G = d.num_q_heads / d.num_kv_heads;
  a.rows = plan->rows;
  a.dv = d.v_dim;
  a.fixed = plan->fixed ? 1 : 0;
  a.max_splits = plan->max_group_splits;
  cudaError_t e = launch_combine(a, true, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the combine kernel");
  return SPLITKV_OK;
}

splitkv_status splitkv_combine(const float* o_part, const float* lse_part, int32_t n_parts,
                               int32_t rows, int32_t dv, void* out_bf16, float* out_f32,
                               float* lse_out, void* stream) {
  if (!o_part || !lse_part) return fail(SPLITKV_EINVAL, "o_part and lse_part must not be NULL");
  if (n_parts < 1 || rows < 0) return fail(SPLITKV_EINVAL, "n_parts must be >= 1 and rows >= 0");
  if (dv < 4 || dv % 4) return fail(SPLITKV_EINVAL, "dv must be a positive multiple of 4");
  if (!out_bf16 && !out_f32 && !lse_out) return fail(SPLITKV_EINVAL, "no output given");
  if (!aligned16(o_part) || (out_f32 && !aligned16(out_f32)) ||
      (out_bf16 && (reinterpret_cast<uintptr_t>(out_bf16) & 7u)))
    return fail(SPLITKV_EINVAL, "misaligned buffers");
  cudaError_t e = launch_combine_raw(o_part, lse_part, n_parts, rows, dv, out_bf16, out_f32,
                                     lse_out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the combine kernel");
  return SPLITKV_OK;
}

splitkv_status splitkv_read_stats(const splitkv_plan_t* plan, const void* workspace,
                                  int32_t* cta_log_host, int32_t capacity, int32_t* status_host,
                                  void* stream) {
  if (!plan || !workspace) return fail(SPLITKV_EINVAL, "plan and workspace must not be NULL");
  if (cta_log_host && capacity < plan->n_ctas)
    return fail(SPLITKV_EINVAL, "cta log capacity %d < %d CTAs", capacity, plan->n_ctas);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned char* ws = static_cast<const unsigned char*>(workspace);
  cudaError_t e = cudaSuccess;
  if (cta_log_host && plan->n_ctas)
    e = cudaMemcpyAsync(cta_log_host, ws + plan->off_log,
                        size_t(plan->n_ctas) * kLogFields * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && status_host)
    e = cudaMemcpyAsync(status_host, ws + plan->off_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the statistics");
  return SPLITKV_OK;
}

splitkv_status splitkv_debug_gather(const splitkv_desc_t* desc, const void* pages,
                                    int32_t row_elems, const int32_t* block_table, int32_t b,
                                    int32_t h_kv, int32_t n_keys, void* dst, void* stream) {
  splitkv_status st = validate_desc(desc);
  if (st != SPLITKV_OK) return st;
  if (!pages || !block_table || !dst) return fail(SPLITKV_EINVAL, "NULL pointer");
  if (b < 0 || b >= desc->batch || h_kv < 0 || h_kv >= desc->num_kv_heads)
    return fail(SPLITKV_EINVAL, "b or h_kv out of range");
  if (n_keys < 0 || int64_t(n_keys) > int64_t(desc->max_pages_per_seq) * desc->page_size)
    return fail(SPLITKV_EINVAL, "n_keys out of range");
  if (!aligned16(pages) || !aligned16(dst)) return fail(SPLITKV_EINVAL, "misaligned buffers");
  if (family_of(*desc) == Family::kMla) {
    // the latent key rows (qk_dim wide) or a separate V tensor (v_dim wide)
    if (row_elems != desc->qk_dim && !(row_elems == desc->v_dim && !desc->v_shares_k))
      return fail(SPLITKV_EINVAL, "row_elems (%d) must be qk_dim, or v_dim for a separate V tensor",
                  row_elems);
    TmaDesc t;
    const int64_t rows_total = int64_t(desc->num_pages_total) * desc->page_size;
    const bool fp8 = desc->kv_dtype == SPLITKV_FP8_E4M3;
    const int box_rows = desc->page_size < 64 ? desc->page_size : 64;
    st = fp8 ? make_u8_map(&t, pages, row_elems, rows_total, box_rows)
             : make_bf16_map(&t, pages, row_elems, rows_total, box_rows);
    if (st != SPLITKV_OK) return st;
    cudaError_t e = launch_mla_debug_gather(t, fp8, block_table + size_t(b) * desc->max_pages_per_seq,
                                            desc->page_size, desc->num_pages_total, row_elems,
                                            n_keys, dst, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the gather kernel");
    return SPLITKV_OK;
  }
  if (row_elems != 128) return fail(SPLITKV_EINVAL, "GQA rows are 128 wide");
  const bool fp8 = desc->kv_dtype == SPLITKV_FP8_E4M3;
  TmaDesc t;
  st = make_gqa_map(&t, pages, fp8, desc->page_size, desc->num_kv_heads, desc->num_pages_total, 1,
                    desc->kv_layout == SPLITKV_LAYOUT_NHD);
  if (st != SPLITKV_OK) return st;
  cudaError_t e = launch_debug_gather(t, fp8, block_table + size_t(b) * desc->max_pages_per_seq,
                                      h_kv, desc->page_size, n_keys, dst, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the gather kernel");
  return SPLITKV_OK;
}

}  // extern "C"
