// Internal declarations shared by the planner, the C-ABI layer and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime_api.h>

#include "splitkv.h"

namespace splitkv {

constexpr int kMaxSplits = 64;     // cap on splits per sequence
constexpr int kItemOverhead = 96;  // planner: fixed cost of one work item, 1/16-page units
constexpr int kCombineCost = 2;    // planner: merge cost per split, 1/16-page units
constexpr int kMaxWaves = 8;       // planner: candidate granularities, 1..8 items per slot
constexpr int kGqaCtasPerSm = 3;   // resident CTAs per SM of the GQA kernel
constexpr int kGroupFields = 4;    // {b, first h_kv, S_b, first slot}
constexpr int kLogFields = 4;      // per-CTA log record
constexpr size_t kAlign = 256;

// Which kernel family serves a descriptor.
enum class Family { kGqa, kMla, kNone };

Family family_of(const splitkv_desc_t& d);

// KV heads one work item covers (consecutive, from the item's h_kv): for the
// e4m3 GQA path with at most 8 query rows per head, 2 when Hkv is even (one
// TMA box brings a 16-key tile of both), else 1; otherwise 1.
int heads_per_item(const splitkv_desc_t& d);

// Query rows one work item produces: heads_per_item * T * G.
inline int rows_per_item(const splitkv_desc_t& d) {
  return heads_per_item(d) * d.q_tokens * (d.num_q_heads / d.num_kv_heads);
}

// CTAs launched per work item (1 for GQA; token tiles x CTA pair for MLA).
int ctas_per_item(const splitkv_desc_t& d);

// Resident CTAs per SM the planner counts on (kGqaCtasPerSm for GQA, 1 for MLA).
int ctas_per_sm(const splitkv_desc_t& d);

}  // namespace splitkv

struct splitkv_plan_s {
  splitkv_desc_t desc;
  int32_t num_splits = 0;  // as requested (0 = planner's choice)
  bool fixed = false;      // capacity plan whose work list a kernel rewrites (splitkv_plan_fixed)
  int32_t num_sms = 0;
  std::vector<int32_t> seq_lens;
  std::vector<int32_t> items;   // n_items * SPLITKV_ITEM_FIELDS, launch order
  std::vector<int32_t> groups;  // n_groups * kGroupFields, (b, h_kv) order
  int32_t n_items = 0, n_groups = 0, n_slots = 0, rows = 0, n_ctas = 0;
  int32_t max_group_splits = 0;  // largest S of a combine group (0: no group)
  // workspace byte offsets
  size_t off_status = 0, off_items = 0, off_groups = 0, off_seqlens = 0, off_tickets = 0;
  size_t off_log = 0, off_lse = 0, off_o = 0, upload_bytes = 0, total = 0;
  std::vector<unsigned char> upload;  // host image of [0, upload_bytes)
};

namespace splitkv {

// Planner (plan.cpp, host only).  Fills items/groups/offsets of `p` from
// p->desc, p->seq_lens, p->num_splits, p->num_sms.
void build_plan(splitkv_plan_s* p);

// Capacity plan (plan.cpp): items (b, head group, s) for every s < num_splits,
// all marked unused (NSPLIT = 0) until splitkv_plan_refresh rewrites them on
// the device; one combine group per (b, head group) when num_splits > 1.
void build_fixed_plan(splitkv_plan_s* p);

// Thread-local error text (api.cu).
splitkv_status fail(splitkv_status s, const char* fmt, ...);

// ----------------------------------------------------------------- kernels

// Shape of a capacity plan's work list, from which the kernels derive each
// item and combine group from the device lengths (fixed_plan.cuh).
struct FixedShape {
  const int32_t* seq_lens;  // device lengths [B], read after the dependency wait
  int32_t S;                // items per (sequence, head group)
  int32_t U;                // head groups per sequence (Hkv / heads per item)
  int32_t hpi;              // KV heads per item
  int32_t P;                // page size
  int32_t T;                // query tokens
  int64_t cap;              // max_pages_per_seq * P
};

struct DecodeArgs {
  const int32_t* items;
  const int32_t* groups;
  const int32_t* plan_lens;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const void* q;
  void* out;
  float* lse;
  float* o_part;
  float* lse_part;
  int32_t* tickets;
  int32_t* cta_log;
  int32_t* status;
  int32_t n_items, n_groups;
  int32_t batch, T, Hq, Hkv, G, P, max_pages, num_pages, rows, dv;
  float qk_scale_log2;  // scale * kv_scale (FP8 only) * log2(e)
  float o_scale;        // factor applied to the normalised output (FP8: kv_scale)
  int32_t fused;        // 1: last CTA of a group merges
  int32_t hpi;          // KV heads per item (e4m3 boxes are [hpi][16][128])
  const float* k_scale;  // e4m3 per-KV-head scales [Hkv] (device) or null: the
  const float* v_scale;  //   kernel multiplies qk_scale_log2 / o_scale by them
  int32_t fixed;         // 1: the work list was written by a kernel (read it after the
                         //    dependency wait); items with NSPLIT = 0 are unused
  int32_t max_splits;    // largest S of a combine group (sizes the combine kernel's loads)
  FixedShape fx;         // capacity plans: the kernels derive items and groups from it
  int32_t deep_ring;     // 1: at most one CTA per SM, so the GQA kernel may take the
                         //    deeper (four-stage) ring instead of sharing the SM
};

// Raw 128-byte tensor map storage (CUtensorMap), built by the API layer.
struct alignas(64) TmaDesc {
  unsigned char bytes[128];
};

cudaError_t launch_gqa(const DecodeArgs& a, const TmaDesc& tk, const TmaDesc& tv, bool fp8,
                       void* stream);
// tv: the V map of a cache with separate V rows, or null when V is the first
// columns of the key rows
// fp8: tk is an unswizzled uint8 map over e4m3 latent rows (tv must be null)
cudaError_t launch_mla(const DecodeArgs& a, const TmaDesc& tk, const TmaDesc* tv, bool fp8,
                       void* stream);
cudaError_t launch_combine(const DecodeArgs& a, bool pdl, void* stream);
// The FixedShape of a capacity plan over device lengths `seq_lens`.
FixedShape fixed_shape(const splitkv_plan_s& p, const int32_t* seq_lens);
cudaError_t launch_refresh(const splitkv_plan_s& p, void* workspace, const int32_t* seq_lens,
                           void* stream);
cudaError_t launch_combine_raw(const float* o_part, const float* lse_part, int n_parts, int rows,
                               int dv, void* out_bf16, float* out_f32, float* lse_out,
                               void* stream);
cudaError_t launch_debug_gather(const TmaDesc& t, bool fp8, const int32_t* table_row,
                                int32_t h_kv, int32_t P, int32_t n_keys, void* dst, void* stream);
// The MLA family's gather (2-D latent or separate-V map, row_elems 576 or 512).
cudaError_t launch_mla_debug_gather(const TmaDesc& t, bool fp8, const int32_t* table_row, int32_t P,
                                    int32_t num_pages, int32_t row_elems, int32_t n_keys, void* dst,
                                    void* stream);

}  // namespace splitkv
