// Device-side rewrite of a capacity plan's work list (splitkv_plan_refresh).
//
// A CUDA graph fixes every launch's grid, while the sequence lengths of a
// serving batch change from step to step ("Shipped: 484.5 tok/s on one GB300
// ...", table "What shipped": splitting was enabled for one captured shape
// only).  A capacity plan launches num_splits items per (sequence, KV-head
// group); this kernel turns the current device lengths into the same split
// page ranges the host planner gives for that num_splits -- S_b = min(S,
// ceil(L_b / P)), split s covering pages [floor(s n / S_b), floor((s+1) n /
// S_b)) -- and marks the remaining capacity items unused (NSPLIT = 0), which
// the decode kernels skip.  Partial-result slots and combine groups keep
// fixed places: group g = b * U + u owns slots [g S, g S + S).
#include <cuda_runtime.h>

#include "fixed_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace splitkv {
namespace {

using namespace ptx;

__global__ void refresh_kernel(const FixedShape f, int n_items, int32_t* items, int32_t* groups,
                               int32_t* plan_lens, int32_t* status) {
  // Programmatic dependent launch: a following kernel may start its prologue
  // now; this kernel rewrites the work list only once the previous kernel on
  // the stream (which may still read it) has finished.
  launch_dependents();
  wait_prerequisites();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items) return;
  int32_t it[SPLITKV_ITEM_FIELDS];
  int L;
  bool bad;
  fixed_item(f, i, it, &L, &bad);
  const int s = it[SPLITKV_ITEM_SPLIT], u = it[SPLITKV_ITEM_HKV] / f.hpi, b = it[SPLITKV_ITEM_B];
  if (bad && s == 0 && u == 0) atomicOr(status, SPLITKV_DEVERR_SEQLEN);
  int32_t* dst = items + size_t(i) * SPLITKV_ITEM_FIELDS;
#pragma unroll
  for (int k = 0; k < SPLITKV_ITEM_FIELDS; ++k) dst[k] = it[k];
  if (s == 0 && groups) {
    int gb, ghkv, gS, slot0;
    fixed_group(f, b * f.U + u, &gb, &ghkv, &gS, &slot0);
    int32_t* gr = groups + size_t(b * f.U + u) * kGroupFields;
    gr[0] = gb;
    gr[1] = ghkv;
    gr[2] = gS;  // 0: nothing to merge (the split kernel wrote the output)
    gr[3] = slot0;
  }
  if (s == 0 && u == 0) plan_lens[b] = L;
}

}  // namespace

FixedShape fixed_shape(const splitkv_plan_s& p, const int32_t* seq_lens) {
  const splitkv_desc_t& d = p.desc;
  const int hpi = heads_per_item(d);
  FixedShape f;
  f.seq_lens = seq_lens;
  f.S = p.num_splits;
  f.U = d.num_kv_heads / hpi;
  f.hpi = hpi;
  f.P = d.page_size;
  f.T = d.q_tokens;
  f.cap = int64_t(d.max_pages_per_seq) * d.page_size;
  return f;
}

cudaError_t launch_refresh(const splitkv_plan_s& p, void* workspace, const int32_t* seq_lens,
                           void* stream) {
  if (p.n_items == 0) return cudaSuccess;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const int threads = 128, blocks = (p.n_items + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, refresh_kernel, fixed_shape(p, seq_lens), p.n_items,
                            reinterpret_cast<int32_t*>(ws + p.off_items),
                            p.n_groups ? reinterpret_cast<int32_t*>(ws + p.off_groups) : nullptr,
                            reinterpret_cast<int32_t*>(ws + p.off_seqlens),
                            reinterpret_cast<int32_t*>(ws + p.off_status));
}

}  // namespace splitkv
