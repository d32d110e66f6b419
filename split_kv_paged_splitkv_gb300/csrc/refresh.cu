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

#include "internal.h"

namespace splitkv {
namespace {

__global__ void refresh_kernel(const int32_t* __restrict__ seq_lens, int32_t* items, int32_t* groups,
                               int32_t* plan_lens, int32_t* status, int B, int U, int hpi, int S,
                               int P, int T, int64_t cap) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * U * S) return;
  const int s = i % S, u = (i / S) % U, b = i / (S * U);
  int L = seq_lens[b];
  if (L < 0 || int64_t(L) > cap || (L > 0 && L < T)) {
    // not a length the plan can serve: the sequence is treated as empty
    if (s == 0 && u == 0) atomicOr(status, SPLITKV_DEVERR_SEQLEN);
    L = 0;
  }
  const int n = (L + P - 1) / P;
  const int Sb = n > 0 ? min(S, n) : 1;
  const int g = b * U + u;
  const bool split = Sb > 1;
  int32_t f[SPLITKV_ITEM_FIELDS] = {b, u * hpi, s, 0, 0, 0, -1, -1};
  if (s < Sb) {
    f[SPLITKV_ITEM_NSPLIT] = Sb;
    f[SPLITKV_ITEM_PAGE0] = n > 0 ? int32_t((int64_t(s) * n) / Sb) : 0;
    f[SPLITKV_ITEM_PAGE1] = n > 0 ? int32_t((int64_t(s + 1) * n) / Sb) : 0;
    f[SPLITKV_ITEM_SLOT] = split ? g * S + s : -1;
    f[SPLITKV_ITEM_GROUP] = split ? g : -1;
  }
  int32_t* it = items + size_t(i) * SPLITKV_ITEM_FIELDS;
#pragma unroll
  for (int k = 0; k < SPLITKV_ITEM_FIELDS; ++k) it[k] = f[k];
  if (s == 0 && groups) {
    int32_t* gr = groups + size_t(g) * kGroupFields;
    gr[0] = b;
    gr[1] = u * hpi;
    gr[2] = split ? Sb : 0;  // 0: nothing to merge (the split kernel wrote the output)
    gr[3] = g * S;
  }
  if (s == 0 && u == 0) plan_lens[b] = L;
}

}  // namespace

cudaError_t launch_refresh(const splitkv_plan_s& p, void* workspace, const int32_t* seq_lens,
                           void* stream) {
  const splitkv_desc_t& d = p.desc;
  if (p.n_items == 0) return cudaSuccess;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const int hpi = heads_per_item(d);
  const int threads = 128, blocks = (p.n_items + threads - 1) / threads;
  refresh_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      seq_lens, reinterpret_cast<int32_t*>(ws + p.off_items),
      p.n_groups ? reinterpret_cast<int32_t*>(ws + p.off_groups) : nullptr,
      reinterpret_cast<int32_t*>(ws + p.off_seqlens), reinterpret_cast<int32_t*>(ws + p.off_status),
      d.batch, d.num_kv_heads / hpi, hpi, p.num_splits, d.page_size, d.q_tokens,
      int64_t(d.max_pages_per_seq) * d.page_size);
  return cudaGetLastError();
}

}  // namespace splitkv
