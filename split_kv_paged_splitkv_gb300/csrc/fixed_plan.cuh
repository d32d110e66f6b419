// Work items of a capacity plan (splitkv_plan_fixed), derived on the device
// from the current sequence lengths.  The plan launches S items per
// (sequence, KV-head group) in (b, group, s) order and keeps fixed partial
// slots (group g = b * U + u owns slots [g S, g S + S)); these functions give
// each item the page range the host planner gives for S splits --
// S_b = min(S, ceil(L_b / P)), split s covering pages [floor(s n / S_b),
// floor((s + 1) n / S_b)) -- and mark items s >= S_b unused (NSPLIT = 0).
// The split kernels, the combine kernel and splitkv_plan_refresh all call
// them, so the three agree by construction.
#pragma once

#include <cstdint>

#include "internal.h"

namespace splitkv {

// The length served for a sequence of length L: L when the plan can serve it
// (0 <= L <= cap, and L >= T unless L == 0), else 0 -- an empty sequence,
// with `bad` set.
__device__ __forceinline__ int fixed_len_of(const FixedShape& f, int L, bool* bad) {
  *bad = L < 0 || int64_t(L) > f.cap || (L > 0 && L < f.T);
  return *bad ? 0 : L;
}

// The length served for sequence b (seq_lens[b], validated as above).
__device__ __forceinline__ int fixed_len(const FixedShape& f, int b, bool* bad) {
  return fixed_len_of(f, f.seq_lens[b], bad);
}

// The sequence of item i.
__device__ __forceinline__ int fixed_seq(const FixedShape& f, int i) { return i / (f.S * f.U); }

// Splits of sequence b for length L (1 for an empty sequence).
__device__ __forceinline__ int fixed_splits(const FixedShape& f, int L) {
  const int n = (L + f.P - 1) / f.P;
  return n > 0 ? min(f.S, n) : 1;
}

// Work-list fields of item i (SPLITKV_ITEM_* order) when its sequence has
// length L_raw; *L receives the length served and *bad whether L_raw was
// replaced by 0.
__device__ __forceinline__ void fixed_item_at(const FixedShape& f, int i, int L_raw,
                                              int32_t (&it)[SPLITKV_ITEM_FIELDS], int* L,
                                              bool* bad) {
  const int s = i % f.S, u = (i / f.S) % f.U, b = fixed_seq(f, i);
  *L = fixed_len_of(f, L_raw, bad);
  const int n = (*L + f.P - 1) / f.P;
  const int Sb = fixed_splits(f, *L);
  const int g = b * f.U + u;
  const bool split = Sb > 1;
  it[SPLITKV_ITEM_B] = b;
  it[SPLITKV_ITEM_HKV] = u * f.hpi;
  it[SPLITKV_ITEM_SPLIT] = s;
  it[SPLITKV_ITEM_NSPLIT] = s < Sb ? Sb : 0;
  it[SPLITKV_ITEM_PAGE0] = s < Sb && n > 0 ? int32_t((int64_t(s) * n) / Sb) : 0;
  it[SPLITKV_ITEM_PAGE1] = s < Sb && n > 0 ? int32_t((int64_t(s + 1) * n) / Sb) : 0;
  it[SPLITKV_ITEM_SLOT] = s < Sb && split ? g * f.S + s : -1;
  it[SPLITKV_ITEM_GROUP] = s < Sb && split ? g : -1;
}

// The same from the current device length seq_lens[b].
__device__ __forceinline__ void fixed_item(const FixedShape& f, int i,
                                           int32_t (&it)[SPLITKV_ITEM_FIELDS], int* L,
                                           bool* bad) {
  fixed_item_at(f, i, f.seq_lens[fixed_seq(f, i)], it, L, bad);
}

// Combine group g = b * U + u: (b, first KV head, splits to merge -- 0 when
// the split kernel wrote the output itself --, first slot).
__device__ __forceinline__ void fixed_group(const FixedShape& f, int g, int* b, int* hkv, int* S,
                                            int* slot0) {
  *b = g / f.U;
  *hkv = (g % f.U) * f.hpi;
  bool bad;
  const int Sb = fixed_splits(f, fixed_len(f, *b, &bad));
  *S = Sb > 1 ? Sb : 0;
  *slot0 = g * f.S;
}

// The combine-group entry (b, first KV head, splits to merge or 0, first
// slot) of the group of item `it`, written by the group's item s == 0: a
// capacity plan's group table is not uploaded, since S_b follows the lengths.
// The combine kernel reads it after its dependency wait.
__device__ __forceinline__ void fixed_write_group(const FixedShape& f, int32_t* groups,
                                                  const int32_t (&it)[SPLITKV_ITEM_FIELDS]) {
  if (groups == nullptr || f.S <= 1 || it[SPLITKV_ITEM_SPLIT] != 0) return;
  const int g = it[SPLITKV_ITEM_B] * f.U + it[SPLITKV_ITEM_HKV] / f.hpi;
  const int Sb = it[SPLITKV_ITEM_NSPLIT];
  int32_t* gr = groups + size_t(g) * kGroupFields;
  gr[0] = it[SPLITKV_ITEM_B];
  gr[1] = it[SPLITKV_ITEM_HKV];
  gr[2] = Sb > 1 ? Sb : 0;
  gr[3] = g * f.S;
}

}  // namespace splitkv
