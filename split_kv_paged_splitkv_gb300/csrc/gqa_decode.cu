// Split-KV partial attention for thin query groups (GQA), sm_103a.
//
// One CTA per work item (b, HPI consecutive KV heads, split, page range).
// The split's pages are streamed HBM -> shared memory by TMA: one tiled box
// per 16-key tile of K and one of V, covering the item's HPI heads, through
// tensor maps whose coordinates are (dims, key in page, [column half,] KV
// head, page) whether the pools are HND or NHD, with the 128-byte swizzle so
// the ldmatrix reads below are bank-conflict free.  The boxes land in a ring
// of NST stages guarded by mbarriers: two 32 KB stages, so that three CTAs
// share an SM, or four for a grid of at most one CTA per SM, whose producer
// also warms L2 with its first tiles before the dependency wait (a capacity
// plan's CTA picks those tiles from a speculative read of the device length;
// its real item comes from the length read after the wait).  One
// producer warp issues the copies (four, taking the tiles round-robin, in
// the four-stage form, whose CTA has an SM to itself).  The four consumer
// warps form slots (head slot, row group): each slot serves query rows
// [8 rg, 8 rg + 8) of KV head h0 + hs, and a slot's warps take its tiles
// round-robin.
//
// Per 16-key tile a consumer warp computes, on the warp tensor-core path:
//   S^T[16 keys x 8 rows] = K_tile[16 x 128] . Q^T      (m16n8k16, keys on M)
//   online softmax over the keys of each query row (shuffle reductions)
//   O^T[128 x 8 rows]   += V_tile^T[128 x 16] . P^T     (m16n8k16, dims on M)
// so a row group of up to 8 query rows fills the MMA's N side (9 to 16 rows
// per KV head -- speculative decode -- take two row groups over the same
// tiles, 17 to 32 four) and the 16-key tile fills M with no padding.  P^T is turned from
// accumulator layout into operand layout in registers with movmatrix.  FP8
// e4m3 tiles are converted to f16 in registers (exact, ptx::e4m3x2_*) and
// use the f16 MMA; BF16 tiles go straight to the bf16 MMA.
//
// The (m, l, O) of the warps sharing a slot are merged in shared memory; the
// item's result is written as the final bf16 output (S_b == 1) or as an fp32
// partial with its natural-log LSE.  With the fused combine, the last CTA of
// a (b, head group) group -- or, past 8 splits, of each bundle of 8 splits
// and then of the bundles (atomic tickets, no waiting) -- merges the partials.
//
// This is the split partial of "vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can
// Be 48% Slower", section "What SplitKV is trying to do"; the merge gives
// partials with LSE = -inf zero weight (section "Why the result is still
// correct").  FP8 KV with BF16 queries: "Xqa decode kernels", section
// "Purpose".
#include <cuda_runtime.h>

#include <cfloat>

#include "fixed_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace splitkv {
namespace {

using namespace ptx;

// A tile is 16 keys of the item's HPI KV heads: its K box ([HPI][16 rows])
// then its V box.  A stage -- the unit one mbarrier phase covers -- is TPS
// tiles (32 KB).  Measured on GB300, one CTA keeps only about one stage's
// worth of TMA boxes in flight however deep its ring is, and small boxes
// stream more slowly than large ones, so per-SM bandwidth comes from several
// CTAs per SM (a two-stage ring and 160 threads let three CTAs share an SM)
// and from boxes that span several heads (HPI > 1, e4m3 only).  A grid of at
// most one CTA per SM cannot share SMs; its CTAs take a four-stage ring
// instead (128 KB, a whole item of a few thousand keys in flight at once).
template <bool FP8, int HPI, int NRG = 1, int NST_ = 2>
struct Gqa {
  static_assert(HPI == 1 || (FP8 && (HPI == 2 || HPI == 4)), "heads per item");
  static_assert(NRG == 1 || ((NRG == 2 || NRG == 4) && HPI == 1) || (NRG == 2 && HPI == 2),
                "row groups per head");
  static constexpr int D = 128;
  static constexpr int TK = 16;                            // keys per tile
  static constexpr int KT_BYTES = TK * D * (FP8 ? 1 : 2);  // one head's K (or V) rows
  static constexpr int TILE = 2 * HPI * KT_BYTES;          // K + V boxes of one tile
  static constexpr int STAGE = 32768;
  static constexpr int TPS = STAGE / TILE;                 // tiles per stage
  static constexpr int NST = NST_;                         // stages in the ring
  // Consumer warps: eight when two or four row groups share a one-wave CTA
  // (more warps per row group shorten the chain of tiles each scores: on the
  // 5.9k shape two tokens of a G = 8 group took 7.35 -> 7.11 us per call,
  // four 8.82 -> 8.41), else four.
  static constexpr int NCW = NST_ == 4 && NRG >= 2 ? 8 : 4;
  // Producer warps: four for the one-wave four-stage ring (tiles go to them
  // round-robin; measured on GB300, a CTA's cold 48 KB lands about 13 %
  // sooner when four warps issue its boxes than when one does), one for the
  // two-stage ring, whose three CTAs per SM have no threads to spare.
  static constexpr int NPROD = NST_ == 4 ? 4 : 1;
  // A slot is (head slot hs, row group rg) = (slot % HPI, slot / HPI): the
  // warps of a slot score query rows [8 rg, 8 rg + 8) of KV head h0 + hs.
  static constexpr int SLOTS = HPI * NRG;
  static constexpr int WPH = NCW / SLOTS;                  // warps per slot
  static constexpr int THREADS = (NCW + NPROD) * 32;
  static constexpr int MIN_CTAS = NST_ == 4 ? 1 : kGqaCtasPerSm;  // resident CTAs per SM
  static constexpr int RING = NST * STAGE;
  static constexpr int ROWS = 8 * SLOTS;                   // merge rows (8 per slot)
  // The warps' O rows in the merge area are MO_STRIDE floats apart: 4 more
  // than D, so that the 4 rows (2 ti) a warp's lanes store at once fall on
  // different banks (a 128-float stride put them on the same 8 banks).
  static constexpr int MO_STRIDE = D + 4;
  static constexpr int MERGE = NCW * 8 * MO_STRIDE * 4 + NCW * 8 * 2 * 4;
  static_assert(MERGE + 64 * ROWS * 4 <= RING, "merge area and staged LSEs alias the ring");
  // Warp w takes tiles w / HPI, w / HPI + WPH, ...: its successive visits to
  // one stage must be exactly one barrier phase apart (parity waits cannot
  // tell phase k from k + 2).  That holds when a warp visits every stage in
  // turn (TPS a multiple of WPH) or steps WPH / TPS stages at a time with that
  // step dividing NST.
  static constexpr bool kVisitsEveryStage = TPS % WPH == 0;
  static constexpr int kStageStep = WPH >= TPS ? WPH / TPS : 1;
  static_assert(kVisitsEveryStage || (WPH % TPS == 0 && NST % kStageStep == 0),
                "stage/warp aliasing");
  static constexpr int BARS = 2 * NST * 8;
  static constexpr int PT_CHUNK = 1024;  // block-table entries staged at a time
  // The four-stage form has shared memory to spare: its merge area is its
  // own, so each consumer warp stores its (m, l, O) as soon as its tiles are
  // done (in the two-stage form the area aliases the ring, and the warps
  // first wait for one another to drain it).
  static constexpr bool SEP_MERGE = NST_ == 4;
  static constexpr int SMEM = 1024 + RING + BARS + 64 + NPROD * PT_CHUNK * 4 + (SEP_MERGE ? MERGE : 0);
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a tile stored
// as 128-byte rows with the TMA 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// BF16 tiles are two 64-column halves, each [16 rows][128 B], 2 KB apart.
__device__ __forceinline__ uint32_t swz_bf16(int row, int d) {
  return static_cast<uint32_t>((d >> 6) * 2048) + swz(row, (d & 63) >> 3);
}

// Sums DPT consecutive floats of `x` (DPT a multiple of 4) into `acc` with weight w.
template <int DPT>
__device__ __forceinline__ void axpy(float (&acc)[DPT], float w, const float* x) {
#pragma unroll
  for (int i = 0; i < DPT; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    acc[i] += w * v.x; acc[i + 1] += w * v.y; acc[i + 2] += w * v.z; acc[i + 3] += w * v.w;
  }
}

// Writes DPT outputs of one query row: bf16 to `out` or fp32 to `dst`.
template <int DPT>
__device__ __forceinline__ void store_row(const float (&acc)[DPT], __nv_bfloat16* out, float* dst) {
#pragma unroll
  for (int i = 0; i < DPT; i += 4) {
    if (out) {
      uint2 v;
      v.x = pack_bf16(acc[i], acc[i + 1]);
      v.y = pack_bf16(acc[i + 2], acc[i + 3]);
      *reinterpret_cast<uint2*>(out + i) = v;
    } else {
      *reinterpret_cast<float4*>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    }
  }
}

// Merges the (m, l, O) of the warps sharing each slot and writes the item's
// result.  Runs on the NT = NCW * 32 consumer threads: merge row n = tid /
// TPR (slot n / 8, i.e. head slot hs and row group rg; query row rg * 8 +
// n % 8 of that head), DPT = 128 / TPR consecutive dims from d0.  `mo` is
// [NCW][8][MO_STRIDE] fp32, `mm`/`ml` [NCW][8]; m is in log2 units.  Partial rows
// are numbered hs * T*G + row.
template <bool FP8, int HPI, int NRG, int NST>
__device__ __forceinline__ void merge_and_store(const DecodeArgs& a, int tid, const float* mo,
                                                const float* mm, const float* ml, int b, int h0,
                                                int slot) {
  using C = Gqa<FP8, HPI, NRG, NST>;
  constexpr int NT = C::NCW * 32, TPR = NT / C::ROWS, DPT = 128 / TPR;
  const int n = tid / TPR;           // merge row
  const int sl = n >> 3, r8 = n & 7;
  const int hs = sl % HPI, r = (sl / HPI) * 8 + r8;  // head slot, query row of that head
  const int d0 = (tid % TPR) * DPT;  // first of DPT consecutive dims
  float M = -INFINITY;
#pragma unroll
  for (int j = 0; j < C::WPH; ++j) M = fmaxf(M, mm[(sl + C::SLOTS * j) * 8 + r8]);
  float acc[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int j = 0; j < C::WPH; ++j) {
      const int w = sl + C::SLOTS * j;
      const float sc = ex2(mm[w * 8 + r8] - M);
      lsum += sc * ml[w * 8 + r8];
      axpy<DPT>(acc, sc, mo + (w * 8 + r8) * C::MO_STRIDE + d0);
    }
  }
  float lse_n = -INFINITY;
  const float osc = a.v_scale ? __ldg(a.v_scale + h0 + hs) : a.o_scale;
  // (lsum is a sum of at most a few million terms of at most 1: far below
  // the 2^126 where the fast divide loses range)
  const float inv = lsum > 0.f ? __fdividef(osc, lsum) : 0.f;
#pragma unroll
  for (int i = 0; i < DPT; ++i) acc[i] *= inv;
  if (lsum > 0.f) lse_n = (M + lg2(lsum)) * kLn2;
  const int rph = a.T * a.G;  // query rows per head
  if (r >= rph) return;
  if (slot < 0) {
    const int t = r / a.G, g = r - (r / a.G) * a.G;
    const size_t row = (size_t(b) * a.T + t) * a.Hq + size_t(h0 + hs) * a.G + g;
    store_row<DPT>(acc, static_cast<__nv_bfloat16*>(a.out) + row * 128 + d0, nullptr);
    if (d0 == 0 && a.lse) a.lse[row] = lse_n;
  } else {
    const int pr = hs * rph + r;
    store_row<DPT>(acc, nullptr, a.o_part + (size_t(slot) * a.rows + pr) * 128 + d0);
    if (d0 == 0) a.lse_part[size_t(slot) * a.rows + pr] = lse_n;
  }
}

// Log-sum-exp merge of `count` partials of one (b, head group) group -- the
// slots first, first + stride, ... -- by one CTA.  NT threads over ROWS =
// 8 * HPI * NRG merge rows.  The count x rows LSE values are first staged in shared
// memory (`sl`, [count][ROWS]) by all threads at once; then thread (row n,
// DPT dims from d0) accumulates the weighted partials with U partials' loads
// in flight per step, so the L2 round trips overlap instead of serialising.
// out_slot < 0: the result is the final bf16 output and LSE; otherwise it is
// written as a partial (fp32 O, natural-log LSE) into slot out_slot, which may
// be one of the slots read (each thread reads its own elements before writing
// them, and the LSEs were staged before any is written).
template <int NT, int HPI, int NRG>
__device__ __forceinline__ void merge_group(const DecodeArgs& a, int tid, int b, int h0, int first,
                                            int count, int stride, int out_slot, float* sl) {
  constexpr int ROWS = 8 * HPI * NRG, TPR = NT / ROWS, DPT = 128 / TPR, U = 64 / DPT;
  const int rows = a.rows, rph = a.T * a.G;
  // merge row n: slot n / 8 = (head slot, row group), query row of that head
  auto hs_of = [](int n) { return (n >> 3) % HPI; };
  auto r_of = [](int n) { return ((n >> 3) / HPI) * 8 + (n & 7); };
  for (int i = tid; i < count * ROWS; i += NT) {
    const int s = i / ROWS, n = i % ROWS, hs = hs_of(n), r = r_of(n);
    sl[i] = r < rph ? __ldcg(a.lse_part + size_t(first + s * stride) * rows + hs * rph + r) : -INFINITY;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  const int n = tid / TPR;
  const int hs = hs_of(n), r = r_of(n);
  const int d0 = (tid % TPR) * DPT;
  if (r >= rph) return;
  float M = -INFINITY;
  for (int s = 0; s < count; ++s) M = fmaxf(M, sl[s * ROWS + n]);
  float acc[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    const size_t sstride = size_t(stride) * rows * 128;
    const float* base = a.o_part + (size_t(first) * rows + hs * rph + r) * 128 + d0;
    for (int s0 = 0; s0 < count; s0 += U) {
      float4 x[U][DPT / 4];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < DPT / 4; ++v)
          if (s0 + u < count)
            x[u][v] = __ldcg(reinterpret_cast<const float4*>(base + size_t(s0 + u) * sstride) + v);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (s0 + u < count) {
          const float w = ex2((sl[(s0 + u) * ROWS + n] - M) * kLog2e);
          wsum += w;
#pragma unroll
          for (int v = 0; v < DPT / 4; ++v) {
            acc[4 * v] += w * x[u][v].x; acc[4 * v + 1] += w * x[u][v].y;
            acc[4 * v + 2] += w * x[u][v].z; acc[4 * v + 3] += w * x[u][v].w;
          }
        }
      }
    }
  }
  float lse_n = -INFINITY;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int i = 0; i < DPT; ++i) acc[i] *= inv;
  if (wsum > 0.f) lse_n = M + lg2(wsum) * kLn2;
  if (out_slot >= 0) {
    const int pr = hs * rph + r;
    store_row<DPT>(acc, nullptr, a.o_part + (size_t(out_slot) * rows + pr) * 128 + d0);
    if (d0 == 0) a.lse_part[size_t(out_slot) * rows + pr] = lse_n;
    return;
  }
  const int t = r / a.G, g = r - (r / a.G) * a.G;
  const size_t row = (size_t(b) * a.T + t) * a.Hq + size_t(h0 + hs) * a.G + g;
  store_row<DPT>(acc, static_cast<__nv_bfloat16*>(a.out) + row * 128 + d0, nullptr);
  if (d0 == 0 && a.lse) a.lse[row] = lse_n;
}

// L2 prefetches of the tiles an item's ring takes first, issued by the
// producer warp while the previous kernel on the stream finishes (only in a
// one-wave grid, whose CTAs all start early; later waves of a larger grid
// start with nothing to overlap, measured 0.5-1 % slower): one lane per tile
// reads its block-table entry speculatively (a relaxed load; the previous
// kernel may still be writing the table) and prefetches its K and V boxes.
// A stale entry only warms the wrong page; the copies proper are issued after
// the dependency wait from entries read again.
template <class C, bool FP8>
__device__ __forceinline__ void prefetch_first_tiles(const DecodeArgs& a, const CUtensorMap* tk,
                                                     const CUtensorMap* tv, int b, int h0,
                                                     int k_begin, int n_tiles, int lane) {
  const int t = lane;
  if (t >= n_tiles || t >= C::NST * C::TPS) return;
  const int key0 = k_begin + t * 16;
  const int page = key0 / a.P;
  const int ph = ld_relaxed_gpu(a.block_table + size_t(b) * a.max_pages + page);
  if (ph < 0 || ph >= a.num_pages) return;
  const int kp = key0 - page * a.P;
  if (FP8) {
    tma_prefetch_4d(tk, 0, kp, h0, ph);
    tma_prefetch_4d(tv, 0, kp, h0, ph);
  } else {
    tma_prefetch_5d(tk, 0, kp, 0, h0, ph);
    tma_prefetch_5d(tv, 0, kp, 0, h0, ph);
  }
}

template <bool FP8, int HPI, int NRG, int NST>
__global__ void __launch_bounds__(Gqa<FP8, HPI, NRG, NST>::THREADS, Gqa<FP8, HPI, NRG, NST>::MIN_CTAS)
    gqa_splitkv_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv) {
  using C = Gqa<FP8, HPI, NRG, NST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::RING);
  uint64_t* empty = full + C::NST;
  int* misc = reinterpret_cast<int*>(empty + C::NST);  // [0] merge flag, [1] keys scored
  int* pt = misc + 16;                                 // staged block-table entries, per producer

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A host plan's item comes from the uploaded work list, with the plan's
  // copy of the sequence length (read first, so that these loads overlap the
  // rest of the prologue).
  int32_t it[SPLITKV_ITEM_FIELDS];
  int L = 0;
  if (!a.fixed) {
    const int32_t* src = a.items + size_t(blockIdx.x) * SPLITKV_ITEM_FIELDS;
#pragma unroll
    for (int k = 0; k < SPLITKV_ITEM_FIELDS; ++k) it[k] = src[k];
    L = a.plan_lens[it[SPLITKV_ITEM_B]];
  }

  // Prologue: only shared memory, the tensor maps and the uploaded work list,
  // so it may overlap the previous kernel on the stream (programmatic
  // dependent launch).  Everything a previous kernel may write -- the caller's
  // inputs and this workspace's partials and tickets -- is touched only after
  // griddepcontrol.wait.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), C::TPS * C::SLOTS);  // one arrival per tile and slot
    }
    misc[0] = 0;
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == C::NCW && lane == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  __syncthreads();  // barriers initialised before any thread uses them
  launch_dependents();
  // The plan's copy of the length is never written by a kernel; the caller's
  // device copy is only checked against it, after the wait and off the
  // critical path.  A capacity plan's item is derived from the device length
  // after the wait; before it, a relaxed read of that length (which the
  // previous kernel may still be writing) gives a speculative item whose
  // first tiles are only prefetched into L2, so a stale value costs nothing
  // but the prefetch.  Only the first producer warp issues the prefetches:
  // the other warps go straight to the dependency wait.
  if (a.fixed) {
    if (a.deep_ring && warp == C::NCW) {
      int Ls;
      bool bad_s;
      fixed_item_at(a.fx, blockIdx.x, ld_relaxed_gpu(a.fx.seq_lens + fixed_seq(a.fx, blockIdx.x)),
                    it, &Ls, &bad_s);
      if (it[SPLITKV_ITEM_NSPLIT] > 0) {
        const int kb = it[SPLITKV_ITEM_PAGE0] * a.P, ke = min(it[SPLITKV_ITEM_PAGE1] * a.P, Ls);
        prefetch_first_tiles<C, FP8>(a, &tk, &tv, it[SPLITKV_ITEM_B], it[SPLITKV_ITEM_HKV], kb,
                                     ke > kb ? (ke - kb + 15) >> 4 : 0, lane);
      }
    }
    wait_prerequisites();
    bool bad;
    fixed_item(a.fx, blockIdx.x, it, &L, &bad);
    if (threadIdx.x == 0) fixed_write_group(a.fx, const_cast<int32_t*>(a.groups), it);
  } else {
    if (a.deep_ring && warp == C::NCW) {
      const int kb = it[SPLITKV_ITEM_PAGE0] * a.P, ke = min(it[SPLITKV_ITEM_PAGE1] * a.P, L);
      prefetch_first_tiles<C, FP8>(a, &tk, &tv, it[SPLITKV_ITEM_B], it[SPLITKV_ITEM_HKV], kb,
                                   ke > kb ? (ke - kb + 15) >> 4 : 0, lane);
    }
    wait_prerequisites();
  }
  const int b = it[SPLITKV_ITEM_B], h0 = it[SPLITKV_ITEM_HKV];  // heads h0 .. h0+HPI-1
  const int split = it[SPLITKV_ITEM_SPLIT], nsplit = it[SPLITKV_ITEM_NSPLIT];
  const int p0 = it[SPLITKV_ITEM_PAGE0], p1 = it[SPLITKV_ITEM_PAGE1];
  const int slot = it[SPLITKV_ITEM_SLOT], group = it[SPLITKV_ITEM_GROUP];
  if (nsplit == 0) {  // a capacity item the current sequence lengths leave unused
    if (threadIdx.x == 0) {
      int32_t* lg = a.cta_log + size_t(blockIdx.x) * kLogFields;
      lg[0] = p0;
      lg[1] = p1;
      lg[2] = 0;
      lg[3] = 0;
    }
    return;
  }
  const int k_begin = p0 * a.P;
  const int k_end = min(p1 * a.P, L);
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + 15) >> 4 : 0;
  if (threadIdx.x == 0 && a.seq_lens[b] != L) atomicOr(a.status, SPLITKV_DEVERR_SEQLEN);

  if (warp >= C::NCW) {
    // --------------------------------------------------------------- producers
    // Each producer warp stages up to PT_CHUNK physical page ids of this item
    // in its own shared-memory array (coalesced loads; the warps read the same
    // entries, so they never wait for one another), then walks the tiles,
    // issuing its own (tile t goes to producer warp t % NPROD) from one elected
    // lane of the converged warp (copies issued by a converged warp cost a
    // fraction of the issue cycles of copies issued by a lane that branched
    // away from its warp).  The warp owning a stage's first tile arms the
    // stage's barrier with the stage's bytes; every warp waits for a ring slot
    // to be released before writing into it again.
    const int pw = warp - C::NCW;
    int32_t* ptw = pt + pw * C::PT_CHUNK;
    const int32_t* trow = a.block_table + size_t(b) * a.max_pages;
    const int pg_end = (k_end + a.P - 1) / a.P;
    const int tiles_per_page = a.P >> 4;
    // Last stage this warp issued into (a stage holds TPS >= NPROD tiles, so
    // every full stage holds a tile of every producer warp).
    static_assert(C::TPS >= C::NPROD, "every full stage has a tile of every producer warp");
    int last_j = -1;
    int t = 0;
    bool ok = true;
    for (int pc = p0; pc < pg_end && ok; pc += C::PT_CHUNK) {
      const int cnt = min(C::PT_CHUNK, pg_end - pc);
      __syncwarp();
      for (int x = lane; x < cnt; x += 32) {
        int ph = __ldg(trow + pc + x);
        if (ph < 0 || ph >= a.num_pages) {
          if (pw == 0) atomicOr(a.status, SPLITKV_DEVERR_PAGE);
          ph = 0;
        }
        ptw[x] = ph;
      }
      __syncwarp();
      const int t_end = min(n_tiles, (pc + cnt) * tiles_per_page - p0 * tiles_per_page);
      for (; t < t_end; ++t) {
        if (C::NPROD > 1 && t % C::NPROD != pw) continue;
        const int key0 = k_begin + t * 16;
        const int page = key0 / a.P;
        const int ph = ptw[page - pc];
        const int j = t / C::TPS, u = t - j * C::TPS, st = j % C::NST;
        const uint32_t bar = smem_u32(full + st);
        // the first of this warp's tiles in stage j (u < NPROD) waits for the
        // slot's release
        if (j >= C::NST && u < C::NPROD) {
          ok = __all_sync(kFull, mbar_wait(smem_u32(empty + st), ((j / C::NST) - 1) & 1));
          if (!ok) {
            if (lane == 0) atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
            break;
          }
        }
        if (u == 0) mbar_arrive_expect_tx_warp(bar, min(C::TPS, n_tiles - t) * C::TILE);
        last_j = j;
        const uint32_t dk = smem_u32(ring + st * C::STAGE + u * C::TILE);
        const uint32_t dv = dk + HPI * C::KT_BYTES;
        // The maps' coordinates are (dims, key in page, [column half,] KV
        // head, page) in either page layout; one box per operand and tile.
        const int kp = key0 - page * a.P;
        if (FP8) {  // [HPI heads][16 keys][128]
          tma_load_4d_warp(dk, &tk, bar, 0, kp, h0, ph);
          tma_load_4d_warp(dv, &tv, bar, 0, kp, h0, ph);
        } else {    // [2 halves][16 keys][64]
          tma_load_5d_warp(dk, &tk, bar, 0, kp, 0, h0, ph);
          tma_load_5d_warp(dv, &tv, bar, 0, kp, 0, h0, ph);
        }
      }
    }
    // Stay resident until every copy this warp issued has landed: the CTA
    // must not exit (and free its shared memory) with TMA writes in flight,
    // even when a consumer gave up on a timed-out wait.  Each ring slot is
    // waited on at the latest phase it reached: the item's last stage in that
    // slot, which covers the earlier phases (and, were a warp's own last
    // phase in a slot used instead, another warp's tile of the item's final
    // stage could complete one more phase there, leaving the barrier at the
    // parity the wait asks for).  A warp that gave up waits only on the
    // phases it used itself; the stage it stopped at cannot complete, so no
    // slot runs further.  Normally these waits return at once.
    const int final_j = !ok ? last_j : n_tiles > 0 ? (n_tiles - 1) / C::TPS : -1;
    if (lane == 0) {
      for (int st = 0; st < C::NST; ++st) {
        const int j = final_j - ((final_j - st + C::NST) % C::NST);
        if (j < 0) continue;
        if (!mbar_wait(smem_u32(full + st), (j / C::NST) & 1)) {
          atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
          break;
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int tid = threadIdx.x;  // consumer threads 0 .. NCW*32-1
  const int gi = lane >> 2, ti = lane & 3;
  const int slot_w = warp % C::SLOTS;  // this warp's slot:
  const int hs = slot_w % HPI;         //   KV head h0 + hs,
  const int rg = slot_w / HPI;         //   query rows [8 rg, 8 rg + 8) of that head
  const int hkv = h0 + hs;
  const int rph = a.T * a.G;           // query rows per KV head
  // scores -> log2 units: scale (and the e4m3 K scale, per KV head if given)
  const float qk_l2 = a.k_scale ? a.qk_scale_log2 * __ldg(a.k_scale + hkv) : a.qk_scale_log2;
  // Per query row of this lane's scores (rows 2ti, 2ti + 1 of the slot's row
  // group): qk_l2 times the inverse of the power of two the row's f16 query
  // fragments were scaled by (e4m3 path; 1 for bf16).
  float qk0 = qk_l2, qk1 = qk_l2;

  // Q^T operand fragments: query row n = 8 rg + gi of this head, dims by ti
  // (see the layout notes); rows past the head's T*G rows are zero.
  uint32_t qf[8][2];
  {
    const int n = rg * 8 + gi;
    if (!FP8) {
      if (n < rph) {
        const int t = n / a.G, g = n - t * a.G;
        const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) +
                                  ((size_t(b) * a.T + t) * a.Hq + size_t(hkv) * a.G + g) * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qf[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qp + ks * 16 + 2 * ti));
          qf[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qp + ks * 16 + 2 * ti + 8));
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) qf[ks][0] = qf[ks][1] = 0u;
      }
    } else {
      // The f16 MMA needs f16 queries, whose range (|x| < 65,520, normal from
      // 2^-14) is far narrower than bf16's.  Each row is scaled by 2^k so that
      // its largest component lies in [2^14, 2^15): a power of two is exact,
      // and every component then rounds to f16 without loss unless it is
      // below 2^-29 of the row maximum (a term 2^-29 of the largest one).  The
      // row's score scale takes the factor 2^-k.  The four lanes ti of a row
      // (lanes 4 gi .. 4 gi + 3) hold its 128 dims.
      float f[8][4];
      float amax = 0.f;
      if (n < rph) {
        const int t = n / a.G, g = n - t * a.G;
        const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) +
                                  ((size_t(b) * a.T + t) * a.Hq + size_t(hkv) * a.G + g) * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          // k = 2ti, 2ti+1 <-> d = 16ks+4ti, +1 ; k = 2ti+8, 2ti+9 <-> d = 16ks+4ti+2, +3
          // (the byte order of the e4m3 K operand, see the QK product below)
          const uint2 raw = __ldg(reinterpret_cast<const uint2*>(qp + ks * 16 + 4 * ti));
          f[ks][0] = __uint_as_float(raw.x << 16);
          f[ks][1] = __uint_as_float(raw.x & 0xffff0000u);
          f[ks][2] = __uint_as_float(raw.y << 16);
          f[ks][3] = __uint_as_float(raw.y & 0xffff0000u);
#pragma unroll
          for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(f[ks][i]));
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) f[ks][0] = f[ks][1] = f[ks][2] = f[ks][3] = 0.f;
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      // k = 14 - floor(log2 amax), within [-113, 126] so that 2^k and 2^-k are
      // normal floats (a zero row keeps k = 0)
      int k = 0;
      if (amax > 0.f) k = min(126, max(-113, 14 - (int((__float_as_uint(amax) >> 23) & 0xff) - 127)));
      const float up = __uint_as_float(uint32_t(127 + k) << 23);
      const float down = __uint_as_float(uint32_t(127 - k) << 23);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qf[ks][0] = pack_f16(f[ks][0] * up, f[ks][1] * up);
        qf[ks][1] = pack_f16(f[ks][2] * up, f[ks][3] * up);
      }
      // rows 2ti and 2ti + 1 are held by lanes 8 ti and 8 ti + 4
      qk0 = qk_l2 * __shfl_sync(kFull, down, 8 * ti);
      qk1 = qk_l2 * __shfl_sync(kFull, down, 8 * ti + 4);
    }
  }
  // Visible-key limits of the two query rows whose scores this lane holds.
  int lim0 = -1, lim1 = -1;
  {
    const int n0 = rg * 8 + 2 * ti, n1 = n0 + 1;
    if (n0 < rph) lim0 = L - a.T + n0 / a.G;
    if (n1 < rph) lim1 = L - a.T + n1 / a.G;
  }
  const int min_lim = L - a.T;

  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int keys_scored = 0;

  for (int i = warp / C::SLOTS; i < n_tiles; i += C::WPH) {
    const int j = i / C::TPS, st = j % C::NST;
    const bool arrived = __all_sync(kFull, mbar_wait(smem_u32(full + st), (j / C::NST) & 1));
    if (!arrived) {
      if (lane == 0) atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      break;
    }
    uint8_t* kt = ring + st * C::STAGE + (i - j * C::TPS) * C::TILE + hs * C::KT_BYTES;
    uint8_t* vt = kt + HPI * C::KT_BYTES;
    const int key0 = k_begin + i * 16;
    const int valid = min(16, k_end - key0);
    if (slot_w == 0) keys_scored += valid;
    if (valid < 16) {
      // Slots past the last visible key may hold anything (even NaN): zero
      // those V rows so that 0 * V stays 0 in the PV product.
      const int rows_bad = 16 - valid;
      const int halves = FP8 ? 1 : 2;
      for (int x = lane; x < rows_bad * 8 * halves; x += 32) {
        const int r = valid + (x >> 3) % rows_bad;
        const int h = x / (8 * rows_bad);
        *reinterpret_cast<uint4*>(vt + h * 2048 + r * 128 + (x & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      // order these generic-proxy writes before the stage's next TMA refill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // ---- S^T = K . Q^T (two accumulator chains: even and odd k-steps)
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t kbase = smem_u32(kt);
    const int mi = lane >> 3, mr = lane & 7;
    if (!FP8) {
      const int krow = (mi & 1) * 8 + mr;
      uint32_t af[8][4];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) ldsm_x4(kbase + swz_bf16(krow, ks * 16 + (mi >> 1) * 8), af[ks]);
#pragma unroll
      for (int ks = 0; ks < 8; ks += 2) {
        mma_bf16(sc, af[ks], qf[ks][0], qf[ks][1]);
        mma_bf16(sd, af[ks + 1], qf[ks + 1][0], qf[ks + 1][1]);
      }
    } else {
      const int krow = (mi & 1) * 8 + mr;
      uint32_t x[4][4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) ldsm_x4(kbase + swz(krow, 2 * kk + (mi >> 1)), x[kk]);
      // a lane holds dims 4ti..4ti+3 of one key row per word: dims (4ti, 4ti+1)
      // feed k = (2ti, 2ti+1) and dims (4ti+2, 4ti+3) feed k = (2ti+8, 2ti+9)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t af[4] = {e4m3x2_lo(x[kk][0]), e4m3x2_lo(x[kk][1]), e4m3x2_hi(x[kk][0]), e4m3x2_hi(x[kk][1])};
        mma_f16(sc, af, qf[2 * kk][0], qf[2 * kk][1]);
        uint32_t ag[4] = {e4m3x2_lo(x[kk][2]), e4m3x2_lo(x[kk][3]), e4m3x2_hi(x[kk][2]), e4m3x2_hi(x[kk][3])};
        mma_f16(sd, ag, qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) sc[r] += sd[r];

    // ---- scores in log2 units, masked
    float s0 = sc[0] * qk0, s1 = sc[1] * qk1;
    float s2 = sc[2] * qk0, s3 = sc[3] * qk1;
    if (key0 + 15 > min_lim) {
      const int ka = key0 + gi, kb = ka + 8;
      s0 = ka <= lim0 ? s0 : -INFINITY;
      s1 = ka <= lim1 ? s1 : -INFINITY;
      s2 = kb <= lim0 ? s2 : -INFINITY;
      s3 = kb <= lim1 ? s3 : -INFINITY;
    }
    float t0 = fmaxf(s0, s2), t1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, off));
      t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, off));
    }
    const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
    if (__any_sync(kFull, n0 > m0 || n1 > m1)) {
      const float a0 = ex2(m0 - (n0 == -INFINITY ? 0.f : n0));
      const float a1 = ex2(m1 - (n1 == -INFINITY ? 0.f : n1));
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      l0 *= a0;
      l1 *= a1;
      m0 = n0;
      m1 = n1;
    }
    const float ms0 = m0 == -INFINITY ? 0.f : m0, ms1 = m1 == -INFINITY ? 0.f : m1;
    const float p0 = ex2(s0 - ms0), p1 = ex2(s1 - ms1), p2 = ex2(s2 - ms0), p3 = ex2(s3 - ms1);
    l0 += p0 + p2;
    l1 += p1 + p3;

    // ---- P^T into operand layout: keys on K, query rows on N
    const uint32_t pk0 = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
    const uint32_t pk1 = FP8 ? pack_f16(p2, p3) : pack_bf16(p2, p3);
    const uint32_t pb0 = movmatrix_t(pk0), pb1 = movmatrix_t(pk1);

    // ---- O^T += V^T . P^T
    const uint32_t vbase = smem_u32(vt);
    if (!FP8) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t af[4];
        ldsm_x4_t(vbase + swz_bf16((mi >> 1) * 8 + mr, mt * 16 + (mi & 1) * 8), af);
        mma_bf16(o[mt], af, pb0, pb1);
      }
    } else {
      const int vr = (mi & 1) * 8 + mr;
      // a lane's word holds keys (2ti, 2ti+1) x dims (2gi, 2gi+1) as bytes
      // (k, d), (k, d+1), (k+1, d), (k+1, d+1): regroup into one key pair per
      // dim, so MMA row gi <-> dim 2gi and row gi + 8 <-> dim 2gi + 1
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t x[4];
        ldsm_x4_t(vbase + swz(vr, 2 * cc + (mi >> 1)), x);
#pragma unroll
        for (int q = 0; q < 4; ++q) x[q] = prmt(x[q], 0u, 0x3120u);
        uint32_t af[4] = {e4m3x2_lo(x[0]), e4m3x2_hi(x[0]), e4m3x2_lo(x[1]), e4m3x2_hi(x[1])};
        mma_f16(o[2 * cc], af, pb0, pb1);
        uint32_t ag[4] = {e4m3x2_lo(x[2]), e4m3x2_hi(x[2]), e4m3x2_lo(x[3]), e4m3x2_hi(x[3])};
        mma_f16(o[2 * cc + 1], ag, pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + st));
  }

  // ---- warp totals of l over the 8 lanes sharing each row pair
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
  }
  if (lane == 0) atomicAdd(&misc[1], keys_scored);

  // ---- cross-warp merge through shared memory (its own area in the
  // four-stage form, else the drained ring)
  if (!C::SEP_MERGE) asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
  float* mo = C::SEP_MERGE ? reinterpret_cast<float*>(pt + C::NPROD * C::PT_CHUNK)
                           : reinterpret_cast<float*>(ring);
  float* mm = mo + C::NCW * 8 * C::MO_STRIDE;
  float* ml = mm + C::NCW * 8;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    int da, db;
    if (!FP8) {
      da = mt * 16 + gi;
      db = da + 8;
    } else {
      da = mt * 16 + 2 * gi;
      db = da + 1;
    }
    float* w0 = mo + (warp * 8 + 2 * ti) * C::MO_STRIDE;
    float* w1 = w0 + C::MO_STRIDE;
    w0[da] = o[mt][0];
    w1[da] = o[mt][1];
    w0[db] = o[mt][2];
    w1[db] = o[mt][3];
  }
  if (gi == 0) {
    mm[warp * 8 + 2 * ti] = m0;
    mm[warp * 8 + 2 * ti + 1] = m1;
    ml[warp * 8 + 2 * ti] = l0;
    ml[warp * 8 + 2 * ti + 1] = l1;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
  merge_and_store<FP8, HPI, NRG, NST>(a, tid, mo, mm, ml, b, h0, slot);

  // Fused combine: last-arriver merges, no waiting.  With S <= kBundle splits
  // the CTA that finishes last merges the group's S partials into the output.
  // With more, the splits form bundles of kBundle consecutive splits: the
  // last CTA of a bundle merges it in place into the bundle's first slot,
  // and the last bundle to finish merges the bundle partials into the output
  // (two reads of at most kBundle partials instead of one read of S).
  // Bundle tickets live after the group tickets, indexed by slot.
  int merged = 0;
  if (slot >= 0 && a.fused) {
    constexpr int kBundle = 8;
    float* sl = reinterpret_cast<float*>(ring) + C::NCW * 8 * C::MO_STRIDE + 2 * C::NCW * 8;
    const int slot0 = slot - split;
    const bool two_level = nsplit > kBundle;
    const int bslot = slot0 + (split / kBundle) * kBundle;
    const int bcount = min(kBundle, nsplit - (bslot - slot0));
    asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
    if (tid == 0)
      misc[0] = two_level ? (atom_add_acq_rel_gpu(a.tickets + a.n_groups + bslot, 1) == bcount - 1)
                          : (atom_add_acq_rel_gpu(a.tickets + group, 1) == nsplit - 1);
    asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
    if (misc[0] && !two_level) {
      merge_group<C::NCW * 32, HPI, NRG>(a, tid, b, h0, slot0, nsplit, 1, -1, sl);
      if (tid == 0) a.tickets[group] = 0;
      merged = 1;
    } else if (misc[0]) {
      merge_group<C::NCW * 32, HPI, NRG>(a, tid, b, h0, bslot, bcount, 1, bslot, sl);
      if (tid == 0) a.tickets[a.n_groups + bslot] = 0;
      merged = 2;
      const int nb = (nsplit + kBundle - 1) / kBundle;
      asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
      if (tid == 0) misc[0] = (atom_add_acq_rel_gpu(a.tickets + group, 1) == nb - 1);
      asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
      if (misc[0]) {
        merge_group<C::NCW * 32, HPI, NRG>(a, tid, b, h0, slot0, nb, kBundle, -1, sl);
        if (tid == 0) a.tickets[group] = 0;
        merged = 3;
      }
    }
  }
  if (tid == 0) {
    int32_t* lg = a.cta_log + size_t(blockIdx.x) * kLogFields;
    lg[0] = p0;
    lg[1] = p1;
    lg[2] = misc[1];
    lg[3] = merged;
  }
}

// Copies keys [0, n_keys) of one KV head through the block table with the
// same tensor-map boxes and swizzled shared-memory addressing as the decode
// kernel.  One CTA of 128 threads; tiles are loaded one at a time.
template <bool FP8>
__global__ void __launch_bounds__(128) gather_debug_kernel(const __grid_constant__ CUtensorMap tm,
                                                           const int32_t* table_row, int h_kv,
                                                           int P, int n_keys, uint8_t* dst,
                                                           int32_t* status) {
  constexpr int KT = Gqa<FP8, 1>::KT_BYTES;
  __shared__ __align__(1024) uint8_t tile[KT];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int n_tiles = (n_keys + 15) / 16;
  for (int i = 0; i < n_tiles; ++i) {
    const int key0 = i * 16;
    if (threadIdx.x == 0) {
      const int ph = table_row[key0 / P];
      mbar_arrive_expect_tx(smem_u32(&bar), KT);
      // the decode kernel's maps: (dims, key in page, [column half,] head, page)
      if (FP8)
        tma_load_4d(smem_u32(tile), &tm, smem_u32(&bar), 0, key0 % P, h_kv, ph);
      else
        tma_load_5d(smem_u32(tile), &tm, smem_u32(&bar), 0, key0 % P, 0, h_kv, ph);
    }
    if (!__syncthreads_and(mbar_wait(smem_u32(&bar), i & 1))) {
      if (threadIdx.x == 0 && status) atomicOr(status, SPLITKV_DEVERR_TIMEOUT);
      // one more bounded wait so the copy is not left writing into freed smem
      if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), i & 1);
      __syncthreads();
      return;
    }
    // 16 rows x 16 chunks (bf16) or 8 chunks (fp8) of 16 bytes each
    constexpr int CH = FP8 ? 8 : 16;
    for (int x = threadIdx.x; x < 16 * CH; x += blockDim.x) {
      const int r = x / CH, c = x % CH;
      if (key0 + r >= n_keys) continue;
      const uint32_t off = FP8 ? swz(r, c) : swz_bf16(r, c * 8);
      *reinterpret_cast<uint4*>(dst + (size_t(key0 + r) * CH + c) * 16) =
          *reinterpret_cast<const uint4*>(tile + off);
    }
    __syncthreads();
  }
}

}  // namespace

namespace {

// One-time shared-memory opt-in of an instantiation, then a launch with
// programmatic dependent launch: the kernel's prologue may overlap the tail
// of the previous kernel on the stream; it waits (griddepcontrol.wait)
// before touching anything that kernel could have written.
template <bool FP8, int HPI, int NRG = 1, int NST = 2>
cudaError_t launch_gqa_t(const DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                         cudaStream_t s) {
  using C = Gqa<FP8, HPI, NRG, NST>;
  // The shared-memory opt-in is a per-process attribute: set it on first use only.
  static cudaError_t attr = cudaFuncSetAttribute(
      gqa_splitkv_kernel<FP8, HPI, NRG, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_items, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = la;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_splitkv_kernel<FP8, HPI, NRG, NST>, a, mk, mv);
}

constexpr int kDeepStages = 4;

// Picks the instantiation for the query rows per KV head, the cache type and
// the KV heads per item.
template <int NST>
cudaError_t launch_gqa_nst(const DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                           bool fp8, cudaStream_t s) {
  if (a.T * a.G > 16) {  // 17..32 query rows per KV head: four row groups
    if (a.hpi != 1) return cudaErrorInvalidValue;
    return fp8 ? launch_gqa_t<true, 1, 4, NST>(a, mk, mv, s)
               : launch_gqa_t<false, 1, 4, NST>(a, mk, mv, s);
  }
  if (a.T * a.G > 8) {  // 9..16 query rows per KV head: two row groups
    if (fp8 && a.hpi == 2) return launch_gqa_t<true, 2, 2, NST>(a, mk, mv, s);
    if (a.hpi != 1) return cudaErrorInvalidValue;
    return fp8 ? launch_gqa_t<true, 1, 2, NST>(a, mk, mv, s)
               : launch_gqa_t<false, 1, 2, NST>(a, mk, mv, s);
  }
  if (!fp8) return a.hpi == 1 ? launch_gqa_t<false, 1, 1, NST>(a, mk, mv, s) : cudaErrorInvalidValue;
  switch (a.hpi) {
    case 1: return launch_gqa_t<true, 1, 1, NST>(a, mk, mv, s);
    case 2: return launch_gqa_t<true, 2, 1, NST>(a, mk, mv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gqa(const DecodeArgs& a, const TmaDesc& tk, const TmaDesc& tv, bool fp8,
                       void* stream) {
  const CUtensorMap& mk = *reinterpret_cast<const CUtensorMap*>(&tk);
  const CUtensorMap& mv = *reinterpret_cast<const CUtensorMap*>(&tv);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.n_items == 0) return cudaSuccess;
  // A grid of at most one CTA per SM does not share SMs, so its CTAs take the
  // four-stage ring (more bytes in flight per SM); a larger grid keeps the
  // two-stage ring that lets kGqaCtasPerSm CTAs share each SM.
  if (a.deep_ring) return launch_gqa_nst<kDeepStages>(a, mk, mv, fp8, s);
  return launch_gqa_nst<2>(a, mk, mv, fp8, s);
}

cudaError_t launch_debug_gather(const TmaDesc& t, bool fp8, const int32_t* table_row,
                                int32_t h_kv, int32_t P, int32_t n_keys, void* dst, void* stream) {
  const CUtensorMap& m = *reinterpret_cast<const CUtensorMap*>(&t);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = nullptr;
  if (fp8)
    gather_debug_kernel<true><<<1, 128, 0, s>>>(m, table_row, h_kv, P, n_keys,
                                                static_cast<uint8_t*>(dst), status);
  else
    gather_debug_kernel<false><<<1, 128, 0, s>>>(m, table_row, h_kv, P, n_keys,
                                                 static_cast<uint8_t*>(dst), status);
  return cudaGetLastError();
}

}  // namespace splitkv
