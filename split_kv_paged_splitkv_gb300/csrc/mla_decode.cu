// Split-KV partial attention for the MLA-style decode (128 query heads of up
// to 16 tokens sharing one 576-wide latent KV head, V = its first 512
// columns), on the 5th-generation tensor cores (tcgen05, accumulators in
// TMEM).  This is the dense case of the split-KV decode: "Shipped: 484.5
// tok/s on one GB300 ...", table "What shipped" (MLA decode of one request at
// 6 tokens per step, split 4 ways), with the per-split partial and the
// log-sum-exp merge of "vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48%
// Slower", section "What SplitKV is trying to do".
//
// Work: two CTAs per (work item, query token), one per half h of the 512 V
// columns.  The 128 heads of the token are the MMA rows (M = 128); a
// 128 x 512 fp32 output tile would fill all of TMEM, hence the V halves.
// Each CTA computes the full 576-wide scores of its token itself, so the
// two CTAs never exchange anything (on this part, moving a 64-key block of
// fp32 partial scores between the CTAs of a cluster took about three times
// as long as computing the scores).
//
// The nine 64-column chunks of a key row split by where the matching query
// chunk lives.  Four score-only chunks pair with query chunks held in TMEM;
// the CTA's four V chunks (columns [256 h, 256 h + 256)) and the rope chunk
// pair with query chunks in shared memory.  They stream through two rings
// of two slots, each fed by its own producer warp:
//   N ring: the four TMEM-paired chunks of a block, released as soon as the
//           block's score MMAs have read them;
//   V ring: the V chunks and the rope chunk, released after the block's PV
//           (the score product reads them last).
// S is double-buffered; P is written over the first 32 columns of its own
// S buffer, so the scores of block j + 1 accumulate while the softmax warps
// work on block j, and the scores of block j + 2 wait only for PV(j).
// Keys stream in blocks of 64.  A page of 16 or 32 keys fills a block chunk
// with 4 or 2 TMA boxes of one page each; a page of 64 keys or a multiple of
// 64 holds whole blocks (the split's first key is then a multiple of 64).
// Per 64-key block:
//   1. S_b = Q . K^T      (tcgen05, M=128 N=64 K=576, b = j % 2)
//   2. softmax warps: online softmax with a lazy reference maximum (O is
//      rescaled only when a row maximum grows by more than 2^8, after PV(j-1)
//      has finished); P (bf16) goes into S_b
//   3. O_h += P . V_h      (tcgen05, M=128 N=256 K=64, P from TMEM)
// TMEM columns: S_0 [0, 64), S_1 [64, 128), Q's four TMEM chunks [128, 256),
// O_h [256, 512).  Warp roles: warp 0 N-ring producer and TMEM owner, warp 1
// MMA issuer (whole warps run the issue loops; one elected lane issues),
// warps 2-5 load Q, then softmax and epilogue (thread = query head = TMEM
// lane), warp 6 V-ring producer.
//
// FP8 (an e4m3 latent cache with a per-tensor scale, V in its first 512
// columns): TMA lands each block's e4m3 rows in the upper half of the ring
// slot, four converter warps turn them into f16 over the whole slot (the
// hardware e4m3 -> f16 pair conversion is exact), and the MMAs run on f16:
// the query rows are scaled by a power of two each into f16's range (exact;
// the row's score scale takes the inverse), P is packed as f16, and the
// cache scale multiplies the scores and the output once.  "Xqa decode
// kernels", section "Purpose": an FP8 KV cache read with 16-bit queries.
//
// Separate V (SEPV: a cache whose V rows are their own 512-wide tensor, not
// the first columns of the key rows): the V-ring slot of block j first holds
// the five key chunks as above; once the score MMAs of block j have read
// them, warp 7 loads block j's V half over the first four of them, and PV(j)
// waits for that load.  Shared memory and TMEM are laid out as for the
// shared latent row; each V-ring slot is filled twice per use.
#include <cuda_runtime.h>

#include "fixed_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace splitkv {
namespace {

using namespace ptx;

struct Mla {
  static constexpr int DK = 576, DV = 512;
  static constexpr int ROWS = 128;          // query heads of one token
  static constexpr int BK = 64;             // keys per block
  static constexpr int NN = 4;              // N-ring chunks (query chunk in TMEM)
  static constexpr int NV = 4;              // V chunks of this CTA's half
  static constexpr int NX = NV + 1;         // V-ring chunks: the V chunks and the rope chunk
  static constexpr int K_CH = BK * 128;     // one key chunk: 64 keys x 64 bf16 = 8 KB
  static constexpr int Q_CH = ROWS * 128;   // one Q chunk: 128 rows x 64 bf16 = 16 KB
  static constexpr int NST = 2;             // slots per ring
  static constexpr int N_SLOT = NN * K_CH;
  static constexpr int V_SLOT = NX * K_CH;
  static constexpr int OFF_Q = 0;                       // Q's V-ring chunks (K-major, swizzled)
  static constexpr int OFF_N = OFF_Q + NX * Q_CH;       // N ring
  static constexpr int OFF_V = OFF_N + NST * N_SLOT;    // V ring
  static constexpr int OFF_BAR = OFF_V + NST * V_SLOT;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr int THREADS = 224;       // 256 with separate V (warp 7 loads V),
                                            // 352 with FP8 (warps 7-10 convert)
  static constexpr int CONV_WARP0 = 7;      // FP8: first converter warp
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 0, Q_COL = 128, O_COL = 256;  // S_b at S_COL + 64 b
  static constexpr float RESCALE_LOG2 = 8.f;  // lazy maximum: rescale when it grows by > 2^8
};
static_assert(Mla::Q_COL + Mla::NN * 32 <= Mla::O_COL, "Q overlaps O in TMEM");
static_assert(Mla::S_COL + 2 * 64 <= Mla::Q_COL, "S buffers overlap Q in TMEM");
static_assert(Mla::SMEM <= 227 * 1024, "shared memory budget");

constexpr float kLn2m = 0.6931471805599453f;

// Where a CTA gave up on a timed-out wait, for the per-CTA log: the first
// site recorded wins.  (role << 24) | (x << 12) | y with role 1 the N-ring
// producer, 2 the V-ring producer, 3 the V producer of a separate V tensor
// (y = block), 4 the MMA issuer (bit 23: the N-ring half of QK(x) issued;
// x = next QK block, y = next PV block), 5 the softmax warps (x = 1 waiting
// for S, 2 for PV(y - 1) before a rescale; y = block), 6 the epilogue.
__device__ __forceinline__ void note_abort(int* site, int code) { atomicCAS(site, 0, code); }

// Barrier slots (8 bytes each) after OFF_BAR.
enum {
  B_QFULL = 0,                      // Q written to TMEM and shared memory (128 threads)
  B_NFULL = 1,                      // [NST]
  B_NEMPTY = B_NFULL + Mla::NST,    // [NST]
  B_VFULL = B_NEMPTY + Mla::NST,    // [NST]
  B_VEMPTY = B_VFULL + Mla::NST,    // [NST]
  B_SFULL = B_VEMPTY + Mla::NST,    // [2] S_b complete
  B_PFULL = B_SFULL + 2,            // [2] P written over S_b (128); one barrier per
                                    // buffer, so no barrier runs two phases ahead
  B_PFREE = B_PFULL + 2,            // [2] PV(j) done for j % 2 = b: P read out of S_b,
                                    // O stable.  One barrier per buffer: QK(j) waits
                                    // for PV(j - 2), and with a single barrier PV(j - 2)
                                    // and PV(j - 1) could both complete before that test,
                                    // leaving the barrier two phases ahead of it
  B_DONE = B_PFREE + 2,             // every MMA this CTA issued has completed
  B_XKDONE,                         // [NST] separate V: the score MMAs have read the
                                    // key chunks of V slot s
  B_VDATA = B_XKDONE + Mla::NST,    // [NST] separate V: V rows landed in V slot s
  B_NCONV = B_VDATA + Mla::NST,     // [NST] FP8: N slot s converted to f16 (4 warps)
  B_VCONV = B_NCONV + Mla::NST,     // [NST] FP8: V slot s converted to f16 (4 warps)
  B_COUNT = B_VCONV + Mla::NST
};
static_assert(B_COUNT * 8 + 12 <= 256, "barrier area (then the TMEM slot and two flags)");

// Column chunk (of the nine) in N-ring slot chunk i / V-ring slot chunk k of half h.
__device__ __forceinline__ int n_chunk(int h, int i) { return h == 0 ? 4 + i : i; }
__device__ __forceinline__ int v_chunk(int h, int k) { return k < 4 ? 4 * h + k : 8; }

// FP8: converts the e4m3 rows TMA left in the upper half of a ring slot
// (NCH chunks of [64 rows][64 B], one byte per element) into the f16 chunks
// the MMAs read ([64 rows][128 B] each, 128-byte swizzle) over the whole slot.
// Run by the 128 converter threads (ct = 0..127): each first reads all its
// staged 16-byte segments, the converters then meet at named barrier 2 (the
// f16 rows of the first chunks overwrite the staging area of later ones), and
// each writes its segments as f16, 16 elements -> two 16-byte pieces.
template <int NCH>
__device__ __forceinline__ void convert_slot(uint8_t* slot, int ct) {
  constexpr int PER = NCH * 64 * 4 / 128;  // 16-byte staged segments per thread
  const uint8_t* stage = slot + NCH * Mla::K_CH / 2;
  uint4 x[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) x[i] = *reinterpret_cast<const uint4*>(stage + (i * 128 + ct) * 16);
  asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int g = i * 128 + ct;  // segment: chunk g / 256, row (g / 4) % 64, columns 16 (g % 4) ..
    const int k = g >> 8, r = (g >> 2) & 63, c4 = g & 3;
    uint8_t* row = slot + k * Mla::K_CH + r * 128;
    const uint4 lo = make_uint4(e4m3x2_lo(x[i].x), e4m3x2_hi(x[i].x), e4m3x2_lo(x[i].y),
                                e4m3x2_hi(x[i].y));
    const uint4 hi = make_uint4(e4m3x2_lo(x[i].z), e4m3x2_hi(x[i].z), e4m3x2_lo(x[i].w),
                                e4m3x2_hi(x[i].w));
    *reinterpret_cast<uint4*>(row + (((2 * c4) ^ (r & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((2 * c4 + 1) ^ (r & 7)) << 4)) = hi;
  }
}

// Page walk of a producer warp over its split's 64-key blocks.  Pages of
// 64 keys or a multiple of 64 hold whole blocks: a block is one box at row
// offset `off` of page `pg`.  Pages of 16 or 32 keys (SMALLP) take 4 or 2
// boxes per block chunk, one page each.  The warp holds the physical ids of
// pages chunk0 + lane (0 past the split's last page p1, whose keys are
// masked anyway) and refreshes them when a block reaches past that window.
// No division: the walk advances by whole pages or by 64 rows.
template <bool SMALLP>
struct PageWalk {
  static constexpr int NB = SMALLP ? 4 : 1;  // boxes per block chunk, at most
  int pg, off = 0, chunk0 = -32, phys = 0;

  __device__ __forceinline__ explicit PageWalk(int p0) : pg(p0) {}

  // First rows (the MLA cache has one KV head) of the current block's boxes;
  // with pages of 32 keys y[2], y[3] repeat y[1].  `report` flags
  // out-of-range page ids.
  __device__ __forceinline__ void rows(const DecodeArgs& a, const int32_t* trow, int p1, int lane,
                                       bool report, int (&y)[NB]) {
    const int nb = SMALLP ? Mla::BK / a.P : 1;
    if (pg + nb > chunk0 + 32) {
      chunk0 = pg;
      const int my = chunk0 + lane;
      phys = 0;
      if (my < p1) {
        phys = __ldg(trow + my);
        if (phys < 0 || phys >= a.num_pages) {
          if (report) atomicOr(a.status, SPLITKV_DEVERR_PAGE);
          phys = 0;
        }
      }
    }
    if (SMALLP) {
#pragma unroll
      for (int r = 0; r < NB; ++r) y[r] = __shfl_sync(kFull, phys, pg + min(r, nb - 1) - chunk0) * a.P;
    } else {
      y[0] = __shfl_sync(kFull, phys, pg - chunk0) * a.P + off;
    }
  }

  __device__ __forceinline__ void next(int P) {
    if (SMALLP) {
      pg += Mla::BK / P;
    } else if ((off += Mla::BK) == P) {
      ++pg;
      off = 0;
    }
  }
};

template <bool SEPV, bool SMALLP, bool FP8>
__global__ void __launch_bounds__(SEPV ? Mla::THREADS + 32 : (FP8 ? Mla::THREADS + 128 : Mla::THREADS), 1)
    mla_splitkv_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv) {
  static_assert(!(SEPV && FP8), "FP8 latent caches hold V in the key rows");
  using C = Mla;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* conv_abort = abort_flag + 1;  // FP8: a converter warp gave up
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x & 1;  // V half: columns [256 h, 256 h + 256)
  const int pair = blockIdx.x >> 1;
  const int item = pair / a.T;
  const int t = pair - item * a.T;

  // A capacity plan's item is derived from the device lengths (read after the
  // dependency wait); a host plan's comes from the uploaded work list.
  int32_t it[SPLITKV_ITEM_FIELDS];
  int L_fixed = 0;
  if (a.fixed) {
    wait_prerequisites();
    bool bad;
    fixed_item(a.fx, item, it, &L_fixed, &bad);
    // one CTA of the item (token 0, V half 0) writes its group's entry
    if (threadIdx.x == 0 && blockIdx.x % (2 * a.T) == 0)
      fixed_write_group(a.fx, const_cast<int32_t*>(a.groups), it);
  } else {
    const int32_t* src = a.items + size_t(item) * SPLITKV_ITEM_FIELDS;
#pragma unroll
    for (int k = 0; k < SPLITKV_ITEM_FIELDS; ++k) it[k] = src[k];
  }
  const int b = it[SPLITKV_ITEM_B];
  const int p0 = it[SPLITKV_ITEM_PAGE0], p1 = it[SPLITKV_ITEM_PAGE1];
  const int slot = it[SPLITKV_ITEM_SLOT];
  if (it[SPLITKV_ITEM_NSPLIT] == 0) {  // a capacity item the current lengths leave unused
    if (threadIdx.x == 0) {
      int32_t* lg = a.cta_log + size_t(blockIdx.x) * kLogFields;
      lg[0] = p0;
      lg[1] = p1;
      lg[2] = 0;
      lg[3] = 0;
    }
    return;
  }

  // ---- prologue (shared memory, TMEM, tensor map, work list only)
  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 128);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(B_NFULL + s), 1);
      mbar_init(bar(B_NEMPTY + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_PFULL + 1), 128);
    mbar_init(bar(B_PFREE), 1);
    mbar_init(bar(B_PFREE + 1), 1);
    mbar_init(bar(B_DONE), 1);
    if (SEPV) {
      for (int s = 0; s < C::NST; ++s) {
        mbar_init(bar(B_XKDONE + s), 1);
        mbar_init(bar(B_VDATA + s), 1);
      }
    }
    if (FP8) {
      for (int s = 0; s < C::NST; ++s) {
        mbar_init(bar(B_NCONV + s), 4);
        mbar_init(bar(B_VCONV + s), 4);
      }
    }
    *abort_flag = 0;
    *conv_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    if (lane == 0) {
      prefetch_tmap(&tk);
      if (SEPV) prefetch_tmap(&tv);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // plan's sequence length (uploaded, never written by a kernel): read before the wait
  const int L = a.fixed ? L_fixed : a.plan_lens[b];
  const int k_begin = p0 * a.P;
  const int k_end = min(p1 * a.P, L);
  const int nblk = k_end > k_begin ? (k_end - k_begin + C::BK - 1) / C::BK : 0;
  // last key this CTA scores: visible to its token and inside the split (a
  // split of 16- or 32-key pages may end inside a 64-key block; with larger
  // pages a split ends at a block end or at L)
  const int lim = SMALLP ? min(L - a.T + t, k_end - 1) : L - a.T + t;
  launch_dependents();
  wait_prerequisites();
  if (threadIdx.x == 0 && h == 0 && t == 0 && a.seq_lens[b] != L)
    atomicOr(a.status, SPLITKV_DEVERR_SEQLEN);

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ producers
    // Warp 0 loads the score-only chunks of block j into N slot j % NST (free
    // once the score MMAs of block j - NST are done); warp 6 loads the V
    // chunks into V slot j % NST (free once PV(j - NST) is done).
    const bool vring = warp == 6;
    const int nchk = vring ? C::NX : C::NN;
    const uint32_t full0 = vring ? B_VFULL : B_NFULL, empty0 = vring ? B_VEMPTY : B_NEMPTY;
    const int slot_bytes = vring ? C::V_SLOT : C::N_SLOT;
    uint8_t* ring = sm + (vring ? C::OFF_V : C::OFF_N);
    const int32_t* trow = a.block_table + size_t(b) * a.max_pages;
    bool ok = true;
    int issued = 0;
    PageWalk<SMALLP> walk(p0);
    const int br = SMALLP ? a.P : C::BK;  // rows per box
    for (int j = 0; j < nblk && ok; ++j, walk.next(a.P)) {
      int yr[PageWalk<SMALLP>::NB];
      walk.rows(a, trow, p1, lane, true, yr);
      const int st = j % C::NST;
      if (j >= C::NST) ok = __all_sync(kFull, mbar_wait(bar(empty0 + st), ((j / C::NST) - 1) & 1));
      if (!ok) break;
      // bf16: the chunks straight into the slot; FP8: the e4m3 rows (64 bytes
      // each) into its upper half, for the converter warps
      mbar_arrive_expect_tx_warp(bar(full0 + st), FP8 ? slot_bytes / 2 : slot_bytes);
#pragma unroll
      for (int r = 0; r < PageWalk<SMALLP>::NB; ++r) {
        if (r * br >= C::BK) break;
        for (int k = 0; k < nchk; ++k) {
          uint8_t* dst = FP8 ? ring + st * slot_bytes + slot_bytes / 2 + k * (C::K_CH / 2) + r * br * 64
                             : ring + st * slot_bytes + k * C::K_CH + r * br * 128;
          tma_load_2d_warp(smem_u32(dst), &tk, bar(full0 + st),
                           (vring ? v_chunk(h, k) : n_chunk(h, k)) * 64, yr[r]);
        }
      }
      if (!vring) {
        // The V-ring slot of block j is refilled only once PV(j - 2) is done,
        // a few hundred cycles before the score MMAs need it, while this ring
        // is refilled some 3,000 cycles earlier: warm L2 with block j's
        // V-ring rows (and, with a separate V tensor, its V rows) now, so that
        // copy hits L2 instead of waiting out a DRAM round trip.
#pragma unroll
        for (int r = 0; r < PageWalk<SMALLP>::NB; ++r) {
          if (r * br >= C::BK) break;
          for (int k = 0; k < C::NX; ++k) tma_prefetch_2d_warp(&tk, v_chunk(h, k) * 64, yr[r]);
          if (SEPV)
            for (int k = 0; k < C::NV; ++k) tma_prefetch_2d_warp(&tv, (4 * h + k) * 64, yr[r]);
        }
      }
      issued = j + 1;
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      note_abort(abort_flag, ((vring ? 2 : 1) << 24) | (issued & 0xfff));
    }
    // stay until every issued copy has landed
    if (lane == 0) {
      for (int st = 0; st < C::NST && st < issued; ++st) {
        const int last = st + C::NST * ((issued - 1 - st) / C::NST);
        if (!mbar_wait(bar(full0 + st), (last / C::NST) & 1)) break;
      }
    }
  } else if (SEPV && warp == 7) {
    // ----------------------------------------------------- V producer (SEPV)
    // Block j's V half into the first NV chunks of V slot j % NST, once the
    // score MMAs of block j have read the key chunks there.
    const int32_t* trow = a.block_table + size_t(b) * a.max_pages;
    bool ok = true;
    int issued = 0;
    PageWalk<SMALLP> walk(p0);
    const int br = SMALLP ? a.P : C::BK;
    for (int j = 0; j < nblk && ok; ++j, walk.next(a.P)) {
      int yr[PageWalk<SMALLP>::NB];  // (out-of-range page ids are reported by the key producer)
      walk.rows(a, trow, p1, lane, false, yr);
      const int st = j % C::NST;
      ok = __all_sync(kFull, mbar_wait(bar(B_XKDONE + st), (j / C::NST) & 1));
      if (!ok) break;
      mbar_arrive_expect_tx_warp(bar(B_VDATA + st), C::NV * C::K_CH);
#pragma unroll
      for (int r = 0; r < PageWalk<SMALLP>::NB; ++r) {
        if (r * br >= C::BK) break;
        for (int k = 0; k < C::NV; ++k)
          tma_load_2d_warp(smem_u32(sm + C::OFF_V + st * C::V_SLOT + k * C::K_CH + r * br * 128),
                           &tv, bar(B_VDATA + st), (4 * h + k) * 64, yr[r]);
      }
      issued = j + 1;
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      note_abort(abort_flag, (3 << 24) | (issued & 0xfff));
    }
    // stay until every issued copy has landed
    if (lane == 0) {
      for (int st = 0; st < C::NST && st < issued; ++st) {
        const int last = st + C::NST * ((issued - 1 - st) / C::NST);
        if (!mbar_wait(bar(B_VDATA + st), (last / C::NST) & 1)) break;
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // Issue order follows readiness: PV(jp) as soon as P(jp) is in TMEM (and,
    // with separate V, its V rows have landed; it frees a V slot); else the
    // next half of QK(jq) into S_{jq % 2}: the
    // N-ring chunks once their slot landed and PV(jq - 2) has read the P
    // that shares that S buffer, then the V-ring chunks once their slot landed.
    const uint32_t idesc_qk = FP8 ? umma_idesc_f16(128, 64, 0, 0) : umma_idesc_bf16(128, 64, 0, 0);
    const uint32_t idesc_pv = FP8 ? umma_idesc_f16(128, 256, 0, 1) : umma_idesc_bf16(128, 256, 0, 1);
    // FP8: a slot is ready for the MMAs once converted, not when its TMA lands
    const uint32_t nready0 = FP8 ? B_NCONV : B_NFULL, vready0 = FP8 ? B_VCONV : B_VFULL;
    bool ok = __all_sync(kFull, mbar_wait(bar(B_QFULL), 0));
    int jq = 0, jp = 0;
    bool qk_half = false;  // the N-ring half of QK(jq) has been issued
    long long t_idle = clock64();
    while (ok && jp < nblk) {
      if (jp < jq &&
          __shfl_sync(kFull,
                      mbar_test(bar(B_PFULL + (jp & 1)), (jp >> 1) & 1) &&
                          (!SEPV || mbar_test(bar(B_VDATA + jp % C::NST), (jp / C::NST) & 1)),
                      0)) {  // O_h += P.V
        const int vs = jp % C::NST;
        tc_fence_after();
        uint8_t* vst = sm + C::OFF_V + vs * C::V_SLOT;  // its first NV chunks hold V_h
        const int valid = min(C::BK, k_end - (k_begin + jp * C::BK));
        if (valid < C::BK) {
          // key slots past the last key may hold anything (even NaN): zero their
          // V rows so that 0 * V stays 0 in the PV product (QK(jp) is complete)
          for (int x = lane; x < (C::BK - valid) * 8 * C::NV; x += 32) {
            const int r = valid + (x >> 5), ch = (x >> 3) & 3, c16 = x & 7;
            *reinterpret_cast<uint4*>(vst + ch * C::K_CH + r * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        const uint32_t pcol = C::S_COL + uint32_t(64 * (jp & 1));  // P over S_{jp % 2}
#pragma unroll
        for (int kin = 0; kin < 4; ++kin) {
          const uint64_t bd = umma_desc(smem_u32(vst) + kin * 16 * 128, C::K_CH, 1024, 2);
          umma_bf16_ta_warp(tmem + C::O_COL, tmem + pcol + uint32_t(kin * 8), bd, idesc_pv,
                            (jp | kin) != 0);
        }
        umma_commit_warp(bar(B_VEMPTY + vs));
        umma_commit_warp(bar(B_PFREE + (jp & 1)));
        __syncwarp();
        ++jp;
        t_idle = clock64();
        continue;
      }
      const int qs = jq % C::NST;
      const uint32_t scol = C::S_COL + uint32_t(64 * (jq & 1));
      if (jq < nblk && !qk_half) {  // N-ring chunks of QK(jq), Q from TMEM
        const bool rdy = __shfl_sync(
            kFull,
            mbar_test(bar(nready0 + qs), (jq / C::NST) & 1) &&
                (jq < 2 || mbar_test(bar(B_PFREE + (jq & 1)), ((jq - 2) >> 1) & 1)),
            0);
        if (rdy) {
          tc_fence_after();
          const uint32_t nst = smem_u32(sm + C::OFF_N + qs * C::N_SLOT);
#pragma unroll
          for (int i = 0; i < C::NN; ++i)
#pragma unroll
            for (int kin = 0; kin < 4; ++kin)
              umma_bf16_ta_warp(tmem + scol, tmem + C::Q_COL + uint32_t(i * 32 + kin * 8),
                                umma_desc(nst + i * C::K_CH + kin * 32, 16, 1024, 2), idesc_qk,
                                (i | kin) != 0);
          umma_commit_warp(bar(B_NEMPTY + qs));
          __syncwarp();
          qk_half = true;
          t_idle = clock64();
          continue;
        }
      } else if (jq < nblk) {  // V-ring chunks of QK(jq), Q from shared memory
        if (__shfl_sync(kFull, mbar_test(bar(vready0 + qs), (jq / C::NST) & 1), 0)) {
          tc_fence_after();
          const uint32_t vst = smem_u32(sm + C::OFF_V + qs * C::V_SLOT);
#pragma unroll
          for (int k = 0; k < C::NX; ++k)
#pragma unroll
            for (int kin = 0; kin < 4; ++kin)
              umma_bf16_warp(tmem + scol,
                             umma_desc(smem_u32(sm + C::OFF_Q + k * C::Q_CH) + kin * 32, 16, 1024, 2),
                             umma_desc(vst + k * C::K_CH + kin * 32, 16, 1024, 2), idesc_qk, 1u);
          umma_commit_warp(bar(B_SFULL + (jq & 1)));
          if (SEPV) umma_commit_warp(bar(B_XKDONE + qs));  // its key chunks may be overwritten
          __syncwarp();
          ++jq;
          qk_half = false;
          t_idle = clock64();
          continue;
        }
      }
      __nanosleep(32);  // leave issue slots to the softmax warp on this SM sub-partition
      ok = __shfl_sync(kFull, clock64() - t_idle < kWaitTimeoutCycles, 0);
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      note_abort(abort_flag, (4 << 24) | (qk_half ? 1 << 23 : 0) | ((jq & 0x7ff) << 12) | (jp & 0xfff));
    }
    // every MMA issued above completes before TMEM can be released
    umma_commit_warp(bar(B_DONE));
    __syncwarp();
    mbar_wait(bar(B_DONE), 0);
  } else if (FP8 && warp >= C::CONV_WARP0) {
    // ----------------------------------------------------- converters (FP8)
    // Per block j: N slot j % NST, then V slot j % NST, each once its e4m3
    // rows have landed.  A warp whose wait timed out raises conv_abort before
    // the next named barrier, after which all four warps leave together (a
    // named barrier has no timeout, so no warp may skip one alone).
    const int ct = threadIdx.x - C::CONV_WARP0 * 32;
    int done = 0;
    bool aborted = false;
    for (int j = 0; j < nblk && !aborted; ++j) {
      const int st = j % C::NST;
      for (int rg = 0; rg < 2; ++rg) {
        const bool ok = __all_sync(kFull, mbar_wait(bar((rg ? B_VFULL : B_NFULL) + st), (j / C::NST) & 1));
        if (!ok && lane == 0) *conv_abort = 1;
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (*conv_abort) {
          aborted = true;
          break;
        }
        if (rg == 0)
          convert_slot<C::NN>(sm + C::OFF_N + st * C::N_SLOT, ct);
        else
          convert_slot<C::NX>(sm + C::OFF_V + st * C::V_SLOT, ct);
        // order the f16 writes before the tensor cores' reads (and the slot's
        // next TMA refill)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar((rg ? B_VCONV : B_NCONV) + st));
      }
      done = j + 1;
    }
    if (aborted && ct == 0) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      note_abort(abort_flag, (7 << 24) | (done & 0xfff));
    }
  } else {
    // -------------------------------------------------------------- softmax warps
    const int g = warp & 3;          // TMEM lane group of this warp
    const int r = g * 32 + lane;     // query head = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(g * 32) << 16);

    // Q row r: its N-ring chunks -> TMEM (32-bit column c of a chunk holds
    // dims 2c, 2c + 1, the even one in the low half: the A-from-TMEM layout);
    // its V-ring chunks -> shared memory, 128-byte swizzled K-major rows
    // scores -> log2 units for this row (FP8: times the inverse of the
    // power of two the row's f16 query was scaled by)
    float sl2 = a.qk_scale_log2;
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                         ((size_t(b) * a.T + t) * a.Hq + r) * C::DK);
      // FP8: the f16 products need f16 queries, whose range is far narrower
      // than bf16's; the row is scaled by 2^k so that its largest component
      // lies in [2^14, 2^15) (exact, and every component rounds to f16
      // without loss unless it is below 2^-29 of the row maximum)
      float up = 1.f;
      if (FP8) {
        float amax = 0.f;
#pragma unroll 4
        for (int v = 0; v < C::DK / 8; ++v) {
          const uint4 x = __ldg(qrow + v);
          const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[e] << 16)),
                                     fabsf(__uint_as_float(wv[e] & 0xffff0000u))));
        }
        int k = 0;
        if (amax > 0.f) k = min(126, max(-113, 14 - (int((__float_as_uint(amax) >> 23) & 0xff) - 127)));
        up = __uint_as_float(uint32_t(127 + k) << 23);
        sl2 *= __uint_as_float(uint32_t(127 - k) << 23);
      }
      // bf16 pair -> f16 pair times `up` (FP8), or the bf16 pair itself
      auto cvt = [&](uint32_t w) -> uint32_t {
        if (!FP8) return w;
        return pack_f16(__uint_as_float(w << 16) * up, __uint_as_float(w & 0xffff0000u) * up);
      };
#pragma unroll 1
      for (int i = 0; i < C::NN; ++i) {
        const uint4* src = qrow + n_chunk(h, i) * 8;
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = __ldg(src + v);
          w[4 * v] = cvt(x.x);
          w[4 * v + 1] = cvt(x.y);
          w[4 * v + 2] = cvt(x.z);
          w[4 * v + 3] = cvt(x.w);
        }
        tmem_st32u(lane_base + C::Q_COL + uint32_t(i * 32), w);
      }
#pragma unroll 1
      for (int k = 0; k < C::NX; ++k) {
        const uint4* src = qrow + v_chunk(h, k) * 8;
        uint8_t* dst = sm + C::OFF_Q + k * C::Q_CH + r * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = __ldg(src + v);
          *reinterpret_cast<uint4*>(dst + ((v ^ (r & 7)) << 4)) =
              make_uint4(cvt(x.x), cvt(x.y), cvt(x.z), cvt(x.w));
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_QFULL));
    }

    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    int fail_at = 0;  // (wait kind << 12) | block, for the abort record
    for (int j = 0; j < nblk && ok; ++j) {
      const uint32_t scol = C::S_COL + uint32_t(64 * (j & 1));
      ok = __all_sync(kFull, mbar_wait(bar(B_SFULL + (j & 1)), (j >> 1) & 1));
      if (!ok) {
        fail_at = (1 << 12) | (j & 0xfff);
        break;
      }
      tc_fence_after();
      float s[64];
      {
        float x[32];
        tmem_ld32(lane_base + scol, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = x[i];
        tmem_ld32(lane_base + scol + 32, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 + i] = x[i];
      }

      // row maximum (the thread owns its row), taken on the raw scores: the
      // scale is positive (checked on the host), so it commutes with the
      // maximum and is applied inside the exponent below.  Only a block that
      // reaches past the last visible key is masked.
      const int key0 = k_begin + j * C::BK;
      if (key0 + C::BK - 1 > lim) {
#pragma unroll
        for (int k = 0; k < 64; ++k) s[k] = (key0 + k <= lim) ? s[k] : -INFINITY;
      }
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmaxf(s[i], s[8 + i]);
#pragma unroll
      for (int k = 16; k < 64; k += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[k + i]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
      float alpha = 1.f;
      bool rescale_o = false;
      if (mx > m_ref + C::RESCALE_LOG2 || (m_ref == -INFINITY && mx != -INFINITY)) {
        alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - mx);
        rescale_o = m_ref != -INFINITY;
        m_ref = mx;
        l *= alpha;
      }
      const float nms = m_ref == -INFINITY ? 0.f : -m_ref;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pv[i] = ex2(fmaf(s[8 * c + i], sl2, nms));
        l += ((pv[0] + pv[1]) + (pv[2] + pv[3])) + ((pv[4] + pv[5]) + (pv[6] + pv[7]));
#pragma unroll
        for (int i = 0; i < 4; ++i)
          pk[4 * c + i] = FP8 ? pack_f16(pv[2 * i], pv[2 * i + 1]) : pack_bf16(pv[2 * i], pv[2 * i + 1]);
      }
      // O may only be rescaled once PV(j-1) has finished accumulating into it
      if (__any_sync(kFull, rescale_o)) {
        if (j >= 1)
          ok = __all_sync(kFull, mbar_wait(bar(B_PFREE + ((j - 1) & 1)), ((j - 1) >> 1) & 1));
        if (!ok) {
          fail_at = (2 << 12) | (j & 0xfff);
          break;
        }
        tc_fence_after();
        for (int c0 = 0; c0 < 256; c0 += 32) {
          float o[32];
          tmem_ld32(lane_base + C::O_COL + uint32_t(c0), o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_base + C::O_COL + uint32_t(c0), o);
        }
      }
      // P over the first 32 columns of S_b (S_b has been read into registers)
      tmem_st32u(lane_base + scol, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + (j & 1)));
    }
    if (!ok) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      note_abort(abort_flag, (5 << 24) | fail_at);
    }

    // ---- epilogue: O / l for this CTA's 256 V columns
    const int row_n = t * C::ROWS + r;  // row of the item's partial block
    float lse_n = -INFINITY;
    if (l > 0.f) lse_n = (m_ref + lg2(l)) * kLn2m;
    const float inv = l > 0.f ? a.o_scale / l : 0.f;  // o_scale: the FP8 cache scale, else 1
    bool have_o = ok && nblk > 0;
    // PV(nblk - 1) complete (its commit covers every earlier MMA, PV(nblk - 2) too)
    if (have_o && !__all_sync(kFull, mbar_wait(bar(B_PFREE + ((nblk - 1) & 1)),
                                               ((nblk - 1) >> 1) & 1))) {
      have_o = false;
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      note_abort(abort_flag, 6 << 24);
    }
    if (have_o) tc_fence_after();
    const size_t out_row = (size_t(b) * a.T + t) * a.Hq + r;
    for (int c0 = 0; c0 < 256; c0 += 32) {
      float o[32];
      if (have_o) {
        tmem_ld32(lane_base + C::O_COL + uint32_t(c0), o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      const int d0 = h * 256 + c0;
      if (slot < 0) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + out_row * C::DV + d0;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 w;
          w.x = pack_bf16(o[i] * inv, o[i + 1] * inv);
          w.y = pack_bf16(o[i + 2] * inv, o[i + 3] * inv);
          w.z = pack_bf16(o[i + 4] * inv, o[i + 5] * inv);
          w.w = pack_bf16(o[i + 6] * inv, o[i + 7] * inv);
          *reinterpret_cast<uint4*>(dst + i) = w;
        }
      } else {
        float* dst = a.o_part + (size_t(slot) * a.rows + row_n) * C::DV + d0;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + i) =
              make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
      }
    }
    if (h == 0) {  // both halves hold the same (m, l)
      if (slot < 0) {
        if (a.lse) a.lse[out_row] = lse_n;
      } else {
        a.lse_part[size_t(slot) * a.rows + row_n] = lse_n;
      }
    }
  }

  // ---- teardown: TMEM is freed by the warp that allocated it
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    int32_t* lg = a.cta_log + size_t(blockIdx.x) * kLogFields;
    lg[0] = p0;
    lg[1] = p1;
    lg[2] = k_end > k_begin ? k_end - k_begin : 0;
    lg[3] = *abort_flag;
  }
}

// Copies keys [0, n_keys) of one sequence's latent (or separate V) rows
// through the block table with the decode kernel's tensor map, boxes and
// 128-byte-swizzled shared-memory addressing: per 64-key block and 64-column
// chunk, one box of 64 rows at the block's row offset (pages of 64 keys or a
// multiple of 64), or one box of P rows per page written P * 128 bytes apart
// (pages of 16 or 32 keys).  One CTA of 128 threads; one chunk at a time.
// Page ids outside [0, num_pages) are read as page 0, as in the decode kernel.
template <bool FP8>
__global__ void __launch_bounds__(128) mla_gather_debug_kernel(const __grid_constant__ CUtensorMap tm,
                                                               const int32_t* table_row, int P,
                                                               int num_pages, int row_elems,
                                                               int n_keys, uint8_t* dst) {
  constexpr int RB = FP8 ? 64 : 128;  // bytes of one 64-column row of a box
  __shared__ __align__(1024) uint8_t chunk[Mla::K_CH];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int small = P < Mla::BK;
  const int br = small ? P : Mla::BK;  // rows per box
  const int n_pages = (n_keys + P - 1) / P;
  const int n_chunks = row_elems / 64;
  int phase = 0;
  for (int key0 = 0; key0 < n_keys; key0 += Mla::BK) {
    for (int c = 0; c < n_chunks; ++c, ++phase) {
      if (threadIdx.x == 0) {
        const int nb = small ? min(Mla::BK / P, n_pages - key0 / P) : 1;
        mbar_arrive_expect_tx(smem_u32(&bar), uint32_t(nb * br * RB));
        for (int r = 0; r < nb; ++r) {
          const int page = small ? key0 / P + r : key0 / P;
          const int off = small ? 0 : key0 - page * P;
          int ph = table_row[page];
          if (ph < 0 || ph >= num_pages) ph = 0;
          tma_load_2d_warp_lane(smem_u32(chunk + r * br * RB), &tm, smem_u32(&bar), c * 64,
                                ph * P + off);
        }
      }
      if (!__syncthreads_and(mbar_wait(smem_u32(&bar), phase & 1))) {
        // one more bounded wait so the copy is not left writing into freed smem
        if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), phase & 1);
        __syncthreads();
        return;
      }
      const int rows = min(Mla::BK, n_keys - key0);
      constexpr int SEGS = RB / 16;  // 16-byte segments of a row
      for (int x = threadIdx.x; x < rows * SEGS; x += blockDim.x) {
        const int i = x / SEGS, seg = x % SEGS;
        // bf16: the 128-byte swizzle of the decode kernel's boxes; e4m3: the
        // unswizzled rows its converter warps read
        const uint32_t off = FP8 ? uint32_t(i * 64 + seg * 16) : uint32_t(i * 128 + ((seg ^ (i & 7)) << 4));
        *reinterpret_cast<uint4*>(dst + size_t(key0 + i) * row_elems * (FP8 ? 1 : 2) +
                                  (c * 64) * (FP8 ? 1 : 2) + seg * 16) =
            *reinterpret_cast<const uint4*>(chunk + off);
      }
      __syncthreads();
    }
  }
}

}  // namespace

namespace {

template <bool SEPV, bool SMALLP, bool FP8 = false>
cudaError_t launch_mla_t(const DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                         cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(
      mla_splitkv_kernel<SEPV, SMALLP, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, Mla::SMEM);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_items * a.T * 2, 1, 1);
  cfg.blockDim = dim3(SEPV ? Mla::THREADS + 32 : (FP8 ? Mla::THREADS + 128 : Mla::THREADS), 1, 1);
  cfg.dynamicSmemBytes = Mla::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_splitkv_kernel<SEPV, SMALLP, FP8>, a, mk, mv);
}

}  // namespace

cudaError_t launch_mla(const DecodeArgs& a, const TmaDesc& tk, const TmaDesc* tv, bool fp8,
                       void* stream) {
  if (a.n_items == 0) return cudaSuccess;
  const CUtensorMap& mk = *reinterpret_cast<const CUtensorMap*>(&tk);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // pages of 16 or 32 keys: several boxes per 64-key block
  const bool small = a.P < Mla::BK;
  if (fp8) {
    if (tv) return cudaErrorInvalidValue;  // FP8 latent caches hold V in the key rows
    return small ? launch_mla_t<false, true, true>(a, mk, mk, s)
                 : launch_mla_t<false, false, true>(a, mk, mk, s);
  }
  if (tv) {
    const CUtensorMap& mv = *reinterpret_cast<const CUtensorMap*>(tv);
    return small ? launch_mla_t<true, true>(a, mk, mv, s) : launch_mla_t<true, false>(a, mk, mv, s);
  }
  return small ? launch_mla_t<false, true>(a, mk, mk, s) : launch_mla_t<false, false>(a, mk, mk, s);
}

cudaError_t launch_mla_debug_gather(const TmaDesc& t, bool fp8, const int32_t* table_row, int32_t P,
                                    int32_t num_pages, int32_t row_elems, int32_t n_keys, void* dst,
                                    void* stream) {
  const CUtensorMap& m = *reinterpret_cast<const CUtensorMap*>(&t);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fp8)
    mla_gather_debug_kernel<true><<<1, 128, 0, s>>>(m, table_row, P, num_pages, row_elems, n_keys,
                                                    static_cast<uint8_t*>(dst));
  else
    mla_gather_debug_kernel<false><<<1, 128, 0, s>>>(m, table_row, P, num_pages, row_elems, n_keys,
                                                     static_cast<uint8_t*>(dst));
  return cudaGetLastError();
}

}  // namespace splitkv
