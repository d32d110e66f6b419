// Split-KV partial attention for the MLA-style decode (128 query heads of up
// to 16 tokens sharing one 576-wide latent KV head, V = its first 512
// columns), on the 5th-generation tensor cores (tcgen05, accumulators in
// TMEM).  This is the dense case of the split-KV decode: "Shipped: 484.5
// tok/s on one GB300 ...", table "What shipped" (MLA decode of one request at
// 6 tokens per step, split 4 ways), with the per-split partial and the
// log-sum-exp merge of "vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48%
// Slower", section "What SplitKV is trying to do".
//
// Work: one 2-CTA cluster per (work item, query token).  The 128 heads of the
// token are the MMA rows (M = 128).  A 128 x 512 fp32 output tile would fill
// all of TMEM and its 128 x 576 bf16 query tile most of shared memory, so the
// pair splits the 576-wide contraction:
//   rank 0: dims [0, 256) and [512, 576)   (5 chunks of 64)
//   rank 1: dims [256, 512)                (4 chunks of 64)
// Each rank's chunks contain the 256 V columns it owns (rank r: V columns
// [256 r, 256 r + 256)), so the keys it loads serve both its QK part and its
// PV part.  Per 64-key block (one page):
//   1. S_r = Q_r . K_r^T                      (tcgen05, M=128 N=64, TMEM)
//   2. softmax warps read S_r, send it to the peer through distributed shared
//      memory, receive S_peer, and form S = S_r + S_peer (the same sum on both
//      ranks: fp32 addition is commutative), then online softmax with a lazy
//      reference maximum (O is rescaled only when a row maximum grows by more
//      than 2^8) and write P (bf16) to shared memory;
//   3. O_r += P . V_r                         (tcgen05, M=128 N=256, TMEM)
// Warp roles: warp 0 TMA producer and TMEM owner, warp 1 MMA issuer, warps
// 2-5 softmax / exchange / epilogue (thread = query head = TMEM lane).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace splitkv {
namespace {

using namespace ptx;

struct Mla {
  static constexpr int DK = 576, DV = 512;
  static constexpr int ROWS = 128;         // query heads of one token
  static constexpr int BK = 64;            // keys per block (= one page)
  static constexpr int NCH_MAX = 5;        // 64-dim chunks held by rank 0
  static constexpr int Q_CH = ROWS * 128;  // one Q chunk: 128 rows x 64 bf16 = 16 KB
  static constexpr int K_CH = BK * 128;    // one K chunk: 64 keys x 64 bf16 = 8 KB
  static constexpr int NST = 2;            // key-block stages
  static constexpr int Q_BYTES = NCH_MAX * Q_CH;
  static constexpr int K_STAGE = NCH_MAX * K_CH;
  static constexpr int P_BYTES = ROWS * BK * 2;  // P: 128 rows x 64 keys bf16
  static constexpr int X_BYTES = ROWS * BK * 4;  // peer scores: 128 x 64 fp32
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_P = OFF_K + NST * K_STAGE;
  static constexpr int OFF_X = OFF_P + P_BYTES;
  static constexpr int OFF_BAR = OFF_X + X_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 512;  // S buffers at cols 0 and 64, O at 256
  static constexpr uint32_t O_COL = 256;
  static constexpr float RESCALE_LOG2 = 8.f;  // lazy maximum: rescale when it grows by > 2^8
};

constexpr float kLn2m = 0.6931471805599453f;

// Barrier slots (8 bytes each) after OFF_BAR.
enum {
  B_QFULL = 0,
  B_KFULL = 1,   // [2]
  B_KEMPTY = 3,  // [2]
  B_SFULL = 5,   // [2]
  B_SFREE = 7,   // [2]
  B_PFULL = 9,
  B_PFREE = 10,
  B_XIN = 11,    // peer's scores arrived in my X buffer
  B_XOUT = 12,   // peer has read the scores I sent (my send buffer at the peer is free)
  B_COUNT = 13
};

__device__ __forceinline__ int chunk_of(int rank, int slot) {
  return rank == 0 ? (slot < 4 ? slot : 8) : 4 + slot;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Mla::THREADS, 1)
    mla_splitkv_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tk) {
  using C = Mla;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int item = pair / a.T;
  const int t = pair - item * a.T;
  const int nch = rank == 0 ? 5 : 4;

  const int32_t* it = a.items + size_t(item) * SPLITKV_ITEM_FIELDS;
  const int b = it[SPLITKV_ITEM_B];
  const int p0 = it[SPLITKV_ITEM_PAGE0], p1 = it[SPLITKV_ITEM_PAGE1];
  const int slot = it[SPLITKV_ITEM_SLOT];

  // ---- prologue (shared memory, TMEM, tensor maps, work list only)
  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SFREE + s), 128);
    }
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_PFREE), 1);
    mbar_init(bar(B_XIN), 128);
    mbar_init(bar(B_XOUT), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // plan's sequence length (uploaded, never written by a kernel): read before the wait
  const int L = a.plan_lens[b];
  const int k_begin = p0 * C::BK;
  const int k_end = min(p1 * C::BK, L);
  const int nblk = k_end > k_begin ? (k_end - k_begin + C::BK - 1) / C::BK : 0;
  const int lim = L - a.T + t;  // last key visible to this token
  launch_dependents();
  wait_prerequisites();
  if (threadIdx.x == 0 && rank == 0 && t == 0 && a.seq_lens[b] != L)
    atomicOr(a.status, SPLITKV_DEVERR_SEQLEN);

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    const int32_t* trow = a.block_table + size_t(b) * a.max_pages;
    bool ok = true;
    int issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(B_QFULL), nch * C::Q_CH);
      const int qrow = (b * a.T + t) * C::ROWS;
      for (int i = 0; i < nch; ++i)
        tma_load_2d(smem_u32(sm + C::OFF_Q + i * C::Q_CH), &tq, bar(B_QFULL), chunk_of(rank, i) * 64, qrow);
    }
    int phys = 0, chunk0 = -32;
    for (int j = 0; j < nblk && ok; ++j) {
      const int page = p0 + j;
      if (page >= chunk0 + 32) {
        chunk0 = page;
        const int my = chunk0 + lane;
        phys = 0;
        if (my < p1) {
          phys = __ldg(trow + my);
          if (phys < 0 || phys >= a.num_pages) {
            atomicOr(a.status, SPLITKV_DEVERR_PAGE);
            phys = 0;
          }
        }
      }
      const int ph = __shfl_sync(kFull, phys, page - chunk0);
      if (lane == 0) {
        const int st = j % C::NST;
        if (j >= C::NST && !mbar_wait(bar(B_KEMPTY + st), ((j / C::NST) - 1) & 1)) {
          atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
        } else {
          mbar_arrive_expect_tx(bar(B_KFULL + st), nch * C::K_CH);
          for (int i = 0; i < nch; ++i)
            tma_load_2d(smem_u32(sm + C::OFF_K + st * C::K_STAGE + i * C::K_CH), &tk,
                        bar(B_KFULL + st), chunk_of(rank, i) * 64, (ph * a.Hkv) * a.P);
          issued = j + 1;
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
    }
    // stay until every issued copy has landed
    if (lane == 0) {
      mbar_wait(bar(B_QFULL), 0);
      for (int st = 0; st < C::NST && st < issued; ++st) {
        const int last = st + C::NST * ((issued - 1 - st) / C::NST);
        if (!mbar_wait(bar(B_KFULL + st), (last / C::NST) & 1)) break;
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    const uint32_t idesc_qk = umma_idesc_bf16(128, 64, 0, 0);
    const uint32_t idesc_pv = umma_idesc_bf16(128, 256, 0, 1);
    bool ok = __all_sync(kFull, mbar_wait(bar(B_QFULL), 0));
    for (int j = 0; j <= nblk && ok; ++j) {
      if (j < nblk) {  // S[j % 2] = Q . K_j^T
        const int st = j % C::NST;
        bool w = mbar_wait(bar(B_KFULL + st), (j / C::NST) & 1);
        if (w && j >= C::NST) w = mbar_wait(bar(B_SFREE + st), ((j / C::NST) - 1) & 1);
        ok = __all_sync(kFull, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t d = tmem + uint32_t(st * C::BK);
          for (int i = 0; i < nch; ++i)
            for (int kin = 0; kin < 4; ++kin) {
              const uint64_t ad = umma_desc(smem_u32(sm + C::OFF_Q + i * C::Q_CH) + kin * 32, 16, 1024, 2);
              const uint64_t bd =
                  umma_desc(smem_u32(sm + C::OFF_K + st * C::K_STAGE + i * C::K_CH) + kin * 32, 16, 1024, 2);
              umma_bf16(d, ad, bd, idesc_qk, (i | kin) != 0);
            }
          umma_commit(bar(B_SFULL + st));
        }
        __syncwarp();
      }
      if (j >= 1) {  // O += P_{j-1} . V_{j-1}
        const int jj = j - 1, st = jj % C::NST;
        ok = __all_sync(kFull, mbar_wait(bar(B_PFULL), jj & 1));
        if (!ok) break;
        tc_fence_after();
        const int valid = min(C::BK, k_end - (k_begin + jj * C::BK));
        if (valid < C::BK) {
          // key slots past the last key may hold anything (even NaN): zero their
          // V rows so that 0 * V stays 0 in the PV product
          uint8_t* kst = sm + C::OFF_K + st * C::K_STAGE;
          for (int x = lane; x < (C::BK - valid) * 8 * 4; x += 32) {
            const int r = valid + (x >> 5), ch = (x >> 3) & 3, c16 = x & 7;
            *reinterpret_cast<uint4*>(kst + ch * C::K_CH + r * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        if (lane == 0) {
          for (int kin = 0; kin < 4; ++kin) {
            const uint64_t ad = umma_desc(smem_u32(sm + C::OFF_P) + kin * 32, 16, 1024, 2);
            const uint64_t bd =
                umma_desc(smem_u32(sm + C::OFF_K + st * C::K_STAGE) + kin * 16 * 128, C::K_CH, 1024, 2);
            umma_bf16(tmem + C::O_COL, ad, bd, idesc_pv, (jj | kin) != 0);
          }
          umma_commit(bar(B_KEMPTY + st));
          umma_commit(bar(B_PFREE));
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else {
    // -------------------------------------------------------------- softmax warps
    const int g = warp & 3;          // TMEM lane group of this warp
    const int r = g * 32 + lane;     // query head = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(g * 32) << 16);
    const uint32_t x_local = smem_u32(sm + C::OFF_X);
    const uint32_t x_remote = map_to_rank(x_local, peer);
    const uint32_t xin_remote = map_to_rank(bar(B_XIN), peer);
    const uint32_t xout_remote = map_to_rank(bar(B_XOUT), peer);
    uint8_t* prow = sm + C::OFF_P + r * 128;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk && ok; ++j) {
      const int st = j % C::NST;
      ok = __all_sync(kFull, mbar_wait(bar(B_SFULL + st), (j / C::NST) & 1));
      if (!ok) break;
      tc_fence_after();
      float s[64];
      {
        float h[32];
        tmem_ld32(lane_base + uint32_t(st * C::BK), h);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = h[i];
        tmem_ld32(lane_base + uint32_t(st * C::BK + 32), h);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 + i] = h[i];
      }
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + st));

      // exchange the partial scores with the peer: [16 chunks][128 rows][16 B]
      if (j >= 1) ok = __all_sync(kFull, mbar_wait_cluster(bar(B_XOUT), (j - 1) & 1));
      if (!ok) break;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_cluster_v4(x_remote + uint32_t((c * 128 + r) * 16), s[4 * c], s[4 * c + 1], s[4 * c + 2],
                      s[4 * c + 3]);
      mbar_arrive_remote(xin_remote);
      ok = __all_sync(kFull, mbar_wait_cluster(bar(B_XIN), j & 1));
      if (!ok) break;
      const float4* xr = reinterpret_cast<const float4*>(sm + C::OFF_X);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 v = xr[c * 128 + r];
        s[4 * c] += v.x;
        s[4 * c + 1] += v.y;
        s[4 * c + 2] += v.z;
        s[4 * c + 3] += v.w;
      }
      mbar_arrive_remote(xout_remote);

      // scale into log2 units, mask, row maximum (the thread owns its row)
      const int key0 = k_begin + j * C::BK;
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        float v = s[k] * a.qk_scale_log2;
        v = (key0 + k <= lim) ? v : -INFINITY;
        s[k] = v;
        mx = fmaxf(mx, v);
      }
      float alpha = 1.f;
      bool rescale_o = false;
      if (mx > m_ref + C::RESCALE_LOG2 || (m_ref == -INFINITY && mx != -INFINITY)) {
        alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - mx);
        rescale_o = m_ref != -INFINITY;
        m_ref = mx;
        l *= alpha;
      }
      const float ms = m_ref == -INFINITY ? 0.f : m_ref;

      // P(j) may only be written after PV(j-1) has read P(j-1)
      if (j >= 1) ok = __all_sync(kFull, mbar_wait(bar(B_PFREE), (j - 1) & 1));
      if (!ok) break;
      tc_fence_after();
      if (__any_sync(kFull, rescale_o)) {
        for (int c0 = 0; c0 < 256; c0 += 32) {
          float o[32];
          tmem_ld32(lane_base + C::O_COL + uint32_t(c0), o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_base + C::O_COL + uint32_t(c0), o);
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pv[i] = ex2(s[8 * c + i] - ms);
          l += pv[i];
        }
        uint4 w;
        w.x = pack_bf16(pv[0], pv[1]);
        w.y = pack_bf16(pv[2], pv[3]);
        w.z = pack_bf16(pv[4], pv[5]);
        w.w = pack_bf16(pv[6], pv[7]);
        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = w;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    if (!ok) {
      atomicOr(a.status, SPLITKV_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }

    // ---- epilogue: O / l for this rank's 256 V columns
    const int row_n = t * C::ROWS + r;  // row of the item's partial block
    float lse_n = -INFINITY;
    if (l > 0.f) lse_n = (m_ref + lg2(l)) * kLn2m;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const bool have_o = ok && nblk > 0 &&
                        __all_sync(kFull, mbar_wait(bar(B_PFREE), (nblk - 1) & 1));
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
      const int d0 = int(rank) * 256 + c0;
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
    if (rank == 0) {
      if (slot < 0) {
        if (a.lse) a.lse[out_row] = lse_n;
      } else {
        a.lse_part[size_t(slot) * a.rows + row_n] = lse_n;
      }
    }
  }

  // ---- teardown: no CTA of the pair may leave while the other can still
  // touch its shared memory; TMEM is freed by the warp that allocated it.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
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

}  // namespace

cudaError_t launch_mla(const DecodeArgs& a, const TmaDesc& tq, const TmaDesc& tk, void* stream) {
  if (a.n_items == 0) return cudaSuccess;
  static cudaError_t attr = cudaFuncSetAttribute(
      mla_splitkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Mla::SMEM);
  if (attr != cudaSuccess) return attr;
  const CUtensorMap& mq = *reinterpret_cast<const CUtensorMap*>(&tq);
  const CUtensorMap& mk = *reinterpret_cast<const CUtensorMap*>(&tk);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_items * a.T * 2, 1, 1);
  cfg.blockDim = dim3(Mla::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Mla::SMEM;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_splitkv_kernel, a, mq, mk);
}

}  // namespace splitkv
