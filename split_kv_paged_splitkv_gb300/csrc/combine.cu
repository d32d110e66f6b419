// Log-sum-exp combine of split partials (separate-kernel mode and the
// standalone splitkv_combine entry point).
//
// For a row with partials (O_s, lse_s), s < S:  M = max_s lse_s,
// lse = M + ln sum_s exp(lse_s - M),  out = sum_s exp(lse_s - lse) O_s.
// Partials with lse_s = -inf weigh nothing; a row whose partials are all
// -inf gets out = 0 and lse = -inf.  This is the merge step of "vLLM 0.30.0
// FA4 SplitKV Bug: H100 Decode Can Be 48% Slower", section "Why the result
// is still correct" (empty splits contribute zero weight).
#include <cuda_runtime.h>

#include "fixed_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace splitkv {
namespace {

using namespace ptx;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One CTA of 128 threads per (group, row, 64-dim chunk): 16 lanes x 4 float
// dims each, and 8 "ways" that take every 8th split.  A thread loads the LSE
// and the O values of up to PER_WAY of its splits at once (one L2 round trip
// for up to 8 * PER_WAY splits), keeps a running maximum across further
// chunks of splits, and the 8 ways are merged through shared memory at the
// end.  Measured on the 5.9k decode (64 splits, 16 rows): 1.98 us against
// 2.18 with 128-dim chunks (4 ways of 32 lanes, 16 loads each: twice the
// bytes per CTA and 168 registers a thread).  Groups of at most 16 splits use
// one warp per row instead (below), which matters when there are thousands
// of rows (the MLA merge: 768 rows x 4 column chunks).
//   plan mode (groups != nullptr): group g = blockIdx.x covers slots
//     slot0 .. slot0+S-1 with `rows` rows each; row n -> (t, head) of (b, the
//     group's KV heads).
//   raw mode: one group, S = n_parts, slot0 = 0, output row n.
constexpr int kCombineThreads = 128;

// WAYS > 1: one row per CTA; DL = 128 / WAYS lanes of 4 dims each cover
// 4 * DL dims, the WAYS groups take every WAYS-th split and merge through
// shared memory.  WAYS = 1 (small groups; PER_WAY splits per pass): each warp
// (DL = 32) merges a row of its own over all the splits, 4 rows per CTA,
// with no shared memory and no CTA barrier.
template <int WAYS, int PER_WAY, bool CAP>
__device__ __forceinline__ void combine_body(
    const float* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ groups, int n_parts, int rows, int dv, int T, int Hq, int G,
    void* out_bf16, float* out_f32, float* lse_out, int pdl, int fixed, const FixedShape& fx) {
  __shared__ float4 red[kCombineThreads];
  __shared__ float red_w[kCombineThreads], red_m[kCombineThreads];
  launch_dependents();
  // The group table of a host plan is uploaded with the plan and never
  // written by a kernel: it is read before waiting for the split kernel, off
  // the critical path.  A capacity plan's group g = b * U + u has its slots
  // [g S, g S + S) fixed, but its split count follows the device length of
  // sequence b: after the wait that length is read together with the
  // partials of every slot of the group, and the splits past the count are
  // dropped by select (those slots may hold anything).  A group with no
  // splits to merge (S_b <= 1) leaves the output the split kernel wrote.
  // Without the lengths (the standalone merge of a capacity plan's
  // workspace) the group table the split kernel wrote is read after the wait.
  if (!CAP && fixed && pdl) wait_prerequisites();
  static_assert(WAYS == 1 || WAYS == 8, "ways");
  constexpr int DL = WAYS == 1 ? 32 : kCombineThreads / WAYS;  // dim lanes of a way
  constexpr int RPC = WAYS == 1 ? kCombineThreads / 32 : 1;    // rows per CTA
  const int n = blockIdx.y * RPC + (WAYS == 1 ? int(threadIdx.x >> 5) : 0);
  if (WAYS == 1 && n >= rows) return;
  int S = n_parts, slot0 = 0;
  size_t orow = n;
  // CAP: the groups of a capacity plan (groups != nullptr)
  constexpr bool cap = CAP;
  int S_load = n_parts;  // CAP: the slots loaded, every slot of the group
  int bcap = 0;  // CAP: the group's sequence
  if constexpr (CAP) {
    const int b = blockIdx.x / fx.U, hkv = (blockIdx.x % fx.U) * fx.hpi;
    bcap = b;
    slot0 = blockIdx.x * fx.S;
    S_load = fx.S;
    const int hs = n / (T * G), r = n - hs * (T * G);
    const int t = r / G, gg = r - t * G;
    orow = (size_t(b) * T + t) * Hq + size_t(hkv + hs) * G + gg;
    if (pdl) wait_prerequisites();
  } else {
    if (groups) {
      const int32_t* g = groups + size_t(blockIdx.x) * kGroupFields;
      const int b = g[0], hkv = g[1];
      S = g[2];
      slot0 = g[3];
      // rows are numbered hs * T*G + t * G + gg over the group's heads hkv + hs
      const int hs = n / (T * G), r = n - hs * (T * G);
      const int t = r / G, gg = r - t * G;
      orow = (size_t(b) * T + t) * Hq + size_t(hkv + hs) * G + gg;
      if (S == 0) return;
    }
    if (pdl) wait_prerequisites();
  }
  const int tid = threadIdx.x, dl = tid % DL, way = WAYS == 1 ? 0 : tid / DL;
  const int d = blockIdx.z * (DL * 4) + dl * 4;
  const bool dim_ok = d < dv;
  const float* lp = lse_part + size_t(slot0) * rows + n;
  const float* op = o_part + (size_t(slot0) * rows + n) * dv + (dim_ok ? d : 0);
  const size_t ostride = size_t(rows) * dv;

  float m_run = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool have_S = !cap;  // (a compile-time true without CAP)
  const int S_end = CAP ? S_load : S;
  for (int s0 = way; s0 < S_end; s0 += WAYS * PER_WAY) {
    float lv[PER_WAY];
    float4 x[PER_WAY];
#pragma unroll
    for (int u = 0; u < PER_WAY; ++u) {
      const int s = s0 + u * WAYS;
      lv[u] = -INFINITY;
      x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s < S_end) {
        lv[u] = lp[size_t(s) * rows];
        if (dim_ok) x[u] = *reinterpret_cast<const float4*>(op + size_t(s) * ostride);
      }
    }
    if (!have_S) {
      // the group's device length, read after the partials' loads are
      // issued (read before them it measured 0.25 us slower per 5.9k call)
      bool bad;
      const int Sb = fixed_splits(fx, fixed_len_of(fx, fx.seq_lens[bcap], &bad));
      S = Sb > 1 ? Sb : 0;
      have_S = true;
    }
    if constexpr (CAP) {
#pragma unroll
      for (int u = 0; u < PER_WAY; ++u)
        if (s0 + u * WAYS >= S) {  // past the group's splits: a slot of no split
          lv[u] = -INFINITY;
          x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float m_new = m_run;
#pragma unroll
    for (int u = 0; u < PER_WAY; ++u) m_new = fmaxf(m_new, lv[u]);
    if (m_new == -INFINITY) continue;  // every split so far is empty
    const float rs = ex2((m_run - m_new) * kLog2e);  // 0 when m_run is -inf
    acc.x *= rs; acc.y *= rs; acc.z *= rs; acc.w *= rs;
    wsum *= rs;
#pragma unroll
    for (int u = 0; u < PER_WAY; ++u) {
      const float w = ex2((lv[u] - m_new) * kLog2e);  // 0 for empty splits
      wsum += w;
      acc.x += w * x[u].x; acc.y += w * x[u].y; acc.z += w * x[u].z; acc.w += w * x[u].w;
    }
    m_run = m_new;
  }
  if (!have_S) {  // a way with no slot of the group (S_load <= way)
    bool bad;
    const int Sb = fixed_splits(fx, fixed_len_of(fx, fx.seq_lens[bcap], &bad));
    S = Sb > 1 ? Sb : 0;
  }
  if (cap && S == 0) return;  // the same for the whole CTA (one group)
  float M = m_run, wtot = wsum;
  float4 tot = acc;
  if constexpr (WAYS > 1) {
    // Every thread rescales its own way's sums to the maximum M over the
    // WAYS ways of its dim lane; the ways are then added pairwise within a
    // warp (the two ways of a warp sit 16 lanes apart) and the warps' sums
    // through shared memory, all threads at once (a single way adding the
    // others one after another took ~1,000 cycles on the 5.9k call).
    static_assert(WAYS == 8 && DL == 16, "two ways per warp");
    red_m[tid] = m_run;
    __syncthreads();
    M = -INFINITY;
#pragma unroll
    for (int k = 0; k < WAYS; ++k) M = fmaxf(M, red_m[dl + DL * k]);
    const float sc = m_run == -INFINITY ? 0.f : ex2((m_run - M) * kLog2e);
    float4 v = make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
    float w = wsum * sc;
    v.x += __shfl_xor_sync(kFull, v.x, 16);
    v.y += __shfl_xor_sync(kFull, v.y, 16);
    v.z += __shfl_xor_sync(kFull, v.z, 16);
    v.w += __shfl_xor_sync(kFull, v.w, 16);
    w += __shfl_xor_sync(kFull, w, 16);
    const int wp = tid >> 5;  // warp: ways 2 wp and 2 wp + 1
    if ((tid & 16) == 0) {
      red[wp * DL + dl] = v;
      red_w[wp * DL + dl] = w;
    }
    __syncthreads();
    if (tid >= DL) return;
    tot = red[dl];
    wtot = red_w[dl];
#pragma unroll
    for (int k = 1; k < WAYS / 2; ++k) {
      const float4 o = red[k * DL + dl];
      tot.x += o.x; tot.y += o.y; tot.z += o.z; tot.w += o.w;
      wtot += red_w[k * DL + dl];
    }
  }
  float lse_n = -INFINITY;
  if (wtot > 0.f) {
    const float inv = __frcp_rn(wtot);
    tot.x *= inv; tot.y *= inv; tot.z *= inv; tot.w *= inv;
    lse_n = M + lg2(wtot) * kLn2;
  }
  if (dim_ok) {
    if (out_bf16) {
      uint2 v;
      v.x = pack_bf16(tot.x, tot.y);
      v.y = pack_bf16(tot.z, tot.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out_bf16) + orow * dv + d) = v;
    }
    if (out_f32) *reinterpret_cast<float4*>(out_f32 + orow * dv + d) = tot;
  }
  if (dl == 0 && blockIdx.z == 0 && lse_out) lse_out[orow] = lse_n;
}

// Host plans and the standalone merge: the group table (or one raw group).
template <int WAYS, int PER_WAY>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ groups, int n_parts, int rows, int dv, int T, int Hq, int G,
    void* out_bf16, float* out_f32, float* lse_out, int pdl, int fixed) {
  combine_body<WAYS, PER_WAY, false>(o_part, lse_part, groups, n_parts, rows, dv, T, Hq, G,
                                     out_bf16, out_f32, lse_out, pdl, fixed, FixedShape{});
}

// Capacity plans: each group's split count from the device lengths.
template <int WAYS, int PER_WAY>
__global__ void __launch_bounds__(kCombineThreads) combine_cap_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ groups, int n_parts, int rows, int dv, int T, int Hq, int G,
    void* out_bf16, float* out_f32, float* lse_out, int pdl, const FixedShape fx) {
  combine_body<WAYS, PER_WAY, true>(o_part, lse_part, groups, n_parts, rows, dv, T, Hq, G,
                                    out_bf16, out_f32, lse_out, pdl, 1, fx);
}

}  // namespace

namespace {

// Groups of at most kSmallGroup splits take the warp-per-row form, kSmallLoads
// splits per pass.  Measured on the MLA merge (768 rows x 512 dims, 12
// splits): 4.1 us with 8 loads per pass, 4.8 with 16 (162 registers), 5.8
// with the 4-way form at 4 loads per way, 14.3 at 16 loads per way.  Above
// kSmallLoads splits that form needs a second dependent pass over L2, which
// only pays when the launch has rows enough to fill the GPU: a merge of a few
// rows (one short GQA sequence, 16 rows, 9 to 16 splits) took ~0.5 us longer
// per call than with 8 or 17 splits, so there the 8-way form (one pass for up
// to 64 splits) is used instead.
constexpr int kSmallGroup = 16;
constexpr int kSmallLoads = 8;
constexpr long kManyRowCtas = 256;  // warp-per-row CTAs that fill the GPU

bool warp_per_row(int max_splits, long groups, int rows, int dv) {
  if (max_splits <= kSmallLoads) return true;
  if (max_splits > kSmallGroup) return false;
  return groups * ((rows + 3) / 4) * ((dv + 127) / 128) >= kManyRowCtas;
}

// Shared-memory carveout: the kernel's 3 KB of shared memory would otherwise
// cap the resident CTAs below what the registers allow.  Set once per
// instantiation.
template <int WAYS, int PER_WAY, bool CAP>
cudaError_t combine_attrs() {
  static cudaError_t e =
      CAP ? cudaFuncSetAttribute(combine_cap_kernel<WAYS, PER_WAY>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout, 50)
          : cudaFuncSetAttribute(combine_kernel<WAYS, PER_WAY>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout, 50);
  return e;
}

template <int WAYS, int PER_WAY, bool CAP>
cudaError_t launch_combine_t(const DecodeArgs& a, bool pdl, cudaStream_t s) {
  cudaError_t e = combine_attrs<WAYS, PER_WAY, CAP>();
  if (e != cudaSuccess) return e;
  constexpr int RPC = WAYS == 1 ? kCombineThreads / 32 : 1;
  constexpr int DIMS = WAYS == 1 ? 128 : 4 * kCombineThreads / WAYS;  // dims per CTA
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_groups, (a.rows + RPC - 1) / RPC, (a.dv + DIMS - 1) / DIMS);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if constexpr (CAP)
    return cudaLaunchKernelEx(&cfg, combine_cap_kernel<WAYS, PER_WAY>,
                              static_cast<const float*>(a.o_part), static_cast<const float*>(a.lse_part),
                              a.groups, 0, a.rows, a.dv, a.T, a.Hq, a.G, a.out,
                              static_cast<float*>(nullptr), a.lse, pdl ? 1 : 0, a.fx);
  else
    return cudaLaunchKernelEx(&cfg, combine_kernel<WAYS, PER_WAY>,
                              static_cast<const float*>(a.o_part), static_cast<const float*>(a.lse_part),
                              a.groups, 0, a.rows, a.dv, a.T, a.Hq, a.G, a.out,
                              static_cast<float*>(nullptr), a.lse, pdl ? 1 : 0, a.fixed);
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, bool pdl, void* stream) {
  if (a.n_groups == 0) return cudaSuccess;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // A capacity plan's decode passes its lengths (a.fx); the standalone merge
  // of its workspace does not, and reads the group table instead.
  const bool cap = a.fixed && a.fx.seq_lens != nullptr && a.fx.U > 0 && a.fx.S > 0;
  if (warp_per_row(a.max_splits, a.n_groups, a.rows, a.dv))
    return cap ? launch_combine_t<1, kSmallLoads, true>(a, pdl, s)
               : launch_combine_t<1, kSmallLoads, false>(a, pdl, s);
  return cap ? launch_combine_t<8, 8, true>(a, pdl, s) : launch_combine_t<8, 8, false>(a, pdl, s);
}

cudaError_t launch_combine_raw(const float* o_part, const float* lse_part, int n_parts, int rows,
                               int dv, void* out_bf16, float* out_f32, float* lse_out,
                               void* stream) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(1, rows, (dv + 127) / 128), block(kCombineThreads, 1, 1);  // (small groups)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (warp_per_row(n_parts, 1, rows, dv)) {
    cudaError_t e = combine_attrs<1, kSmallLoads, false>();
    if (e != cudaSuccess) return e;
    grid.y = (rows + 3) / 4;
    combine_kernel<1, kSmallLoads><<<grid, block, 0, s>>>(o_part, lse_part, nullptr, n_parts, rows,
                                                          dv, 1, 1, 1, out_bf16, out_f32, lse_out,
                                                          0, 0);
  } else {
    cudaError_t e = combine_attrs<8, 8, false>();
    if (e != cudaSuccess) return e;
    grid.z = (dv + 63) / 64;
    combine_kernel<8, 8><<<grid, block, 0, s>>>(o_part, lse_part, nullptr, n_parts, rows, dv, 1, 1,
                                                1, out_bf16, out_f32, lse_out, 0, 0);
  }
  return cudaGetLastError();
}

}  // namespace splitkv
