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

#include "internal.h"
#include "ptx.cuh"

namespace splitkv {
namespace {

using namespace ptx;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One CTA of 128 threads per (group, row).  The row's S LSE values are staged
// in shared memory by all threads at once.  Each thread owns 4 dims (float4)
// and 1/W of the splits, W = 128 / (dv / 4) "ways"; it keeps 8 splits' loads
// in flight per step, and the W ways are summed through shared memory.
//   plan mode (groups != nullptr): group g = blockIdx.x covers slots
//     slot0 .. slot0+S-1 with `rows` rows each; row n -> (t, head) of (b, h_kv).
//   raw mode: one group, S = n_parts, slot0 = 0, output row n.
constexpr int kCombineThreads = 128;
constexpr int kCombineMaxParts = 1024;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ groups, int n_parts, int rows, int dv, int T, int Hq, int G,
    void* out_bf16, float* out_f32, float* lse_out, int pdl) {
  __shared__ float sl[kCombineMaxParts];
  __shared__ float4 red[kCombineThreads];
  __shared__ float wred[kCombineThreads];
  launch_dependents();
  if (pdl) wait_prerequisites();
  const int n = blockIdx.y;
  int S = n_parts, slot0 = 0;
  size_t orow = n;
  if (groups) {
    const int32_t* g = groups + size_t(blockIdx.x) * kGroupFields;
    const int b = g[0], hkv = g[1];
    S = g[2];
    slot0 = g[3];
    const int t = n / G, gg = n - t * G;
    orow = (size_t(b) * T + t) * Hq + size_t(hkv) * G + gg;
  }
  const int tid = threadIdx.x;
  for (int s = tid; s < S; s += kCombineThreads) sl[s] = lse_part[size_t(slot0 + s) * rows + n];
  __syncthreads();
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, sl[s]);

  const int lanes = dv >> 2;                 // threads per row of dims
  const int ways = kCombineThreads / lanes;  // splits interleaved over this many threads
  const int dl = tid % lanes, way = tid / lanes;
  const int d = dl * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY && way < ways) {
    const size_t stride = size_t(rows) * dv;
    const float* base = o_part + (size_t(slot0) * rows + n) * dv + d;
    for (int s0 = way; s0 < S; s0 += 8 * ways) {
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + u * ways;
        if (s < S) x[u] = *reinterpret_cast<const float4*>(base + size_t(s) * stride);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + u * ways;
        if (s < S) {
          const float w = ex2((sl[s] - M) * kLog2e);
          wsum += w;
          acc.x += w * x[u].x;
          acc.y += w * x[u].y;
          acc.z += w * x[u].z;
          acc.w += w * x[u].w;
        }
      }
    }
  }
  red[tid] = acc;
  wred[tid] = wsum;
  __syncthreads();
  if (way != 0) return;
  for (int k = 1; k < ways; ++k) {
    const float4 o = red[tid + k * lanes];
    acc.x += o.x;
    acc.y += o.y;
    acc.z += o.z;
    acc.w += o.w;
    wsum += wred[tid + k * lanes];
  }
  float lse_n = -INFINITY;
  if (wsum > 0.f) {
    const float inv = 1.f / wsum;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    lse_n = M + lg2(wsum) * kLn2;
  }
  if (out_bf16) {
    uint2 v;
    v.x = pack_bf16(acc.x, acc.y);
    v.y = pack_bf16(acc.z, acc.w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out_bf16) + orow * dv + d) = v;
  }
  if (out_f32) *reinterpret_cast<float4*>(out_f32 + orow * dv + d) = acc;
  if (tid == 0 && lse_out) lse_out[orow] = lse_n;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, bool pdl, void* stream) {
  if (a.n_groups == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_groups, a.rows, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const float*>(a.o_part),
                            static_cast<const float*>(a.lse_part), a.groups, 0, a.rows, a.dv, a.T,
                            a.Hq, a.G, a.out, static_cast<float*>(nullptr), a.lse, pdl ? 1 : 0);
}

cudaError_t launch_combine_raw(const float* o_part, const float* lse_part, int n_parts, int rows,
                               int dv, void* out_bf16, float* out_f32, float* lse_out,
                               void* stream) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(1, rows, 1), block(kCombineThreads, 1, 1);
  combine_kernel<<<grid, block, 0, static_cast<cudaStream_t>(stream)>>>(
      o_part, lse_part, nullptr, n_parts, rows, dv, 1, 1, 1, out_bf16, out_f32, lse_out, 0);
  return cudaGetLastError();
}

}  // namespace splitkv
