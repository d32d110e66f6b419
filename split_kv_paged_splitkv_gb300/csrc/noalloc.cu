// splitkv_decode_noalloc: the decode call for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at all: code that
// runs inside another framework's memory budget, plugins whose host forbids
// device allocations after start-up, or real-time loops that must not risk an
// allocation stall or failure mid-step.  For them this entry point keeps the
// decode workspace (work list, merge tickets, partial outputs) in one
// file-scope device array instead of a caller buffer.
//
// The array is kNoAllocScratchBytes (16 MiB) and lives as long as the library
// is loaded: every GPU that loads the library holds it until the process exits.
// Host code may not use the array's name as an address (on the host it names a
// stand-in object, not device memory); its device address is fetched once per
// device with cudaGetSymbolAddress and passed to the kernels like any other
// workspace pointer.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace splitkv {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
splitkv_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SPLITKV_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(SPLITKV_EUNSUPPORTED, "device %d is beyond the %d devices supported", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(SPLITKV_ECUDA, "cudaGetSymbolAddress of the decode scratch array: %s",
                  cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SPLITKV_OK;
}

}  // namespace
}  // namespace splitkv

using namespace splitkv;

extern "C" splitkv_status splitkv_decode_noalloc(const splitkv_plan_t* plan, const void* q,
                                                 const void* k_pages, const void* v_pages,
                                                 const int32_t* block_table,
                                                 const int32_t* seq_lens, int32_t num_splits,
                                                 float scale, float kv_scale, void* out,
                                                 float* lse, void* stream) {
  if (!plan) return fail(SPLITKV_EINVAL, "plan is NULL");
  if (plan->total > kNoAllocScratchBytes)
    return fail(SPLITKV_EWORKSPACE,
                "this plan needs %zu bytes of scratch; splitkv_decode_noalloc holds at most %zu "
                "bytes (16 MiB) -- use splitkv_decode with a caller-allocated workspace",
                plan->total, kNoAllocScratchBytes);
  void* scratch = nullptr;
  splitkv_status st = scratch_for_current_device(&scratch);
  if (st != SPLITKV_OK) return st;
  // Every call re-writes the work list and zeroes the tickets and the status
  // word: the array still holds whatever the previous call left there.
  st = splitkv_plan_upload(plan, scratch, kNoAllocScratchBytes, stream);
  if (st != SPLITKV_OK) return st;
  // (a capacity plan's items are derived from the device lengths by the kernels)
  return splitkv_decode(plan, scratch, q, k_pages, v_pages, block_table, seq_lens, num_splits,
                        scale, kv_scale, out, lse, stream);
}

// The status word and per-CTA log of the last splitkv_decode_noalloc call on
// the current device live in the scratch array, whose address callers never
// see: this reads them the way splitkv_read_stats reads a caller workspace.
extern "C" splitkv_status splitkv_noalloc_read_stats(const splitkv_plan_t* plan,
                                                     int32_t* cta_log_host, int32_t capacity,
                                                     int32_t* status_host, void* stream) {
  if (!plan) return fail(SPLITKV_EINVAL, "plan is NULL");
  if (plan->total > kNoAllocScratchBytes)
    return fail(SPLITKV_EWORKSPACE,
                "this plan needs %zu bytes of scratch, more than splitkv_decode_noalloc holds "
                "(%zu bytes), so it never ran there",
                plan->total, kNoAllocScratchBytes);
  void* scratch = nullptr;
  splitkv_status st = scratch_for_current_device(&scratch);
  if (st != SPLITKV_OK) return st;
  return splitkv_read_stats(plan, scratch, cta_log_host, capacity, status_host, stream);
}
