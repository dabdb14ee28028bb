// Paged prefill for callers that cannot allocate device memory.
//
// nvfp4_paged_prefill() takes a caller-provided workspace for its work
// schedule.  Some callers have no way to provide one: an inference engine that
// plans every device buffer up front and forbids cudaMalloc on its serving
// path (an allocation can synchronize the device and stall other streams), or
// a host framework that hands a kernel plugin its inputs and outputs but no
// scratch pointer.  This entry point keeps the schedule in a fixed-size
// array compiled into the library instead, so it allocates nothing.
//
// Only the schedule lives in the array: the call always runs the in-kernel
// mode of the prefill (V dequantized inside the attention kernel), never the
// repack mode whose per-tile records would need far more room.  Its results
// are bit for bit those of nvfp4_paged_prefill() given a schedule-only
// workspace.
//
// The array lives in every GPU that loads the library until the process exits
// (kNoAllocScratchBytes per device).  Its device address is looked up once
// per device, with that device current, on the first call; make that first
// call before any stream capture.  The cached address assumes one CUDA
// context per device for the life of the process (a cudaDeviceReset followed
// by further calls is not supported).  Every call shares the one array and it
// keeps the last call's contents: the schedule kernel rewrites all of it that
// a call reads, so nothing has to start at zero, but two calls whose work
// overlaps on the GPU (different streams without ordering between them) race
// on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.cuh"
#include "nvfp4kv.h"

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB: ~65,000 (request, q tile, kv head) units

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device; the host-side symbol itself is not a device address).  The
// device must already have passed the library's capability check.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return NVFP4KV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return NVFP4KV_OK;
}

}  // namespace

extern "C" {

size_t nvfp4_paged_prefill_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

int nvfp4_paged_prefill_noalloc(const void* q, int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                                const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                                const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale,
                                int32_t variant, float q_global_scale, void* o, float* lse, void* stream) {
  if (!cache || num_q_heads <= 0 || cache->num_kv_heads <= 0) return NVFP4KV_ERR_ARG;
  // the schedule alone: a workspace of exactly this size pins in-kernel mode
  const size_t need =
      nvfp4_workspace_bytes(NVFP4KV_OP_PREFILL, batch, num_q_heads, cache->num_kv_heads, total_q, 0);
  if (need == 0 && (batch != 0 || total_q != 0)) return NVFP4KV_ERR_ARG;
  if (need > kNoAllocScratchBytes) return NVFP4KV_ERR_WORKSPACE;  // schedule would not fit the static scratch
  // An unsupported device is reported as such before the symbol lookup,
  // which would fail there for want of an sm_103a image.
  int rc = nvfp4kv::current_device_status();
  if (rc) return rc;
  void* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch))) return rc;
  return nvfp4_paged_prefill(q, total_q, num_q_heads, cache, page_table, max_pages_per_req, kv_lens, qo_indptr,
                             batch, causal, sm_scale, variant, q_global_scale, o, lse, scratch, need, stream);
}

}  // extern "C"
