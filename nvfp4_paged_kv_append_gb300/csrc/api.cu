// C ABI of libnvfp4kv.so: argument validation on the host, the device status
// word, and kernel launches.  No entry point
// allocates device memory; nothing throws across the boundary.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.cuh"
#include "nvfp4kv.h"

using namespace nvfp4kv;

namespace {

__device__ int g_status_word;  // bit set of kDev* conditions, read + cleared by nvfp4kv_get_device_status

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool init = false;
  int rc = NVFP4KV_OK;
  int num_sms = 0;
  int append_ctas = 1;    // resident append CTAs per SM
  int* status = nullptr;  // device address of g_status_word on this device
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Kernels whose shared-memory attributes are set on a device.
struct KernelAttr {
  int dev;
  const void* kernel;
  int bytes;
};
std::mutex g_attr_mu;
KernelAttr g_attr[256];
int g_n_attr = 0;

// Per-device set-up on first use (device current): capability check, SM
// count, status word address.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return NVFP4KV_ERR_CUDA;
    }
    d.num_sms = sms;
    if (major != 10 || minor != 3) {
      d.rc = NVFP4KV_ERR_UNSUPPORTED;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return NVFP4KV_ERR_CUDA;
      d.status = static_cast<int*>(p);
      d.append_ctas = append_ctas_per_sm();
      d.rc = NVFP4KV_OK;
    }
    d.init = true;
  }
  *out = &d;
  return d.rc;
}

}  // namespace

// Capability check of the current device for code outside this file (the
// allocation-free entry point checks the device before it touches its
// static array): NVFP4KV_OK, NVFP4KV_ERR_UNSUPPORTED or NVFP4KV_ERR_CUDA.
int nvfp4kv::current_device_status() {
  DeviceState* d = nullptr;
  return device_state(&d);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool finite_pos(float x) { return std::isfinite(x) && x > 0.0f; }

int check_cache(const nvfp4kv_cache_t* c) {
  if (!c) return NVFP4KV_ERR_ARG;
  if (!c->k_data || !c->k_scale || !c->v_data || !c->v_scale) return NVFP4KV_ERR_ARG;
  if (!aligned16(c->k_data) || !aligned16(c->k_scale) || !aligned16(c->v_data) || !aligned16(c->v_scale))
    return NVFP4KV_ERR_ARG;
  if (c->page_size != kPageSize || c->head_dim != kHeadDim) return NVFP4KV_ERR_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->num_kv_heads > 255) return NVFP4KV_ERR_ARG;
  if (static_cast<int64_t>(c->num_pages) * c->num_kv_heads * kPageSize >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  if (!finite_pos(c->k_global_scale) || !finite_pos(c->v_global_scale)) return NVFP4KV_ERR_ARG;
  return NVFP4KV_OK;
}

int check_fp8_cache(const fp8kv_cache_t* c) {
  if (!c) return NVFP4KV_ERR_ARG;
  if (!c->k_data || !c->v_data || !aligned16(c->k_data) || !aligned16(c->v_data)) return NVFP4KV_ERR_ARG;
  if (c->page_size != kPageSize || c->head_dim != kHeadDim) return NVFP4KV_ERR_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->num_kv_heads > 255) return NVFP4KV_ERR_ARG;
  if (static_cast<int64_t>(c->num_pages) * c->num_kv_heads * kPageSize >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  if (!finite_pos(c->k_scale) || !finite_pos(c->v_scale)) return NVFP4KV_ERR_ARG;
  return NVFP4KV_OK;
}

// One layer's cache as the kernels see it: NVFP4 (codes + block scales +
// per-tensor scales) or FP8 (codes + per-tensor scales, no scale pools).
struct CacheView {
  const uint8_t *k_data, *k_scale, *v_data, *v_scale;
  int num_pages, num_kv_heads;
  float k_g, v_g;
  bool fp8;
};

CacheView view_of(const nvfp4kv_cache_t* c) {
  return CacheView{static_cast<const uint8_t*>(c->k_data), static_cast<const uint8_t*>(c->k_scale),
                   static_cast<const uint8_t*>(c->v_data), static_cast<const uint8_t*>(c->v_scale),
                   c->num_pages, c->num_kv_heads, c->k_global_scale, c->v_global_scale, false};
}

CacheView view_of(const fp8kv_cache_t* c) {
  return CacheView{static_cast<const uint8_t*>(c->k_data), nullptr, static_cast<const uint8_t*>(c->v_data), nullptr,
                   c->num_pages, c->num_kv_heads, c->k_scale, c->v_scale, true};
}

int log2_exact(int x) {
  if (x <= 0 || (x & (x - 1)) != 0) return -1;
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

int64_t prefill_max_items(int64_t total_q, int batch, int num_q_heads, int num_kv_heads) {
  const int64_t group = num_q_heads / num_kv_heads;
  return (static_cast<int64_t>((total_q * group + kBM - 1) / kBM) + batch) * num_kv_heads;
}

// Prefill workspace: [16 B header][items: 16 B each][unit prefix][tile
// prefix][unit table: 16 B per unit, split KV only] padded to 1 KB, then
// (repack mode) one record for every (request, kv head, KV tile) the batch can
// hold: 64 KB per 128-key tile for the dequant-ahead kernel, 37 KB per 112-key
// tile for the A4Q kernel; then (split KV) one partial slot per (unit, part).
constexpr size_t kRepackRecordBytesDq = 65536;
size_t prefill_repack_bytes(int variant, int batch, int num_kv_heads, int64_t max_kv_len);
int64_t units_table_offset(int64_t max_items, int batch) {  // in ints, 16-byte aligned
  return (4 + 4 * max_items + 2 * (static_cast<int64_t>(batch) + 1) + 3) & ~int64_t(3);
}
size_t prefill_sched_bytes(int64_t max_units, int split, int batch) {
  const int64_t max_items = max_units * split;
  size_t b = 4 * static_cast<size_t>(units_table_offset(max_items, batch));
  if (split > 1) b += 16 * static_cast<size_t>(max_units);
  return (b + 1023) & ~size_t(1023);
}
size_t prefill_part_bytes(int64_t max_units, int split) {
  return split > 1 ? static_cast<size_t>(max_units) * split * kPartFloats * sizeof(float) : 0;
}
// Split KV: when the (request, q tile, kv head) units are fewer than the CTAs
// of the attention kernel, each unit's KV range may be cut into parts (the
// plan picks how many for the actual units); this is the most parts the
// workspace is laid out for.  Workspace sizing assumes the kernels with one
// CTA per SM on 152 SMs and 128-key tiles; with more SMs at run time the
// split shrinks to what the workspace holds.
constexpr int kSplitSizingCtas = 152;
int split_cap(int64_t max_units, int64_t max_tiles, int ctas) {
  if (max_units <= 0 || max_units >= ctas) return 1;
  int64_t s = (4 * ctas + max_units - 1) / max_units;  // room for about four items per CTA
  if (s > kMaxSplit) s = kMaxSplit;
  if (s > max_tiles / kMinSplitTiles) s = max_tiles / kMinSplitTiles;
  return s > 1 ? static_cast<int>(s) : 1;
}
size_t prefill_repack_tiles(int batch, int num_kv_heads, int64_t max_kv_len, int bn) {
  if (max_kv_len <= 0) return 0;
  return static_cast<size_t>(batch) * num_kv_heads * static_cast<size_t>((max_kv_len + bn - 1) / bn);
}
// Keys per KV tile of the attention kernel that runs (variant, mode).
int prefill_tile_keys(int variant, bool repack) { return (variant == 0 && repack) ? prefill_a4q_2cta_tile_keys() : kBN; }
size_t prefill_repack_bytes(int variant, int batch, int num_kv_heads, int64_t max_kv_len) {
  if (variant == NVFP4KV_VARIANT_A4Q)
    return prefill_a4q_2cta_record_bytes() *
           prefill_repack_tiles(batch, num_kv_heads, max_kv_len, prefill_a4q_2cta_tile_keys());
  if (variant == NVFP4KV_VARIANT_A4Q_FP4PV)
    return prefill_fp4pv_record_bytes() * prefill_repack_tiles(batch, num_kv_heads, max_kv_len, kBN);
  return kRepackRecordBytesDq * prefill_repack_tiles(batch, num_kv_heads, max_kv_len, kBN);
}

}  // namespace

cudaError_t nvfp4kv::set_kernel_smem(const void* kernel, int bytes, bool max_carveout) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (int i = 0; i < g_n_attr; ++i)
    if (g_attr[i].dev == dev && g_attr[i].kernel == kernel && g_attr[i].bytes == bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && max_carveout)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && g_n_attr < 256) g_attr[g_n_attr++] = {dev, kernel, bytes};
  return e;
}

namespace {

int launch_rc(cudaError_t e) { return e == cudaSuccess ? NVFP4KV_OK : NVFP4KV_ERR_CUDA; }

// Decode workspace starts with the item schedule: a 16-byte header, then one
// 16-byte record per (request, kv head, split).
size_t decode_sched_bytes(int batch, int num_kv_heads, size_t splits) {
  return 16 + 16 * static_cast<size_t>(batch) * num_kv_heads * splits;
}

// A wait that can only end by its time limit (nothing arrives on `bar`).
__global__ void nvfp4_debug_wait_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_barrier_init();
  mbar_wait(&bar, 0, status, limit_ns);
}

// Cache write of either format: validation of the tensors, one persistent
// wave of the format's append kernel.
int append_impl(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, const CacheView& c,
                void* stream) {
  int rc;
  if (num_tokens < 0) return NVFP4KV_ERR_ARG;
  if (num_tokens == 0) return NVFP4KV_OK;
  if (!k || !v || !slot_mapping || !aligned16(k) || !aligned16(v)) return NVFP4KV_ERR_ARG;
  const int64_t rows = num_tokens * c.num_kv_heads;
  if (num_tokens >= (int64_t(1) << 31) || rows >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  AppendArgs a;
  a.k = k;
  a.v = v;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.num_kv_heads = c.num_kv_heads;
  a.num_slots = static_cast<int64_t>(c.num_pages) * kPageSize;
  a.k_data = const_cast<uint8_t*>(c.k_data);
  a.k_scale = const_cast<uint8_t*>(c.k_scale);
  a.v_data = const_cast<uint8_t*>(c.v_data);
  a.v_scale = const_cast<uint8_t*>(c.v_scale);
  a.k_scale_g = c.k_g;
  a.v_scale_g = c.v_g;
  a.row_magic = ((uint64_t(1) << 40) + c.num_kv_heads - 1) / c.num_kv_heads;
  a.status = d->status;
  // one persistent wave (as many CTAs of 256 threads as fit on every SM);
  // each warp step covers four rows, 2 * rows rows of K and V in all
  const int64_t warps = (2 * rows + 3) / 4;
  const int64_t want = (warps + 7) / 8;
  const int64_t cap = static_cast<int64_t>(d->num_sms) * d->append_ctas;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (c.fp8) fp8_kv_append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  else nvfp4_kv_append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_rc(cudaGetLastError());
}

}  // namespace

extern "C" {

size_t nvfp4_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (num_pages <= 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0) return 0;
  return 2ull * static_cast<size_t>(num_pages) * page_size * num_kv_heads * (head_dim / 2 + head_dim / 16);
}

size_t nvfp4_workspace_bytes(int32_t op, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int64_t total_q,
                             int32_t max_kv_len) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
  if (op == NVFP4KV_OP_PREFILL) {
    if (total_q < 0) return 0;
    const int64_t units = prefill_max_items(total_q, batch, num_q_heads, num_kv_heads);
    size_t rec = 0;  // the largest records of any variant
    for (int v : {NVFP4KV_VARIANT_A4Q, NVFP4KV_VARIANT_DQ_AHEAD, NVFP4KV_VARIANT_A4Q_FP4PV}) {
      const size_t r = prefill_repack_bytes(v, batch, num_kv_heads, max_kv_len);
      rec = r > rec ? r : rec;
    }
    const int split = split_cap(units, max_kv_len > 0 ? (max_kv_len + kBN - 1) / kBN : 0, kSplitSizingCtas);
    return prefill_sched_bytes(units, split, batch) + rec + prefill_part_bytes(units, split);
  }
  if (op == NVFP4KV_OP_DECODE) {
    if (max_kv_len < 0) return 0;
    const size_t splits = (static_cast<size_t>(max_kv_len) + kDecSplit - 1) / kDecSplit;
    return decode_sched_bytes(batch, num_kv_heads, splits) +
           static_cast<size_t>(batch) * splits * num_q_heads * (kHeadDim + 1) * sizeof(float);
  }
  return 0;
}

int nvfp4_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                    const nvfp4kv_cache_t* cache, void* stream) {
  const int rc = check_cache(cache);
  if (rc) return rc;
  return append_impl(k, v, slot_mapping, num_tokens, view_of(cache), stream);
}

int fp8_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                  const fp8kv_cache_t* cache, void* stream) {
  const int rc = check_fp8_cache(cache);
  if (rc) return rc;
  return append_impl(k, v, slot_mapping, num_tokens, view_of(cache), stream);
}

}  // extern "C"

namespace {

enum PrefillStage { kStagePlan = 1, kStageRun = 2 };

// Validates the arguments, fills the kernel argument blocks and launches the
// requested stages.  q/o/lse/sm_scale are only used by the run stage.  An FP8
// cache always runs in repack mode (records converted once per KV tile, then
// the dequant-ahead attention), so its workspace must hold the records.
int prefill_stages(int stages, const void* q, int64_t total_q, int32_t num_q_heads, const CacheView& c,
                   const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                   const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale, int32_t variant,
                   float q_global_scale, void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  int rc;
  if (batch < 0 || total_q < 0 || max_pages_per_req <= 0) return NVFP4KV_ERR_ARG;
  if (num_q_heads <= 0 || num_q_heads % c.num_kv_heads != 0) return NVFP4KV_ERR_ARG;
  const int lg = log2_exact(num_q_heads / c.num_kv_heads);
  if (lg < 0 || lg > 7) return NVFP4KV_ERR_ARG;
  if (causal != 0 && causal != 1) return NVFP4KV_ERR_ARG;
  if (variant != NVFP4KV_VARIANT_A4Q && variant != NVFP4KV_VARIANT_DQ_AHEAD && variant != NVFP4KV_VARIANT_A4Q_FP4PV)
    return NVFP4KV_ERR_ARG;
  const bool fp4pv = variant == NVFP4KV_VARIANT_A4Q_FP4PV;
  if (fp4pv && c.fp8) return NVFP4KV_ERR_ARG;
  if ((stages & kStageRun) && !std::isfinite(sm_scale)) return NVFP4KV_ERR_ARG;
  if (!std::isfinite(q_global_scale) || q_global_scale < 0.0f) return NVFP4KV_ERR_ARG;
  if (total_q * num_q_heads >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  if (batch == 0 || total_q == 0) return NVFP4KV_OK;
  if (!page_table || !kv_lens || !qo_indptr) return NVFP4KV_ERR_ARG;
  if ((stages & kStageRun) && (!q || !o || !aligned16(q) || !aligned16(o))) return NVFP4KV_ERR_ARG;
  const int64_t max_units = prefill_max_items(total_q, batch, num_q_heads, c.num_kv_heads);
  if (max_units >= (int64_t(1) << 30) / kMaxSplit) return NVFP4KV_ERR_ARG;
  const int64_t max_kv = static_cast<int64_t>(max_pages_per_req) * kPageSize;
  if (max_kv / prefill_a4q_2cta_tile_keys() >= 65535) return NVFP4KV_ERR_ARG;  // tile indices fit 16 bits
  const size_t sched1 = prefill_sched_bytes(max_units, 1, batch);
  if (!workspace || !aligned16(workspace) || workspace_bytes < sched1) return NVFP4KV_ERR_WORKSPACE;
  // Repack mode (each V tile dequantized once, into the workspace) when the
  // workspace holds a tile for every (request, kv head, KV tile) the page
  // table allows and each record would be read by enough q tiles: requests
  // average at least eight q tiles per kv head for A4Q, two for dequant-ahead
  // (whose in-kernel mode converts K as well).  (A4Q on GB300, whole calls:
  // six q tiles per kv head, 4 x 192 over 2K, in-kernel 52.9 against repack
  // 56.0 us; eight, 4 x 256 over 4K, 80.5 against 81.5 us; sixteen, 2 x 512
  // over 8K, repack 122.5 against 131.7 us.)
  const size_t rbytes = prefill_repack_bytes(variant, batch, c.num_kv_heads, max_kv);
  const int64_t qtiles = (total_q * (num_q_heads / c.num_kv_heads) + kBM - 1) / kBM;
  const int64_t min_qtiles = variant == NVFP4KV_VARIANT_A4Q ? 8 : 2;
  bool repack = workspace_bytes >= sched1 + rbytes && qtiles >= min_qtiles * batch;
  if (c.fp8 || fp4pv) {  // these read only repacked records
    if (workspace_bytes < sched1 + rbytes) return NVFP4KV_ERR_WORKSPACE;
    repack = true;
  }
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  // Split KV when the units are fewer than the attention kernel's CTAs and
  // the workspace has room for the partial results -- for the kernels with
  // one CTA per SM.  (On the two-CTA A4Q kernel of repack mode, measured on
  // 4 x 128 queries over 2K keys, the split items' prologues and the merge
  // cost more than the parallelism gained: 61 against 54 us.)
  const int bn = prefill_tile_keys(variant, repack);
  const bool two_cta = repack && variant == NVFP4KV_VARIANT_A4Q && !c.fp8;
  const int ctas = d->num_sms;
  // (The FP4 PV variant codes P against a reference that each KV range
  // would restart, so it always runs each unit whole.)
  int split = (two_cta || fp4pv) ? 1 : split_cap(max_units, (max_kv + bn - 1) / bn, ctas);
  while (split > 1 && workspace_bytes < prefill_sched_bytes(max_units, split, batch) + (repack ? rbytes : 0) +
                                            prefill_part_bytes(max_units, split))
    --split;
  const int64_t max_items = max_units * split;
  const size_t sched = prefill_sched_bytes(max_units, split, batch);

  PlanArgs plan;
  plan.kv_lens = kv_lens;
  plan.qo_indptr = qo_indptr;
  plan.total_q = total_q;
  plan.batch = batch;
  plan.max_pages = max_pages_per_req;
  plan.num_kv_heads = c.num_kv_heads;
  plan.log2_group = lg;
  plan.causal = causal;
  plan.bn = bn;
  plan.split = split;
  plan.ctas = ctas;
  plan.work = static_cast<int*>(workspace);
  plan.max_units = static_cast<int>(max_units);
  plan.max_items = static_cast<int>(max_items);
  plan.units = split > 1 ? reinterpret_cast<int4*>(static_cast<int*>(workspace) + units_table_offset(max_items, batch))
                         : nullptr;
  plan.status = d->status;

  PrefillArgs a;
  a.q = q;
  a.k_data = c.k_data;
  a.k_scale = c.k_scale;
  a.v_data = c.v_data;
  a.v_scale = c.v_scale;
  a.page_table = page_table;
  a.kv_lens = kv_lens;
  a.qo_indptr = qo_indptr;
  a.total_q = total_q;
  a.batch = batch;
  a.max_pages = max_pages_per_req;
  a.num_pages = c.num_pages;
  a.num_kv_heads = c.num_kv_heads;
  a.num_q_heads = num_q_heads;
  a.group = 1 << lg;
  a.log2_group = lg;
  a.causal = causal;
  a.sm_scale = sm_scale;
  a.k_g = c.k_g;
  a.v_g = c.v_g;
  a.q_g = variant != NVFP4KV_VARIANT_DQ_AHEAD ? q_global_scale : 0.0f;
  a.o = o;
  a.lse = lse;
  a.work = static_cast<const int*>(workspace);
  a.tile_prefix = static_cast<const int*>(workspace) + 4 + 4 * max_items + (batch + 1);
  a.units = plan.units;
  a.repack = repack ? static_cast<uint8_t*>(workspace) + sched : nullptr;
  a.part = split > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + sched + (repack ? rbytes : 0))
                     : nullptr;
  a.split = split;
  a.max_units = static_cast<int>(max_units);
  a.status = d->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.fp8) return launch_rc(launch_prefill_fp8(a, plan, d->num_sms, st));  // plan + repack + attention (+ merge)
  if (stages & kStagePlan) {
    if ((rc = launch_rc(launch_prefill_plan(a, plan, variant, repack, d->num_sms, st)))) return rc;
  }
  if (stages & kStageRun) {
    if ((rc = launch_rc(launch_prefill_attend(a, variant, repack, d->num_sms, st)))) return rc;
    if (split > 1) return launch_rc(launch_prefill_merge(a, st));
  }
  return NVFP4KV_OK;
}

// Paged decode of either format.
int decode_impl(const void* q, int32_t num_q_heads, const CacheView& c, const int32_t* page_table,
                int32_t max_pages_per_req, const int32_t* kv_lens, int32_t batch, float sm_scale, void* o, float* lse,
                void* workspace, size_t workspace_bytes, void* stream) {
  int rc;
  if (batch < 0 || max_pages_per_req <= 0) return NVFP4KV_ERR_ARG;
  if (num_q_heads <= 0 || num_q_heads % c.num_kv_heads != 0) return NVFP4KV_ERR_ARG;
  const int lg = log2_exact(num_q_heads / c.num_kv_heads);
  if (lg < 0 || lg > 4) return NVFP4KV_ERR_ARG;
  if (!std::isfinite(sm_scale)) return NVFP4KV_ERR_ARG;
  if (batch == 0) return NVFP4KV_OK;
  if (!q || !o || !page_table || !kv_lens || !aligned16(q) || !aligned16(o)) return NVFP4KV_ERR_ARG;
  const int64_t max_kv = static_cast<int64_t>(max_pages_per_req) * kPageSize;
  if (max_kv >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  const size_t need = nvfp4_workspace_bytes(NVFP4KV_OP_DECODE, batch, num_q_heads, c.num_kv_heads, 0,
                                            static_cast<int32_t>(max_kv));
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return NVFP4KV_ERR_WORKSPACE;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  DecodeArgs a;
  a.q = q;
  a.k_data = c.k_data;
  a.k_scale = c.k_scale;
  a.v_data = c.v_data;
  a.v_scale = c.v_scale;
  a.page_table = page_table;
  a.kv_lens = kv_lens;
  a.max_pages = max_pages_per_req;
  a.num_pages = c.num_pages;
  a.num_kv_heads = c.num_kv_heads;
  a.num_q_heads = num_q_heads;
  a.max_splits = static_cast<int>((max_kv + kDecSplit - 1) / kDecSplit);
  a.k_g = c.k_g;
  a.v_g = c.v_g;
  a.sm_scale = sm_scale;
  a.o = o;
  a.lse = lse;
  a.batch = batch;
  a.sched = static_cast<int*>(workspace);
  float* ws = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       decode_sched_bytes(batch, c.num_kv_heads, a.max_splits));
  a.part_o = ws;
  a.part_lse = ws + static_cast<size_t>(batch) * a.max_splits * num_q_heads * kHeadDim;
  a.status = d->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return launch_rc(c.fp8 ? launch_decode_fp8(a, batch, d->num_sms, st) : launch_decode(a, batch, d->num_sms, st));
}

}  // namespace

extern "C" {

int nvfp4_paged_prefill(const void* q, int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                        const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                        const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale, int32_t variant,
                        float q_global_scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream) {
  const int rc = check_cache(cache);
  if (rc) return rc;
  return prefill_stages(kStagePlan | kStageRun, q, total_q, num_q_heads, view_of(cache), page_table,
                        max_pages_per_req, kv_lens, qo_indptr, batch, causal, sm_scale, variant, q_global_scale, o,
                        lse, workspace, workspace_bytes, stream);
}

int nvfp4_paged_prefill_plan(int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                             const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                             const int32_t* qo_indptr, int32_t batch, int32_t causal, int32_t variant,
                             void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = check_cache(cache);
  if (rc) return rc;
  return prefill_stages(kStagePlan, nullptr, total_q, num_q_heads, view_of(cache), page_table, max_pages_per_req,
                        kv_lens, qo_indptr, batch, causal, 0.0f, variant, 0.0f, nullptr, nullptr, workspace,
                        workspace_bytes, stream);
}

int nvfp4_paged_prefill_run(const void* q, int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                            const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                            const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale,
                            int32_t variant, float q_global_scale, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  const int rc = check_cache(cache);
  if (rc) return rc;
  return prefill_stages(kStageRun, q, total_q, num_q_heads, view_of(cache), page_table, max_pages_per_req, kv_lens,
                        qo_indptr, batch, causal, sm_scale, variant, q_global_scale, o, lse, workspace,
                        workspace_bytes, stream);
}

int nvfp4_paged_decode(const void* q, int32_t num_q_heads, const nvfp4kv_cache_t* cache, const int32_t* page_table,
                       int32_t max_pages_per_req, const int32_t* kv_lens, int32_t batch, float sm_scale, void* o,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = check_cache(cache);
  if (rc) return rc;
  return decode_impl(q, num_q_heads, view_of(cache), page_table, max_pages_per_req, kv_lens, batch, sm_scale, o, lse,
                     workspace, workspace_bytes, stream);
}

size_t fp8_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (num_pages <= 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return 2ull * static_cast<size_t>(num_pages) * page_size * num_kv_heads * head_dim;
}

size_t fp8_workspace_bytes(int32_t op, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int64_t total_q,
                           int32_t max_kv_len) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
  if (op == NVFP4KV_OP_PREFILL) {
    if (total_q < 0 || max_kv_len <= 0) return 0;
    const int64_t units = prefill_max_items(total_q, batch, num_q_heads, num_kv_heads);
    const int split = split_cap(units, (max_kv_len + kBN - 1) / kBN, kSplitSizingCtas);
    return prefill_sched_bytes(units, split, batch) + prefill_repack_bytes(1, batch, num_kv_heads, max_kv_len) +
           prefill_part_bytes(units, split);
  }
  return nvfp4_workspace_bytes(op, batch, num_q_heads, num_kv_heads, total_q, max_kv_len);
}

int fp8_paged_prefill(const void* q, int64_t total_q, int32_t num_q_heads, const fp8kv_cache_t* cache,
                      const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                      const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale, void* o, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = check_fp8_cache(cache);
  if (rc) return rc;
  return prefill_stages(kStagePlan | kStageRun, q, total_q, num_q_heads, view_of(cache), page_table,
                        max_pages_per_req, kv_lens, qo_indptr, batch, causal, sm_scale, NVFP4KV_VARIANT_DQ_AHEAD,
                        0.0f, o, lse, workspace, workspace_bytes, stream);
}

int fp8_paged_decode(const void* q, int32_t num_q_heads, const fp8kv_cache_t* cache, const int32_t* page_table,
                     int32_t max_pages_per_req, const int32_t* kv_lens, int32_t batch, float sm_scale, void* o,
                     float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = check_fp8_cache(cache);
  if (rc) return rc;
  return decode_impl(q, num_q_heads, view_of(cache), page_table, max_pages_per_req, kv_lens, batch, sm_scale, o, lse,
                     workspace, workspace_bytes, stream);
}

int nvfp4_quantize_rows(const void* x, int64_t rows, int32_t mode, float global_scale, void* packed, void* scales,
                        float* row_scales, void* stream) {
  if (rows < 0 || (mode != NVFP4KV_QUANT_GLOBAL && mode != NVFP4KV_QUANT_PER_ROW)) return NVFP4KV_ERR_ARG;
  if (mode == NVFP4KV_QUANT_GLOBAL && !finite_pos(global_scale)) return NVFP4KV_ERR_ARG;
  if (rows == 0) return NVFP4KV_OK;
  if (!x || !packed || !scales || !aligned16(x) || (reinterpret_cast<uintptr_t>(packed) & 7u)) return NVFP4KV_ERR_ARG;
  if (mode == NVFP4KV_QUANT_PER_ROW && !row_scales) return NVFP4KV_ERR_ARG;
  if (rows * 32 / 256 + 1 >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  DeviceState* d = nullptr;
  int rc;
  if ((rc = device_state(&d))) return rc;
  QuantArgs a{x, rows, mode, global_scale, static_cast<uint8_t*>(packed), static_cast<uint8_t*>(scales), row_scales};
  nvfp4_quantize_rows_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_rc(cudaGetLastError());
}

int nvfp4_dequantize_rows(const void* packed, const void* scales, int64_t rows, const float* row_scales,
                          float global_scale, void* out, void* stream) {
  if (rows < 0) return NVFP4KV_ERR_ARG;
  if (!row_scales && !finite_pos(global_scale)) return NVFP4KV_ERR_ARG;
  if (rows == 0) return NVFP4KV_OK;
  if (!packed || !scales || !out || (reinterpret_cast<uintptr_t>(packed) & 3u) || !aligned16(out)) return NVFP4KV_ERR_ARG;
  if (rows * 16 / 256 + 1 >= (int64_t(1) << 31)) return NVFP4KV_ERR_ARG;
  DeviceState* d = nullptr;
  int rc;
  if ((rc = device_state(&d))) return rc;
  DequantArgs a{static_cast<const uint8_t*>(packed), static_cast<const uint8_t*>(scales), rows, row_scales,
                global_scale, out};
  nvfp4_dequantize_rows_kernel<<<static_cast<unsigned>((rows * 16 + 255) / 256), 256, 0,
                                 static_cast<cudaStream_t>(stream)>>>(a);
  return launch_rc(cudaGetLastError());
}

int nvfp4_v_token_major(const nvfp4kv_cache_t* cache, const int32_t* page_ids, int32_t num_ids, void* codes,
                        void* scales, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (num_ids < 0) return NVFP4KV_ERR_ARG;
  if (num_ids == 0) return NVFP4KV_OK;
  if (!page_ids || !codes || !scales || (reinterpret_cast<uintptr_t>(codes) & 7u)) return NVFP4KV_ERR_ARG;
  if (static_cast<int64_t>(num_ids) * cache->num_kv_heads * kHeadDim >= (int64_t(1) << 40)) return NVFP4KV_ERR_ARG;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  TokenMajorArgs a{static_cast<const uint8_t*>(cache->v_data), static_cast<const uint8_t*>(cache->v_scale), page_ids,
                   num_ids, cache->num_pages, cache->num_kv_heads, static_cast<uint8_t*>(codes),
                   static_cast<uint8_t*>(scales), d->status};
  return launch_rc(launch_v_token_major(a, d->num_sms, static_cast<cudaStream_t>(stream)));
}

int nvfp4kv_get_device_status(void* stream) {
  DeviceState* d = nullptr;
  int rc;
  if ((rc = device_state(&d))) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return NVFP4KV_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NVFP4KV_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return NVFP4KV_ERR_CUDA;
  if (word & kDevTimeout) return NVFP4KV_ERR_TIMEOUT;
  if (word & (kDevBadPage | kDevBadSlot)) return NVFP4KV_ERR_DEVICE_INDEX;
  if (word & kDevBadShape) return NVFP4KV_ERR_SHAPE;
  return NVFP4KV_OK;
}

const char* nvfp4kv_status_string(int status) {
  switch (status) {
    case NVFP4KV_OK: return "ok";
    case NVFP4KV_ERR_ARG: return "invalid argument";
    case NVFP4KV_ERR_SHAPE: return "invalid request shape (q_len > kv_len for causal, or kv_len beyond the page table)";
    case NVFP4KV_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4KV_ERR_CUDA: return "CUDA call failed";
    case NVFP4KV_ERR_TIMEOUT: return "device pipeline wait timed out";
    case NVFP4KV_ERR_DEVICE_INDEX: return "page id or slot out of range";
    case NVFP4KV_ERR_UNSUPPORTED: return "device is not sm_103";
    default: return "unknown status";
  }
}

int nvfp4kv_debug_wait_timeout(uint32_t limit_ns, void* stream) {
  DeviceState* d = nullptr;
  int rc;
  if ((rc = device_state(&d))) return rc;
  uint64_t lim = limit_ns < 1000u ? 1000u : limit_ns;
  if (lim > 1000000000ull) lim = 1000000000ull;
  nvfp4_debug_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(lim, d->status);
  return launch_rc(cudaGetLastError());
}

const char* nvfp4kv_version(void) { return "nvfp4kv 0.1 sm_103a"; }

}  // extern "C"
