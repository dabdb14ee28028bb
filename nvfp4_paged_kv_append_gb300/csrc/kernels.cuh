// Kernel argument blocks and launch-shape constants shared by the kernel
// translation units and the C-ABI host code.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "codec.cuh"
#include "ptx.cuh"

namespace nvfp4kv {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;

struct AppendArgs {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int num_kv_heads;
  int64_t num_slots;  // num_pages * page_size
  uint8_t* k_data;
  uint8_t* k_scale;
  uint8_t* v_data;
  uint8_t* v_scale;
  float k_scale_g;
  float v_scale_g;
  uint64_t row_magic;  // ceil(2^40 / num_kv_heads): row / Hkv as a multiply-shift
  int* status;
};

struct QuantArgs {
  const void* x;
  int64_t rows;
  int mode;
  float global_scale;
  uint8_t* packed;
  uint8_t* scales;
  float* row_scales;
};

struct DequantArgs {
  const uint8_t* packed;
  const uint8_t* scales;
  int64_t rows;
  const float* row_scales;
  float global_scale;
  void* out;
};

// ---- decode --------------------------------------------------------------------
// Decode work items cover kDecSplit << k tokens (one partial result each),
// k = 0 .. kDecSplitSteps - 1, chosen per call by the schedule kernel; the
// workspace holds the partials of the shortest.
constexpr int kDecSplit = 1024;
constexpr int kDecSplitSteps = 4;
constexpr int kDecUnit = 256;    // tokens per shared-memory stage (16 pages)
constexpr int kDecWarps = 4;

struct DecodeArgs {
  const void* q;  // bf16 [B][Hq][128]
  const uint8_t* k_data;
  const uint8_t* k_scale;
  const uint8_t* v_data;
  const uint8_t* v_scale;
  const int32_t* page_table;
  const int32_t* kv_lens;
  int max_pages;
  int num_pages;
  int num_kv_heads;
  int num_q_heads;
  int max_splits;
  int batch;
  int ctas;           // CTAs of the attention grid (the schedule sizes items for it)
  int* sched;         // [0] item count, [1] claim counter, [2] split length; records (int4 b, h, split, n_tok) from sched + 4
  float k_g, v_g, sm_scale;
  void* o;            // bf16 [B][Hq][128]
  float* lse;         // optional [B][Hq]
  float* part_o;      // [B][max_splits][Hq][128]
  float* part_lse;    // [B][max_splits][Hq]  (log2 domain)
  int* status;
};

// ---- prefill -------------------------------------------------------------------
constexpr int kBM = 128;        // query rows per tile (tokens x grouped heads)
constexpr int kBN = 128;        // keys per KV tile (8 pages)
constexpr int kPagesPerTile = kBN / kPageSize;

struct PrefillArgs {
  const void* q;  // bf16 [total_q][Hq][128]
  const uint8_t* k_data;
  const uint8_t* k_scale;
  const uint8_t* v_data;
  const uint8_t* v_scale;
  const int32_t* page_table;
  const int32_t* kv_lens;
  const int32_t* qo_indptr;
  int64_t total_q;
  int batch;
  int max_pages;
  int num_pages;
  int num_kv_heads;
  int num_q_heads;
  int group;        // num_q_heads / num_kv_heads (power of two)
  int log2_group;
  int causal;
  float sm_scale, k_g, v_g;
  float q_g;        // A4Q query scale: 0 = per row (amax/2688), > 0 = this scale for every row
  void* o;          // bf16 [total_q][Hq][128]
  float* lse;       // optional [total_q][Hq]
  const int* work;  // [0] item count, [1] repacked tile count, [2] unit count; items (int4) from work + 4
  const int* tile_prefix;  // [batch+1] per-request KV-tile prefix (repack mode)
  const int4* units;       // split > 1: per unit (request, q tile << 8 | kv head, parts, 0)
  uint8_t* repack;         // repack mode: one record per (request, kv head, KV tile)
  float* part;             // split > 1: kPartFloats per partial slot (unit * split + part)
  int split;               // most KV parts per unit (1: no split)
  int max_units;           // bound on the number of units (grid of the merge)
  int* status;
};

// Split KV: at most kMaxSplit parts per unit, each of at least kMinSplitTiles
// KV tiles.
constexpr int kMaxSplit = 16;
constexpr int kMinSplitTiles = 4;

// A split item writes its unnormalized O (fp32, relative to its running max),
// running max (log2 units) and running sum into one partial slot:
// O [128 rows][128] | m [128] | l [128].
constexpr int kPartFloats = kBM * kHeadDim + 2 * kBM;

struct PlanArgs {
  const int32_t* kv_lens;
  const int32_t* qo_indptr;
  int64_t total_q;
  int batch;
  int max_pages;
  int num_kv_heads;
  int log2_group;
  int causal;
  int bn;     // keys per KV tile of the attention kernel the schedule is for
  int split;  // most KV parts per (request, q tile, kv head) unit (1: no split)
  int ctas;   // CTAs of the attention kernel (the plan picks the parts for them)
  int* work;  // output schedule
  int max_units;  // bound on the units (request, q tile, kv head)
  int max_items;  // max_units * split: room for items in the schedule
  int4* units;  // split > 1: unit table for the merge
  int* status;
};

// Per-device set-up and capability check of the current device (api.cu):
// NVFP4KV_OK, NVFP4KV_ERR_UNSUPPORTED (not sm_103) or NVFP4KV_ERR_CUDA.
int current_device_status();

// Kernels (defined in append.cu, decode.cu, prefill.cu).
__global__ void nvfp4_kv_append_kernel(AppendArgs a);
int append_ctas_per_sm();  // resident CTAs of 256 threads per SM of the append kernel
// FP8 cache write (same arguments; the scale pointers are unused, k_scale_g /
// v_scale_g are the per-tensor FP8 scales)
__global__ void fp8_kv_append_kernel(AppendArgs a);
__global__ void nvfp4_quantize_rows_kernel(QuantArgs a);
__global__ void nvfp4_dequantize_rows_kernel(DequantArgs a);

// Launchers that hide templates (decode.cu / prefill.cu).
cudaError_t launch_decode(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s);
// The same over an FP8 cache (k_data / v_data hold E4M3 codes, 128 B per token row).
cudaError_t launch_decode_fp8(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s);
// Schedule (+ repack pre-pass) and the attention kernel, launched separately.
cudaError_t launch_prefill_plan(const PrefillArgs& a, const PlanArgs& plan, int variant, bool repack, int num_sms,
                                cudaStream_t s);
cudaError_t launch_prefill_attend(const PrefillArgs& a, int variant, bool repack, int num_sms, cudaStream_t s);
// Split KV: merge the partial results of units split into several items.
cudaError_t launch_prefill_merge(const PrefillArgs& a, cudaStream_t s);
// FP8 cache: schedule, repack of the FP8 pages into dequant-ahead records
// (K BF16 | V FP16 per 128-key tile), then the dequant-ahead attention.
cudaError_t launch_prefill_fp8(const PrefillArgs& a, const PlanArgs& plan, int num_sms, cudaStream_t s);
// A4Q in repack mode: two CTAs per SM, 112-key tiles (prefill_a4q.cu).
// FP4 PV: repack record size (per 128-key tile) and the page re-layout
struct TokenMajorArgs {
  const uint8_t* v_data;
  const uint8_t* v_scale;
  const int32_t* page_ids;
  int n_ids;
  int num_pages;
  int num_kv_heads;
  uint8_t* codes;   // [n_ids][Hkv][128][8]
  uint8_t* scales;  // [n_ids][Hkv][128]
  int* status;
};
size_t prefill_fp4pv_record_bytes();
cudaError_t launch_v_token_major(const TokenMajorArgs& a, int num_sms, cudaStream_t s);
size_t prefill_a4q_2cta_record_bytes();
int prefill_a4q_2cta_tile_keys();
cudaError_t launch_prefill_a4q_2cta_repack(const PrefillArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_a4q_2cta(const PrefillArgs& a, int num_sms, cudaStream_t s);
// Sets a kernel's dynamic shared-memory limit (and, for the kernels that pair
// two CTAs per SM, the largest shared-memory carveout) once per device: the
// calls are host work that a short launch would otherwise wait on.
cudaError_t set_kernel_smem(const void* kernel, int bytes, bool max_carveout);

}  // namespace nvfp4kv
