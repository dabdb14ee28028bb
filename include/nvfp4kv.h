/*
 * nvfp4kv -- NVFP4 paged KV cache: append, A4Q paged prefill, paged decode.
 * C ABI of libnvfp4kv.so (built for sm_103a only).
 *
 * The cache format is the one described on "NVFP4 KV cache prefill vs decode
 * performance", section "NVFP4 stores 4.5 bits per value before padding"
 * (packed E2M1 pairs, one E4M3 scale per 16 values) and "NVFP4 KV cache vs
 * NVFP4 weights", section "NVFP4 KV cache vs NVFP4 weights" (a second,
 * per-tensor FP32 scale).  Per layer the caller owns four device pools:
 *
 *   k_data, v_data   uint8 [num_pages][num_kv_heads][page_size][head_dim/2]
 *                    two E2M1 codes per byte, element 2i in the low nibble
 *   k_scale, v_scale uint8 [num_pages][num_kv_heads][page_size][head_dim/16]
 *                    one E4M3 (FN) block scale per 16 values, linear order
 *
 * A stored value decodes as e2m1(code) * e4m3(scale) * global_scale.  A token
 * lives in slot = page * page_size + offset.  head_dim must be 128 and
 * page_size 16; 144 bytes per (token, kv head) for K+V scales and codes of
 * one tensor pair -- 4.5 bits per value, 56.25% of an FP8 cache.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless a comment says HOST.  The
 *     caller owns every buffer; the library allocates no device memory (the
 *     prefill and decode calls take a caller-provided workspace).
 *   - Calls are asynchronous on `stream` (a cudaStream_t, passed as void*;
 *     NULL = legacy default stream) and return before the GPU work finishes.
 *   - Return 0 (NVFP4KV_OK) or a negative NVFP4KV_ERR_* code.  Argument
 *     errors are detected on the host before anything is launched.  Errors
 *     that only the device can see (an out-of-range page id or slot, a causal
 *     request with q_len > kv_len, a pipeline wait that timed out) are
 *     recorded in a device status word and reported by
 *     nvfp4kv_get_device_status(); the offending entries are skipped.
 *   - Nothing crosses the ABI as an exception; nothing calls exit().
 *   - Bounds: num_pages * page_size * num_kv_heads < 2^31 token-heads,
 *     total_q * num_q_heads < 2^31, and an append's num_tokens *
 *     num_kv_heads < 2^31.
 */
#ifndef NVFP4KV_H
#define NVFP4KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4KV_OK 0
#define NVFP4KV_ERR_ARG (-1)          /* null pointer, bad size, misaligned pool */
#define NVFP4KV_ERR_SHAPE (-2)        /* device saw q_len > kv_len (causal) or kv_len > table */
#define NVFP4KV_ERR_WORKSPACE (-3)    /* workspace NULL or smaller than required */
#define NVFP4KV_ERR_CUDA (-4)         /* a CUDA runtime/driver call failed */
#define NVFP4KV_ERR_TIMEOUT (-5)      /* a bounded device wait gave up */
#define NVFP4KV_ERR_DEVICE_INDEX (-6) /* device saw a page id / slot out of range */
#define NVFP4KV_ERR_UNSUPPORTED (-7)  /* current device is not sm_103 */

#define NVFP4KV_HEAD_DIM 128
#define NVFP4KV_PAGE_SIZE 16

/* Prefill variants ("NVFP4 KV cache A4Q prefill explained", sections
 * "Quantize Q instead of expanding K" and "Compare A4Q with dequantize-ahead
 * repacking"). */
#define NVFP4KV_VARIANT_A4Q 0      /* Q quantized to NVFP4 in-kernel, QK on block-scaled FP4 MMA */
#define NVFP4KV_VARIANT_DQ_AHEAD 1 /* K tile dequantized once to BF16, QK on BF16 MMA with BF16 Q */
/* An experiment beyond the pages' design, which keeps PV wide because the V
 * block scales run along the head dimension while PV reduces over tokens
 * ("NVFP4 KV cache A4Q prefill explained", sections "Why NVFP4 KV cache A4Q
 * prefill exists" and "Compare A4Q with dequantize-ahead repacking"): A4Q QK,
 * and PV on block-scaled FP4 MMA too.  V is re-coded once per call along
 * tokens (nvfp4_v_token_major's blocks, with slots past kv_len as zeros) into
 * the workspace; P is coded per 16 keys by the cache's block codec with
 * global scale fl32(16/2688), against a running reference that moves in
 * whole log2 steps when a 128-key tile's largest score exceeds it by more
 * than 4 (the kernel folds each block's reciprocal scale into the exponent,
 * which moves a code decision only when p lies within about 1e-6 relative of
 * a rounding boundary); the row sum uses the uncoded P.  Needs the repack
 * workspace. */
#define NVFP4KV_VARIANT_A4Q_FP4PV 2

/* Quantize-rows modes. */
#define NVFP4KV_QUANT_GLOBAL 0  /* one caller-given global scale for every row */
#define NVFP4KV_QUANT_PER_ROW 1 /* per-row scale amax/2688 (the A4Q query scheme) */

/* Workspace queries. */
#define NVFP4KV_OP_PREFILL 0
#define NVFP4KV_OP_DECODE 1

/* Descriptor of one layer's cache (a HOST struct; the pools are device
 * memory, each 16-byte aligned). */
typedef struct nvfp4kv_cache {
  void* k_data;
  void* k_scale;
  void* v_data;
  void* v_scale;
  int32_t num_pages;
  int32_t page_size;    /* must be 16 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* must be 128 */
  float k_global_scale; /* decode multiplier of K (> 0, finite) */
  float v_global_scale; /* decode multiplier of V (> 0, finite) */
} nvfp4kv_cache_t;

/* Cache append ("NVFP4 KV cache prefill vs decode performance", section
 * "NVFP4 stores 4.5 bits per value before padding": the cache write quantizes
 * BF16 input, creates packed FP4 data, writes block scales and maps the result
 * into paged cache slots).
 *
 * k, v:          bf16 [num_tokens][num_kv_heads][128], row-contiguous.
 * slot_mapping:  int64 [num_tokens]; token t goes to slot_mapping[t]; a
 *                negative slot skips the token; a slot >= num_pages*page_size
 *                is skipped and flagged (NVFP4KV_ERR_DEVICE_INDEX).
 * Per 16-value block: s = amax/(6*g) rounded to E4M3 (nearest even,
 * saturating at 448); codes = x * (1/(g*s)) rounded to E2M1 (nearest even,
 * ties to the even code, saturating at 6); zero scale -> zero codes.
 * num_tokens == 0 is a no-op. */
int nvfp4_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                    const nvfp4kv_cache_t* cache, void* stream);

/* Causal (or full) paged prefill attention over the NVFP4 cache
 * ("NVFP4 KV cache A4Q prefill explained": A4Q quantizes each query tile to
 * block-scaled FP4 and runs QK on native FP4 MMA against the cache's packed K
 * and scales; PV stays wide with V dequantized).
 *
 * q:          bf16 [total_q][num_q_heads][128] (ragged requests, packed).
 * qo_indptr:  int32 [batch+1], request b's queries are rows
 *             qo_indptr[b] .. qo_indptr[b+1]-1 of q (qo_indptr[batch] <= total_q).
 * kv_lens:    int32 [batch], cached tokens of each request (including the
 *             new ones, which must already be appended).
 * page_table: int32 [batch][max_pages_per_req]; entries past a request's
 *             ceil(kv_len/16) pages are never read.
 * causal:     1 = query i of a request sees keys j <= kv_len - q_len + i
 *             (bottom-right alignment); 0 = every query sees all kv_len keys.
 * sm_scale:   softmax scale applied to q.k (e.g. 1/sqrt(128)).
 * variant:    NVFP4KV_VARIANT_A4Q, NVFP4KV_VARIANT_DQ_AHEAD or
 *             NVFP4KV_VARIANT_A4Q_FP4PV (NVFP4 cache only; returns
 *             NVFP4KV_ERR_WORKSPACE unless the workspace holds the repack
 *             records, 18 KB per 128-key tile).
 * q_global_scale: the A4Q query scale scheme ("NVFP4 KV cache A4Q prefill
 *             explained", section "Make query accuracy a release gate": the
 *             scheme is a recorded choice).  0 = per (token, head) row, dual
 *             level: g_row = amax_row/2688.  > 0 = this one fp32 scale for
 *             every query row: a per-tensor dual-level scheme when the caller
 *             passes amax(Q)/2688, a single-level scheme when it passes 1.
 *             Either way the row is then coded with the cache's 16-value
 *             block codec.  Must be finite and >= 0; ignored by
 *             NVFP4KV_VARIANT_DQ_AHEAD (its query stays BF16); used by
 *             NVFP4KV_VARIANT_A4Q_FP4PV as by NVFP4KV_VARIANT_A4Q.
 * o:          bf16 [total_q][num_q_heads][128] output (rows of q not covered
 *             by qo_indptr are left untouched).
 * lse:        optional fp32 [total_q][num_q_heads] natural-log sum-exp of the
 *             scaled scores; NULL to skip.
 * workspace:  device buffer of at least
 *             nvfp4_workspace_bytes(NVFP4KV_OP_PREFILL, batch, num_q_heads,
 *             num_kv_heads, total_q, 0) bytes, 16-byte aligned; its contents
 *             are overwritten (it holds the work schedule).  Given
 *             nvfp4_workspace_bytes(..., total_q, max_pages_per_req * 16)
 *             bytes, the call may also run in repack mode:
 *             when requests average enough q tiles (128 rows of query
 *             tokens x grouped heads) per kv head -- eight for A4Q, two for
 *             dequant-ahead -- V (and K for the
 *             dequant-ahead variant) is first dequantized once per KV
 *             tile (112 keys for A4Q, 128 for dequant-ahead) into the
 *             workspace ("NVFP4 KV cache A4Q prefill explained", section
 *             "Compare A4Q with dequantize-ahead repacking"), instead of
 *             once per q tile inside the kernel.
 *             Both modes compute the same attention; they differ only in
 *             KV tile size and so in the order of the fp32 accumulation.
 * num_q_heads must be a multiple of num_kv_heads with a power-of-two ratio
 * of at most 128.  q_len == 0 requests produce nothing. */
int nvfp4_paged_prefill(const void* q, int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                        const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                        const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale, int32_t variant,
                        float q_global_scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream);

/* The two halves of nvfp4_paged_prefill, for callers that time or overlap
 * them separately.  nvfp4_paged_prefill_plan writes the work schedule into
 * the workspace and, in repack mode, the repacked K/V tile records of this
 * cache; nvfp4_paged_prefill_run launches only the attention kernel, which
 * reads them.  run must follow plan on the same stream with the same
 * arguments (the pair computes the same mode from them) and the same
 * workspace, with the cache unchanged in between; otherwise its result is
 * undefined.  nvfp4_paged_prefill(...) is plan(...) then run(...).  Arguments
 * and errors as for nvfp4_paged_prefill (plan takes no q, o, lse,
 * sm_scale or q_global_scale).  Neither allocates. */
int nvfp4_paged_prefill_plan(int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                             const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                             const int32_t* qo_indptr, int32_t batch, int32_t causal, int32_t variant,
                             void* workspace, size_t workspace_bytes, void* stream);
int nvfp4_paged_prefill_run(const void* q, int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                            const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                            const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale,
                            int32_t variant, float q_global_scale, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/* nvfp4_paged_prefill without a workspace argument, for callers that cannot
 * allocate device memory: an engine that plans all device memory up front and
 * allows no cudaMalloc on its serving path (an allocation can synchronize the
 * device), or a host that passes a kernel only its inputs and outputs.  The
 * pages have no counterpart of this call; it is a packaging of the same
 * kernels.  The work schedule lives in a static device array of
 * nvfp4_paged_prefill_noalloc_max_bytes() bytes (1 MiB) that every GPU which
 * loads the library holds until the process exits; only the schedule is
 * stored there, so the call always runs in-kernel mode (V dequantized inside
 * the attention kernel) and its output equals, bit for bit, that of
 * nvfp4_paged_prefill given a schedule-only workspace.  Arguments and results
 * are those of nvfp4_paged_prefill.  Returns NVFP4KV_ERR_WORKSPACE when the
 * schedule of the call (nvfp4_workspace_bytes(NVFP4KV_OP_PREFILL, ..., 0)) is
 * larger than the array, and NVFP4KV_ERR_UNSUPPORTED on a device that is not
 * sm_103; NVFP4KV_VARIANT_A4Q_FP4PV, which reads only repacked records, is
 * refused with NVFP4KV_ERR_WORKSPACE.  The first call on a device looks up the
 * array's device address
 * (make it before any stream capture); the address is kept for the life of
 * the process, which assumes one CUDA context per device.  All calls share
 * the array: calls that overlap on the GPU race.  Allocates nothing. */
int nvfp4_paged_prefill_noalloc(const void* q, int64_t total_q, int32_t num_q_heads, const nvfp4kv_cache_t* cache,
                                const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                                const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale,
                                int32_t variant, float q_global_scale, void* o, float* lse, void* stream);

/* Size in bytes of the static schedule array used by
 * nvfp4_paged_prefill_noalloc.  Host-only. */
size_t nvfp4_paged_prefill_noalloc_max_bytes(void);

/* Paged decode: one query token per request attends to all kv_lens[b] cached
 * tokens ("NVFP4 KV cache prefill vs decode performance", section "Decode can
 * win on fewer bytes read": decode reads the long cache for one new token and
 * is bandwidth-bound).  The query stays BF16; K and V are dequantized.
 * Each (request, kv head) is cut into items of S tokens, S the longest of
 * 1024, 2048, 4096 and 8192 that still gives every attention CTA two items
 * (chosen on the device from kv_lens); the items' partial results are merged
 * by their log-sum-exp.  The output does not depend on which CTA runs which
 * item.
 * q, o:       bf16 [batch][num_q_heads][128].
 * lse:        optional fp32 [batch][num_q_heads].
 * workspace:  nvfp4_workspace_bytes(NVFP4KV_OP_DECODE, batch, num_q_heads,
 *             num_kv_heads, 0, max_pages_per_req*16) bytes: the split
 *             schedule and the split-KV partials.  Rewritten by every call,
 *             so calls that share a workspace must be ordered on one
 *             stream.
 * kv_lens[b] == 0 gives a zero output row (lse -inf); a kv_lens[b] above
 * max_pages_per_req*16 does too and sets NVFP4KV_ERR_SHAPE in the device
 * status. */
int nvfp4_paged_decode(const void* q, int32_t num_q_heads, const nvfp4kv_cache_t* cache, const int32_t* page_table,
                       int32_t max_pages_per_req, const int32_t* kv_lens, int32_t batch, float sm_scale, void* o,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for op.  NVFP4KV_OP_PREFILL: the schedule for total_q
 * query tokens, plus, when max_kv_len > 0, room for the repack records of
 * any variant (per request and kv head: 37 KB per 112-key A4Q tile, 64 KB
 * per 128-key dequant-ahead tile or 18 KB per 128-key FP4 PV tile of
 * max_kv_len, the largest total).  NVFP4KV_OP_DECODE: the split-KV partials
 * for max_kv_len.  Host-only, no CUDA call.  Returns 0 for
 * bad arguments. */
size_t nvfp4_workspace_bytes(int32_t op, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int64_t total_q,
                             int32_t max_kv_len);

/* Bytes of one layer's four pools ("NVFP4 KV cache prefill vs decode
 * performance", section "A worked per-token cache estimate"):
 * 2 * num_pages * page_size * num_kv_heads * (head_dim/2 + head_dim/16).
 * Host-only.  Returns 0 for non-positive sizes or head_dim % 16 != 0. */
size_t nvfp4_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);

/* The device quantizer of the cache write and of the A4Q query, exposed for
 * standalone quantization ("NVFP4 KV cache A4Q prefill explained", section
 * "Preserve the capacity and decode case": GPU quantize kernels with a linear
 * block-scale layout).
 * x:          bf16 [rows][128].
 * packed:     uint8 [rows][64]; scales: uint8 [rows][8].
 * mode:       NVFP4KV_QUANT_GLOBAL (uses global_scale > 0) or
 *             NVFP4KV_QUANT_PER_ROW (writes fp32 row_scales[rows]). */
int nvfp4_quantize_rows(const void* x, int64_t rows, int32_t mode, float global_scale, void* packed, void* scales,
                        float* row_scales, void* stream);

/* Inverse of nvfp4_quantize_rows: out bf16 [rows][128] =
 * e2m1(code) * e4m3(scale) * (row_scales ? row_scales[r] : global_scale),
 * rounded to bf16 (exact when the product has at most 8 significant bits). */
int nvfp4_dequantize_rows(const void* packed, const void* scales, int64_t rows, const float* row_scales,
                          float global_scale, void* out, void* stream);

/* The token-major re-layout of V that NVFP4KV_VARIANT_A4Q_FP4PV reads (an
 * experiment: "NVFP4 KV cache A4Q prefill explained", section "Why NVFP4 KV
 * cache A4Q prefill exists", notes that the cache's V block scales do not
 * follow PV's reduction axis).  A page holds 16 tokens, so each (page, kv
 * head, head dimension d) is one block along tokens: the 16 slots' values at
 * d, decoded without the tensor scale (e2m1 * e4m3, exact), re-coded by the
 * cache's block codec (as nvfp4_kv_append) with global scale 1.  A value
 * decodes as e2m1(code) * e4m3(scale) * v_global_scale.
 * page_ids:  device int32 [num_ids]; an id outside [0, num_pages) gives zeros
 *            and is flagged (NVFP4KV_ERR_DEVICE_INDEX).
 * codes:     device uint8 [num_ids][num_kv_heads][128][8], 8-byte aligned;
 *            slot 2i in the low nibble of byte i.
 * scales:    device uint8 [num_ids][num_kv_heads][128].
 * Every slot of a listed page is used as written (the prefill variant
 * treats slots past a request's kv_len as zeros). */
int nvfp4_v_token_major(const nvfp4kv_cache_t* cache, const int32_t* page_ids, int32_t num_ids, void* codes,
                        void* scales, void* stream);

/* ---- FP8 (E4M3) comparison cache --------------------------------------------
 * The format the pages weigh NVFP4 against ("NVFP4 KV cache prefill vs decode
 * performance", sections "NVFP4 stores 4.5 bits per value before padding" and
 * "A worked per-token cache estimate": one 8-bit FP8 value per element, 2 * L
 * * H * D bytes per token, scale metadata kept apart; "NVFP4 KV cache A4Q
 * prefill explained", section "Build the benchmark matrix": run FP8 and the
 * NVFP4 paths on the same revision).  One fp32 scale per tensor; a value
 * decodes as e4m3(code) * scale.  Per layer the caller owns two device pools
 * (16-byte aligned):
 *
 *   k_data, v_data   uint8 [num_pages][num_kv_heads][page_size][head_dim]
 *
 * 256 bytes per (token, kv head) for K and V.  Slots, page tables, request
 * metadata, workspaces, errors and streams follow the NVFP4 calls. */
typedef struct fp8kv_cache {
  void* k_data;
  void* v_data;
  int32_t num_pages;
  int32_t page_size;    /* must be 16 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* must be 128 */
  float k_scale;        /* decode multiplier of K (> 0, finite) */
  float v_scale;        /* decode multiplier of V (> 0, finite) */
} fp8kv_cache_t;

/* FP8 cache write: code = E4M3(x * (1/scale)) with 1/scale the correctly
 * rounded fp32 reciprocal, nearest even, saturating at +-448; a negative value
 * that rounds to zero keeps its sign bit.  Arguments as for nvfp4_kv_append. */
int fp8_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                  const fp8kv_cache_t* cache, void* stream);

/* Paged prefill over the FP8 cache with a BF16 query: K and V are converted
 * once per (request, kv head, 128-key tile) into the workspace (E4M3 is exact
 * in BF16 and FP16), then QK runs on BF16 and PV on FP16 tensor-core MMA --
 * the FP8 baseline of the comparison.  Arguments as for nvfp4_paged_prefill
 * without variant and q_global_scale; the workspace must hold
 * fp8_workspace_bytes(NVFP4KV_OP_PREFILL, batch, num_q_heads, num_kv_heads,
 * total_q, max_pages_per_req * 16) bytes (NVFP4KV_ERR_WORKSPACE otherwise). */
int fp8_paged_prefill(const void* q, int64_t total_q, int32_t num_q_heads, const fp8kv_cache_t* cache,
                      const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
                      const int32_t* qo_indptr, int32_t batch, int32_t causal, float sm_scale, void* o, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Paged decode over the FP8 cache (BF16 query, one token per request).
 * Arguments, workspace and results as for nvfp4_paged_decode. */
int fp8_paged_decode(const void* q, int32_t num_q_heads, const fp8kv_cache_t* cache, const int32_t* page_table,
                     int32_t max_pages_per_req, const int32_t* kv_lens, int32_t batch, float sm_scale, void* o,
                     float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of the FP8 calls (NVFP4KV_OP_PREFILL: the schedule plus the
 * converted tiles for max_kv_len, which must be > 0; NVFP4KV_OP_DECODE: as for
 * NVFP4).  Host-only; 0 for bad arguments. */
size_t fp8_workspace_bytes(int32_t op, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int64_t total_q,
                           int32_t max_kv_len);

/* Bytes of one layer's two FP8 pools: 2 * num_pages * page_size *
 * num_kv_heads * head_dim ("A worked per-token cache estimate").  Host-only. */
size_t fp8_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device: 0, or the NVFP4KV_ERR_* code of the first recorded
 * condition (TIMEOUT before DEVICE_INDEX before SHAPE). */
int nvfp4kv_get_device_status(void* stream);

/* Static English text for a status code. */
const char* nvfp4kv_status_string(int status);

/* Test hook for the failure path: launches one thread that waits on a
 * shared-memory barrier nothing will ever complete, with a wall-time limit of
 * limit_ns (clamped to [1 us, 1 s]).  The wait gives up, records
 * NVFP4KV_ERR_TIMEOUT in the status word and the kernel returns normally:
 * the context stays usable.  Used to test nvfp4kv_get_device_status(). */
int nvfp4kv_debug_wait_timeout(uint32_t limit_ns, void* stream);

/* Library version, e.g. "nvfp4kv 0.1 sm_103a". */
const char* nvfp4kv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4KV_H */
