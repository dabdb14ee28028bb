// Paged prefill attention over the NVFP4 cache, run A4Q-style
// ("NVFP4 KV cache A4Q prefill explained", sections "Quantize Q instead of
// expanding K" and "Compare A4Q with dequantize-ahead repacking").
//
// One persistent CTA per SM walks a schedule of work items (request, q tile,
// kv head), longest first.  A q tile is 128 MMA rows = 128/G query tokens x
// the G query heads of one kv head, so each K/V tile fetched serves the whole
// GQA group.  Per KV tile of 128 keys (8 pages):
//
//   producer warp   TMA: packed K pages (64B-swizzled, straight into the
//                   FP4 MMA operand layout), K scales, packed V, V scales
//   transform WG    A4Q: K block scales -> TMEM (UE4M3 scale operand of the
//                   block-scaled MMA); DQ-ahead: K -> BF16 once per tile.
//                   V -> FP16 in the MMA's MN-major layout (exact).
//                   At each item start: Q tile -> NVFP4 (per-row dual level
//                   scale) + Q block scales -> TMEM (A4Q), or Q -> smem (BF16).
//   MMA warp        S = Q K^T: tcgen05 kind::mxf4nvf4 (scale_vec 4X, UE4M3),
//                   or kind::f16 BF16 (DQ-ahead), fp32 S in TMEM (double
//                   buffered).  O += P V: kind::f16 with P read from TMEM.
//   softmax WG      one TMEM lane (= one row) per thread: causal mask, online
//                   softmax in the log2 domain with lazy O rescaling, P as
//                   FP16 written back over S; epilogue O * v_scale / l.
//
// PV runs on FP16 operands: every dequantized V value (E2M1 x E4M3) is exact
// in FP16 (and in BF16), while FP16 keeps 3 more mantissa bits of P.
#include "kernels.cuh"

namespace nvfp4kv {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before O is rescaled

constexpr int kThreads = 320;  // warps 0-3 transform, 4-7 softmax, 8 producer, 9 MMA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

// TMEM columns
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColSFA = 384, kColSFB = 392;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kStageKData = 8192, kStageKScale = 1024, kStageVData = 8192, kStageVScale = 1024;
constexpr uint32_t kStageBytes = kStageKData + kStageKScale + kStageVData + kStageVScale;  // 18 KB
constexpr uint32_t kTileBuf16 = 32768;  // 128 keys x 128 values x 2 B

template <int VARIANT>
struct Layout {
  static constexpr bool kA4Q = VARIANT == 0;
  static constexpr int kStages = kA4Q ? 3 : 2;
  static constexpr uint32_t kQBytes = kA4Q ? 8192u : 32768u;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffStage = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffStage + kStages * kStageBytes;
  static constexpr uint32_t kOffK = kOffV + 2 * kTileBuf16;  // DQ-ahead only
  static constexpr uint32_t kOffSmall = kOffK + (kA4Q ? 0u : 2 * kTileBuf16);
  static constexpr uint32_t kOffQScale = kOffSmall;            // 128 floats
  static constexpr uint32_t kOffSfaStage = kOffQScale + 512;   // 128 x 8 B
  static constexpr uint32_t kOffMask = kOffSfaStage + 1024;    // per-stage page mask
  static constexpr uint32_t kOffBar = kOffMask + 64;
  static constexpr uint32_t kNumBars = 32;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffTmemSlot + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1 KB alignment
};

struct Bars {
  uint64_t* kv_full;   // [3]
  uint64_t* kv_empty;  // [3]
  uint64_t* sfb_full;  // [2] (A4Q: K scales in TMEM; DQ-ahead: K tile in BF16)
  uint64_t* s_full;    // [2]
  uint64_t* p_full;    // [2]
  uint64_t* vdq_full;  // [2]
  uint64_t* pv_done;   // [2]
  uint64_t* o_full;
  uint64_t* o_empty;
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* drain;
  uint64_t* qs_empty;   // softmax has read the item's row scales
  uint64_t* sfa_ready;  // transform warps have staged the item's Q block scales
};

__device__ __forceinline__ Bars make_bars(uint64_t* base) {
  Bars b;
  b.kv_full = base + 0;
  b.kv_empty = base + 3;
  b.sfb_full = base + 6;
  b.s_full = base + 8;
  b.p_full = base + 10;
  b.vdq_full = base + 12;
  b.pv_done = base + 14;
  b.o_full = base + 16;
  b.o_empty = base + 17;
  b.q_full = base + 18;
  b.q_empty = base + 19;
  b.drain = base + 20;
  b.qs_empty = base + 21;
  b.sfa_ready = base + 22;
  return b;
}

struct Item {
  int b, qt, kvh;
  int q_start, q_len, kv_len;
  int tok0, n_tok, n_tiles;
};

// Items are sorted by decreasing cost; CTAs take them in snake order.
__device__ __forceinline__ bool get_item(const PrefillArgs& a, int round, Item& it) {
  const int n_items = a.work[0];
  const int grid = gridDim.x;
  const int idx = round * grid + ((round & 1) ? (grid - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x));
  if (idx >= n_items) return false;
  const int2 w = reinterpret_cast<const int2*>(a.work + 4)[idx];
  it.b = w.x;
  it.qt = w.y >> 8;
  it.kvh = w.y & 255;
  it.q_start = a.qo_indptr[it.b];
  it.q_len = a.qo_indptr[it.b + 1] - it.q_start;
  it.kv_len = a.kv_lens[it.b];
  const int tpq = kBM >> a.log2_group;
  it.tok0 = it.qt * tpq;
  it.n_tok = min(tpq, it.q_len - it.tok0);
  const int last_key = a.causal ? it.kv_len - it.q_len + it.tok0 + it.n_tok - 1 : it.kv_len - 1;
  it.n_tiles = last_key / kBN + 1;
  return true;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16-byte chunk `cc` (0..7) of row `r` in a 128B-swizzled [rows][128 B] tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t cc) { return r * 128u + (((cc ^ r) & 7u) << 4); }
// 16-byte chunk `c` (0..3) of row `r` in a 64B-swizzled [rows][64 B] tile.
__device__ __forceinline__ uint32_t sw64_off(uint32_t r, uint32_t c) { return r * 64u + (((c ^ (r >> 1)) & 3u) << 4); }

// ---------------------------------------------------------------------------
// producer warp
template <int VARIANT>
__device__ void producer_loop(const PrefillArgs& a, const CUtensorMap* tmap_k, uint8_t* smem, const Bars& bars,
                              int lane) {
  using L = Layout<VARIANT>;
  int* mask_slot = reinterpret_cast<int*>(smem + L::kOffMask);
  uint32_t it_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round) {
    for (int j = 0; j < item.n_tiles; ++j, ++it_ctr) {
      const uint32_t st = it_ctr % L::kStages, ph = (it_ctr / L::kStages) & 1u;
      int pid = -1;
      const int page_idx = j * kPagesPerTile + lane;
      if (lane < kPagesPerTile && page_idx * kPageSize < item.kv_len) {
        pid = a.page_table[static_cast<int64_t>(item.b) * a.max_pages + page_idx];
        if (pid < 0 || pid >= a.num_pages) {
          set_status(a.status, kDevBadPage);
          pid = -1;
        }
      }
      const unsigned valid = __ballot_sync(0xffffffffu, pid >= 0);
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&bars.kv_empty[st], ph ^ 1u, a.status);
        if (ok) {
          mask_slot[st] = static_cast<int>(valid);
          mbar_arrive_expect_tx(&bars.kv_full[st], __popc(valid) * (kStageBytes / kPagesPerTile));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) return;
      if (pid >= 0) {
        uint8_t* stage = smem + L::kOffStage + st * kStageBytes;
        const int64_t row = (static_cast<int64_t>(pid) * a.num_kv_heads + item.kvh) * kPageSize;
        tma_load_2d(stage + lane * 1024, tmap_k, 0, static_cast<int32_t>(row), &bars.kv_full[st]);
        bulk_load(stage + kStageKData + lane * 128, a.k_scale + row * 8, 128, &bars.kv_full[st]);
        bulk_load(stage + kStageKData + kStageKScale + lane * 1024, a.v_data + row * 64, 1024, &bars.kv_full[st]);
        bulk_load(stage + kStageKData + kStageKScale + kStageVData + lane * 128, a.v_scale + row * 8, 128,
                  &bars.kv_full[st]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// MMA warp (lane 0 only)
template <int VARIANT>
__device__ void mma_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase) {
  using L = Layout<VARIANT>;
  const uint32_t q_s = smem_u32(smem + L::kOffQ);
  const uint32_t idesc_pv = idesc_f16(128, 128, 0, 0, 0, 1);
  const uint32_t idesc_qk = L::kA4Q ? idesc_mxf4nvf4(128, 128) : idesc_f16(128, 128, 1, 1, 0, 0);
  uint32_t it_ctr = 0, item_ctr = 0;
  Item item;
  auto do_pv = [&](uint32_t it, bool first) -> bool {
    const uint32_t b = it & 1u, ph = (it >> 1) & 1u;
    if (!mbar_wait(&bars.p_full[b], ph, a.status)) return false;
    if (!mbar_wait(&bars.vdq_full[b], ph, a.status)) return false;
    if (first && !mbar_wait(bars.o_empty, (item_ctr & 1u) ^ 1u, a.status)) return false;
    tc_fence_after();
    const uint32_t v_s = smem_u32(smem + L::kOffV + b * kTileBuf16);
    const uint32_t s_col = b ? kColS1 : kColS0;
#pragma unroll
    for (uint32_t k = 0; k < 8; ++k) {
      mma_f16_ts(tbase + kColO, tbase + s_col + 8 * k, smem_desc(v_s + k * 2048, 16384, 1024, kSwz128), idesc_pv,
                 (first && k == 0) ? 0u : 1u);
    }
    tc_commit(&bars.pv_done[b]);
    return true;
  };
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    if (!mbar_wait(bars.q_full, item_ctr & 1u, a.status)) return;
    tc_fence_after();
    for (int j = 0; j < item.n_tiles; ++j) {
      const uint32_t it = it_ctr + j;
      const uint32_t st = it % L::kStages, b = it & 1u;
      if (!mbar_wait(&bars.kv_full[st], (it / L::kStages) & 1u, a.status)) return;
      if (!mbar_wait(&bars.sfb_full[b], (it >> 1) & 1u, a.status)) return;
      if (it >= 2 && !mbar_wait(&bars.pv_done[b], ((it >> 1) - 1u) & 1u, a.status)) return;
      tc_fence_after();
      const uint32_t s_col = b ? kColS1 : kColS0;
      if constexpr (L::kA4Q) {
        const uint32_t k_s = smem_u32(smem + L::kOffStage + st * kStageBytes);
#pragma unroll
        for (uint32_t s = 0; s < 2; ++s) {
          mma_nvf4_ss(tbase + s_col, smem_desc(q_s + 32 * s, 16, 512, kSwz64), smem_desc(k_s + 32 * s, 16, 512, kSwz64),
                      idesc_qk, tbase + kColSFA + 4 * s, tbase + kColSFB + 8 * b + 4 * s, s > 0 ? 1u : 0u);
        }
      } else {
        const uint32_t k_s = smem_u32(smem + L::kOffK + b * kTileBuf16);
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_f16_ss(tbase + s_col, smem_desc(q_s + off, 16, 1024, kSwz128), smem_desc(k_s + off, 16, 1024, kSwz128),
                     idesc_qk, k > 0 ? 1u : 0u);
        }
      }
      tc_commit(&bars.s_full[b]);
      tc_commit(&bars.kv_empty[st]);
      if (j == item.n_tiles - 1) tc_commit(bars.q_empty);
      if (j >= 1 && !do_pv(it - 1, j == 1)) return;
    }
    if (!do_pv(it_ctr + item.n_tiles - 1, item.n_tiles == 1)) return;
    tc_commit(bars.o_full);
    it_ctr += item.n_tiles;
  }
}

// ---------------------------------------------------------------------------
// transform warpgroup (warps 0-3): thread = Q row / TMEM lane
template <int VARIANT>
__device__ void transform_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase, int tid) {
  using L = Layout<VARIANT>;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = a.group, lg = a.log2_group;
  float* qscale = reinterpret_cast<float*>(smem + L::kOffQScale);
  uint2* sfa_stage = reinterpret_cast<uint2*>(smem + L::kOffSfaStage);
  const int* mask_slot = reinterpret_cast<const int*>(smem + L::kOffMask);
  uint32_t it_ctr = 0, item_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    // The previous item's Q tile, Q block scales and row scales must be
    // consumed (last QK issued and finished; softmax has read its row scales)
    // before they are overwritten.  Waiting on both also keeps the softmax
    // less than one q_full phase behind.
    if (item_ctr > 0 && !mbar_wait_warp(bars.q_empty, (item_ctr - 1) & 1u, a.status)) return;
    if (item_ctr > 0 && !mbar_wait_warp(bars.qs_empty, (item_ctr - 1) & 1u, a.status)) return;
    // ---- Q tile ------------------------------------------------------------
    {
      const int r = tid;
      const int tq = item.tok0 + (r >> lg);
      const bool valid = (r >> lg) < item.n_tok;
      const int hq = item.kvh * G + (r & (G - 1));
      uint32_t w[64];
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                          (static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq) * kHeadDim);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint4 v = src[i];
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) w[i] = 0u;
      }
      if constexpr (L::kA4Q) {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float lo, hi;
          bf16x2_to_f32(w[i], lo, hi);
          amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
        }
        const float g_row = __fdiv_rn(amax, 2688.0f);
        uint32_t codes[16];
        uint32_t sc[8];
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          float x[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) bf16x2_to_f32(w[8 * blk + i], x[2 * i], x[2 * i + 1]);
          if (g_row != 0.0f) {
            sc[blk] = quant_block16(x, g_row, codes[2 * blk], codes[2 * blk + 1]);
          } else {
            sc[blk] = 0u;
            codes[2 * blk] = codes[2 * blk + 1] = 0u;
          }
        }
        uint8_t* qrow = smem + L::kOffQ;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(qrow + sw64_off(r, c)) =
              make_uint4(codes[4 * c], codes[4 * c + 1], codes[4 * c + 2], codes[4 * c + 3]);
        sfa_stage[r] = make_uint2(sc[0] | (sc[1] << 8) | (sc[2] << 16) | (sc[3] << 24),
                                  sc[4] | (sc[5] << 8) | (sc[6] << 16) | (sc[7] << 24));
        qscale[r] = g_row;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sfa_ready);
        if (!mbar_wait_warp(bars.sfa_ready, item_ctr & 1u, a.status)) return;
        // Q block scales -> TMEM: lane i of each quadrant, column 4s+j holds
        // the four scales of k-step s for row 32j+i (replicated per quadrant).
        uint32_t va[8];
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint2 v = sfa_stage[32 * j + lane];
            va[4 * s + j] = s ? v.y : v.x;
          }
        tmem_st8(tmem_addr(tbase, 32 * warp, kColSFA), va);
        tmem_wait_st();
      } else {
        uint8_t* qt = smem + L::kOffQ;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(qt + (c >> 3) * 16384 + sw128_off(r, c & 7)) =
              make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        qscale[r] = 1.0f;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.q_full);
    }
    // ---- KV tiles ------------------------------------------------------------
    for (int j = 0; j < item.n_tiles; ++j) {
      const uint32_t it = it_ctr + j;
      const uint32_t st = it % L::kStages, b = it & 1u;
      if (!mbar_wait_warp(&bars.kv_full[st], (it / L::kStages) & 1u, a.status)) return;
      const uint8_t* stage = smem + L::kOffStage + st * kStageBytes;
      const int valid_pages = mask_slot[st];
      const int key_base = j * kBN;
      if (it >= 2 && !mbar_wait_warp(&bars.s_full[b], ((it >> 1) - 1u) & 1u, a.status)) return;
      if constexpr (L::kA4Q) {
        // K block scales -> TMEM (same replicated layout as Q's)
        const uint8_t* ks = stage + kStageKData;
        uint32_t vb[8];
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) vb[4 * s + jj] = *reinterpret_cast<const uint32_t*>(ks + (32 * jj + lane) * 8 + 4 * s);
        tmem_st8(tmem_addr(tbase, 32 * warp, kColSFB + 8 * b), vb);
        tmem_wait_st();
        tc_fence_before();
      } else {
        // K -> BF16 (exact), K-major 128B-swizzled operand
        uint8_t* kb = smem + L::kOffK + b * kTileBuf16;
        const uint8_t* kd = stage;
        const uint8_t* ks = stage + kStageKData;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int u = tid + 128 * i;
          const int key = u >> 2, c = u & 3;
          const uint4 src = *reinterpret_cast<const uint4*>(kd + sw64_off(key, c));
          const uint32_t sc01 = *reinterpret_cast<const uint16_t*>(ks + key * 8 + 2 * c);
          const uint32_t s0 = scale_bf16x2_x2p112(sc01 & 0xFFu), s1 = scale_bf16x2_x2p112(sc01 >> 8);
          uint32_t o0[4], o1[4], o2[4], o3[4];
          dequant8_bf16(src.x, s0, o0);
          dequant8_bf16(src.y, s0, o1);
          dequant8_bf16(src.z, s1, o2);
          dequant8_bf16(src.w, s1, o3);
          uint8_t* dst = kb + (c >> 1) * 16384;
          const uint32_t cc = (c & 1) * 4;
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 0)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 1)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 2)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 3)) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sfb_full[b]);
      // ---- V -> FP16, MN-major 128B-swizzled operand ---------------------------
      if (it >= 2 && !mbar_wait_warp(&bars.pv_done[b], ((it >> 1) - 1u) & 1u, a.status)) return;
      {
        uint8_t* vb = smem + L::kOffV + b * kTileBuf16;
        const uint8_t* vd = stage + kStageKData + kStageKScale;
        const uint8_t* vs = vd + kStageVData;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int u = tid + 128 * i;
          const int key = u >> 2, c = u & 3;
          const bool live = (key_base + key < item.kv_len) && ((valid_pages >> (key >> 4)) & 1);
          uint32_t o0[4] = {0, 0, 0, 0}, o1[4] = {0, 0, 0, 0}, o2[4] = {0, 0, 0, 0}, o3[4] = {0, 0, 0, 0};
          if (live) {
            const uint4 src = *reinterpret_cast<const uint4*>(vd + key * 64 + 16 * c);
            const uint32_t sc01 = *reinterpret_cast<const uint16_t*>(vs + key * 8 + 2 * c);
            const uint32_t s0 = scale_f16x2(sc01 & 0xFFu), s1 = scale_f16x2(sc01 >> 8);
            dequant8_f16(src.x, s0, o0);
            dequant8_f16(src.y, s0, o1);
            dequant8_f16(src.z, s1, o2);
            dequant8_f16(src.w, s1, o3);
          }
          uint8_t* dst = vb + (c >> 1) * 16384;
          const uint32_t cc = (c & 1) * 4;
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 0)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 1)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 2)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(key, cc + 3)) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.vdq_full[b]);
        mbar_arrive(&bars.kv_empty[st]);
      }
    }
    it_ctr += item.n_tiles;
  }
}

// ---------------------------------------------------------------------------
// softmax warpgroup (warps 4-7): thread = TMEM lane = row
template <int VARIANT>
__device__ void softmax_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase, int r) {
  using L = Layout<VARIANT>;
  const int quad = r >> 5, lane = r & 31;
  const int G = a.group, lg = a.log2_group;
  const float* qscale = reinterpret_cast<const float*>(smem + L::kOffQScale);
  const uint32_t lane_base = tmem_addr(tbase, 32 * quad, 0);
  uint32_t it_ctr = 0, item_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    if (!mbar_wait_warp(bars.q_full, item_ctr & 1u, a.status)) return;
    const int tq = item.tok0 + (r >> lg);
    const bool valid = (r >> lg) < item.n_tok;
    const int hq = item.kvh * G + (r & (G - 1));
    const int limit = !valid ? -1 : (a.causal ? item.kv_len - item.q_len + tq : item.kv_len - 1);
    const float c_r = (L::kA4Q ? qscale[r] : 1.0f) * a.k_g * a.sm_scale * kLog2e;
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.qs_empty);
    float m_run = -INFINITY, l_run = 0.0f;
    for (int j = 0; j < item.n_tiles; ++j) {
      const uint32_t it = it_ctr + j;
      const uint32_t b = it & 1u;
      const uint32_t s_col = b ? kColS1 : kColS0;
      if (!mbar_wait_warp(&bars.s_full[b], (it >> 1) & 1u, a.status)) return;
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_wait_ld();
      float* s = reinterpret_cast<float*>(sr);
      const int key0 = j * kBN;
      // Tiles crossing the row's last visible key are scaled and masked here;
      // all others fold the scale into the exponent's FMA.
      const bool masked = key0 + kBN - 1 > limit;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (key0 + c > limit) ? -INFINITY : s[c] * c_r;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 2) mx = fmaxf(mx, fmaxf(s[c], s[c + 1]));
      const float m_tile = masked ? mx : mx * c_r;
      // Lazy rescale: a row moves its running max only when the tile max
      // exceeds it by more than 2^8.  O is rescaled by the whole warp (TMEM
      // loads/stores are warp-collective), with factor 1 for rows that keep
      // their max.
      float alpha = 1.0f;
      const bool need = m_tile > m_run + kRescaleThreshold;
      if (need) {
        alpha = fast_exp2(m_run - m_tile);  // 0 when m_run = -inf
        l_run *= alpha;
        m_run = m_tile;
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O must hold PV of the previous tile before it is rescaled
        const uint32_t pit = it - 1u;
        if (!mbar_wait_warp(&bars.pv_done[pit & 1u], (pit >> 1) & 1u, a.status)) return;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kColO + 32 * c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st16(lane_base + kColO + 32 * c, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
          tmem_st16(lane_base + kColO + 32 * c + 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[16]));
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      const float cs = masked ? 1.0f : c_r;
      float lsum = 0.0f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = fast_exp2(fmaf(s[2 * c], cs, -m_use));
        const float p1 = fast_exp2(fmaf(s[2 * c + 1], cs, -m_use));
        lsum += p0 + p1;
        pk[c] = pack_f16x2(p0, p1);
      }
      l_run += lsum;
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_st16(lane_base + s_col + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * c]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[b]);
    }
    // ---- epilogue ---------------------------------------------------------------
    if (!mbar_wait_warp(bars.o_full, item_ctr & 1u, a.status)) return;
    tc_fence_after();
    const float inv_l = (l_run > 0.0f) ? a.v_g / l_run : 0.0f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) +
                          (static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq) * kHeadDim;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t ov[32];
      tmem_ld32(lane_base + kColO + 32 * c, ov);
      tmem_wait_ld();
      if (valid) {
        uint32_t pb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
          pb[i] = *reinterpret_cast<uint32_t*>(&v);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
        dst[0] = make_uint4(pb[0], pb[1], pb[2], pb[3]);
        dst[1] = make_uint4(pb[4], pb[5], pb[6], pb[7]);
        dst[2] = make_uint4(pb[8], pb[9], pb[10], pb[11]);
        dst[3] = make_uint4(pb[12], pb[13], pb[14], pb[15]);
      }
    }
    if (valid && a.lse)
      a.lse[static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq] =
          (l_run > 0.0f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.o_empty);
    it_ctr += item.n_tiles;
  }
}

template <int VARIANT>
__device__ __forceinline__ void prefill_body(const PrefillArgs& a, const CUtensorMap* tmap_k) {
  using L = Layout<VARIANT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  const Bars bars = make_bars(bar_base);
  if (tid == 0) {
    for (int i = 0; i < L::kStages; ++i) {
      mbar_init(&bars.kv_full[i], 1);
      mbar_init(&bars.kv_empty[i], 5);  // QK commit + one arrive per transform warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.sfb_full[i], 4);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);
      mbar_init(&bars.vdq_full[i], 4);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(bars.o_full, 1);
    mbar_init(bars.o_empty, 4);
    mbar_init(bars.q_full, 4);
    mbar_init(bars.q_empty, 1);
    mbar_init(bars.drain, 1);
    mbar_init(bars.qs_empty, 4);
    mbar_init(bars.sfa_ready, 4);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) prefetch_tmap(tmap_k);
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp < 4) {
    transform_loop<VARIANT>(a, smem, bars, tbase, tid);
  } else if (warp < 8) {
    softmax_loop<VARIANT>(a, smem, bars, tbase, tid - 128);
  } else if (warp == kProducerWarp) {
    producer_loop<VARIANT>(a, tmap_k, smem, bars, lane);
  } else {
    if (lane == 0) {
      mma_loop<VARIANT>(a, smem, bars, tbase);
      // drain: every MMA issued by this thread has finished before TMEM is freed
      tc_commit(bars.drain);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    if (lane == 0) mbar_wait(bars.drain, 0, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_prefill_a4q_sm103_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmap_k) {
  prefill_body<0>(a, &tmap_k);
}

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_prefill_dqahead_sm103_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmap_k) {
  prefill_body<1>(a, &tmap_k);
}

// ---------------------------------------------------------------------------
// schedule: items (request, q tile, kv head) sorted by decreasing KV-tile count
constexpr int kMaxCostBins = 4096;

__global__ void __launch_bounds__(1024) nvfp4_prefill_plan_kernel(PlanArgs a) {
  __shared__ int hist[kMaxCostBins];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  int* prefix = a.work + 4 + 2 * a.max_items;  // [batch + 1] unit prefix (scratch)
  const int tpq_shift = 7 - a.log2_group;      // log2(tokens per q tile)
  for (int i = tid; i < kMaxCostBins; i += blockDim.x) hist[i] = 0;
  if (tid == 0) {
    int total = 0;
    for (int b = 0; b < a.batch; ++b) {
      prefix[b] = total;
      const int q0 = a.qo_indptr[b], q1 = a.qo_indptr[b + 1];
      const int q_len = q1 - q0, kv_len = a.kv_lens[b];
      bool bad = q_len < 0 || q0 < 0 || q1 > a.total_q || kv_len < 0 ||
                 kv_len > a.max_pages * kPageSize || (a.causal && q_len > kv_len);
      if (bad) {
        set_status(a.status, kDevBadShape);
        continue;
      }
      const int n_qt = (q_len + (1 << tpq_shift) - 1) >> tpq_shift;
      const int add = n_qt * a.num_kv_heads;
      if (total + add > a.max_items) {
        set_status(a.status, kDevBadShape);
        continue;
      }
      total += add;
    }
    prefix[a.batch] = total;
    s_total = total;
    a.work[0] = total;
  }
  __syncthreads();
  const int total = s_total;
  auto cost_of = [&](int u, int& b, int& qt, int& kvh) -> int {
    int lo = 0, hi = a.batch - 1;  // last b with prefix[b] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int r = u - prefix[b];
    qt = r / a.num_kv_heads;
    kvh = r - qt * a.num_kv_heads;
    const int q_len = a.qo_indptr[b + 1] - a.qo_indptr[b], kv_len = a.kv_lens[b];
    const int tok0 = qt << tpq_shift;
    const int n_tok = min(1 << tpq_shift, q_len - tok0);
    const int last_key = a.causal ? kv_len - q_len + tok0 + n_tok - 1 : kv_len - 1;
    return min(last_key / kBN + 1, kMaxCostBins - 1);
  };
  for (int u = tid; u < total; u += blockDim.x) {
    int b, qt, kvh;
    atomicAdd(&hist[cost_of(u, b, qt, kvh)], 1);
  }
  __syncthreads();
  if (tid == 0) {  // exclusive offsets, largest cost first
    int run = 0;
    for (int c = kMaxCostBins - 1; c >= 0; --c) {
      const int n = hist[c];
      hist[c] = run;
      run += n;
    }
  }
  __syncthreads();
  int2* items = reinterpret_cast<int2*>(a.work + 4);
  for (int u = tid; u < total; u += blockDim.x) {
    int b, qt, kvh;
    const int c = cost_of(u, b, qt, kvh);
    const int pos = atomicAdd(&hist[c], 1);
    items[pos] = make_int2(b, (qt << 8) | kvh);
  }
}

}  // namespace

size_t prefill_smem_bytes(int variant) { return variant == 0 ? Layout<0>::kAlloc : Layout<1>::kAlloc; }

cudaError_t launch_prefill(const PrefillArgs& a, const PlanArgs& plan, const CUtensorMap& tmap_k, int variant,
                           int num_sms, cudaStream_t s) {
  nvfp4_prefill_plan_kernel<<<1, 1024, 0, s>>>(plan);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (variant == 0) {
    e = cudaFuncSetAttribute(nvfp4_prefill_a4q_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<0>::kAlloc);
    if (e != cudaSuccess) return e;
    nvfp4_prefill_a4q_sm103_kernel<<<num_sms, kThreads, Layout<0>::kAlloc, s>>>(a, tmap_k);
  } else {
    e = cudaFuncSetAttribute(nvfp4_prefill_dqahead_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<1>::kAlloc);
    if (e != cudaSuccess) return e;
    nvfp4_prefill_dqahead_sm103_kernel<<<num_sms, kThreads, Layout<1>::kAlloc, s>>>(a, tmap_k);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4kv
