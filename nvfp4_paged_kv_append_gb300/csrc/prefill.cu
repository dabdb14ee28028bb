// Paged prefill attention over the NVFP4 cache, run A4Q-style
// ("NVFP4 KV cache A4Q prefill explained", sections "Quantize Q instead of
// expanding K" and "Compare A4Q with dequantize-ahead repacking").
//
// One persistent CTA per SM walks a schedule of work items (request, q tile,
// kv head), longest first.  A q tile is 128 MMA rows = 128/G query tokens x
// the G query heads of one kv head, so each K/V tile fetched serves the whole
// GQA group.  Per KV tile of 128 keys (8 pages):
//
//   loader warps    In-kernel mode: cp.async gathers of the tile's 8 pages
//                   (K codes into the 64B-swizzled FP4 MMA operand layout, K
//                   block scales into the MMA's scale-factor atoms, V codes and
//                   scales as stored).  Repack mode: one bulk copy of the
//                   tile's record, prepared once per (request, kv head, tile)
//                   by the repack pre-pass in the exact shared-memory layout.
//   transform WG    At each item start: Q tile -> NVFP4 (per-row dual level
//                   scale) + Q block scales -> TMEM (A4Q), or Q -> shared
//                   memory as BF16 (dequant-ahead).  In-kernel mode, per KV
//                   tile: V -> FP16 in the MMA's MN-major layout (exact), and
//                   for the dequant-ahead variant K -> BF16.
//   MMA warp        K block scales -> scale-factor atoms -> TMEM (tcgen05.cp);
//                   S = Q K^T: tcgen05 kind::mxf4nvf4 (scale_vec 4X, UE4M3),
//                   or kind::f16 BF16 (dequant-ahead); fp32 S in TMEM, double
//                   buffered.  O += P V: kind::f16 with P read from TMEM.
//   softmax WGs     two warpgroups, one TMEM lane (= one row) per thread, each
//                   owning 64 of the tile's 128 keys (and 64 of O's columns):
//                   causal mask, row max exchanged through shared memory,
//                   online softmax in the log2 domain with lazy O rescaling,
//                   P as FP16 written back over S; epilogue O * v_scale / l.
//
// Repack mode follows the pages' "convert an NVFP4 tile once before repeated
// MMA use": every q tile of a request that visits a KV tile would otherwise
// dequantize the same V values again.  It is used when the caller's workspace
// has room and requests have enough q tiles per kv head on average (eight for
// A4Q, two for dequant-ahead).
//
// PV runs on FP16 operands: every dequantized V value (E2M1 x E4M3) is exact
// in FP16 (and in BF16), while FP16 keeps 3 more mantissa bits of P.
//
// The FP4 PV variant (an experiment: the pages keep PV wide because the
// cache's V block scales run along the head dimension while PV reduces over
// tokens, "NVFP4 KV cache A4Q prefill explained", sections "Why NVFP4 KV cache
// A4Q prefill exists" and "Compare A4Q with dequantize-ahead repacking") runs
// PV on kind::mxf4nvf4 too.  Its repack records carry V re-coded along
// tokens (one E4M3 scale per 16 tokens of one head dimension, the cache's
// block codec with global scale 1) as an MMA B operand beside K; the softmax
// codes P per 16 keys with the same codec and global scale 2^4/2688, against
// a running reference that only takes whole values (so a moved reference
// scales P and O by exact powers of two), and writes P's codes and scale
// atoms to shared memory for the PV MMA.
#include "prefill_common.cuh"

namespace nvfp4kv {

namespace {

using namespace prefill_detail;

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^d for a whole number d <= 0 (or -inf), exactly; 0 below the normal range.
__device__ __forceinline__ float exp2_whole(float d) {
  return d < -126.0f ? 0.0f : __int_as_float((static_cast<int>(d) + 127) << 23);
}

// warps 0 QK issue (and TMEM allocation), 1-2 loaders, 3 PV issue, 4-7
// transform, 8-11 softmax half 0, 12-15 softmax half 1.  A warp reaches only
// the TMEM lane quadrant (warp id % 4), which the transform and softmax
// warpgroups keep: row r of a tile lives in quadrant r / 32.
constexpr int kThreads = 512;
constexpr int kMmaWarp = 0, kPvWarp = 3;
constexpr int kLoaderWarp0 = 1, kLoaderWarp1 = 2;
constexpr int kLoaderThreads = 64;
constexpr int kTransformTid0 = 128, kSoftmaxTid0 = 256;

// TMEM columns: S double buffer (fp32; each half's P as FP16 pairs over the
// first 32 of its 64 columns), O (fp32), Q block scales, K block scales
// (double buffer); FP4 PV: P and V block scales (double buffered)
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColSFA = 448, kColSFB = 456;
constexpr uint32_t kColSFP = 384, kColSFV = 400;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kKData = 8192, kKScale = 1024, kVData = 8192, kVScale = 1024;
constexpr uint32_t kTile16 = 32768;  // 128 keys x 128 values x 2 B
constexpr uint32_t kPBuf = 8192 + 1024;  // FP4 PV: P codes (64B-swizzled rows) + two scale atoms

// FP4 PV: P <= 2^kTauFp4 against the whole-number reference, coded with
// global scale fl32(2^kTauFp4 / 2688) so that its block scales never saturate.
constexpr float kTauFp4 = 4.0f;
constexpr float kPScale = 16.0f / 2688.0f;
constexpr float kPInvSixG = 28.0f;  // 1 / (6 g_P): a block scale is amax * 28

// Shared-memory layout per (variant, mode).  Stage contents:
//   in-kernel:     K codes 8 KB | K scales 1 KB | V codes 8 KB | V scales 1 KB
//   A4Q repack:    K codes 8 KB | K scales 1 KB | V tile (FP16) 32 KB
//   DQ repack:     K tile (BF16) 32 KB | V tile (FP16) 32 KB
//   FP4 PV repack: K codes 8 KB | K scales 1 KB | token-major V codes 8 KB
//                  (64B-swizzled [head dim][64 B]) | their scale atoms 1 KB
// K codes are 64B-swizzled [key][64 B] rows.  A4Q K scales are two 512-byte
// scale-factor atoms (k-steps 0 and 1: key n's four block scales at byte
// (n % 32) * 16 + (n / 32) * 4), ready for tcgen05.cp; dequant-ahead keeps
// them as stored ([key][8 B]).  A repack-mode stage is one record of the
// repack pre-pass, byte for byte.
template <int VARIANT, bool REPACK>
struct Layout {
  static constexpr bool kA4Q = VARIANT != 1;    // FP4 query, block-scaled FP4 QK
  static constexpr bool kFp4Pv = VARIANT == 2;  // FP4 P x token-major FP4 V
  static_assert(!kFp4Pv || REPACK, "the FP4 PV variant reads repacked records");
  static constexpr int kStages = REPACK ? (kFp4Pv ? 6 : kA4Q ? 5 : 2) : (kA4Q ? 6 : 3);
  static constexpr uint32_t kStageBytes =
      REPACK ? (kFp4Pv ? kKData + kKScale + kVData + kVScale : kA4Q ? kKData + kKScale + kTile16 : 2 * kTile16)
             : kKData + kKScale + kVData + kVScale;
  static constexpr uint32_t kStageV = REPACK ? (kA4Q ? kKData + kKScale : kTile16) : kKData + kKScale;
  static constexpr uint32_t kQBytes = kA4Q ? 8192u : 32768u;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffStage = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffStage + kStages * kStageBytes;            // in-kernel V buffers
  static constexpr uint32_t kOffK = kOffV + (REPACK ? 0u : 2 * kTile16);          // in-kernel DQ K buffers
  static constexpr uint32_t kOffP = kOffK + ((!REPACK && !kA4Q) ? 2 * kTile16 : 0u);  // FP4 PV: P [2]
  static constexpr uint32_t kOffSmall = kOffP + (kFp4Pv ? 2 * kPBuf : 0u);
  static constexpr uint32_t kOffQScale = kOffSmall;            // 128 floats
  static constexpr uint32_t kOffSfaStage = kOffQScale + 512;   // 128 x 8 B
  static constexpr uint32_t kOffXmax = kOffSfaStage + 1024;    // [2 parity][2 half][128] row maxima
  static constexpr uint32_t kOffXl = kOffXmax + 2048;          // [2 half][128] row sums
  static constexpr uint32_t kOffBar = kOffXl + 1024;
  static constexpr uint32_t kNumBars = 36;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffTmemSlot + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1 KB alignment
  static_assert(kAlloc <= 227 * 1024, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kStageV % 1024 == 0, "1 KB aligned operands");
};

struct Bars {
  uint64_t* kv_full;   // [6]
  uint64_t* kv_empty;  // [6]
  uint64_t* sfb_full;  // [2] in-kernel dequant-ahead: K tile in BF16
  uint64_t* s_full;    // [2]
  uint64_t* s_free;    // [2] FP4 PV: softmax has loaded S, the buffer may take the next QK
  uint64_t* p_full;    // [2]
  uint64_t* vdq_full;  // [2] in-kernel mode: V tile in FP16
  uint64_t* pv_done;   // [2]
  uint64_t* o_full;
  uint64_t* o_empty;
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* drain;
  uint64_t* qs_empty;   // softmax has read the item's row scales
  uint64_t* sfa_ready;  // transform warps have staged the item's Q block scales
  uint64_t* xchg;       // [4] per TMEM quadrant: the two softmax halves of a row meet
};

__device__ __forceinline__ Bars make_bars(uint64_t* base) {
  Bars b;
  b.kv_full = base + 0;
  b.kv_empty = base + 6;
  b.sfb_full = base + 12;
  b.s_full = base + 14;
  b.p_full = base + 16;
  b.vdq_full = base + 18;
  b.pv_done = base + 20;
  b.o_full = base + 22;
  b.o_empty = base + 23;
  b.q_full = base + 24;
  b.q_empty = base + 25;
  b.drain = base + 26;
  b.qs_empty = base + 27;
  b.sfa_ready = base + 28;
  b.xchg = base + 29;  // 29..32
  b.s_free = base + 33;  // 33..34
  return b;
}

// ---------------------------------------------------------------------------
// loader warps (1 and 2): t = 0..63.  In-kernel mode, thread t gathers a
// slice of page p = t / 8 of the tile with cp.async; a page past kv_len (or
// with an invalid id) reads as zeros.  Repack mode: thread 0 issues the one
// bulk copy of the tile's record.
template <int VARIANT, bool REPACK>
__device__ void loader_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, int t) {
  using L = Layout<VARIANT, REPACK>;
  const int p = t >> 3, sub = t & 7;
  uint32_t it_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round) {
    for (int j = 0; j < item.n_tiles; ++j, ++it_ctr) {
      const uint32_t st = it_ctr % L::kStages, ph = (it_ctr / L::kStages) & 1u;
      uint8_t* stage = smem + L::kOffStage + st * L::kStageBytes;
      if constexpr (REPACK) {
        if (t == 0) {
          if (!mbar_wait(&bars.kv_empty[st], ph ^ 1u, a.status)) return;
          mbar_arrive_expect_tx(&bars.kv_full[st], L::kStageBytes);
          bulk_load(stage, a.repack + repack_index(a, item.b, item.kvh, item.t0 + j) * L::kStageBytes, L::kStageBytes,
                    &bars.kv_full[st]);
        }
      } else {
        int pid = -1;
        const int page_idx = (item.t0 + j) * kPagesPerTile + p;
        if (page_idx * kPageSize < item.kv_len) {
          pid = a.page_table[static_cast<int64_t>(item.b) * a.max_pages + page_idx];
          if (pid < 0 || pid >= a.num_pages) {
            if (sub == 0) set_status(a.status, kDevBadPage);
            pid = -1;
          }
        }
        const uint32_t n16 = pid >= 0 ? 16u : 0u, n4 = pid >= 0 ? 4u : 0u;
        const int64_t row0 = (static_cast<int64_t>(pid >= 0 ? pid : 0) * a.num_kv_heads + item.kvh) * kPageSize;
        if (!mbar_wait_warp(&bars.kv_empty[st], ph ^ 1u, a.status)) return;
        const uint32_t st_s = smem_u32(stage);
        const uint8_t* kd = a.k_data + row0 * 64;
        const uint8_t* vd = a.v_data + row0 * 64;
        // codes: the page's 64 chunks of 16 B, chunk q = token q/4, quarter q%4
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int q = sub + 8 * i, n = p * kPageSize + (q >> 2), c = q & 3;
          cp_async16(st_s + sw64_off(n, c), kd + q * 16, n16);
          cp_async16(st_s + kKData + kKScale + n * 64 + c * 16, vd + q * 16, n16);
        }
        // V scales: 16 B = two tokens' 8 scale bytes
        cp_async16(st_s + kKData + kKScale + kVData + (p * kPageSize + 2 * sub) * 8,
                   a.v_scale + row0 * 8 + sub * 16, n16);
        if constexpr (L::kA4Q) {
          // K scales into the scale-factor atoms: 4 bytes = one token's scales
          // for one 64-value k-step
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int q = sub + 8 * i, r = q >> 1, ks = q & 1, n = p * kPageSize + r;
            cp_async4(st_s + kKData + ks * 512 + (n & 31) * 16 + (n >> 5) * 4, a.k_scale + (row0 + r) * 8 + 4 * ks,
                      n4);
          }
        } else {
          cp_async16(st_s + kKData + (p * kPageSize + 2 * sub) * 8, a.k_scale + row0 * 8 + sub * 16, n16);
        }
        cp_async_mbar_arrive(&bars.kv_full[st]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issue: one thread issues every QK (warp 0, lane 0) and another every PV
// (warp 3, lane 0).  A thread that issues tcgen05.mma is held until the
// tensor core has nearly finished it, so with a single issuer every barrier
// wait, commit and fence would sit between MMAs; with two, one thread's
// bookkeeping overlaps the other's MMAs.  Each thread's commits track its own
// MMAs.  The two streams meet only through the softmax: P(it) exists only
// after S(it) was read, so PV(it) finishing implies QK(it) finished.
template <int VARIANT, bool REPACK>
__device__ void qk_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase) {
  using L = Layout<VARIANT, REPACK>;
  const uint32_t q_s = smem_u32(smem + L::kOffQ);
  const uint32_t idesc_qk = L::kA4Q ? idesc_mxf4nvf4(128, 128) : idesc_f16(128, 128, 1, 1, 0, 0);
  uint32_t it_ctr = 0, item_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    if (!mbar_wait(bars.q_full, item_ctr & 1u, a.status)) return;
    for (int j = 0; j < item.n_tiles; ++j) {
      const uint32_t it = it_ctr + j;
      const uint32_t st = it % L::kStages, b = it & 1u;
      if (!mbar_wait(&bars.kv_full[st], (it / L::kStages) & 1u, a.status)) return;
      if constexpr (!L::kA4Q && !REPACK) {
        if (!mbar_wait(&bars.sfb_full[b], (it >> 1) & 1u, a.status)) return;
      }
      // S buffer b held S(it-2), and P(it-2) over it, until PV(it-2) read P
      // (FP4 PV: P is in shared memory, so until the softmax loaded S)
      if (it >= 2 && !mbar_wait(L::kFp4Pv ? &bars.s_free[b] : &bars.pv_done[b], ((it >> 1) - 1u) & 1u, a.status))
        return;
      tc_fence_after();
      const uint32_t s_col = b ? kColS1 : kColS0;
      const uint32_t stage_s = smem_u32(smem + L::kOffStage + st * L::kStageBytes);
      if constexpr (L::kA4Q) {
        // In-kernel mode the K codes and scale atoms arrived through
        // cp.async (generic proxy); the tensor core reads them next.
        if constexpr (!REPACK) fence_proxy_async_smem();
        // SFB buffer b was last read by QK(it-2), finished before the wait above.
        const uint32_t at_s = stage_s + kKData;
        tc_cp_32x128b_warpx4(tbase + kColSFB + 8 * b, smem_desc(at_s, 0, 128, kSwzNone));
        tc_cp_32x128b_warpx4(tbase + kColSFB + 8 * b + 4, smem_desc(at_s + 512, 0, 128, kSwzNone));
#pragma unroll
        for (uint32_t s = 0; s < 2; ++s) {
          mma_nvf4_ss(tbase + s_col, smem_desc(q_s + 32 * s, 16, 512, kSwz64),
                      smem_desc(stage_s + 32 * s, 16, 512, kSwz64), idesc_qk, tbase + kColSFA + 4 * s,
                      tbase + kColSFB + 8 * b + 4 * s, s > 0 ? 1u : 0u);
        }
      } else {
        const uint32_t k_s = REPACK ? stage_s : smem_u32(smem + L::kOffK + b * kTile16);
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_f16_ss(tbase + s_col, smem_desc(q_s + off, 16, 1024, kSwz128), smem_desc(k_s + off, 16, 1024, kSwz128),
                     idesc_qk, k > 0 ? 1u : 0u);
        }
      }
      tc_commit(&bars.s_full[b]);
      if (!REPACK) tc_commit(&bars.kv_empty[st]);  // the stage's K has been read
      if (j == item.n_tiles - 1) tc_commit(bars.q_empty);
    }
    it_ctr += item.n_tiles;
  }
}

template <int VARIANT, bool REPACK>
__device__ void pv_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase) {
  using L = Layout<VARIANT, REPACK>;
  const uint32_t idesc_pv = L::kFp4Pv ? idesc_mxf4nvf4(128, 128) : idesc_f16(128, 128, 0, 0, 0, 1);
  uint32_t it_ctr = 0, item_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    for (int j = 0; j < item.n_tiles; ++j) {
      const uint32_t it = it_ctr + j;
      const uint32_t st = it % L::kStages, b = it & 1u, ph = (it >> 1) & 1u;
      if (!mbar_wait(&bars.p_full[b], ph, a.status)) return;
      if (!REPACK && !mbar_wait(&bars.vdq_full[b], ph, a.status)) return;
      // the first PV of an item overwrites O: the previous item's epilogue
      // must have read it
      if (j == 0 && !mbar_wait(bars.o_empty, (item_ctr & 1u) ^ 1u, a.status)) return;
      tc_fence_after();
      const uint32_t v_s = REPACK ? smem_u32(smem + L::kOffStage + st * L::kStageBytes + L::kStageV)
                                  : smem_u32(smem + L::kOffV + b * kTile16);
      const uint32_t s_col = b ? kColS1 : kColS0;  // P(it) is over the first half of each half's S
      if constexpr (L::kFp4Pv) {
        // P (codes and scale atoms, written by the softmax warps) and the
        // record's token-major V.  Scale buffer b was last read by PV(it-2),
        // which had finished before the softmax wrote P(it).
        const uint32_t p_s = smem_u32(smem + L::kOffP + b * kPBuf);
        tc_cp_32x128b_warpx4(tbase + kColSFP + 8 * b, smem_desc(p_s + 8192, 0, 128, kSwzNone));
        tc_cp_32x128b_warpx4(tbase + kColSFP + 8 * b + 4, smem_desc(p_s + 8192 + 512, 0, 128, kSwzNone));
        tc_cp_32x128b_warpx4(tbase + kColSFV + 8 * b, smem_desc(v_s + kVData, 0, 128, kSwzNone));
        tc_cp_32x128b_warpx4(tbase + kColSFV + 8 * b + 4, smem_desc(v_s + kVData + 512, 0, 128, kSwzNone));
#pragma unroll
        for (uint32_t s = 0; s < 2; ++s) {
          mma_nvf4_ss(tbase + kColO, smem_desc(p_s + 32 * s, 16, 512, kSwz64), smem_desc(v_s + 32 * s, 16, 512, kSwz64),
                      idesc_pv, tbase + kColSFP + 8 * b + 4 * s, tbase + kColSFV + 8 * b + 4 * s,
                      (j == 0 && s == 0) ? 0u : 1u);
        }
      } else {
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k) {
          mma_f16_ts(tbase + kColO, tbase + s_col + (k < 4 ? 8 * k : 64 + 8 * (k - 4)),
                     smem_desc(v_s + k * 2048, 16384, 1024, kSwz128), idesc_pv, (j == 0 && k == 0) ? 0u : 1u);
        }
      }
      tc_commit(&bars.pv_done[b]);
      if (REPACK) tc_commit(&bars.kv_empty[st]);  // the stage's V tile has been read
    }
    tc_commit(bars.o_full);
    it_ctr += item.n_tiles;
  }
}

// ---------------------------------------------------------------------------
// The transform warpgroup's conversion of one 128-key tile of packed codes
// into a 128B-swizzled 16-bit operand tile: 512 units of 32 values (one key,
// group c of its 128 head dimensions), four per thread.  src(key, c, codes,
// scales) loads a unit's 16 code bytes and two block-scale bytes and returns
// false for a unit that stays zero.  Thread (warp w, lane l = 8 p + j), pass
// i takes key 8 (4 i + w) + 4 (p >> 1) + (j >> 1) and group c = (j & 1) |
// (((j >> 2) ^ p) & 1) << 1: the eight lanes of a phase hold four consecutive
// keys with both parities under each group, so their 16-byte code loads and
// each of their four 16-byte stores land in eight different bank groups, and
// key mod 8 (hence the swizzled chunk offsets) is the same in every pass.
template <bool BF16, class Src>
__device__ __forceinline__ void tf_convert_tile(uint8_t* tile, int tid, Src src) {
  const int lane = tid & 31, j8 = lane & 7, ph = lane >> 3;
  const int key_lo = 4 * (ph >> 1) + (j8 >> 1);
  const int c = (j8 & 1) | ((((j8 >> 2) ^ ph) & 1) << 1);
  const uint32_t cc = (c & 1) * 4, kx = key_lo & 7;
  uint8_t* dst0 = tile + (c >> 1) * 16384 + key_lo * 128;
  const uint32_t ch0 = ((cc + 0) ^ kx) << 4, ch1 = ((cc + 1) ^ kx) << 4;
  const uint32_t ch2 = ((cc + 2) ^ kx) << 4, ch3 = ((cc + 3) ^ kx) << 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key8 = 8 * (4 * i + (tid >> 5));
    uint32_t o0[4] = {0, 0, 0, 0}, o1[4] = {0, 0, 0, 0}, o2[4] = {0, 0, 0, 0}, o3[4] = {0, 0, 0, 0};
    uint4 v;
    uint32_t sc;
    if (src(key8 + key_lo, c, v, sc)) dequant_unit<BF16>(v, sc, o0, o1, o2, o3);
    uint8_t* dst = dst0 + key8 * 128;
    *reinterpret_cast<uint4*>(dst + ch0) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
    *reinterpret_cast<uint4*>(dst + ch1) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    *reinterpret_cast<uint4*>(dst + ch2) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
    *reinterpret_cast<uint4*>(dst + ch3) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
  }
}

// ---------------------------------------------------------------------------
// transform warpgroup (warps 4-7): thread = Q row / TMEM lane
template <int VARIANT, bool REPACK>
__device__ void transform_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase, int tid) {
  using L = Layout<VARIANT, REPACK>;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = a.group, lg = a.log2_group;
  float* qscale = reinterpret_cast<float*>(smem + L::kOffQScale);
  uint2* sfa_stage = reinterpret_cast<uint2*>(smem + L::kOffSfaStage);
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
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                        (static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq) * kHeadDim);
      if constexpr (L::kA4Q) {
        float g_row;
        sfa_stage[r] = quantize_q_row(src, valid, smem + L::kOffQ, r, a.q_g, g_row);
        qscale[r] = g_row;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sfa_ready);
        if (!mbar_wait_warp(bars.sfa_ready, item_ctr & 1u, a.status)) return;
        // Q block scales -> TMEM: lane i of each quadrant, column 4s+j holds
        // the four scales of k-step s for row 32j+i (replicated per quadrant).
        uint32_t va[8];
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint2 v = sfa_stage[32 * j + lane];
            va[4 * s2 + j] = s2 ? v.y : v.x;
          }
        tmem_st8(tmem_addr(tbase, 32 * warp, kColSFA), va);
        tmem_wait_st();
      } else {
        uint8_t* qt = smem + L::kOffQ;
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
          const uint4 v = valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(qt + (c >> 3) * 16384 + sw128_off(r, c & 7)) = v;
        }
        qscale[r] = 1.0f;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.q_full);
    }
    // ---- KV tiles (in-kernel mode: dequantize V, and K for dequant-ahead) ----
    if constexpr (!REPACK) {
      for (int j = 0; j < item.n_tiles; ++j) {
        const uint32_t it = it_ctr + j;
        const uint32_t st = it % L::kStages, b = it & 1u;
        // A4Q: the stage and the V buffer (read by PV(it-2)) are usually both
        // complete by now, and are tested at once so that the two round
        // trips overlap
        const uint32_t kv_ph = (it / L::kStages) & 1u, prev_ph = ((it >> 1) - 1u) & 1u;
        if (L::kA4Q && it >= 2 ? !mbar_wait2_warp(&bars.kv_full[st], kv_ph, &bars.pv_done[b], prev_ph, a.status)
                               : !mbar_wait_warp(&bars.kv_full[st], kv_ph, a.status))
          return;
        const uint8_t* stage = smem + L::kOffStage + st * L::kStageBytes;
        const int key_base = (item.t0 + j) * kBN;
        if constexpr (!L::kA4Q) {
          // K -> BF16 (exact), K-major 128B-swizzled operand; buffer b was
          // read by QK(it-2)
          if (it >= 2 && !mbar_wait_warp(&bars.s_full[b], prev_ph, a.status)) return;
          tf_convert_tile<true>(smem + L::kOffK + b * kTile16, tid, [&](int key, int c, uint4& v, uint32_t& sc) {
            v = *reinterpret_cast<const uint4*>(stage + sw64_off(key, c));
            sc = *reinterpret_cast<const uint16_t*>(stage + kKData + key * 8 + 2 * c);
            return true;
          });
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.sfb_full[b]);
        }
        // ---- V -> FP16, MN-major 128B-swizzled operand; buffer b was read by
        // PV(it-2) (A4Q: waited for above)
        if (!L::kA4Q && it >= 2 && !mbar_wait_warp(&bars.pv_done[b], prev_ph, a.status)) return;
        {
          const uint8_t* vd = stage + kKData + kKScale;
          const uint8_t* vs = vd + kVData;
          tf_convert_tile<false>(smem + L::kOffV + b * kTile16, tid, [&](int key, int c, uint4& v, uint32_t& sc) {
            if (key_base + key >= item.kv_len) return false;  // invalid pages were loaded as zeros
            v = *reinterpret_cast<const uint4*>(vd + key * 64 + 16 * c);
            sc = *reinterpret_cast<const uint16_t*>(vs + key * 8 + 2 * c);
            return true;
          });
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars.vdq_full[b]);
          mbar_arrive(&bars.kv_empty[st]);
        }
      }
    }
    it_ctr += item.n_tiles;
  }
}

// ---------------------------------------------------------------------------
// softmax warpgroups (warps 8-15): thread = TMEM lane = row; warpgroup `half`
// owns keys 64*half .. 64*half+63 of every tile and O columns of the same range
template <int VARIANT, bool REPACK>
__device__ void softmax_loop(const PrefillArgs& a, uint8_t* smem, const Bars& bars, uint32_t tbase, int r,
                             int half) {
  using L = Layout<VARIANT, REPACK>;
  const int quad = r >> 5, lane = r & 31;
  const int G = a.group, lg = a.log2_group;
  const float* qscale = reinterpret_cast<const float*>(smem + L::kOffQScale);
  float* xmax = reinterpret_cast<float*>(smem + L::kOffXmax);  // [parity][half][row]
  float* xl = reinterpret_cast<float*>(smem + L::kOffXl);      // [half][row]
  const uint32_t lane_base = tmem_addr(tbase, 32 * quad, 0);
  const uint32_t ocol = kColO + 64 * half;
  uint32_t it_ctr = 0, item_ctr = 0, xphase = 0;
  Item item;
  // The two halves of a row meet on xchg[quad]; every meeting is one phase.
  auto meet = [&]() -> bool {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.xchg[quad]);
    const bool ok = mbar_wait_warp(&bars.xchg[quad], xphase & 1u, a.status);
    ++xphase;
    tc_fence_after();
    return ok;
  };
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    if (!mbar_wait_warp(bars.q_full, item_ctr & 1u, a.status)) return;
    const int tq = item.tok0 + (r >> lg);
    const bool valid = (r >> lg) < item.n_tok;
    const int hq = item.kvh * G + (r & (G - 1));
    const int limit = !valid ? -1 : (a.causal ? item.kv_len - item.q_len + tq : item.kv_len - 1);
    const float c_r = (L::kA4Q ? qscale[r] : 1.0f) * a.k_g * a.sm_scale * kLog2e;
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.qs_empty);
    // A warp whose 32 rows all lie past the q tile's rows (a short q tile:
    // a tail of few query tokens, a request's last tile) computes nothing:
    // it waits for each S and arrives as if it had written its P, and its P
    // and O rows are never read out.  (Both halves of a row agree, so the
    // pair skips its meetings together.  QK(it+2) waits for PV(it), so such
    // a warp cannot run ahead by a phase; FP4 PV, whose QK waits only for
    // the S reads, keeps the full path.)
    const bool idle = !L::kFp4Pv && 32 * quad >= (item.n_tok << lg);
    float m_run = -INFINITY;
    float2 lacc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int j = 0; j < item.n_tiles; ++j) {
      const uint32_t it = it_ctr + j;
      const uint32_t b = it & 1u;
      const uint32_t s_col = b ? kColS1 : kColS0;
      if (!mbar_wait_warp(&bars.s_full[b], (it >> 1) & 1u, a.status)) return;
      if (idle) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[b]);
        continue;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(lane_base + s_col + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(lane_base + s_col + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      // FP4 PV: S is in registers and P goes to shared memory, so the
      // buffer may take QK(it+2) (otherwise P(it) is written over it and
      // QK(it+2) waits for PV(it))
      if constexpr (L::kFp4Pv) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.s_free[b]);
      }
      float* s = reinterpret_cast<float*>(sr);
      const int key0 = (item.t0 + j) * kBN + 64 * half;
      // Keys past the row's last visible one are masked (scale applied here);
      // unmasked halves fold the scale into the exponent's FMA below.
      const bool masked = key0 + 63 > limit;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = (key0 + c > limit) ? -INFINITY : s[c] * c_r;
      }
      float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
#pragma unroll
      for (int c = 6; c < 62; c += 4) {
        mx0 = fmax3(mx0, s[c], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
      }
      const float mx = fmax3(mx0, mx1, fmaxf(s[62], s[63]));
      const float m_half = masked ? mx : mx * c_r;
      float* xm = xmax + (j & 1) * 256;
      xm[half * 128 + r] = m_half;
      if (!meet()) return;  // both halves have read their S and published their max
      const float m_tile = fmaxf(m_half, xm[(half ^ 1) * 128 + r]);
      // Lazy rescale: the running max moves only when the tile max exceeds it
      // by more than 2^15.  TMEM loads/stores are warp-collective, so the
      // whole warp rescales its 64 O columns, with factor 1 for rows that keep
      // their max.  Both halves take identical decisions (same m_tile).
      // (FP4 PV: the threshold is 2^4 and the reference a whole number, so
      // alpha is an exact power of two and P <= 16 fits P's global scale.)
      float alpha = 1.0f;
      const bool need = m_tile > m_run + (L::kFp4Pv ? kTauFp4 : kRescaleThreshold);
      if (need) {
        if constexpr (L::kFp4Pv) {
          const float m_new = ceilf(m_tile);
          alpha = exp2_whole(m_run - m_new);
          m_run = m_new;
        } else {
          alpha = fast_exp2(m_run - m_tile);  // 0 when m_run = -inf
          m_run = m_tile;
        }
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < 4; ++i) lacc[i] = __fmul2_rn(lacc[i], a2);
      }
      const bool rescale_o = j > 0 && __any_sync(0xffffffffu, need);
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      const float cs = masked ? 1.0f : c_r;
      const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-m_use, -m_use);
      uint32_t pk[32];
      uint32_t pw[8], psc = 0u;  // FP4 PV: this half's P codes (4 blocks x 8 B) and block scales
      if constexpr (L::kFp4Pv) {
        // P coded per 16 keys by the block codec with global scale g_P: the
        // block scale from the block's largest p, which is 2^(its largest t)
        // since ex2 is monotone; each code from p * inv = 2^(t - log2(g_P *
        // scale)), the reciprocal folded into the exponent's addend.  These
        // roundings differ from the codec's own steps by about 1e-6 relative
        // only.  The row sum takes p = (code input) * g_P * scale, uncoded.
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const float* sb = s + 16 * blk;
          float mb = fmax3(sb[0], sb[1], sb[2]);
#pragma unroll
          for (int i = 3; i < 15; i += 2) mb = fmax3(mb, sb[i], sb[i + 1]);
          mb = fmaxf(mb, sb[15]);
          const float amax = fast_exp2(fmaf(mb, cs, -m_use));
          const uint32_t sc = cvt_e4m3x2(amax * kPInvSixG, 0.0f) & 0xFFu;
          const float sdec = e4m3_to_f32(sc);
          const float f = sdec > 0.0f ? kPScale * sdec : 1.0f;
          const float add = -m_use - fast_log2(f);
          const float2 add2 = make_float2(add, add);
          float2 qsum = make_float2(0.0f, 0.0f);
          uint32_t wlo = 0u, whi = 0u;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float2 t = __ffma2_rn(make_float2(sb[2 * c], sb[2 * c + 1]), cs2, add2);
            const float2 qq = make_float2(fast_exp2(t.x), fast_exp2(t.y));
            qsum = __fadd2_rn(qsum, qq);
            const uint32_t byte = cvt_e2m1x2(qq.x, qq.y);
            if (c < 4) wlo |= byte << (8 * c);
            else whi |= byte << (8 * (c - 4));
          }
          const bool live = sdec > 0.0f;  // a zero scale codes the block as zeros
          pw[2 * blk] = live ? wlo : 0u;
          pw[2 * blk + 1] = live ? whi : 0u;
          psc |= sc << (8 * blk);
          lacc[blk] = __ffma2_rn(qsum, make_float2(f, f), lacc[blk]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 t = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), cs2, nm2);
          const float2 p = make_float2(fast_exp2(t.x), fast_exp2(t.y));
          lacc[c & 3] = __fadd2_rn(lacc[c & 3], p);
          pk[c] = pack_f16x2(p.x, p.y);
        }
      }
      if constexpr (L::kFp4Pv) {
        // P buffer b was read by PV(it-2); O may be rescaled only once PV(it-1)
        // has finished (the later wait covers the earlier PV).
        if (rescale_o || it >= 2) {
          const uint32_t pit = it - (rescale_o ? 1u : 2u);
          if (!mbar_wait_warp(&bars.pv_done[pit & 1u], (pit >> 1) & 1u, a.status)) return;
          tc_fence_after();
        }
      } else if (rescale_o) {
        // O belongs to the tensor core until PV(it-1) has finished.  (P(it)
        // goes over S(it), which no PV reads before PV(it).)
        const uint32_t pit = it - 1u;
        if (!mbar_wait_warp(&bars.pv_done[pit & 1u], (pit >> 1) & 1u, a.status)) return;
        tc_fence_after();
      }
      if (rescale_o) {
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + ocol + 32 * c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st16(lane_base + ocol + 32 * c, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
          tmem_st16(lane_base + ocol + 32 * c + 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[16]));
        }
      }
      if constexpr (L::kFp4Pv) {
        // keys 64*half.. are chunks 2*half, 2*half+1 of row r and k-step
        // `half` of the scale atoms; the tensor core reads them next
        uint8_t* pb = smem + L::kOffP + b * kPBuf;
        *reinterpret_cast<uint4*>(pb + sw64_off(r, 2 * half)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(pb + sw64_off(r, 2 * half + 1)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
        *reinterpret_cast<uint32_t*>(pb + 8192 + 512 * half + (r & 31) * 16 + (r >> 5) * 4) = psc;
        fence_proxy_async_smem();
      } else {
        // P of keys 64*half.. over the first 32 of this half's S columns
        // (already read into registers; the other half's are not touched)
        tmem_st16(lane_base + s_col + 64 * half, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_st16(lane_base + s_col + 64 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[b]);
    }
    // ---- epilogue: combine the halves' row sums, scale this half of O ---------
    if (idle) {
      if (!mbar_wait_warp(bars.o_full, item_ctr & 1u, a.status)) return;
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.o_empty);
      it_ctr += item.n_tiles;
      continue;
    }
    const float l_half = (lacc[0].x + lacc[0].y) + (lacc[1].x + lacc[1].y) + (lacc[2].x + lacc[2].y) +
                         (lacc[3].x + lacc[3].y);
    xl[half * 128 + r] = l_half;
    if (!meet()) return;
    const float l_run = l_half + xl[(half ^ 1) * 128 + r];
    if (!mbar_wait_warp(bars.o_full, item_ctr & 1u, a.status)) return;
    tc_fence_after();
    // FP4 PV: O accumulated P's codes times its block scales; its global
    // scale is applied here
    const float o_mul = L::kFp4Pv ? kPScale : 1.0f;
    const float inv_l = (l_run > 0.0f) ? a.v_g * o_mul / l_run : 0.0f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) +
                          (static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq) * kHeadDim + 64 * half;
    float* prow = item.part >= 0 ? part_slot(a, item) : nullptr;  // split item: partial O, m, l
    if (prow && half == 0) {
      prow[kBM * kHeadDim + r] = m_run;
      prow[kBM * kHeadDim + kBM + r] = l_run;
    }
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t ov[32];
      tmem_ld32(lane_base + ocol + 32 * c, ov);
      tmem_wait_ld();
      if (prow) {
        float4* dst = reinterpret_cast<float4*>(prow + r * kHeadDim + 64 * half + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(ov[4 * i]) * o_mul, __uint_as_float(ov[4 * i + 1]) * o_mul,
                               __uint_as_float(ov[4 * i + 2]) * o_mul, __uint_as_float(ov[4 * i + 3]) * o_mul);
      } else if (valid) {
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
    if (!prow && half == 0 && valid && a.lse)
      a.lse[static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq] =
          (l_run > 0.0f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.o_empty);
    it_ctr += item.n_tiles;
  }
}

template <int VARIANT, bool REPACK>
__device__ __forceinline__ void prefill_body(const PrefillArgs& a) {
  using L = Layout<VARIANT, REPACK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  const Bars bars = make_bars(bar_base);
  if (tid == 0) {
    for (int i = 0; i < L::kStages; ++i) {
      mbar_init(&bars.kv_full[i], REPACK ? 1 : kLoaderThreads);  // bulk copy + tx, or one cp.async arrival per loader thread
      // one MMA commit, plus one arrive per transform warp when the transform
      // warpgroup reads the stage (in-kernel mode)
      mbar_init(&bars.kv_empty[i], REPACK ? 1 : 5);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.sfb_full[i], 4);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], 8);
      mbar_init(&bars.p_full[i], 8);
      mbar_init(&bars.vdq_full[i], 4);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(bars.o_full, 1);
    mbar_init(bars.o_empty, 8);
    mbar_init(bars.q_full, 4);
    mbar_init(bars.q_empty, 1);
    mbar_init(bars.drain, 2);  // one commit per MMA-issuing thread
    mbar_init(bars.qs_empty, 8);
    mbar_init(bars.sfa_ready, 4);
    for (int i = 0; i < 4; ++i) mbar_init(&bars.xchg[i], 2);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // The set-up above overlapped the tail of the schedule or repack kernel
  // before this one; its results are read only after this wait.  The merge
  // kernel, if any, may start its set-up now.
  grid_dep_launch();
  grid_dep_wait();

  if (tid >= kSoftmaxTid0) {
    softmax_loop<VARIANT, REPACK>(a, smem, bars, tbase, (tid - kSoftmaxTid0) & 127, (tid - kSoftmaxTid0) >> 7);
  } else if (tid >= kTransformTid0) {
    transform_loop<VARIANT, REPACK>(a, smem, bars, tbase, tid - kTransformTid0);
  } else if (warp == kLoaderWarp0 || warp == kLoaderWarp1) {
    loader_loop<VARIANT, REPACK>(a, smem, bars, (warp == kLoaderWarp0 ? 0 : 32) + lane);
  } else if ((warp == kMmaWarp || warp == kPvWarp) && lane == 0) {
    if (warp == kMmaWarp) qk_loop<VARIANT, REPACK>(a, smem, bars, tbase);
    else pv_loop<VARIANT, REPACK>(a, smem, bars, tbase);
    // drain: every MMA this thread issued has finished before TMEM is freed
    tc_commit(bars.drain);
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

// Kernel names carry the variant and the V path, so a trace shows which ran.
// (A4Q in repack mode runs the two-CTA kernel of prefill_a4q.cu.)
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_prefill_a4q_sm103_kernel(const PrefillArgs a) {
  prefill_body<0, false>(a);
}
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_prefill_dqahead_sm103_kernel(const PrefillArgs a) {
  prefill_body<1, false>(a);
}
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_prefill_dqahead_repack_sm103_kernel(const PrefillArgs a) {
  prefill_body<1, true>(a);
}
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_prefill_a4q_fp4pv_sm103_kernel(const PrefillArgs a) {
  prefill_body<2, true>(a);
}

// ---------------------------------------------------------------------------
// Token-major V (FP4 PV).  One block per (16 token rows, head dimension d):
// the rows' codes [16][64 B] and block scales [16][8 B] staged in shared
// memory; the 16 values at d decoded without the tensor scale (exact: E2M1 x
// E4M3) and coded by the cache's block codec with global scale 1.  Returns
// the block's scale byte; codes in w0 (rows 0-7) and w1 (rows 8-15), row 2i in
// the low nibble.
__device__ __forceinline__ uint32_t token_major_block(const uint8_t* codes, const uint8_t* scales, int d,
                                                      uint32_t& w0, uint32_t& w1) {
  float x[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const uint32_t h2 = cvt_e2m1x2_to_f16x2(codes[t * 64 + (d >> 1)]);
    const float e = __half2float(__ushort_as_half(static_cast<unsigned short>((d & 1) ? (h2 >> 16) : (h2 & 0xFFFFu))));
    x[t] = e * e4m3_to_f32(scales[t * 8 + (d >> 4)]);
  }
  return quant_block16(x, 1.0f, w0, w1);
}

// FP4 PV repack pre-pass: each (request, kv head, KV tile) once -> one 18 KB
// record laid out like a stage: K codes (64B-swizzled rows) | K scale atoms |
// token-major V codes (64B-swizzled [head dim][128 keys / 2]) | their scale
// atoms (k-step s: head dim d's four block scales at (d % 32) * 16 +
// (d / 32) * 4).  Keys past kv_len are zeros, in K and in the V blocks.
__global__ void __launch_bounds__(128) nvfp4_prefill_repack_fp4pv_kernel(PrefillArgs a) {
  using L = Layout<2, true>;
  __shared__ __align__(16) uint8_t sv[kBN * 64];  // the tile's V codes, as stored
  __shared__ __align__(16) uint8_t ss[kBN * 8];   // and V block scales
  grid_dep_launch();
  grid_dep_wait();  // the schedule
  const int tid = threadIdx.x;
  const int total = a.work[1];
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    int lo = 0, hi = a.batch - 1;  // last b with tile_prefix[b] * Hkv <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_prefix[mid] * a.num_kv_heads <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int n_t = a.tile_prefix[b + 1] - a.tile_prefix[b];
    const int r = t - a.tile_prefix[b] * a.num_kv_heads;
    const int h = r / n_t, j = r - h * n_t;
    const int kv_len = a.kv_lens[b];
    uint8_t* rec = a.repack + static_cast<int64_t>(t) * L::kStageBytes;
    auto row_of = [&](int key) -> int64_t {
      const int abs_key = j * kBN + key;
      if (abs_key >= kv_len) return -1;
      const int pid = a.page_table[static_cast<int64_t>(b) * a.max_pages + (abs_key >> 4)];
      if (pid < 0 || pid >= a.num_pages) {
        set_status(a.status, kDevBadPage);
        return -1;
      }
      return (static_cast<int64_t>(pid) * a.num_kv_heads + h) * kPageSize + (abs_key & 15);
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = tid + 128 * i, key = u >> 2, c = u & 3;
      const int64_t row = row_of(key);
      uint4 kw = make_uint4(0u, 0u, 0u, 0u), vw = make_uint4(0u, 0u, 0u, 0u);
      if (row >= 0) {
        kw = *reinterpret_cast<const uint4*>(a.k_data + row * 64 + 16 * c);
        vw = *reinterpret_cast<const uint4*>(a.v_data + row * 64 + 16 * c);
      }
      *reinterpret_cast<uint4*>(rec + sw64_off(key, c)) = kw;
      *reinterpret_cast<uint4*>(sv + key * 64 + 16 * c) = vw;
    }
    {
      const int key = tid;
      const int64_t row = row_of(key);
      uint2 ks = make_uint2(0u, 0u), vs = make_uint2(0u, 0u);
      if (row >= 0) {
        ks = *reinterpret_cast<const uint2*>(a.k_scale + row * 8);
        vs = *reinterpret_cast<const uint2*>(a.v_scale + row * 8);
      }
      *reinterpret_cast<uint32_t*>(rec + kKData + (key & 31) * 16 + (key >> 5) * 4) = ks.x;
      *reinterpret_cast<uint32_t*>(rec + kKData + 512 + (key & 31) * 16 + (key >> 5) * 4) = ks.y;
      *reinterpret_cast<uint2*>(ss + key * 8) = vs;
    }
    __syncthreads();
    // thread = head dimension: eight 16-key blocks along the tile's tokens
    const int d = tid;
    uint8_t* vt = rec + L::kStageV;
    uint32_t sc[2] = {0u, 0u};
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      uint32_t w0, w1;
      const uint32_t sb = token_major_block(sv + kb * 16 * 64, ss + kb * 16 * 8, d, w0, w1);
      *reinterpret_cast<uint2*>(vt + sw64_off(d, kb >> 1) + 8 * (kb & 1)) = make_uint2(w0, w1);
      sc[kb >> 2] |= sb << (8 * (kb & 3));
    }
    *reinterpret_cast<uint32_t*>(vt + kVData + (d & 31) * 16 + (d >> 5) * 4) = sc[0];
    *reinterpret_cast<uint32_t*>(vt + kVData + 512 + (d & 31) * 16 + (d >> 5) * 4) = sc[1];
    __syncthreads();  // the staging buffers take the next tile
  }
}

// The token-major blocks of whole pages, every slot as written: one CTA of
// 128 threads (one per head dimension) per (listed page, kv head).
__global__ void __launch_bounds__(128) nvfp4_v_token_major_kernel(TokenMajorArgs a) {
  __shared__ __align__(16) uint8_t sv[kPageSize * 64];
  __shared__ __align__(16) uint8_t ss[kPageSize * 8];
  const int tid = threadIdx.x;
  const int64_t total = static_cast<int64_t>(a.n_ids) * a.num_kv_heads;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    const int i = static_cast<int>(w / a.num_kv_heads), h = static_cast<int>(w - static_cast<int64_t>(i) * a.num_kv_heads);
    const int pid = a.page_ids[i];
    const bool ok = pid >= 0 && pid < a.num_pages;
    if (!ok && tid == 0) set_status(a.status, kDevBadPage);
    const int64_t row0 = (static_cast<int64_t>(ok ? pid : 0) * a.num_kv_heads + h) * kPageSize;
    if (tid < 64)
      *reinterpret_cast<uint4*>(sv + tid * 16) =
          ok ? *reinterpret_cast<const uint4*>(a.v_data + row0 * 64 + tid * 16) : make_uint4(0u, 0u, 0u, 0u);
    else if (tid < 72)
      *reinterpret_cast<uint4*>(ss + (tid - 64) * 16) =
          ok ? *reinterpret_cast<const uint4*>(a.v_scale + row0 * 8 + (tid - 64) * 16) : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    uint32_t w0, w1;
    const uint32_t sb = token_major_block(sv, ss, tid, w0, w1);
    *reinterpret_cast<uint2*>(a.codes + (w * kHeadDim + tid) * 8) = make_uint2(w0, w1);
    a.scales[w * kHeadDim + tid] = static_cast<uint8_t>(sb);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Dequant-ahead repack pre-pass: each (request, kv head, KV tile) once -> one
// record laid out exactly like a repack-mode stage, so the attention kernel
// moves it with a single bulk copy: K (BF16, K-major 128B-swizzled) | V (FP16,
// MN-major 128B-swizzled).  Keys past kv_len are zeros.  (A4Q records are
// written by the repack kernel of prefill_a4q.cu.)
__global__ void __launch_bounds__(128) nvfp4_prefill_repack_kernel(PrefillArgs a) {
  using L = Layout<1, true>;
  grid_dep_launch();
  grid_dep_wait();  // the schedule
  const int tid = threadIdx.x;
  const int total = a.work[1];
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    int lo = 0, hi = a.batch - 1;  // last b with tile_prefix[b] * Hkv <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_prefix[mid] * a.num_kv_heads <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int n_t = a.tile_prefix[b + 1] - a.tile_prefix[b];
    const int r = t - a.tile_prefix[b] * a.num_kv_heads;
    const int h = r / n_t, j = r - h * n_t;
    const int kv_len = a.kv_lens[b];
    uint8_t* rec = a.repack + static_cast<int64_t>(t) * L::kStageBytes;
    // cache row of key `key` of this tile, or -1 (past kv_len / invalid page)
    auto row_of = [&](int key) -> int64_t {
      const int abs_key = j * kBN + key;
      if (abs_key >= kv_len) return -1;
      const int pid = a.page_table[static_cast<int64_t>(b) * a.max_pages + (abs_key >> 4)];
      if (pid < 0 || pid >= a.num_pages) {
        set_status(a.status, kDevBadPage);
        return -1;
      }
      return (static_cast<int64_t>(pid) * a.num_kv_heads + h) * kPageSize + (abs_key & 15);
    };
    for (int tensor = 0; tensor < 2; ++tensor) {
      const uint8_t* data = tensor ? a.v_data : a.k_data;
      const uint8_t* scl = tensor ? a.v_scale : a.k_scale;
      uint8_t* dst = rec + (tensor ? L::kStageV : 0u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int u = tid + 128 * i;
        const int key = u >> 2, c = u & 3;
        const int64_t row = row_of(key);
        uint32_t o0[4] = {0, 0, 0, 0}, o1[4] = {0, 0, 0, 0}, o2[4] = {0, 0, 0, 0}, o3[4] = {0, 0, 0, 0};
        if (row >= 0) {
          const uint4 src = *reinterpret_cast<const uint4*>(data + row * 64 + 16 * c);
          const uint32_t sc01 = *reinterpret_cast<const uint16_t*>(scl + row * 8 + 2 * c);
          if (tensor) dequant_unit<false>(src, sc01, o0, o1, o2, o3);
          else dequant_unit<true>(src, sc01, o0, o1, o2, o3);
        }
        uint8_t* d = dst + (c >> 1) * 16384;
        const uint32_t cc = (c & 1) * 4;
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 0)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 1)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 2)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 3)) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) cache, the pages' comparison format: the attention of the
// dequant-ahead repack mode (BF16 QK with a BF16 query, FP16 PV) over records
// converted once per (request, kv head, 128-key tile) from FP8 pages of 128
// code bytes per token row.  Every E4M3 value is exact in FP16 and in BF16;
// the per-tensor scales are applied as k_g (in the score scale) and v_g (in
// the epilogue), as for NVFP4.
__device__ __forceinline__ void fp8_group_to_16bit(uint4 w0, uint4 w1, bool bf16, uint32_t (&o0)[4],
                                                   uint32_t (&o1)[4], uint32_t (&o2)[4], uint32_t (&o3)[4]) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t h[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[2 * i] = cvt_e4m3x2_to_f16x2(w[i] & 0xFFFFu);
    h[2 * i + 1] = cvt_e4m3x2_to_f16x2(w[i] >> 16);
  }
  if (bf16) {
    // f16 -> bf16 by moving the exponent field (value * 2^-112, exact for
    // every E4M3 value), then * 2^112 in bf16 (exact)
    const uint32_t two112 = 0x77807780u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t a = ((h[i] & 0x7FFF7FFFu) >> 3) | (h[i] & 0x80008000u);
      __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&two112));
      h[i] = *reinterpret_cast<uint32_t*>(&r);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o0[i] = h[i];
    o1[i] = h[4 + i];
    o2[i] = h[8 + i];
    o3[i] = h[12 + i];
  }
}

__global__ void __launch_bounds__(128) fp8_prefill_repack_kernel(PrefillArgs a) {
  using L = Layout<1, true>;
  grid_dep_launch();
  grid_dep_wait();  // the schedule
  const int tid = threadIdx.x;
  const int total = a.work[1];
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    int lo = 0, hi = a.batch - 1;  // last b with tile_prefix[b] * Hkv <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_prefix[mid] * a.num_kv_heads <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int n_t = a.tile_prefix[b + 1] - a.tile_prefix[b];
    const int r = t - a.tile_prefix[b] * a.num_kv_heads;
    const int h = r / n_t, j = r - h * n_t;
    const int kv_len = a.kv_lens[b];
    uint8_t* rec = a.repack + static_cast<int64_t>(t) * L::kStageBytes;
    for (int tensor = 0; tensor < 2; ++tensor) {
      const uint8_t* data = tensor ? a.v_data : a.k_data;
      uint8_t* dst = rec + (tensor ? L::kStageV : 0u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int u = tid + 128 * i;
        const int key = u >> 2, c = u & 3;
        const int abs_key = j * kBN + key;
        int64_t row = -1;
        if (abs_key < kv_len) {
          const int pid = a.page_table[static_cast<int64_t>(b) * a.max_pages + (abs_key >> 4)];
          if (pid < 0 || pid >= a.num_pages) set_status(a.status, kDevBadPage);
          else row = (static_cast<int64_t>(pid) * a.num_kv_heads + h) * kPageSize + (abs_key & 15);
        }
        uint32_t o0[4] = {0, 0, 0, 0}, o1[4] = {0, 0, 0, 0}, o2[4] = {0, 0, 0, 0}, o3[4] = {0, 0, 0, 0};
        if (row >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(data + row * kHeadDim + 32 * c);
          fp8_group_to_16bit(src[0], src[1], tensor == 0, o0, o1, o2, o3);
        }
        uint8_t* d = dst + (c >> 1) * 16384;
        const uint32_t cc = (c & 1) * 4;
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 0)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 1)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 2)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 3)) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
      }
    }
  }
}

// The dequant-ahead repack attention over records converted from FP8 pages
// (named for the format so that a trace shows which cache ran).
__global__ void __launch_bounds__(kThreads, 1) fp8_prefill_repack_sm103_kernel(const PrefillArgs a) {
  prefill_body<1, true>(a);
}

// ---------------------------------------------------------------------------
// schedule: items (request, q tile, kv head) sorted by decreasing KV-tile
// count, and the per-request KV-tile prefix used by repack mode
constexpr int kMaxCostBins = 4096;

// Inclusive prefix sum over the 1024 threads of the block.
__device__ __forceinline__ int block_inclusive_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) nvfp4_prefill_plan_kernel(PlanArgs a) {
  __shared__ int hist[kMaxCostBins];
  __shared__ int warp_sums[32];
  grid_dep_launch();  // the next kernel may start its set-up
  const int tid = threadIdx.x;
  int* prefix = a.work + 4 + 4 * a.max_items;  // [batch + 1] unit prefix (after the int4 items)
  int* tprefix = prefix + a.batch + 1;         // [batch + 1] KV-tile prefix
  const int tpq_shift = 7 - a.log2_group;      // log2(tokens per q tile)
  for (int i = tid; i < kMaxCostBins; i += blockDim.x) hist[i] = 0;
  // 1) units per request (q tiles x kv heads), KV tiles per request, prefixes
  int carry = 0, tcarry = 0;
  for (int base = 0; base < a.batch; base += blockDim.x) {
    const int b = base + tid;
    int cnt = 0, tiles = 0;
    if (b < a.batch) {
      const int q0 = a.qo_indptr[b], q1 = a.qo_indptr[b + 1];
      const int q_len = q1 - q0, kv_len = a.kv_lens[b];
      const bool bad = q_len < 0 || q0 < 0 || q1 > a.total_q || kv_len < 0 ||
                       kv_len > a.max_pages * kPageSize || (a.causal && q_len > kv_len);
      if (bad) {
        set_status(a.status, kDevBadShape);
      } else if (q_len > 0) {
        cnt = ((q_len + (1 << tpq_shift) - 1) >> tpq_shift) * a.num_kv_heads;
        tiles = max(1, (kv_len + a.bn - 1) / a.bn);
      }
    }
    const int incl = block_inclusive_scan(cnt, warp_sums);
    if (b < a.batch) prefix[b] = carry + incl - cnt;
    carry += warp_sums[31];  // block total of this chunk
    __syncthreads();
    const int tincl = block_inclusive_scan(tiles, warp_sums);
    if (b < a.batch) tprefix[b] = tcarry + tincl - tiles;
    tcarry += warp_sums[31];
    __syncthreads();
  }
  int total = carry;
  if (total > a.max_units) {  // cannot happen when qo_indptr is non-decreasing
    set_status(a.status, kDevBadShape);
    total = a.max_units;
  }
  if (tid == 0) {
    prefix[a.batch] = total;
    tprefix[a.batch] = tcarry;
    a.work[1] = tcarry * a.num_kv_heads;
    a.work[2] = total;
  }
  __shared__ int n_items;
  if (tid == 0) n_items = 0;
  __syncthreads();
  // unit u -> (request, q tile, kv head) and its KV tile count
  auto unit_of = [&](int u, int& b, int& qt, int& kvh) -> int {
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
    return last_key / a.bn + 1;
  };
  // Split KV: a unit of n tiles becomes min(split, n) items over contiguous
  // tile ranges (the part p of `parts` covers tiles n*p/parts .. n*(p+1)/parts - 1)
  // The number of parts S (at most a.split) minimizes the estimated makespan
  // ceil(units * S / ctas) / S of equal units on the kernel's CTAs; a unit is
  // cut into at most S parts of at least kMinSplitTiles tiles.
  __shared__ int s_split;
  if (tid == 0) {
    int best = 1;
    float best_t = static_cast<float>((total + a.ctas - 1) / max(a.ctas, 1));
    for (int sp = 2; sp <= a.split; ++sp) {
      const float t_sp = static_cast<float>((total * sp + a.ctas - 1) / a.ctas) / sp;
      if (t_sp < best_t * 0.999f) {
        best = sp;
        best_t = t_sp;
      }
    }
    s_split = best;
  }
  __syncthreads();
  const int split = s_split;
  auto parts_of = [&](int n) { return split > 1 ? min(split, max(1, n / kMinSplitTiles)) : 1; };
  // 2) histogram of item costs (tiles per item) and the item count
  for (int u = tid; u < total; u += blockDim.x) {
    int b, qt, kvh;
    const int n = unit_of(u, b, qt, kvh);
    const int parts = parts_of(n);
    for (int p = 0; p < parts; ++p) {
      const int cost = (n * (p + 1)) / parts - (n * p) / parts;
      atomicAdd(&hist[min(cost, kMaxCostBins - 1)], 1);
    }
    atomicAdd(&n_items, parts);
    if (a.split > 1) a.units[u] = make_int4(b, (qt << 8) | kvh, parts, n);
  }
  __syncthreads();
  if (tid == 0) a.work[0] = min(n_items, a.max_items);
  // 3) exclusive offsets, largest cost first: thread t owns 4 bins from the top
  constexpr int kPer = kMaxCostBins / 1024;
  int v[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = hist[kMaxCostBins - 1 - (tid * kPer + i)];
    sum += v[i];
  }
  int run = block_inclusive_scan(sum, warp_sums) - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    hist[kMaxCostBins - 1 - (tid * kPer + i)] = run;
    run += v[i];
  }
  __syncthreads();
  // 4) scatter the items: (request, q tile << 8 | kv head, first tile |
  // tiles << 16, partial slot or -1)
  int4* items = reinterpret_cast<int4*>(a.work + 4);
  for (int u = tid; u < total; u += blockDim.x) {
    int b, qt, kvh;
    const int n = unit_of(u, b, qt, kvh);
    const int parts = parts_of(n);
    for (int p = 0; p < parts; ++p) {
      const int t0 = (n * p) / parts, cnt = (n * (p + 1)) / parts - t0;
      const int pos = atomicAdd(&hist[min(cnt, kMaxCostBins - 1)], 1);
      if (pos < a.max_items)
        items[pos] = make_int4(b, (qt << 8) | kvh, t0 | (cnt << 16), parts > 1 ? u * a.split + p : -1);
    }
  }
}

// Split KV: merge the partial results of every unit that was split into
// several items.  One warp per row (16 rows per CTA), four head dimensions per
// lane: M = max_p m_p, w_p = 2^(m_p - M), O = sum_p w_p O_p / sum_p w_p l_p,
// times the V tensor scale (log-sum-exp combination in the log2 domain).
constexpr int kMergeRowsPerCta = 16;
constexpr int kMergeGroup = 8;  // parts whose rows a lane loads at once
__global__ void __launch_bounds__(32 * kMergeRowsPerCta) nvfp4_prefill_merge_kernel(PrefillArgs a) {
  grid_dep_wait();  // the attention kernel's partials
  const int u = blockIdx.x;
  const int4 info = a.units[u];  // (grid = the most units the workspace holds)
  if (u >= a.work[2]) return;
  const int parts = info.z;
  if (parts <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kMergeRowsPerCta + warp;
  const int b = info.x, qt = info.y >> 8, kvh = info.y & 255;
  const int G = a.group, lg = a.log2_group;
  const float* base = a.part + static_cast<int64_t>(u) * a.split * kPartFloats;
  // Loads that depend only on (unit, row) go out together: the request's
  // bounds, each part's row max and sum (lane p < parts), and the first
  // kMergeGroup parts' rows (r < kBM: inside the slot even for padding rows)
  const int q_start = a.qo_indptr[b], q_end = a.qo_indptr[b + 1];
  const float mp = lane < parts ? base[lane * kPartFloats + kBM * kHeadDim + r] : -INFINITY;
  const float lp = lane < parts ? base[lane * kPartFloats + kBM * kHeadDim + kBM + r] : 0.0f;
  float4 o4[kMergeGroup];
#pragma unroll
  for (int i = 0; i < kMergeGroup; ++i)
    o4[i] = i < parts ? reinterpret_cast<const float4*>(base + i * kPartFloats + r * kHeadDim)[lane]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  const int tok0 = qt * (kBM >> lg);
  const int n_rows = min(kBM >> lg, q_end - q_start - tok0) << lg;
  if (r >= n_rows) return;
  float m = mp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float mu = (m == -INFINITY) ? 0.0f : m;
  const float wp = lane < parts ? fast_exp2(mp - mu) : 0.0f;  // 0 for a part with no visible key
  float L = wp * lp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMergeGroup; ++i) {
    const float w = __shfl_sync(0xffffffffu, wp, i);  // 0 for i >= parts
    acc.x += w * o4[i].x;
    acc.y += w * o4[i].y;
    acc.z += w * o4[i].z;
    acc.w += w * o4[i].w;
  }
  for (int p = kMergeGroup; p < parts; ++p) {
    const float w = __shfl_sync(0xffffffffu, wp, p);
    const float4 v = reinterpret_cast<const float4*>(base + p * kPartFloats + r * kHeadDim)[lane];
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float sc = L > 0.0f ? a.v_g / L : 0.0f;
  const int tq = tok0 + (r >> lg), hq = kvh * G + (r & (G - 1));
  const int64_t orow = static_cast<int64_t>(q_start + tq) * a.num_q_heads + hq;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * sc, acc.y * sc), hi = __floats2bfloat162_rn(acc.z * sc, acc.w * sc);
  reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.o) + orow * kHeadDim)[lane] =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lane == 0 && a.lse) a.lse[orow] = (L > 0.0f) ? (mu + __log2f(L)) * kLn2 : -INFINITY;
}

template <typename K>
cudaError_t launch_main(K kernel, uint32_t smem, const PrefillArgs& a, int num_sms, cudaStream_t s) {
  cudaError_t e = set_kernel_smem(reinterpret_cast<const void*>(kernel), smem, false);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(num_sms), dim3(kThreads), smem, s, a);
}

}  // namespace

cudaError_t launch_prefill_plan(const PrefillArgs& a, const PlanArgs& plan, int variant, bool repack, int num_sms,
                                cudaStream_t s) {
  nvfp4_prefill_plan_kernel<<<1, 1024, 0, s>>>(plan);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !repack) return e;
  if (variant == 0) return launch_prefill_a4q_2cta_repack(a, num_sms, s);
  return launch_pdl(variant == 2 ? nvfp4_prefill_repack_fp4pv_kernel : nvfp4_prefill_repack_kernel,
                    dim3(num_sms * 8), dim3(128), 0, s, a);
}

size_t prefill_fp4pv_record_bytes() { return Layout<2, true>::kStageBytes; }

cudaError_t launch_v_token_major(const TokenMajorArgs& a, int num_sms, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(a.n_ids) * a.num_kv_heads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  nvfp4_v_token_major_kernel<<<static_cast<unsigned>(total < cap ? total : cap), 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_fp8(const PrefillArgs& a, const PlanArgs& plan, int num_sms, cudaStream_t s) {
  nvfp4_prefill_plan_kernel<<<1, 1024, 0, s>>>(plan);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(fp8_prefill_repack_kernel, dim3(num_sms * 8), dim3(128), 0, s, a)) != cudaSuccess) return e;
  if ((e = launch_main(fp8_prefill_repack_sm103_kernel, Layout<1, true>::kAlloc, a, num_sms, s)) != cudaSuccess)
    return e;
  return a.split > 1 ? launch_prefill_merge(a, s) : cudaSuccess;
}

cudaError_t launch_prefill_merge(const PrefillArgs& a, cudaStream_t s) {
  return launch_pdl(nvfp4_prefill_merge_kernel, dim3(a.max_units, kBM / kMergeRowsPerCta),
                    dim3(32 * kMergeRowsPerCta), 0, s, a);
}

cudaError_t launch_prefill_attend(const PrefillArgs& a, int variant, bool repack, int num_sms, cudaStream_t s) {
  if (variant == 2) return launch_main(nvfp4_prefill_a4q_fp4pv_sm103_kernel, Layout<2, true>::kAlloc, a, num_sms, s);
  if (variant == 0)
    return repack ? launch_prefill_a4q_2cta(a, num_sms, s)
                  : launch_main(nvfp4_prefill_a4q_sm103_kernel, Layout<0, false>::kAlloc, a, num_sms, s);
  return repack ? launch_main(nvfp4_prefill_dqahead_repack_sm103_kernel, Layout<1, true>::kAlloc, a, num_sms, s)
                : launch_main(nvfp4_prefill_dqahead_sm103_kernel, Layout<1, false>::kAlloc, a, num_sms, s);
}

}  // namespace nvfp4kv
