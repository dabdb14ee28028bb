// A4Q paged prefill, repack mode, two CTAs per SM ("NVFP4 KV cache A4Q
// prefill explained", sections "Quantize Q instead of expanding K" and
// "Compare A4Q with dequantize-ahead repacking").
//
// Same method as prefill.cu (per-row NVFP4 Q, block-scaled FP4 QK on the
// cache's own codes and scales, online softmax, FP16 PV on V converted once
// per tile), arranged so that two independent CTAs share each SM.  Each CTA
// owns one 128-row q tile at a time and 256 TMEM columns:
//
//   S half 0 (columns 0-63, keys 0-63 of the KV tile; its P as FP16 pairs
//   over 0-31), S half 1 (64-111, keys 64-111; P over 64-87), Q block scales
//   (112-119), K block scales (120-127), O (128-255, fp32)
//
// which is why a KV tile is 112 keys (7 pages).  The two halves of S work as
// a double buffer: the QK of one half runs while the softmax works on the
// other, and each half's PV starts as soon as its P is written.  The tensor
// operations of one thread run in issue order, so a QK queued right behind
// the PV of the same half overwrites S only after the PV has read P from it.
// The other CTA on the SM fills the tensor core's remaining gaps.  A softmax
// thread owns one whole row, so no row statistics are exchanged between
// warps.
//
//   warp 0 lane 0   TMEM allocation; every tensor operation: at each item
//                   start the tcgen05.cp of the item's Q scale atoms; per
//                   half, the tcgen05.cp of its K scale atoms, QK
//                   (kind::mxf4nvf4, N = 64 or 48), PV (kind::f16, P from
//                   TMEM)
//   warp 1 lane 0   one bulk copy per tile of the repacked record
//   warps 2-3       Q of the CTA's next item -> NVFP4 (two rows a thread)
//                   into the other of two Q buffers, with its block scales
//                   in the tcgen05.cp layout and the row scales, so that an
//                   item's first QK can run during the previous epilogue
//   warps 4-7       thread = row: Q of the CTA's first item (the same way),
//                   the softmax of every half tile, the epilogue
#include "prefill_common.cuh"

namespace nvfp4kv {

namespace {

using namespace prefill_detail;

constexpr int kBN2 = 112;
// A tile is two halves, keys 0-63 (h = 0) and 64-111 (h = 1), each with its
// own S columns, QK and PV, so that the QK of one half runs while the softmax
// works on the other.
__host__ __device__ constexpr int half_keys(int h) { return h == 0 ? 64 : kBN2 - 64; }
__host__ __device__ constexpr uint32_t half_col(int h) { return h == 0 ? 0u : 64u; }
constexpr int kThreads2 = 256;
constexpr int kStages2 = 2;
constexpr uint32_t kCols2 = 256;
constexpr uint32_t kColS2 = 0, kColSFA2 = 112, kColSFB2 = 120, kColO2 = 128;
constexpr uint32_t kKCodes2 = kBN2 * 64;                         // 7 KB, 64B-swizzled rows
constexpr uint32_t kKAtoms2 = 2048;  // per half: two k-steps x 512 B, the half's keys from row 0
constexpr uint32_t kVChunk2 = kBN2 * 128;                        // 64 head dims x 112 keys, FP16
constexpr uint32_t kRecord2 = kKCodes2 + kKAtoms2 + 2 * kVChunk2;  // 37 KB
static_assert(kRecord2 % 1024 == 0 && (kKCodes2 + kKAtoms2) % 1024 == 0, "1 KB aligned operands");

// per-thread register budgets: issue/loader warpgroup and softmax warpgroup
constexpr uint32_t kRegsIssue2 = 56, kRegsSoftmax2 = 200;
static_assert(128 * (kRegsIssue2 + kRegsSoftmax2) <= kThreads2 * 128, "register budgets exceed the launch");

// shared memory
constexpr uint32_t kOffQ2 = 0;                                   // [2] 8 KB FP4 Q tiles
constexpr uint32_t kOffStage2 = 16384;
constexpr uint32_t kOffQa2 = kOffStage2 + kStages2 * kRecord2;   // [2] Q scale atoms (two k-steps x 512 B)
constexpr uint32_t kOffQg2 = kOffQa2 + 2048;                     // [2][128] fp32 Q row scales
constexpr uint32_t kOffBar2 = kOffQg2 + 1024;
constexpr uint32_t kNumBars2 = 16;
constexpr uint32_t kOffSlot2 = kOffBar2 + kNumBars2 * 8;
constexpr uint32_t kAlloc2 = kOffSlot2 + 16 + 1024;              // + slack for 1 KB alignment
static_assert(2 * kAlloc2 <= 228 * 1024, "two CTAs per SM");

struct Bars2 {
  uint64_t* kv_full;   // [2]
  uint64_t* kv_empty;  // [2]
  uint64_t* s_full;    // [half] S of the half is in TMEM
  uint64_t* p_full;    // [half] P of the half written over its S (4 softmax warps)
  uint64_t* pv_done;   // [half] PV of the half finished
  uint64_t* q_full;    // [2] Q buffer b holds the item's Q tile and scales (warps 2-3)
  uint64_t* q_empty;   // [2] the item's last QK has finished and the softmax has its row scales
  uint64_t* o_empty;   // the epilogue has read O (4 softmax warps)
  uint64_t* drain;
};

__device__ __forceinline__ Bars2 make_bars2(uint64_t* base) {
  Bars2 b;
  b.kv_full = base + 0;
  b.kv_empty = base + 2;
  b.s_full = base + 4;
  b.p_full = base + 6;
  b.pv_done = base + 8;
  b.q_full = base + 10;   // 10, 11
  b.q_empty = base + 12;  // 12, 13
  b.o_empty = base + 14;
  b.drain = base + 15;
  return b;
}

// ---------------------------------------------------------------------------
// MMA thread.  Issue order, one 112-key tile j at a time:
//     PV_0(j)  QK_0(j+1)  PV_1(j)  QK_1(j+1)
// (half h: scale copy, then QK into the half's S; PV once the softmax has
// written the half's P).  The tensor operations of one thread run in issue
// order, so QK_h(j+1) overwrites S only after PV_h(j) has read P from it, and
// the scale copy for one half only after the other half's QK has read the
// previous scales.
template <int h>
__device__ __forceinline__ void qk_half(uint32_t q_s, uint32_t stage_s, uint32_t tbase) {
  const uint32_t at_s = stage_s + kKCodes2 + 1024u * h;
  tc_cp_32x128b_warpx4(tbase + kColSFB2, smem_desc(at_s, 0, 128, kSwzNone));
  tc_cp_32x128b_warpx4(tbase + kColSFB2 + 4, smem_desc(at_s + 512, 0, 128, kSwzNone));
  const uint32_t idesc = idesc_mxf4nvf4(128, half_keys(h));
  const uint32_t k_s = stage_s + 64u * 64u * h;  // K code rows of the half (64 B each)
#pragma unroll
  for (uint32_t s = 0; s < 2; ++s)
    mma_nvf4_ss(tbase + kColS2 + half_col(h), smem_desc(q_s + 32 * s, 16, 512, kSwz64),
                smem_desc(k_s + 32 * s, 16, 512, kSwz64), idesc, tbase + kColSFA2 + 4 * s, tbase + kColSFB2 + 4 * s,
                s > 0 ? 1u : 0u);
}

// The item's Q block scales: two tcgen05.cp of the staged atoms (k-steps 0, 1).
__device__ __forceinline__ void copy_q_scales(uint32_t qa_s, uint32_t tbase) {
  tc_cp_32x128b_warpx4(tbase + kColSFA2, smem_desc(qa_s, 0, 128, kSwzNone));
  tc_cp_32x128b_warpx4(tbase + kColSFA2 + 4, smem_desc(qa_s + 512, 0, 128, kSwzNone));
}

template <int h>
__device__ __forceinline__ void pv_half(uint32_t stage_s, uint32_t tbase, bool first, uint32_t idesc_pv) {
  const uint32_t v_s = stage_s + kKCodes2 + kKAtoms2;
#pragma unroll
  for (int k = 0; k < half_keys(h) / 16; ++k) {
    const int kk = (h == 0 ? 0 : 4) + k;  // 16-key step within the tile
    mma_f16_ts(tbase + kColO2, tbase + kColS2 + half_col(h) + 8 * k,
               smem_desc(v_s + kk * 2048, kVChunk2, 1024, kSwz128), idesc_pv, (first && kk == 0) ? 0u : 1u);
  }
}

__device__ __forceinline__ void mma_thread(const PrefillArgs& a, uint8_t* smem, const Bars2& bars, uint32_t tbase) {
  const uint32_t idesc_pv = idesc_f16(128, 128, 0, 0, 0, 1);
  uint32_t it = 0, item_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    const uint32_t qb = item_ctr & 1u;
    const uint32_t q_s = smem_u32(smem + kOffQ2 + qb * 8192);
    if (!mbar_wait(&bars.q_full[qb], (item_ctr >> 1) & 1u, a.status)) return;
    // prologue: the item's Q scales, both halves of tile 0 (the previous
    // item's QKs, issued earlier, have read the scale columns)
    uint32_t stage_s = smem_u32(smem + kOffStage2 + (it % kStages2) * kRecord2);
    if (!mbar_wait(&bars.kv_full[it % kStages2], (it / kStages2) & 1u, a.status)) return;
    tc_fence_after();
    copy_q_scales(smem_u32(smem + kOffQa2 + qb * 1024), tbase);
    qk_half<0>(q_s, stage_s, tbase);
    tc_commit(&bars.s_full[0]);
    qk_half<1>(q_s, stage_s, tbase);
    tc_commit(&bars.s_full[1]);
    if (item.n_tiles == 1) tc_commit(&bars.q_empty[qb]);
    for (int j = 0; j < item.n_tiles; ++j, ++it) {
      const uint32_t st = it % kStages2;
      const bool more = j + 1 < item.n_tiles;
      const uint32_t next_s = smem_u32(smem + kOffStage2 + ((it + 1) % kStages2) * kRecord2);
      // the item's first PV overwrites O: the previous epilogue must have read it
      if (j == 0 && !mbar_wait(bars.o_empty, (item_ctr & 1u) ^ 1u, a.status)) return;
      // half 0: PV of tile j, then QK of tile j + 1
      if (!mbar_wait(&bars.p_full[0], it & 1u, a.status)) return;
      tc_fence_after();
      pv_half<0>(stage_s, tbase, j == 0, idesc_pv);
      tc_commit(&bars.pv_done[0]);
      if (more) {
        if (!mbar_wait(&bars.kv_full[(it + 1) % kStages2], ((it + 1) / kStages2) & 1u, a.status)) return;
        tc_fence_after();
        qk_half<0>(q_s, next_s, tbase);
        tc_commit(&bars.s_full[0]);
      }
      // half 1
      if (!mbar_wait(&bars.p_full[1], it & 1u, a.status)) return;
      tc_fence_after();
      pv_half<1>(stage_s, tbase, j == 0, idesc_pv);
      tc_commit(&bars.pv_done[1]);
      tc_commit(&bars.kv_empty[st]);
      if (more) {
        qk_half<1>(q_s, next_s, tbase);
        tc_commit(&bars.s_full[1]);
        if (j + 2 == item.n_tiles) tc_commit(&bars.q_empty[qb]);
      }
      stage_s = next_s;
    }
  }
}

// ---------------------------------------------------------------------------
// Loader thread: one bulk copy per tile.
__device__ __forceinline__ void load_thread(const PrefillArgs& a, uint8_t* smem, const Bars2& bars) {
  uint32_t it = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round) {
    for (int j = 0; j < item.n_tiles; ++j, ++it) {
      const uint32_t st = it % kStages2;
      if (!mbar_wait(&bars.kv_empty[st], ((it / kStages2) & 1u) ^ 1u, a.status)) return;
      mbar_arrive_expect_tx(&bars.kv_full[st], kRecord2);
      bulk_load(smem + kOffStage2 + st * kRecord2, a.repack + repack_index(a, item.b, item.kvh, item.t0 + j) * kRecord2,
                kRecord2, &bars.kv_full[st]);
    }
  }
}

// ---------------------------------------------------------------------------
// Q warps (warps 2-3, thread t = 0..63): the Q tile of each of the CTA's
// items, rows t and t + 64, into Q buffer (item & 1) once the item two back
// has released it: FP4 codes (64B-swizzled rows), the block scales in the
// layout tcgen05.cp 32x128b.warpx4 expects (row 32 j + i at byte 16 i + 4 j
// of each k-step's 512 B), and the row scales.
__device__ __forceinline__ void stage_q_row(const PrefillArgs& a, uint8_t* smem, const Item& item, uint32_t qb, int r) {
  const int G = a.group, lg = a.log2_group;
  const int tq = item.tok0 + (r >> lg);
  const bool valid = (r >> lg) < item.n_tok;
  const int hq = item.kvh * G + (r & (G - 1));
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                    (static_cast<int64_t>(item.q_start + (valid ? tq : 0)) *
                                                         a.num_q_heads + hq) * kHeadDim);
  float g_row;
  const uint2 sw = quantize_q_row(src, valid, smem + kOffQ2 + qb * 8192, r, a.q_g, g_row);
  reinterpret_cast<float*>(smem + kOffQg2)[qb * 128 + r] = g_row;
  uint8_t* atoms = smem + kOffQa2 + qb * 1024;
  const int off = (r & 31) * 16 + (r >> 5) * 4;
  *reinterpret_cast<uint32_t*>(atoms + off) = sw.x;
  *reinterpret_cast<uint32_t*>(atoms + 512 + off) = sw.y;
}

// From the second item on (the softmax warps stage the first one).
__device__ __forceinline__ void q_warps(const PrefillArgs& a, uint8_t* smem, const Bars2& bars, int t) {
  uint32_t item_ctr = 1;
  Item item;
  for (int round = 1; get_item(a, round, item); ++round, ++item_ctr) {
    const uint32_t qb = item_ctr & 1u;
    if (item_ctr >= 2 && !mbar_wait_warp(&bars.q_empty[qb], ((item_ctr >> 1) - 1) & 1u, a.status)) return;
#pragma unroll 1
    for (int r = t; r < kBM; r += 64) stage_q_row(a, smem, item, qb, r);
    fence_proxy_async_smem();
    __syncwarp();
    if ((t & 31) == 0) mbar_arrive(&bars.q_full[qb]);
  }
}

// Softmax of half h of tile j for row lane_base's thread: S -> P (over S),
// running max and sum.  Returns false when a wait timed out.
template <int h>
__device__ __forceinline__ bool softmax_half(const PrefillArgs& a, const Bars2& bars, uint32_t lane_base, int lane,
                                             int j, int jt, uint32_t it, int limit, float c_r, float& m_run,
                                             float2 (&lacc)[4]) {
  constexpr int kMaxKeys = 64;
  constexpr int nk = half_keys(h);
  if (!mbar_wait_warp(&bars.s_full[h], it & 1u, a.status)) return false;
  tc_fence_after();
  uint32_t sr[kMaxKeys];
  const uint32_t s_addr = lane_base + kColS2 + half_col(h);
  tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
  if (h == 0) tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
  else tmem_ld16(s_addr + 32, *reinterpret_cast<uint32_t(*)[16]>(&sr[32]));
  tmem_wait_ld();
  float* s = reinterpret_cast<float*>(sr);
  const int key0 = jt * kBN2 + 64 * h;  // jt: the tile's index in the request
  // On a half with masked keys the kept scores are scaled here, so that a
  // zero row scale (an all-zero query row, or a row past the request) never
  // multiplies -inf
  const bool masked = key0 + nk - 1 > limit;
  if (masked) {
#pragma unroll
    for (int c = 0; c < nk; ++c) s[c] = (key0 + c > limit) ? -INFINITY : s[c] * c_r;
  }
  // half maximum (c_r >= 0 commutes with the maximum)
  float mxq[4];
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const float* sq = s + (nk / 4) * q4;
    float m = fmax3(sq[0], sq[1], sq[2]);
#pragma unroll
    for (int c = 3; c + 1 < nk / 4; c += 2) m = fmax3(m, sq[c], sq[c + 1]);
    if ((nk / 4) % 2 == 0) m = fmaxf(m, sq[nk / 4 - 1]);
    mxq[q4] = m;
  }
  const float mx = fmaxf(fmax3(mxq[0], mxq[1], mxq[2]), mxq[3]);
  const float m_tile = masked ? mx : mx * c_r;
  // Lazy rescale: the running max moves only when the half exceeds it by
  // more than 2^15 (P stays inside FP16).  O then holds the other
  // half's latest PV, which may still be running: wait for it first.
  const bool need = m_tile > m_run + kRescaleThreshold;
  float alpha = 1.0f;
  if (need) {
    alpha = fast_exp2(m_run - m_tile);  // 0 when m_run = -inf
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int i = 0; i < 4; ++i) lacc[i] = __fmul2_rn(lacc[i], a2);
    m_run = m_tile;
  }
  if ((h == 1 || j > 0) && __any_sync(0xffffffffu, need)) {
    if (!mbar_wait_warp(&bars.pv_done[1 - h], (h == 0 ? it - 1 : it) & 1u, a.status)) return false;
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t ov[32];
      tmem_ld32(lane_base + kColO2 + 32 * c, ov);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
      tmem_st16(lane_base + kColO2 + 32 * c, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
      tmem_st16(lane_base + kColO2 + 32 * c + 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[16]));
    }
  }
  const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
  const float cs = masked ? 1.0f : c_r;
  const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-m_use, -m_use);
  uint32_t pk[kMaxKeys / 2];
#pragma unroll
  for (int c = 0; c < nk / 2; ++c) {
    const float2 t = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), cs2, nm2);
    const float2 p = make_float2(fast_exp2(t.x), fast_exp2(t.y));
    lacc[c & 3] = __fadd2_rn(lacc[c & 3], p);
    pk[c] = pack_f16x2(p.x, p.y);
  }
  // P over the half's first nk/2 S columns (already read into registers)
  tmem_st16(s_addr, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
  if (h == 0) tmem_st16(s_addr + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
  else tmem_st8(s_addr + 16, *reinterpret_cast<uint32_t(*)[8]>(&pk[16]));
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.p_full[h]);
  return true;
}

// ---------------------------------------------------------------------------
// Softmax warpgroup: thread r = TMEM lane r = row r of the q tile.
__device__ __forceinline__ void softmax_rows(const PrefillArgs& a, uint8_t* smem, const Bars2& bars, uint32_t tbase,
                                             int r) {
  const int quad = r >> 5, lane = r & 31;
  const int G = a.group, lg = a.log2_group;
  const uint32_t lane_base = tmem_addr(tbase, 32 * quad, 0);
  uint32_t it = 0, item_ctr = 0;
  Item item;
  for (int round = 0; get_item(a, round, item); ++round, ++item_ctr) {
    const int tq = item.tok0 + (r >> lg);
    const bool valid = (r >> lg) < item.n_tok;
    const int hq = item.kvh * G + (r & (G - 1));
    const int limit = !valid ? -1 : (a.causal ? item.kv_len - item.q_len + tq : item.kv_len - 1);
    // ---- the item's row scale from the Q warps; its Q buffer is then free
    // as far as this warp is concerned
    const uint32_t qb = item_ctr & 1u;
    if (item_ctr == 0) {
      // the first item's Q: one row per thread, all four warps, then two
      // arrivals (as the Q warps make) once every row is staged
      stage_q_row(a, smem, item, 0, r);
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (lane == 0 && quad < 2) mbar_arrive(&bars.q_full[0]);
    }
    if (!mbar_wait_warp(&bars.q_full[qb], (item_ctr >> 1) & 1u, a.status)) return;
    const float c_r = reinterpret_cast<const float*>(smem + kOffQg2)[qb * 128 + r] * a.k_g * a.sm_scale * kLog2e;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.q_empty[qb]);

    float m_run = -INFINITY;
    float2 lacc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int j = 0; j < item.n_tiles; ++j, ++it) {
      if (!softmax_half<0>(a, bars, lane_base, lane, j, item.t0 + j, it, limit, c_r, m_run, lacc)) return;
      if (!softmax_half<1>(a, bars, lane_base, lane, j, item.t0 + j, it, limit, c_r, m_run, lacc)) return;
    }
    // ---- epilogue: O * v_scale / l -------------------------------------------
    const float l_run = (lacc[0].x + lacc[0].y) + (lacc[1].x + lacc[1].y) + (lacc[2].x + lacc[2].y) +
                        (lacc[3].x + lacc[3].y);
    if (!mbar_wait_warp(&bars.pv_done[1], (it - 1) & 1u, a.status)) return;
    tc_fence_after();
    const float inv_l = (l_run > 0.0f) ? a.v_g / l_run : 0.0f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) +
                          (static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq) * kHeadDim;
    float* prow = item.part >= 0 ? part_slot(a, item) : nullptr;  // split item: partial O, m, l
    if (prow) {
      prow[kBM * kHeadDim + r] = m_run;
      prow[kBM * kHeadDim + kBM + r] = l_run;
    }
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t ov[32];
      tmem_ld32(lane_base + kColO2 + 32 * c, ov);
      tmem_wait_ld();
      if (prow) {
        float4* dst = reinterpret_cast<float4*>(prow + r * kHeadDim + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                               __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
      } else if (valid) {
        uint32_t pb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __nv_bfloat162 v =
              __floats2bfloat162_rn(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
          pb[i] = *reinterpret_cast<uint32_t*>(&v);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
        dst[0] = make_uint4(pb[0], pb[1], pb[2], pb[3]);
        dst[1] = make_uint4(pb[4], pb[5], pb[6], pb[7]);
        dst[2] = make_uint4(pb[8], pb[9], pb[10], pb[11]);
        dst[3] = make_uint4(pb[12], pb[13], pb[14], pb[15]);
      }
    }
    if (!prow && valid && a.lse)
      a.lse[static_cast<int64_t>(item.q_start + tq) * a.num_q_heads + hq] =
          (l_run > 0.0f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.o_empty);
  }
}

__global__ void __launch_bounds__(kThreads2, 2) nvfp4_prefill_a4q_2cta_sm103_kernel(const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Bars2 bars = make_bars2(reinterpret_cast<uint64_t*>(smem + kOffBar2));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot2);
  if (tid == 0) {
    for (int i = 0; i < kStages2; ++i) {
      mbar_init(&bars.kv_full[i], 1);
      mbar_init(&bars.kv_empty[i], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bars.s_full[h], 1);
      mbar_init(&bars.p_full[h], 4);
      mbar_init(&bars.pv_done[h], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.q_full[b], 2);   // the two Q warps
      mbar_init(&bars.q_empty[b], 5);  // the item's last QK (commit) + the 4 softmax warps
    }
    mbar_init(bars.o_empty, 4);
    mbar_init(bars.drain, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kCols2);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // The set-up above overlapped the tail of the repack pre-pass (or the
  // schedule kernel) before this one; their results are read only now.
  grid_dep_launch();
  grid_dep_wait();
  // Register budgets (launched with 128 per thread): warps 0-3 give up to 56,
  // the softmax warpgroup takes 200; 128 x (56 + 200) = 32,768 = 256 x 128.
  if (warp >= 4) {
    regs_inc<kRegsSoftmax2>();
    softmax_rows(a, smem, bars, tbase, tid - 128);
  } else {
    regs_dec<kRegsIssue2>();
    if (warp == 0 && lane == 0) {
      mma_thread(a, smem, bars, tbase);
      tc_commit(bars.drain);  // every MMA of this thread has finished before TMEM is freed
    } else if (warp == 1 && lane == 0) {
      load_thread(a, smem, bars);
    } else if (warp >= 2) {
      q_warps(a, smem, bars, tid - 64);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) mbar_wait(bars.drain, 0, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kCols2);
  }
}

// ---------------------------------------------------------------------------
// Repack pre-pass for this kernel: each (request, kv head, 112-key tile) once
// -> one 37 KB record laid out exactly like a stage: K codes (64B-swizzled
// rows), the K scale atoms of each half (its keys from row 0, the remaining
// rows zero), V as FP16 in the MN-major 128B-swizzled operand layout (two
// chunks of 64 head dims x 112 keys).  Keys past kv_len are zeros.
__global__ void __launch_bounds__(128) nvfp4_prefill_repack112_kernel(PrefillArgs a) {
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
    const int rr = t - a.tile_prefix[b] * a.num_kv_heads;
    const int h = rr / n_t, j = rr - h * n_t;
    const int kv_len = a.kv_lens[b];
    uint8_t* rec = a.repack + static_cast<int64_t>(t) * kRecord2;
    auto row_of = [&](int key) -> int64_t {
      const int abs_key = j * kBN2 + key;
      if (key >= kBN2 || abs_key >= kv_len) return -1;
      const int pid = a.page_table[static_cast<int64_t>(b) * a.max_pages + (abs_key >> 4)];
      if (pid < 0 || pid >= a.num_pages) {
        set_status(a.status, kDevBadPage);
        return -1;
      }
      return (static_cast<int64_t>(pid) * a.num_kv_heads + h) * kPageSize + (abs_key & 15);
    };
    // K codes: 112 rows x 4 chunks of 16 B
    for (int u = tid; u < kBN2 * 4; u += 128) {
      const int key = u >> 2, c = u & 3;
      const int64_t row = row_of(key);
      const uint4 v = row >= 0 ? *reinterpret_cast<const uint4*>(a.k_data + row * 64 + 16 * c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(rec + sw64_off(key, c)) = v;
    }
    // K scale atoms of each half: 128 rows (the half's keys, then zeros) x 2
    // k-steps; half h starts at key 64 h
    for (int u = tid; u < 512; u += 128) {
      const int h = u >> 8, r = (u >> 1) & 127, ks = u & 1;
      const int key = 64 * h + r;
      const int64_t row = (r < half_keys(h)) ? row_of(key) : -1;
      const uint32_t w = row >= 0 ? *reinterpret_cast<const uint32_t*>(a.k_scale + row * 8 + 4 * ks) : 0u;
      *reinterpret_cast<uint32_t*>(rec + kKCodes2 + 1024 * h + ks * 512 + (r & 31) * 16 + (r >> 5) * 4) = w;
    }
    // V: 112 keys x 4 groups of 32 values -> FP16, MN-major 128B-swizzled
    uint8_t* vt = rec + kKCodes2 + kKAtoms2;
    for (int u = tid; u < kBN2 * 4; u += 128) {
      const int key = u >> 2, c = u & 3;
      const int64_t row = row_of(key);
      uint32_t o0[4] = {0, 0, 0, 0}, o1[4] = {0, 0, 0, 0}, o2[4] = {0, 0, 0, 0}, o3[4] = {0, 0, 0, 0};
      if (row >= 0) {
        const uint4 src = *reinterpret_cast<const uint4*>(a.v_data + row * 64 + 16 * c);
        const uint32_t sc01 = *reinterpret_cast<const uint16_t*>(a.v_scale + row * 8 + 2 * c);
        dequant_unit<false>(src, sc01, o0, o1, o2, o3);
      }
      uint8_t* d = vt + (c >> 1) * kVChunk2;
      const uint32_t cc = (c & 1) * 4;
      *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 0)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
      *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 1)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
      *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 2)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
      *reinterpret_cast<uint4*>(d + sw128_off(key, cc + 3)) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
    }
  }
}

}  // namespace

size_t prefill_a4q_2cta_record_bytes() { return kRecord2; }
int prefill_a4q_2cta_tile_keys() { return kBN2; }

cudaError_t launch_prefill_a4q_2cta_repack(const PrefillArgs& a, int num_sms, cudaStream_t s) {
  return launch_pdl(nvfp4_prefill_repack112_kernel, dim3(num_sms * 8), dim3(128), 0, s, a);
}

cudaError_t launch_prefill_a4q_2cta(const PrefillArgs& a, int num_sms, cudaStream_t s) {
  cudaError_t e = set_kernel_smem(reinterpret_cast<const void*>(nvfp4_prefill_a4q_2cta_sm103_kernel), kAlloc2, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(nvfp4_prefill_a4q_2cta_sm103_kernel, dim3(2 * num_sms), dim3(kThreads2), kAlloc2, s, a);
}

}  // namespace nvfp4kv
