// Paged decode over the NVFP4 cache: one query token per request attends to
// every cached token ("NVFP4 KV cache prefill vs decode performance", section
// "Decode can win on fewer bytes read": decode re-reads the whole history and
// is bandwidth-bound, so fewer bytes per token is the win).
//
// Split-KV: a work item is (request, kv head, split of up to S tokens), S one
// of 1024, 2048, 4096 or 8192: the schedule kernel takes the longest that
// still gives every attention CTA two items (each item costs a prologue, a
// merge of the four warps and a partial result).  It writes one record per
// item, full splits first and then the shorter last splits, longest first;
// one persistent wave of CTAs (3 per SM) claims records from a counter.  An item streams through two shared-memory
// stages of 256 tokens (K/V codes 1 KB + scales 128 B per page, gathered with
// cp.async by all threads and completing on one mbarrier), so the next unit's
// bytes are in flight while the current one is computed.  (Per-page bulk
// copies cost the copy engine a fixed time each, which capped the rate;
// cp.async spreads the same bytes over the load units.)  The schedule, the
// attention kernel and the combine kernel are chained by programmatic
// dependent launch.
//
// Four warps take 16-token chunks of a unit; the packed codes are dequantized
// (exactly: e2m1 x e4m3 fits f16) straight into MMA fragment registers, so no
// dequantized copy of K or V is ever written.
//   S^T = K q^T   m16n8k16 with the chunk's 16 tokens as the M rows and the
//               query heads as N.  The head dimension is permuted inside the
//               MMA's K index so that each lane converts 16 contiguous code
//               bytes of each of its two tokens; the query carries the same
//               permutation.
//   O^T += V^T P^T   m16n8k16 with head dimensions as the M rows (eight
//               m-tiles), the chunk's tokens as K and the heads as N.  P^T's
//               operand comes from the scores by one 8x8 transpose
//               (movmatrix) per token half, and lane (g, t) reads one 8-byte
//               code run (head dims 16g..16g+15, one scale block) per token.
// Queries are bf16; each head is multiplied by a power of two (exact) to sit
// inside f16's range and the factor is removed from the scores in fp32.  The
// running max moves lazily.  Partial (o, lse) per split are merged by a
// second kernel.
#include "kernels.cuh"

namespace nvfp4kv {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void mma_f16_16816(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// 8x8 transpose of b16 elements held in the MMA fragment layout: lane (g, t)
// gives row g, columns 2t, 2t+1 and receives row g, columns 2t, 2t+1 of the
// transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Dequantize four code bytes (eight values) times an f16x2 scale: out[i] holds
// the values of byte i (low nibble in the low half).  The bytes are taken as
// sub-registers of the word, so no shifts are needed.
__device__ __forceinline__ void dq4_f16(uint32_t w, uint32_t sc, uint32_t (&out)[4]) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
  const __half2 s2 = *reinterpret_cast<const __half2*>(&sc);
  __half2 r0 = __hmul2(*reinterpret_cast<__half2*>(&h0), s2), r1 = __hmul2(*reinterpret_cast<__half2*>(&h1), s2);
  __half2 r2 = __hmul2(*reinterpret_cast<__half2*>(&h2), s2), r3 = __hmul2(*reinterpret_cast<__half2*>(&h3), s2);
  out[0] = *reinterpret_cast<uint32_t*>(&r0);
  out[1] = *reinterpret_cast<uint32_t*>(&r1);
  out[2] = *reinterpret_cast<uint32_t*>(&r2);
  out[3] = *reinterpret_cast<uint32_t*>(&r3);
}

// log2 units: a head's running max moves only when a chunk exceeds it by more
// than this (P <= 2^15 stays inside FP16)
constexpr float kDecRescaleThreshold = 15.0f;

// Per-format layout of a shared-memory stage.  NVFP4: 64 code bytes and 8
// scale bytes per token row, 256-token units (K, K scales, V, V scales: 36 KB).
// FP8: 128 code bytes per token row, 128-token units (K, V: 32 KB), each row's
// 16-byte chunks XOR-swizzled by the row's low three bits so that the fragment
// loads of a warp spread over the banks.
template <bool FP8>
struct DecFmt {
  static constexpr int kUnit = FP8 ? 128 : 256;
  static constexpr int kRow = FP8 ? 128 : 64;        // code bytes per token row
  static constexpr int kBytesK = kUnit * kRow;
  static constexpr int kBytesS = FP8 ? 0 : kUnit * 8;
  static constexpr int kStage = 2 * (kBytesK + kBytesS);
  static constexpr int kPagesPerUnit = kUnit / kPageSize;
  static constexpr int kThrPerPage = 128 / kPagesPerUnit;  // gather threads per page
  static constexpr int kSmem = 2 * kStage + 1024;          // two stages + alignment slack
  // The four warps' partial O are merged through the stage just consumed:
  // [warp][head][kRedRow] fp32, rows padded by two words (where they fit) so
  // that the accumulator stores of a warp spread over the banks.
  static constexpr int kRedRow = (kDecWarps * 16 * (kHeadDim + 2) * 4 <= kStage) ? kHeadDim + 2 : kHeadDim;
  static_assert(kDecWarps * 16 * kRedRow * 4 <= kStage, "merge buffer fits one stage");
  static_assert(kThrPerPage == 8 || kThrPerPage == 16, "gather split");
};
constexpr int kDecCtasPerSm = 3;

struct DecItem {
  int b, h, split, tok0, n_tok, n_units;
};

// The schedule lists item records (request, kv head, split, tokens): full
// S-token items first, then the shorter last splits.  CTAs claim records in
// that order from a counter (sched[1]), so the short items fill the tail.
template <bool FP8>
__device__ __forceinline__ DecItem item_of(int4 r, int split_len) {
  DecItem it;
  it.b = r.x;
  it.h = r.y;
  it.split = r.z;
  it.tok0 = r.z * split_len;
  it.n_tok = r.w;
  it.n_units = (r.w + DecFmt<FP8>::kUnit - 1) / DecFmt<FP8>::kUnit;
  return it;
}

// Claimed records of this CTA in claim order, four deep: the copy cursor runs
// at most two units ahead of the compute, so at most three items are live.
struct ClaimRing {
  int4 rec[4];
  int n_valid;    // records claimed so far that hold an item
  int done;       // the schedule is exhausted
  int split_len;  // S of this call (sched[2])
};

// Claim the next record.  Every thread calls it, every time (its barrier
// must be met by all threads); only thread 0 reads or writes the ring's
// state before the barrier, and it claims nothing once the schedule is
// exhausted.
__device__ __forceinline__ void claim_item(const DecodeArgs& a, ClaimRing* ring) {
  if (threadIdx.x == 0 && !ring->done) {
    const int idx = atomicAdd(a.sched + 1, 1);
    if (idx < a.sched[0]) {
      ring->rec[ring->n_valid & 3] = reinterpret_cast<const int4*>(a.sched + 4)[idx];
      ++ring->n_valid;
    } else {
      ring->done = 1;
    }
  }
  __syncthreads();
}

// Tokens of unit u of an item (at most one unit).
template <bool FP8>
__device__ __forceinline__ int unit_tokens(const DecItem& it, int u) {
  return min(DecFmt<FP8>::kUnit, it.n_tok - u * DecFmt<FP8>::kUnit);
}

// Raw page id of the page this thread gathers for unit u of an item (page
// tid / 8 of the unit), or -1 past the unit.  Loaded one unit ahead so that
// the global-load latency is off the path of the gather; checked there.
template <bool FP8>
__device__ __forceinline__ int unit_page(const DecodeArgs& a, const DecItem& it, int u, int tid) {
  const int p = tid / DecFmt<FP8>::kThrPerPage;
  if (p * kPageSize >= unit_tokens<FP8>(it, u)) return -1;
  return a.page_table[static_cast<int64_t>(it.b) * a.max_pages +
                      (it.tok0 + u * DecFmt<FP8>::kUnit) / kPageSize + p];
}

// All 128 threads gather unit u of an item into `stage` with cp.async: thread
// t serves page t / 8 (K and V codes, 16 B at a time, plus one 16-byte piece
// of each scale page; V code rows are permuted, see the PV step).  A page with an invalid id (flagged) reads as zeros,
// and so do the V scales of tokens past the item's end -- their values are
// then exactly 0 whatever codes the page holds.  Each thread arrives on `bar`
// once its copies land.
template <bool FP8>
__device__ __forceinline__ void issue_unit(const DecodeArgs& a, const DecItem& it, int u, int pid, uint8_t* stage,
                                           uint64_t* bar, int* page_ok, int tid) {
  using F = DecFmt<FP8>;
  constexpr int kThrPerPage = F::kThrPerPage;
  const int p = tid / kThrPerPage, sub = tid % kThrPerPage;
  const int n_tok = unit_tokens<FP8>(it, u);
  if constexpr (FP8) {
    // FP8: thread t copies 8 of the 128 16-byte chunks of page t / 16 of K
    // and of V.  Rows of tokens past the item's end, and pages with an
    // invalid id (flagged), read as zeros: E4M3 has NaN codes, and a NaN V
    // value would reach the output through a zero softmax weight.
    if (p * kPageSize < n_tok) {
      if (pid >= a.num_pages || pid < 0) {
        if (sub == 0) set_status(a.status, kDevBadPage);
        pid = -1;
      }
      if (sub == 0) page_ok[p] = pid >= 0;
      const int live = pid >= 0 ? min(n_tok - p * kPageSize, kPageSize) : 0;
      const int64_t row = (static_cast<int64_t>(pid >= 0 ? pid : 0) * a.num_kv_heads + it.h) * kPageSize;
      const uint32_t sK = smem_u32(stage), sV = sK + F::kBytesK;
      const uint8_t* gk = a.k_data + row * 128;
      const uint8_t* gv = a.v_data + row * 128;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = sub + 16 * i;       // chunk of the page: token c / 8, piece c % 8
        const int tok = c >> 3, r = p * kPageSize + tok;
        const uint32_t n = tok < live ? 16u : 0u;
        const uint32_t dst = r * 128 + (((c & 7) ^ (r & 7)) << 4);
        cp_async16(sK + dst, gk + c * 16, n);
        cp_async16(sV + dst, gv + c * 16, n);
      }
    }
    cp_async_mbar_arrive(bar);
    return;
  }
  if (p * kPageSize < n_tok) {
    if (pid >= a.num_pages || pid < 0) {
      if (sub == 0) set_status(a.status, kDevBadPage);
      pid = -1;
    }
    if (sub == 0) page_ok[p] = pid >= 0;
    const uint32_t n16 = pid >= 0 ? 16u : 0u;
    // V scales of tokens 2 ps, 2 ps + 1 of this page: 8 bytes per live token
    const int ps = sub & 7;
    const int live = min(max(n_tok - p * kPageSize - 2 * ps, 0), 2);
    const uint32_t nvs = pid >= 0 ? 8u * live : 0u;
    const int64_t row = (static_cast<int64_t>(pid >= 0 ? pid : 0) * a.num_kv_heads + it.h) * kPageSize;
    const uint32_t sK = smem_u32(stage), sKs = sK + F::kBytesK, sV = sKs + F::kBytesS, sVs = sV + F::kBytesK;
    const uint8_t* gk = a.k_data + row * 64;
    const uint8_t* gv = a.v_data + row * 64;
#pragma unroll
    for (int i = 0; i < 64 / kThrPerPage; ++i) {
      const int c = sub + kThrPerPage * i;
      const int vrow = c >> 2, vprow = vrow ^ ((vrow >> 1) & 1);  // V row permutation (bank spread)
      cp_async16(sK + p * 1024 + c * 16, gk + c * 16, n16);
      cp_async16(sV + p * 1024 + (vprow * 4 + (c & 3)) * 16, gv + c * 16, n16);
    }
    if (kThrPerPage == 8 || sub < 8) cp_async16(sKs + p * 128 + ps * 16, a.k_scale + row * 8 + ps * 16, n16);
    if (kThrPerPage == 8 || sub >= 8) cp_async16(sVs + p * 128 + ps * 16, a.v_scale + row * 8 + ps * 16, nvs);
  }
  cp_async_mbar_arrive(bar);
}

// Raw bf16 query rows of an item for lane (g, t): d = 32t .. 32t+31 of heads
// g and g+8 (zeros past the group).  Loaded one item ahead.
template <int G>
__device__ __forceinline__ void load_q_raw(const DecodeArgs& a, const DecItem& it, int g, int t, uint4 (&qr)[2][4]) {
  const uint16_t* qb =
      reinterpret_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(it.b) * a.num_q_heads + it.h * G) * kHeadDim;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int head = g + 8 * r;
    const bool live = (r == 0 || G > 8) && head < G;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      qr[r][i] = live ? reinterpret_cast<const uint4*>(qb + head * kHeadDim + 32 * t)[i] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The copy cursor: (claimed item ci, unit u) of the next unit to gather.
struct UnitCursor {
  int ci, u;
  bool has;
  DecItem it;
};
template <bool FP8>
__device__ __forceinline__ void cursor_load(ClaimRing* ring, UnitCursor& c) {
  c.has = c.ci < ring->n_valid;
  if (c.has) c.it = item_of<FP8>(ring->rec[c.ci & 3], ring->split_len);
}
template <bool FP8>
__device__ __forceinline__ void cursor_start(const DecodeArgs& a, ClaimRing* ring, UnitCursor& c) {
  c.ci = 0;
  c.u = 0;
  claim_item(a, ring);
  cursor_load<FP8>(ring, c);
}
template <bool FP8>
__device__ __forceinline__ void cursor_next(const DecodeArgs& a, ClaimRing* ring, UnitCursor& c) {
  if (++c.u >= c.it.n_units) {
    c.u = 0;
    ++c.ci;
    claim_item(a, ring);
    cursor_load<FP8>(ring, c);
  }
}

// Persistent: CTAs claim items from the schedule.  Each item (up to S
// tokens) streams through two shared-memory stages of one unit (256 tokens
// of NVFP4, 128 of FP8), so the copies of the next unit run while the current
// one is computed; the four warps' partial results are merged once per item.
template <int G, bool FP8>
__device__ __forceinline__ void decode_body(const DecodeArgs& a) {
  using F = DecFmt<FP8>;
  constexpr bool kTwoRows = G > 8;  // MMA rows g+8 carry heads 8..15
  constexpr int kHeadBlocks = kTwoRows ? 2 : 1;
  extern __shared__ __align__(128) uint8_t dsmem_raw[];
  uint8_t* dsmem = dsmem_raw + ((128u - (smem_u32(dsmem_raw) & 127u)) & 127u);
  __shared__ uint64_t bars[2];
  __shared__ int page_ok_sh[2][F::kPagesPerUnit];
  __shared__ float red_m[kDecWarps][16], red_l[kDecWarps][16];
  __shared__ float mw[kDecWarps][16];   // merge weights exp2(m_w - m) / L per head
  __shared__ ClaimRing ring;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  if (tid == 0) {
    mbar_init(&bars[0], 128);  // one cp.async arrival per thread
    mbar_init(&bars[1], 128);
    fence_barrier_init();
    ring.n_valid = 0;
    ring.done = 0;
  }
  __syncthreads();
  grid_dep_launch();  // the combine grid may be scheduled as CTAs finish
  grid_dep_wait();    // the schedule written by the plan kernel
  if (tid == 0) ring.split_len = a.sched[2];  // seen by all after the first claim's barrier
  // issue cursor: two units ahead of the compute
  UnitCursor ic;
  cursor_start<FP8>(a, &ring, ic);
  for (int s = 0; s < 2 && ic.has; ++s) {
    issue_unit<FP8>(a, ic.it, ic.u, unit_page<FP8>(a, ic.it, ic.u, tid), dsmem + s * F::kStage, &bars[s],
                    page_ok_sh[s], tid);
    cursor_next<FP8>(a, &ring, ic);
  }
  DecItem it;
  uint4 qr[2][4];
  bool q_ready = false;  // qr holds the query rows of the next item to compute
  uint32_t uc = 0;  // units consumed: stage uc & 1, phase (uc >> 1) & 1
  for (int k = 0; k < ring.n_valid; ++k) {
    it = item_of<FP8>(ring.rec[k & 3], ring.split_len);
    const int b = it.b, h = it.h;
    if (!q_ready) load_q_raw<G>(a, it, g, t, qr);
    q_ready = false;
    // ---- query fragments from the rows loaded one item ahead ------------------
    // B operand of S^T = K q^T: lane (g, t) owns head dims 32t .. 32t+31 of
    // head g (+8 for the second block); MMA j's k positions 2t, 2t+1 are dims
    // 32t + 4j + {0, 1} and positions 2t+8, 2t+9 are dims 32t + 4j + {2, 3}.
    uint32_t qb[kHeadBlocks][8][2];
    float crow[kHeadBlocks][2];  // score scale of heads 2t, 2t+1 (+8 nb)
#pragma unroll
    for (int nb = 0; nb < kHeadBlocks; ++nb) {
      float x[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 w = qr[nb][i];
        bf16x2_to_f32(w.x, x[8 * i + 0], x[8 * i + 1]);
        bf16x2_to_f32(w.y, x[8 * i + 2], x[8 * i + 3]);
        bf16x2_to_f32(w.z, x[8 * i + 4], x[8 * i + 5]);
        bf16x2_to_f32(w.w, x[8 * i + 6], x[8 * i + 7]);
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // power of two bringing the head's amax into [2^14, 2^15): exact in f16
      const int e = (amax > 0.0f) ? (14 - ilogbf(amax)) : 0;
      const float up = ldexpf(1.0f, e);
      const float c_own = a.sm_scale * a.k_g * kLog2e * ldexpf(1.0f, -e);  // head g (+8 nb)
      crow[nb][0] = __shfl_sync(0xffffffffu, c_own, 8 * t);
      crow[nb][1] = __shfl_sync(0xffffffffu, c_own, 8 * t + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qb[nb][j][0] = pack_f16x2(x[4 * j] * up, x[4 * j + 1] * up);
        qb[nb][j][1] = pack_f16x2(x[4 * j + 2] * up, x[4 * j + 3] * up);
      }
    }

    // Row state of heads 2t, 2t+1 (+8 nb): all lanes of a column group t hold
    // the same running max, and a partial sum over their own tokens.
    float m_run[kHeadBlocks][2], l_run[kHeadBlocks][2];
#pragma unroll
    for (int nb = 0; nb < kHeadBlocks; ++nb) {
      m_run[nb][0] = m_run[nb][1] = -INFINITY;
      l_run[nb][0] = l_run[nb][1] = 0.0f;
    }
    // O^T accumulators: m-tile mt holds head dims 16g + 2mt (row g) and
    // 16g + 2mt + 1 (row g+8) for heads 2t, 2t+1 (+8 for the second block)
    float acc[kHeadBlocks][8][4];
#pragma unroll
    for (int nb = 0; nb < kHeadBlocks; ++nb)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[nb][mt][0] = acc[nb][mt][1] = acc[nb][mt][2] = acc[nb][mt][3] = 0.0f;

    for (int u = 0; u < it.n_units; ++u, ++uc) {
      const int stg = uc & 1;
      uint8_t* sK = dsmem + stg * F::kStage;
      uint8_t* sKs = sK + F::kBytesK;  // NVFP4 only
      uint8_t* sV = sKs + F::kBytesS;
      uint8_t* sVs = sV + F::kBytesK;  // NVFP4 only
      const int* page_ok = page_ok_sh[stg];
      const int n_tok = unit_tokens<FP8>(it, u);
      // the page this thread gathers for the unit issued after this one, and
      // the next item's query rows once that item is claimed
      const int pid_next = ic.has ? unit_page<FP8>(a, ic.it, ic.u, tid) : -1;
      if (!q_ready && k + 1 < ring.n_valid) {
        load_q_raw<G>(a, item_of<FP8>(ring.rec[(k + 1) & 3], ring.split_len), g, t, qr);
        q_ready = true;
      }
      const bool ok = mbar_wait(&bars[stg], (uc >> 1) & 1, a.status);
      const int n_chunks = ok ? (n_tok + 15) / 16 : 0;
      for (int c = warp; c < n_chunks; c += kDecWarps) {
        const int cbase = c * 16;
        const bool page_valid = page_ok[c] != 0;
        // ---- S^T = K q^T: m rows are the chunk's tokens (lane rows g, g+8),
        // n columns the heads.  Each lane converts 16 code bytes of each of
        // its two tokens, whose byte pairs are the A registers of MMAs 2wi and
        // 2wi + 1.
        float s[kHeadBlocks][4];
#pragma unroll
        for (int nb = 0; nb < kHeadBlocks; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.0f;
        if constexpr (FP8) {
          // lane (g, t): 32 code bytes (head dims 32t .. 32t+31) of tokens g
          // and g + 8; word j holds dims 32t + 4j + 0..3, whose halves are the
          // A registers (k positions 2t, 2t+1 and 2t+8, 2t+9) of MMA j.  The
          // per-tensor scale is part of the score scale.
          const int tok0 = cbase + g, tok1 = tok0 + 8;
          const int x0 = tok0 & 7, x1 = tok1 & 7;  // chunk swizzle of the rows
          const uint4 k0a = *reinterpret_cast<const uint4*>(sK + tok0 * 128 + (((2 * t) ^ x0) << 4));
          const uint4 k0b = *reinterpret_cast<const uint4*>(sK + tok0 * 128 + (((2 * t + 1) ^ x0) << 4));
          const uint4 k1a = *reinterpret_cast<const uint4*>(sK + tok1 * 128 + (((2 * t) ^ x1) << 4));
          const uint4 k1b = *reinterpret_cast<const uint4*>(sK + tok1 * 128 + (((2 * t + 1) ^ x1) << 4));
          const uint32_t kw0[8] = {k0a.x, k0a.y, k0a.z, k0a.w, k0b.x, k0b.y, k0b.z, k0b.w};
          const uint32_t kw1[8] = {k1a.x, k1a.y, k1a.z, k1a.w, k1b.x, k1b.y, k1b.z, k1b.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t a0 = cvt_e4m3x2_to_f16x2(kw0[j] & 0xFFFFu), a2 = cvt_e4m3x2_to_f16x2(kw0[j] >> 16);
            const uint32_t a1 = cvt_e4m3x2_to_f16x2(kw1[j] & 0xFFFFu), a3 = cvt_e4m3x2_to_f16x2(kw1[j] >> 16);
#pragma unroll
            for (int nb = 0; nb < kHeadBlocks; ++nb)
              mma_f16_16816(s[nb][0], s[nb][1], s[nb][2], s[nb][3], a0, a1, a2, a3, qb[nb][j][0], qb[nb][j][1]);
          }
        } else {
          const int tok0 = cbase + g, tok1 = tok0 + 8;
          const uint4 k0 = *reinterpret_cast<const uint4*>(sK + tok0 * 64 + 16 * t);
          const uint4 k1 = *reinterpret_cast<const uint4*>(sK + tok1 * 64 + 16 * t);
          const uint32_t hs0 = cvt_e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sKs + tok0 * 8 + 2 * t));
          const uint32_t hs1 = cvt_e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sKs + tok1 * 8 + 2 * t));
          const uint32_t sc0[2] = {prmt(hs0, hs0, 0x1010u), prmt(hs0, hs0, 0x3232u)};
          const uint32_t sc1[2] = {prmt(hs1, hs1, 0x1010u), prmt(hs1, hs1, 0x3232u)};
          const uint32_t kw0[4] = {k0.x, k0.y, k0.z, k0.w}, kw1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            uint32_t h0[4], h1[4];
            dq4_f16(kw0[wi], sc0[wi >> 1], h0);
            dq4_f16(kw1[wi], sc1[wi >> 1], h1);
#pragma unroll
            for (int nb = 0; nb < kHeadBlocks; ++nb) {
              mma_f16_16816(s[nb][0], s[nb][1], s[nb][2], s[nb][3], h0[0], h1[0], h0[1], h1[1], qb[nb][2 * wi][0],
                            qb[nb][2 * wi][1]);
              mma_f16_16816(s[nb][0], s[nb][1], s[nb][2], s[nb][3], h0[2], h1[2], h0[3], h1[3],
                            qb[nb][2 * wi + 1][0], qb[nb][2 * wi + 1][1]);
            }
          }
        }
        // ---- online softmax (log2 domain), lazy rescale.  Lane (g, t) holds
        // tokens g and g+8 of heads 2t, 2t+1 (+8 nb).
        const int lim = page_valid ? n_tok - cbase : 0;
        const bool live0 = g < lim, live1 = g + 8 < lim;
        uint32_t pb[kHeadBlocks][2];
#pragma unroll
        for (int nb = 0; nb < kHeadBlocks; ++nb) {
          float x[4];
          x[0] = live0 ? s[nb][0] * crow[nb][0] : -INFINITY;
          x[1] = live0 ? s[nb][1] * crow[nb][1] : -INFINITY;
          x[2] = live1 ? s[nb][2] * crow[nb][0] : -INFINITY;
          x[3] = live1 ? s[nb][3] * crow[nb][1] : -INFINITY;
          // The running max moves only when the chunk exceeds it by more than
          // 2^15, so P stays inside FP16.  A head's chunk max can pass that
          // bound only if one of its lanes does, so the reduction over the
          // eight lanes of a column group runs only then.
          float cm0 = fmaxf(x[0], x[2]), cm1 = fmaxf(x[1], x[3]);
          if (__any_sync(0xffffffffu, cm0 > m_run[nb][0] + kDecRescaleThreshold ||
                                          cm1 > m_run[nb][1] + kDecRescaleThreshold)) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, o));
              cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, o));
            }
            const bool need0 = cm0 > m_run[nb][0] + kDecRescaleThreshold;
            const bool need1 = cm1 > m_run[nb][1] + kDecRescaleThreshold;
            const float al0 = need0 ? fast_exp2(m_run[nb][0] - cm0) : 1.0f;  // 0 when m_run = -inf
            const float al1 = need1 ? fast_exp2(m_run[nb][1] - cm1) : 1.0f;
            if (need0) m_run[nb][0] = cm0;
            if (need1) m_run[nb][1] = cm1;
            l_run[nb][0] *= al0;
            l_run[nb][1] *= al1;
            // O^T columns 2t, 2t+1 are this lane's heads
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              acc[nb][mt][0] *= al0;
              acc[nb][mt][1] *= al1;
              acc[nb][mt][2] *= al0;
              acc[nb][mt][3] *= al1;
            }
          }
          const float mu0 = (m_run[nb][0] == -INFINITY) ? 0.0f : m_run[nb][0];
          const float mu1 = (m_run[nb][1] == -INFINITY) ? 0.0f : m_run[nb][1];
          const float p0 = fast_exp2(x[0] - mu0), p1 = fast_exp2(x[1] - mu1);
          const float p2 = fast_exp2(x[2] - mu0), p3 = fast_exp2(x[3] - mu1);
          l_run[nb][0] += p0 + p2;
          l_run[nb][1] += p1 + p3;
          // P^T as the B operand of PV: an 8x8 transpose of each token half
          pb[nb][0] = movmatrix_trans(pack_f16x2(p0, p1));
          pb[nb][1] = movmatrix_trans(pack_f16x2(p2, p3));
        }
        // ---- O^T += V^T P^T: A = V^T (rows: head dims, k: tokens), B = P^T
        // Lane (g, t) needs tokens 2t, 2t+1, 8+2t, 9+2t at code bytes 8g..8g+7
        // (head dims 16g..16g+15: one scale block).  The nibbles of a token
        // pair (a, b) are interleaved byte by byte before conversion, so each
        // converted f16 pair is (token a, token b) at one head dimension: an
        // A-fragment register as it stands.  The pair's two scales form one
        // f16x2 multiplier.  V rows sit in shared memory with row r stored at
        // r ^ ((r >> 1) & 1), so the four rows 2t + c of a load hit both
        // halves of the banks.
        uint32_t va[2][16];  // [pair][2j + e]: head dim 16g + 2j + e, j = 0..7
        if constexpr (FP8) {
          // FP8: 16 code bytes (head dims 16g .. 16g+15) of each token of the
          // pair; byte i of token a and byte i of token b form one E4M3 pair,
          // converted to the f16 pair (a, b) at head dim 16g + i.
#pragma unroll
          for (int tp = 0; tp < 2; ++tp) {
            const int tok_a = cbase + 8 * tp + 2 * t, tok_b = tok_a + 1;
            const uint4 ca = *reinterpret_cast<const uint4*>(sV + tok_a * 128 + ((g ^ (tok_a & 7)) << 4));
            const uint4 cb = *reinterpret_cast<const uint4*>(sV + tok_b * 128 + ((g ^ (tok_b & 7)) << 4));
            const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w}, wb[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint32_t lo = prmt(wa[w], wb[w], 0x5140u), hi = prmt(wa[w], wb[w], 0x7362u);
              va[tp][4 * w + 0] = cvt_e4m3x2_to_f16x2(lo & 0xFFFFu);
              va[tp][4 * w + 1] = cvt_e4m3x2_to_f16x2(lo >> 16);
              va[tp][4 * w + 2] = cvt_e4m3x2_to_f16x2(hi & 0xFFFFu);
              va[tp][4 * w + 3] = cvt_e4m3x2_to_f16x2(hi >> 16);
            }
          }
        } else {
#pragma unroll
        for (int tp = 0; tp < 2; ++tp) {
          const int tok_a = cbase + 8 * tp + 2 * t;
          const uint2 ca = *reinterpret_cast<const uint2*>(sV + (tok_a ^ (t & 1)) * 64 + 8 * g);
          const uint2 cb = *reinterpret_cast<const uint2*>(sV + ((tok_a + 1) ^ (t & 1)) * 64 + 8 * g);
          const uint32_t sab =
              static_cast<uint32_t>(sVs[tok_a * 8 + g]) | (static_cast<uint32_t>(sVs[(tok_a + 1) * 8 + g]) << 8);
          const uint32_t sc = cvt_e4m3x2_to_f16x2(sab);
          const uint32_t wa[2] = {ca.x, ca.y}, wb[2] = {cb.x, cb.y};
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint32_t ev = (wa[h2] & 0x0F0F0F0Fu) | ((wb[h2] << 4) & 0xF0F0F0F0u);
            const uint32_t od = ((wa[h2] >> 4) & 0x0F0F0F0Fu) | (wb[h2] & 0xF0F0F0F0u);
            uint32_t e4[4], o4[4];
            dq4_f16(ev, sc, e4);
            dq4_f16(od, sc, o4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              va[tp][2 * (4 * h2 + i)] = e4[i];
              va[tp][2 * (4 * h2 + i) + 1] = o4[i];
            }
          }
        }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const uint32_t a0 = va[0][2 * mt], a1 = va[0][2 * mt + 1], a2 = va[1][2 * mt], a3 = va[1][2 * mt + 1];
#pragma unroll
          for (int nb = 0; nb < kHeadBlocks; ++nb)
            mma_f16_16816(acc[nb][mt][0], acc[nb][mt][1], acc[nb][mt][2], acc[nb][mt][3], a0, a1, a2, a3, pb[nb][0],
                          pb[nb][1]);
        }
      }
      const bool last = u == it.n_units - 1;
      if (last) {
        // ---- merge the four warps through this stage's shared memory ---------
#pragma unroll
        for (int nb = 0; nb < kHeadBlocks; ++nb)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            l_run[nb][0] += __shfl_xor_sync(0xffffffffu, l_run[nb][0], o);
            l_run[nb][1] += __shfl_xor_sync(0xffffffffu, l_run[nb][1], o);
          }
        __syncthreads();  // every warp is done reading the stage
        float* red_o = reinterpret_cast<float*>(sK);  // [warp][G][F::kRedRow]
#pragma unroll
        for (int r = 0; r < kHeadBlocks; ++r) {
          if (g == 0) {
            red_m[warp][8 * r + 2 * t] = m_run[r][0];
            red_l[warp][8 * r + 2 * t] = l_run[r][0];
            red_m[warp][8 * r + 2 * t + 1] = m_run[r][1];
            red_l[warp][8 * r + 2 * t + 1] = l_run[r][1];
          }
          if (8 * r + 2 * t < G) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int d = 16 * g + 2 * mt;
              float* o0 = red_o + (warp * G + 8 * r + 2 * t) * F::kRedRow;
              *reinterpret_cast<float2*>(o0 + d) = make_float2(acc[r][mt][0], acc[r][mt][2]);
              if (8 * r + 2 * t + 1 < G)
                *reinterpret_cast<float2*>(o0 + F::kRedRow + d) = make_float2(acc[r][mt][1], acc[r][mt][3]);
            }
          }
        }
        __syncthreads();
        const bool single = a.kv_lens[b] <= ring.split_len;
        // per head: the combined max and sum, and each warp's weight
        // exp2(m_w - m) / L, computed once
        if (tid < G) {
          const int head = tid;
          float m = -INFINITY;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, red_m[w][head]);
          const float mu = (m == -INFINITY) ? 0.0f : m;
          float f[kDecWarps], L = 0.0f;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) {
            f[w] = fast_exp2(red_m[w][head] - mu);
            L += red_l[w][head] * f[w];
          }
          const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) mw[w][head] = f[w] * inv;
          const float lse2 = (L > 0.0f) ? mu + __log2f(L) : -INFINITY;
          const int hq = h * G + head;
          if (single) {
            if (a.lse) a.lse[static_cast<int64_t>(b) * a.num_q_heads + hq] = lse2 * kLn2;
          } else {
            a.part_lse[(static_cast<int64_t>(b) * a.max_splits + it.split) * a.num_q_heads + hq] = lse2;
          }
        }
        __syncthreads();
        for (int i = tid; i < G * kHeadDim; i += 128) {
          const int head = i >> 7, d = i & 127;
          float on = 0.0f;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) on += red_o[(w * G + head) * F::kRedRow + d] * mw[w][head];
          const int hq = h * G + head;
          if (single) {
            reinterpret_cast<__nv_bfloat16*>(a.o)[(static_cast<int64_t>(b) * a.num_q_heads + hq) * kHeadDim + d] =
                __float2bfloat16_rn(on * a.v_g);
          } else {
            a.part_o[((static_cast<int64_t>(b) * a.max_splits + it.split) * a.num_q_heads + hq) * kHeadDim + d] = on;
          }
        }
      }
      __syncthreads();  // every thread is done with this stage
      if (ic.has) {
        issue_unit<FP8>(a, ic.it, ic.u, pid_next, dsmem + stg * F::kStage, &bars[stg], page_ok_sh[stg], tid);
        cursor_next<FP8>(a, &ring, ic);
      }
    }
  }
}

template <int G>
__global__ void __launch_bounds__(128, kDecCtasPerSm) nvfp4_paged_decode_kernel(DecodeArgs a) {
  decode_body<G, false>(a);
}
template <int G>
__global__ void __launch_bounds__(128, kDecCtasPerSm) fp8_paged_decode_kernel(DecodeArgs a) {
  decode_body<G, true>(a);
}

// Block-wide exclusive prefix sums of two counts (returns the exclusive
// values; *total receives the sums).  blockDim.x is a multiple of 32.
__device__ __forceinline__ int2 block_exclusive_scan2(int2 v, int2* warp_sums, int2* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int2 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(0xffffffffu, x.x, o), ny = __shfl_up_sync(0xffffffffu, x.y, o);
    if (lane >= o) {
      x.x += nx;
      x.y += ny;
    }
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int2 w = lane < nw ? warp_sums[lane] : make_int2(0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nx = __shfl_up_sync(0xffffffffu, w.x, o), ny = __shfl_up_sync(0xffffffffu, w.y, o);
      if (lane >= o) {
        w.x += nx;
        w.y += ny;
      }
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int2 before = wid > 0 ? warp_sums[wid - 1] : make_int2(0, 0);
  *total = warp_sums[nw - 1];
  __syncthreads();
  return make_int2(x.x + before.x - v.x, x.y + before.y - v.y);
}

// Schedule: one record per (request, kv head, S-token split).  S is the
// longest of kDecSplit << k (k < kDecSplitSteps) whose items number at least
// two per attention CTA, else kDecSplit.  All full splits come first; then
// each request's shorter last split, longest first, so that the items
// claimed last are the shortest.  Requests are taken kPlanThreads at a time
// (one pass for the usual batch sizes); the longest-first order holds within
// each such chunk.  Every CTA of the grid computes the same S and prefix
// sums and writes its share of the records.
constexpr int kPlanThreads = 256, kPlanCtas = 16;
static_assert(kDecSplitSteps == 4, "the split choice reduces four counts");
__global__ void __launch_bounds__(kPlanThreads) nvfp4_decode_plan_kernel(DecodeArgs a) {
  grid_dep_launch();  // the attention grid may start its prologue now
  __shared__ int2 warp_sums[32];
  __shared__ int req_len[kPlanThreads], req_first[kPlanThreads], req_fpos[kPlanThreads], req_ppos[kPlanThreads];
  int4* items = reinterpret_cast<int4*>(a.sched + 4);
  const int tid = threadIdx.x, H = a.num_kv_heads, cap = a.max_pages * kPageSize;
  // ---- the split length S
  int split_len = kDecSplit;
  {
    int c[kDecSplitSteps] = {0, 0, 0, 0};  // items per kv head for each candidate
    for (int b = tid; b < a.batch; b += blockDim.x) {
      const int kv = a.kv_lens[b];
      if (kv > 0 && kv <= cap)
#pragma unroll
        for (int k = 0; k < kDecSplitSteps; ++k) c[k] += (kv + (kDecSplit << k) - 1) / (kDecSplit << k);
    }
    int2 t01, t23;
    block_exclusive_scan2(make_int2(c[0], c[1]), warp_sums, &t01);
    block_exclusive_scan2(make_int2(c[2], c[3]), warp_sums, &t23);
    const int tot[kDecSplitSteps] = {t01.x, t01.y, t23.x, t23.y};
#pragma unroll
    for (int k = 1; k < kDecSplitSteps; ++k)
      if (static_cast<int64_t>(tot[k]) * H >= 2 * static_cast<int64_t>(a.ctas)) split_len = kDecSplit << k;
  }
  // total of the full items of all requests (the partial ones follow them)
  int n_full_total = 0;
  if (a.batch > static_cast<int>(blockDim.x)) {
    for (int base = 0; base < a.batch; base += blockDim.x) {
      const int b = base + tid;
      const int kv_len = b < a.batch ? a.kv_lens[b] : 0;
      int2 tot;
      block_exclusive_scan2(make_int2(kv_len > 0 && kv_len <= cap ? kv_len / split_len : 0, 0), warp_sums, &tot);
      n_full_total += tot.x * H;
    }
  }
  int full_carry = 0, part_carry = 0;
  for (int base = 0; base < a.batch; base += blockDim.x) {
    const int b = base + tid;
    const int n_req = min(static_cast<int>(blockDim.x), a.batch - base);
    int kv_len = 0;
    if (b < a.batch) {
      kv_len = a.kv_lens[b];
      if (kv_len > cap) set_status(a.status, kDevBadShape);
      if (kv_len < 0 || kv_len > cap) kv_len = 0;
    }
    const int full = kv_len / split_len, plen = kv_len % split_len;
    req_len[tid] = plen;
    int2 tot;
    const int2 ex = block_exclusive_scan2(make_int2(full, plen > 0 ? 1 : 0), warp_sums, &tot);
    if (a.batch <= static_cast<int>(blockDim.x)) n_full_total = tot.x * H;
    // rank of this request's last split among the chunk's: longer first,
    // then request order
    int rank = 0;
    if (plen > 0) {
      for (int j = 0; j < n_req; ++j) {
        const int lj = req_len[j];
        rank += (lj > plen || (lj == plen && j < tid)) ? 1 : 0;
      }
    }
    __syncthreads();  // every thread has read req_len
    req_len[tid] = kv_len;
    req_fpos[tid] = full_carry + ex.x * H;
    req_ppos[tid] = n_full_total + part_carry + rank * H;
    req_first[tid] = (ex.x + ex.y) * H;
    __syncthreads();
    const int rtot = (tot.x + tot.y) * H;
    for (int i = tid + blockIdx.x * blockDim.x; i < rtot; i += blockDim.x * gridDim.x) {
      int lo = 0, hi = n_req - 1;  // last request of the chunk with req_first <= i
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (req_first[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const int len = req_len[lo], rfull = len / split_len;
      const int j = i - req_first[lo];
      const int sp = j / H, h = j - sp * H;
      if (sp < rfull) items[req_fpos[lo] + sp * H + h] = make_int4(base + lo, h, sp, split_len);
      else items[req_ppos[lo] + h] = make_int4(base + lo, h, rfull, len - rfull * split_len);
    }
    __syncthreads();
    full_carry += tot.x * H;
    part_carry += tot.y * H;
  }
  if (tid == 0 && blockIdx.x == 0) {
    a.sched[0] = full_carry + part_carry;
    a.sched[1] = 0;  // claim counter of the attention kernel
    a.sched[2] = split_len;
  }
}

// Merge the split partials of requests with more than one split; write zeros
// for empty requests.  One CTA per (q head, request), one thread per head
// dimension.  Every thread reads the splits' lse and its own column of the
// partial O eight splits at a time, all loads of a group issued together,
// and merges online (running max, rescaled sum and accumulator), so the
// merge costs about one memory round trip per eight splits and needs no
// shared memory or barrier.
constexpr int kCombineGroup = 8;
__global__ void __launch_bounds__(128) nvfp4_decode_combine_kernel(DecodeArgs a) {
  grid_dep_wait();  // the attention kernel's partials
  const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int kv_len = a.kv_lens[b];
  const int64_t orow = (static_cast<int64_t>(b) * a.num_q_heads + hq) * kHeadDim;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
  if (kv_len <= 0 || kv_len > a.max_pages * kPageSize) {  // empty, or flagged by the plan
    o[orow + d] = __float2bfloat16_rn(0.0f);
    if (a.lse && d == 0) a.lse[static_cast<int64_t>(b) * a.num_q_heads + hq] = -INFINITY;
    return;
  }
  const int split_len = a.sched[2];
  const int n_s = (kv_len + split_len - 1) / split_len;
  if (n_s <= 1) return;
  const int64_t stride = static_cast<int64_t>(a.num_q_heads);
  const float* pl = a.part_lse + static_cast<int64_t>(b) * a.max_splits * a.num_q_heads + hq;
  const float* po = a.part_o + (static_cast<int64_t>(b) * a.max_splits * a.num_q_heads + hq) * kHeadDim + d;
  float m = -INFINITY, L = 0.0f, acc = 0.0f;
  for (int s0 = 0; s0 < n_s; s0 += kCombineGroup) {
    float lv[kCombineGroup], ov[kCombineGroup];
#pragma unroll
    for (int i = 0; i < kCombineGroup; ++i) {
      const bool in = s0 + i < n_s;
      lv[i] = in ? pl[(s0 + i) * stride] : -INFINITY;
      ov[i] = in ? po[(s0 + i) * stride * kHeadDim] : 0.0f;
    }
    float mg = m;
#pragma unroll
    for (int i = 0; i < kCombineGroup; ++i) mg = fmaxf(mg, lv[i]);
    const float mu = (mg == -INFINITY) ? 0.0f : mg;
    const float r = fast_exp2(m - mu);  // 0 while nothing is merged (m = -inf)
    L *= r;
    acc *= r;
#pragma unroll
    for (int i = 0; i < kCombineGroup; ++i) {
      const float w = fast_exp2(lv[i] - mu);  // 0 past the last split
      L += w;
      acc += w * ov[i];
    }
    m = mg;
  }
  const float mu = (m == -INFINITY) ? 0.0f : m;
  o[orow + d] = __float2bfloat16_rn((L > 0.0f ? acc / L : 0.0f) * a.v_g);
  if (a.lse && d == 0)
    a.lse[static_cast<int64_t>(b) * a.num_q_heads + hq] = (L > 0.0f) ? (mu + __log2f(L)) * kLn2 : -INFINITY;
}

// Launch with programmatic stream serialization: the kernel may begin while
// the previous one in the stream finishes, and waits for it in grid_dep_wait.
cudaError_t launch_dependent(void (*kernel)(DecodeArgs), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             const DecodeArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int G, bool FP8>
cudaError_t launch_decode_g(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s) {
  DecodeArgs b = a;
  b.ctas = num_sms * kDecCtasPerSm;
  nvfp4_decode_plan_kernel<<<kPlanCtas, kPlanThreads, 0, s>>>(b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  void (*kern)(DecodeArgs) = FP8 ? fp8_paged_decode_kernel<G> : nvfp4_paged_decode_kernel<G>;
  e = set_kernel_smem(reinterpret_cast<const void*>(kern), DecFmt<FP8>::kSmem, false);
  if (e != cudaSuccess) return e;
  e = launch_dependent(kern, dim3(b.ctas), dim3(128), DecFmt<FP8>::kSmem, s, b);
  if (e != cudaSuccess) return e;
  return launch_dependent(nvfp4_decode_combine_kernel, dim3(a.num_q_heads, batch), dim3(128), 0, s, b);
}

template <bool FP8>
cudaError_t launch_decode_fmt(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_decode_g<1, FP8>(a, batch, num_sms, s);
    case 2: return launch_decode_g<2, FP8>(a, batch, num_sms, s);
    case 4: return launch_decode_g<4, FP8>(a, batch, num_sms, s);
    case 8: return launch_decode_g<8, FP8>(a, batch, num_sms, s);
    case 16: return launch_decode_g<16, FP8>(a, batch, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s) {
  return launch_decode_fmt<false>(a, batch, num_sms, s);
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s) {
  return launch_decode_fmt<true>(a, batch, num_sms, s);
}

}  // namespace nvfp4kv
