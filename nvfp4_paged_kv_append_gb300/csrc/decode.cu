// Paged decode over the NVFP4 cache: one query token per request attends to
// every cached token ("NVFP4 KV cache prefill vs decode performance", section
// "Decode can win on fewer bytes read": decode re-reads the whole history and
// is bandwidth-bound, so fewer bytes per token is the win).
//
// Split-KV: a work item is (request, kv head, 256-token split).  A small
// schedule kernel turns kv_lens into per-request item prefixes; then one
// persistent wave of CTAs (3 per SM) walks the items.  For each item all
// threads gather its pages (K/V codes 1 KB + scales 128 B per page) with
// cp.async into one of two shared-memory stages, completing on one mbarrier,
// so the next item's bytes are in flight while the current one is computed.
// (Per-page bulk copies cost the copy engine a fixed time each, which capped
// the item rate; cp.async spreads the same bytes over the load units.)  Four warps take
// 16-token chunks of the item.  The G query heads of the kv group are the
// M rows of an m16n8k16 f16 MMA: the packed codes are dequantized (exactly,
// e2m1 x e4m3 fits f16) straight into B-fragment registers, so no dequantized
// copy of K or V is ever written.  The head dimension is permuted inside the
// MMA's K index so that each lane's fragment is 16 contiguous code bytes; the
// query carries the same permutation.  Queries are bf16; each head is
// multiplied by a power of two (exact) to sit inside f16's range and the
// factor is removed from the scores in fp32.  Partial (o, lse) per split are
// merged by a second kernel.
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

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// dequantize one code byte (two values) times an f16x2 scale
__device__ __forceinline__ uint32_t dq2(uint32_t byte, uint32_t sc) {
  uint32_t h = cvt_e2m1x2_to_f16x2(byte);
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&h), *reinterpret_cast<__half2*>(&sc));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Token (relative to a 16-token chunk) carried by MMA column n of QK n-tile
// nt, which is also row 8*nt + n of the PV K index.  Lanes reading "k index
// 2t" then touch four consecutive token rows (no shared-memory bank clash).
__device__ __forceinline__ int chunk_token(int nt, int n) { return 8 * nt + (n >> 1) + 4 * (n & 1); }

constexpr int kSplitBytesK = kDecSplit * 64;
constexpr int kSplitBytesS = kDecSplit * 8;
constexpr int kStageBytes = 2 * (kSplitBytesK + kSplitBytesS);  // 36 KB: K, K scales, V, V scales
constexpr int kDecCtasPerSm = 3;
constexpr int kDecSmem = 2 * kStageBytes + 1024;                 // two stages + alignment slack

struct DecItem {
  int b, h, split, n_tok, n_pages;
};

// Items are (request, kv head, split) in request-major order; the prefix of
// items per request (written by the schedule kernel) maps an index back.
__device__ __forceinline__ bool decode_item(const DecodeArgs& a, int idx, DecItem& it) {
  const int total = a.sched[0];
  if (idx >= total) return false;
  const int* prefix = a.sched + 4;
  int lo = 0, hi = a.batch - 1;  // last b with prefix[b] <= idx
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  const int kv_len = a.kv_lens[lo];
  const int n_s = (kv_len + kDecSplit - 1) / kDecSplit;
  const int r = idx - prefix[lo];
  it.b = lo;
  it.h = r / n_s;
  it.split = r - it.h * n_s;
  it.n_tok = min(kDecSplit, kv_len - it.split * kDecSplit);
  it.n_pages = (it.n_tok + kPageSize - 1) / kPageSize;
  return true;
}

// All 128 threads gather the item's pages into `stage` with cp.async: thread
// t serves page t / 8 (K and V codes, 16 B at a time, plus one 16-byte piece
// of each scale page); a page past the item or with an invalid id is skipped
// or zero-filled.  Each thread then arrives on `bar` once its copies land.
__device__ __forceinline__ void issue_item(const DecodeArgs& a, const DecItem& it, uint8_t* stage, uint64_t* bar,
                                           int* page_ok, int tid) {
  const int p = tid >> 3, sub = tid & 7;
  if (p < it.n_pages) {
    int pid = a.page_table[static_cast<int64_t>(it.b) * a.max_pages + it.split * 16 + p];
    if (pid < 0 || pid >= a.num_pages) {
      if (sub == 0) set_status(a.status, kDevBadPage);
      pid = -1;
    }
    if (sub == 0) page_ok[p] = pid >= 0;
    const uint32_t n16 = pid >= 0 ? 16u : 0u;
    const int64_t row = (static_cast<int64_t>(pid >= 0 ? pid : 0) * a.num_kv_heads + it.h) * kPageSize;
    const uint32_t sK = smem_u32(stage), sKs = sK + kSplitBytesK, sV = sKs + kSplitBytesS, sVs = sV + kSplitBytesK;
    const uint8_t* gk = a.k_data + row * 64;
    const uint8_t* gv = a.v_data + row * 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = sub + 8 * i;
      cp_async16(sK + p * 1024 + c * 16, gk + c * 16, n16);
      cp_async16(sV + p * 1024 + c * 16, gv + c * 16, n16);
    }
    cp_async16(sKs + p * 128 + sub * 16, a.k_scale + row * 8 + sub * 16, n16);
    cp_async16(sVs + p * 128 + sub * 16, a.v_scale + row * 8 + sub * 16, n16);
  }
  cp_async_mbar_arrive(bar);
}

// Persistent: CTA c takes items c, c + grid, ...; two shared-memory stages so
// that the copies of item k+1 run while item k is computed.
template <int G>
__global__ void __launch_bounds__(128, kDecCtasPerSm) nvfp4_paged_decode_kernel(DecodeArgs a) {
  constexpr bool kTwoRows = G > 8;  // MMA rows g+8 carry heads 8..15
  extern __shared__ __align__(128) uint8_t dsmem_raw[];
  uint8_t* dsmem = dsmem_raw + ((128u - (smem_u32(dsmem_raw) & 127u)) & 127u);
  __shared__ uint64_t bars[2];
  __shared__ int page_ok_sh[2][16];
  __shared__ float red_m[kDecWarps][16], red_l[kDecWarps][16];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  if (tid == 0) {
    mbar_init(&bars[0], 128);  // one cp.async arrival per thread
    mbar_init(&bars[1], 128);
    fence_barrier_init();
  }
  __syncthreads();
  DecItem nxt;
  for (int k = 0; k < 2; ++k)
    if (decode_item(a, blockIdx.x + k * gridDim.x, nxt)) issue_item(a, nxt, dsmem + k * kStageBytes, &bars[k], page_ok_sh[k], tid);
  DecItem it;
  for (int k = 0; decode_item(a, blockIdx.x + k * gridDim.x, it); ++k) {
    const int stg = k & 1;
    uint8_t* sK = dsmem + stg * kStageBytes;
    uint8_t* sKs = sK + kSplitBytesK;
    uint8_t* sV = sKs + kSplitBytesS;
    uint8_t* sVs = sV + kSplitBytesK;
    const int* page_ok = page_ok_sh[stg];
    const int b = it.b, h = it.h, n_tok = it.n_tok, n_pages = it.n_pages;

    // ---- query fragments (overlap the copies) ------------------------------
    // Lane (g, t) owns d = 32t .. 32t+31 of heads g and g+8.
    const uint16_t* qb =
        reinterpret_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(b) * a.num_q_heads + h * G) * kHeadDim;
    uint32_t qa[8][4];
    float crow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int head = g + 8 * r;
      float x[32];
      if ((r == 0 || kTwoRows) && head < G) {
        const uint4* src = reinterpret_cast<const uint4*>(qb + head * kHeadDim + 32 * t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 w = src[i];
          bf16x2_to_f32(w.x, x[8 * i + 0], x[8 * i + 1]);
          bf16x2_to_f32(w.y, x[8 * i + 2], x[8 * i + 3]);
          bf16x2_to_f32(w.z, x[8 * i + 4], x[8 * i + 5]);
          bf16x2_to_f32(w.w, x[8 * i + 6], x[8 * i + 7]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.0f;
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // power of two bringing the head's amax into [2^14, 2^15): exact in f16
      const int e = (amax > 0.0f) ? (14 - ilogbf(amax)) : 0;
      const float up = ldexpf(1.0f, e);
      crow[r] = a.sm_scale * a.k_g * kLog2e * ldexpf(1.0f, -e);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        qa[s][r] = pack_f16x2(x[4 * s] * up, x[4 * s + 1] * up);
        qa[s][r + 2] = pack_f16x2(x[4 * s + 2] * up, x[4 * s + 3] * up);
      }
    }

    const bool ok = mbar_wait(&bars[stg], (k >> 1) & 1, a.status);
    // zero the V scales of tokens that hold no data (past kv_len, or a page
    // that was not loaded) so that their values are exactly 0
    if (ok) {
      for (int i = tid; i < n_pages * kPageSize; i += 128) {
        if (i >= n_tok || !page_ok[i >> 4]) *reinterpret_cast<uint2*>(sVs + i * 8) = make_uint2(0u, 0u);
      }
    }
    __syncthreads();

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;

    const int n_chunks = ok ? n_pages : 0;
    for (int c = warp; c < n_chunks; c += kDecWarps) {
      const int cbase = c * 16;
      const bool page_valid = page_ok[c] != 0;
      // ---- S = q K^T for the chunk's two 8-token n-tiles
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
        const int tok = cbase + chunk_token(nt, g);
        const uint4 kc = *reinterpret_cast<const uint4*>(sK + tok * 64 + 16 * t);
        const uint32_t ks = *reinterpret_cast<const uint16_t*>(sKs + tok * 8 + 2 * t);
        const uint32_t sc0 = scale_f16x2(ks & 0xFFu), sc1 = scale_f16x2(ks >> 8);
        const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w};
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const uint32_t w = kw[st >> 1] >> (16 * (st & 1));
          const uint32_t sc = st < 4 ? sc0 : sc1;
          const uint32_t b0 = dq2(w & 0xFFu, sc), b1 = dq2((w >> 8) & 0xFFu, sc);
          mma_f16_16816(s[nt][0], s[nt][1], s[nt][2], s[nt][3], qa[st][0], qa[st][1], qa[st][2], qa[st][3], b0, b1);
        }
      }
      // ---- online softmax (log2 domain); rows g and g+8
      float p[2][4];
#pragma unroll
      for (int r = 0; r < (kTwoRows ? 2 : 1); ++r) {
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nt = i >> 1, col = 2 * t + (i & 1);
          const int tok = cbase + chunk_token(nt, col);
          x[i] = (page_valid && tok < n_tok) ? s[nt][2 * r + (i & 1)] * crow[r] : -INFINITY;
        }
        float cm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
        const float m_new = fmaxf(m_run[r], cm);
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = fast_exp2(m_run[r] - m_use);
        m_run[r] = m_new;
        float ps = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float e = fast_exp2(x[i] - m_use);
          p[i >> 1][2 * r + (i & 1)] = e;
          ps += e;
        }
        l_run[r] = l_run[r] * alpha + ps;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          acc[j][2 * r] *= alpha;
          acc[j][2 * r + 1] *= alpha;
        }
      }
      if (!kTwoRows) {
        p[0][2] = p[0][3] = p[1][2] = p[1][3] = 0.0f;
      }
      const uint32_t pa0 = pack_f16x2(p[0][0], p[0][1]), pa1 = pack_f16x2(p[0][2], p[0][3]);
      const uint32_t pa2 = pack_f16x2(p[1][0], p[1][1]), pa3 = pack_f16x2(p[1][2], p[1][3]);
      // ---- O += P V; lane's V rows: tokens t, t+4 (k 2t, 2t+1) and 8+t, 12+t
      uint32_t vx[4][4], vy[4][4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int tok = cbase + (q4 & 1) * 4 + (q4 >> 1) * 8 + t;
        const uint2 vc = *reinterpret_cast<const uint2*>(sV + tok * 64 + 8 * g);
        const uint32_t sc = scale_f16x2(sVs[tok * 8 + g]);
        dequant8_f16(vc.x, sc, vx[q4]);
        dequant8_f16(vc.y, sc, vy[q4]);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        // value index j of the lane's 16-wide d block: word j/2 (of vx|vy), half j%2
        const int w = (j >> 1) & 3;
        const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
        const uint32_t* A0 = (j < 8) ? vx[0] : vy[0];
        const uint32_t* A1 = (j < 8) ? vx[1] : vy[1];
        const uint32_t* A2 = (j < 8) ? vx[2] : vy[2];
        const uint32_t* A3 = (j < 8) ? vx[3] : vy[3];
        const uint32_t b0 = prmt(A0[w], A1[w], sel);
        const uint32_t b1 = prmt(A2[w], A3[w], sel);
        mma_f16_16816(acc[j][0], acc[j][1], acc[j][2], acc[j][3], pa0, pa1, pa2, pa3, b0, b1);
      }
    }

    // ---- merge the four warps (the stage's shared memory is free now) -------
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
    __syncthreads();
    float* red_o = reinterpret_cast<float*>(sK);  // [warp][16 heads][128]: 32 KB of the 36 KB stage
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int head = g + 8 * r;
      if (r == 1 && !kTwoRows) break;
      if (t == 0) {
        red_m[warp][head] = m_run[r];
        red_l[warp][head] = l_run[r];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        red_o[(warp * 16 + head) * kHeadDim + 16 * (2 * t) + j] = acc[j][2 * r];
        red_o[(warp * 16 + head) * kHeadDim + 16 * (2 * t + 1) + j] = acc[j][2 * r + 1];
      }
    }
    __syncthreads();
    const int kv_len = a.kv_lens[b];
    const bool single = kv_len <= kDecSplit;
    for (int i = tid; i < G * kHeadDim; i += 128) {
      const int head = i >> 7, d = i & 127;
      float m = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, red_m[w][head]);
      const float mu = (m == -INFINITY) ? 0.0f : m;
      float L = 0.0f, o = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = fast_exp2(red_m[w][head] - mu);
        L += red_l[w][head] * f;
        o += red_o[(w * 16 + head) * kHeadDim + d] * f;
      }
      const float on = (L > 0.0f) ? o / L : 0.0f;
      const float lse2 = (L > 0.0f) ? mu + __log2f(L) : -INFINITY;
      const int hq = h * G + head;
      if (single) {
        reinterpret_cast<__nv_bfloat16*>(a.o)[(static_cast<int64_t>(b) * a.num_q_heads + hq) * kHeadDim + d] =
            __float2bfloat16_rn(on * a.v_g);
        if (a.lse && d == 0) a.lse[static_cast<int64_t>(b) * a.num_q_heads + hq] = lse2 * kLn2;
      } else {
        const int64_t pi = (static_cast<int64_t>(b) * a.max_splits + it.split) * a.num_q_heads + hq;
        a.part_o[pi * kHeadDim + d] = on;
        if (d == 0) a.part_lse[pi] = lse2;
      }
    }
    __syncthreads();  // every thread is done with this stage
    if (decode_item(a, blockIdx.x + (k + 2) * gridDim.x, nxt))
      issue_item(a, nxt, dsmem + stg * kStageBytes, &bars[stg], page_ok_sh[stg], tid);
  }
}

// Schedule: items per request (splits x kv heads) and their prefix.
__global__ void __launch_bounds__(1024) nvfp4_decode_plan_kernel(DecodeArgs a) {
  __shared__ int warp_sums[32];
  int* prefix = a.sched + 4;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int carry = 0;
  for (int base = 0; base < a.batch; base += blockDim.x) {
    const int b = base + tid;
    int cnt = 0;
    if (b < a.batch) {
      const int kv_len = a.kv_lens[b];
      if (kv_len > a.max_pages * kPageSize) set_status(a.status, kDevBadShape);
      else if (kv_len > 0) cnt = ((kv_len + kDecSplit - 1) / kDecSplit) * a.num_kv_heads;
    }
    int v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[wid] = v;
    __syncthreads();
    if (wid == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = v + (wid > 0 ? warp_sums[wid - 1] : 0);
    if (b < a.batch) prefix[b] = carry + incl - cnt;
    carry += warp_sums[31];
    __syncthreads();
  }
  if (tid == 0) {
    prefix[a.batch] = carry;
    a.sched[0] = carry;
  }
}

// Merge the split partials of requests with more than one split; write zeros
// for empty requests.
__global__ void __launch_bounds__(128) nvfp4_decode_combine_kernel(DecodeArgs a) {
  const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int kv_len = a.kv_lens[b];
  const int64_t orow = (static_cast<int64_t>(b) * a.num_q_heads + hq) * kHeadDim;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
  if (kv_len <= 0) {
    o[orow + d] = __float2bfloat16_rn(0.0f);
    if (a.lse && d == 0) a.lse[static_cast<int64_t>(b) * a.num_q_heads + hq] = -INFINITY;
    return;
  }
  const int n_s = (kv_len + kDecSplit - 1) / kDecSplit;
  if (n_s <= 1) return;
  const int64_t base = static_cast<int64_t>(b) * a.max_splits * a.num_q_heads + hq;
  float m = -INFINITY;
  for (int s = 0; s < n_s; ++s) m = fmaxf(m, a.part_lse[base + static_cast<int64_t>(s) * a.num_q_heads]);
  const float mu = (m == -INFINITY) ? 0.0f : m;
  float L = 0.0f, acc = 0.0f;
  for (int s = 0; s < n_s; ++s) {
    const int64_t pi = base + static_cast<int64_t>(s) * a.num_q_heads;
    const float w = fast_exp2(a.part_lse[pi] - mu);
    L += w;
    acc += w * a.part_o[pi * kHeadDim + d];
  }
  const float on = (L > 0.0f) ? acc / L : 0.0f;
  o[orow + d] = __float2bfloat16_rn(on * a.v_g);
  if (a.lse && d == 0) a.lse[static_cast<int64_t>(b) * a.num_q_heads + hq] = (L > 0.0f) ? (mu + __log2f(L)) * kLn2 : -INFINITY;
}

template <int G>
cudaError_t launch_decode_g(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s) {
  nvfp4_decode_plan_kernel<<<1, 1024, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(nvfp4_paged_decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
  if (e != cudaSuccess) return e;
  nvfp4_paged_decode_kernel<G><<<num_sms * kDecCtasPerSm, 128, kDecSmem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  nvfp4_decode_combine_kernel<<<dim3(a.num_q_heads, batch), 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int batch, int num_sms, cudaStream_t s) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_decode_g<1>(a, batch, num_sms, s);
    case 2: return launch_decode_g<2>(a, batch, num_sms, s);
    case 4: return launch_decode_g<4>(a, batch, num_sms, s);
    case 8: return launch_decode_g<8>(a, batch, num_sms, s);
    case 16: return launch_decode_g<16>(a, batch, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4kv
