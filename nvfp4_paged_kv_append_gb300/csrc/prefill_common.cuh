// Device helpers shared by the prefill kernels (prefill.cu: one CTA per SM,
// 128-key tiles; prefill_a4q.cu: two CTAs per SM, 112-key tiles).
#pragma once
#include "kernels.cuh"

namespace nvfp4kv {

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes (its set-up overlapping that
// kernel's tail) and waits for it in grid_dep_wait before reading its results.
template <class Args>
inline cudaError_t launch_pdl(void (*kernel)(Args), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              const Args& a) {
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

namespace prefill_detail {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// log2 units: a row's running max moves (and O is rescaled) only when a tile
// exceeds it by more than this, so P stays <= 2^15, inside FP16's range.
constexpr float kRescaleThreshold = 15.0f;

// A work item: one (request, q tile, kv head) unit over KV tiles t0 ..
// t0 + n_tiles - 1 (all of the unit's tiles unless the unit is split), and the
// partial slot it writes (-1: the item covers the unit and writes the output).
struct Item {
  int b, qt, kvh;
  int q_start, q_len, kv_len;
  int tok0, n_tok;
  int t0, n_tiles, part;
};

// Items are sorted by decreasing cost; CTAs take them in snake order.
__device__ __forceinline__ bool get_item(const PrefillArgs& a, int round, Item& it) {
  const int n_items = a.work[0];
  const int grid = gridDim.x;
  const int idx = round * grid + ((round & 1) ? (grid - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x));
  if (idx >= n_items) return false;
  const int4 w = reinterpret_cast<const int4*>(a.work + 4)[idx];
  it.b = w.x;
  it.qt = w.y >> 8;
  it.kvh = w.y & 255;
  it.t0 = w.z & 0xFFFF;
  it.n_tiles = w.z >> 16;
  it.part = w.w;
  it.q_start = a.qo_indptr[it.b];
  it.q_len = a.qo_indptr[it.b + 1] - it.q_start;
  it.kv_len = a.kv_lens[it.b];
  const int tpq = kBM >> a.log2_group;
  it.tok0 = it.qt * tpq;
  it.n_tok = min(tpq, it.q_len - it.tok0);
  return true;
}

// Epilogue of a split item: row r's unnormalized O (32 columns starting at
// col), and its running max (log2 units) and sum.
__device__ __forceinline__ float* part_slot(const PrefillArgs& a, const Item& it) {
  return a.part + static_cast<int64_t>(it.part) * kPartFloats;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16-byte chunk `cc` (0..7) of row `r` in a 128B-swizzled [rows][128 B] tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t cc) { return r * 128u + (((cc ^ r) & 7u) << 4); }

// 16-byte chunk `c` (0..3) of row `r` in a 64B-swizzled [rows][64 B] tile.
__device__ __forceinline__ uint32_t sw64_off(uint32_t r, uint32_t c) { return r * 64u + (((c ^ (r >> 1)) & 3u) << 4); }

// Dequantize 32 values (16 code bytes, two 16-value blocks) of one row.
template <bool BF16>
__device__ __forceinline__ void dequant_unit(uint4 src, uint32_t sc01, uint32_t (&o0)[4], uint32_t (&o1)[4],
                                             uint32_t (&o2)[4], uint32_t (&o3)[4]) {
  if (BF16) {
    const uint32_t s0 = scale_bf16x2_x2p112(sc01 & 0xFFu), s1 = scale_bf16x2_x2p112(sc01 >> 8);
    dequant8_bf16(src.x, s0, o0);
    dequant8_bf16(src.y, s0, o1);
    dequant8_bf16(src.z, s1, o2);
    dequant8_bf16(src.w, s1, o3);
  } else {
    // both scale bytes in one conversion (byte 0 -> low half), then each
    // broadcast to a pair
    const uint32_t h = cvt_e4m3x2_to_f16x2(sc01 & 0xFFFFu);
    const uint32_t s0 = __byte_perm(h, 0u, 0x1010u), s1 = __byte_perm(h, 0u, 0x3232u);
    dequant8_f16(src.x, s0, o0);
    dequant8_f16(src.y, s0, o1);
    dequant8_f16(src.z, s1, o2);
    dequant8_f16(src.w, s1, o3);
  }
}

// Index of the repacked tile (request b, kv head h, KV tile j).
__device__ __forceinline__ int64_t repack_index(const PrefillArgs& a, int b, int h, int j) {
  const int p0 = a.tile_prefix[b], n_t = a.tile_prefix[b + 1] - p0;
  return static_cast<int64_t>(p0) * a.num_kv_heads + static_cast<int64_t>(h) * n_t + j;
}

// Quantize one 128-value bf16 row of Q A4Q-style ("NVFP4 KV cache A4Q prefill
// explained", section "Quantize Q instead of expanding K"; the section "Make
// query accuracy a release gate" leaves the scale scheme open).  With q_g = 0
// the scale is per row, dual level: g_row = amax/2688; with q_g > 0 every row
// uses q_g (one per-tensor scale, or 1 for a single-level scheme).  Then the
// cache's 16-value block codec.  Writes the 64 code bytes into row r of a
// 64B-swizzled FP4 tile and returns the eight E4M3 block scales as two words
// (k-steps 0 and 1); zeros for an invalid row.
__device__ __forceinline__ uint2 quantize_q_row(const uint4* src, bool valid, uint8_t* qtile, int r, float q_g,
                                                float& g_row) {
  float amax = 0.0f;
  if (valid && q_g == 0.0f) {
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const uint4 v = src[i];
      const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float lo, hi;
        bf16x2_to_f32(ww[k], lo, hi);
        amax = fmax3(amax, fabsf(lo), fabsf(hi));
      }
    }
  }
  g_row = q_g != 0.0f ? q_g : __fdiv_rn(amax, 2688.0f);
  uint32_t sw0 = 0u, sw1 = 0u;  // the eight scale bytes, k-step 0 and 1 (kept in registers)
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t cw[4] = {0u, 0u, 0u, 0u};
    if (valid && g_row != 0.0f) {
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint4 v0 = src[4 * c + 2 * blk], v1 = src[4 * c + 2 * blk + 1];
        float x[16];
        bf16x2_to_f32(v0.x, x[0], x[1]);
        bf16x2_to_f32(v0.y, x[2], x[3]);
        bf16x2_to_f32(v0.z, x[4], x[5]);
        bf16x2_to_f32(v0.w, x[6], x[7]);
        bf16x2_to_f32(v1.x, x[8], x[9]);
        bf16x2_to_f32(v1.y, x[10], x[11]);
        bf16x2_to_f32(v1.z, x[12], x[13]);
        bf16x2_to_f32(v1.w, x[14], x[15]);
        const uint32_t sc = quant_block16(x, g_row, cw[2 * blk], cw[2 * blk + 1]);
        const uint32_t sh = 8u * ((2 * c + blk) & 3);
        if (c < 2) sw0 |= sc << sh;
        else sw1 |= sc << sh;
      }
    }
    *reinterpret_cast<uint4*>(qtile + sw64_off(r, c)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  }
  return make_uint2(sw0, sw1);
}

}  // namespace prefill_detail
}  // namespace nvfp4kv
