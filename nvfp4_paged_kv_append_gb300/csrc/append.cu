// Cache append: BF16 K/V -> NVFP4 codes + E4M3 block scales scattered into
// paged slots ("NVFP4 KV cache prefill vs decode performance", section "NVFP4
// stores 4.5 bits per value before padding": the cache write quantizes the new
// vectors, chooses block scales, packs FP4 data and maps it into paged slots).
//
// HBM-bound: per (token, kv head) and tensor, 256 B are read and 72 B written.
// A lane owns one 16-value block (32 B of bf16, two 16-byte streaming loads)
// and writes its 8 code bytes and its scale byte; eight lanes cover a row, so
// a warp reads four consecutive rows (1 KB) per step and writes each row's 64
// code bytes and 8 scale bytes contiguously.  Rows of K come first, then rows
// of V.  One persistent wave of CTAs (as many as fit on every SM) strides
// over the rows, and each lane loads its next block before it encodes the
// current one, so the encode of one step overlaps the loads of the next.
#include "kernels.cuh"

namespace nvfp4kv {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

namespace {

// One lane's 16-value block, loaded one step ahead of its encoding.
struct AppendBlock {
  uint4 lo, hi;  // the 16 bf16 values
  int64_t slot;  // destination slot of the row's token
  int row;       // token * Hkv + head within the tensor
  int tensor;    // 0 = K, 1 = V, -1 = no block (past the end)
};

// token of a row: floor(row / Hkv) by a multiply-shift (exact for
// row < 2^31 and Hkv <= 255, which the host checks)
__device__ __forceinline__ int row_token(int row, uint64_t magic) {
  return static_cast<int>((static_cast<uint64_t>(row) * magic) >> 40);
}

__device__ __forceinline__ void append_fetch(const AppendArgs& a, int64_t step, int lane, AppendBlock& blk) {
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  const int64_t gr = step * 4 + (lane >> 3);
  blk.tensor = -1;
  if (gr >= 2 * rows) return;
  blk.tensor = gr >= rows;
  blk.row = static_cast<int>(gr - blk.tensor * rows);
  const uint16_t* src =
      reinterpret_cast<const uint16_t*>(blk.tensor ? a.v : a.k) + static_cast<int64_t>(blk.row) * kHeadDim + (lane & 7) * 16;
  blk.lo = ld_stream_v4(src);
  blk.hi = ld_stream_v4(src + 8);
  blk.slot = a.slot_mapping[row_token(blk.row, a.row_magic)];
}

__device__ __forceinline__ void append_encode(const AppendArgs& a, const AppendBlock& blk, int lane) {
  if (blk.tensor < 0 || blk.slot < 0) return;  // past the end, or a padding token
  if (blk.slot >= a.num_slots) {
    set_status(a.status, kDevBadSlot);
    return;
  }
  float x[16];
  bf16x2_to_f32(blk.lo.x, x[0], x[1]);
  bf16x2_to_f32(blk.lo.y, x[2], x[3]);
  bf16x2_to_f32(blk.lo.z, x[4], x[5]);
  bf16x2_to_f32(blk.lo.w, x[6], x[7]);
  bf16x2_to_f32(blk.hi.x, x[8], x[9]);
  bf16x2_to_f32(blk.hi.y, x[10], x[11]);
  bf16x2_to_f32(blk.hi.z, x[12], x[13]);
  bf16x2_to_f32(blk.hi.w, x[14], x[15]);
  uint32_t c0, c1;
  const uint32_t sc = quant_block16(x, blk.tensor ? a.v_scale_g : a.k_scale_g, c0, c1);
  const int h = blk.row - row_token(blk.row, a.row_magic) * a.num_kv_heads;
  const int64_t tok_row = ((blk.slot >> 4) * a.num_kv_heads + h) * kPageSize + (blk.slot & 15);
  const int b = lane & 7;
  *reinterpret_cast<uint2*>((blk.tensor ? a.v_data : a.k_data) + tok_row * (kHeadDim / 2) + b * 8) = make_uint2(c0, c1);
  (blk.tensor ? a.v_scale : a.k_scale)[tok_row * (kHeadDim / 16) + b] = static_cast<uint8_t>(sc);
}

}  // namespace

// A warp's step covers four rows (of K, then of V); warps stride over the
// steps with one block per lane in flight ahead of the one being encoded.
__global__ void __launch_bounds__(256) nvfp4_kv_append_kernel(AppendArgs a) {
  const int64_t steps = (2 * a.num_tokens * a.num_kv_heads + 3) / 4;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  AppendBlock cur, next;
  cur.tensor = -1;
  if (w0 < steps) append_fetch(a, w0, lane, cur);
  for (int64_t st = w0; st < steps; st += nw) {
    next.tensor = -1;
    if (st + nw < steps) append_fetch(a, st + nw, lane, next);
    append_encode(a, cur, lane);
    cur = next;
  }
}

// FP8 cache write (the comparison format: one E4M3 code per value and one
// fp32 scale per tensor, "NVFP4 KV cache prefill vs decode performance",
// section "A worked per-token cache estimate").  code = E4M3(x * (1/g)),
// nearest even and saturating at 448 (hardware cvt), with 1/g the correctly
// rounded reciprocal.  Same lane layout as the NVFP4 append: a lane encodes
// 16 values of a row and writes 16 code bytes.
__global__ void __launch_bounds__(256) fp8_kv_append_kernel(AppendArgs a) {
  const int64_t steps = (2 * a.num_tokens * a.num_kv_heads + 3) / 4;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float inv_k = __frcp_rn(a.k_scale_g), inv_v = __frcp_rn(a.v_scale_g);
  AppendBlock cur, next;
  cur.tensor = -1;
  if (w0 < steps) append_fetch(a, w0, lane, cur);
  for (int64_t st = w0; st < steps; st += nw) {
    next.tensor = -1;
    if (st + nw < steps) append_fetch(a, st + nw, lane, next);
    if (cur.tensor >= 0 && cur.slot >= 0) {
      if (cur.slot >= a.num_slots) {
        set_status(a.status, kDevBadSlot);
      } else {
        const float inv = cur.tensor ? inv_v : inv_k;
        const uint32_t w[8] = {cur.lo.x, cur.lo.y, cur.lo.z, cur.lo.w, cur.hi.x, cur.hi.y, cur.hi.z, cur.hi.w};
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float x0, x1, x2, x3;
          bf16x2_to_f32(w[2 * i], x0, x1);
          bf16x2_to_f32(w[2 * i + 1], x2, x3);
          pk[i] = cvt_e4m3x2(__fmul_rn(x0, inv), __fmul_rn(x1, inv)) |
                  (cvt_e4m3x2(__fmul_rn(x2, inv), __fmul_rn(x3, inv)) << 16);
        }
        const int h = cur.row - row_token(cur.row, a.row_magic) * a.num_kv_heads;
        const int64_t tok_row = ((cur.slot >> 4) * a.num_kv_heads + h) * kPageSize + (cur.slot & 15);
        *reinterpret_cast<uint4*>((cur.tensor ? a.v_data : a.k_data) + tok_row * kHeadDim + (lane & 7) * 16) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    cur = next;
  }
}

int append_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4_kv_append_kernel, 256, 0) != cudaSuccess || n < 1)
    return 1;
  return n;
}

// Standalone quantizer (same codec; GLOBAL or PER_ROW scale).  One warp per
// row: lane i owns values 4i..4i+3; the row amax (PER_ROW) is a warp max.
__global__ void __launch_bounds__(256) nvfp4_quantize_rows_kernel(QuantArgs a) {
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const uint16_t* src = reinterpret_cast<const uint16_t*>(a.x) + row * kHeadDim;
  // gather the 16-value block of this lane's group: lanes 4b..4b+3 share block b
  float x[16];
  const uint4 w0 = *reinterpret_cast<const uint4*>(src + (lane >> 2) * 16);
  const uint4 w1 = *reinterpret_cast<const uint4*>(src + (lane >> 2) * 16 + 8);
  bf16x2_to_f32(w0.x, x[0], x[1]);
  bf16x2_to_f32(w0.y, x[2], x[3]);
  bf16x2_to_f32(w0.z, x[4], x[5]);
  bf16x2_to_f32(w0.w, x[6], x[7]);
  bf16x2_to_f32(w1.x, x[8], x[9]);
  bf16x2_to_f32(w1.y, x[10], x[11]);
  bf16x2_to_f32(w1.z, x[12], x[13]);
  bf16x2_to_f32(w1.w, x[14], x[15]);
  float g = a.global_scale;
  if (a.mode == 1) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    g = __fdiv_rn(amax, 2688.0f);
    if (lane == 0) a.row_scales[row] = g;
  }
  uint32_t c0 = 0, c1 = 0, sc = 0;
  if (g != 0.0f) sc = quant_block16(x, g, c0, c1);
  if ((lane & 3) == 0) {
    uint8_t* p = a.packed + row * (kHeadDim / 2) + (lane >> 2) * 8;
    *reinterpret_cast<uint2*>(p) = make_uint2(c0, c1);
    a.scales[row * (kHeadDim / 16) + (lane >> 2)] = static_cast<uint8_t>(sc);
  }
}

// Inverse quantizer: bf16 out = code * scale * (row scale or global scale).
__global__ void __launch_bounds__(256) nvfp4_dequantize_rows_kernel(DequantArgs a) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid >> 4;  // 16 threads per row, 8 values each
  const int part = static_cast<int>(gid & 15);
  if (row >= a.rows) return;
  const uint32_t codes = *reinterpret_cast<const uint32_t*>(a.packed + row * (kHeadDim / 2) + part * 4);
  const float s = e4m3_to_f32(a.scales[row * (kHeadDim / 16) + (part >> 1)]);
  const float g = a.row_scales ? a.row_scales[row] : a.global_scale;
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h = cvt_e2m1x2_to_f16x2((codes >> (8 * i)) & 0xFFu);
    float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    __nv_bfloat162 r = __floats2bfloat162_rn(f.x * s * g, f.y * s * g);
    out[i] = *reinterpret_cast<uint32_t*>(&r);
  }
  *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + row * kHeadDim + part * 8) =
      make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace nvfp4kv
