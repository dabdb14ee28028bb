// Cache append: BF16 K/V -> NVFP4 codes + E4M3 block scales scattered into
// paged slots ("NVFP4 KV cache prefill vs decode performance", section "NVFP4
// stores 4.5 bits per value before padding": the cache write quantizes the new
// vectors, chooses block scales, packs FP4 data and maps it into paged slots).
//
// HBM-bound: per (token, kv head) and tensor, 256 B are read and 72 B written.
// Four threads share one 128-value row: each reads 64 contiguous bytes (four
// 16-byte streaming loads), encodes two 16-value blocks and writes one 16-byte
// vector of codes plus a 2-byte scale pair; the four threads of a row write
// the row's 64 code bytes and 8 scale bytes contiguously.
#include "kernels.cuh"

namespace nvfp4kv {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One unit = 32 values (64 B of bf16) of one (token, kv head) row of K or V:
// two 16-value blocks -> 16 code bytes + 2 scale bytes.
struct AppendUnit {
  uint4 w[4];
  int64_t slot;
};

__device__ __forceinline__ void append_load(const AppendArgs& a, int64_t u, int64_t units_per_tensor,
                                            AppendUnit& x) {
  const int tensor = u >= units_per_tensor;
  const int64_t uu = u - tensor * units_per_tensor;
  const int64_t row = uu >> 2;  // token * Hkv + head
  const int part = static_cast<int>(uu & 3);
  const uint16_t* src = reinterpret_cast<const uint16_t*>(tensor ? a.v : a.k) + row * kHeadDim + part * 32;
#pragma unroll
  for (int i = 0; i < 4; ++i) x.w[i] = ld_stream_v4(src + 8 * i);
  x.slot = a.slot_mapping[row / a.num_kv_heads];
}

__device__ __forceinline__ void append_store(const AppendArgs& a, int64_t u, int64_t units_per_tensor,
                                             const AppendUnit& x) {
  if (x.slot < 0) return;
  if (x.slot >= a.num_slots) {
    set_status(a.status, kDevBadSlot);
    return;
  }
  const int tensor = u >= units_per_tensor;
  const int64_t uu = u - tensor * units_per_tensor;
  const int64_t row = uu >> 2;
  const int part = static_cast<int>(uu & 3);
  const int h = static_cast<int>(row % a.num_kv_heads);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    bf16x2_to_f32(x.w[i].x, v[8 * i + 0], v[8 * i + 1]);
    bf16x2_to_f32(x.w[i].y, v[8 * i + 2], v[8 * i + 3]);
    bf16x2_to_f32(x.w[i].z, v[8 * i + 4], v[8 * i + 5]);
    bf16x2_to_f32(x.w[i].w, v[8 * i + 6], v[8 * i + 7]);
  }
  const float g = tensor ? a.v_scale_g : a.k_scale_g;
  uint4 codes;
  const uint32_t s0 = quant_block16(v, g, codes.x, codes.y);
  const uint32_t s1 = quant_block16(v + 16, g, codes.z, codes.w);
  const int64_t page = x.slot >> 4, off = x.slot & 15;
  const int64_t tok_row = (page * a.num_kv_heads + h) * kPageSize + off;
  uint8_t* data = tensor ? a.v_data : a.k_data;
  uint8_t* scale = tensor ? a.v_scale : a.k_scale;
  *reinterpret_cast<uint4*>(data + tok_row * (kHeadDim / 2) + part * 16) = codes;
  *reinterpret_cast<uint16_t*>(scale + tok_row * (kHeadDim / 16) + part * 2) = static_cast<uint16_t>(s0 | (s1 << 8));
}

// Grid-stride over all units of K then V, two units per thread per step so
// that 128 B of loads per thread are in flight before any is consumed.
__global__ void __launch_bounds__(256) nvfp4_kv_append_kernel(AppendArgs a) {
  const int64_t per_tensor = a.num_tokens * a.num_kv_heads * 4;
  const int64_t total = 2 * per_tensor;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; u + stride < total; u += 2 * stride) {
    AppendUnit x0, x1;
    append_load(a, u, per_tensor, x0);
    append_load(a, u + stride, per_tensor, x1);
    append_store(a, u, per_tensor, x0);
    append_store(a, u + stride, per_tensor, x1);
  }
  if (u < total) {
    AppendUnit x0;
    append_load(a, u, per_tensor, x0);
    append_store(a, u, per_tensor, x0);
  }
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
