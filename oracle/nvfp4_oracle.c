/*
 * CPU oracle for the NVFP4 paged KV-cache path.  TEST INFRASTRUCTURE ONLY:
 * loaded by tests/, the smoke check and bench.py's cpu_baseline/reference
 * legs, never by the product path.  Plain loops, written for checking by eye
 * against the definitions; no blocking, fusion or reordering.
 *
 * Every function cites the passage it follows; the readings R1..R8 are
 * stated in nvfp4_oracle.h.  Compile with -ffp-contract=off: each fp32 step
 * below is one IEEE operation rounded to nearest even.
 */
#include "nvfp4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* E2M1 magnitudes indexed by the 3 low code bits: the value set of a 1-sign,
 * 2-exponent, 1-mantissa float with exponent bias 1 ([W] "NVFP4 KV cache vs
 * NVFP4 weights": 4-bit E2M1 values). */
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(unsigned code) {
  double mag = kE2M1Mag[code & 7u];
  return (code & 8u) ? -mag : mag;
}

/* OCP FP8 E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, max finite 448 ([W]: "an E4M3 scale for
 * each block of 16 values"). */
double orc_e4m3_value(unsigned byte) {
  unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  double v;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -v : v;
}

/* R1: nearest non-negative finite E4M3 value, ties to the even code.  The
 * codes 0x00..0x7E are in increasing value order, so a brute-force search over
 * them is the definition of round-to-nearest; anything above 448 lands on
 * 0x7E, which is the saturating behaviour. */
unsigned orc_e4m3_encode(float x) {
  double xd = (double)x;
  /* Saturation first: far above 448 every candidate's distance rounds to the
   * same double and the search below could not tell them apart. */
  if (xd >= 448.0) return 0x7Eu;
  unsigned best = 0;
  double best_err = fabs(xd - orc_e4m3_value(0));
  for (unsigned c = 1; c <= 0x7Eu; ++c) {
    double err = fabs(xd - orc_e4m3_value(c));
    if (err < best_err || (err == best_err && (c & 1u) == 0u && (best & 1u))) {
      best = c;
      best_err = err;
    }
  }
  return best;
}

/* R2: sign bit of q, then the nearest E2M1 magnitude with ties to the even
 * code; magnitudes above 6 land on 6 (saturation). */
unsigned orc_e2m1_encode(float q) {
  double a = fabs((double)q);
  if (a >= 6.0) return (signbit(q) ? 8u : 0u) | 7u; /* saturation, as above */
  unsigned best = 0;
  double best_err = a;
  for (unsigned c = 1; c < 8u; ++c) {
    double err = fabs(a - kE2M1Mag[c]);
    if (err < best_err || (err == best_err && (c & 1u) == 0u && (best & 1u))) {
      best = c;
      best_err = err;
    }
  }
  return (signbit(q) ? 8u : 0u) | best;
}

/* The codes of n values, one orc_e2m1_encode call each (a batch entry point
 * for the format tests' sweeps; no arithmetic of its own). */
void orc_e2m1_encode_n(const float* q, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)orc_e2m1_encode(q[i]);
}

/* One block ([PD] "NVFP4 stores 4.5 bits per value before padding": one E4M3
 * scale for each group of 16 elements; packed E2M1 pairs), steps R1..R4. */
void orc_quantize_block16(const float* x, float g, uint8_t* packed8,
                          uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float six_g = 6.0f * g;                 /* fl32(6*g) */
  float s_real = (amax == 0.0f) ? 0.0f : amax / six_g; /* fl32(amax/(6g)) */
  unsigned sc = orc_e4m3_encode(s_real);
  *scale = (uint8_t)sc;
  unsigned codes[16];
  double sdec = orc_e4m3_value(sc);
  if (sdec == 0.0) { /* R3 */
    for (int i = 0; i < 16; ++i) codes[i] = 0u;
  } else {
    float denom = g * (float)sdec;        /* fl32(g * e4m3(s)) */
    float inv = 1.0f / denom;             /* fl32(1 / denom) */
    for (int i = 0; i < 16; ++i) {
      float q = x[i] * inv;               /* fl32(x * inv) */
      codes[i] = orc_e2m1_encode(q);
    }
  }
  for (int i = 0; i < 8; ++i) /* R4 */
    packed8[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
}

void orc_quantize_rows(const float* x, int64_t rows, int D, int mode, float g,
                       uint8_t* packed, uint8_t* scales, float* row_g) {
  for (int64_t r = 0; r < rows; ++r) {
    const float* xr = x + r * (int64_t)D;
    float gr = g;
    if (mode == 1) { /* R6: dual level, one fp32 scale per row */
      float amax = 0.0f;
      for (int d = 0; d < D; ++d) {
        float a = fabsf(xr[d]);
        if (a > amax) amax = a;
      }
      gr = amax / 2688.0f; /* 2688 = 6 * 448, the largest FP4 x E4M3 product */
      if (row_g) row_g[r] = gr;
      if (gr == 0.0f) {
        memset(packed + r * (int64_t)(D / 2), 0, (size_t)(D / 2));
        memset(scales + r * (int64_t)(D / 16), 0, (size_t)(D / 16));
        continue;
      }
    }
    for (int b = 0; b < D / 16; ++b)
      orc_quantize_block16(xr + 16 * b, gr,
                           packed + r * (int64_t)(D / 2) + 8 * b,
                           scales + r * (int64_t)(D / 16) + b);
  }
}

/* R5 ([W]: the FP4 value, its block scale and the second scale). */
void orc_dequantize_rows(const uint8_t* packed, const uint8_t* scales,
                         int64_t rows, int D, const float* row_g, float g,
                         double* out) {
  for (int64_t r = 0; r < rows; ++r) {
    double gr = row_g ? (double)row_g[r] : (double)g;
    for (int d = 0; d < D; ++d) {
      uint8_t byte = packed[r * (int64_t)(D / 2) + d / 2];
      unsigned code = (d & 1) ? (byte >> 4) : (byte & 15u);
      double s = orc_e4m3_value(scales[r * (int64_t)(D / 16) + d / 16]);
      out[r * (int64_t)D + d] = orc_e2m1_value(code) * s * gr;
    }
  }
}

/* Byte offset of (slot, head) inside a pool whose per-token row is `row`
 * bytes wide (R8). */
static int64_t pool_offset(int64_t page, int64_t off, int head, int Hkv,
                           int page_size, int row) {
  return ((page * Hkv + head) * page_size + off) * (int64_t)row;
}

/* [PD] "NVFP4 stores 4.5 bits per value before padding": the cache write
 * quantizes the new K and V, creates packed FP4 data, writes the block scales
 * and maps the result into paged cache slots. */
int orc_kv_append(const float* k, const float* v, const int64_t* slot_mapping,
                  int64_t T, int Hkv, int D, int page_size, int64_t num_pages,
                  float k_g, float v_g, uint8_t* k_data, uint8_t* k_scale,
                  uint8_t* v_data, uint8_t* v_scale) {
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_pages * page_size) return -1;
    int64_t page = slot / page_size, off = slot % page_size;
    for (int h = 0; h < Hkv; ++h) {
      const float* kr = k + (t * Hkv + h) * (int64_t)D;
      const float* vr = v + (t * Hkv + h) * (int64_t)D;
      orc_quantize_rows(kr, 1, D, 0, k_g,
                        k_data + pool_offset(page, off, h, Hkv, page_size, D / 2),
                        k_scale + pool_offset(page, off, h, Hkv, page_size, D / 16),
                        NULL);
      orc_quantize_rows(vr, 1, D, 0, v_g,
                        v_data + pool_offset(page, off, h, Hkv, page_size, D / 2),
                        v_scale + pool_offset(page, off, h, Hkv, page_size, D / 16),
                        NULL);
    }
  }
  return 0;
}

int orc_gather_decode(const uint8_t* data, const uint8_t* scale,
                      const int32_t* page_row, int kv_len, int head, int Hkv,
                      int D, int page_size, int64_t num_pages, float g,
                      double* out) {
  for (int j = 0; j < kv_len; ++j) {
    int64_t page = page_row[j / page_size];
    int64_t off = j % page_size;
    if (page < 0 || page >= num_pages) return -1;
    orc_dequantize_rows(data + pool_offset(page, off, head, Hkv, page_size, D / 2),
                        scale + pool_offset(page, off, head, Hkv, page_size, D / 16),
                        1, D, NULL, g, out + (int64_t)j * D);
  }
  return 0;
}

/* Softmax attention from its definition; the causal bound is R7. */
void orc_attention_rows(const double* q, const int32_t* pos, int n_rows,
                        int q_len, const double* k, const double* v,
                        int kv_len, int D, int causal, double sm_scale,
                        double* out, double* lse) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
  for (int r = 0; r < n_rows; ++r) {
    const double* qr = q + (int64_t)r * D;
    double* o = out + (int64_t)r * D;
    int last = causal ? kv_len - q_len + pos[r] : kv_len - 1; /* last key seen */
    if (last > kv_len - 1) last = kv_len - 1;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (last < 0) { /* no visible key: output 0, lse -inf */
      if (lse) lse[r] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int j = 0; j <= last; ++j) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qr[d] * k[(int64_t)j * D + d];
      s[j] = sm_scale * dot;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j <= last; ++j) {
      double p = exp(s[j] - m);
      l += p;
      for (int d = 0; d < D; ++d) o[d] += p * v[(int64_t)j * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    if (lse) lse[r] = m + log(l);
  }
  free(s);
}

/* [PD] "A worked per-token cache estimate" and "NVFP4 stores 4.5 bits per
 * value before padding": K and V each hold D/2 packed bytes and D/16 scale
 * bytes per (token, kv head). */
int64_t orc_cache_bytes(int64_t num_pages, int page_size, int Hkv, int D) {
  return 2 * num_pages * (int64_t)page_size * Hkv * (int64_t)(D / 2 + D / 16);
}

/* ---- FP8 (E4M3) cache, the comparison format of the pages -----------------
 * "NVFP4 KV cache prefill vs decode performance", sections "NVFP4 stores 4.5
 * bits per value before padding" (an 8-bit FP8 value per element) and "A
 * worked per-token cache estimate" (FP8 bytes per token = 2 * L * H * D, one
 * byte per value before any separate scale metadata).  Readings F1..F3 are
 * stated in nvfp4_oracle.h. */

/* F2: sign of x, then the nearest E4M3 magnitude (R1's encoder, which
 * saturates at 448 and breaks ties to the even code). */
unsigned orc_fp8_encode(float x) {
  unsigned mag = orc_e4m3_encode(fabsf(x));
  return (signbit(x) ? 0x80u : 0u) | mag;
}

/* F1, F2: one per-tensor scale g; each value times the correctly rounded
 * reciprocal of g, then coded. */
void orc_fp8_quantize_rows(const float* x, int64_t n, float g, uint8_t* out) {
  float inv = 1.0f / g; /* fl32(1 / g) */
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_fp8_encode(x[i] * inv);
}

/* Cache write of the FP8 format: token t of K and V into slot
 * slot_mapping[t] (R8 layout with D bytes per token row). */
int orc_fp8_kv_append(const float* k, const float* v, const int64_t* slot_mapping,
                      int64_t T, int Hkv, int D, int page_size, int64_t num_pages,
                      float k_g, float v_g, uint8_t* k_data, uint8_t* v_data) {
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_pages * page_size) return -1;
    int64_t page = slot / page_size, off = slot % page_size;
    for (int h = 0; h < Hkv; ++h) {
      orc_fp8_quantize_rows(k + (t * Hkv + h) * (int64_t)D, D, k_g,
                            k_data + pool_offset(page, off, h, Hkv, page_size, D));
      orc_fp8_quantize_rows(v + (t * Hkv + h) * (int64_t)D, D, v_g,
                            v_data + pool_offset(page, off, h, Hkv, page_size, D));
    }
  }
  return 0;
}

/* F3: x = e4m3(byte) * g, exact in fp64. */
int orc_fp8_gather_decode(const uint8_t* data, const int32_t* page_row, int kv_len,
                          int head, int Hkv, int D, int page_size, int64_t num_pages,
                          float g, double* out) {
  for (int j = 0; j < kv_len; ++j) {
    int64_t page = page_row[j / page_size];
    int64_t off = j % page_size;
    if (page < 0 || page >= num_pages) return -1;
    const uint8_t* row = data + pool_offset(page, off, head, Hkv, page_size, D);
    for (int d = 0; d < D; ++d) out[(int64_t)j * D + d] = orc_e4m3_value(row[d]) * (double)g;
  }
  return 0;
}

/* "A worked per-token cache estimate": 2 * pages * page_size * Hkv * D. */
int64_t orc_fp8_cache_bytes(int64_t num_pages, int page_size, int Hkv, int D) {
  return 2 * num_pages * (int64_t)page_size * Hkv * (int64_t)D;
}

/* X1 ([A4Q] "Why NVFP4 KV cache A4Q prefill exists": the cache's V scales
 * follow the head dimension while PV reduces over tokens).  One block per
 * head dimension d: the page's 16 slots at d, coded by R1..R4 with g = 1. */
void orc_v_token_major_page(const float* x, int D, uint8_t* codes,
                            uint8_t* scales) {
  float block[16];
  for (int d = 0; d < D; ++d) {
    for (int t = 0; t < 16; ++t) block[t] = x[(int64_t)t * D + d];
    orc_quantize_block16(block, 1.0f, codes + 8 * (int64_t)d, scales + d);
  }
}

/* The E2M1 rounding boundaries (midpoints of neighbouring magnitudes). */
static const double kE2M1Mid[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};

/* Largest change of one coded value of a block if the decision that coded it
 * had gone the other way: per element, a code decision within relative eps
 * of an E2M1 boundary may take the neighbouring magnitude; the block scale,
 * if amax/(6g) lies within relative eps of an E4M3 midpoint, may take the
 * neighbouring byte, which re-codes the whole block (R1..R3). */
static void block_flip_bound(const float* x, float g, const uint8_t* packed,
                             unsigned sc, double eps, double* delta) {
  double sdec = orc_e4m3_value(sc);
  for (int i = 0; i < 16; ++i) delta[i] = 0.0;
  if (sdec != 0.0) {
    float inv = 1.0f / (g * (float)sdec);
    for (int i = 0; i < 16; ++i) {
      double q = fabs((double)(x[i] * inv));
      unsigned code = (packed[i / 2] >> (4 * (i % 2))) & 7u;
      for (int b = 0; b < 7; ++b) {
        if (fabs(q - kE2M1Mid[b]) <= eps * kE2M1Mid[b]) {
          unsigned alt = (code == (unsigned)b) ? (unsigned)b + 1u : (unsigned)b;
          double d = fabs(kE2M1Mag[alt] - kE2M1Mag[code]) * sdec * (double)g;
          if (d > delta[i]) delta[i] = d;
        }
      }
    }
  }
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i)
    if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
  double s_real = (double)(amax / (6.0f * g));
  for (int nb = -1; nb <= 1; nb += 2) {
    int alt = (int)sc + nb;
    if (alt < 0 || alt > 0x7E || amax == 0.0f) continue;
    double mid = 0.5 * (orc_e4m3_value(sc) + orc_e4m3_value((unsigned)alt));
    if (fabs(s_real - mid) > eps * mid) continue;
    double adec = orc_e4m3_value((unsigned)alt);
    float ainv = 1.0f / (g * (float)adec);
    for (int i = 0; i < 16; ++i) {
      unsigned code = (packed[i / 2] >> (4 * (i % 2))) & 15u;
      unsigned acode = orc_e2m1_encode(x[i] * ainv);
      double d = fabs(orc_e2m1_value(acode) * adec - orc_e2m1_value(code) * sdec) * (double)g;
      if (d > delta[i]) delta[i] = d;
    }
  }
}

/* X2..X5 ([A4Q] "Compare A4Q with dequantize-ahead repacking": A4Q keeps a
 * wide PV; this is the FP4 alternative, P coded by the cache's block codec
 * against a whole-number running reference).  With slack != NULL, also the
 * per-row, per-dimension bound on how far o moves when P decisions lying
 * within relative eps of a rounding boundary go the other way
 * (block_flip_bound), so that a result computed from scores that differ in
 * the last bits can be checked against what is unique. */
void orc_fp4pv_attention_rows(const double* q, const int32_t* pos, int n_rows,
                              int q_len, const double* k, const double* vhat,
                              int kv_len, int D, int causal, double sm_scale,
                              int tile, int tau, float g_p, double eps,
                              double* out, double* lse, double* slack) {
  const double log2e = 1.0 / log(2.0);
  int n = kv_len > 0 ? kv_len : 1;
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  double* m_of = (double*)malloc(sizeof(double) * (size_t)(n / tile + 1));
  for (int r = 0; r < n_rows; ++r) {
    const double* qr = q + (int64_t)r * D;
    double* o = out + (int64_t)r * D;
    double* sl = slack ? slack + (int64_t)r * D : NULL;
    int last = causal ? kv_len - q_len + pos[r] : kv_len - 1; /* R7 */
    if (last > kv_len - 1) last = kv_len - 1;
    for (int d = 0; d < D; ++d) {
      o[d] = 0.0;
      if (sl) sl[d] = 0.0;
    }
    if (last < 0) {
      if (lse) lse[r] = -INFINITY;
      continue;
    }
    /* X2 */
    for (int j = 0; j <= last; ++j) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qr[d] * k[(int64_t)j * D + d];
      s[j] = sm_scale * log2e * dot;
    }
    /* X3: the reference each tile is coded against */
    int n_tiles = last / tile + 1;
    double m = -INFINITY;
    for (int t = 0; t < n_tiles; ++t) {
      double mt = -INFINITY;
      for (int j = t * tile; j < (t + 1) * tile && j <= last; ++j)
        if (s[j] > mt) mt = s[j];
      if (mt > m + (double)tau) m = ceil(mt);
      m_of[t] = m;
    }
    double m_end = m;
    double l = 0.0;
    for (int j = 0; j <= last; ++j) l += exp2(s[j] - m_end);
    /* X4, X5 */
    for (int b0 = 0; b0 <= last; b0 += 16) {
      int t = b0 / tile;
      float p[16];
      uint8_t packed[8], sc;
      for (int i = 0; i < 16; ++i) {
        int j = b0 + i;
        p[i] = (j <= last) ? (float)exp2(s[j] - m_of[t]) : 0.0f;
      }
      orc_quantize_block16(p, g_p, packed, &sc);
      double wt = exp2(m_of[t] - m_end);
      double w = wt * orc_e4m3_value(sc) * (double)g_p;
      double delta[16];
      if (sl) block_flip_bound(p, g_p, packed, sc, eps, delta);
      for (int i = 0; i < 16 && b0 + i <= last; ++i) {
        unsigned code = (packed[i / 2] >> (4 * (i % 2))) & 15u; /* R4 */
        double ph = w * orc_e2m1_value(code);
        const double* vr = vhat + (int64_t)(b0 + i) * D;
        for (int d = 0; d < D; ++d) o[d] += ph * vr[d];
        if (sl && delta[i] > 0.0)
          for (int d = 0; d < D; ++d) sl[d] += wt * delta[i] * fabs(vr[d]);
      }
    }
    for (int d = 0; d < D; ++d) {
      o[d] /= l;
      if (sl) sl[d] /= l;
    }
    if (lse) lse[r] = (m_end + log2(l)) * log(2.0);
  }
  free(m_of);
  free(s);
}
