/*
 * CPU oracle for the NVFP4 paged KV-cache path.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check in __graft_entry__.py and the cpu_baseline /
 * reference legs of bench.py may load this library.  The product path (the
 * CUDA library and its Python binding) never links, imports or calls it.  It
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Precision: every attention quantity is computed in fp64 from the decoded
 * cache values.  The codec follows the rounding steps stated below in plain
 * IEEE fp32 (compiled with -ffp-contract=off so no step is fused).
 *
 * Source pages (cited by page title and section):
 *   [W]  "NVFP4 KV cache vs NVFP4 weights", section "NVFP4 KV cache vs NVFP4
 *        weights": 4-bit E2M1 values, one E4M3 scale per 16 values, and a
 *        second (tensor) scale mapping the tensor into the FP4 x block-scale
 *        range.
 *   [PD] "NVFP4 KV cache prefill vs decode performance", section "NVFP4 stores
 *        4.5 bits per value before padding": packed E2M1 pairs, one E4M3 scale
 *        per 16 elements, 72 bits per 16 values; the same cache write
 *        quantizes, chooses block scales, packs, and maps into paged slots.
 *   [A4Q] "NVFP4 KV cache A4Q prefill explained", sections "Quantize Q instead
 *        of expanding K" and "Make query accuracy a release gate": Q is
 *        quantized to block-scaled FP4 per tile; the Q-scale scheme (single or
 *        dual level) and rounding must be recorded.
 *
 * Readings taken where the pages are silent (each one also listed in the
 * design notes):
 *   R1 block scale   s = fl32(amax16 / fl32(6*g)), stored as E4M3 with
 *                    round-to-nearest-even, saturating to 448, subnormals kept.
 *   R2 codes         q = fl32(x * fl32(1 / fl32(g * e4m3(s)))) -- the value
 *                    times the correctly rounded reciprocal of the QUANTIZED
 *                    scale, the way NVFP4 quantizers apply a block scale --
 *                    then E2M1 round-to-nearest-even with
 *                    ties to the even code, saturating to 6.  The sign bit of
 *                    q is kept, so a negative value that rounds to zero is
 *                    code 0x8 (decodes to -0, equal to 0).
 *   R3 zero scale    if e4m3(s) decodes to 0 the 16 codes are all 0x0.
 *   R4 nibble order  element 2i in the low nibble, 2i+1 in the high nibble.
 *   R5 decode        x = e2m1(code) * e4m3(scale) * g (exact in fp64).
 *   R6 Q scheme      dual level per (token, head) row of D values:
 *                    g_row = fl32(amax_row / 2688) then R1..R4 with g = g_row;
 *                    an all-zero row has g_row = 0 and all codes/scales 0.
 *   R7 causal        bottom-right aligned: query i of a request with lengths
 *                    (q_len, kv_len) sees keys j <= kv_len - q_len + i.
 *   R8 cache layout  data [page][kv_head][page_size][D/2] bytes,
 *                    scales [page][kv_head][page_size][D/16] bytes,
 *                    slot = page * page_size + offset, negative slot = skip.
 *
 * The FP8 comparison cache ("NVFP4 KV cache prefill vs decode performance",
 * sections "NVFP4 stores 4.5 bits per value before padding" and "A worked
 * per-token cache estimate": one 8-bit FP8 value per element, scale metadata
 * kept apart):
 *   F1 scale         one fp32 scale per tensor (K and V), value = e4m3 * g.
 *   F2 encode        code = sign | E4M3 magnitude nearest-even, saturating at
 *                    448, of fl32(x * fl32(1 / g)) (R1's encoder on |q|); a
 *                    negative value that rounds to zero keeps its sign (0x80).
 *   F3 layout        data [page][kv_head][page_size][D] bytes, slots as R8;
 *                    decode x = e4m3(byte) * g, exact in fp64.
 *
 * The FP4 PV experiment ("NVFP4 KV cache A4Q prefill explained", sections
 * "Why NVFP4 KV cache A4Q prefill exists" and "Compare A4Q with
 * dequantize-ahead repacking": the cache's V block scales run along the head
 * dimension, not along the token axis that PV reduces over, so the pages keep
 * PV wide).  The pages define no FP4 PV; these readings define the one built
 * here:
 *   X1 token-major V one block per (page, kv head, head dim d): the page's 16
 *                    slots of V at d, decoded by R5 without g (e2m1 * e4m3,
 *                    exact) with slots at or past the request's kv_len taken
 *                    as 0, coded by R1..R4 with g = 1 (slot 2i in the low
 *                    nibble).  Decoded value: e2m1 * e4m3 * v_g.
 *   X2 scores        s_j = sm_scale * log2(e) * <q, k_j> (log2 units), q the
 *                    A4Q query (R6 or a given scale), k_j by R5.
 *   X3 reference     keys in tiles of T (keys T*t .. T*t+T-1 of the
 *                    request); a reference m starts at -inf; a tile whose
 *                    largest visible score mt exceeds m + tau sets
 *                    m = ceil(mt); tile t is coded against the m in force
 *                    after its own update (m_t).  m is a whole number, so two
 *                    references differ by a power of two.
 *   X4 P codes       p_j = fl32(2^(s_j - m_t)) for visible keys, 0 for the
 *                    others; every 16 keys from a multiple of 16 are one
 *                    block coded by R1..R4 with g = g_p; p <= 2^tau, so
 *                    g_p = fl32(2^tau / 2688) keeps the block scale unsaturated.
 *   X5 output        o = sum_j 2^(m_t(j) - m_end) * phat_j * vhat_j / l with
 *                    l = sum_j 2^(s_j - m_end) (unquantized p),
 *                    lse = (m_end + log2 l) * ln 2; a row that sees no key
 *                    has o = 0 and lse = -inf.
 *                    The kernel takes T = 128 and tau = 4.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Format definitions ([W], [PD]). */
double orc_e2m1_value(unsigned code);   /* code in 0..15 */
double orc_e4m3_value(unsigned byte);   /* OCP E4M3FN; NaN for 0x7F/0xFF */
unsigned orc_e4m3_encode(float x);      /* x >= 0, finite: R1 rounding */
unsigned orc_e2m1_encode(float q);      /* R2 rounding, returns 4-bit code */
void orc_e2m1_encode_n(const float* q, int64_t n, uint8_t* codes); /* the same, n values */

/* One 16-value block with scale g (R1..R4): writes 8 packed bytes and one
 * scale byte. */
void orc_quantize_block16(const float* x, float g, uint8_t* packed8,
                          uint8_t* scale);

/* Quantize `rows` rows of D values (D % 16 == 0).
 * mode 0 (GLOBAL): every row uses g.  mode 1 (PER_ROW): R6, g ignored and
 * the per-row scale written to row_g[r] (row_g may be NULL in mode 0). */
void orc_quantize_rows(const float* x, int64_t rows, int D, int mode, float g,
                       uint8_t* packed, uint8_t* scales, float* row_g);

/* Decode rows (R5) with one g per row (row_g) or a single g (row_g NULL). */
void orc_dequantize_rows(const uint8_t* packed, const uint8_t* scales,
                         int64_t rows, int D, const float* row_g, float g,
                         double* out);

/* Cache write ([PD] "NVFP4 stores 4.5 bits per value before padding"):
 * quantize K and V [T][Hkv][D] with their tensor scales and write the codes
 * and scales of token t into slot slot_mapping[t] (R8).  Slots outside
 * [0, num_pages*page_size) other than negative ones return -1. */
int orc_kv_append(const float* k, const float* v, const int64_t* slot_mapping,
                  int64_t T, int Hkv, int D, int page_size, int64_t num_pages,
                  float k_g, float v_g, uint8_t* k_data, uint8_t* k_scale,
                  uint8_t* v_data, uint8_t* v_scale);

/* Decode the first kv_len tokens of kv-head `head` of one request from a pool
 * through its page-table row (R8, R5): out is [kv_len][D] fp64.
 * Returns -1 on an out-of-range page id. */
int orc_gather_decode(const uint8_t* data, const uint8_t* scale,
                      const int32_t* page_row, int kv_len, int head, int Hkv,
                      int D, int page_size, int64_t num_pages, float g,
                      double* out);

/* Scaled dot-product attention for selected query rows of one (request,
 * q-head), straight from the definition in fp64:
 *   s_j = sm_scale * <q_i, k_j> for the keys row i may see (R7 when causal),
 *   p_j = exp(s_j - max_j s_j),  o_i = sum_j p_j v_j / sum_j p_j,
 *   lse_i = max_j s_j + log(sum_j p_j)  (natural log).
 * q: [n_rows][D] (already decoded), pos[r] = index of row r within the
 * request's q_len queries, k and v: [kv_len][D].  out: [n_rows][D]. */
void orc_attention_rows(const double* q, const int32_t* pos, int n_rows,
                        int q_len, const double* k, const double* v,
                        int kv_len, int D, int causal, double sm_scale,
                        double* out, double* lse);

/* FP8 cache (F1..F3). */
unsigned orc_fp8_encode(float x);
void orc_fp8_quantize_rows(const float* x, int64_t n, float g, uint8_t* out);
int orc_fp8_kv_append(const float* k, const float* v, const int64_t* slot_mapping,
                      int64_t T, int Hkv, int D, int page_size, int64_t num_pages,
                      float k_g, float v_g, uint8_t* k_data, uint8_t* v_data);
int orc_fp8_gather_decode(const uint8_t* data, const int32_t* page_row, int kv_len,
                          int head, int Hkv, int D, int page_size, int64_t num_pages,
                          float g, double* out);
int64_t orc_fp8_cache_bytes(int64_t num_pages, int page_size, int Hkv, int D);

/* X1: the token-major blocks of one page of V.  x: [16][D] values of the
 * page's 16 slots (already decoded without g; zero rows for slots past
 * kv_len).  Writes codes [D][8] (slot 2i in the low nibble of byte i) and
 * scales [D]. */
void orc_v_token_major_page(const float* x, int D, uint8_t* codes,
                            uint8_t* scales);

/* X2..X5: attention with FP4 P and the token-major V, for selected query
 * rows of one (request, q-head).  q: [n_rows][D] decoded A4Q queries, k:
 * [kv_len][D] decoded keys, vhat: [kv_len][D] token-major V decoded by X1
 * (v_g included).  tile = T, tau as in X3, g_p as in X4.  slack (optional,
 * [n_rows][D]): how far each output element can move when the P decisions
 * (E2M1 codes, E4M3 block scales) that lie within relative eps of a rounding
 * boundary go the other way -- the part of the result that scores differing
 * in their last bits may legitimately change. */
void orc_fp4pv_attention_rows(const double* q, const int32_t* pos, int n_rows,
                              int q_len, const double* k, const double* vhat,
                              int kv_len, int D, int causal, double sm_scale,
                              int tile, int tau, float g_p, double eps,
                              double* out, double* lse, double* slack);

/* Cache bytes for one layer's K and V pools ([PD] "A worked per-token cache
 * estimate"): 2 * pages * page_size * Hkv * (D/2 + D/16). */
int64_t orc_cache_bytes(int64_t num_pages, int page_size, int Hkv, int D);

#ifdef __cplusplus
}
#endif
#endif
