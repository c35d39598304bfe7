/*
 * kvq_oracle.h -- plain single-threaded CPU oracle for the quantized paged
 * KV-cache hot path (quantize-on-write + paged decode attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load or call this library.  It shares
 * no code, header, table or constant with the CUDA library; the only thing the
 * two have in common is the byte layout of a page, which both write out from
 * the written layout specification.
 *
 * Precision: quantization decisions are taken in fp32 with IEEE
 * round-to-nearest-even and no fused multiply-add (build with
 * -ffp-contract=off), as the pages' formulas are written for fp32 tensors;
 * attention is computed in fp64 from the stored codes and scales.
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  KVQO_FP8_PER_TENSOR = 1,
  KVQO_INT8_PER_TOKEN_HEAD = 2,
  KVQO_FP8_PER_TOKEN_HEAD = 3,
  KVQO_NVFP4 = 4,
  KVQO_INT4_PER_TOKEN_HEAD = 5,
  KVQO_NVFP4_4OVER6 = 6,
  KVQO_KVARN_K4V2_G128 = 16
};

/* ---- number formats ---- */
double kvqo_e4m3_decode(uint8_t code);
uint8_t kvqo_e4m3_encode(float v);          /* RNE, saturating to +-448 */
double kvqo_e2m1_decode(uint8_t nibble);
uint8_t kvqo_e2m1_encode(float v);          /* RNE, saturating to +-6 */
int kvqo_int8_encode(float v);              /* clamp(rint(v), -127, 127) */
int kvqo_int4_encode(float v);              /* clamp(rint(v), -7, 7) */

/* ---- scales ---- */
float kvqo_fp8_tensor_scale(float amax);    /* amax/448, 1.0 for an all-zero tensor */
float kvqo_nvfp4_tensor_scale(float amax);  /* amax/(448*6), 1.0 for an all-zero tensor */
float kvqo_amax(const float* x, size_t n);

/* ---- single-row quantizers (one token x one kv head, D values) ---- */
void kvqo_quant_row_fp8_pt(const float* x, int D, float s, uint8_t* q);
void kvqo_quant_row_int8_pth(const float* x, int D, int8_t* q, float* s);
void kvqo_quant_row_fp8_pth(const float* x, int D, uint8_t* q, float* s);
void kvqo_quant_row_nvfp4(const float* x, int D, float s_t, uint8_t* packed, uint8_t* block_scales);
void kvqo_quant_row_int4_pth(const float* x, int D, uint8_t* packed, float* s);
/* nvfp4_4over6: per block, the max/6 or the max/4 block scale, whichever
 * reconstructs the block with the smaller fp32 sum of squared errors;
 * choice_out (may be NULL) gets 6 or 4 per block. */
void kvqo_quant_row_nvfp4_4over6(const float* x, int D, float s_t, uint8_t* packed, uint8_t* block_scales,
                                 uint8_t* choice_out);
float kvqo_nvfp4_block_sse(const float* x, const uint8_t* codes, float den); /* 16 values */

/* ---- KVarN k4v2 g128 pieces ---- */
float kvqo_inv_sqrt128(void);
void kvqo_fwht128_f32(float* y);                          /* in place, normalised */
float kvqo_sum128(const float* v);                        /* fixed pairwise tree */
void kvqo_kvarn_normalize(float* Y, float* r, float* c, int steps); /* Y [128][128] */
void kvqo_kvarn_tile(const float* X, int is_value, uint8_t* codes, float* scale, float* zero,
                     float* r, float* c);                 /* X, codes [128][128] */
void kvqo_hadamard_f64(double* x, int n);                 /* normalised, in place */

/* ---- paged pool ---- */
size_t kvqo_header_bytes(void);
size_t kvqo_block_bytes(int mode, int page_size, int head_dim);
size_t kvqo_pool_bytes(int mode, int num_pages, int page_size, int num_kv_heads, int head_dim);

/* Quantize N tokens of K and V ([N][Hkv][D] fp32) into the pool at slot_mapping.
 * k_scale / v_scale are the per-tensor scales (FP8 per-tensor s, NVFP4 s_t).
 * Returns 0, or -1 on a bad argument (KVarN: tokens must form whole tiles). */
int kvqo_write(int mode, uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
               int head_dim, const float* k, const float* v, const int32_t* slot_mapping,
               int num_tokens, float k_scale, float v_scale);

/* Dequantize one stored row (token `slot`, kv head `h`, side 0=K 1=V) to fp64. */
int kvqo_dequant_row(int mode, const uint8_t* pool, int num_pages, int page_size,
                     int num_kv_heads, int head_dim, float k_scale, float v_scale,
                     int64_t slot, int h, int side, double* out);

/* Paged decode attention in fp64.  q [B][Hq][D] fp32; out [B][Hq][D] fp64.
 * rows: list of (b*Hq + hq) to compute (NULL = all).  Returns 0 or -1. */
int kvqo_decode(int mode, const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                int head_dim, float k_scale, float v_scale, const float* q,
                const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                int num_seqs, int num_q_heads, double softmax_scale, const int32_t* rows,
                int n_rows, double* out);

/* KVarN decode with an open tile: sequence b's first seq_len - seq_len % 128
 * tokens come from its quantized tiles (dequantized and rotated back to the
 * input domain, x^ = H x^'), the remaining seq_len % 128 from rows 0.. of its
 * raw tail (tail_k / tail_v [num_seqs][128][Hkv][D] fp32); fp64 attention over
 * all of them.  Returns 0 or -1. */
int kvqo_decode_kvarn_tail(const uint8_t* pool, int num_pages, int num_kv_heads, const float* q,
                           const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                           int num_seqs, int num_q_heads, double softmax_scale, const float* tail_k,
                           const float* tail_v, const int32_t* rows, int n_rows, double* out);

#ifdef __cplusplus
}
#endif
#endif
