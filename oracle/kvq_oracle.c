/*
 * kvq_oracle.c -- plain single-threaded CPU oracle for the quantized paged
 * KV-cache hot path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg are its only users.
 *
 * Every function is written out from the definition it cites, with no
 * blocking, fusion or reordering beyond what that definition states.  Sources
 * (web pages, cited by title and section):
 *
 *  [P1] "KV Cache 量化深度解析：Per-Tensor、Per-Token-Head 与 NVFP4"
 *       sec. 2.1 (FP8 per-tensor), sec. 2.2 (per-token-head scale loop),
 *       sec. 2.3 (NVFP4 block scale along head_dim).
 *  [P2] "KVarN：华为推出的原生 vLLM KV-cache 量化后端，打破性能与精度的权衡"
 *       section 技术原理 (four stages: tile, Hadamard rotation, iterative
 *       variance normalisation, asymmetric round-to-nearest), section
 *       配置与部署 (preset kvarn_k4v2_g128), section 注意事项 (tile = 128).
 *  [P3] "KV Cache 量化 · LLM Glossary", first section (s = max|x|/127,
 *       q = clip(round(x/s), -127, 127), x^ = s q), fake-quant listing
 *       (scale clamped at 1e-8 before the divide; torch.round = half-even).
 *  [P4] "KV 量化" (rustineverything.app), sections on FP8 per-tensor
 *       write/read (divide by scale before the cast, multiply on read) and on
 *       scales stored in the page next to the data.
 *  [P5] "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化", sections
 *       "NVFP4 中的 4 bit 表示什么" (E2M1 values), "双层缩放怎样恢复动态范围"
 *       (q_i = Q_E2M1(x_i/(s_t s_b)), x^_i = s_t s_b q_i),
 *       "用一组数直观看缩放的作用" (block max maps to about 6),
 *       "K 与 V 的量化误差进入 attention 的位置不同" (A = softmax(QK^T/sqrt(d)), O = AV).
 *
 * Readings where the pages are silent are listed in the project's design
 * notes; each is restated at the function that applies it.
 */
#include "kvq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* E4M3 ("fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no      */
/* infinities, S.1111.111 is NaN, largest finite 448, smallest subnormal 2^-9. */
/* ------------------------------------------------------------------------- */
double kvqo_e4m3_decode(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);          /* subnormal: 0.mmm x 2^(1-7) */
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 1.mmm x 2^(e-7) */
  return s ? -mag : mag;
}

/* Round |v| to the nearest of the 127 finite non-negative E4M3 values; an
 * exact tie goes to the code with an even mantissa (round-to-nearest-even);
 * magnitudes at or above 448 saturate to 448.  The sign of v is kept, so a
 * negative value that rounds to zero encodes as 0x80. */
uint8_t kvqo_e4m3_encode(float v) {
  uint8_t sign, mag;
  double a, dl, dh;
  int lo, hi;
  if (isnan(v)) return 0x7F;
  sign = signbit(v) ? 0x80 : 0x00;
  a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  lo = 0;
  hi = 0x7E; /* invariant: decode(lo) <= a < decode(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (kvqo_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  dl = a - kvqo_e4m3_decode((uint8_t)lo);
  dh = kvqo_e4m3_decode((uint8_t)hi) - a;
  if (dl < dh) mag = (uint8_t)lo;
  else if (dh < dl) mag = (uint8_t)hi;
  else mag = (uint8_t)((lo & 1) ? hi : lo);
  return (uint8_t)(sign | mag);
}

/* E2M1 [P5 "NVFP4 中的 4 bit 表示什么"]: 1 sign, 2 exponent (bias 1), 1 mantissa
 * bit; non-negative values 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double kvqo_e2m1_decode(uint8_t nibble) {
  int s = (nibble >> 3) & 1;
  int e = (nibble >> 1) & 3;
  int m = nibble & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* Q_E2M1 [P5 "双层缩放"]: "round to the nearest E2M1 value and handle inputs out
 * of range" -- read as round-to-nearest-even with saturation to +-6. */
uint8_t kvqo_e2m1_encode(float v) {
  uint8_t sign, mag;
  double a, dl, dh;
  int lo, hi;
  if (isnan(v)) return 0x7; /* E2M1 has no NaN; never produced for finite inputs */
  sign = signbit(v) ? 0x8 : 0x0;
  a = fabs((double)v);
  if (a >= 6.0) return (uint8_t)(sign | 0x7);
  lo = 0;
  hi = 7; /* invariant: decode(lo) <= a < decode(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (kvqo_e2m1_decode((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  dl = a - kvqo_e2m1_decode((uint8_t)lo);
  dh = kvqo_e2m1_decode((uint8_t)hi) - a;
  if (dl < dh) mag = (uint8_t)lo;
  else if (dh < dl) mag = (uint8_t)hi;
  else mag = (uint8_t)((lo & 1) ? hi : lo);
  return (uint8_t)(sign | mag);
}

/* [P3 first section]: q = clip(round(v), -127, 127); round is half-to-even as
 * torch.round in the fake-quant listing (C rintf in the default mode). */
int kvqo_int8_encode(float v) {
  float r = rintf(v);
  if (r > 127.0f) r = 127.0f;
  if (r < -127.0f) r = -127.0f;
  return (int)r;
}

/* INT4 code [P4 "scale 和数据放在一起" names int4_per_token_head and its
 * head_size/2 bytes per head, nothing more]: read as the 4-bit analogue of
 * the int8 rule, q = clip(round(v), -7, 7), round half-to-even; the code is
 * stored as a 4-bit two's-complement nibble. */
int kvqo_int4_encode(float v) {
  float r = rintf(v);
  if (r > 7.0f) r = 7.0f;
  if (r < -7.0f) r = -7.0f;
  return (int)r;
}

/* ------------------------------------------------------------------------- */
/* Scales                                                                     */
/* ------------------------------------------------------------------------- */
float kvqo_amax(const float* x, size_t n) {
  float a = 0.0f;
  size_t i;
  for (i = 0; i < n; i++) a = fmaxf(a, fabsf(x[i]));
  return a;
}

/* Per-tensor FP8 scale [P1 sec. 2.1: K_fp8 = K/scale]: the scale is taken as
 * global amax/448 so the largest magnitude maps to the E4M3 maximum; an
 * all-zero tensor keeps the default scale 1.0 ([P4]: missing scales are 1.0). */
float kvqo_fp8_tensor_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

/* NVFP4 global scale s_t [P5 "双层缩放"]: amax/(448*6), so that block scales
 * amax_b/(6 s_t) stay inside the E4M3 range while each block max maps to ~6. */
float kvqo_nvfp4_tensor_scale(float amax) { return amax > 0.0f ? amax / 2688.0f : 1.0f; }

/* ------------------------------------------------------------------------- */
/* Row quantizers                                                             */
/* ------------------------------------------------------------------------- */
/* [P1 sec. 2.1], [P4 写和读]: divide by the per-tensor scale, cast to E4M3. */
void kvqo_quant_row_fp8_pt(const float* x, int D, float s, uint8_t* q) {
  int d;
  for (d = 0; d < D; d++) q[d] = kvqo_e4m3_encode(x[d] / s);
}

/* [P1 sec. 2.2] scale[i][j] = max|K[i,j,:]| / MAX; K_quant = round(k / scale),
 * with [P3]'s clamp of the max at 1e-8 before the divide and MAX = 127. */
void kvqo_quant_row_int8_pth(const float* x, int D, int8_t* q, float* s_out) {
  float amax = 0.0f, s;
  int d;
  for (d = 0; d < D; d++) amax = fmaxf(amax, fabsf(x[d]));
  s = fmaxf(amax, 1e-8f) / 127.0f;
  for (d = 0; d < D; d++) q[d] = (int8_t)kvqo_int8_encode(x[d] / s);
  *s_out = s;
}

/* [P1 sec. 2.2] with FP8_MAX = 448 and the E4M3 cast in place of round(). */
void kvqo_quant_row_fp8_pth(const float* x, int D, uint8_t* q, float* s_out) {
  float amax = 0.0f, s;
  int d;
  for (d = 0; d < D; d++) amax = fmaxf(amax, fabsf(x[d]));
  s = fmaxf(amax, 1e-8f) / 448.0f;
  for (d = 0; d < D; d++) q[d] = kvqo_e4m3_encode(x[d] / s);
  *s_out = s;
}

/* NVFP4 [P5 "双层缩放", "用一组数直观看缩放的作用"], [P1 sec. 2.3]: blocks of 16
 * consecutive head_dim values; s_b = E4M3(amax_b / (6 s_t)) so the block max
 * maps to ~6; q_i = Q_E2M1(x_i / (s_t s_b)) with the product s_t s_b rounded
 * to fp32 first.  A block whose scale rounds to zero stores all-zero codes.
 * Two codes per byte, the even head_dim index in the low nibble. */
void kvqo_quant_row_nvfp4(const float* x, int D, float s_t, uint8_t* packed, uint8_t* bs) {
  float six_st = 6.0f * s_t;
  int b, i;
  for (b = 0; b < D / 16; b++) {
    float amax = 0.0f, sbf, den;
    uint8_t sb, codes[16];
    for (i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(x[16 * b + i]));
    sb = kvqo_e4m3_encode(amax / six_st);
    bs[b] = sb;
    sbf = (float)kvqo_e4m3_decode(sb);
    den = s_t * sbf;
    for (i = 0; i < 16; i++) codes[i] = (sbf == 0.0f) ? 0 : kvqo_e2m1_encode(x[16 * b + i] / den);
    for (i = 0; i < 8; i++) packed[8 * b + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
  }
}

/* Squared reconstruction error of one 16-value NVFP4 block, fp32: x^_i =
 * E2M1value(code_i) * den, e_i = (x_i - x^_i)^2, summed as a pairwise tree of
 * neighbours ((e0 + e1) + (e2 + e3)) + ... , each operation rounded once. */
float kvqo_nvfp4_block_sse(const float* x, const uint8_t* codes, float den) {
  float e[16];
  int i, w;
  for (i = 0; i < 16; i++) {
    float xh = (float)kvqo_e2m1_decode(codes[i]) * den;
    float d = x[i] - xh;
    e[i] = d * d;
  }
  for (w = 1; w < 16; w <<= 1)
    for (i = 0; i < 16; i += 2 * w) e[i] = e[i] + e[i + w];
  return e[0];
}

/* nvfp4_4over6 [P5 "用一组数直观看缩放的作用", last paragraph: a max-based scale
 * is not always the one with the smallest reconstruction error; the mode picks,
 * per block, between scales of the max/6 and the max/4 kind by reconstruction
 * error].  Both candidates are plain NVFP4 blocks under the same s_t:
 *   max/6: s_b = E4M3(amax_b / (6 s_t))  (block max lands near code 6)
 *   max/4: s_b = E4M3(amax_b / (4 s_t))  (block max lands near code 4)
 * each coded as in kvqo_quant_row_nvfp4; the block keeps the candidate with the
 * smaller kvqo_nvfp4_block_sse, max/6 on a tie.  Storage and reconstruction are
 * NVFP4's. */
void kvqo_quant_row_nvfp4_4over6(const float* x, int D, float s_t, uint8_t* packed, uint8_t* bs,
                                 uint8_t* choice_out) {
  float six_st = 6.0f * s_t, four_st = 4.0f * s_t;
  int b, i, c;
  for (b = 0; b < D / 16; b++) {
    const float* xb = x + 16 * b;
    float amax = 0.0f, err[2];
    uint8_t sb[2], codes[2][16];
    for (i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(xb[i]));
    for (c = 0; c < 2; c++) {
      float sbf, den;
      sb[c] = kvqo_e4m3_encode(amax / (c == 0 ? six_st : four_st));
      sbf = (float)kvqo_e4m3_decode(sb[c]);
      den = s_t * sbf;
      for (i = 0; i < 16; i++) codes[c][i] = (sbf == 0.0f) ? 0 : kvqo_e2m1_encode(xb[i] / den);
      err[c] = kvqo_nvfp4_block_sse(xb, codes[c], den);
    }
    c = err[1] < err[0] ? 1 : 0;
    bs[b] = sb[c];
    if (choice_out) choice_out[b] = (uint8_t)(c ? 4 : 6);
    for (i = 0; i < 8; i++) packed[8 * b + i] = (uint8_t)(codes[c][2 * i] | (codes[c][2 * i + 1] << 4));
  }
}

/* int4_per_token_head [P4 "scale 和数据放在一起": per token and kv head a
 * dynamic fp32 scale stored in the page after head_size/2 bytes of data]:
 * the per-token-head rule of [P1 sec. 2.2] with MAX = 7 (the largest
 * magnitude of the symmetric 4-bit range, as 127 is for int8) and [P3]'s
 * clamp of the max at 1e-8: s = max(max|x|, 1e-8) / 7, q = clip(rint(x/s),
 * -7, 7).  Two codes per byte, the even head_dim index in the low nibble. */
void kvqo_quant_row_int4_pth(const float* x, int D, uint8_t* packed, float* s_out) {
  float amax = 0.0f, s;
  int d;
  for (d = 0; d < D; d++) amax = fmaxf(amax, fabsf(x[d]));
  s = fmaxf(amax, 1e-8f) / 7.0f;
  for (d = 0; d < D; d += 2) {
    int lo = kvqo_int4_encode(x[d] / s) & 15, hi = kvqo_int4_encode(x[d + 1] / s) & 15;
    packed[d / 2] = (uint8_t)(lo | (hi << 4));
  }
  *s_out = s;
}

/* ------------------------------------------------------------------------- */
/* KVarN k4v2 g128 [P2 技术原理]                                                */
/* ------------------------------------------------------------------------- */
float kvqo_inv_sqrt128(void) { return (float)(1.0 / sqrt(128.0)); }

/* Stage 2, Hadamard rotation along channels: the Sylvester-ordered fast
 * Walsh-Hadamard transform, butterflies (a, b) -> (a+b, a-b) on pairs
 * (j, j+h) for h = 1, 2, ..., 64 in that order, then the 1/sqrt(128)
 * normalisation that makes it orthogonal. fp32, each operation rounded. */
void kvqo_fwht128_f32(float* y) {
  int h, i, j;
  float c = kvqo_inv_sqrt128();
  for (h = 1; h < 128; h <<= 1)
    for (i = 0; i < 128; i += 2 * h)
      for (j = i; j < i + h; j++) {
        float a = y[j], b = y[j + h];
        y[j] = a + b;
        y[j + h] = a - b;
      }
  for (j = 0; j < 128; j++) y[j] = y[j] * c;
}

/* The fixed summation order of the normalisation statistics: a pairwise tree
 * v[i] += v[i+off] for off = 64, 32, ..., 1. */
float kvqo_sum128(const float* v) {
  float t[128];
  int off, i;
  memcpy(t, v, sizeof t);
  for (off = 64; off >= 1; off >>= 1)
    for (i = 0; i < off; i++) t[i] = t[i] + t[i + off];
  return t[0];
}

/* Population standard deviation of 128 values. */
static float std128(const float* v) {
  float d2[128], mean, var;
  int i;
  mean = kvqo_sum128(v) / 128.0f;
  for (i = 0; i < 128; i++) {
    float d = v[i] - mean;
    d2[i] = d * d;
  }
  var = kvqo_sum128(d2) / 128.0f;
  return sqrtf(var);
}

/* Stage 3, iterative variance normalisation: alternating standard-deviation
 * normalisation of tokens (columns of the channels x tokens tile) and of
 * channels (rows), tokens first.  Each step divides every token (or channel)
 * by its own std via y * (1/std) and multiplies that std into the token
 * factor r_t (or channel factor c_d); accumulating the factors by product is
 * the same as summing their logarithms ("in log space").  A std below 1e-8
 * leaves that token or channel unchanged.  Y is [token][channel]. */
void kvqo_kvarn_normalize(float* Y, float* r, float* c, int steps) {
  float vec[128], sd[128];
  int k, i, j;
  for (i = 0; i < 128; i++) { r[i] = 1.0f; c[i] = 1.0f; }
  for (k = 0; k < steps; k++) {
    int per_token = (k % 2) == 0;
    for (i = 0; i < 128; i++) {
      for (j = 0; j < 128; j++) vec[j] = per_token ? Y[i * 128 + j] : Y[j * 128 + i];
      sd[i] = std128(vec);
    }
    for (i = 0; i < 128; i++) {
      float inv;
      if (sd[i] < 1e-8f) continue;
      inv = 1.0f / sd[i];
      for (j = 0; j < 128; j++) {
        float* y = per_token ? &Y[i * 128 + j] : &Y[j * 128 + i];
        *y = *y * inv;
      }
      if (per_token) r[i] = r[i] * sd[i]; else c[i] = c[i] * sd[i];
    }
  }
}

/* Stages 1-4 for one 128-token x 128-channel tile of one kv head.
 * Stage 4, asymmetric round-to-nearest: keys get a scale and zero per
 * channel over the tile's tokens (4 bits, 15 steps), values per token over
 * the channels (2 bits, 3 steps); zero is the minimum, scale = (max-min)/steps,
 * code = clamp(rint((y - min)/scale), 0, steps); a zero scale stores code 0.
 * Reconstruction: x^_td = r_t * c_d * (scale * code + zero), in the rotated
 * domain. */
void kvqo_kvarn_tile(const float* X, int is_value, uint8_t* codes, float* scale, float* zero,
                     float* r, float* c) {
  float* Y = (float*)malloc(sizeof(float) * 128 * 128);
  int t, d;
  memcpy(Y, X, sizeof(float) * 128 * 128);
  for (t = 0; t < 128; t++) kvqo_fwht128_f32(Y + 128 * t);
  kvqo_kvarn_normalize(Y, r, c, 8);
  if (!is_value) {
    for (d = 0; d < 128; d++) {
      float mn = Y[d], mx = Y[d], s;
      for (t = 1; t < 128; t++) { mn = fminf(mn, Y[t * 128 + d]); mx = fmaxf(mx, Y[t * 128 + d]); }
      s = (mx - mn) / 15.0f;
      scale[d] = s;
      zero[d] = mn;
      for (t = 0; t < 128; t++) {
        float qv;
        if (s == 0.0f) { codes[t * 128 + d] = 0; continue; }
        qv = rintf((Y[t * 128 + d] - mn) / s);
        if (qv < 0.0f) qv = 0.0f;
        if (qv > 15.0f) qv = 15.0f;
        codes[t * 128 + d] = (uint8_t)qv;
      }
    }
  } else {
    for (t = 0; t < 128; t++) {
      float mn = Y[t * 128], mx = Y[t * 128], s;
      for (d = 1; d < 128; d++) { mn = fminf(mn, Y[t * 128 + d]); mx = fmaxf(mx, Y[t * 128 + d]); }
      s = (mx - mn) / 3.0f;
      scale[t] = s;
      zero[t] = mn;
      for (d = 0; d < 128; d++) {
        float qv;
        if (s == 0.0f) { codes[t * 128 + d] = 0; continue; }
        qv = rintf((Y[t * 128 + d] - mn) / s);
        if (qv < 0.0f) qv = 0.0f;
        if (qv > 3.0f) qv = 3.0f;
        codes[t * 128 + d] = (uint8_t)qv;
      }
    }
  }
  free(Y);
}

/* Normalised Sylvester Hadamard transform in fp64 (H is symmetric and
 * orthonormal, so it is its own inverse). */
void kvqo_hadamard_f64(double* x, int n) {
  int h, i, j;
  double c = 1.0 / sqrt((double)n);
  for (h = 1; h < n; h <<= 1)
    for (i = 0; i < n; i += 2 * h)
      for (j = i; j < i + h; j++) {
        double a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
  for (j = 0; j < n; j++) x[j] *= c;
}

/* ------------------------------------------------------------------------- */
/* Paged pool layout (the written layout specification of the library):       */
/*   pool = 256-byte header, then one block per (page, kv head), page-major.    */
/*   FP8 per-tensor : K[P][D] e4m3 | V[P][D] e4m3                               */
/*   INT8/FP8 PTH   : K[P][D] | V[P][D] | K scale[P] f32 | V scale[P] f32       */
/*   NVFP4, 4over6  : K[P][D/2] | V[P/2][D] | K s_b[P][D/16] | V s_b[P][D/16]   */
/*   INT4 PTH       : K[P][D/2] | V[P/2][D] | K scale[P] f32 | V scale[P] f32   */
/*     with its own nibble order inside each 32-bit word (see int4_k_nibble,    */
/*     int4_v_nibble)                                                            */
/*   KVarN (P=D=128): K[128][64] 4-bit | V[128][32] 2-bit |                      */
/*                    K scale[D] zero[D] c[D] r[P] | V scale[P] zero[P] r[P] c[D] */
/* 4-bit: even index in the low nibble (4-bit V of NVFP4 and INT4: byte [k][d] */
/* holds channel d of tokens 2k (low nibble) and 2k+1); 2-bit: element 4i+j in */
/* bits 2j..2j+1.                                                              */
/* ------------------------------------------------------------------------- */
size_t kvqo_header_bytes(void) { return 256; }

size_t kvqo_block_bytes(int mode, int P, int D) {
  switch (mode) {
    case KVQO_FP8_PER_TENSOR: return (size_t)2 * P * D;
    case KVQO_INT8_PER_TOKEN_HEAD:
    case KVQO_FP8_PER_TOKEN_HEAD: return (size_t)2 * P * D + (size_t)8 * P;
    case KVQO_NVFP4:
    case KVQO_NVFP4_4OVER6: return (size_t)P * D + (size_t)P * D / 8;
    case KVQO_INT4_PER_TOKEN_HEAD: return (size_t)P * D + (size_t)8 * P;
    case KVQO_KVARN_K4V2_G128:
      return (size_t)P * D / 2 + (size_t)P * D / 4 + (size_t)4 * (3 * D + P) + (size_t)4 * (3 * P + D);
    default: return 0;
  }
}

size_t kvqo_pool_bytes(int mode, int num_pages, int P, int Hkv, int D) {
  return kvqo_header_bytes() + (size_t)num_pages * Hkv * kvqo_block_bytes(mode, P, D);
}

static uint8_t* block_at(uint8_t* pool, int mode, int P, int Hkv, int D, int64_t page, int h) {
  return pool + kvqo_header_bytes() + ((size_t)page * Hkv + h) * kvqo_block_bytes(mode, P, D);
}

static void put_f32(uint8_t* p, float v) { memcpy(p, &v, 4); }
static float get_f32(const uint8_t* p) { float v; memcpy(&v, p, 4); return v; }

/* INT4 storage order.  Inside each 4-byte word of a K row (8 channels 8m ..
 * 8m+7) nibble k (bits 4k .. 4k+3) holds channel 8m + 2k for k < 4 and
 * 8m + 2(k-4) + 1 for k >= 4: even channels in the low half-word, odd ones in
 * the high half-word.  Inside each 4-byte word of a V token-pair row (channels
 * 4m .. 4m+3 of tokens 2j, 2j+1) nibble k holds channel 4m + k of token 2j for
 * k < 4 and channel 4m + k - 4 of token 2j+1 for k >= 4.  These give the byte
 * and the shift of one code. */
static void int4_k_nibble(int d, int* byte, int* shift) {
  int e = d % 8, k = (e & 1) ? 4 + e / 2 : e / 2;
  *byte = 4 * (d / 8) + k / 2;
  *shift = 4 * (k & 1);
}
static void int4_v_nibble(int t, int d, int* byte, int* shift) {
  int k = 4 * (t & 1) + d % 4;
  *byte = 4 * (d / 4) + k / 2;
  *shift = 4 * (k & 1);
}

/* Token `off`'s value codes (packed two per byte, even channel low) into its
 * nibble of each byte of its token pair's row. */
static void put_pair_nibbles(uint8_t* pair, int D, const uint8_t* packed, int off) {
  int d, sh = 4 * (off & 1);
  for (d = 0; d < D; d++) {
    uint8_t code = (d & 1) ? (uint8_t)(packed[d / 2] >> 4) : (uint8_t)(packed[d / 2] & 15);
    pair[d] = (uint8_t)((pair[d] & ~(15 << sh)) | (code << sh));
  }
}

static void write_kvarn_side(uint8_t* blk, int is_value, const uint8_t* codes, const float* scale,
                             const float* zero, const float* r, const float* c) {
  const int P = 128, D = 128;
  int t, i;
  if (!is_value) {
    uint8_t* pay = blk;
    uint8_t* meta = blk + P * D / 2 + P * D / 4;
    for (t = 0; t < P; t++)
      for (i = 0; i < D / 2; i++)
        pay[t * (D / 2) + i] = (uint8_t)(codes[t * D + 2 * i] | (codes[t * D + 2 * i + 1] << 4));
    for (i = 0; i < D; i++) put_f32(meta + 4 * i, scale[i]);
    for (i = 0; i < D; i++) put_f32(meta + 4 * (D + i), zero[i]);
    for (i = 0; i < D; i++) put_f32(meta + 4 * (2 * D + i), c[i]);
    for (i = 0; i < P; i++) put_f32(meta + 4 * (3 * D + i), r[i]);
  } else {
    uint8_t* pay = blk + P * D / 2;
    uint8_t* meta = blk + P * D / 2 + P * D / 4 + 4 * (3 * D + P);
    for (t = 0; t < P; t++)
      for (i = 0; i < D / 4; i++)
        pay[t * (D / 4) + i] = (uint8_t)(codes[t * D + 4 * i] | (codes[t * D + 4 * i + 1] << 2) |
                                         (codes[t * D + 4 * i + 2] << 4) | (codes[t * D + 4 * i + 3] << 6));
    for (i = 0; i < P; i++) put_f32(meta + 4 * i, scale[i]);
    for (i = 0; i < P; i++) put_f32(meta + 4 * (P + i), zero[i]);
    for (i = 0; i < P; i++) put_f32(meta + 4 * (2 * P + i), r[i]);
    for (i = 0; i < D; i++) put_f32(meta + 4 * (3 * P + i), c[i]);
  }
}

/* Quantize-on-write.  A negative slot is skipped; a slot beyond the pool is
 * skipped and counted.  KVarN writes whole tiles only: each run of 128 tokens
 * must fill one page in order, otherwise that tile is skipped and counted.
 * Returns the number of skipped-and-counted tokens, or -1 on a bad argument. */
int kvqo_write(int mode, uint8_t* pool, int num_pages, int P, int Hkv, int D, const float* k,
               const float* v, const int32_t* slots, int N, float k_scale, float v_scale) {
  int bad = 0, n, h, side;
  if (!pool || !slots || N < 0 || num_pages < 0 || Hkv <= 0 || kvqo_block_bytes(mode, P, D) == 0)
    return -1;
  if (mode == KVQO_KVARN_K4V2_G128) {
    float* X;
    uint8_t* codes;
    float scale[128], zero[128], r[128], c[128];
    int tile, t, d;
    if (P != 128 || D != 128 || N % 128 != 0) return -1;
    X = (float*)malloc(sizeof(float) * 128 * 128);
    codes = (uint8_t*)malloc(128 * 128);
    for (tile = 0; tile < N / 128; tile++) {
      int32_t s0 = slots[tile * 128];
      int ok = s0 >= 0 && s0 % 128 == 0 && s0 / 128 < num_pages;
      for (t = 1; t < 128 && ok; t++) ok = slots[tile * 128 + t] == s0 + t;
      if (!ok) { bad += 128; continue; }
      for (h = 0; h < Hkv; h++)
        for (side = 0; side < 2; side++) {
          const float* src = side ? v : k;
          uint8_t* blk = block_at(pool, mode, P, Hkv, D, s0 / 128, h);
          for (t = 0; t < 128; t++)
            for (d = 0; d < 128; d++) X[t * 128 + d] = src[((size_t)(tile * 128 + t) * Hkv + h) * D + d];
          kvqo_kvarn_tile(X, side, codes, scale, zero, r, c);
          write_kvarn_side(blk, side, codes, scale, zero, r, c);
        }
    }
    free(X);
    free(codes);
    return bad;
  }
  for (n = 0; n < N; n++) {
    int32_t slot = slots[n];
    int64_t page;
    int off;
    if (slot < 0) continue;
    page = slot / P;
    off = slot % P;
    if (page >= num_pages) { bad++; continue; }
    for (h = 0; h < Hkv; h++) {
      uint8_t* blk = block_at(pool, mode, P, Hkv, D, page, h);
      for (side = 0; side < 2; side++) {
        const float* x = (side ? v : k) + ((size_t)n * Hkv + h) * D;
        float s;
        switch (mode) {
          case KVQO_FP8_PER_TENSOR:
            kvqo_quant_row_fp8_pt(x, D, side ? v_scale : k_scale, blk + (size_t)side * P * D + (size_t)off * D);
            break;
          case KVQO_INT8_PER_TOKEN_HEAD:
            kvqo_quant_row_int8_pth(x, D, (int8_t*)(blk + (size_t)side * P * D + (size_t)off * D), &s);
            put_f32(blk + (size_t)2 * P * D + (size_t)side * 4 * P + 4 * off, s);
            break;
          case KVQO_FP8_PER_TOKEN_HEAD:
            kvqo_quant_row_fp8_pth(x, D, blk + (size_t)side * P * D + (size_t)off * D, &s);
            put_f32(blk + (size_t)2 * P * D + (size_t)side * 4 * P + 4 * off, s);
            break;
          case KVQO_NVFP4:
          case KVQO_NVFP4_4OVER6:
          case KVQO_INT4_PER_TOKEN_HEAD: {
            /* K: row `off` of [P][D/2]; V: this token's nibbles of its token pair's row */
            uint8_t packed[512];
            uint8_t* dst = side ? packed : blk + (size_t)off * D / 2;
            if (D > 1024) return -1;
            if (mode == KVQO_INT4_PER_TOKEN_HEAD) {
              uint8_t* row = side ? blk + (size_t)P * D / 2 + (size_t)(off / 2) * D : blk + (size_t)off * D / 2;
              int d, by, sh;
              kvqo_quant_row_int4_pth(x, D, packed, &s);
              put_f32(blk + (size_t)P * D + (size_t)side * 4 * P + 4 * off, s);
              for (d = 0; d < D; d++) {           /* the storage order above */
                uint8_t code = (d & 1) ? (uint8_t)(packed[d / 2] >> 4) : (uint8_t)(packed[d / 2] & 15);
                if (side) int4_v_nibble(off, d, &by, &sh); else int4_k_nibble(d, &by, &sh);
                row[by] = (uint8_t)((row[by] & ~(15 << sh)) | (code << sh));
              }
              break;
            } else {
              uint8_t* bs = blk + (size_t)P * D + (size_t)side * P * D / 16 + (size_t)off * D / 16;
              if (mode == KVQO_NVFP4) kvqo_quant_row_nvfp4(x, D, side ? v_scale : k_scale, dst, bs);
              else kvqo_quant_row_nvfp4_4over6(x, D, side ? v_scale : k_scale, dst, bs, NULL);
            }
            if (side) put_pair_nibbles(blk + (size_t)P * D / 2 + (size_t)(off / 2) * D, D, packed, off);
            break;
          }
          default: return -1;
        }
      }
    }
  }
  return bad;
}

/* Reconstruction x^ of one stored row, in fp64 (every product of a code and
 * a stored fp32 scale is exact in fp64; KVarN's triple product is rounded
 * once per operation in fp64). */
int kvqo_dequant_row(int mode, const uint8_t* pool, int num_pages, int P, int Hkv, int D,
                     float k_scale, float v_scale, int64_t slot, int h, int side, double* out) {
  int64_t page = slot / P;
  int t = (int)(slot % P), d;
  const uint8_t* blk;
  if (slot < 0 || page >= num_pages || h < 0 || h >= Hkv) return -1;
  blk = block_at((uint8_t*)pool, mode, P, Hkv, D, page, h);
  switch (mode) {
    case KVQO_FP8_PER_TENSOR: {
      double s = side ? v_scale : k_scale;
      const uint8_t* row = blk + (size_t)side * P * D + (size_t)t * D;
      for (d = 0; d < D; d++) out[d] = s * kvqo_e4m3_decode(row[d]);
      return 0;
    }
    case KVQO_INT8_PER_TOKEN_HEAD:
    case KVQO_FP8_PER_TOKEN_HEAD: {
      const uint8_t* row = blk + (size_t)side * P * D + (size_t)t * D;
      double s = get_f32(blk + (size_t)2 * P * D + (size_t)side * 4 * P + 4 * t);
      for (d = 0; d < D; d++)
        out[d] = s * (mode == KVQO_INT8_PER_TOKEN_HEAD ? (double)(int8_t)row[d] : kvqo_e4m3_decode(row[d]));
      return 0;
    }
    case KVQO_INT4_PER_TOKEN_HEAD: {
      const uint8_t* row = side ? blk + (size_t)P * D / 2 + (size_t)(t / 2) * D : blk + (size_t)t * D / 2;
      double s = get_f32(blk + (size_t)P * D + (size_t)side * 4 * P + 4 * t);
      for (d = 0; d < D; d++) {
        int by, sh, nib;
        if (side) int4_v_nibble(t, d, &by, &sh); else int4_k_nibble(d, &by, &sh);
        nib = (row[by] >> sh) & 15;
        out[d] = s * (double)(nib >= 8 ? nib - 16 : nib);
      }
      return 0;
    }
    case KVQO_NVFP4:
    case KVQO_NVFP4_4OVER6: {
      double st = side ? v_scale : k_scale;
      const uint8_t* row = blk + (size_t)t * D / 2;                               /* K */
      const uint8_t* pair = blk + (size_t)P * D / 2 + (size_t)(t / 2) * D;         /* V */
      const uint8_t* bs = blk + (size_t)P * D + (size_t)side * P * D / 16 + (size_t)t * D / 16;
      for (d = 0; d < D; d++) {
        uint8_t nib = side ? (uint8_t)((pair[d] >> (4 * (t & 1))) & 15)
                           : ((d & 1) ? (uint8_t)(row[d / 2] >> 4) : (uint8_t)(row[d / 2] & 15));
        out[d] = st * kvqo_e4m3_decode(bs[d / 16]) * kvqo_e2m1_decode(nib);
      }
      return 0;
    }
    case KVQO_KVARN_K4V2_G128: {
      if (P != 128 || D != 128) return -1;
      if (!side) {
        const uint8_t* row = blk + (size_t)t * (D / 2);
        const uint8_t* meta = blk + P * D / 2 + P * D / 4;
        double r = get_f32(meta + 4 * (3 * D + t));
        for (d = 0; d < D; d++) {
          int code = (d & 1) ? (row[d / 2] >> 4) : (row[d / 2] & 15);
          double sc = get_f32(meta + 4 * d), z = get_f32(meta + 4 * (D + d)), c = get_f32(meta + 4 * (2 * D + d));
          out[d] = r * c * (sc * code + z);
        }
      } else {
        const uint8_t* row = blk + P * D / 2 + (size_t)t * (D / 4);
        const uint8_t* meta = blk + P * D / 2 + P * D / 4 + 4 * (3 * D + P);
        double sc = get_f32(meta + 4 * t), z = get_f32(meta + 4 * (P + t)), r = get_f32(meta + 4 * (2 * P + t));
        for (d = 0; d < D; d++) {
          int code = (row[d / 4] >> (2 * (d % 4))) & 3;
          double c = get_f32(meta + 4 * (3 * P + d));
          out[d] = r * c * (sc * code + z);
        }
      }
      return 0;
    }
    default: return -1;
  }
}

/* Paged decode attention [P5 "K 与 V 的量化误差..."]: for query head hq of
 * sequence b, o = sum_t softmax_t(q . k^_t * softmax_scale) v^_t over the
 * sequence's tokens, read through the block table; the softmax subtracts the
 * maximum logit.  GQA [P5 "GQA"]: query head hq reads kv head hq / (Hq/Hkv).
 * Tokens whose page id is out of range are left out.  An empty sequence gives
 * o = 0.  KVarN: keys live in the rotated domain, so q' = H q and o = H o'. */
int kvqo_decode(int mode, const uint8_t* pool, int num_pages, int P, int Hkv, int D, float k_scale,
                float v_scale, const float* q, const int32_t* block_table, int max_pages,
                const int32_t* seq_lens, int B, int Hq, double softmax_scale, const int32_t* rows,
                int n_rows, double* out) {
  int G, nr, ri, d;
  double *qv, *kv, *vv, *s, *acc;
  if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return -1;
  G = Hq / Hkv;
  nr = rows ? n_rows : B * Hq;
  qv = (double*)malloc(sizeof(double) * D);
  kv = (double*)malloc(sizeof(double) * D);
  vv = (double*)malloc(sizeof(double) * D);
  acc = (double*)malloc(sizeof(double) * D);
  for (ri = 0; ri < nr; ri++) {
    int row = rows ? rows[ri] : ri;
    int b = row / Hq, hq = row % Hq, kvh = hq / G, n = seq_lens[b], t, valid = 0;
    double m = -INFINITY, l = 0.0;
    double* o = out + (size_t)row * D;
    for (d = 0; d < D; d++) qv[d] = q[(size_t)row * D + d];
    if (mode == KVQO_KVARN_K4V2_G128) kvqo_hadamard_f64(qv, D);
    s = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
    for (t = 0; t < n; t++) {
      int32_t page = (t / P < max_pages) ? block_table[(size_t)b * max_pages + t / P] : -1;
      double dot = 0.0;
      if (page < 0 || page >= num_pages) { s[t] = -INFINITY; continue; }
      kvqo_dequant_row(mode, pool, num_pages, P, Hkv, D, k_scale, v_scale, (int64_t)page * P + t % P, kvh, 0, kv);
      for (d = 0; d < D; d++) dot += qv[d] * kv[d];
      s[t] = dot * softmax_scale;
      if (s[t] > m) m = s[t];
      valid++;
    }
    for (d = 0; d < D; d++) acc[d] = 0.0;
    for (t = 0; t < n && valid; t++) {
      int32_t page = (t / P < max_pages) ? block_table[(size_t)b * max_pages + t / P] : -1;
      double p;
      if (page < 0 || page >= num_pages) continue;
      p = exp(s[t] - m);
      l += p;
      kvqo_dequant_row(mode, pool, num_pages, P, Hkv, D, k_scale, v_scale, (int64_t)page * P + t % P, kvh, 1, vv);
      for (d = 0; d < D; d++) acc[d] += p * vv[d];
    }
    for (d = 0; d < D; d++) o[d] = valid ? acc[d] / l : 0.0;
    if (mode == KVQO_KVARN_K4V2_G128 && valid) kvqo_hadamard_f64(o, D);
    free(s);
  }
  free(qv);
  free(kv);
  free(vv);
  free(acc);
  return 0;
}

/* KVarN with an open tile [P2 注意事项: a tile is one 128-token page, and the
 * backend keeps a small fixed decode workspace].  Read as: a sequence's last,
 * incomplete tile is not quantized yet; its raw rows sit in a tail buffer and
 * attention covers the quantized tiles plus those raw rows.  Written in the
 * input domain: each stored row is dequantized and rotated back (x^ = H x^',
 * H symmetric orthonormal), then o = sum_t softmax_t(q . k_t * scale) v_t over
 * the sequence's tokens, max-subtracted, in fp64.  Tokens of an out-of-range
 * page are left out; an empty sequence gives 0. */
int kvqo_decode_kvarn_tail(const uint8_t* pool, int num_pages, int Hkv, const float* q,
                           const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                           int Hq, double softmax_scale, const float* tail_k, const float* tail_v,
                           const int32_t* rows, int n_rows, double* out) {
  const int P = 128, D = 128;
  int G, nr, ri, d;
  double kv[128], vv[128], acc[128];
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  G = Hq / Hkv;
  nr = rows ? n_rows : B * Hq;
  for (ri = 0; ri < nr; ri++) {
    int row = rows ? rows[ri] : ri;
    int b = row / Hq, hq = row % Hq, kvh = hq / G, n = seq_lens[b], nf = n - n % P, t, valid = 0;
    double m = -INFINITY, l = 0.0, *s;
    double* o = out + (size_t)row * D;
    const float* qr = q + (size_t)row * D;
    s = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
    for (t = 0; t < n; t++) {               /* pass 1: scores */
      double dot = 0.0;
      if (t < nf) {
        int32_t page = (t / P < max_pages) ? block_table[(size_t)b * max_pages + t / P] : -1;
        if (page < 0 || page >= num_pages) { s[t] = -INFINITY; continue; }
        kvqo_dequant_row(KVQO_KVARN_K4V2_G128, pool, num_pages, P, Hkv, D, 1.0f, 1.0f,
                         (int64_t)page * P + t % P, kvh, 0, kv);
        kvqo_hadamard_f64(kv, D);
      } else {
        for (d = 0; d < D; d++) kv[d] = tail_k[(((size_t)b * P + (t - nf)) * Hkv + kvh) * D + d];
      }
      for (d = 0; d < D; d++) dot += (double)qr[d] * kv[d];
      s[t] = dot * softmax_scale;
      if (s[t] > m) m = s[t];
      valid++;
    }
    for (d = 0; d < D; d++) acc[d] = 0.0;
    for (t = 0; t < n && valid; t++) {      /* pass 2: weights and values */
      double p;
      if (s[t] == -INFINITY) continue;
      p = exp(s[t] - m);
      l += p;
      if (t < nf) {
        int32_t page = block_table[(size_t)b * max_pages + t / P];
        kvqo_dequant_row(KVQO_KVARN_K4V2_G128, pool, num_pages, P, Hkv, D, 1.0f, 1.0f,
                         (int64_t)page * P + t % P, kvh, 1, vv);
        kvqo_hadamard_f64(vv, D);
      } else {
        for (d = 0; d < D; d++) vv[d] = tail_v[(((size_t)b * P + (t - nf)) * Hkv + kvh) * D + d];
      }
      for (d = 0; d < D; d++) acc[d] += p * vv[d];
    }
    for (d = 0; d < D; d++) o[d] = valid ? acc[d] / l : 0.0;
    free(s);
  }
  return 0;
}
