// kvq_write.cu -- quantize-on-write kernels and per-tensor scale setup.
//
// Compiled with -fmad=false and written with explicit _rn intrinsics so every
// fp32 operation is individually rounded: the quantized bytes and scales are
// bit-identical to the specification.
//
// Sources (web pages, by title and section):
//  "KV Cache 量化深度解析：Per-Tensor、Per-Token-Head 与 NVFP4", sec. 2.1-2.3;
//  "KV Cache 量化 · LLM Glossary", first section (s = max|x|/127, q = clip(round(x/s)));
//  "KV 量化" (rustineverything.app), 写和读 (divide by the scale, cast, store as uint8),
//     scale 和数据放在一起 (int4_per_token_head: head_size/2 bytes plus an fp32 scale);
//  "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化", 双层缩放 (q = Q_E2M1(x/(s_t s_b))),
//     KV 的写入与读取路径 (compute scales, round and clip to E2M1, pack two per byte),
//     用一组数直观看缩放的作用 (nvfp4_4over6: a max/6 or max/4 block scale by
//     reconstruction error);
//  "KVarN：华为推出的原生 vLLM KV-cache 量化后端...", 技术原理 (tile, Hadamard rotation,
//     alternating std normalisation, asymmetric RTN), 配置与部署 (k4v2, tile 128) and
//     注意事项 (tile = page; the open tile's raw rows wait in a tail buffer).
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

struct WriteArgs {
  uint8_t* pool;
  const void* k;
  const void* v;
  const int32_t* slots;
  long long num_tokens;
  int Hkv, P, log2P, num_pages;
  size_t block_bytes;
  // KVarN open tiles (kvq_kvarn_append): sequence of each token, and the tail
  // buffer, K rows [num_seqs][128][Hkv][D] then V rows, io dtype
  const int32_t* seq_ids;
  uint8_t* tail;
  int num_seqs;
  // the pool's blocks and the tail buffer, as spans (debug-build store checks)
  Span pool_span, tail_span;
  // -0.0f, as a value the compiler cannot see: the addend that turns a packed
  // fused multiply-add into an exactly rounded product (see mul2z)
  float neg_zero = -0.0f;
};

template <typename T>
__device__ __forceinline__ void load16(const T* p, float* f);
template <>
__device__ __forceinline__ void load16<__half>(const __half* p, float* f) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
template <>
__device__ __forceinline__ void load16<float>(const float* p, float* f) {
  float4 u = __ldg(reinterpret_cast<const float4*>(p));
  f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}

// 16 loaded bytes -> fp32 values (exact widening of fp16; fp32 as is).
template <typename T>
__device__ __forceinline__ void widen16(const uint4& u, float* f);
template <>
__device__ __forceinline__ void widen16<__half>(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(u32_as_h2(w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
template <>
__device__ __forceinline__ void widen16<float>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}

template <int N>
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint32_t* w);
template <int N>
__device__ __forceinline__ void store_bytes_chk(uint8_t* dst, const uint32_t* w, const WriteArgs& a) {
  if (in_span(dst, N, a.pool_span, a.pool)) store_bytes<N>(dst, w);
}
template <>
__device__ __forceinline__ void store_bytes<2>(uint8_t* dst, const uint32_t* w) {
  *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w[0]);
}
template <>
__device__ __forceinline__ void store_bytes<4>(uint8_t* dst, const uint32_t* w) {
  *reinterpret_cast<uint32_t*>(dst) = w[0];
}
template <>
__device__ __forceinline__ void store_bytes<8>(uint8_t* dst, const uint32_t* w) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
}

// x / d for a constant divisor d, given rd = RN(1/d): q0 = RN(x rd), the
// remainder r = x - q0 d (exact, one FMA), q = RN(q0 + r rd) -- Markstein's
// correction step ("Computation of elementary functions on the IBM RISC
// System/6000 processor", 1990).  For the divisors and inputs used here it
// returns the IEEE quotient RN(x/d) for every input, checked exhaustively over
// all fp32 values: d = 127, 448, 7 with x >= 1e-8 (scales of max(amax, 1e-8))
// and d = 15, 3 with any finite x >= 0 (KVarN ranges, zero and subnormals
// included); infinities and NaN take the IEEE division.
__device__ __forceinline__ float div_const(float x, float d, float rd) {
  if (!(x <= 0x1.fffffep127f)) return __fdiv_rn(x, d);  // inf and NaN keep IEEE semantics
  const float q0 = __fmul_rn(x, rd);
  const float r = __fmaf_rn(-q0, d, x);
  return __fmaf_rn(r, rd, q0);
}
constexpr float kRcp127 = 0x1.020408p-7f, kRcp448 = 0x1.24924ap-9f, kRcp7 = 0x1.24924ap-3f;
constexpr float kRcp15 = 0x1.111112p-4f, kRcp3 = 0x1.555556p-2f;

// The reciprocals are RN(1/d): checked here against the compiler's own
// correctly rounded constant division.
static_assert(kRcp127 == 1.0f / 127.0f && kRcp448 == 1.0f / 448.0f && kRcp7 == 1.0f / 7.0f,
              "reciprocal constants of the per-token-head scales");
static_assert(kRcp15 == 1.0f / 15.0f && kRcp3 == 1.0f / 3.0f, "reciprocal constants of the RTN scales");

// Packed fp32 pairs (f32x2): each lane is rounded on its own, exactly as the
// scalar __fadd_rn / __fmul_rn, so a pair op is two of the specification's
// operations in one instruction.  Written as PTX with the explicit .rn
// modifier, which keeps the compiler from contracting a product and a sum
// into one fused multiply-add (the packed intrinsics were contracted).
__device__ __forceinline__ unsigned long long f2_bits(float2 a) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 bits_f2(unsigned long long r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
// The code generator fuses a packed product into a packed sum that consumes it
// (explicit .rn and -fmad=false notwithstanding; measured on GB300: 18% of
// (a b) + c pairs differed from the two rounded steps).  A product that feeds
// a sum is therefore written as fma(a, b, -0): a b + (-0) rounded once is the
// rounded product, for every a b (a zero keeps its sign), and a fused
// multiply-add has nothing left to fuse with.  z = (-0, -0) must come from a
// kernel argument so that the addend is not folded away.
__device__ __forceinline__ float2 mul2z(float2 a, float2 b, float2 z) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(z)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }

// Encoding of the IEEE quotient RN(x/s) without a division on the common path.
// With r the hardware's approximate reciprocal of s (relative error below
// 2^-21 = 8u, u = 2^-24), rlo = RN(r(1 - 2^-20)) and rhi = RN(r(1 + 2^-20)),
// the products RN(x rlo) and RN(x rhi) enclose RN(x/s): their relative
// distance to x/s is at least 16u - 8u - 2u on each side, while RN(x/s) is
// within u of it.  Every encoder used here (round-to-nearest-even onto a
// grid, with saturation) is monotone, so when both ends encode to the same
// code, that is the code of RN(x/s); when they differ the quotient is computed
// exactly.  Scales whose reciprocal is not a comfortable normal number always
// divide.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
struct QDiv {
  float s, rlo, rhi;
  bool fast;
  __device__ __forceinline__ explicit QDiv(float s_) : s(s_) {
    const float r = rcp_approx(s_);
    fast = r >= 0x1p-100f && r <= 0x1p100f;
    rlo = __fmul_rn(r, 1.0f - 0x1p-20f);
    rhi = __fmul_rn(r, 1.0f + 0x1p-20f);
  }
  // E4M3 codes of x1:x0 (x0 in the low byte)
  __device__ __forceinline__ uint32_t e4m3x2(float x1, float x0) const {
    const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(x1, rlo), __fmul_rn(x0, rlo));
    const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(x1, rhi), __fmul_rn(x0, rhi));
    if (fast && lo == hi) return lo;
    return f32x2_to_e4m3x2(__fdiv_rn(x1, s), __fdiv_rn(x0, s));
  }
  // Four int8 codes clamp(rint(x/s), -127, 127), x[0] in the low byte.  rint
  // is done by adding 1.5 * 2^23: round-to-nearest-even leaves the integer in
  // the low mantissa bits, whose low byte is the two's-complement code.  The
  // fast path also requires both ends inside [-127, 127] (bit patterns
  // 0x4B400000 -127 .. +127), so neither the clamp nor a NaN can reach it.
  // (The products and the additions run as packed pairs; z = (-0, -0), see mul2z.)
  __device__ __forceinline__ uint32_t int8x4(const float* x, float2 z) const {
    const float2 magic = dup2(12582912.0f);  // 1.5 * 2^23
    uint32_t lo[4], bad = fast ? 0u : 1u;
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const float2 x2 = make_float2(x[e], x[e + 1]);
      const float2 l2 = add2(mul2z(x2, dup2(rlo), z), magic), h2 = add2(mul2z(x2, dup2(rhi), z), magic);
      lo[e] = __float_as_uint(l2.x);
      lo[e + 1] = __float_as_uint(l2.y);
      bad |= (lo[e] ^ __float_as_uint(h2.x)) | static_cast<uint32_t>(lo[e] - 0x4B3FFF81u > 254u);
      bad |= (lo[e + 1] ^ __float_as_uint(h2.y)) | static_cast<uint32_t>(lo[e + 1] - 0x4B3FFF81u > 254u);
    }
    if (bad == 0) return prmt(prmt(lo[0], lo[1], 0x0040u), prmt(lo[2], lo[3], 0x0040u), 0x5410u);
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float qv = fminf(fmaxf(rintf(__fdiv_rn(x[e], s)), -127.0f), 127.0f);
      w |= (static_cast<uint32_t>(__float2int_rn(qv)) & 0xFFu) << (8 * e);
    }
    return w;
  }
  // N <= 8 signed 4-bit codes clamp(rint(x/s), -7, 7) of x[0..N), two's
  // complement.  Same rint as int8x4; the fast path requires both ends inside
  // [-7, 7] (bit patterns 0x4B400000 -7 .. +7), whose low nibble is then the
  // code.  KEY = false: x[e] in nibble e.  KEY = true, the key-word order of
  // an 8-channel group: x[e] in nibble e/2 for even e, 4 + e/2 for odd e.
  template <int N, bool KEY = false>
  __device__ __forceinline__ uint32_t int4x8(const float* x, float2 z) const {
    static_assert(N % 2 == 0, "pairs");
    const float2 magic = dup2(12582912.0f);  // 1.5 * 2^23
    uint32_t lo[N], bad = fast ? 0u : 1u;
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      const float2 x2 = make_float2(x[e], x[e + 1]);
      const float2 l2 = add2(mul2z(x2, dup2(rlo), z), magic), h2 = add2(mul2z(x2, dup2(rhi), z), magic);
      lo[e] = __float_as_uint(l2.x);
      lo[e + 1] = __float_as_uint(l2.y);
      bad |= (lo[e] ^ __float_as_uint(h2.x)) | static_cast<uint32_t>(lo[e] - 0x4B3FFFF9u > 14u);
      bad |= (lo[e + 1] ^ __float_as_uint(h2.y)) | static_cast<uint32_t>(lo[e + 1] - 0x4B3FFFF9u > 14u);
    }
    if (bad != 0) {
#pragma unroll
      for (int e = 0; e < N; ++e) {
        const float qv = fminf(fmaxf(rintf(__fdiv_rn(x[e], s)), -7.0f), 7.0f);
        lo[e] = static_cast<uint32_t>(__float2int_rn(qv));
      }
    }
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < N; ++e) w |= (lo[e] & 0xFu) << (4 * (KEY ? ((e & 1) ? 4 + e / 2 : e / 2) : e));
    return w;
  }
  // eight E2M1 codes (pairs packed low nibble first) of x[0..n)
  template <int N>
  __device__ __forceinline__ uint32_t e2m1x8(const float* x) const {
    float ylo[8], yhi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ylo[i] = i < N ? __fmul_rn(x[i], rlo) : 0.0f;
      yhi[i] = i < N ? __fmul_rn(x[i], rhi) : 0.0f;
    }
    const uint32_t lo = f32x8_to_e2m1x8(ylo), hi = f32x8_to_e2m1x8(yhi);
    if (fast && lo == hi) return lo;
#pragma unroll
    for (int i = 0; i < 8; ++i) ylo[i] = i < N ? __fdiv_rn(x[i], s) : 0.0f;
    return f32x8_to_e2m1x8(ylo);
  }
};

// Group max over TPR consecutive lanes (TPR a power of two <= 32).
template <int TPR>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = 1; o < TPR; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Squared reconstruction error of a 16-value block whose codes (w, this
// thread's VEC of them) reconstruct as E2M1(code) * den: fp32, every operation
// rounded alone, summed as a pairwise tree of neighbours -- within the thread
// for its VEC consecutive values, then across the TPB lanes of the block
// (xor 1, 2: each level adds two neighbouring subtrees, and fp32 addition is
// commutative, so every lane holds the same total).
// Packed: values i and i + VEC/2 share a pair, so the neighbour levels of the
// tree are pair additions and the last one adds the pair's two halves.
template <int VEC, int TPB>
__device__ __forceinline__ float block_sse(const float* x, uint32_t w, float den, float2 z) {
  constexpr int H = VEC / 2;
  uint32_t h[4];
  e2m1x8_to_f16x2x4(w, h);
  float val[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const __half2 p = u32_as_h2(h[i / 2]);
    val[i] = (i & 1) ? __high2float(p) : __low2float(p);
  }
  float2 e[H];  // (error^2 of value k, of value k + H)
#pragma unroll
  for (int k = 0; k < H; ++k) {
    const float2 d = sub2(make_float2(x[k], x[k + H]), mul2z(make_float2(val[k], val[k + H]), dup2(den), z));
    e[k] = mul2z(d, d, z);
  }
#pragma unroll
  for (int st = 1; st < H; st <<= 1)
#pragma unroll
    for (int k = 0; k < H; k += 2 * st) e[k] = add2(e[k], e[k + st]);
  float t = __fadd_rn(e[0].x, e[0].y);
#pragma unroll
  for (int o = 1; o < TPB; o <<= 1) t = __fadd_rn(t, __shfl_xor_sync(kFull, t, o));
  return t;
}

// NVFP4 codes of a thread's VEC values (its 16-value block shared with TPB =
// 16 / VEC lanes): the E4M3 block scale byte sb and the E2M1 codes packed two
// per byte, even channel in the low nibble (sb = 0 gives all-zero codes).
// F46 (nvfp4_4over6): the block is also coded with the max/4 scale
// E4M3(amax / (4 s_t)), and that coding is kept when its block_sse is smaller.
// q6, q4: the quotient brackets of RN(6 s_t) and RN(4 s_t).
template <int VEC, int TPB, bool F46>
__device__ __forceinline__ void nvfp4_codes(const float* x, float st, const QDiv& q6, const QDiv& q4, float2 z,
                                            uint32_t& w, uint32_t& sb) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = group_max<TPB>(amax);
  sb = q6.e4m3x2(0.0f, amax) & 0xFFu;  // E4M3(RN(amax / (6 s_t)))
  const float sbf = e4m3_to_f32(sb);
  const float den = __fmul_rn(st, sbf);
  w = sbf != 0.0f ? QDiv(den).e2m1x8<VEC>(x) : 0u;
  if constexpr (F46) {
    const uint32_t sb4 = q4.e4m3x2(0.0f, amax) & 0xFFu;  // E4M3(RN(amax / (4 s_t)))
    const float sbf4 = e4m3_to_f32(sb4);
    const float den4 = __fmul_rn(st, sbf4);
    const uint32_t w4 = sbf4 != 0.0f ? QDiv(den4).e2m1x8<VEC>(x) : 0u;
    if (block_sse<VEC, TPB>(x, w4, den4, z) < block_sse<VEC, TPB>(x, w, den, z)) {
      w = w4;
      sb = sb4;
    }
  }
}

template <int MODE>
constexpr bool kFourBit = MODE == KVQ_NVFP4 || MODE == KVQ_NVFP4_4OVER6 || MODE == KVQ_INT4_PER_TOKEN_HEAD;

// The n = 4 or 8 codes packed in w (two per byte) spread one per byte, in the
// low nibble: bytes c0, c1, c2, c3 (| c4..c7).
__device__ __forceinline__ uint2 spread_codes(uint32_t w) {
  const uint32_t even = w & 0x0F0F0F0Fu, odd = (w >> 4) & 0x0F0F0F0Fu;
  return make_uint2(prmt(even, odd, 0x5140u), prmt(even, odd, 0x7362u));
}

// The side's per-tensor scale (FP8 per-tensor s, NVFP4 s_t) and the quotient
// brackets built from it, set up once per thread: the pool header does not
// change during a write.
struct TensorScale {
  float st;
  QDiv qs;  // FP8 per-tensor: x / s; NVFP4: amax / (6 s_t)
  QDiv q4;  // NVFP4 4over6: amax / (4 s_t)
  template <int MODE>
  __device__ __forceinline__ static TensorScale make(const WriteArgs& a, int side) {
    const float st = *reinterpret_cast<const float*>(a.pool + (side ? kHdrVScaleOffset : kHdrKScaleOffset));
    return TensorScale{st, QDiv(MODE == KVQ_FP8_PER_TENSOR ? st : __fmul_rn(6.0f, st)), QDiv(__fmul_rn(4.0f, st))};
  }
};

// Quantize one (token, kv head, side) row of D values, held by a group of TPR
// threads with VEC values each (thread j: values j*VEC ..), and store it at
// slot (skipped when slot < 0; flagged and skipped when out of range).
template <int MODE, int D, int VEC, int TPR>
__device__ __forceinline__ void quantize_row(const WriteArgs& a, int h, int side, int slot, int j, const float* x,
                                             const TensorScale& ts) {
  bool active = slot >= 0;
  const int page = slot >> a.log2P;
  const int off = slot & (a.P - 1);
  if (active && page >= a.num_pages) {
    if (j == 0) set_error(a.pool, KVQ_DEVERR_SLOT_RANGE);
    active = false;
  }
  uint8_t* blk = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes;

  if constexpr (MODE == KVQ_FP8_PER_TENSOR) {
    const QDiv& q = ts.qs;
    uint32_t w[VEC / 4];
#pragma unroll
    for (int i = 0; i < VEC; i += 4) w[i / 4] = q.e4m3x2(x[i + 1], x[i]) | (q.e4m3x2(x[i + 3], x[i + 2]) << 16);
    if (active) store_bytes_chk<VEC>(blk + (size_t)side * a.P * D + (size_t)off * D + j * VEC, w, a);
  } else if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD || MODE == KVQ_FP8_PER_TOKEN_HEAD) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = group_max<TPR>(amax);
    const float s = MODE == KVQ_INT8_PER_TOKEN_HEAD ? div_const(fmaxf(amax, 1e-8f), 127.0f, kRcp127)
                                                    : div_const(fmaxf(amax, 1e-8f), 448.0f, kRcp448);
    const QDiv q(s);
    uint32_t w[VEC / 4];
#pragma unroll
    for (int i = 0; i < VEC; i += 4) {
      if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD) {
        w[i / 4] = q.int8x4(x + i, dup2(a.neg_zero));
      } else {
        w[i / 4] = q.e4m3x2(x[i + 1], x[i]) | (q.e4m3x2(x[i + 3], x[i + 2]) << 16);
      }
    }
    if (active) {
      store_bytes_chk<VEC>(blk + (size_t)side * a.P * D + (size_t)off * D + j * VEC, w, a);
      if (j == 0) st_chk(reinterpret_cast<float*>(blk + (size_t)2 * a.P * D + (size_t)side * 4 * a.P + 4 * off), s, a.pool_span, a.pool);
    }
  } else if constexpr (MODE == KVQ_NVFP4 || MODE == KVQ_NVFP4_4OVER6) {  // keys; values: pair_values_pass
    constexpr int TPB = 16 / VEC;  // threads per 16-value block
    uint32_t w[1], sb;
    nvfp4_codes<VEC, TPB, MODE == KVQ_NVFP4_4OVER6>(x, ts.st, ts.qs, ts.q4, dup2(a.neg_zero), w[0], sb);
    if (active) {
      store_bytes_chk<VEC / 2>(blk + (size_t)off * D / 2 + j * VEC / 2, w, a);
      if ((j % TPB) == 0)
        st_chk(blk + (size_t)a.P * D + (size_t)off * D / 16 + (j * VEC) / 16, static_cast<uint8_t>(sb), a.pool_span, a.pool);
    }
  } else if constexpr (MODE == KVQ_INT4_PER_TOKEN_HEAD) {  // keys; values: pair_values_pass
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = group_max<TPR>(amax);
    const float s = div_const(fmaxf(amax, 1e-8f), 7.0f, kRcp7);
    // a key word holds an 8-channel group, even channels in its low half-word:
    // with 4 values per thread, two lanes fill one word (the odd lane's
    // channels 4..7 sit one byte higher) and the even lane stores it
    uint32_t w[1] = {QDiv(s).int4x8<VEC, true>(x, dup2(a.neg_zero))};
    if constexpr (VEC == 4) {
      if (j & 1) w[0] <<= 8;
      w[0] |= __shfl_xor_sync(kFull, w[0], 1);
    }
    if (active) {
      if (VEC == 8 || (j & 1) == 0) store_bytes_chk<4>(blk + (size_t)off * D / 2 + (j * VEC / 8) * 4, w, a);
      if (j == 0) st_chk(reinterpret_cast<float*>(blk + (size_t)a.P * D + 4 * off), s, a.pool_span, a.pool);
    }
  }
}


// 4-bit values (NVFP4, NVFP4 4over6, INT4): token-pair rows, byte (k, d) of a
// page holding channel d of tokens 2k (low nibble) and 2k + 1.  A token with
// an even slot whose successor in the batch holds the next slot stores the
// pair's bytes whole and the successor stores nothing; every other token
// writes its own nibbles with 32-bit atomic AND/OR (two tokens never share a
// nibble, so these commute), e.g. the one new token of a decode step.  The
// successor's codes come from the next row group of the same warp (a shuffle)
// when a warp holds two row groups (TPR = 16), else through shared memory
// (whole CTA, one barrier).  Scales (NVFP4 block scales, the INT4 token
// scale) are per token and stored directly.
template <int MODE, int D, int VEC, int TPR, int NTOK, int R, typename T>
__device__ __forceinline__ void pair_values_pass(const WriteArgs& a, int h, const int* slot, const uint4* raw,
                                                 int j, const TensorScale& ts) {
  constexpr int TPB = 16 / VEC;
  constexpr int TOK = NTOK / R;
  constexpr bool kInWarp = TPR == 16;
  __shared__ uint32_t codes[kInWarp ? 1 : NTOK * TPR];
  __shared__ int vslot[kInWarp ? 1 : NTOK];
  const int g = threadIdx.x / TPR;
  uint32_t wr[R];
  int sr[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float x[VEC];
    widen16<T>(raw[r], x);
    const int s = slot[r];
    bool active = s >= 0;
    const int page = s >> a.log2P, off = s & (a.P - 1);
    if (active && page >= a.num_pages) {
      if (j == 0) set_error(a.pool, KVQ_DEVERR_SLOT_RANGE);
      active = false;
    }
    uint8_t* blk = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes;
    if constexpr (MODE == KVQ_INT4_PER_TOKEN_HEAD) {
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(x[i]));
      amax = group_max<TPR>(amax);
      const float sc = div_const(fmaxf(amax, 1e-8f), 7.0f, kRcp7);
      wr[r] = QDiv(sc).int4x8<VEC>(x, dup2(a.neg_zero));
      if (active && j == 0)
        st_chk(reinterpret_cast<float*>(blk + (size_t)a.P * D + (size_t)4 * a.P + 4 * off), sc, a.pool_span, a.pool);
    } else {
      uint32_t sb;
      nvfp4_codes<VEC, TPB, MODE == KVQ_NVFP4_4OVER6>(x, ts.st, ts.qs, ts.q4, dup2(a.neg_zero), wr[r], sb);
      if (active && (j % TPB) == 0)
        st_chk(blk + (size_t)a.P * D + (size_t)a.P * D / 16 + (size_t)off * D / 16 + (j * VEC) / 16, static_cast<uint8_t>(sb),
               a.pool_span, a.pool);
    }
    sr[r] = active ? s : -1;
    if constexpr (!kInWarp) {
      const int li = g + TOK * r;
      codes[li * TPR + j] = wr[r];
      if (j == 0) vslot[li] = sr[r];
    }
  }
  if constexpr (!kInWarp) __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int s = sr[r];
    int next, prev;
    uint32_t other;
    if constexpr (kInWarp) {  // lanes 0-15: row group g (even), lanes 16-31: g + 1
      const bool lower = (threadIdx.x & 16) == 0;
      const int up = __shfl_down_sync(0xffffffffu, s, 16), down = __shfl_up_sync(0xffffffffu, s, 16);
      other = __shfl_down_sync(0xffffffffu, wr[r], 16);
      next = lower ? up : -1;
      prev = lower ? -1 : down;
    } else {
      const int li = g + TOK * r;
      next = li + 1 < NTOK ? vslot[li + 1] : -1;
      prev = li > 0 ? vslot[li - 1] : -1;
      other = li + 1 < NTOK ? codes[(li + 1) * TPR + j] : 0u;
    }
    if (s < 0 || ((s & 1) && prev == s - 1)) continue;  // nothing, or written with the pair's first token
    const int page = s >> a.log2P, off = s & (a.P - 1);
    uint8_t* dst = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes + (size_t)a.P * D / 2 +
                   (size_t)(off >> 1) * D + j * VEC;
    if constexpr (MODE == KVQ_INT4_PER_TOKEN_HEAD) {
      // INT4 pair-row word: 4 channels of the even token in the low half-word,
      // the same channels of the odd token in the high half-word
      if (!(s & 1) && next == s + 1) {
        const uint2 both = make_uint2(prmt(wr[r], other, 0x5410u), prmt(wr[r], other, 0x7632u));
        if constexpr (VEC == 8) st_chk(reinterpret_cast<uint2*>(dst), both, a.pool_span, a.pool);
        else st_chk(reinterpret_cast<uint32_t*>(dst), both.x, a.pool_span, a.pool);
      } else {
        const int sh = 16 * (off & 1);
        const uint32_t m = 0xFFFFu << sh;
        unsigned int* wd = reinterpret_cast<unsigned int*>(dst);
        if (!in_span(wd, VEC == 8 ? 8 : 4, a.pool_span, a.pool)) continue;
        atomicAnd(wd, ~m);
        atomicOr(wd, (wr[r] & 0xFFFFu) << sh);
        if constexpr (VEC == 8) {
          atomicAnd(wd + 1, ~m);
          atomicOr(wd + 1, (wr[r] >> 16) << sh);
        }
      }
      continue;
    }
    if (!(s & 1) && next == s + 1) {
      // even channels: my low nibbles | the successor's low nibbles << 4; odd
      // channels: my high nibbles >> 4 | the successor's high nibbles; then
      // interleave the bytes back into channel order
      const uint32_t ev = bitsel(wr[r], other << 4, 0x0F0F0F0Fu);
      const uint32_t od = bitsel(wr[r] >> 4, other, 0x0F0F0F0Fu);
      const uint2 both = make_uint2(prmt(ev, od, 0x5140u), prmt(ev, od, 0x7362u));
      if constexpr (VEC == 8) st_chk(reinterpret_cast<uint2*>(dst), both, a.pool_span, a.pool);
      else st_chk(reinterpret_cast<uint32_t*>(dst), both.x, a.pool_span, a.pool);
    } else {
      const uint2 mine = spread_codes(wr[r]);
      const int sh = 4 * (off & 1);
      const uint32_t m = 0x0F0F0F0Fu << sh;
      unsigned int* wd = reinterpret_cast<unsigned int*>(dst);
      if (!in_span(wd, VEC == 8 ? 8 : 4, a.pool_span, a.pool)) continue;
      atomicAnd(wd, ~m);
      atomicOr(wd, mine.x << sh);
      if constexpr (VEC == 8) {
        atomicAnd(wd + 1, ~m);
        atomicOr(wd + 1, mine.y << sh);
      }
    }
  }
}

// Rows of D values, one per group of TPR threads (VEC = 16 bytes of input per
// thread), kRowsPerThread rows per thread with every load issued before the
// first row is converted, so that enough bytes are in flight to cover HBM
// latency.  Grid: (token blocks, kv head, side), so no index needs a division;
// a block's consecutive tokens land in consecutive rows of the same pages.
// Modes 1-4.
#ifndef KVQ_WRITE_ROWS
#define KVQ_WRITE_ROWS 4
#endif
constexpr int kRowsPerThread = KVQ_WRITE_ROWS;

template <int MODE, typename T, int D>
__global__ void __launch_bounds__(256) write_rows_kernel(WriteArgs a) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int TPR = D / VEC;
  constexpr int TOK = 256 / TPR;  // tokens per block and row pass
  constexpr int R = kRowsPerThread;
  static_assert(TPR >= 2 && TPR <= 32 && (TPR & (TPR - 1)) == 0, "row group");
  const int h = blockIdx.y, side = blockIdx.z;
  const long long tok0 = (long long)blockIdx.x * (TOK * R) + threadIdx.x / TPR;
  const int j = threadIdx.x % TPR;
  const T* src = static_cast<const T*>(side ? a.v : a.k);

  int slot[R];
  uint4 raw[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const long long token = tok0 + (long long)r * TOK;
    const bool in = token < a.num_tokens;
    slot[r] = in ? __ldg(a.slots + token) : -1;
    raw[r] = in ? __ldg(reinterpret_cast<const uint4*>(src + (token * a.Hkv + h) * D + j * VEC))
                : make_uint4(0u, 0u, 0u, 0u);
  }
  const TensorScale ts = TensorScale::make<MODE>(a, side);  // unused (and dropped) by the per-token-head modes
  if constexpr (kFourBit<MODE>) {
    if (side == 1) {
      pair_values_pass<MODE, D, VEC, TPR, TOK * R, R, T>(a, h, slot, raw, j, ts);
      return;
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float x[VEC];
    widen16<T>(raw[r], x);
    quantize_row<MODE, D, VEC, TPR>(a, h, side, slot[r], j, x, ts);
  }
}

// ------------------------------------------------------------------ KVarN
// One CTA of 256 threads per (128-token tile, kv head, side).
//  1. Load + rotate: thread (token t, half) holds channels 64 half .. +63;
//     Walsh-Hadamard stages h = 1 .. 32 run in registers, h = 64 between the
//     two halves' lanes, then the fp32 1/sqrt(128) (0x3DB504F3).  The tile is
//     staged in shared memory once (row stride 144 floats).
//  2. Normalise: thread (warp w, lane l) holds y[i][j] for tokens
//     t = tl + 16 i and channels d = dl + 16 j (i, j = 0..7), with dl = l & 15
//     and tl = (l >> 4) | (w << 1).  The canonical 128-sum (v[i] += v[i + off],
//     off = 64, 32, .., 1) therefore takes its first three levels inside the
//     thread on either axis.  Token sums finish with lane shuffles on
//     d bits 3, 2, 1, 0 -- recursive halving, so that afterwards each lane
//     owns one of its eight tokens and computes that token's sqrt and
//     reciprocal once; channel sums finish through shared memory on t bits
//     3, 2, 1, 0 (one thread per channel).  Every fp32 operation is the
//     specification's, rounded alone (-fmad=false); a line whose std is below
//     1e-8 is multiplied by exactly 1 instead of being skipped.
//  3. Round: asymmetric RTN, keys per channel over tokens (4 bits), values
//     per token over channels (2 bits); codes staged as bytes in shared
//     memory, then packed and stored as 16-byte rows.
constexpr int kKvTile = 128;
constexpr int kKvThreads = 256;
constexpr int kKvYS = 144;  // floats per staged token row (banks: +16 per row)
// Staged position of channel d in token row t: its 4-channel chunk index is
// XORed with (d's bit 6, t's bit 1), so that the rotation's 16-byte stores
// (8 threads: 4 rows x 2 halves, one chunk each) hit 8 distinct bank groups,
// while the normalisation's loads (16 channels of row 2k, 16 of row 2k + 1)
// still fill the 32 banks once.
__device__ __forceinline__ int kv_ypos(int t, int d) { return d ^ ((d >> 4) & 4) ^ ((t << 2) & 8); }
constexpr int kKvCS = 144;  // bytes per staged code row
struct KvSmem {
  float Y[kKvTile * kKvYS];     // rotated tile; later the code bytes
  float part[16 * kKvYS];       // per-channel partial sums / minima [t_lo][d]
  float part2[16 * kKvYS];      // per-channel maxima [t_lo][d]
  float st0[kKvTile], st1[kKvTile];  // per-line statistics
  float fr[kKvTile], fc[kKvTile];    // final factors r_t, c_d
  float tm[kKvTile], ti[kKvTile];    // per-token mean, 1/std of the token steps, [tl][i]: token tl + 16 i
};
constexpr size_t kKvSmem = sizeof(KvSmem);
#ifndef KVQ_KVARN_PAIR_UNROLL
#define KVQ_KVARN_PAIR_UNROLL 1
#endif
constexpr int kKvPairUnroll = KVQ_KVARN_PAIR_UNROLL;  // normalisation pairs unrolled

// In-thread levels 64, 32, 16 of the canonical sum over eight values whose
// index bits are the line's bits 6, 5, 4 (v[k] = element 16 k + lo).
__device__ __forceinline__ float tree8(const float* v) {
  const float a0 = __fadd_rn(v[0], v[4]), a1 = __fadd_rn(v[1], v[5]);
  const float a2 = __fadd_rn(v[2], v[6]), a3 = __fadd_rn(v[3], v[7]);
  return __fadd_rn(__fadd_rn(a0, a2), __fadd_rn(a1, a3));
}

// Canonical levels 8, 4, 2, 1 over lane bits 3..0 for the thread's eight
// tokens (p[i] = partial of token tl + 16 i).  Returns the full sum of token
// tl + 16 (4 b3 + 2 b2 + b1), b = lane bits; lanes differing in bit 0 agree.
__device__ __forceinline__ float row_tree(const float* p, int lane) {
  const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  float q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b3 ? p[i + 4] : p[i], send = b3 ? p[i] : p[i + 4];
    q[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 8));
  }
  float q2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b2 ? q[i + 2] : q[i], send = b2 ? q[i] : q[i + 2];
    q2[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 4));
  }
  const float q3 = __fadd_rn(b1 ? q2[1] : q2[0], __shfl_xor_sync(kFull, b1 ? q2[0] : q2[1], 2));
  return __fadd_rn(q3, __shfl_xor_sync(kFull, q3, 1));
}
// Lane holding row_tree's result for the thread's token index i.
__device__ __forceinline__ int row_owner(int lane, int i) {
  return (lane & 16) | (((i >> 2) & 1) << 3) | (((i >> 1) & 1) << 2) | ((i & 1) << 1);
}
// Same recursive halving for a minimum and a maximum (order-free).
__device__ __forceinline__ void row_minmax(const float* mn8, const float* mx8, int lane, float& mn, float& mx) {
  const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  float a[4], b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[i] = fminf(b3 ? mn8[i + 4] : mn8[i], __shfl_xor_sync(kFull, b3 ? mn8[i] : mn8[i + 4], 8));
    b[i] = fmaxf(b3 ? mx8[i + 4] : mx8[i], __shfl_xor_sync(kFull, b3 ? mx8[i] : mx8[i + 4], 8));
  }
  float a2[2], b2v[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    a2[i] = fminf(b2 ? a[i + 2] : a[i], __shfl_xor_sync(kFull, b2 ? a[i] : a[i + 2], 4));
    b2v[i] = fmaxf(b2 ? b[i + 2] : b[i], __shfl_xor_sync(kFull, b2 ? b[i] : b[i + 2], 4));
  }
  float a3 = fminf(b1 ? a2[1] : a2[0], __shfl_xor_sync(kFull, b1 ? a2[0] : a2[1], 2));
  float b3v = fmaxf(b1 ? b2v[1] : b2v[0], __shfl_xor_sync(kFull, b1 ? b2v[0] : b2v[1], 2));
  mn = fminf(a3, __shfl_xor_sync(kFull, a3, 1));
  mx = fmaxf(b3v, __shfl_xor_sync(kFull, b3v, 1));
}
// Canonical levels 8, 4, 2, 1 over the 16 partials of one channel (row i of
// part = t_lo i).
__device__ __forceinline__ float col_tree(const float* part, int d) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = part[i * kKvYS + d];
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
    for (int i = 0; i < off; ++i) v[i] = __fadd_rn(v[i], v[i + off]);
  return v[0];
}

// code = clamp(rint(x / s), 0, steps) for x >= 0 (x = y - min); s == 0 gives 0.
__device__ __forceinline__ uint32_t rtn_code(float x, const QDiv& q, float steps) {
  if (q.s == 0.0f) return 0u;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it leaves rint(v) in the low bits
  const uint32_t lo = __float_as_uint(__fadd_rn(__fmul_rn(x, q.rlo), kMagic));
  const uint32_t hi = __float_as_uint(__fadd_rn(__fmul_rn(x, q.rhi), kMagic));
  if (q.fast && lo == hi && lo - 0x4B400000u <= static_cast<uint32_t>(steps)) return lo & 0xFFu;
  const float qv = fminf(fmaxf(rintf(__fdiv_rn(x, q.s)), 0.0f), steps);
  return static_cast<uint32_t>(__float2int_rn(qv));
}

// tree8 of two interleaved lines at once (component-wise).
__device__ __forceinline__ float2 tree8x2(const float2* v) {
  const float2 a0 = add2(v[0], v[4]), a1 = add2(v[1], v[5]);
  const float2 a2 = add2(v[2], v[6]), a3 = add2(v[3], v[7]);
  return add2(add2(a0, a2), add2(a1, a3));
}
// rtn_code of two values with their own divisors: the two products and the
// two magic-number additions are packed; the checks are per value.
__device__ __forceinline__ uint32_t rtn_finish(float x, const QDiv& q, float steps, uint32_t lo, uint32_t hi) {
  if (q.s == 0.0f) return 0u;
  if (q.fast && lo == hi && lo - 0x4B400000u <= static_cast<uint32_t>(steps)) return lo & 0xFFu;
  const float qv = fminf(fmaxf(rintf(__fdiv_rn(x, q.s)), 0.0f), steps);
  return static_cast<uint32_t>(__float2int_rn(qv));
}
__device__ __forceinline__ void rtn_code2(float2 x, const QDiv& qa, const QDiv& qb, float steps, float2 z, uint32_t& ca,
                                          uint32_t& cb) {
  const float2 magic = dup2(12582912.0f);  // 1.5 * 2^23, as in rtn_code
  const float2 lo = add2(mul2z(x, make_float2(qa.rlo, qb.rlo), z), magic);
  const float2 hi = add2(mul2z(x, make_float2(qa.rhi, qb.rhi), z), magic);
  ca = rtn_finish(x.x, qa, steps, __float_as_uint(lo.x), __float_as_uint(hi.x));
  cb = rtn_finish(x.y, qb, steps, __float_as_uint(lo.y), __float_as_uint(hi.y));
}

// TAIL = false: tile blockIdx.x is batch rows 128 x .. 128 x + 127 of k / v.
// TAIL = true (kvq_kvarn_append): CTA blockIdx.x looks at batch token x; when
// that token filled the last row of its tile (slot % 128 == 127), the tile is
// the 128 rows of its sequence's tail, written to the token's page.
template <typename T, bool TAIL>
__global__ void __launch_bounds__(kKvThreads, 2) kvarn_write_kernel(WriteArgs a) {
  extern __shared__ __align__(16) unsigned char kv_smem[];
  KvSmem& sm = *reinterpret_cast<KvSmem*>(kv_smem);
  const int h = blockIdx.y, side = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int D = 128;

  const long long t0 = TAIL ? 0 : (long long)blockIdx.x * kKvTile;
  const T* src;
  int page = 0;
  if constexpr (TAIL) {  // uniform per CTA; argument errors were flagged by the tail copy
    const int slot = __ldg(a.slots + blockIdx.x), seq = __ldg(a.seq_ids + blockIdx.x);
    if (slot < 0 || slot % kKvTile != kKvTile - 1 || slot / kKvTile >= a.num_pages || seq < 0 || seq >= a.num_seqs)
      return;
    page = slot / kKvTile;
    // The call must not also carry rows of another tile of this sequence: the
    // copy would have overwritten rows of this one.  Such a tile is not
    // written, and the error is flagged.
    int other = 0;
    for (long long i = tid; i < a.num_tokens; i += kKvThreads) {
      const int s2 = __ldg(a.slots + i);
      other |= __ldg(a.seq_ids + i) == seq && s2 >= 0 && s2 / kKvTile < a.num_pages && s2 / kKvTile != page;
    }
    if (__syncthreads_or(other)) {
      if (tid == 0 && h == 0 && side == 0) set_error(a.pool, KVQ_DEVERR_PARTIAL_TILE);
      return;
    }
    const size_t side_bytes = (size_t)a.num_seqs * kKvTile * a.Hkv * D * sizeof(T);
    src = reinterpret_cast<const T*>(a.tail + side * side_bytes) + (size_t)seq * kKvTile * a.Hkv * D;
  } else {
    src = static_cast<const T*>(side ? a.v : a.k);
  }
  // This thread's half token (64 channels), loaded before the slot check so
  // that the two memory latencies overlap (rows t0 .. t0 + 127 always exist).
  const int t = tid >> 1, half = tid & 1;
  constexpr int NRAW = 64 * (int)sizeof(T) / 16;
  uint4 raw[NRAW];
  {
    const uint4* row = reinterpret_cast<const uint4*>(src + ((t0 + t) * a.Hkv + h) * D + 64 * half);
#pragma unroll
    for (int k = 0; k < NRAW; ++k) raw[k] = __ldg(row + k);
  }

  if constexpr (!TAIL) {
    // A tile must be 128 consecutive slots starting a page.
    const int s0 = __ldg(a.slots + t0);
    int ok = 1;
    if (tid < kKvTile) ok = (__ldg(a.slots + t0 + tid) == s0 + tid);
    ok = __syncthreads_and(ok && s0 >= 0 && (s0 % kKvTile) == 0 && s0 / kKvTile < a.num_pages);
    if (!ok) {
      if (tid == 0 && h == 0 && side == 0) set_error(a.pool, KVQ_DEVERR_PARTIAL_TILE);
      return;
    }
    page = s0 / kKvTile;
  }
  if (tid < kKvTile) {
    sm.fr[tid] = 1.0f;  // token factors r_t
    sm.fc[tid] = 1.0f;  // channel factors c_d
  }

  // ---- 1. Walsh-Hadamard along channels.  Adjacent channels travel as f32x2
  //      pairs from stage h = 2 on (stage 1 mixes the two halves of a pair).
  {
    float2 v2[32];  // channels 2m, 2m + 1 of this thread's half token
    {
      float v[64];
#pragma unroll
      for (int k = 0; k < NRAW; ++k) widen16<T>(raw[k], v + k * (16 / (int)sizeof(T)));
#pragma unroll
      for (int m = 0; m < 32; ++m) v2[m] = make_float2(__fadd_rn(v[2 * m], v[2 * m + 1]), __fsub_rn(v[2 * m], v[2 * m + 1]));
    }
#pragma unroll
    for (int hp = 1; hp <= 16; hp <<= 1)  // stage h = 2 hp: the butterflies of pairs m and m + hp
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int m = (k / hp) * 2 * hp + k % hp;
        const float2 x = v2[m], y = v2[m + hp];
        v2[m] = add2(x, y);
        v2[m + hp] = sub2(x, y);
      }
    // stage h = 64 between the two halves' lanes, then the fp32 1/sqrt(128):
    // the upper half takes p - v as (-v) + p, the same rounding
    const float2 sg = dup2(half ? -1.0f : 1.0f), c2 = dup2(__int_as_float(0x3DB504F3));
    float* dst = sm.Y + t * kKvYS;
#pragma unroll
    for (int m = 0; m < 32; m += 2) {
      float2 r[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float2 pv = make_float2(__shfl_xor_sync(kFull, v2[m + u].x, 1), __shfl_xor_sync(kFull, v2[m + u].y, 1));
        r[u] = mul2(add2(mul2(v2[m + u], sg), pv), c2);
      }
      *reinterpret_cast<float4*>(dst + kv_ypos(t, 64 * half + 2 * m)) = make_float4(r[0].x, r[0].y, r[1].x, r[1].y);
    }
  }
  __syncthreads();

  // ---- 2. eight alternating std normalisation steps, tokens first.  The
  //      thread's eight tokens travel as f32x2 pairs (tokens tl + 32 i2 and
  //      tl + 32 i2 + 16): per-token work is component-wise, and the per-channel
  //      tree over the eight tokens takes its levels 64 and 32 on the pairs and
  //      its level 16 inside each pair.
  const int dl = lane & 15, tl = (lane >> 4) | (warp << 1);
  // the lane that finishes token tl + 16 rr's sums (lanes 2k and 2k+1 agree)
  const int rr = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
  const float2 nz = dup2(a.neg_zero);
  float2 y[4][8];  // y[i2][j] = (token tl + 32 i2, token tl + 32 i2 + 16), channel dl + 16 j
#pragma unroll
  for (int i2 = 0; i2 < 4; ++i2)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      y[i2][j] = make_float2(sm.Y[(tl + 32 * i2) * kKvYS + kv_ypos(tl, dl + 16 * j)],
                             sm.Y[(tl + 32 * i2 + 16) * kKvYS + kv_ypos(tl, dl + 16 * j)]);
  // Steps alternate tokens, channels, ...; written as four (token, channel)
  // pairs so that no branch joins the two forms of the loop body.
#pragma unroll kKvPairUnroll
  for (int pair = 0; pair < 4; ++pair) {
    {  // per token: sums over channels
      float p[8];
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const float2 sum = tree8x2(y[i2]);
        p[2 * i2] = sum.x;
        p[2 * i2 + 1] = sum.y;
      }
      // each lane's finished token goes to shared memory; the warp's sixteen
      // tokens are its own, so a warp barrier orders the exchange
      const float mine = __fmul_rn(row_tree(p, lane), 0.0078125f);
      if ((lane & 1) == 0) sm.tm[tl * 8 + rr] = mine;
      __syncwarp();
      float m8[8];
      *reinterpret_cast<float4*>(m8) = *reinterpret_cast<const float4*>(sm.tm + tl * 8);
      *reinterpret_cast<float4*>(m8 + 4) = *reinterpret_cast<const float4*>(sm.tm + tl * 8 + 4);
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const float2 mean = make_float2(m8[2 * i2], m8[2 * i2 + 1]);
        float2 d2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 dv = sub2(y[i2][j], mean);
          d2[j] = mul2z(dv, dv, nz);
        }
        const float2 sum = tree8x2(d2);
        p[2 * i2] = sum.x;
        p[2 * i2 + 1] = sum.y;
      }
      float sd = __fsqrt_rn(__fmul_rn(row_tree(p, lane), 0.0078125f));
      float inv = __frcp_rn(sd);
      if (sd < 1e-8f) {  // std below 1e-8: the token stays as it is
        sd = 1.0f;
        inv = 1.0f;
      }
      if ((lane & 1) == 0) {
        sm.fr[tl + 16 * rr] = __fmul_rn(sm.fr[tl + 16 * rr], sd);
        sm.ti[tl * 8 + rr] = inv;
      }
      __syncwarp();
      float i8[8];
      *reinterpret_cast<float4*>(i8) = *reinterpret_cast<const float4*>(sm.ti + tl * 8);
      *reinterpret_cast<float4*>(i8 + 4) = *reinterpret_cast<const float4*>(sm.ti + tl * 8 + 4);
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const float2 iv = make_float2(i8[2 * i2], i8[2 * i2 + 1]);
#pragma unroll
        for (int j = 0; j < 8; ++j) y[i2][j] = mul2z(y[i2][j], iv, nz);
      }
    }
    {  // per channel: sums over tokens; tree8 over tokens i = 2 i2 + e:
       // (v0 + v4, v1 + v5), (v2 + v6, v3 + v7), then their sums, then within
      auto col8 = [](const float2* c) -> float {  // c[i2] = (v[2 i2], v[2 i2 + 1])
        const float2 s = add2(add2(c[0], c[2]), add2(c[1], c[3]));
        return __fadd_rn(s.x, s.y);
      };
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 col[4] = {y[0][j], y[1][j], y[2][j], y[3][j]};
        sm.part[tl * kKvYS + dl + 16 * j] = col8(col);
      }
      __syncthreads();
      if (tid < D) sm.st0[tid] = __fmul_rn(col_tree(sm.part, tid), 0.0078125f);
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 mean = dup2(sm.st0[dl + 16 * j]);
        float2 col[4];
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const float2 dv = sub2(y[i2][j], mean);
          col[i2] = mul2z(dv, dv, nz);
        }
        sm.part[tl * kKvYS + dl + 16 * j] = col8(col);
      }
      __syncthreads();
      if (tid < D) {
        const float sd = __fsqrt_rn(__fmul_rn(col_tree(sm.part, tid), 0.0078125f));
        const bool keep = sd < 1e-8f;  // std below 1e-8: the channel stays as it is
        sm.st1[tid] = keep ? 1.0f : __frcp_rn(sd);
        sm.fc[tid] = __fmul_rn(sm.fc[tid], keep ? 1.0f : sd);
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 iv = dup2(sm.st1[dl + 16 * j]);
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) y[i2][j] = mul2z(y[i2][j], iv, nz);
      }
    }
  }
  // ---- 3. asymmetric round-to-nearest
  uint8_t* blk = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes;
  uint8_t* codes = reinterpret_cast<uint8_t*>(sm.Y);  // [128][kKvCS]; Y is in registers now
  __syncthreads();  // every thread has read its y from sm.Y
  if (side == 0) {  // keys: per channel over the tile's tokens, 4 bits
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float mn = fminf(y[0][j].x, y[0][j].y), mx = fmaxf(y[0][j].x, y[0][j].y);
#pragma unroll
      for (int i2 = 1; i2 < 4; ++i2) {
        mn = fminf(mn, fminf(y[i2][j].x, y[i2][j].y));
        mx = fmaxf(mx, fmaxf(y[i2][j].x, y[i2][j].y));
      }
      sm.part[tl * kKvYS + dl + 16 * j] = mn;
      sm.part2[tl * kKvYS + dl + 16 * j] = mx;
    }
    __syncthreads();
    float* meta = reinterpret_cast<float*>(blk + kKvTile * D / 2 + kKvTile * D / 4);
    if (tid < D) {
      float mn = sm.part[tid], mx = sm.part2[tid];
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        mn = fminf(mn, sm.part[i * kKvYS + tid]);
        mx = fmaxf(mx, sm.part2[i * kKvYS + tid]);
      }
      const float sc = div_const(__fsub_rn(mx, mn), 15.0f, kRcp15);
      sm.st0[tid] = sc;
      sm.st1[tid] = mn;
      st_chk(meta + tid, sc, a.pool_span, a.pool);
      st_chk(meta + D + tid, mn, a.pool_span, a.pool);
      st_chk(meta + 2 * D + tid, sm.fc[tid], a.pool_span, a.pool);
      st_chk(meta + 3 * D + tid, sm.fr[tid], a.pool_span, a.pool);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d = dl + 16 * j;
      const float2 mn = dup2(sm.st1[d]);
      const QDiv q(sm.st0[d]);
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        uint32_t c0, c1;
        rtn_code2(sub2(y[i2][j], mn), q, q, 15.0f, nz, c0, c1);
        codes[(tl + 32 * i2) * kKvCS + d] = static_cast<uint8_t>(c0);
        codes[(tl + 32 * i2 + 16) * kKvCS + d] = static_cast<uint8_t>(c1);
      }
    }
  } else {  // values: per token over the channels, 2 bits
    float mn8[8], mx8[8];
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
      float a0 = y[i2][0].x, a1 = y[i2][0].x, b0 = y[i2][0].y, b1 = y[i2][0].y;
#pragma unroll
      for (int j = 1; j < 8; ++j) {
        a0 = fminf(a0, y[i2][j].x);
        a1 = fmaxf(a1, y[i2][j].x);
        b0 = fminf(b0, y[i2][j].y);
        b1 = fmaxf(b1, y[i2][j].y);
      }
      mn8[2 * i2] = a0; mx8[2 * i2] = a1;
      mn8[2 * i2 + 1] = b0; mx8[2 * i2 + 1] = b1;
    }
    float mn, mx;
    row_minmax(mn8, mx8, lane, mn, mx);
    const float sc = div_const(__fsub_rn(mx, mn), 3.0f, kRcp3);
    float* meta = reinterpret_cast<float*>(blk + kKvTile * D / 2 + kKvTile * D / 4 + 4 * (3 * D + kKvTile));
    if ((lane & 1) == 0) {  // lanes 2k (+16) own token tl + 16 (4 b3 + 2 b2 + b1)
      const int t = tl + 16 * (((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1));
      st_chk(meta + t, sc, a.pool_span, a.pool);
      st_chk(meta + kKvTile + t, mn, a.pool_span, a.pool);
    }
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
      const int sa = row_owner(lane, 2 * i2), sb = row_owner(lane, 2 * i2 + 1);
      const float2 mni = make_float2(__shfl_sync(kFull, mn, sa), __shfl_sync(kFull, mn, sb));
      const QDiv qa(__shfl_sync(kFull, sc, sa)), qb(__shfl_sync(kFull, sc, sb));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t c0, c1;
        rtn_code2(sub2(y[i2][j], mni), qa, qb, 3.0f, nz, c0, c1);
        codes[(tl + 32 * i2) * kKvCS + dl + 16 * j] = static_cast<uint8_t>(c0);
        codes[(tl + 32 * i2 + 16) * kKvCS + dl + 16 * j] = static_cast<uint8_t>(c1);
      }
    }
    if (tid < kKvTile) {
      st_chk(meta + 2 * kKvTile + tid, sm.fr[tid], a.pool_span, a.pool);
      st_chk(meta + 3 * kKvTile + tid, sm.fc[tid], a.pool_span, a.pool);
    }
  }
  __syncthreads();

  // ---- pack the code bytes and store 16-byte rows
  if (side == 0) {  // [128][64]: even channel in the low nibble; 32 codes per chunk
    uint8_t* pay = blk;
    for (int c = tid; c < kKvTile * 4; c += kKvThreads) {
      const int t = c >> 2, k0 = (c & 3) * 32;
      const uint4 u0 = *reinterpret_cast<const uint4*>(codes + t * kKvCS + k0);
      const uint4 u1 = *reinterpret_cast<const uint4*>(codes + t * kKvCS + k0 + 16);
      const uint32_t in[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      uint32_t out[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t x0 = in[2 * q] | (in[2 * q] >> 4), x1 = in[2 * q + 1] | (in[2 * q + 1] >> 4);
        out[q] = prmt(x0, x1, 0x6420u);  // bytes 0, 2 of each: (c0 | c1 << 4), (c2 | c3 << 4)
      }
      st_chk(reinterpret_cast<uint4*>(pay + t * 64 + (c & 3) * 16), make_uint4(out[0], out[1], out[2], out[3]), a.pool_span,
             a.pool);
    }
  } else {  // [128][32]: element 4i + j in bits 2j..2j+1; 64 codes per chunk
    uint8_t* pay = blk + kKvTile * D / 2;
    const int t = tid >> 1, k0 = (tid & 1) * 64;
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = *reinterpret_cast<const uint4*>(codes + t * kKvCS + k0 + 16 * q);
      const uint32_t in[4] = {u.x, u.y, u.z, u.w};
      uint32_t b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) b[e] = (in[e] | (in[e] >> 6) | (in[e] >> 12) | (in[e] >> 18)) & 0xFFu;
      out[q] = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    }
    st_chk(reinterpret_cast<uint4*>(pay + t * 32 + (tid & 1) * 16), make_uint4(out[0], out[1], out[2], out[3]), a.pool_span,
           a.pool);
  }
}

// ------------------------------------------------------------------ debug self-test
// A store at pool byte 41 against the span [40, 41): outside it, so a debug
// build skips it and flags KVQ_DEVERR_BOUNDS (byte 41 is inside the header,
// unused, so even a missing check could not touch anything but that byte).
__global__ void bounds_selftest_kernel(uint8_t* pool) {
  const Span s{pool + 40, pool + 41};
  st_chk(pool + 41, static_cast<uint8_t>(0x5A), s, pool);
}

// ------------------------------------------------------------------ scales
template <typename T>
__global__ void __launch_bounds__(256) amax_kernel(const T* x, size_t n, uint32_t* out) {
  float m = 0.0f;
  constexpr int VEC = 16 / sizeof(T);
  const size_t nvec = n / VEC;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    float f[VEC];
    load16<T>(x + i * VEC, f);
#pragma unroll
    for (int e = 0; e < VEC; ++e) m = fmaxf(m, fabsf(f[e]));
  }
  for (size_t i = nvec * VEC + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    m = fmaxf(m, fabsf(static_cast<float>(x[i])));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));  // m >= 0: bit order is value order
}

__global__ void scales_from_amax_kernel(uint8_t* pool, const float* ak, const float* av, float div) {
  const float a0 = *ak, a1 = *av;
  *reinterpret_cast<float*>(pool + kHdrKScaleOffset) = a0 > 0.0f ? __fdiv_rn(a0, div) : 1.0f;
  *reinterpret_cast<float*>(pool + kHdrVScaleOffset) = a1 > 0.0f ? __fdiv_rn(a1, div) : 1.0f;
}

template <int MODE, typename T, int D>
cudaError_t launch_rows(const WriteArgs& a, cudaStream_t s) {
  constexpr int TOK = 256 / (D / (16 / sizeof(T))) * kRowsPerThread;
  const long long blocks = (a.num_tokens + TOK - 1) / TOK;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL || a.Hkv > 65535) return cudaErrorInvalidValue;
  write_rows_kernel<MODE, T, D><<<dim3(static_cast<unsigned>(blocks), a.Hkv, 2), 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_mode(int mode, const WriteArgs& a, cudaStream_t s) {
  switch (mode) {
    case KVQ_FP8_PER_TENSOR: return launch_rows<KVQ_FP8_PER_TENSOR, T, D>(a, s);
    case KVQ_INT8_PER_TOKEN_HEAD: return launch_rows<KVQ_INT8_PER_TOKEN_HEAD, T, D>(a, s);
    case KVQ_FP8_PER_TOKEN_HEAD: return launch_rows<KVQ_FP8_PER_TOKEN_HEAD, T, D>(a, s);
    case KVQ_NVFP4: return launch_rows<KVQ_NVFP4, T, D>(a, s);
    case KVQ_INT4_PER_TOKEN_HEAD: return launch_rows<KVQ_INT4_PER_TOKEN_HEAD, T, D>(a, s);
    case KVQ_NVFP4_4OVER6: return launch_rows<KVQ_NVFP4_4OVER6, T, D>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, bool TAIL>
cudaError_t launch_kvarn(const WriteArgs& a, cudaStream_t s) {
  const long long tiles = TAIL ? a.num_tokens : a.num_tokens / kKvTile;
  if (tiles == 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL || a.Hkv > 65535) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kvarn_write_kernel<T, TAIL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kKvSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(tiles), a.Hkv, 2);
  kvarn_write_kernel<T, TAIL><<<grid, kKvThreads, kKvSmem, s>>>(a);
  return cudaGetLastError();
}

// KVarN open tiles: token i's K and V rows (16 bytes per thread) go to row
// slot % 128 of sequence seq_ids[i]'s tail.  A negative slot skips the token;
// a slot past the pool or a sequence id outside [0, num_seqs) skips it and
// sets its error bit.
template <typename T>
__global__ void __launch_bounds__(256) kvarn_tail_copy_kernel(WriteArgs a) {
  constexpr int D = 128, CH = D * (int)sizeof(T) / 16;  // 16-byte chunks per row
  const long long n = a.num_tokens * a.Hkv * 2 * CH;
  const size_t side_bytes = (size_t)a.num_seqs * kKvTile * a.Hkv * D * sizeof(T);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx % CH);
    const long long r = idx / CH;
    const int side = (int)(r % 2);
    const long long th = r / 2;
    const int h = (int)(th % a.Hkv);
    const long long i = th / a.Hkv;
    const int slot = __ldg(a.slots + i), seq = __ldg(a.seq_ids + i);
    if (slot < 0) continue;
    if (slot / kKvTile >= a.num_pages) {
      if (c == 0 && h == 0 && side == 0) set_error(a.pool, KVQ_DEVERR_SLOT_RANGE);
      continue;
    }
    if (seq < 0 || seq >= a.num_seqs) {
      if (c == 0 && h == 0 && side == 0) set_error(a.pool, KVQ_DEVERR_SEQ_ID);
      continue;
    }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(side ? a.v : a.k) +
                                                         (i * a.Hkv + h) * D) + c);
    uint4* dst = reinterpret_cast<uint4*>(a.tail + side * side_bytes +
                                          ((((size_t)seq * kKvTile + slot % kKvTile) * a.Hkv + h) * D) * sizeof(T));
    st_chk(dst + c, v, a.tail_span, a.pool);
  }
}

template <typename T>
cudaError_t launch_kvarn_tail(const WriteArgs& a, cudaStream_t s) {
  const long long chunks = a.num_tokens * a.Hkv * 2 * (128 * (long long)sizeof(T) / 16);
  long long blocks = (chunks + 255) / 256;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) return cudaSuccess;
  kvarn_tail_copy_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_kvarn<T, true>(a, s);
}

}  // namespace

// The span of the pool's (page, kv head) blocks: every store a write kernel makes.
Span pool_blocks(const kvq_cache* c) {
  uint8_t* lo = c->base + kHeaderBytes;
  return Span{lo, lo + (size_t)c->cfg.num_pages * c->cfg.num_kv_heads * c->block_bytes};
}

cudaError_t launch_write(const kvq_cache* c, const void* k, const void* v, const int32_t* slots, int num_tokens,
                         cudaStream_t stream) {
  WriteArgs a;
  a.pool = c->base;
  a.k = k;
  a.v = v;
  a.slots = slots;
  a.num_tokens = num_tokens;
  a.Hkv = c->cfg.num_kv_heads;
  a.P = c->cfg.page_size;
  a.log2P = 0;
  while ((1 << a.log2P) < a.P) ++a.log2P;  // page sizes are powers of two
  a.num_pages = c->cfg.num_pages;
  a.block_bytes = c->block_bytes;
  const int mode = c->cfg.mode, D = c->cfg.head_dim;
  const bool f16 = c->cfg.io_dtype == KVQ_F16;
  a.seq_ids = nullptr;
  a.tail = nullptr;
  a.num_seqs = 0;
  a.pool_span = pool_blocks(c);
  a.tail_span = Span{nullptr, nullptr};
  if (mode == KVQ_KVARN_K4V2_G128)
    return f16 ? launch_kvarn<__half, false>(a, stream) : launch_kvarn<float, false>(a, stream);
  if (D == 128) return f16 ? launch_mode<__half, 128>(mode, a, stream) : launch_mode<float, 128>(mode, a, stream);
  if (D == 32) return f16 ? launch_mode<__half, 32>(mode, a, stream) : launch_mode<float, 32>(mode, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_kvarn_append(const kvq_cache* c, const void* k, const void* v, const int32_t* slots,
                                const int32_t* seq_ids, int num_tokens, void* tail, int num_seqs,
                                cudaStream_t stream) {
  WriteArgs a;
  a.pool = c->base;
  a.k = k;
  a.v = v;
  a.slots = slots;
  a.num_tokens = num_tokens;
  a.Hkv = c->cfg.num_kv_heads;
  a.P = c->cfg.page_size;
  a.log2P = 7;
  a.num_pages = c->cfg.num_pages;
  a.block_bytes = c->block_bytes;
  a.seq_ids = seq_ids;
  a.tail = static_cast<uint8_t*>(tail);
  a.num_seqs = num_seqs;
  a.pool_span = pool_blocks(c);
  const size_t esz = c->cfg.io_dtype == KVQ_F16 ? 2 : 4;
  a.tail_span = Span{a.tail, a.tail + (size_t)2 * num_seqs * 128 * a.Hkv * c->cfg.head_dim * esz};
  return c->cfg.io_dtype == KVQ_F16 ? launch_kvarn_tail<__half>(a, stream) : launch_kvarn_tail<float>(a, stream);
}

cudaError_t launch_bounds_selftest(uint8_t* pool, cudaStream_t stream) {
  bounds_selftest_kernel<<<1, 1, 0, stream>>>(pool);
  return cudaGetLastError();
}

cudaError_t launch_amax(const void* x, int dtype, size_t n, float* out, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), stream);
  if (e != cudaSuccess || n == 0) return e;
  const int vec = dtype == KVQ_F16 ? 8 : 4;
  size_t blocks = (n / vec + 255) / 256;
  const size_t cap = (size_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  if (dtype == KVQ_F16)
    amax_kernel<__half><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const __half*>(x), n,
                                                              reinterpret_cast<uint32_t*>(out));
  else
    amax_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const float*>(x), n,
                                                             reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_scales_from_amax(uint8_t* pool, const float* ak, const float* av, float div,
                                   cudaStream_t stream) {
  scales_from_amax_kernel<<<1, 1, 0, stream>>>(pool, ak, av, div);
  return cudaGetLastError();
}

}  // namespace kvq
