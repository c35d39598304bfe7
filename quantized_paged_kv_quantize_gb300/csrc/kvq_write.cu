// kvq_write.cu -- quantize-on-write kernels and per-tensor scale setup.
//
// Compiled with -fmad=false and written with explicit _rn intrinsics so every
// fp32 operation is individually rounded: the quantized bytes and scales are
// bit-identical to the specification.
//
// Sources (web pages, by title and section):
//  "KV Cache 量化深度解析：Per-Tensor、Per-Token-Head 与 NVFP4", sec. 2.1-2.3;
//  "KV Cache 量化 · LLM Glossary", first section (s = max|x|/127, q = clip(round(x/s)));
//  "KV 量化" (rustineverything.app), 写和读 (divide by the scale, cast, store as uint8);
//  "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化", 双层缩放 (q = Q_E2M1(x/(s_t s_b))),
//     KV 的写入与读取路径 (compute scales, round and clip to E2M1, pack two per byte);
//  "KVarN：华为推出的原生 vLLM KV-cache 量化后端...", 技术原理 (tile, Hadamard rotation,
//     alternating std normalisation, asymmetric RTN) and 配置与部署 (k4v2, tile 128).
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

template <int N>
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint32_t* w);
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

// Encoding of the IEEE quotient RN(x/s) without a division on the common path.
// With r = RN(1/s), rlo = RN(r(1 - 2^-20)) and rhi = RN(r(1 + 2^-20)), the
// products RN(x rlo) and RN(x rhi) enclose RN(x/s): their relative distance to
// x/s is at least 16u - 3u (u = 2^-24) on each side, while RN(x/s) is within u
// of it.  Every encoder used here (round-to-nearest-even onto a grid, with
// saturation) is monotone, so when both ends encode to the same code, that is
// the code of RN(x/s); when they differ the quotient is computed exactly.
// Scales whose reciprocal is not a comfortable normal number always divide.
struct QDiv {
  float s, rlo, rhi;
  bool fast;
  __device__ __forceinline__ explicit QDiv(float s_) : s(s_) {
    const float r = __frcp_rn(s_);
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
  __device__ __forceinline__ uint32_t int8x4(const float* x) const {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    uint32_t lo[4], bad = fast ? 0u : 1u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo[e] = __float_as_uint(__fadd_rn(__fmul_rn(x[e], rlo), kMagic));
      const uint32_t hi = __float_as_uint(__fadd_rn(__fmul_rn(x[e], rhi), kMagic));
      bad |= (lo[e] ^ hi) | static_cast<uint32_t>(lo[e] - 0x4B3FFF81u > 254u);
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

// One (token, kv head, side) row of D values per group of TPR threads; each
// thread converts VEC = 16 bytes of input.  Grid: (token blocks, kv head,
// side), so no index needs a division; a block's consecutive tokens land in
// consecutive rows of the same pages.  Modes 1-4.
template <int MODE, typename T, int D>
__global__ void __launch_bounds__(256) write_rows_kernel(WriteArgs a) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int TPR = D / VEC;
  constexpr int TOK = 256 / TPR;  // tokens per block
  static_assert(TPR >= 2 && TPR <= 32 && (TPR & (TPR - 1)) == 0, "row group");
  const int h = blockIdx.y, side = blockIdx.z;
  const long long token = (long long)blockIdx.x * TOK + threadIdx.x / TPR;
  const int j = threadIdx.x % TPR;

  bool active = token < a.num_tokens;
  int slot = active ? __ldg(a.slots + token) : -1;
  active = active && slot >= 0;
  const int page = slot >> a.log2P;
  const int off = slot & (a.P - 1);
  if (active && page >= a.num_pages) {
    if (j == 0) set_error(a.pool, KVQ_DEVERR_SLOT_RANGE);
    active = false;
  }
  const long long r = token * a.Hkv + h;  // (token, head) row of the input

  float x[VEC];
  if (active) {
    const T* src = static_cast<const T*>(side ? a.v : a.k) + r * D + j * VEC;
    load16<T>(src, x);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) x[i] = 0.0f;
  }
  uint8_t* blk = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes;

  if constexpr (MODE == KVQ_FP8_PER_TENSOR) {
    const QDiv q(*reinterpret_cast<const float*>(a.pool + (side ? kHdrVScaleOffset : kHdrKScaleOffset)));
    uint32_t w[VEC / 4];
#pragma unroll
    for (int i = 0; i < VEC; i += 4) w[i / 4] = q.e4m3x2(x[i + 1], x[i]) | (q.e4m3x2(x[i + 3], x[i + 2]) << 16);
    if (active) store_bytes<VEC>(blk + (size_t)side * a.P * D + (size_t)off * D + j * VEC, w);
  } else if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD || MODE == KVQ_FP8_PER_TOKEN_HEAD) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = group_max<TPR>(amax);
    const float s = __fdiv_rn(fmaxf(amax, 1e-8f), MODE == KVQ_INT8_PER_TOKEN_HEAD ? 127.0f : 448.0f);
    const QDiv q(s);
    uint32_t w[VEC / 4];
#pragma unroll
    for (int i = 0; i < VEC; i += 4) {
      if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD) {
        w[i / 4] = q.int8x4(x + i);
      } else {
        w[i / 4] = q.e4m3x2(x[i + 1], x[i]) | (q.e4m3x2(x[i + 3], x[i + 2]) << 16);
      }
    }
    if (active) {
      store_bytes<VEC>(blk + (size_t)side * a.P * D + (size_t)off * D + j * VEC, w);
      if (j == 0) *reinterpret_cast<float*>(blk + (size_t)2 * a.P * D + (size_t)side * 4 * a.P + 4 * off) = s;
    }
  } else if constexpr (MODE == KVQ_NVFP4) {
    constexpr int TPB = 16 / VEC;  // threads per 16-value block
    const float st = *reinterpret_cast<const float*>(a.pool + (side ? kHdrVScaleOffset : kHdrKScaleOffset));
    const float six_st = __fmul_rn(6.0f, st);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = group_max<TPB>(amax);
    const uint32_t sb = f32x2_to_e4m3x2(0.0f, __fdiv_rn(amax, six_st)) & 0xFFu;
    const float sbf = e4m3_to_f32(sb);
    const float den = __fmul_rn(st, sbf);
    uint32_t w[1] = {0u};
    if (sbf != 0.0f) w[0] = QDiv(den).e2m1x8<VEC>(x);
    if (active) {
      store_bytes<VEC / 2>(blk + (size_t)side * a.P * D / 2 + (size_t)off * D / 2 + j * VEC / 2, w);
      if ((j % TPB) == 0)
        blk[(size_t)a.P * D + (size_t)side * a.P * D / 16 + (size_t)off * D / 16 + (j * VEC) / 16] =
            static_cast<uint8_t>(sb);
    }
  }
}

// ------------------------------------------------------------------ KVarN
// One CTA per (128-token tile, kv head, side).  The tile is held in shared
// memory as Y[token][channel] (row stride 129 floats: both row-wise and
// column-wise warp accesses are bank-conflict free).
constexpr int kKvTile = 128;
constexpr int kKvStride = 129;
constexpr int kKvThreads = 256;
constexpr size_t kKvSmem = sizeof(float) * (kKvTile * kKvStride + 4 * kKvTile) + kKvTile * kKvTile;

// Canonical 128-sum: lane l holds elements l, l+32, l+64, l+96; the pairwise
// tree adds v[i] + v[i+off] for off = 64, 32 (in thread) then 16 .. 1 (lanes).
__device__ __forceinline__ float tree_sum128(const float* v) {
  float s = __fadd_rn(__fadd_rn(v[0], v[2]), __fadd_rn(v[1], v[3]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(kFull, s, o));
  return s;
}

template <typename T>
__global__ void __launch_bounds__(kKvThreads) kvarn_write_kernel(WriteArgs a) {
  extern __shared__ __align__(16) unsigned char kv_smem[];
  float* Y = reinterpret_cast<float*>(kv_smem);
  float* fac_r = Y + kKvTile * kKvStride;  // per-token factor r_t
  float* fac_c = fac_r + kKvTile;          // per-channel factor c_d
  float* qscale = fac_c + kKvTile;         // RTN scale (K: per channel, V: per token)
  float* qzero = qscale + kKvTile;         // RTN zero (minimum)
  uint8_t* codes = reinterpret_cast<uint8_t*>(qzero + kKvTile);  // [128][128]

  const int tile = blockIdx.x, h = blockIdx.y, side = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int D = 128;

  // A tile must be 128 consecutive slots starting a page.
  const long long t0 = (long long)tile * kKvTile;
  const int s0 = __ldg(a.slots + t0);
  int ok = 1;
  if (tid < kKvTile) ok = (__ldg(a.slots + t0 + tid) == s0 + tid);
  ok = __syncthreads_and(ok && s0 >= 0 && (s0 % kKvTile) == 0 && s0 / kKvTile < a.num_pages);
  if (!ok) {
    if (tid == 0 && h == 0 && side == 0) set_error(a.pool, KVQ_DEVERR_PARTIAL_TILE);
    return;
  }
  const int page = s0 / kKvTile;
  if (tid < kKvTile) { fac_r[tid] = 1.0f; fac_c[tid] = 1.0f; }

  // Stage 1-2: load each token's 128 channels (lane holds d = 4l..4l+3),
  // Walsh-Hadamard butterflies h = 1, 2 (in thread), 4 .. 64 (lanes), then
  // the 1/sqrt(128) normalisation (fp32 0x3DB504F3).
  const T* src = static_cast<const T*>(side ? a.v : a.k);
  const float inv_sqrt128 = __int_as_float(0x3DB504F3);
  for (int t = warp; t < kKvTile; t += kKvThreads / 32) {
    const T* row = src + ((t0 + t) * a.Hkv + h) * D + 4 * lane;
    float v[4];
    if constexpr (sizeof(T) == 2) {
      uint2 u = __ldg(reinterpret_cast<const uint2*>(row));
      float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      v[0] = p0.x; v[1] = p0.y; v[2] = p1.x; v[3] = p1.y;
    } else {
      float4 u = __ldg(reinterpret_cast<const float4*>(row));
      v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    float w0 = __fadd_rn(v[0], v[1]), w1 = __fsub_rn(v[0], v[1]);
    float w2 = __fadd_rn(v[2], v[3]), w3 = __fsub_rn(v[2], v[3]);
    v[0] = __fadd_rn(w0, w2); v[2] = __fsub_rn(w0, w2);
    v[1] = __fadd_rn(w1, w3); v[3] = __fsub_rn(w1, w3);
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __shfl_xor_sync(kFull, v[i], o);
        v[i] = upper ? __fsub_rn(p, v[i]) : __fadd_rn(v[i], p);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) Y[t * kKvStride + 4 * lane + i] = __fmul_rn(v[i], inv_sqrt128);
  }
  __syncthreads();

  // Stage 3: eight alternating std normalisation steps, tokens first.
  for (int step = 0; step < 8; ++step) {
    const bool per_token = (step & 1) == 0;
    for (int L = warp; L < kKvTile; L += kKvThreads / 32) {
      float v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        v[m] = per_token ? Y[L * kKvStride + lane + 32 * m] : Y[(lane + 32 * m) * kKvStride + L];
      const float mean = __fmul_rn(tree_sum128(v), 0.0078125f);
      float sq[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float d = __fsub_rn(v[m], mean);
        sq[m] = __fmul_rn(d, d);
      }
      const float var = __fmul_rn(tree_sum128(sq), 0.0078125f);
      const float sd = __fsqrt_rn(var);
      if (!(sd < 1e-8f)) {
        const float inv = __frcp_rn(sd);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float y = __fmul_rn(v[m], inv);
          if (per_token) Y[L * kKvStride + lane + 32 * m] = y;
          else Y[(lane + 32 * m) * kKvStride + L] = y;
        }
        if (lane == 0) {
          if (per_token) fac_r[L] = __fmul_rn(fac_r[L], sd);
          else fac_c[L] = __fmul_rn(fac_c[L], sd);
        }
      }
    }
    __syncthreads();
  }

  // Stage 4: asymmetric round-to-nearest.  K: per channel over the tile's
  // tokens, 4 bits; V: per token over the channels, 2 bits.
  {
    const bool by_channel = side == 0;
    const float steps = by_channel ? 15.0f : 3.0f;
    for (int L = warp; L < kKvTile; L += kKvThreads / 32) {
      float v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        v[m] = by_channel ? Y[(lane + 32 * m) * kKvStride + L] : Y[L * kKvStride + lane + 32 * m];
      float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
      float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      }
      const float sc = __fdiv_rn(__fsub_rn(mx, mn), steps);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float qv = 0.0f;
        if (sc != 0.0f) {
          qv = rintf(__fdiv_rn(__fsub_rn(v[m], mn), sc));
          qv = fminf(fmaxf(qv, 0.0f), steps);
        }
        const int e = lane + 32 * m;
        codes[by_channel ? e * kKvTile + L : L * kKvTile + e] = static_cast<uint8_t>(__float2int_rn(qv));
      }
      if (lane == 0) { qscale[L] = sc; qzero[L] = mn; }
    }
  }
  __syncthreads();

  // Pack and store payload + metadata of this side.
  uint8_t* blk = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes;
  if (side == 0) {
    uint8_t* pay = blk;  // [128][64]: even channel in the low nibble
    for (int c = tid; c < kKvTile * 4; c += kKvThreads) {  // 16-byte chunks: 32 channels of one token
      const int t = c >> 2, k0 = (c & 3) * 32;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int d = k0 + 8 * q + 2 * b;
          word |= (uint32_t)(codes[t * kKvTile + d] | (codes[t * kKvTile + d + 1] << 4)) << (8 * b);
        }
        w[q] = word;
      }
      *reinterpret_cast<uint4*>(pay + t * 64 + (c & 3) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    float* meta = reinterpret_cast<float*>(blk + kKvTile * D / 2 + kKvTile * D / 4);
    if (tid < kKvTile) {
      meta[tid] = qscale[tid];
      meta[D + tid] = qzero[tid];
      meta[2 * D + tid] = fac_c[tid];
      meta[3 * D + tid] = fac_r[tid];
    }
  } else {
    uint8_t* pay = blk + kKvTile * D / 2;  // [128][32]: element 4i+j in bits 2j..2j+1
    for (int c = tid; c < kKvTile * 2; c += kKvThreads) {  // 16-byte chunks: 64 channels of one token
      const int t = c >> 1, k0 = (c & 1) * 64;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int d = k0 + 16 * q + 4 * b;
          const uint8_t* cp = codes + t * kKvTile + d;
          word |= (uint32_t)(cp[0] | (cp[1] << 2) | (cp[2] << 4) | (cp[3] << 6)) << (8 * b);
        }
        w[q] = word;
      }
      *reinterpret_cast<uint4*>(pay + t * 32 + (c & 1) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    float* meta = reinterpret_cast<float*>(blk + kKvTile * D / 2 + kKvTile * D / 4 + 4 * (3 * D + kKvTile));
    if (tid < kKvTile) {
      meta[tid] = qscale[tid];
      meta[kKvTile + tid] = qzero[tid];
      meta[2 * kKvTile + tid] = fac_r[tid];
      meta[3 * kKvTile + tid] = fac_c[tid];
    }
  }
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
  constexpr int TOK = 256 / (D / (16 / sizeof(T)));
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
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_kvarn(const WriteArgs& a, cudaStream_t s) {
  const long long tiles = a.num_tokens / kKvTile;
  if (tiles == 0) return cudaSuccess;
  static bool attr_set = false;  // one attribute per instantiation, set before first launch
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kvarn_write_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kKvSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(static_cast<unsigned>(tiles), a.Hkv, 2);
  kvarn_write_kernel<T><<<grid, kKvThreads, kKvSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

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
  if (mode == KVQ_KVARN_K4V2_G128)
    return f16 ? launch_kvarn<__half>(a, stream) : launch_kvarn<float>(a, stream);
  if (D == 128) return f16 ? launch_mode<__half, 128>(mode, a, stream) : launch_mode<float, 128>(mode, a, stream);
  if (D == 32) return f16 ? launch_mode<__half, 32>(mode, a, stream) : launch_mode<float, 32>(mode, a, stream);
  return cudaErrorInvalidValue;
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
