// kvq_stats.cu -- tensor-level quantization error of the rows a pool holds
// against the rows they were written from (kvq_tensor_error_stats).
//
// Source: "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化", 量化误差该怎样测, 张量层:
// record MSE and normalised MSE, max absolute error, cosine similarity, zero
// ratio, clipping / saturation ratio and the scale distribution, per head, K
// and V apart.  The dequantization follows the pool layout of kvq.h (the same
// values the decode kernels use): codes times their scales, KVarN rows
// r_t c_d (scale q + zero) rotated back by the normalised Walsh-Hadamard
// transform.  Diagnostic only, not on the decode path.
//
// Grid: (blocks, kv head, side); each warp takes one token row at a time (D/32
// values per lane), accumulates in registers (fp64), and the block merges its
// warps in shared memory before one set of global atomics.
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kWarps = 8;

struct StatsArgs {
  const uint8_t* pool;
  const void* k;
  const void* v;
  const int32_t* slots;
  long long num_tokens;
  int Hkv, P, D, num_pages, mode, f32io;
  size_t block_bytes;
  kvq_error_stats* out;  // [2][Hkv]
};

__device__ __forceinline__ float e4m3_val(uint32_t byte) { return e4m3_to_f32(byte); }
__device__ __forceinline__ float e2m1_val(uint32_t nib) {
  const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  const float m = mag[nib & 7];
  return (nib & 8) ? -m : m;
}
__device__ __forceinline__ int scale_bin(float s) {
  if (!(s > 0.0f)) return 0;
  if (!(s <= 3.4e38f)) return 63;
  int e = 0;
  (void)frexpf(s, &e);  // s = m 2^e, m in [0.5, 1): floor(log2 s) = e - 1
  const int b = e - 1 + 32;
  return b < 0 ? 0 : (b > 63 ? 63 : b);
}

// Normalised Walsh-Hadamard transform of a 128-vector held as 4 consecutive
// values per lane (lane l: elements 4l .. 4l+3); it is its own inverse.
__device__ __forceinline__ void fwht128(float* v, int lane) {
  float w0 = v[0] + v[1], w1 = v[0] - v[1], w2 = v[2] + v[3], w3 = v[2] - v[3];
  v[0] = w0 + w2; v[2] = w0 - w2; v[1] = w1 + w3; v[3] = w1 - w3;
#pragma unroll
  for (int o = 1; o <= 16; o <<= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __shfl_xor_sync(kFull, v[i], o);
      v[i] = upper ? p - v[i] : v[i] + p;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= 0.08838834764831845f;
}

struct Acc {
  double n = 0, se = 0, sr = 0, sd = 0, dot = 0, mx = 0, zeros = 0, sat = 0, clip = 0;
  // clipped: saturated, and the input beyond the top grid value by more than
  // half the grid's last step (margin), i.e. farther than rounding would put it
  __device__ void add(double x, double xh, bool saturated, double margin) {
    const double e = xh - x;
    n += 1.0;
    se += e * e;
    sr += x * x;
    sd += xh * xh;
    dot += x * xh;
    mx = fmax(mx, fabs(e));
    zeros += xh == 0.0 ? 1.0 : 0.0;
    sat += saturated ? 1.0 : 0.0;
    clip += (saturated && fabs(x) - fabs(xh) > margin) ? 1.0 : 0.0;
  }
};

__global__ void __launch_bounds__(kWarps * 32) error_stats_kernel(const StatsArgs a) {
  __shared__ double red[kWarps][9];
  __shared__ unsigned int hist[64];
  const int h = blockIdx.y, side = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 64; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int D = a.D, P = a.P, VPL = D / 32;  // values per lane (4 or 1), lane l: elements VPL l ..
  const float* hdr = reinterpret_cast<const float*>(a.pool + (side ? kHdrVScaleOffset : kHdrKScaleOffset));
  const float st = *hdr;  // per-tensor scale (FP8 per-tensor s, NVFP4 s_t)
  const bool kvarn = a.mode == KVQ_KVARN_K4V2_G128;
  Acc acc;
  for (long long t = (long long)blockIdx.x * kWarps + warp; t < a.num_tokens; t += (long long)gridDim.x * kWarps) {
    const int slot = __ldg(a.slots + t);
    if (slot < 0) continue;
    const int page = slot / P, off = slot % P;
    if (page >= a.num_pages) {
      if (lane == 0 && h == 0 && side == 0) set_error(const_cast<uint8_t*>(a.pool), KVQ_DEVERR_SLOT_RANGE);
      continue;
    }
    const uint8_t* blk = a.pool + kHeaderBytes + ((size_t)page * a.Hkv + h) * a.block_bytes;
    // the input row
    float x[4];
    {
      const size_t base = ((size_t)t * a.Hkv + h) * D + (size_t)VPL * lane;
      const void* src = side ? a.v : a.k;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        x[i] = i < VPL ? (a.f32io ? static_cast<const float*>(src)[base + i]
                                  : __half2float(static_cast<const __half*>(src)[base + i]))
                       : 0.0f;
    }
    float xh[4] = {0.f, 0.f, 0.f, 0.f};
    bool sat[4] = {false, false, false, false};
    float margin[4] = {0.f, 0.f, 0.f, 0.f};
    const int m = a.mode;
    if (m == KVQ_FP8_PER_TENSOR || m == KVQ_INT8_PER_TOKEN_HEAD || m == KVQ_FP8_PER_TOKEN_HEAD) {
      const uint8_t* row = blk + (size_t)side * P * D + (size_t)off * D;
      const float s = m == KVQ_FP8_PER_TENSOR ? st
                                              : *reinterpret_cast<const float*>(blk + (size_t)2 * P * D +
                                                                                 (size_t)side * 4 * P + 4 * off);
      if (lane == 0) atomicAdd(&hist[scale_bin(s)], 1u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i >= VPL) break;
        const uint32_t c = row[VPL * lane + i];
        if (m == KVQ_INT8_PER_TOKEN_HEAD) {
          const int q = static_cast<int8_t>(c);
          xh[i] = (float)q * s;
          sat[i] = q == 127 || q == -127;
          margin[i] = 0.5f * s;
        } else {
          xh[i] = e4m3_val(c) * s;
          sat[i] = (c & 0x7Fu) == 0x7Eu;  // 448; the last step of the grid is 448 - 416
          margin[i] = 16.0f * s;
        }
      }
    } else if (m == KVQ_NVFP4 || m == KVQ_NVFP4_4OVER6) {
      const uint8_t* bs = blk + (size_t)P * D + (size_t)side * P * D / 16 + (size_t)off * D / 16;
      if (lane < D / 16) atomicAdd(&hist[scale_bin(e4m3_val(bs[lane]))], 1u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i >= VPL) break;
        const int d = VPL * lane + i;
        uint32_t nib;
        if (side == 0) nib = (blk[(size_t)off * D / 2 + d / 2] >> (4 * (d & 1))) & 15u;
        else nib = (blk[(size_t)P * D / 2 + (size_t)(off >> 1) * D + d] >> (4 * (off & 1))) & 15u;
        const float den = st * e4m3_val(bs[d / 16]);
        xh[i] = e2m1_val(nib) * den;
        sat[i] = (nib & 7u) == 7u;  // 6; the last step of the grid is 6 - 4
        margin[i] = den;
      }
    } else if (m == KVQ_INT4_PER_TOKEN_HEAD) {
      const float s = *reinterpret_cast<const float*>(blk + (size_t)P * D + (size_t)side * 4 * P + 4 * off);
      if (lane == 0) atomicAdd(&hist[scale_bin(s)], 1u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i >= VPL) break;
        const int d = VPL * lane + i;
        uint32_t word, nib;
        if (side == 0) {  // key word d/8: channel 8m + 2k in nibble k, 8m + 2k + 1 in nibble 4 + k
          word = *reinterpret_cast<const uint32_t*>(blk + (size_t)off * D / 2 + 4 * (d / 8));
          nib = ((d & 1) ? 4 : 0) + (d % 8) / 2;
        } else {          // value pair word d/4: channel 4m + k of the even token in nibble k, odd in 4 + k
          word = *reinterpret_cast<const uint32_t*>(blk + (size_t)P * D / 2 + (size_t)(off >> 1) * D + 4 * (d / 4));
          nib = (d % 4) + ((off & 1) ? 4 : 0);
        }
        const int q = (int)((word >> (4 * nib)) & 15u) - (((word >> (4 * nib)) & 8u) ? 16 : 0);
        xh[i] = (float)q * s;
        sat[i] = q == 7 || q == -7;
        margin[i] = 0.5f * s;
      }
    } else if (kvarn) {  // D = P = 128: 4 values per lane
      const float* km = reinterpret_cast<const float*>(blk + P * D / 2 + P * D / 4);
      const float* vm = km + 3 * D + P;
      float yh[4];
      if (side == 0) {
        const uint8_t* row = blk + (size_t)off * (D / 2);
        const float r = km[3 * D + off];
        if (off == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) atomicAdd(&hist[scale_bin(km[4 * lane + i])], 1u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int d = 4 * lane + i;
          const uint32_t q = (row[d / 2] >> (4 * (d & 1))) & 15u;
          yh[i] = r * km[2 * D + d] * (km[d] * (float)q + km[D + d]);
          sat[i] = q == 15u;
        }
      } else {
        const uint8_t* row = blk + P * D / 2 + (size_t)off * (D / 4);
        const float sc = vm[off], z = vm[P + off], r = vm[2 * P + off];
        if (lane == 0) atomicAdd(&hist[scale_bin(sc)], 1u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int d = 4 * lane + i;
          const uint32_t q = (row[d / 4] >> (2 * (d % 4))) & 3u;
          yh[i] = r * vm[3 * P + d] * (sc * (float)q + z);
          sat[i] = q == 3u;
        }
      }
      // back to the input domain: x^ = H y^; the min/max grid of the asymmetric
      // RTN cannot clip, so nothing counts as clipped
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xh[i] = yh[i];
        margin[i] = INFINITY;
      }
      fwht128(xh, lane);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < VPL) acc.add((double)x[i], (double)xh[i], sat[i], (double)margin[i]);
  }
  // merge: lanes, then warps, then one atomic per field
  double f[9] = {acc.n, acc.se, acc.sr, acc.sd, acc.dot, acc.mx, acc.zeros, acc.sat, acc.clip};
#pragma unroll
  for (int j = 0; j < 9; ++j) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const double y = __shfl_xor_sync(kFull, f[j], o);
      f[j] = j == 5 ? fmax(f[j], y) : f[j] + y;
    }
    if (lane == 0) red[warp][j] = f[j];
  }
  __syncthreads();
  kvq_error_stats* o = a.out + (size_t)side * a.Hkv + h;
  if (threadIdx.x < 9) {
    const int j = threadIdx.x;
    double v = red[0][j];
    for (int w = 1; w < kWarps; ++w) v = j == 5 ? fmax(v, red[w][j]) : v + red[w][j];
    double* dst = &o->count + j;  // the nine leading fields, in order
    if (j == 5) atomicMax(reinterpret_cast<unsigned long long*>(dst), (unsigned long long)__double_as_longlong(v));
    else atomicAdd(dst, v);
  }
  for (int i = threadIdx.x; i < 64; i += blockDim.x)
    if (hist[i]) atomicAdd(&o->scale_hist[i], (double)hist[i]);
}

}  // namespace

cudaError_t launch_error_stats(const kvq_cache* c, const void* k, const void* v, const int32_t* slots, int num_tokens,
                               kvq_error_stats* out, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(kvq_error_stats) * 2 * c->cfg.num_kv_heads, s);
  if (e != cudaSuccess || num_tokens == 0) return e;
  StatsArgs a;
  a.pool = c->base;
  a.k = k;
  a.v = v;
  a.slots = slots;
  a.num_tokens = num_tokens;
  a.Hkv = c->cfg.num_kv_heads;
  a.P = c->cfg.page_size;
  a.D = c->cfg.head_dim;
  a.num_pages = c->cfg.num_pages;
  a.mode = c->cfg.mode;
  a.f32io = c->cfg.io_dtype == KVQ_F32;
  a.block_bytes = c->block_bytes;
  a.out = out;
  long long want = ((long long)num_tokens + kWarps - 1) / kWarps;
  const long long cap = (long long)num_sms() * 4 / (2 * a.Hkv) + 1;
  const int blocks = (int)(want < cap ? want : cap);
  error_stats_kernel<<<dim3(blocks, a.Hkv, 2), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
