// kvq_decode_kvarn.cu -- paged decode attention over the KVarN k4v2 g128 cache.
//
// Source: "KVarN：华为推出的原生 vLLM KV-cache 量化后端，打破性能与精度的权衡",
// section 技术原理: 128-token tiles; a Hadamard rotation along channels, which is
// orthogonal and so leaves attention scores unchanged; variance normalisation;
// asymmetric round-to-nearest whose scales are folded back at read time, keys
// per channel and values per token.  Attention itself follows
// "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化", A = softmax(QK^T/sqrt(d)), O = AV.
//
// Stored tile (per kv head), rotated domain: x^_td = r_t c_d (scale * code + zero)
// with K's scale/zero per channel and V's per token.  With q' = H q:
//   s_t  = r^K_t [ sum_d (q'_d c^K_d scale^K_d) code^K_td + sum_d q'_d c^K_d zero^K_d ]
//   o'_d = c^V_d [ sum_t (p_t r^V_t scale^V_t) code^V_td + sum_t p_t r^V_t zero^V_t ]
//   o    = H o' / sum_t p_t
// so every scale folds into the 8 x 128 query (once per tile) or into the
// probabilities (once per token), and the codes enter the tensor cores as
// small exact f16 values: a key code c (0..15) becomes 1 + c/16 and a value
// code (0..3) becomes 1 + c/4, each by one shift and one bit-select; the
// constant 1 is taken back out with the per-tile sums of the folded query
// and of the scaled probabilities.
//
// GB300 layout: one CTA per (KV split, kv head, sequence); the CTA's warps
// share a ring of 16 KB tile buffers filled by bulk TMA copies (one per tile).
// Per tile the CTA folds the query (channel d per thread) into shared memory
// in mma.sync B-fragment order; each warp then takes 2 of the tile's 8
// 16-token sub-blocks: S^T = K Q^T and O^T += V^T P^T on mma.m16n8k16 (N = the
// GQA group of 8 query heads), online softmax in base 2, f16 hi + lo splits
// for the folded query and for the probabilities.
#include <cuda_fp16.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kT = 128;                              // tokens per tile (= page)
constexpr int kD = 128;                              // head_dim
constexpr int kBlk = 16384;                          // bytes per (tile, kv head)
constexpr int kW = 4;                                // warps per CTA
constexpr int kVOff = kT * kD / 2;                   // V codes [128][32]
constexpr int kKMeta = kVOff + kT * kD / 4;          // K: scale[D] zero[D] c[D] r[T]
constexpr int kVMeta = kKMeta + 4 * (3 * kD + kT);   // V: scale[T] zero[T] r[T] c[D]
constexpr int kPShift = 14;                          // P scaled by 2^14 before the f16 split
constexpr int kMaxTiles = 64;                        // tiles per split (page ids kept in smem)
#ifndef KVQ_KVARN_STAGES
#define KVQ_KVARN_STAGES 2
#endif
constexpr int kS = KVQ_KVARN_STAGES;

// The folded query is the B operand of S^T = K Q^T.  Entry (k-step j, lane
// 4h + tq) holds head h's channels base, base+4, base+1, base+5 with
// base = 32 tq + 8 (j >> 1) + 2 (j & 1), as {b0, b1} in f16 hi then lo; the
// key-code unpacking (kcode) produces the A operand in the same channel order.
// Entries are stored at [j][(4h + tq) ^ 4j]: the MMA warps' loads (one j at a
// time) and the fold's stores (one h at a time) are both conflict-free.
__host__ __device__ constexpr int frag_base(int j, int tq) { return 32 * tq + 8 * (j >> 1) + 2 * (j & 1); }

struct Shared {
  float qrot[8][kD];     // q' = H q per head of the group (set-up only)
  uint4 frag[8][32];     // folded query, see above
  float4 cs[32];         // per tile, entry order (4 j + tq): c_d * scale_d of K
  float4 cz[32];         //                                   c_d * zero_d of K
  float kf[kT];          // r^K_t * softmax_scale * log2(e)
  float vf[kT];          // r^V_t * scale^V_t
  float vz[kT];          // r^V_t * zero^V_t
  float beta[8];         // per head: sum_d q'_d c_d zero_d - 16 sum_d (folded query used)
  float vmax_part[kW];
  int pages[kMaxTiles];
};
constexpr size_t kSmem = (size_t)kS * kBlk + sizeof(Shared);

// Two 4-bit key codes (bits sft..sft+3 and 16+sft..) -> f16x2 {1 + c/16}: c lands in
// mantissa bits 6..9 of 1.0 (0x3C00).
__device__ __forceinline__ uint32_t kcode(uint32_t w, int sft) {
  const uint32_t x = sft >= 6 ? (w >> (sft - 6)) : (w << (6 - sft));
  return (x & 0x03C003C0u) | 0x3C003C00u;
}
// Two 2-bit value codes (bits sft..sft+1 and 16+sft..) -> f16x2 {1 + c/4}: c lands in
// mantissa bits 8..9 of 1.0.
__device__ __forceinline__ uint32_t vcode(uint32_t w, int sft) {
  const uint32_t x = sft >= 8 ? (w >> (sft - 8)) : (w << (8 - sft));
  return (x & 0x03000300u) | 0x3C003C00u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// In-register normalised Walsh-Hadamard transform of one 128-vector held as
// 4 consecutive values per lane (lane l: elements 4l..4l+3).
__device__ __forceinline__ void fwht128_warp(float* v, int lane) {
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
  const float c = 0.08838834764831845f;
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= c;
}

__global__ void __launch_bounds__(kW * 32) kvarn_decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t bars[kS];
  uint8_t* ring = smem_raw;
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw + (size_t)kS * kBlk);

  // b: the query row -- query b % nq of sequence b / nq (nq = 1: the sequence)
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int seq = b / a.nq;
  uint8_t* pool = const_cast<uint8_t*>(a.pool);
  pdl_launch_dependents();

  int n = a.seq_lens[seq];
  const int lim = min(a.max_seq_len, a.max_pages * kT);
  const bool first = tid == 0 && split == 0 && kvh == 0;
  if (n > lim || n < 0) {
    if (first) set_error(pool, KVQ_DEVERR_SEQ_LEN);
    n = n < 0 ? 0 : lim;
  }
  if (n % kT) {  // only whole tiles are quantized: the rest is read from the tail, if there is one
    if (first && a.tail == nullptr) set_error(pool, KVQ_DEVERR_PARTIAL_TILE);
    n -= n % kT;
  }
  // causal: the tokens up to the query's own position (several queries per
  // sequence come without a tail, so the last tile a query sees may end early)
  n = max(n - (a.nq - 1 - b % a.nq), 0);
  // with a tail, every CTA leaves a partial result for the merge kernel
  const bool direct = a.num_splits == 1 && a.tail == nullptr;
  const int t_begin = split * a.tokens_per_split;
  const int t_end = min(n, t_begin + a.tokens_per_split);
  if (t_begin >= t_end) {
    if (direct) {
      for (int i = tid; i < a.G * kD; i += blockDim.x) {
        const long long o = ((long long)b * a.Hq + (long long)kvh * a.G + i / kD) * kD + i % kD;
        store_out(a, o, 0.0f);
      }
    }
    return;
  }
  const int tile0 = t_begin / kT, ntiles = (t_end - t_begin + kT - 1) / kT;

  if (tid < ntiles) {
    int pid = __ldg(a.block_table + (long long)seq * a.max_pages + tile0 + tid);
    if (pid < 0 || pid >= a.num_pages) {
      set_error(pool, KVQ_DEVERR_PAGE_RANGE);
      pid = -1;
    }
    sh.pages[tid] = pid;
  }
  if (tid == 0) {
    for (int s = 0; s < kS; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](int i) {  // thread 0 only
    const int pid = sh.pages[i];
    uint64_t* bar = &bars[i % kS];
    mbar_arrive_expect_tx(bar, pid >= 0 ? (uint32_t)kBlk : 0u);
    if (pid >= 0)
      bulk_g2s(ring + (i % kS) * kBlk, a.pool + kHeaderBytes + ((size_t)pid * a.Hkv + kvh) * kBlk, kBlk, bar);
  };
  if (tid == 0)
    for (int i = 0; i < min(kS, ntiles); ++i) issue(i);

  // q' = H q for the group's heads (zero for heads >= G)
  for (int h = warp; h < 8; h += kW) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (h < a.G) {
      const long long row = ((long long)b * a.Hq + (long long)kvh * a.G + h) * kD + 4 * lane;
      if (a.q_f32) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + row));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
      } else {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(a.q) + row));
        const float2 f0 = __half22float2(u32_as_h2(u.x)), f1 = __half22float2(u32_as_h2(u.y));
        v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
      }
    }
    fwht128_warp(v, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) sh.qrot[h][4 * lane + i] = v[i];
  }
  __syncthreads();
  // this lane's fold entry: k-step fj, channel group ftq, for heads warp and warp + 4
  const int fj = lane >> 2, ftq = lane & 3, fbase = frag_base(fj, ftq);
  float qv[2][4];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float* qr = sh.qrot[warp + kW * hh];
    qv[hh][0] = qr[fbase];
    qv[hh][1] = qr[fbase + 4];
    qv[hh][2] = qr[fbase + 1];
    qv[hh][3] = qr[fbase + 5];
  }

  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  bool timed_out = false;

  for (int i = 0; i < ntiles; ++i) {
    const uint8_t* st = ring + (i % kS) * kBlk;
    const bool ok = mbar_wait_bounded(&bars[i % kS], (i / kS) & 1);
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    const int pid = sh.pages[i];
    if (pid >= 0) {
      const float* km = reinterpret_cast<const float*>(st + kKMeta);
      const float* vm = reinterpret_cast<const float*>(st + kVMeta);
      // ---- fold, part 1: thread tid owns channel d = tid and token t = tid
      {
        const int d = tid;
        // entry (j, tq) and position of channel d (inverse of frag_base)
        const int tqd = d >> 5, w = (d & 31) >> 3, k = d & 7, sd = k & 3, half = k >> 2;
        const int pos = 4 * (4 * (2 * w + (sd >> 1)) + tqd) + 2 * (sd & 1) + half;
        reinterpret_cast<float*>(sh.cs)[pos] = km[2 * kD + d] * km[d];       // c_d * scale_d
        reinterpret_cast<float*>(sh.cz)[pos] = km[2 * kD + d] * km[kD + d];  // c_d * zero_d
        const int t = tid;
        sh.kf[t] = km[3 * kD + t] * a.sm_log2;
        const float f = vm[2 * kT + t] * vm[t];
        sh.vf[t] = f;
        sh.vz[t] = vm[2 * kT + t] * vm[kT + t];
        float fm = fabsf(f);
#pragma unroll
        for (int x = 16; x >= 1; x >>= 1) fm = fmaxf(fm, __shfl_xor_sync(kFull, fm, x));
        if (lane == 0) sh.vmax_part[warp] = fm;
      }
      __syncthreads();
      // ---- fold, part 2: warp w folds heads w and w + 4, lane = entry 4 j + tq
      {
        const float4 cs4 = sh.cs[lane], cz4 = sh.cz[lane];
        const float2 csp[2] = {make_float2(cs4.x, cs4.y), make_float2(cs4.z, cs4.w)};
        const float2 czp[2] = {make_float2(cz4.x, cz4.y), make_float2(cz4.z, cz4.w)};
        float bph[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = warp + kW * hh;
          uint32_t hw[2], lw[2];
          float2 bpp = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int ip = 0; ip < 2; ++ip) {  // entries 2 ip, 2 ip + 1 as a packed pair
            const float2 q2 = make_float2(qv[hh][2 * ip], qv[hh][2 * ip + 1]);
            const float2 qt = __fmul2_rn(q2, csp[ip]);
            const __half2 hi = __floats2half2_rn(qt.x, qt.y);
            const float2 fh = __half22float2(hi);
            const float2 rem = __fadd2_rn(qt, make_float2(-fh.x, -fh.y));
            const __half2 lo = __floats2half2_rn(rem.x, rem.y);
            const float2 fl = __half22float2(lo);
            // the tensor core sees (1 + code/16): take out 16 * the folded query it used
            bpp = __fadd2_rn(bpp, __ffma2_rn(q2, czp[ip], __fmul2_rn(make_float2(-16.0f, -16.0f), __fadd2_rn(fh, fl))));
            hw[ip] = h2_as_u32(hi);
            lw[ip] = h2_as_u32(lo);
          }
          sh.frag[fj][(4 * h + ftq) ^ (4 * fj)] = make_uint4(hw[0], hw[1], lw[0], lw[1]);
          bph[hh] = bpp.x + bpp.y;
        }
        float2 bp = make_float2(bph[0], bph[1]);  // heads warp, warp + kW: one packed warp sum
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
          bp = __fadd2_rn(bp, make_float2(__shfl_xor_sync(kFull, bp.x, o), __shfl_xor_sync(kFull, bp.y, o)));
        if (lane == 0) {
          sh.beta[warp] = bp.x;
          sh.beta[warp + kW] = bp.y;
        }
      }
      __syncthreads();
      const float be0 = sh.beta[2 * tq], be1 = sh.beta[2 * tq + 1];
      const float vmx = fmaxf(fmaxf(sh.vmax_part[0], sh.vmax_part[1]), fmaxf(sh.vmax_part[2], sh.vmax_part[3]));
      int ex = 0;
      (void)frexpf(vmx, &ex);                         // vmx < 2^ex
      const float vnorm = ldexpf(1.0f, -ex);          // p' * vf * vnorm <= 2^kPShift
      const float vback = ldexpf(4.0f, ex);           // undoes vnorm and the 1/4 of the value codes

      // ---- this warp's two 16-token sub-blocks: tokens 16*sa.., 16*sb..
      const int sa = warp, sb = warp + kW;
      float cA[4] = {0.f, 0.f, 0.f, 0.f}, cB[4] = {0.f, 0.f, 0.f, 0.f};
      {
        uint32_t KA0[4], KA8[4], KB0[4], KB8[4];
        lds<4>(st + (16 * sa + g) * 64 + tq * 16, KA0);
        lds<4>(st + (16 * sa + g + 8) * 64 + tq * 16, KA8);
        lds<4>(st + (16 * sb + g) * 64 + tq * 16, KB0);
        lds<4>(st + (16 * sb + g + 8) * 64 + tq * 16, KB8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 fq = sh.frag[j][lane ^ (4 * j)];
          const int w = j >> 1, sft = (j & 1) * 8;
          uint32_t af[4];
          af[0] = kcode(KA0[w], sft);
          af[2] = kcode(KA0[w], sft + 4);
          af[1] = kcode(KA8[w], sft);
          af[3] = kcode(KA8[w], sft + 4);
          mma16816(cA, af, fq.x, fq.y);
          mma16816(cA, af, fq.z, fq.w);
          af[0] = kcode(KB0[w], sft);
          af[2] = kcode(KB0[w], sft + 4);
          af[1] = kcode(KB8[w], sft);
          af[3] = kcode(KB8[w], sft + 4);
          mma16816(cB, af, fq.x, fq.y);
          mma16816(cB, af, fq.z, fq.w);
        }
      }
      const int ta = 16 * sa + g, tb = 16 * sb + g;
      const float kA0 = sh.kf[ta], kA8 = sh.kf[ta + 8], kB0 = sh.kf[tb], kB8 = sh.kf[tb + 8];
      // (heads 2tq, 2tq + 1 of a token travel as packed f32x2 pairs)
      const float2 be = make_float2(be0, be1), c16 = make_float2(16.0f, 16.0f);
      float2 sA[2] = {__fmul2_rn(__ffma2_rn(make_float2(cA[0], cA[1]), c16, be), make_float2(kA0, kA0)),
                      __fmul2_rn(__ffma2_rn(make_float2(cA[2], cA[3]), c16, be), make_float2(kA8, kA8))};
      float2 sB[2] = {__fmul2_rn(__ffma2_rn(make_float2(cB[0], cB[1]), c16, be), make_float2(kB0, kB0)),
                      __fmul2_rn(__ffma2_rn(make_float2(cB[2], cB[3]), c16, be), make_float2(kB8, kB8))};
      const int nv = t_end - (t_begin + i * kT);  // tokens of this tile the query sees
      if (nv < kT) {
        const float2 ninf = make_float2(-INFINITY, -INFINITY);
        if (ta >= nv) sA[0] = ninf;
        if (ta + 8 >= nv) sA[1] = ninf;
        if (tb >= nv) sB[0] = ninf;
        if (tb + 8 >= nv) sB[1] = ninf;
      }
      float bm0 = fmaxf(fmaxf(sA[0].x, sA[1].x), fmaxf(sB[0].x, sB[1].x));
      float bm1 = fmaxf(fmaxf(sA[0].y, sA[1].y), fmaxf(sB[0].y, sB[1].y));
#pragma unroll
      for (int x = 4; x <= 16; x <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, x));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, x));
      }
      const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
      const float z0 = n0 == -INFINITY ? 0.0f : n0, z1 = n1 == -INFINITY ? 0.0f : n1;
      const float al0 = ex2(m0 - z0), al1 = ex2(m1 - z1);
      m0 = n0;
      m1 = n1;
      if (!__all_sync(kFull, al0 == 1.0f && al1 == 1.0f)) {
        const float2 al = make_float2(al0, al1);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float2 a01 = __fmul2_rn(make_float2(o[t][0], o[t][1]), al);
          const float2 a23 = __fmul2_rn(make_float2(o[t][2], o[t][3]), al);
          o[t][0] = a01.x; o[t][1] = a01.y; o[t][2] = a23.x; o[t][3] = a23.y;
        }
      }
      const float2 e01 = make_float2((float)kPShift - z0, (float)kPShift - z1);
      float2 pA[2], pB[2];  // (heads 2tq, 2tq + 1) of tokens ta, ta + 8 and tb, tb + 8
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float2 ua = __fadd2_rn(sA[r], e01), ub = __fadd2_rn(sB[r], e01);
        pA[r] = make_float2(ex2(ua.x), ex2(ua.y));
        pB[r] = make_float2(ex2(ub.x), ex2(ub.y));
      }
      {
        const float2 lsum = __fadd2_rn(__fadd2_rn(pA[0], pA[1]), __fadd2_rn(pB[0], pB[1]));
        l0 = l0 * al0 + lsum.x;
        l1 = l1 * al1 + lsum.y;
      }
      // value-side bias: sum_t p'_t r_t zero_t over this warp's 32 tokens
      const float zA0 = sh.vz[ta], zA8 = sh.vz[ta + 8], zB0 = sh.vz[tb], zB8 = sh.vz[tb + 8];
      float2 bv = __fadd2_rn(__ffma2_rn(pA[0], make_float2(zA0, zA0), __fmul2_rn(pA[1], make_float2(zA8, zA8))),
                             __ffma2_rn(pB[0], make_float2(zB0, zB0), __fmul2_rn(pB[1], make_float2(zB8, zB8))));
      uint32_t bh[4], bl[4];
      {
        const float fA0 = sh.vf[ta] * vnorm, fA8 = sh.vf[ta + 8] * vnorm;
        const float fB0 = sh.vf[tb] * vnorm, fB8 = sh.vf[tb + 8] * vnorm;
        const float2 x[4] = {__fmul2_rn(pA[0], make_float2(fA0, fA0)), __fmul2_rn(pA[1], make_float2(fA8, fA8)),
                             __fmul2_rn(pB[0], make_float2(fB0, fB0)), __fmul2_rn(pB[1], make_float2(fB8, fB8))};
        float2 u = make_float2(0.0f, 0.0f);  // sum of the f16 values the tensor core sees, per head
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __half2 h = __floats2half2_rn(x[k].x, x[k].y);
          const float2 f = __half22float2(h);
          const float2 rem = __fadd2_rn(x[k], make_float2(-f.x, -f.y));
          const __half2 lo = __floats2half2_rn(rem.x, rem.y);
          const float2 fl = __half22float2(lo);
          u = __fadd2_rn(u, __fadd2_rn(f, fl));
          bh[k] = movmatrix_t(h2_as_u32(h));
          bl[k] = movmatrix_t(h2_as_u32(lo));
        }
        // value codes enter as (1 + code/4): take out vback * sum of the probabilities used
        bv = __ffma2_rn(make_float2(-vback, -vback), u, bv);
      }
      float bv0 = bv.x, bv1 = bv.y;
#pragma unroll
      for (int x = 4; x <= 16; x <<= 1) {
        bv0 += __shfl_xor_sync(kFull, bv0, x);
        bv1 += __shfl_xor_sync(kFull, bv1, x);
      }
      // ---- O_tile^T = V^T P^T for both sub-blocks, then the per-channel fold
      float ot[8][4];
#pragma unroll
      for (int t = 0; t < 8; ++t) ot[t][0] = ot[t][1] = ot[t][2] = ot[t][3] = 0.0f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int base = 16 * (half ? sb : sa);
        const uint8_t* vrow = st + kVOff + 4 * g;
        const uint32_t A0 = *reinterpret_cast<const uint32_t*>(vrow + (base + 2 * tq) * 32);
        const uint32_t A1 = *reinterpret_cast<const uint32_t*>(vrow + (base + 2 * tq + 1) * 32);
        const uint32_t A2 = *reinterpret_cast<const uint32_t*>(vrow + (base + 2 * tq + 8) * 32);
        const uint32_t A3 = *reinterpret_cast<const uint32_t*>(vrow + (base + 2 * tq + 9) * 32);
        // codes 0..7 of two rows side by side (low / high halfword), then 8..15
        const uint32_t X01 = prmt(A0, A1, 0x5410u), Y01 = prmt(A0, A1, 0x7632u);
        const uint32_t X23 = prmt(A2, A3, 0x5410u), Y23 = prmt(A2, A3, 0x7632u);
        const uint32_t hb0 = half ? bh[2] : bh[0], hb1 = half ? bh[3] : bh[1];
        const uint32_t lb0 = half ? bl[2] : bl[0], lb1 = half ? bl[3] : bl[1];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint32_t s01 = t < 4 ? X01 : Y01, s23 = t < 4 ? X23 : Y23;
          const int sh2 = 4 * (t & 3);  // code e = 2t (row g) and 2t+1 (row g+8), 2 bits each
          uint32_t av[4];
          av[0] = vcode(s01, sh2);
          av[1] = vcode(s01, sh2 + 2);
          av[2] = vcode(s23, sh2);
          av[3] = vcode(s23, sh2 + 2);
          mma16816(ot[t], av, hb0, hb1);
          mma16816(ot[t], av, lb0, lb1);
        }
      }
      {
        float cv[16];
        lds<4>(reinterpret_cast<const uint8_t*>(vm + 3 * kT + 16 * g), reinterpret_cast<uint32_t*>(cv));
        lds<4>(reinterpret_cast<const uint8_t*>(vm + 3 * kT + 16 * g + 4), reinterpret_cast<uint32_t*>(cv + 4));
        lds<4>(reinterpret_cast<const uint8_t*>(vm + 3 * kT + 16 * g + 8), reinterpret_cast<uint32_t*>(cv + 8));
        lds<4>(reinterpret_cast<const uint8_t*>(vm + 3 * kT + 16 * g + 12), reinterpret_cast<uint32_t*>(cv + 12));
        const float2 vb = make_float2(vback, vback), bvv = make_float2(bv0, bv1);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float2 a01 = __ffma2_rn(make_float2(cv[2 * t], cv[2 * t]), __ffma2_rn(make_float2(ot[t][0], ot[t][1]), vb, bvv),
                                        make_float2(o[t][0], o[t][1]));
          const float2 a23 = __ffma2_rn(make_float2(cv[2 * t + 1], cv[2 * t + 1]),
                                        __ffma2_rn(make_float2(ot[t][2], ot[t][3]), vb, bvv), make_float2(o[t][2], o[t][3]));
          o[t][0] = a01.x; o[t][1] = a01.y; o[t][2] = a23.x; o[t][3] = a23.y;
        }
      }
    }
    __syncthreads();  // every warp is done with this stage
    if (tid == 0 && i + kS < ntiles) {
      fence_proxy_async_smem();
      issue(i + kS);
    }
  }
  if (timed_out && tid == 0) set_error(pool, KVQ_DEVERR_TIMEOUT);

  // ---- merge the warps (the ring is free: every issued copy was waited for)
#pragma unroll
  for (int x = 4; x <= 16; x <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, x);
    l1 += __shfl_xor_sync(kFull, l1, x);
  }
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(ring);   // [W][8][D]
  float* red_m = red_o + kW * 8 * kD;              // [W][8]
  float* red_l = red_m + kW * 8;                   // [W][8]
  float* fin = red_l + kW * 8;                     // [8][D]
  if (g == 0) {
    red_m[warp * 8 + 2 * tq] = m0;
    red_m[warp * 8 + 2 * tq + 1] = m1;
    red_l[warp * 8 + 2 * tq] = l0;
    red_l[warp * 8 + 2 * tq + 1] = l1;
  }
  {
    float* ow = red_o + warp * 8 * kD;
    const int d0 = 16 * g;
#pragma unroll
    for (int t = 0; t < 8; ++t) {  // bank-swizzled columns
      ow[(2 * tq) * kD + merge_col128(2 * tq, d0 + 2 * t)] = o[t][0];
      ow[(2 * tq + 1) * kD + merge_col128(2 * tq + 1, d0 + 2 * t)] = o[t][1];
      ow[(2 * tq) * kD + merge_col128(2 * tq, d0 + 2 * t + 1)] = o[t][2];
      ow[(2 * tq + 1) * kD + merge_col128(2 * tq + 1, d0 + 2 * t + 1)] = o[t][3];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < 8 * kD; idx += blockDim.x) {
    const int h = idx / kD, d = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float L = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kW; ++w) {
        const float e = ex2(red_m[w * 8 + h] - M);
        L += red_l[w * 8 + h] * e;
        O += red_o[(w * 8 + h) * kD + merge_col128(h, d)] * e;
      }
    }
    if (direct) {
      fin[idx] = L > 0.0f ? O / L : 0.0f;
    } else if (h < a.G) {
      const long long pi = ((long long)b * a.Hq + (long long)kvh * a.G + h) * a.num_splits + split;
      store_ws(a, a.ws_o + (pi * kD + d), O);
      if (d == 0) {
        store_ws(a, a.ws_ml + (2 * pi), M);
        store_ws(a, a.ws_ml + (2 * pi + 1), L);
      }
    }
  }
  if (direct) {
    __syncthreads();
    for (int h = warp; h < a.G; h += kW) {  // o = H o'
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = fin[h * kD + 4 * lane + i];
      fwht128_warp(v, lane);
      const long long ob = ((long long)b * a.Hq + (long long)kvh * a.G + h) * kD + 4 * lane;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        store_out(a, ob + i, v[i]);
      }
    }
  }
}

// Merge the splits of each (sequence, query head), then rotate back: o = H o'.
// With a tail (open tiles), the merged tile result stays unnormalised, is
// rotated back (H is linear) and joins the tail rows' terms, computed in the
// input domain: scores q . k_t in fp32 (warp w takes rows w, w + 4, ..; lane l
// channels 4l .. 4l + 3), then one max-subtracted softmax over both parts.
__global__ void __launch_bounds__(kD) kvarn_combine_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float v[kD], wts[kD], red[kD / 32], tsc[kT];
  const int b = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq, d = threadIdx.x;
  const int lane = d & 31, warp = d >> 5;
  pdl_wait_primary();  // the decode grid's partials are complete and visible
  int n = a.seq_lens[b / a.nq];  // b: the query row
  const int lim = min(a.max_seq_len, a.max_pages * kT);
  n = n < 0 ? 0 : (n > lim ? lim : n);
  const int nt = a.tail ? n % kT : 0;  // tail rows (one query per sequence)
  n -= n % kT;
  n = max(n - (a.nq - 1 - b % a.nq), 0);  // causal: as the decode kernel
  const int ns = (n + a.tokens_per_split - 1) / a.tokens_per_split;
  float M = -INFINITY, L = 0.0f;
  const float r0 = merge_split_row<kD>(a, ((long long)b * a.Hq + hq) * a.num_splits, ns, wts, red,
                                       a.tail ? &M : nullptr, &L);
  v[d] = r0;
  __syncthreads();
  for (int h = 1; h < kD; h <<= 1) {  // Sylvester butterflies across threads
    const float mine = v[d], other = v[d ^ h];
    __syncthreads();
    v[d] = (d & h) ? other - mine : mine + other;
    __syncthreads();
  }
  float r = v[d] * 0.08838834764831845f;
  if (a.tail) {
    const int kvh = hq / a.G;
    const size_t esz = a.q_f32 ? 4 : 2;
    const size_t row_elems = (size_t)a.Hkv * kD;                    // one tail row (token)
    const uint8_t* tk = a.tail + ((size_t)b * kT * row_elems + (size_t)kvh * kD) * esz;
    const uint8_t* tv = tk + (size_t)a.B * kT * row_elems * esz;    // the V rows follow the K rows
    auto ld4 = [&](const uint8_t* base, size_t elem, float* x) {  // 4 consecutive elements
      if (a.q_f32) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(base + elem * 4));
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
      } else {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(base + elem * 2));
        const float2 f0 = __half22float2(u32_as_h2(u.x)), f1 = __half22float2(u32_as_h2(u.y));
        x[0] = f0.x; x[1] = f0.y; x[2] = f1.x; x[3] = f1.y;
      }
    };
    float qv[4];
    ld4(static_cast<const uint8_t*>(a.q), ((size_t)b * a.Hq + hq) * kD + 4 * lane, qv);
    for (int t = warp; t < nt; t += kD / 32) {
      float kx[4];
      ld4(tk, (size_t)t * row_elems + 4 * lane, kx);
      float dot = qv[0] * kx[0] + qv[1] * kx[1] + qv[2] * kx[2] + qv[3] * kx[3];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
      if (lane == 0) tsc[t] = dot * a.sm_log2;
    }
    __syncthreads();
    // the tiles' (M, L, H acc) carry the 2^kPShift of the decode kernel's P: their max is M - kPShift
    const float Mq = M - (float)kPShift;
    float mt = Mq;
    for (int t = 0; t < nt; ++t) mt = fmaxf(mt, tsc[t]);
    float Lt = 0.0f, Ot = 0.0f;
    if (mt != -INFINITY) {
      const float wq = exp2f(Mq - mt);
      Lt = L * wq;
      Ot = r * wq;  // H acc, normalised rotation
      for (int t = 0; t < nt; ++t) {
        const float w = exp2f(tsc[t] - mt);
        const uint8_t* vr = tv + ((size_t)t * row_elems + d) * esz;
        Lt += w;
        Ot += w * (a.q_f32 ? *reinterpret_cast<const float*>(vr) : __half2float(*reinterpret_cast<const __half*>(vr)));
      }
    }
    r = Lt > 0.0f ? Ot / Lt : 0.0f;
  }
  const long long oi = ((long long)b * a.Hq + hq) * kD + d;
  store_out(a, oi, r);
}

}  // namespace

int kvarn_resident_ctas() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaFuncSetAttribute(kvarn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmem)) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kvarn_decode_kernel, kW * 32, kSmem) != cudaSuccess ||
      n <= 0) {
    (void)cudaGetLastError();
    n = 4;
  }
  cached.store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_kvarn_decode(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kvarn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.Hkv, a.B);
  kvarn_decode_kernel<<<grid, kW * 32, kSmem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || (a.num_splits == 1 && a.tail == nullptr)) return e;
  e = launch_dependent(kvarn_combine_kernel, dim3(a.B * a.Hq), dim3(kD), s, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvq
