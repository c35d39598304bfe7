// kvq_decode.cu -- paged decode attention over the packed quantized cache,
// dequantization fused into the load path, for the 16-token-page modes (FP8
// per-tensor; INT8, FP8 and INT4 per-token-head; NVFP4, whose storage the
// 4over6 variant shares), plus the split-KV combine kernel.  Several causal
// queries per sequence run as one grid row each (query b % nq of sequence
// b / nq); the combine is launched as a programmatic dependent of the decode.
//
// Sources (web pages, by title and section):
//  "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化": "K 与 V 的量化误差进入 attention 的位置不同"
//     (A = softmax(QK^T/sqrt(d)), O = AV), "KV 的写入与读取路径" (unpack, apply block and tensor
//     scales inside the attention tile load, no dequantized temporary), "GQA";
//  "KV Cache 量化 · LLM Glossary": dequantize while loading inside the attention kernel;
//  "KV 量化" (rustineverything.app), 写和读: read by block table, multiply by the descale;
//     scale 和数据放在一起: the per-token-head modes, int4_per_token_head among them.
//
// Design (GB300): one CTA per (KV split, kv head, sequence), W warps; each
// warp owns a ring of STAGES shared-memory buffers and streams whole
// (page, kv head) blocks into them with TMA (a tiled tensor copy whose
// 128/64-byte swizzle makes the fragment loads bank-conflict free; a plain
// bulk copy for head_dim 32), completion tracked by one mbarrier per stage.
// A 16-token page is one tensor-core step: S^T = K Q^T on mma.m16n8k16 with
// M = 16 tokens, N = 8 query heads of the GQA group, K = 16 channels; then
// O^T += V^T P^T with M = 16 channels, N = 8 heads, K = 16 tokens.  Codes are
// converted to f16 in registers (exact: int8, e4m3, e2m1 x e4m3 are all
// representable), the scales are applied to the fp32 scores and to P, and the
// fp32 probabilities enter the second product as an f16 hi + lo pair so the
// result keeps ~22 bits.  Online softmax in base 2.  Split partials are merged
// inside the CTA and, when a sequence has several splits, by the combine kernel.
#include <cuda_fp16.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kPage = 16;
constexpr int kWarps = 4;
// Pipeline depth (pages in flight per warp) and the resident CTAs per SM the
// register budget is sized for, per payload width; -D overrides exist for tuning.
#ifndef KVQ_FP4_STAGES
#define KVQ_FP4_STAGES 4
#endif
#ifndef KVQ_FP4_MINB
#define KVQ_FP4_MINB 4
#endif
#ifndef KVQ_B1_STAGES
#define KVQ_B1_STAGES 2
#endif
#ifndef KVQ_B1_MINB
#define KVQ_B1_MINB 4
#endif
#ifndef KVQ_PT_STAGES
#define KVQ_PT_STAGES KVQ_B1_STAGES
#endif
// A warp's page ids for one split live in shared memory (at most this many
// pages per warp, so at most kWarps * kIdsPerWarp pages per split).
constexpr int kIdsPerWarp = 256;
constexpr float kLog2e = 1.4426950408889634f;

template <int MODE, int D>
struct Cfg {
  // 4-bit payloads (NVFP4 -- also the storage of NVFP4 4over6 -- and INT4):
  // K rows of D/2 bytes, V token-pair rows of D bytes.
  static constexpr bool FOUR = MODE == KVQ_NVFP4 || MODE == KVQ_INT4_PER_TOKEN_HEAD;
  static constexpr int RW = FOUR ? D / 2 : D;  // payload row bytes
  static constexpr int BLK = (int)block_bytes(MODE, kPage, D);
  static constexpr bool TMA = D == 128;
  // stage stride: a multiple of the swizzle pattern's period (1024 B for SW128,
  // 512 B for SW64), whose phase the hardware takes from the smem address
  static constexpr int SALIGN = !TMA ? 128 : (RW == 128 ? 1024 : 512);
  static constexpr int STAGE = (BLK + SALIGN - 1) / SALIGN * SALIGN;
  static constexpr int KSTEPS = D / 16;
  static constexpr int MTILES = D / 16;
  static constexpr int V_OFF = kPage * RW;            // V payload
  static constexpr int S_OFF = 2 * kPage * RW;        // scales region
  // SW128 for 128-byte rows, SW64 for 64-byte rows (XOR of address bits 7.. into 4..).
  static constexpr int SWZ_MASK = !TMA ? 0 : (RW == 128 ? 7 : 3);
  static constexpr int STAGES = FOUR ? KVQ_FP4_STAGES : MODE == KVQ_FP8_PER_TENSOR ? KVQ_PT_STAGES : KVQ_B1_STAGES;
  static constexpr int MINB = FOUR ? KVQ_FP4_MINB : KVQ_B1_MINB;
  // The running reference max may lag the true max by up to SLACK (log2 units)
  // before it is moved, so probabilities reach 2^SLACK; they are scaled by
  // 2^PSHIFT before the f16 split, with 2^(PSHIFT + SLACK) x (largest V scale
  // folded into P) inside the f16 range: per-token-head V scales of fp16 inputs
  // are at most 65504/127 (INT8), 65504/448 (FP8) or 65504/7 (INT4).
  static constexpr int slack(bool f32io) { return f32io ? 0 : 4; }
  static constexpr int pshift(bool f32io) {
    return MODE == KVQ_INT8_PER_TOKEN_HEAD ? (f32io ? 0 : 2)
         : MODE == KVQ_FP8_PER_TOKEN_HEAD ? (f32io ? 0 : 4)
         : MODE == KVQ_INT4_PER_TOKEN_HEAD ? (f32io ? 0 : -2) : (f32io ? 14 : 10);
  }
  // Channel group (D/8 channels) whose V rows the lanes of MMA row g load and
  // whose outputs they hold.  4-bit V at D = 128 is read as token-pair rows with
  // 128-bit loads under the 64-byte swizzle: the order 0, 4, 1, 5, 2, 6, 3, 7
  // puts the two groups of each 8-lane phase in different bank halves, so the
  // loads are conflict-free (the identity order is 2-way conflicted).
  static __device__ __forceinline__ int cgrp(int g) {
    return (FOUR && D == 128) ? ((g >> 1) | ((g & 1) << 2)) : g;
  }
  // The CTA's warps share one copy of the query fragments in shared memory
  // (one 64-bit load per k-step) instead of 16 registers each: faster for the
  // one-byte modes, slower for NVFP4 (measured on GB300).
  static constexpr bool QSMEM = !FOUR;
};

template <int MASK>
__device__ __forceinline__ int swz(int off) {
  return off ^ (((off >> 7) & MASK) << 4);
}

// One INT4 storage word (eight two's-complement 4-bit codes) -> four exact
// f16x2, out[i] = (nibble i, nibble i + 4): for a key word the channel pairs
// (2i, 2i + 1), for a value word channel i of the even and of the odd token.
// One lop3 per register: with two constant operands it maps each bit to 0, 1,
// w or ~w (LUT 0x6A: per bit (K1, K2) = (0,0) -> 0, (0,1) -> 1, (1,0) -> w,
// (1,1) -> ~w), so it selects two nibbles, flips their top bit (the code
// biased by 8) and supplies f16 1024 (nibble at mantissa bits 0-3) or 64
// (mantissa bits 4-7, step 1); one f16x2 subtraction of 1032 or 72 leaves
// the signed code.
__device__ __forceinline__ uint32_t lop3_sel(uint32_t w, uint32_t k1, uint32_t k2) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(k1), "r"(k2));
  return r;
}
__device__ __forceinline__ void s4w_to_f16x2x4(uint32_t w, uint32_t* out) {
  const __half2 c1032 = u32_as_h2(0x64086408u), c72 = u32_as_h2(0x54805480u);
  const uint32_t w8 = w >> 8;
  out[0] = h2_as_u32(__hsub2(u32_as_h2(lop3_sel(w, 0x000F000Fu, 0x64086408u)), c1032));
  out[1] = h2_as_u32(__hsub2(u32_as_h2(lop3_sel(w, 0x00F000F0u, 0x54805480u)), c72));
  out[2] = h2_as_u32(__hsub2(u32_as_h2(lop3_sel(w8, 0x000F000Fu, 0x64086408u)), c1032));
  out[3] = h2_as_u32(__hsub2(u32_as_h2(lop3_sel(w8, 0x00F000F0u, 0x54805480u)), c72));
}

// int8 pair (bytes 0,1 or 2,3 of w) -> exact f16x2 via 1024 + (x + 128) - 1152.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t biased_w, uint32_t sel) {
  const uint32_t h = prmt(biased_w, 0x64646464u, sel);
  return h2_as_u32(__hsub2(u32_as_h2(h), __half2half2(__ushort_as_half(0x6480))));  // 0x6480 = 1152
}

template <int MODE>
__device__ __forceinline__ void cvt_pair4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  // 4 one-byte codes -> (bytes 0,1) and (bytes 2,3) as f16x2
  if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD) {
    const uint32_t b = w ^ 0x80808080u;
    lo = i8x2_to_f16x2(b, 0x4140u);
    hi = i8x2_to_f16x2(b, 0x4342u);
  } else {
    lo = e4m3x2_to_f16x2(w & 0xFFFFu);
    hi = e4m3x2_to_f16x2(w >> 16);
  }
}

// Like cvt_pair4, but int8 words arrive already biased (x ^ 0x80 per byte).
template <int MODE>
__device__ __forceinline__ void cvt_pair4_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD) {
    lo = i8x2_to_f16x2(w, 0x4140u);
    hi = i8x2_to_f16x2(w, 0x4342u);
  } else {
    cvt_pair4<MODE>(w, lo, hi);
  }
}

// Q as the B operand of S^T = K Q^T: b0 = Q[g][d(j,2tq..2tq+1)], b1 = Q[g][d(j,2tq+8..+9)]
// with d(j, .) = tq*D/4 + 4j + {0,1} and {2,3}.  Heads >= G are zero.
template <int D, bool QF32>
__device__ __forceinline__ void load_q(const DecodeArgs& a, int b, int kvh, int g, int tq, uint32_t (*qh)[2],
                                       uint32_t (*ql)[2]) {
  constexpr int KSTEPS = D / 16;
  const bool ok = g < a.G;
  const long long row = ((long long)b * a.Hq + (long long)kvh * a.G + (ok ? g : 0)) * D + tq * (D / 4);
#pragma unroll
  for (int j = 0; j < KSTEPS; ++j) {
    float x[4];
    if constexpr (QF32) {
      const float4 u = ok ? __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + row + 4 * j))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
      __half2 h0 = __floats2half2_rn(x[0], x[1]), h1 = __floats2half2_rn(x[2], x[3]);
      const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
      qh[j][0] = h2_as_u32(h0);
      qh[j][1] = h2_as_u32(h1);
      ql[j][0] = h2_as_u32(__floats2half2_rn(x[0] - f0.x, x[1] - f0.y));
      ql[j][1] = h2_as_u32(__floats2half2_rn(x[2] - f1.x, x[3] - f1.y));
    } else {
      const uint2 u = ok ? __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(a.q) + row + 4 * j))
                         : make_uint2(0u, 0u);
      qh[j][0] = u.x;
      qh[j][1] = u.y;
    }
  }
}

// S^T = K Q^T for NP staged pages, their k-steps interleaved so the pages'
// MMA chains overlap: c[p][0..1] = token g, c[p][2..3] = token g+8, heads 2tq, 2tq+1.
template <int MODE, int D, bool QF32, int NP>
__device__ __forceinline__ void qk_pages(const uint8_t* const* st, int g, int tq, const uint32_t (*qh)[2],
                                         const uint32_t (*ql)[2], const uint2* qs, int lane, float (*c)[4]) {
  using C = Cfg<MODE, D>;
  constexpr int KSTEPS = C::KSTEPS;
  constexpr int KW = (C::FOUR ? D / 8 : D / 4) / 4;  // words per thread per row
  uint32_t kg[NP][KW], kh8[NP][KW];
  const int rb = tq * (KW * 4);
#pragma unroll
  for (int p = 0; p < NP; ++p)
#pragma unroll
    for (int w = 0; w < KW; w += 4) {
      lds<(KW >= 4 ? 4 : KW)>(st[p] + swz<C::SWZ_MASK>(g * C::RW + rb + 4 * w), kg[p] + w);
      lds<(KW >= 4 ? 4 : KW)>(st[p] + swz<C::SWZ_MASK>((g + 8) * C::RW + rb + 4 * w), kh8[p] + w);
    }
  if constexpr (MODE == KVQ_INT4_PER_TOKEN_HEAD) {  // per-token K scale: applied to the scores
#pragma unroll
    for (int w = 0; w < KW; ++w)
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        uint32_t fg[4], fh[4];
        s4w_to_f16x2x4(kg[p][w], fg);
        s4w_to_f16x2x4(kh8[p][w], fh);
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          const int j = 2 * w + hlf;
          const uint32_t af[4] = {fg[2 * hlf], fh[2 * hlf], fg[2 * hlf + 1], fh[2 * hlf + 1]};
          mma16816(c[p], af, qh[j][0], qh[j][1]);
          if constexpr (QF32) mma16816(c[p], af, ql[j][0], ql[j][1]);
        }
      }
  } else if constexpr (MODE == KVQ_NVFP4) {
    constexpr int SB = D / 16;
    const int blk0 = (tq * (D / 4)) / 16;
    const int base_g = C::S_OFF + g * SB, base_h = C::S_OFF + (g + 8) * SB;
    __half2 sg2[NP], sh2[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      uint32_t sg, sh;
      if constexpr (D / 4 >= 16) {
        sg = *reinterpret_cast<const uint16_t*>(st[p] + swz<C::SWZ_MASK>(base_g + blk0));
        sh = *reinterpret_cast<const uint16_t*>(st[p] + swz<C::SWZ_MASK>(base_h + blk0));
      } else {
        sg = st[p][swz<C::SWZ_MASK>(base_g + blk0)] * 0x0101u;
        sh = st[p][swz<C::SWZ_MASK>(base_h + blk0)] * 0x0101u;
      }
      sg2[p] = u32_as_h2(e4m3x2_to_f16x2(sg));
      sh2[p] = u32_as_h2(e4m3x2_to_f16x2(sh));
    }
#pragma unroll
    for (int w = 0; w < KW; ++w)
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int j = 2 * w + hlf;
        const bool second = (4 * j) >= 16;  // channel offset within the thread's D/4 range
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          uint32_t fg[4], fh[4];
          e2m1x8_to_f16x2x4(kg[p][w], fg);
          e2m1x8_to_f16x2x4(kh8[p][w], fh);
          const __half2 sa = second ? __high2half2(sg2[p]) : __low2half2(sg2[p]);
          const __half2 sb = second ? __high2half2(sh2[p]) : __low2half2(sh2[p]);
          uint32_t af[4];
          af[0] = h2_as_u32(__hmul2(u32_as_h2(fg[2 * hlf]), sa));
          af[1] = h2_as_u32(__hmul2(u32_as_h2(fh[2 * hlf]), sb));
          af[2] = h2_as_u32(__hmul2(u32_as_h2(fg[2 * hlf + 1]), sa));
          af[3] = h2_as_u32(__hmul2(u32_as_h2(fh[2 * hlf + 1]), sb));
          mma16816(c[p], af, qh[j][0], qh[j][1]);
          if constexpr (QF32) mma16816(c[p], af, ql[j][0], ql[j][1]);
        }
      }
  } else {
    static_assert(C::QSMEM, "one-byte modes read the query fragments from shared memory");
#pragma unroll
    for (int j = 0; j < KSTEPS; ++j)
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        uint32_t af[4];
        cvt_pair4<MODE>(kg[p][j], af[0], af[2]);
        cvt_pair4<MODE>(kh8[p][j], af[1], af[3]);
        const uint2 qv = qs[j * 32 + lane];
        mma16816(c[p], af, qv.x, qv.y);
        if constexpr (QF32) {
          const uint2 qw = qs[(KSTEPS + j) * 32 + lane];
          mma16816(c[p], af, qw.x, qw.y);
        }
      }
  }
}

// The V operands of a page pair, moved from the two stages into registers
// before the stages are refilled.  w[row][p][k]: word k of the thread's row of
// page p -- 4-bit modes: token-pair rows tq and tq + 4; one-byte modes: token
// rows 2tq, 2tq + 1, 2tq + 8, 2tq + 9.  NVFP4 adds the block scales of the
// thread's tokens as f16x2 pairs (tokens 2tq, 2tq + 1 and 2tq + 8, 2tq + 9).
template <int MODE, int D>
struct VRegs {
  static constexpr int VW = D / 32;  // words per thread per row, both layouts
  uint32_t w[Cfg<MODE, D>::FOUR ? 2 : 4][2][VW];
  __half2 sc[2][MODE == KVQ_NVFP4 ? 2 : 1];
};

// Load both pages' V operands.  With PARTIAL, rows (tokens) >= nvalid[p] are
// neutralised so that whatever bytes an unwritten slot (or a stage that holds
// no page, nvalid = 0) holds cannot reach the output: one-byte codes are
// zeroed, NVFP4 gets a zero block scale (E2M1 codes are all finite), and INT4
// codes are finite anyway, their tokens entering with p = 0.
template <int MODE, int D, bool PARTIAL>
__device__ __forceinline__ void pv_load(const uint8_t* const* st, int g, int tq, const int* nvalid,
                                        VRegs<MODE, D>& v) {
  using C = Cfg<MODE, D>;
  constexpr int VW = VRegs<MODE, D>::VW;
  const int r0 = 2 * tq, r1 = 2 * tq + 1, r2 = 2 * tq + 8, r3 = 2 * tq + 9;  // tokens
  if constexpr (C::FOUR) {
    // Token-pair rows: byte (k, d) holds channel d of tokens 2k (low nibble)
    // and 2k + 1, so one pair conversion gives the A fragment's (token 2tq,
    // 2tq + 1) f16x2 directly.  Lanes (g, tq) read pair rows tq and tq + 4,
    // channels cgb .. cgb + D/8 - 1.
    const int cgb = (D / 8) * C::cgrp(g);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      lds<VW>(st[p] + swz<C::SWZ_MASK>(C::V_OFF + tq * D + cgb), v.w[0][p]);
      lds<VW>(st[p] + swz<C::SWZ_MASK>(C::V_OFF + (tq + 4) * D + cgb), v.w[1][p]);
    }
    if constexpr (MODE == KVQ_NVFP4) {
      const int vblk = cgb / 16;
      constexpr int VS = C::S_OFF + kPage * (D / 16);  // V block scales [kPage][D/16]
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t b0 = st[p][swz<C::SWZ_MASK>(VS + r0 * (D / 16) + vblk)];
        uint32_t b1 = st[p][swz<C::SWZ_MASK>(VS + r1 * (D / 16) + vblk)];
        uint32_t b2 = st[p][swz<C::SWZ_MASK>(VS + r2 * (D / 16) + vblk)];
        uint32_t b3 = st[p][swz<C::SWZ_MASK>(VS + r3 * (D / 16) + vblk)];
        if constexpr (PARTIAL) {
          const int nv = nvalid[p];
          if (r0 >= nv) b0 = 0;
          if (r1 >= nv) b1 = 0;
          if (r2 >= nv) b2 = 0;
          if (r3 >= nv) b3 = 0;
        }
        v.sc[p][0] = u32_as_h2(e4m3x2_to_f16x2(b0 | (b1 << 8)));
        v.sc[p][1] = u32_as_h2(e4m3x2_to_f16x2(b2 | (b3 << 8)));
      }
    }
  } else {
    const int cb = g * (D / 8);
    const int rows[4] = {r0, r1, r2, r3};
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        lds<VW>(st[p] + swz<C::SWZ_MASK>(C::V_OFF + rows[r] * C::RW + cb), v.w[r][p]);
        if constexpr (PARTIAL) {
#pragma unroll
          for (int k = 0; k < VW; ++k)
            if (rows[r] >= nvalid[p]) v.w[r][p][k] = 0;
        }
      }
  }
}

// O^T += V^T P^T for the page pair in registers (M-tiles interleaved across
// the two pages).  Tile t of the 4-bit layouts uses channel cgb + 2t in MMA
// row g and cgb + 2t + 1 in row g + 8; the one-byte layout interleaves the
// channels of each word with a byte permute.
template <int MODE, int D>
__device__ __forceinline__ void pv_mma(const VRegs<MODE, D>& v, const uint32_t (*bh)[2], const uint32_t (*bl)[2],
                                       float (*o)[4]) {
  constexpr int VW = VRegs<MODE, D>::VW;
  if constexpr (MODE == KVQ_INT4_PER_TOKEN_HEAD) {
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int w = 0; w < VW; ++w) {
        uint32_t f0[4], f2[4];  // byte e of the word: channel cgb + 4w + e
        s4w_to_f16x2x4(v.w[0][p][w], f0);
        s4w_to_f16x2x4(v.w[1][p][w], f2);
        uint32_t av[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          av[u][0] = f0[2 * u];
          av[u][1] = f0[2 * u + 1];
          av[u][2] = f2[2 * u];
          av[u][3] = f2[2 * u + 1];
          mma16816(o[2 * w + u], av[u], bh[p][0], bh[p][1]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) mma16816(o[2 * w + u], av[u], bl[p][0], bl[p][1]);
      }
  } else if constexpr (MODE == KVQ_NVFP4) {
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int w = 0; w < VW; ++w) {
        uint32_t f0[4], f2[4];  // byte e of the word: channel cgb + 4w + e
        e2m1x8_to_f16x2x4(v.w[0][p][w], f0);
        e2m1x8_to_f16x2x4(v.w[1][p][w], f2);
        // hi products of the word's two tiles first, then lo, so that a tile's
        // two MMAs are not issued back to back into the same accumulator
        uint32_t av[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          av[u][0] = h2_as_u32(__hmul2(u32_as_h2(f0[2 * u]), v.sc[p][0]));
          av[u][1] = h2_as_u32(__hmul2(u32_as_h2(f0[2 * u + 1]), v.sc[p][0]));
          av[u][2] = h2_as_u32(__hmul2(u32_as_h2(f2[2 * u]), v.sc[p][1]));
          av[u][3] = h2_as_u32(__hmul2(u32_as_h2(f2[2 * u + 1]), v.sc[p][1]));
          mma16816(o[2 * w + u], av[u], bh[p][0], bh[p][1]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) mma16816(o[2 * w + u], av[u], bl[p][0], bl[p][1]);
      }
  } else {
#pragma unroll
    for (int w = 0; w < VW; ++w)
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t a0 = v.w[0][p][w], a1 = v.w[1][p][w], a2 = v.w[2][p][w], a3 = v.w[3][p][w];
        if constexpr (MODE == KVQ_INT8_PER_TOKEN_HEAD) {  // bias once per word: x + 128
          a0 ^= 0x80808080u; a1 ^= 0x80808080u; a2 ^= 0x80808080u; a3 ^= 0x80808080u;
        }
        const uint32_t x01 = prmt(a0, a1, 0x5140u), y01 = prmt(a0, a1, 0x7362u);
        const uint32_t x23 = prmt(a2, a3, 0x5140u), y23 = prmt(a2, a3, 0x7362u);
        uint32_t av[4], aw[4];
        cvt_pair4_biased<MODE>(x01, av[0], av[1]);
        cvt_pair4_biased<MODE>(x23, av[2], av[3]);
        cvt_pair4_biased<MODE>(y01, aw[0], aw[1]);
        cvt_pair4_biased<MODE>(y23, aw[2], aw[3]);
        mma16816(o[2 * w], av, bh[p][0], bh[p][1]);  // hi of both tiles, then lo
        mma16816(o[2 * w + 1], aw, bh[p][0], bh[p][1]);
        mma16816(o[2 * w], av, bl[p][0], bl[p][1]);
        mma16816(o[2 * w + 1], aw, bl[p][0], bl[p][1]);
      }
  }
}

// Dynamic shared memory of a decode CTA: the warps' stage rings, reused at the
// end by the merge of the warps ([W][8][D] outputs, then [W][8] m and l) and,
// right after that region, by the CTA's own partial for a merge across a
// thread-block cluster ([8] m, [8] l, [8][D] outputs).
template <int D>
constexpr size_t warp_merge_bytes() { return (size_t)kWarps * 8 * (D + 2) * sizeof(float); }
template <int D>
constexpr size_t cluster_part_bytes() { return (size_t)8 * (D + 2) * sizeof(float); }
template <int MODE, int D>
constexpr size_t decode_smem() {
  using C = Cfg<MODE, D>;
  constexpr size_t ring = (size_t)kWarps * C::STAGES * C::STAGE;
  constexpr size_t merge = warp_merge_bytes<D>() + cluster_part_bytes<D>();
  return (ring > merge ? ring : merge) + 1024;  // + the 1024-byte alignment of the ring
}

// Merge of a query row's splits inside their thread-block cluster (one CTA per
// split, ranks in split order).  Each CTA has left (m_h, l_h, o_h) for the G
// heads of its split in `part` ([8] m, [8] l, [8][D] o); CTA r then takes
// every cluster-size-th element (h, d) from r * blockDim on:
// M = max_s m_s, w_s = 2^(m_s - M), out = sum_s o_s w_s / sum_s l_s w_s (0 for
// a row without tokens).  The second barrier keeps every CTA's shared memory
// alive until its peers have read it.
template <int D>
__device__ void merge_in_cluster(const DecodeArgs& a, int b, int kvh, const float* part) {
  cluster_barrier();
  const int r = cluster_rank(), ns = cluster_size();
  const float* pm = part;
  const float* pl = part + 8;
  const float* po = part + 16;
  for (int idx = r * blockDim.x + threadIdx.x; idx < a.G * D; idx += ns * blockDim.x) {
    const int h = idx / D, d = idx % D;
    float ms[8];
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      ms[s] = s < ns ? ld_cluster_f32(pm + h, s) : -INFINITY;
      M = fmaxf(M, ms[s]);
    }
    float L = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        if (s < ns) {
          const float w = exp2f(ms[s] - M);
          L += ld_cluster_f32(pl + h, s) * w;
          O += ld_cluster_f32(po + h * D + d, s) * w;
        }
      }
    }
    store_out(a, ((long long)b * a.Hq + (long long)kvh * a.G + h) * D + d, L > 0.0f ? O / L : 0.0f);
  }
  cluster_barrier();
}

template <int MODE, int D, bool QF32>
__global__ void __launch_bounds__(kWarps * 32, Cfg<MODE, D>::MINB) decode_kernel(const __grid_constant__ DecodeArgs a,
                                                               const __grid_constant__ CUtensorMap tmap) {
  using C = Cfg<MODE, D>;
  constexpr int KSTEPS = C::KSTEPS, MTILES = C::MTILES;
  constexpr int PSHIFT = C::pshift(QF32);
  constexpr float SLACK = (float)C::slack(QF32);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bars[kWarps][C::STAGES];
  __shared__ int page_ids[kWarps * kIdsPerWarp];
  // 1024-byte alignment of the ring (swizzle patterns are address based)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // b: the query row -- query b % nq of sequence b / nq (nq = 1: the sequence)
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int seq = b / a.nq;
  pdl_launch_dependents();

  int n = a.seq_lens[seq];
  const int lim = min(a.max_seq_len, a.max_pages * kPage);
  if (n > lim || n < 0) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0) set_error(const_cast<uint8_t*>(a.pool), KVQ_DEVERR_SEQ_LEN);
    n = n < 0 ? 0 : lim;
  }
  n = max(n - (a.nq - 1 - b % a.nq), 0);  // causal: the tokens up to the query's own position
  const int t_begin = split * a.tokens_per_split;
  const int t_end = min(n, t_begin + a.tokens_per_split);
  float* cpart = reinterpret_cast<float*>(smem + warp_merge_bytes<D>());  // merge across the cluster
  if (t_begin >= t_end) {
    if (a.num_splits == 1) {  // empty sequence: zero output rows
      for (int i = threadIdx.x; i < a.G * D; i += blockDim.x) {
        const long long o = ((long long)b * a.Hq + (long long)kvh * a.G + i / D) * D + i % D;
        store_out(a, o, 0.0f);
      }
    } else if (a.cluster) {  // an empty split still takes part in its cluster's merge
      for (int i = threadIdx.x; i < 8 * (D + 2); i += blockDim.x) cpart[i] = i < 8 ? -INFINITY : 0.0f;
      merge_in_cluster<D>(a, b, kvh, cpart);
    }
    return;
  }
  const int p0 = t_begin / kPage, p1 = (t_end + kPage - 1) / kPage;
  const int my_count = (p1 - p0 - warp + kWarps - 1) / kWarps;  // pages of this warp (<= 32)

  uint8_t* ring = smem + warp * C::STAGES * C::STAGE;
  uint64_t* wb = bars[warp];
  if (lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) mbar_init(&wb[s], 1);
    mbar_fence_init();
    if constexpr (C::TMA) prefetch_tmap(&tmap);
  }
  __syncwarp();

  // the warp's page ids (an out-of-range id is flagged and its page skipped)
  int* ids = page_ids + warp * kIdsPerWarp;
  for (int k = lane; k < my_count; k += 32) {
    int pid = __ldg(a.block_table + (long long)seq * a.max_pages + p0 + warp + kWarps * k);
    if (pid < 0 || pid >= a.num_pages) {
      set_error(const_cast<uint8_t*>(a.pool), KVQ_DEVERR_PAGE_RANGE);
      pid = -1;
    }
    ids[k] = pid;
  }
  __syncwarp();

  // stream page i of this warp into stage i % STAGES: a TMA row coordinate or a
  // byte offset for the plain bulk copy
  auto issue = [&](int i) {
    const int pid = ids[i];
    long long src = kHeaderBytes + ((long long)pid * a.Hkv + kvh) * (long long)C::BLK;
    if constexpr (C::TMA) src /= C::RW;
    if (lane == 0) {
      uint64_t* bar = &wb[i % C::STAGES];
      mbar_arrive_expect_tx(bar, pid >= 0 ? (uint32_t)C::BLK : 0u);
      if (pid >= 0) {
        uint8_t* dst = ring + (i % C::STAGES) * C::STAGE;
        if constexpr (C::TMA)
          tma_g2s_2d(dst, &tmap, 0, (int)src, bar);
        else
          bulk_g2s(dst, a.pool + src, (uint32_t)C::BLK, bar);
      }
    }
  };

  const int npre = my_count < C::STAGES ? my_count : C::STAGES;
  for (int i = 0; i < npre; ++i) issue(i);

  // query fragments: in registers, or one copy in shared memory (C::QSMEM)
  __shared__ uint2 qsm[C::QSMEM ? (QF32 ? 2 : 1) * KSTEPS * 32 : 1];
  uint32_t qh[KSTEPS][2], ql[QF32 ? KSTEPS : 1][2];
  if (!C::QSMEM || warp == 0) load_q<D, QF32>(a, b, kvh, g, tq, qh, ql);
  if constexpr (C::QSMEM) {
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < KSTEPS; ++j) {
        qsm[j * 32 + lane] = make_uint2(qh[j][0], qh[j][1]);
        if constexpr (QF32) qsm[(KSTEPS + j) * 32 + lane] = make_uint2(ql[j][0], ql[j][1]);
      }
    }
    __syncthreads();
  }

  // Scores in log2 units: s = c * kfac (FP8 per-tensor, NVFP4: the K tensor scale
  // is uniform) or c * ks[t] * softmax_scale*log2(e) (per-token-head).  The
  // probabilities enter P V scaled by 2^PSHIFT (added in the exponent); l sums the
  // same scaled values, so O / l needs no correction.
  float kfac = a.sm_log2, vfac = 1.0f;
  if constexpr (MODE == KVQ_FP8_PER_TENSOR || MODE == KVQ_NVFP4) {
    kfac *= *reinterpret_cast<const float*>(a.pool + kHdrKScaleOffset);
    vfac = *reinterpret_cast<const float*>(a.pool + kHdrVScaleOffset);
  }
  constexpr bool kPerToken =
      MODE == KVQ_INT8_PER_TOKEN_HEAD || MODE == KVQ_FP8_PER_TOKEN_HEAD || MODE == KVQ_INT4_PER_TOKEN_HEAD;

  float o[MTILES][4];
#pragma unroll
  for (int i = 0; i < MTILES; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m0 = -1e30f, m1 = -1e30f, l0 = 0.0f, l1 = 0.0f;  // finite start: no inf - inf
  bool timed_out = false;

  for (int i = 0; i < my_count; i += 2) {
    const bool two = i + 1 < my_count;  // warp-uniform
    const int pidA = ids[i];
    const int pidB_raw = ids[two ? i + 1 : i];
    const int pidB = two ? pidB_raw : -1;
    const uint8_t* stA = ring + (i % C::STAGES) * C::STAGE;
    const uint8_t* stB = ring + ((i + 1) % C::STAGES) * C::STAGE;
    if (!mbar_wait_bounded(&wb[i % C::STAGES], (i / C::STAGES) & 1) ||
        (two && !mbar_wait_bounded(&wb[(i + 1) % C::STAGES], ((i + 1) / C::STAGES) & 1))) {
      timed_out = true;
      break;
    }
    const int tokA = (p0 + warp + kWarps * i) * kPage;
    const int tokB = tokA + kWarps * kPage;
    const int nvA = pidA >= 0 ? min(t_end - tokA, kPage) : 0;   // valid rows of each page
    const int nvB = pidB >= 0 ? min(t_end - tokB, kPage) : 0;

    // full pairs take a branch-free path with the two pages interleaved
    const bool full2 = nvA == kPage && nvB == kPage;
    const uint8_t* stAB[2] = {stA, stB};
    float cc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (full2) {
      qk_pages<MODE, D, QF32, 2>(stAB, g, tq, qh, ql, qsm, lane, cc);
    } else {
      if (nvA > 0) qk_pages<MODE, D, QF32, 1>(stAB, g, tq, qh, ql, qsm, lane, cc);
      if (nvB > 0) qk_pages<MODE, D, QF32, 1>(stAB + 1, g, tq, qh, ql, qsm, lane, cc + 1);
    }
    const float* cA = cc[0];
    const float* cB = cc[1];

    float fA0 = kfac, fA8 = kfac, fB0 = kfac, fB8 = kfac;     // score factors of tokens g, g+8
    float vA0 = 1.f, vA8 = 1.f, vB0 = 1.f, vB8 = 1.f;         // V per-token scales
    if constexpr (kPerToken) {
      const float* sa = reinterpret_cast<const float*>(stA + C::S_OFF);  // K scales, then V scales
      const float* sb = reinterpret_cast<const float*>(stB + C::S_OFF);
      fA0 *= sa[g]; fA8 *= sa[g + 8]; vA0 = sa[kPage + g]; vA8 = sa[kPage + g + 8];
      fB0 *= sb[g]; fB8 *= sb[g + 8]; vB0 = sb[kPage + g]; vB8 = sb[kPage + g + 8];
    }
    // The V operands go to registers and both stages are refilled now, so the
    // next pages are in flight during the softmax and the P V products (INT4:
    // after them, measured faster there).
    VRegs<MODE, D> vr;
    if (full2) {
      const int nv2[2] = {kPage, kPage};
      pv_load<MODE, D, false>(stAB, g, tq, nv2, vr);
    } else {
      const int nvAB[2] = {nvA, nvB};
      pv_load<MODE, D, true>(stAB, g, tq, nvAB, vr);
    }
    constexpr bool kEarlyRefill = MODE != KVQ_INT4_PER_TOKEN_HEAD;
    auto refill = [&]() {
      __syncwarp();
      if (i + C::STAGES < my_count) {
        if (lane == 0) fence_proxy_async_smem();
        issue(i + C::STAGES);
        if (i + 1 + C::STAGES < my_count) issue(i + 1 + C::STAGES);
      }
    };
    if constexpr (kEarlyRefill) refill();
    // (heads 2tq, 2tq + 1 of a token travel as packed f32x2 pairs)
    float2 sA[2] = {__fmul2_rn(make_float2(cA[0], cA[1]), make_float2(fA0, fA0)),
                    __fmul2_rn(make_float2(cA[2], cA[3]), make_float2(fA8, fA8))};  // tokens g, g + 8
    float2 sB[2] = {__fmul2_rn(make_float2(cB[0], cB[1]), make_float2(fB0, fB0)),
                    __fmul2_rn(make_float2(cB[2], cB[3]), make_float2(fB8, fB8))};
    if (nvA < kPage || nvB < kPage) {  // rare: a partial or missing page
      if (g >= nvA) { sA[0] = make_float2(-INFINITY, -INFINITY); vA0 = 0.f; }
      if (g + 8 >= nvA) { sA[1] = make_float2(-INFINITY, -INFINITY); vA8 = 0.f; }
      if (g >= nvB) { sB[0] = make_float2(-INFINITY, -INFINITY); vB0 = 0.f; }
      if (g + 8 >= nvB) { sB[1] = make_float2(-INFINITY, -INFINITY); vB8 = 0.f; }
    }
    // Lazy reference max: move it (and rescale) only when some score exceeds it
    // by more than SLACK -- rare once the first pages are seen.
    float bm0 = fmaxf(fmaxf(sA[0].x, sA[1].x), fmaxf(sB[0].x, sB[1].x));  // this thread's max, heads 2tq, 2tq+1
    float bm1 = fmaxf(fmaxf(sA[0].y, sA[1].y), fmaxf(sB[0].y, sB[1].y));
    if (__any_sync(kFull, (bm0 > m0 + SLACK) | (bm1 > m1 + SLACK))) {
#pragma unroll
      for (int x = 4; x <= 16; x <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, x));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, x));
      }
      const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
      const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);  // m starts at a finite -1e30
      m0 = n0;
      m1 = n1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int t = 0; t < MTILES; ++t) {
        o[t][0] *= al0; o[t][2] *= al0;
        o[t][1] *= al1; o[t][3] *= al1;
      }
    }
    const float2 e01 = make_float2((float)PSHIFT - m0, (float)PSHIFT - m1);
    float2 pA[2], pB[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float2 ua = __fadd2_rn(sA[r], e01), ub = __fadd2_rn(sB[r], e01);
      pA[r] = make_float2(ex2(ua.x), ex2(ua.y));
      pB[r] = make_float2(ex2(ub.x), ex2(ub.y));
    }
    {
      const float2 lsum = __fadd2_rn(__fadd2_rn(pA[0], pA[1]), __fadd2_rn(pB[0], pB[1]));
      l0 += lsum.x;
      l1 += lsum.y;
    }
    // P^T as the B operand: f16 hi + lo, each 8x8 block transposed in registers
    uint32_t bh[2][2], bl[2][2];
    {
      float2 x[4] = {pA[0], pA[1], pB[0], pB[1]};  // (heads 2tq, 2tq + 1) of tokens g, g + 8 of A, then B
      if constexpr (kPerToken) {
        x[0] = __fmul2_rn(x[0], make_float2(vA0, vA0));
        x[1] = __fmul2_rn(x[1], make_float2(vA8, vA8));
        x[2] = __fmul2_rn(x[2], make_float2(vB0, vB0));
        x[3] = __fmul2_rn(x[3], make_float2(vB8, vB8));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // hi = x cut to 10 mantissa bits (exact in f16 over P's range; below
        // 2^-14 the f16 conversion rounds it, an error under 2^-24), lo = the
        // exact remainder rounded to f16: together ~22 bits of x
        const float2 hh = make_float2(__uint_as_float(__float_as_uint(x[k].x) & 0xFFFFE000u),
                                      __uint_as_float(__float_as_uint(x[k].y) & 0xFFFFE000u));
        const __half2 h = __floats2half2_rn(hh.x, hh.y);
        const float2 rem = __fadd2_rn(x[k], make_float2(-hh.x, -hh.y));
        const __half2 lo = __floats2half2_rn(rem.x, rem.y);
        bh[k >> 1][k & 1] = movmatrix_t(h2_as_u32(h));
        bl[k >> 1][k & 1] = movmatrix_t(h2_as_u32(lo));
      }
    }
    pv_mma<MODE, D>(vr, bh, bl, o);
    if constexpr (!kEarlyRefill) refill();
  }
  if (timed_out && lane == 0) set_error(const_cast<uint8_t*>(a.pool), KVQ_DEVERR_TIMEOUT);

  // ---------------- merge the warps of this CTA
#pragma unroll
  for (int x = 4; x <= 16; x <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, x);
    l1 += __shfl_xor_sync(kFull, l1, x);
  }
  __syncthreads();  // every warp is done with its ring: reuse it for the merge
  float* red_o = reinterpret_cast<float*>(smem);             // [W][8][D]
  float* red_m = red_o + kWarps * 8 * D;                     // [W][8]
  float* red_l = red_m + kWarps * 8;                         // [W][8]
  if (g == 0) {
    red_m[warp * 8 + 2 * tq] = m0;
    red_m[warp * 8 + 2 * tq + 1] = m1;
    red_l[warp * 8 + 2 * tq] = l0;
    red_l[warp * 8 + 2 * tq + 1] = l1;
  }
  // staged column of (row h, channel d): bank-swizzled at D = 128
  auto col = [](int h, int d) { return D == 128 ? merge_col128(h, d) : d; };
  {
    float* ow = red_o + warp * 8 * D;
    const int d0 = C::cgrp(g) * (D / 8);
#pragma unroll
    for (int t = 0; t < MTILES; ++t) {
      ow[(2 * tq) * D + col(2 * tq, d0 + 2 * t)] = o[t][0];
      ow[(2 * tq + 1) * D + col(2 * tq + 1, d0 + 2 * t)] = o[t][1];
      ow[(2 * tq) * D + col(2 * tq, d0 + 2 * t + 1)] = o[t][2];
      ow[(2 * tq + 1) * D + col(2 * tq + 1, d0 + 2 * t + 1)] = o[t][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < a.G * D; idx += blockDim.x) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float L = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float e = exp2f(red_m[w * 8 + h] - M);
        L += red_l[w * 8 + h] * e;
        O += red_o[(w * 8 + h) * D + col(h, d)] * e;
      }
    }
    const int hq = kvh * a.G + h;
    if (a.num_splits == 1) {
      const float r = L > 0.0f ? O * vfac / L : 0.0f;
      const long long oi = ((long long)b * a.Hq + hq) * D + d;
      store_out(a, oi, r);
    } else if (a.cluster) {
      cpart[16 + h * D + d] = O * vfac;
      if (d == 0) {
        cpart[h] = M;
        cpart[8 + h] = L;
      }
    } else {
      const long long pi = ((long long)b * a.Hq + hq) * a.num_splits + split;
      store_ws(a, a.ws_o + (pi * D + d), O * vfac);
      if (d == 0) {
        store_ws(a, a.ws_ml + (2 * pi), M);
        store_ws(a, a.ws_ml + (2 * pi + 1), L);
      }
    }
  }
  if (a.cluster) merge_in_cluster<D>(a, b, kvh, cpart);
}

// Merge the splits of each (sequence, query head).
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float wts[D], red[D / 32];
  const int b = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq, d = threadIdx.x;  // b: query row
  pdl_wait_primary();  // the decode grid's partials are complete and visible
  int n = a.seq_lens[b / a.nq];
  const int lim = min(a.max_seq_len, a.max_pages * kPage);
  n = n < 0 ? 0 : (n > lim ? lim : n);
  n = max(n - (a.nq - 1 - b % a.nq), 0);
  const int ns = (n + a.tokens_per_split - 1) / a.tokens_per_split;
  const float r = merge_split_row<D>(a, ((long long)b * a.Hq + hq) * a.num_splits, ns, wts, red);
  const long long oi = ((long long)b * a.Hq + hq) * D + d;
  store_out(a, oi, r);
}

// Resident CTAs per SM of one decode kernel instance (occupancy query, cached;
// the register budget's target if the query fails).
template <int MODE, int D, bool QF32>
int resident_ctas() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n > 0) return n;
  auto kern = decode_kernel<MODE, D, QF32>;
  constexpr size_t smem = decode_smem<MODE, D>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarps * 32, smem) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = Cfg<MODE, D>::MINB;
  }
  cached.store(n, std::memory_order_relaxed);
  return n;
}

template <int D, bool QF32>
int resident_ctas_d(int mode) {
  switch (mode) {
    case KVQ_FP8_PER_TENSOR: return resident_ctas<KVQ_FP8_PER_TENSOR, D, QF32>();
    case KVQ_INT8_PER_TOKEN_HEAD: return resident_ctas<KVQ_INT8_PER_TOKEN_HEAD, D, QF32>();
    case KVQ_FP8_PER_TOKEN_HEAD: return resident_ctas<KVQ_FP8_PER_TOKEN_HEAD, D, QF32>();
    case KVQ_NVFP4:
    case KVQ_NVFP4_4OVER6: return resident_ctas<KVQ_NVFP4, D, QF32>();
    case KVQ_INT4_PER_TOKEN_HEAD: return resident_ctas<KVQ_INT4_PER_TOKEN_HEAD, D, QF32>();
    default: return 1;
  }
}

int resident_ctas_of(const kvq_cache* c) {
  const bool f32 = c->cfg.io_dtype == KVQ_F32;
  if (c->cfg.head_dim == 128) return f32 ? resident_ctas_d<128, true>(c->cfg.mode) : resident_ctas_d<128, false>(c->cfg.mode);
  return f32 ? resident_ctas_d<32, true>(c->cfg.mode) : resident_ctas_d<32, false>(c->cfg.mode);
}

template <int MODE, int D, bool QF32>
cudaError_t launch_mode(const kvq_cache* c, const DecodeArgs& a, cudaStream_t s) {
  constexpr size_t smem = decode_smem<MODE, D>();
  auto kern = decode_kernel<MODE, D, QF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.Hkv, a.B);
  if (a.cluster) {  // the splits of a row: one cluster along x, merged on chip
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.num_splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, c->tmap);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  kern<<<grid, kWarps * 32, smem, s>>>(a, c->tmap);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.num_splits == 1) return e;
  e = launch_dependent(combine_kernel<D>, dim3(a.B * a.Hq), dim3(D), s, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, bool QF32>
cudaError_t launch_d(const kvq_cache* c, const DecodeArgs& a, cudaStream_t s) {
  switch (c->cfg.mode) {
    case KVQ_FP8_PER_TENSOR: return launch_mode<KVQ_FP8_PER_TENSOR, D, QF32>(c, a, s);
    case KVQ_INT8_PER_TOKEN_HEAD: return launch_mode<KVQ_INT8_PER_TOKEN_HEAD, D, QF32>(c, a, s);
    case KVQ_FP8_PER_TOKEN_HEAD: return launch_mode<KVQ_FP8_PER_TOKEN_HEAD, D, QF32>(c, a, s);
    case KVQ_NVFP4:  // NVFP4 4over6 shares NVFP4's storage: only the write differs
    case KVQ_NVFP4_4OVER6: return launch_mode<KVQ_NVFP4, D, QF32>(c, a, s);
    case KVQ_INT4_PER_TOKEN_HEAD: return launch_mode<KVQ_INT4_PER_TOKEN_HEAD, D, QF32>(c, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Split plan.  Sequence lengths are known only on the device, so the plan
// takes every sequence to be max_seq_len long.  One CTA per (split, kv head,
// sequence) -- per query row for the mma.sync kernel's multi-query decode --,
// R of them resident per SM; pages per split pps = ceil(pages / s).
//  mma.sync kernel (16-token pages, 1 to kIdsPerWarp per warp) streams at the
//  memory system's pace: a plan with s splits is estimated at
//      ceil(units * s / (R * SMs)) waves  x  (pps + kSplitCostPages).
//  tcgen05 kernel (128-token tiles, all queries of a sequence in one CTA):
//      ceil(units * s / (R * SMs)) waves  x  (tiles per split + kSplitCostUmma).
//  KVarN (the CTA shares each 128-token tile, at most 64 per split) is bound
//  by instruction issue, so a partial wave runs faster and what counts is the
//  busiest SM: ceil(units * s / SMs) x (pps + kSplitCostTiles), with at least
//  one full wave of CTAs (R per SM) to hide latency when there is work for it.
// The overheads are a CTA's cost beyond its pages (start-up, pipeline fill,
// merge, partial write) in page or tile units, fitted to GB300 timings; the
// smallest estimate wins, ties going to the split that divides the pages most
// evenly, then to fewer splits.
constexpr long long kSplitCostPages = 16;
constexpr long long kSplitCostTiles = 2;
constexpr long long kSplitCostUmma = 1;
constexpr int kMaxClusterSplits = 8;  // portable thread-block cluster size

DecodePlan plan_decode(const kvq_cache* c, int num_seqs, int num_q_heads, int max_seq_len, int num_queries) {
  DecodePlan p{1, c->cfg.page_size, 0};
  const int P = c->cfg.page_size;
  const long long pages = (max_seq_len + P - 1) / P;
  if (pages <= 0) return p;
  const long long sms = num_sms();
  const bool kvarn = c->cfg.mode == KVQ_KVARN_K4V2_G128;
  const bool umma = !kvarn && umma_decode_eligible(c, num_q_heads, num_queries);
  const long long rows = (long long)num_seqs * num_queries;  // query rows: the partials' first index
  long long splits = 1;
  long long mma_slots = 0;  // mma.sync kernel: resident CTAs on the whole GPU
  if (umma) {
    const long long units = (long long)num_seqs * c->cfg.num_kv_heads;
    const long long tiles = (pages + 7) / 8;
    const long long cap_tiles = umma_max_pages_per_split() / 8;
    const long long slots = (long long)umma_resident_ctas(c, num_q_heads, num_queries) * sms;
    const long long min_s = (tiles + cap_tiles - 1) / cap_tiles;
    const long long hi = tiles < min_s + 256 ? tiles : min_s + 256;
    long long best = -1, best_ragged = 0;
    splits = min_s;
    for (long long s = min_s; s <= hi; ++s) {
      const long long tps = (tiles + s - 1) / s;
      const long long cost = (units * s + slots - 1) / slots * (tps + kSplitCostUmma);
      const long long ragged = s * tps - tiles;
      if (best < 0 || cost < best || (cost == best && ragged < best_ragged)) {
        best = cost;
        best_ragged = ragged;
        splits = s;
      }
    }
    const long long tps = (tiles + splits - 1) / splits;
    p.tokens_per_split = (int)(tps * 8 * P);
  } else {
    const long long units = rows * c->cfg.num_kv_heads;
    const long long cap = kvarn ? 64 : (long long)kWarps * kIdsPerWarp;
    const long long min_pages = kvarn ? 1 : kWarps;
    long long min_splits = (pages + cap - 1) / cap;
    const long long max_splits = (pages + min_pages - 1) / min_pages;
    const long long slots = (long long)(kvarn ? kvarn_resident_ctas() : resident_ctas_of(c)) * sms;
    if (!kvarn) mma_slots = slots;
    if (kvarn) {  // one full wave when the tiles allow it
      long long full = (slots + units - 1) / units;
      if (full > max_splits) full = max_splits;
      if (full > min_splits) min_splits = full;
    }
    long long best = -1, best_ragged = 0;
    splits = min_splits;
    const long long hi = max_splits < min_splits + 256 ? max_splits : min_splits + 256;
    for (long long s = min_splits; s <= hi; ++s) {
      const long long pps = (pages + s - 1) / s;
      const long long cost = kvarn ? (units * s + sms - 1) / sms * (pps + kSplitCostTiles)
                                   : (units * s + slots - 1) / slots * (pps + kSplitCostPages);
      const long long ragged = s * pps - pages;  // ties: the evener split
      if (best < 0 || cost < best || (cost == best && ragged < best_ragged)) {
        best = cost;
        best_ragged = ragged;
        splits = s;
      }
    }
    if (splits < 1) splits = 1;
    const long long pps = (pages + splits - 1) / splits;
    p.tokens_per_split = (int)(pps * P);
  }
  p.num_splits = (int)((max_seq_len + p.tokens_per_split - 1) / p.tokens_per_split);
  // mma.sync kernel, 2 to 8 splits, every CTA resident at once: the splits of
  // a query row run as one thread-block cluster and merge on chip, so neither
  // the partials' round trip through memory nor a combine launch remains
  p.cluster_merge = mma_slots > 0 && p.num_splits >= 2 && p.num_splits <= kMaxClusterSplits &&
                    rows * c->cfg.num_kv_heads * p.num_splits <= mma_slots;
  if (p.num_splits > 1 && !p.cluster_merge)
    p.workspace_bytes = (size_t)rows * num_q_heads * p.num_splits * (c->cfg.head_dim + 2) * sizeof(float);
  return p;
}

cudaError_t launch_decode(const kvq_cache* c, const DecodePlan& plan, const void* q, const int32_t* block_table,
                          int max_pages, const int32_t* seq_lens, int num_seqs, int num_q_heads, int max_seq_len,
                          float softmax_scale, void* out, int out_dtype, void* workspace, cudaStream_t stream,
                          const void* kvarn_tail, int num_queries) {
  DecodeArgs a;
  a.pool = c->base;
  a.q = q;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.nq = num_queries;
  a.cluster = plan.cluster_merge ? 1 : 0;
  num_seqs *= num_queries;  // query rows: q, out and the split partials are [num_seqs * nq][Hq]..
  a.ws_o = static_cast<float*>(workspace);
  const bool partials = (plan.num_splits > 1 && !plan.cluster_merge) || kvarn_tail;  // split partials in memory
  a.ws_ml = partials
                ? a.ws_o + (size_t)num_seqs * num_q_heads * plan.num_splits * c->cfg.head_dim
                : nullptr;
  a.num_pages = c->cfg.num_pages;
  a.Hkv = c->cfg.num_kv_heads;
  a.Hq = num_q_heads;
  a.G = num_q_heads / c->cfg.num_kv_heads;
  a.B = num_seqs;
  a.max_pages = max_pages;
  a.max_seq_len = max_seq_len;
  a.tokens_per_split = plan.tokens_per_split;
  a.num_splits = plan.num_splits;
  a.out_f32 = out_dtype == KVQ_F32;
  a.q_f32 = c->cfg.io_dtype == KVQ_F32;
  a.sm_log2 = softmax_scale * kLog2e;
  a.block_bytes = c->block_bytes;
  a.tail = static_cast<const uint8_t*>(kvarn_tail);
  a.rows_per_block = c->rows_per_block;
  {
    uint8_t* o = static_cast<uint8_t*>(out);
    const size_t oel = (size_t)num_seqs * num_q_heads * c->cfg.head_dim;  // num_seqs counts query rows here
    a.out_span = Span{o, o + oel * (out_dtype == KVQ_F32 ? 4 : 2)};
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const size_t wbytes = partials
                              ? (size_t)num_seqs * num_q_heads * plan.num_splits * (c->cfg.head_dim + 2) * sizeof(float)
                              : 0;
    a.ws_span = Span{w, w ? w + wbytes : nullptr};
  }
  if (num_seqs == 0) return cudaSuccess;
  if (c->cfg.mode == KVQ_KVARN_K4V2_G128) return launch_kvarn_decode(a, stream);
  if (umma_decode_eligible(c, num_q_heads, num_queries)) {
    cudaError_t e = launch_umma_decode(c, a, stream);
    if (e != cudaSuccess || a.num_splits == 1) return e;
    const int D = c->cfg.head_dim;
    e = D == 128 ? launch_dependent(combine_kernel<128>, dim3(a.B * a.Hq), dim3(128), stream, a) : cudaErrorInvalidValue;
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const bool qf32 = c->cfg.io_dtype == KVQ_F32;
  if (c->cfg.head_dim == 128)
    return qf32 ? launch_d<128, true>(c, a, stream) : launch_d<128, false>(c, a, stream);
  if (c->cfg.head_dim == 32)
    return qf32 ? launch_d<32, true>(c, a, stream) : launch_d<32, false>(c, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
