// kvq_decode_umma.cu -- paged decode attention on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory) for the 4-bit page modes at
// head_dim 128: NVFP4 (also the storage of NVFP4 4over6) and INT4
// per-token-head, with one or several causal queries per sequence.
//
// Sources (web pages, by title and section):
//  "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化": "K 与 V 的量化误差进入 attention 的位置不同"
//     (A = softmax(QK^T/sqrt(d) + M), O = AV; M the causal mask of chunked prefill and
//     speculative decoding, 使用前仍应确认), "KV 的写入与读取路径" (unpack the payload and
//     apply block and tensor scales inside the attention load path), "GQA" (the query heads
//     of a group share each K/V page);
//  "KV 量化" (rustineverything.app), scale 和数据放在一起: int4_per_token_head.
//
// Design (GB300).  One CTA of 256 threads per (KV split, kv head, sequence);
// all the sequence's queries and the GQA group's heads form the N = 16 NT
// columns of both products.  A 128-token tile (8 pages) is the unit:
//  - TMA brings the tile's 8 (page, kv head) blocks into a 3-stage ring
//    (64-byte rows, 64-byte swizzle);
//  - thread (token t, half) dequantizes half of token t's key row to exact f16
//    and stores it into tensor memory, lane t (the A operand of S = K Q^T,
//    M = 128 tokens, K = 128 channels); Q^T is the B operand in shared memory;
//  - thread (channel d, half) dequantizes channel d of half the tile's values
//    into lane d (the A operand of O^T = V^T P^T, M = 128 channels, K = 128
//    tokens);
//  - one thread issues the tcgen05.mma of both products; completion is
//    signalled on mbarriers (tcgen05.commit);
//  - thread (token t, half) reads its row of S from tensor memory, applies the
//    online softmax against a CTA-wide reference max that moves only when a
//    score exceeds it by more than SLACK (rare: a vote at a barrier), and
//    writes P as an f16 hi + lo pair into the B operand P^T;
//  - O^T accumulates in tensor memory over the whole split and is read once.
// The codes are exact in f16 (E2M1 x E4M3 block scale; signed 4-bit integers);
// the per-token INT4 scales go to the fp32 scores (K) and into P (V); the
// per-tensor NVFP4 scales to the scores (K) and the output (V).
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kD = 128;
constexpr int kPage = 16;
constexpr int kTilePages = 8;
constexpr int kTileTok = kTilePages * kPage;
constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kPageSlot = 2560;                      // a block's slot in a stage: 5 periods of the 64-byte swizzle
constexpr int kStageBytes = kTilePages * kPageSlot;  // 20 KB
constexpr int kMaxPages = 1024;                      // pages per split (ids kept in shared memory)
constexpr int kCoreK = 144;                          // bytes between core matrices along K in a B operand
constexpr int kGroup8 = 16 * kCoreK;                 // bytes of one 8-row group of a B operand (K = 128)
constexpr int kTmemCols = 256;                       // A_K 64 | A_V 64 | S N | O N or 2N (| A_V)
constexpr int kColAK = 0, kColAV = 64, kColS = 128;
// Block layout inside a page block (bytes; 4-bit modes, D = 128, P = 16)
constexpr int kVOff = kPage * kD / 2;  // V payload (token-pair rows of 128 bytes)
constexpr int kSOff = kPage * kD;      // scales

template <int MODE>
struct Mode {
  static constexpr bool FP4 = MODE == KVQ_NVFP4;
  static constexpr int BLK = (int)block_bytes(MODE, kPage, kD);
  // P enters A V scaled by 2^PSHIFT; the reference max may lag the row max by
  // up to SLACK (log2 units), so f16 must hold 2^(PSHIFT + SLACK) times the
  // largest V factor folded into P (INT4: the per-token scale, at most 65504/7
  // for fp16 inputs).
  static constexpr int pshift(bool f32io) { return FP4 ? (f32io ? 14 : 10) : (f32io ? 0 : -2); }
  static constexpr int slack(bool f32io) { return f32io ? 0 : 4; }
};

template <int NT, bool QF32, bool FP4>
struct Smem {
  static constexpr int N = 16 * NT;
  static constexpr int BOP = (N / 8) * kGroup8;  // bytes of one K-major B operand (N rows x 128, f16)
  static constexpr int POP = N * kTileTok * 2;    // bytes of P hi (128 token rows x N, f16); P lo the same
  // P hi and lo as one B operand of 2N columns (one MMA per k-step of A V, hi
  // products in O's first N columns, lo in the next N) where tensor memory allows
  static constexpr bool FUSE = 128 + 3 * N <= kTmemCols;
  static constexpr int PC = FUSE ? 2 * N : N;  // columns of a P operand
  static constexpr int OC = FUSE ? 2 * N : N;  // columns of O
  static constexpr int STAGE = 0;
  static constexpr int QT = STAGE + kStages * kStageBytes;
  static constexpr int PT = QT + (QF32 ? 2 : 1) * BOP;  // P hi, then lo (then the second buffer's)
  // A V and P are double-buffered (tile i in buffer i % 2) where the second A V
  // fits in the tensor-memory columns above O and two CTAs still fit an SM
  static constexpr int SINGLE = PT + 2 * POP + (FP4 ? 8 * 64 * 4 : 0) + 4 * N * 4 + kMaxPages * 4 + 1024;
  static constexpr bool DB = 128 + N + OC + 64 <= kTmemCols && 2 * (SINGLE + 2 * POP + 1024) <= 228 * 1024;
  static constexpr int VTAB = PT + (DB ? 4 : 2) * POP;  // NVFP4 V block-scale pairs [8 blocks][64 pairs]
  static constexpr int WRED = VTAB + (FP4 ? 8 * 64 * 4 : 0);
  static constexpr int PAGES = WRED + 4 * N * 4;
  static constexpr int BYTES = PAGES + kMaxPages * 4;
  static constexpr size_t dynamic() { return (size_t)BYTES + 1024; }
};

__device__ __forceinline__ uint32_t lop3_sel(uint32_t w, uint32_t k1, uint32_t k2) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(k1), "r"(k2));
  return r;
}
// Nibble 0 (bits 0-3) and nibble 4 (bits 16-19) of w, two's-complement 4-bit
// codes, as an exact f16 pair: the lop3 flips each code's top bit (code + 8)
// under the f16 exponent of 1024; one subtraction of 1032 leaves the code.
__device__ __forceinline__ uint32_t s4pair_lo(uint32_t w) {
  return h2_as_u32(__hsub2(u32_as_h2(lop3_sel(w, 0x000F000Fu, 0x64086408u)), u32_as_h2(0x64086408u)));
}

template <int MODE, int NT, bool QF32>
__global__ void __launch_bounds__(kThreads, 2) umma_decode_kernel(const __grid_constant__ DecodeArgs a,
                                                                   const __grid_constant__ CUtensorMap tmap) {
  using Md = Mode<MODE>;
  using L = Smem<NT, QF32, Md::FP4>;
  constexpr int N = 16 * NT, CPT = N / 2;
  constexpr int BLK = Md::BLK;
  constexpr int PSHIFT = Md::pshift(QF32);
  constexpr float SLACK = (float)Md::slack(QF32);
  constexpr uint32_t IDESC = umma_idesc_f16(128, N);
  constexpr uint32_t IDESC_PV = umma_idesc_f16_bmn(128, L::PC);
  constexpr int P_LBO = (L::PC / 8) * 128;  // P: 8-token groups (K) after the column groups (MN, 128 B apart)
  constexpr int P_LO = L::FUSE ? (N / 8) * 128 : L::POP;  // P lo: columns N.. of the operand, or its own
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage = sm + L::STAGE;
  uint8_t* qt = sm + L::QT;
  uint8_t* pt = sm + L::PT;
  uint32_t* vtab = reinterpret_cast<uint32_t*>(sm + L::VTAB);
  float* wred = reinterpret_cast<float*>(sm + L::WRED);
  int* pages = reinterpret_cast<int*>(sm + L::PAGES);
  __shared__ uint64_t full_bar[kStages];
  __shared__ uint64_t qk_bar, pv_bar[2];  // A V of tile i commits on pv_bar[i % 2]
  __shared__ uint32_t tmem_base_s;

  const int split = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127, half = tid >> 7;  // token (or channel) of this thread, and its half of the work
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  uint8_t* pool = const_cast<uint8_t*>(a.pool);
  pdl_launch_dependents();

  const int nq = a.nq, G = a.G, Nr = G * nq;  // real columns: (query i, head g) -> r = i G + g
  int n = a.seq_lens[seq];
  const int lim = min(a.max_seq_len, a.max_pages * kPage);
  if (n > lim || n < 0) {
    if (tid == 0 && split == 0 && kvh == 0) set_error(pool, KVQ_DEVERR_SEQ_LEN);
    n = n < 0 ? 0 : lim;
  }
  const int t_begin = split * a.tokens_per_split;
  const int t_end = min(n, t_begin + a.tokens_per_split);
  if (t_begin >= t_end) {
    if (a.num_splits == 1) {  // empty sequence: zero output rows
      for (int idx = tid; idx < Nr * kD; idx += kThreads) {
        const int r = idx / kD, d = idx % kD;
        const long long o = ((long long)(seq * nq + r / G) * a.Hq + (long long)kvh * G + r % G) * kD + d;
        store_out(a, o, 0.0f);
      }
    }
    return;
  }
  const int p0 = t_begin / kPage;
  const int np = (t_end + kPage - 1) / kPage - p0;  // pages of this split (<= kMaxPages by the plan)
  const int ntiles = (np + kTilePages - 1) / kTilePages;

  for (int k = tid; k < np; k += kThreads) {
    int pid = __ldg(a.block_table + (long long)seq * a.max_pages + p0 + k);
    if (pid < 0 || pid >= a.num_pages) {
      set_error(pool, KVQ_DEVERR_PAGE_RANGE);
      pid = -1;
    }
    pages[k] = pid;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[s], kTilePages);  // one arrival per page
    mbar_init(&qk_bar, 1);
    mbar_init(&pv_bar[0], 1);
    mbar_init(&pv_bar[1], 1);
    mbar_fence_init();
    prefetch_tmap(&tmap);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  // Q^T (B operand of S = K Q^T): row c = (r & 1) CPT + (r >> 1) holds query row r
  // (zero rows for r >= Nr); element (c, k) at (c % 8) 16 + (k % 8) 2 + (k / 8) kCoreK + (c / 8) kGroup8.
  for (int it = tid; it < N * 16; it += kThreads) {
    const int c = it >> 4, k8 = it & 15;
    const int r = 2 * (c % CPT) + c / CPT;
    uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
    if (r < Nr) {
      const long long qo = ((long long)(seq * nq + r / G) * a.Hq + (long long)kvh * G + r % G) * kD + 8 * k8;
      if constexpr (QF32) {
        const float4 u0 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + qo));
        const float4 u1 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + qo + 4));
        const float x[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 hh = __floats2half2_rn(x[2 * e], x[2 * e + 1]);
          const float2 hf = __half22float2(hh);
          h[e] = h2_as_u32(hh);
          l[e] = h2_as_u32(__floats2half2_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y));
        }
        hi = make_uint4(h[0], h[1], h[2], h[3]);
        lo = make_uint4(l[0], l[1], l[2], l[3]);
      } else {
        hi = __ldg(reinterpret_cast<const uint4*>(static_cast<const __half*>(a.q) + qo));
      }
    }
    const int off = (c & 7) * 16 + k8 * kCoreK + (c >> 3) * kGroup8;
    *reinterpret_cast<uint4*>(qt + off) = hi;
    if constexpr (QF32) *reinterpret_cast<uint4*>(qt + L::BOP + off) = lo;
  }
  fence_proxy_async_smem();  // Q^T written by the generic proxy, read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_s;
  const uint32_t tAK = tb + kColAK, tAV0 = tb + kColAV, tS = tb + kColS, tO = tb + kColS + N;

  // page p of tile i into stage i % kStages, by one lane of warp p: one arrival
  // with the page's bytes (none for a missing page) on the stage's barrier
  auto issue_page = [&](int i, int p) {
    uint64_t* bar = &full_bar[i % kStages];
    const int k = i * kTilePages + p;
    const int pid = k < np ? pages[k] : -1;
    mbar_arrive_expect_tx(bar, pid >= 0 ? (uint32_t)BLK : 0u);
    if (pid >= 0) {
      const long long r0 = (kHeaderBytes + ((long long)pid * a.Hkv + kvh) * BLK) / 64;
      tma_g2s_2d(stage + (i % kStages) * kStageBytes + p * kPageSlot, &tmap, 0, (int)r0, bar);
    }
  };
  if (elect_one())
    for (int i = 0; i < min(kStages, ntiles); ++i) issue_page(i, warp);
  __syncwarp();
  // B operand descriptors at k-step 0; k-step j starts 2 j kCoreK bytes further (the
  // start-address field holds bytes / 16 and never carries: shared addresses < 2^18)
  const uint64_t dQ = umma_sdesc(smem_u32(qt), kCoreK, kGroup8);
  const uint64_t dQlo = umma_sdesc(smem_u32(qt + (QF32 ? L::BOP : 0)), kCoreK, kGroup8);
  // P (B operand of O^T = V^T P^T) is MN-major: element (token k, column c) at
  // (c % 8) 2 + (k % 8) 16 + (c / 8) 128 + (k / 8) P_LBO, so each thread stores
  // its token's columns as whole 16-byte rows; k-step j starts 2 j P_LBO further
  // (the lo operand and the second buffer as start-address offsets in 16 B units)
  const uint64_t dP = umma_sdesc(smem_u32(pt), P_LBO, 128);
  constexpr uint64_t dPlo = L::POP >> 4;
  constexpr uint64_t kStep = (2 * kCoreK) >> 4;
  constexpr uint64_t kStepP = (2 * P_LBO) >> 4;

  float kfac = a.sm_log2, vfac = 1.0f;
  if constexpr (Md::FP4) {
    kfac *= *reinterpret_cast<const float*>(a.pool + kHdrKScaleOffset);
    vfac = *reinterpret_cast<const float*>(a.pool + kHdrVScaleOffset);
  }
  float m[CPT], l[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    m[k] = -1e30f;  // finite start: no inf - inf
    l[k] = 0.0f;
  }
  // this thread's columns: real ones first (k < nreal), each with its query's
  // causal end (query i sees the tokens before n - (nq - 1 - i))
  const int nreal = (Nr - half + 1) / 2;
  int climit[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) climit[k] = k < nreal ? n - (nq - 1 - (2 * k + half) / G) : 0;
  const int cmin = n - (nq - 1);  // the earliest query's end: tiles below it need no causal mask
  uint32_t qk_phase = 0;
  bool qk_pending = false, o_valid = false, timed_out = false;
  int last_pv = -1;  // the last tile whose A V was issued
  // A V of tile j has completed (and with it every earlier product)
  auto wait_pv = [&](int j) -> bool { return mbar_wait_bounded(&pv_bar[j & 1], (j >> 1) & 1); };

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kStages;
    const uint8_t* st = stage + s * kStageBytes;
    const int tok0 = t_begin + i * kTileTok;  // token of tile row 0
    bool ok = mbar_wait_bounded(&full_bar[s], (i / kStages) & 1);

    // ---- K: token `row`, channels 64 half .. + 63, into lane `row` of A_K
    {
      const uint8_t* pg = st + (row >> 4) * kPageSlot;
      const int r = row & 15, sw = (r >> 1) & 3;
      const uint4 c0 = *reinterpret_cast<const uint4*>(pg + r * 64 + 16 * ((2 * half) ^ sw));
      const uint4 c1 = *reinterpret_cast<const uint4*>(pg + r * 64 + 16 * ((2 * half + 1) ^ sw));
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t f[32];
      if constexpr (Md::FP4) {
        // block scales of blocks 4 half .. + 3 (16 channels = 8 columns each)
        const uint32_t sraw = *reinterpret_cast<const uint32_t*>(pg + kSOff + 8 * r + 4 * half);
        const __half2 s01 = u32_as_h2(e4m3x2_to_f16x2(sraw & 0xFFFFu));
        const __half2 s23 = u32_as_h2(e4m3x2_to_f16x2(sraw >> 16));
        const __half2 sc[4] = {__low2half2(s01), __high2half2(s01), __low2half2(s23), __high2half2(s23)};
#pragma unroll
        for (int mw = 0; mw < 8; ++mw) {
          uint32_t v[4];
          e2m1x8_to_f16x2x4(w[mw], v);
#pragma unroll
          for (int e = 0; e < 4; ++e) f[4 * mw + e] = h2_as_u32(__hmul2(u32_as_h2(v[e]), sc[mw >> 1]));
        }
      } else {
        // INT4 key word: channels 8m + 2i (nibble i) and 8m + 2i + 1 (nibble i + 4)
#pragma unroll
        for (int mw = 0; mw < 8; ++mw) {
          f[4 * mw + 0] = s4pair_lo(w[mw]);
          f[4 * mw + 1] = s4pair_lo(w[mw] >> 4);
          f[4 * mw + 2] = s4pair_lo(w[mw] >> 8);
          f[4 * mw + 3] = s4pair_lo(w[mw] >> 12);
        }
      }
      tmem_st<32>(tAK + lane_base + 32 * half, f);
    }
    // valid tokens of each page of the tile (0 for a missing page)
    auto page_valid = [&](int p) -> int {
      const int k = i * kTilePages + p;
      const int nv = min(kPage, t_end - (p0 + k) * kPage);
      return (k < np && pages[k] >= 0) ? nv : 0;
    };
    if constexpr (Md::FP4) {
      // V block-scale pairs of the tile: entry (block b, pair k) = f16x2 of the
      // scales of tokens 2k, 2k + 1 (0 past the valid tokens: their values vanish)
      for (int e = tid; e < 8 * 64; e += kThreads) {
        const int b = e >> 6, k = e & 63, p = k >> 3, t0 = 2 * (k & 7);
        const uint8_t* pg = st + p * kPageSlot;
        const int nv = page_valid(p);
        uint32_t s0 = pg[kSOff + kPage * 8 + ((8 * t0 + b) ^ 16)];
        uint32_t s1 = pg[kSOff + kPage * 8 + ((8 * (t0 + 1) + b) ^ 16)];
        if (t0 >= nv) s0 = 0;
        if (t0 + 1 >= nv) s1 = 0;
        vtab[e] = e4m3x2_to_f16x2(s0 | (s1 << 8));
      }
    }
    tmem_wait_st();
    tc_fence_before();
    if (__syncthreads_or(!ok)) {  // A_K and the scale table are complete (or a copy never arrived)
      timed_out = true;
      break;
    }
    if (warp == 0) {
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int j = 0; j < 8; ++j) umma_f16_ts(tS, tAK + 8 * j, dQ + j * kStep, IDESC, j > 0 ? 1u : 0u);
        if constexpr (QF32) {
#pragma unroll
          for (int j = 0; j < 8; ++j) umma_f16_ts(tS, tAK + 8 * j, dQlo + j * kStep, IDESC, 1u);
        }
        tc_commit(&qk_bar);
      }
      __syncwarp();
    }
    qk_pending = true;

    // ---- V: channel `row`, tokens 64 half .. + 63, into lane `row` of A_V
    //      (once the previous tile's A V has released A_V and P^T)
    const int buf = L::DB ? (i & 1) : 0;
    const uint32_t tAV = buf ? tb + kColS + N + L::OC : tAV0;  // the second A V: columns above O
    if (i - (L::DB ? 2 : 1) >= 0 && i - (L::DB ? 2 : 1) <= last_pv) ok = wait_pv(i - (L::DB ? 2 : 1)) && ok;
    {
      const int d = row;
      uint32_t f[32];
#pragma unroll
      for (int pl = 0; pl < 4; ++pl) {
        const uint8_t* pg = st + (4 * half + pl) * kPageSlot + kVOff;
        if constexpr (Md::FP4) {
          const uint4* tab = reinterpret_cast<const uint4*>(vtab + (d >> 4) * 64 + 32 * half + 8 * pl);
          const uint4 t01 = tab[0], t23 = tab[1];
          const uint32_t sp[8] = {t01.x, t01.y, t01.z, t01.w, t23.x, t23.y, t23.z, t23.w};
#pragma unroll
          for (int pr = 0; pr < 8; ++pr) {
            const uint32_t byte = pg[128 * pr + (d ^ ((pr & 3) << 4))];
            uint32_t v;
            asm("{\n\t.reg .b8 b0;\n\tcvt.u8.u32 b0, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}" : "=r"(v) : "r"(byte));
            f[8 * pl + pr] = h2_as_u32(__hmul2(u32_as_h2(v), u32_as_h2(sp[pr])));
          }
        } else {
#pragma unroll
          for (int pr = 0; pr < 8; ++pr) {
            const uint32_t word =
                *reinterpret_cast<const uint32_t*>(pg + 128 * pr + ((4 * (d >> 2)) ^ ((pr & 3) << 4)));
            f[8 * pl + pr] = s4pair_lo(word >> (4 * (d & 3)));
          }
        }
      }
      tmem_st<32>(tAV + lane_base + 32 * half, f);
    }

    // ---- scores of token `row` for this thread's columns
    ok = mbar_wait_bounded(&qk_bar, qk_phase) && ok;
    qk_phase ^= 1;
    qk_pending = false;
    tc_fence_after();
    float sc[CPT];
    // a token past the split's end or on a missing page: its stage bytes may be
    // stale (any bit pattern), so its scores and its V factor are replaced
    const bool tok_ok = (row & 15) < page_valid(row >> 4);
    {
      uint32_t sv[CPT];
      tmem_ld<CPT>(tS + lane_base + CPT * half, sv);
      tmem_wait_ld();
      const int p = row >> 4;
      const int pos = tok0 + row;
      float f = kfac;
      if constexpr (!Md::FP4) f *= *reinterpret_cast<const float*>(st + p * kPageSlot + kSOff + 4 * (row & 15));
      if (tok0 + kTileTok <= cmin) {  // CTA-uniform: the whole tile precedes every query
#pragma unroll
        for (int k = 0; k < CPT; ++k) sc[k] = (tok_ok && k < nreal) ? __uint_as_float(sv[k]) * f : -INFINITY;
      } else {
#pragma unroll
        for (int k = 0; k < CPT; ++k) sc[k] = (tok_ok && pos < climit[k]) ? __uint_as_float(sv[k]) * f : -INFINITY;
      }
    }
    bool exceed = false;
#pragma unroll
    for (int k = 0; k < CPT; ++k) exceed |= sc[k] > m[k] + SLACK;
    // ---- P = 2^(s - m + PSHIFT) into P^T (hi, lo), token `row` = K index, with
    //      the current reference maxima; pk keeps each column's p for l
    float vs = 1.0f;
    if constexpr (!Md::FP4)
      vs = tok_ok ? *reinterpret_cast<const float*>(st + (row >> 4) * kPageSlot + kSOff + 64 + 4 * (row & 15)) : 0.0f;
    float pk[CPT];
    auto write_p = [&]() {
      uint32_t ph[CPT / 2], pl[CPT / 2];  // f16 pairs of columns (2e, 2e + 1): hi, lo
#pragma unroll
      for (int e = 0; e < CPT / 2; ++e) {
        float x[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int k = 2 * e + u;
          pk[k] = ex2(sc[k] + ((float)PSHIFT - m[k]));  // ex2(-inf) = 0: masked and padding columns
          x[u] = pk[k];
          if constexpr (!Md::FP4) x[u] *= vs;
        }
        const float h0 = __uint_as_float(__float_as_uint(x[0]) & 0xFFFFE000u);
        const float h1 = __uint_as_float(__float_as_uint(x[1]) & 0xFFFFE000u);
        ph[e] = h2_as_u32(__floats2half2_rn(h0, h1));
        pl[e] = h2_as_u32(__floats2half2_rn(x[0] - h0, x[1] - h1));
      }
      const int kb = (row & 7) * 16 + (row >> 3) * P_LBO + (CPT * half / 8) * 128;
#pragma unroll
      for (int q = 0; q < CPT / 8; ++q) {
        *reinterpret_cast<uint4*>(pt + buf * 2 * L::POP + kb + 128 * q) =
            make_uint4(ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
        *reinterpret_cast<uint4*>(pt + buf * 2 * L::POP + P_LO + kb + 128 * q) =
            make_uint4(pl[4 * q], pl[4 * q + 1], pl[4 * q + 2], pl[4 * q + 3]);
      }
      tmem_wait_st();            // A_V (and a rescaled O) are in tensor memory
      fence_proxy_async_smem();  // P^T, written by the generic proxy, is read by the tensor core
      tc_fence_before();
    };
    write_p();
    // One barrier completes A_V and P^T and the stage's reads, and votes on
    // the maxima: where a score passed its reference max by more than SLACK
    // (rare; always on the first tile) the maxima move, O and l are rescaled
    // and P is written again.
    if (__syncthreads_or(exceed || !ok)) {
      if (__syncthreads_or(!ok)) {
        timed_out = true;
        break;
      }
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const float v = warp_max_xor(sc[k], 1, 16);
        if (lane == 0) wred[(warp & 3) * N + CPT * half + k] = v;
      }
      __syncthreads();
      float alpha[CPT];
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const int c = CPT * half + k;
        const float tmax = fmaxf(fmaxf(wred[c], wred[N + c]), fmaxf(wred[2 * N + c], wred[3 * N + c]));
        const float mn = fmaxf(m[k], tmax);
        alpha[k] = ex2(m[k] - mn);
        m[k] = mn;
        l[k] *= alpha[k];
      }
      if (o_valid) {  // O^T columns of this half, channel `row`, once every A V issued is complete
        if (__syncthreads_or(!wait_pv(last_pv))) {
          timed_out = true;
          break;
        }
#pragma unroll
        for (int part = 0; part < (L::FUSE ? 2 : 1); ++part) {  // hi products, then lo
          uint32_t ov[CPT];
          tmem_ld<CPT>(tO + part * N + lane_base + CPT * half, ov);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < CPT; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha[k]);
          tmem_st<CPT>(tO + part * N + lane_base + CPT * half, ov);
        }
      }
      write_p();
      __syncthreads();  // P^T with the new maxima (and the rescaled O) complete
    }
#pragma unroll
    for (int k = 0; k < CPT; ++k) l[k] += pk[k];
    if (warp == 0) {
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dPb = dP + (uint64_t)((buf * 2 * L::POP) >> 4);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          umma_f16_ts(tO, tAV + 8 * j, dPb + j * kStepP, IDESC_PV, (o_valid || j > 0) ? 1u : 0u);
        if constexpr (!L::FUSE) {
#pragma unroll
          for (int j = 0; j < 8; ++j) umma_f16_ts(tO, tAV + 8 * j, dPb + dPlo + j * kStepP, IDESC_PV, 1u);
        }
        tc_commit(&pv_bar[i & 1]);
      }
      __syncwarp();
    }
    if (i + kStages < ntiles) {  // refill this stage (every thread is done reading it): page `warp`
      if (elect_one()) issue_page(i + kStages, warp);
      __syncwarp();
    }
    last_pv = i;
    o_valid = true;
  }

  // outstanding products must complete before tensor memory is read or freed
  bool ok_end = true;
  if (qk_pending) ok_end = mbar_wait_bounded(&qk_bar, qk_phase) && ok_end;
  if (last_pv >= 0) ok_end = wait_pv(last_pv) && ok_end;
  tc_fence_after();
  if (__syncthreads_or(!ok_end)) timed_out = true;
  if (timed_out) {
    if (tid == 0) set_error(pool, KVQ_DEVERR_TIMEOUT);
  } else {
    // l: sum over the 128 token rows of each column (the stage ring is idle now)
    float* lred = reinterpret_cast<float*>(stage);  // [N][128]
#pragma unroll
    for (int k = 0; k < CPT; ++k) lred[(CPT * half + k) * 128 + row] = l[k];
    __syncthreads();
    float* lsum = lred + N * 128;  // [N]
    for (int c = warp; c < N; c += kThreads / 32) {
      float v = lred[c * 128 + lane] + lred[c * 128 + 32 + lane] + lred[c * 128 + 64 + lane] + lred[c * 128 + 96 + lane];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) lsum[c] = v;
    }
    __syncthreads();
    // O^T row `row` = channel d, this half's columns
    if (o_valid) {
      uint32_t ov[CPT];
      tmem_ld<CPT>(tO + lane_base + CPT * half, ov);
      tmem_wait_ld();
      if constexpr (L::FUSE) {  // O = the hi products + the lo products
        uint32_t ol[CPT];
        tmem_ld<CPT>(tO + N + lane_base + CPT * half, ol);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < CPT; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) + __uint_as_float(ol[k]));
      }
      const int d = row;
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const int r = 2 * k + half;
        if (r >= Nr) continue;
        const float Lc = lsum[CPT * half + k];
        const float O = __uint_as_float(ov[k]) * vfac;
        const long long qrow = (long long)(seq * nq + r / G) * a.Hq + (long long)kvh * G + r % G;
        if (a.num_splits == 1) {
          const float res = Lc > 0.0f ? O / Lc : 0.0f;
          store_out(a, qrow * kD + d, res);
        } else {
          const long long pi = qrow * a.num_splits + split;
          store_ws(a, a.ws_o + (pi * kD + d), Lc > 0.0f ? O : 0.0f);
          if (d == 0) {
            store_ws(a, a.ws_ml + (2 * pi), m[k]);
            store_ws(a, a.ws_ml + (2 * pi + 1), Lc);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kTmemCols);
}

// Resident CTAs per SM, from the per-SM limits (shared memory with its per-CTA
// reserve, registers, threads) and the 512 tensor-memory columns; the
// occupancy query answers 1 for this kernel on GB300 although two CTAs run
// side by side (measured), so it is not used.
template <int MODE, int NT, bool QF32>
int resident() {
  static std::atomic<int> cached{0};
  int r = cached.load(std::memory_order_relaxed);
  if (r > 0) return r;
  auto kern = umma_decode_kernel<MODE, NT, QF32>;
  constexpr size_t smem = Smem<NT, QF32, Mode<MODE>::FP4>::dynamic();
  cudaFuncAttributes fa;
  int dev = 0, smem_sm = 0, reserve = 0, regs_sm = 0, thr_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaFuncGetAttributes(&fa, kern) == cudaSuccess &&
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&reserve, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) == cudaSuccess) {
    const long long per_cta = (long long)fa.sharedSizeBytes + (long long)smem + reserve;
    r = 512 / kTmemCols;
    r = (int)std::min<long long>(r, smem_sm / per_cta);
    r = std::min(r, regs_sm / std::max(1, fa.numRegs * kThreads));
    r = std::min(r, thr_sm / kThreads);
  } else {
    (void)cudaGetLastError();
    r = 1;
  }
  r = std::max(r, 1);
  cached.store(r, std::memory_order_relaxed);
  return r;
}

template <int MODE, int NT, bool QF32>
cudaError_t launch(const kvq_cache* c, const DecodeArgs& a, cudaStream_t s) {
  auto kern = umma_decode_kernel<MODE, NT, QF32>;
  constexpr size_t smem = Smem<NT, QF32, Mode<MODE>::FP4>::dynamic();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.Hkv, a.B / a.nq);
  kern<<<grid, kThreads, smem, s>>>(a, c->tmap);
  return cudaGetLastError();
}

template <int MODE, bool QF32>
int resident_nt(int nt) {
  return nt == 1 ? resident<MODE, 1, QF32>() : nt == 2 ? resident<MODE, 2, QF32>() : resident<MODE, 4, QF32>();
}

template <int MODE, bool QF32>
cudaError_t launch_nt(const kvq_cache* c, const DecodeArgs& a, cudaStream_t s, int nt) {
  return nt == 1 ? launch<MODE, 1, QF32>(c, a, s) : nt == 2 ? launch<MODE, 2, QF32>(c, a, s)
                                                            : launch<MODE, 4, QF32>(c, a, s);
}

}  // namespace

int umma_column_tiles(int group, int num_queries) {
  const int nr = group * num_queries;
  return nr <= 16 ? 1 : nr <= 32 ? 2 : nr <= 64 ? 4 : 0;
}

// Several queries per sequence only: with one query the products have 8 real
// columns, and the tile's conversion and synchronisation work outweigh the
// MMAs it saves against the mma.sync kernel (measured on GB300: NVFP4 B = 32 x
// 32K, 504 us here against 257 us; with 4 queries 730 us against 917 us).
bool umma_decode_eligible(const kvq_cache* c, int num_q_heads, int num_queries) {
  if (num_queries < 2) return false;
  const int m = c->cfg.mode;
  if (c->cfg.head_dim != kD || c->cfg.page_size != kPage || c->rows_per_block == 0) return false;
  if (m != KVQ_NVFP4 && m != KVQ_NVFP4_4OVER6 && m != KVQ_INT4_PER_TOKEN_HEAD) return false;
  return umma_column_tiles(num_q_heads / c->cfg.num_kv_heads, num_queries) > 0;
}

int umma_resident_ctas(const kvq_cache* c, int num_q_heads, int num_queries) {
  const int nt = umma_column_tiles(num_q_heads / c->cfg.num_kv_heads, num_queries);
  const bool f32 = c->cfg.io_dtype == KVQ_F32;
  if (c->cfg.mode == KVQ_INT4_PER_TOKEN_HEAD)
    return f32 ? resident_nt<KVQ_INT4_PER_TOKEN_HEAD, true>(nt) : resident_nt<KVQ_INT4_PER_TOKEN_HEAD, false>(nt);
  return f32 ? resident_nt<KVQ_NVFP4, true>(nt) : resident_nt<KVQ_NVFP4, false>(nt);
}

int umma_max_pages_per_split() { return kMaxPages; }

cudaError_t launch_umma_decode(const kvq_cache* c, const DecodeArgs& a, cudaStream_t s) {
  const int nt = umma_column_tiles(a.G, a.nq);
  const bool f32 = c->cfg.io_dtype == KVQ_F32;
  cudaError_t e;
  if (c->cfg.mode == KVQ_INT4_PER_TOKEN_HEAD)
    e = f32 ? launch_nt<KVQ_INT4_PER_TOKEN_HEAD, true>(c, a, s, nt) : launch_nt<KVQ_INT4_PER_TOKEN_HEAD, false>(c, a, s, nt);
  else
    e = f32 ? launch_nt<KVQ_NVFP4, true>(c, a, s, nt) : launch_nt<KVQ_NVFP4, false>(c, a, s, nt);
  return e;
}

}  // namespace kvq
