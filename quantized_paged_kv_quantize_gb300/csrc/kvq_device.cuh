// kvq_device.cuh -- device-side helpers shared by the libkvq kernels:
// pool layout constants, inline-PTX wrappers for the sm_103a instructions the
// kernels use (mbarrier, bulk / tensor TMA copies, E4M3/E2M1 conversions,
// mma.sync, movmatrix) and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

struct kvq_cache;

namespace kvq {

constexpr int kHeaderBytes = 256;
constexpr int kHdrErrOffset = 12;    // uint32 device error word
constexpr int kHdrKScaleOffset = 16; // float
constexpr int kHdrVScaleOffset = 20; // float

// Bytes of one (page, kv head) block; mirrors the layout documented in kvq.h.
__host__ __device__ constexpr size_t block_bytes(int mode, int P, int D) {
  return mode == KVQ_FP8_PER_TENSOR ? (size_t)2 * P * D
       : (mode == KVQ_INT8_PER_TOKEN_HEAD || mode == KVQ_FP8_PER_TOKEN_HEAD)
             ? (size_t)2 * P * D + (size_t)8 * P
       : (mode == KVQ_NVFP4 || mode == KVQ_NVFP4_4OVER6) ? (size_t)P * D + (size_t)P * D / 8
       : mode == KVQ_INT4_PER_TOKEN_HEAD ? (size_t)P * D + (size_t)8 * P
       : mode == KVQ_KVARN_K4V2_G128
             ? (size_t)P * D / 2 + (size_t)P * D / 4 + (size_t)4 * (3 * D + P) + (size_t)4 * (3 * P + D)
             : 0;
}

__device__ __forceinline__ void set_error(uint8_t* pool, uint32_t bits) {
  atomicOr(reinterpret_cast<uint32_t*>(pool + kHdrErrOffset), bits);
}

// ---------------------------------------------------------------- debug-build store checks
#ifndef KVQ_DEBUG
#define KVQ_DEBUG 0
#endif
// [lo, hi): the bytes one buffer of a kernel's arguments spans.
struct Span {
  uint8_t* lo;
  uint8_t* hi;
};
// In a debug build (-DKVQ_DEBUG=1) every global store checks that its bytes
// lie in the span of its buffer; one that does not is skipped and
// KVQ_DEVERR_BOUNDS is set in the pool's error word.  A release build checks
// nothing.
__device__ __forceinline__ bool in_span(const void* p, size_t bytes, const Span& s, const uint8_t* pool) {
#if KVQ_DEBUG
  const uint8_t* q = static_cast<const uint8_t*>(p);
  if (q < s.lo || q + bytes > s.hi) {
    set_error(const_cast<uint8_t*>(pool), KVQ_DEVERR_BOUNDS);
    return false;
  }
#else
  (void)p; (void)bytes; (void)s; (void)pool;
#endif
  return true;
}
template <typename T>
__device__ __forceinline__ void st_chk(T* p, const T& v, const Span& s, const uint8_t* pool) {
  if (in_span(p, sizeof(T), s, pool)) *p = v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- clusters
// This CTA's rank in its thread-block cluster and the cluster's CTA count.
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return (int)r;
}
// Every thread of every CTA of the cluster: shared-memory writes made before
// the barrier are visible to the cluster's CTAs after it (release / acquire).
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load the float at the address `p` has in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float* p, int rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after `limit` polls (each poll may itself suspend for
// a while) and returns false; callers then record KVQ_DEVERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit = 1u << 22) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) writes into the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// Untiled bulk copy global -> shared, completion counted on `bar`.
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem, const void* gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem)),
      "l"(gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Tiled 2-D tensor copy global -> shared (box given by the tensor map).
__device__ __forceinline__ void tma_g2s_2d(void* smem, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05 (5th-generation tensor cores)
// Tensor memory (TMEM): 128 lanes x 512 columns of 32 bits per SM; an address
// is (lane << 16) | column.  Warp w of a CTA reaches lanes 32 (w % 4) .. + 31.
// Allocation and release are warp-wide; the allocated base is written to
// shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Order tcgen05 operations around a thread barrier (before: issuing side; after: waiting side).
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// One arrival on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// One lane of the (converged) warp gets true: the tcgen05.mma issuer.  Issuing
// from a warp-uniform branch keeps the operands in uniform registers; a
// single-thread branch around the issue loop costs several times as many
// cycles per MMA (measured on GB300).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred P1;\n\telect.sync _|P1, 0xffffffff;\n\tselp.b32 %0, 1, 0, P1;\n\t}" : "=r"(pred));
  return pred != 0;
}
// Shared-memory matrix descriptor, no swizzle: 8-row x 16-byte core matrices,
// `lbo` bytes between core matrices along K, `sbo` bytes between 8-row groups.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}
// Instruction descriptor of kind::f16: f16 A and B (both K-major), f32 accumulate, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with B MN-major (transpose-B bit 16): B's N elements contiguous,
// core matrices of 8 K-rows x 16 bytes of N.
__host__ __device__ constexpr uint32_t umma_idesc_f16_bmn(int M, int N) { return umma_idesc_f16(M, N) | (1u << 16); }
// D[tmem] (+)= A[tmem] * B[smem]; accumulate when acc != 0.  One thread issues.
__device__ __forceinline__ void umma_f16_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 32 bits, N columns: thread i of the warp <-> lane (warp base + i), registers <-> columns.
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t* r);
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t* r);
template <>
__device__ __forceinline__ void tmem_st<4>(uint32_t t, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(t), "r"(r[0]), "r"(r[1]), "r"(r[2]),
               "r"(r[3])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t t, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(t), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t t, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(t),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t t, const uint32_t* r) {
  tmem_st<16>(t, r);
  tmem_st<16>(t + 16, r + 16);
}
template <>
__device__ __forceinline__ void tmem_ld<4>(uint32_t t, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(t)
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t t, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(t)
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t t, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(t)
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t t, uint32_t* r) {
  tmem_ld<16>(t, r);
  tmem_ld<16>(t + 16, r + 16);
}

// ---------------------------------------------------------------- dependent launch
// A decode kernel lets its split-combine kernel be scheduled before it ends
// (the combine's CTAs fill SMs during the decode's last wave); the combine
// waits for the whole decode grid and its memory before reading the partials.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` as a programmatic dependent of the previous kernel on `s`.
template <typename Arg>
inline cudaError_t launch_dependent(void (*kern)(Arg), dim3 grid, dim3 block, cudaStream_t s, const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, arg);
}

// ---------------------------------------------------------------- conversions
// Two fp32 -> two E4M3 (round-to-nearest-even, saturate to +-448);
// `hi` goes to the upper byte of the 16-bit result.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Four fp32 pairs -> eight E2M1 codes packed in a word; pair i gives byte i,
// the first value of each pair in the low nibble.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float* x) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}
// Two E4M3 (16 bits) -> f16x2, element order kept (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two_bytes)));
  return r;
}
// Four bytes of E2M1 pairs -> four f16x2 (byte i -> out[i], low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t* out) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// (a & m) | (b & ~m): LUT over (m, a, b) = (0xF0 & 0xCC) | (~0xF0 & 0xAA) = 0xCA
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(r) : "r"(m), "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
// One E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  return __low2float(u32_as_h2(e4m3x2_to_f16x2(byte & 0xFFu)));
}

// ---------------------------------------------------------------- tensor core
// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float ex2(float x) {  // 2^x on the SFU (rel. error ~2^-22), ex2(-inf) = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory loads of N 32-bit words.
template <int N>
__device__ __forceinline__ void lds(const uint8_t* p, uint32_t* w);
template <>
__device__ __forceinline__ void lds<4>(const uint8_t* p, uint32_t* w) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
}
template <>
__device__ __forceinline__ void lds<2>(const uint8_t* p, uint32_t* w) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  w[0] = u.x; w[1] = u.y;
}
template <>
__device__ __forceinline__ void lds<1>(const uint8_t* p, uint32_t* w) {
  w[0] = *reinterpret_cast<const uint32_t*>(p);
}

__device__ __forceinline__ float warp_max_xor(float v, int first, int last) {
  for (int o = first; o <= last; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Column of (head row h, channel d) in a [8][128] block where the warps of a
// decode CTA stage their m16n8 accumulators for the merge: the writing lanes
// hold rows 2 tq, 2 tq + 1 and channels 16 g' + 2 t, + 1 (g' a permutation of
// g), so XOR-ing channel bits 0..3 with (bits 5..6 of d, bits 1..2 of h) sends
// the 32 lanes of each store to 32 different banks (unswizzled: 16-way), and a
// row's 32 consecutive channels, read back, still fill the 32 banks once.
__device__ __forceinline__ int merge_col128(int h, int d) { return d ^ (((d >> 5) & 3) | ((h >> 1) << 2)); }

// Arguments of the decode kernels (passed by value as a __grid_constant__).
struct DecodeArgs {
  const uint8_t* pool;
  const void* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  float* ws_o;   // [B][Hq][S][D]
  float* ws_ml;  // [B][Hq][S][2]
  int num_pages, Hkv, Hq, G, B, max_pages, max_seq_len;
  int tokens_per_split, num_splits;
  int out_f32;
  int q_f32;
  float sm_log2;  // softmax_scale * log2(e)
  size_t block_bytes;
  int rows_per_block;
  // KVarN open tiles (kvq_kvarn_decode_attention): the tail buffer, K rows
  // [B][128][Hkv][D] then V rows, io dtype; null for whole-tile decode
  const uint8_t* tail;
  // queries per sequence (multi-query decode under the causal mask); B counts
  // query rows, B = sequences * nq
  int nq;
  // 1: the num_splits CTAs of a query row form one thread-block cluster and
  // merge their partials through distributed shared memory (no workspace)
  int cluster;
  // the output [B][Hq][D] and the split workspace, as spans (debug-build checks)
  Span out_span, ws_span;
};
// Checked stores of one output element and of one split partial.
__device__ __forceinline__ void store_out(const DecodeArgs& a, long long i, float v) {
  if (a.out_f32) st_chk(static_cast<float*>(a.out) + i, v, a.out_span, a.pool);
  else st_chk(static_cast<__half*>(a.out) + i, __float2half_rn(v), a.out_span, a.pool);
}
__device__ __forceinline__ void store_ws(const DecodeArgs& a, float* p, float v) { st_chk(p, v, a.ws_span, a.pool); }

// Split-KV merge of one (sequence, query head) row by a CTA of D threads,
// thread d owning channel d; base indexes the row's first split partial.
// M = max_s m_s, w_s = 2^(m_s - M), result sum_s o_s w_s / sum_s l_s w_s (0
// for a row with no tokens).  The weights go through shared memory (wts[D],
// red[D / 32]) in chunks of D splits and each thread keeps eight partial loads
// in flight, so a row costs a few memory round trips whatever the split count.
template <int D>
__device__ float merge_split_row(const DecodeArgs& a, long long base, int ns, float* wts, float* red,
                                 float* m_out = nullptr, float* l_out = nullptr) {
  constexpr int NW = D / 32;
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + base;
  float M = -INFINITY;
  for (int s = d; s < ns; s += D) M = fmaxf(M, ml[s].x);
  M = warp_max_xor(M, 1, 16);
  if (NW > 1) {
    if (lane == 0) red[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red[w]);
    __syncthreads();
  }
  float lsum = 0.0f, acc = 0.0f;
  if (M != -INFINITY) {  // uniform across the CTA
    for (int c = 0; c < ns; c += D) {
      float w = 0.0f;
      if (c + d < ns) {
        const float2 v = ml[c + d];
        w = exp2f(v.x - M);
        lsum += v.y * w;
      }
      wts[d] = w;
      __syncthreads();
      const int cn = min(D, ns - c);
      const float* src = a.ws_o + (base + c) * D + d;
      for (int j0 = 0; j0 < cn; j0 += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j0 + j < cn ? src[(long long)(j0 + j) * D] : 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc += v[j] * (j0 + j < cn ? wts[j0 + j] : 0.0f);
      }
      __syncthreads();
    }
  }
  for (int o = 16; o >= 1; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  if (NW > 1) {
    if (lane == 0) red[warp] = lsum;
    __syncthreads();
    lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) lsum += red[w];
  }
  if (m_out) {  // unnormalised: the caller merges more terms (M = -inf: no split had tokens)
    *m_out = M;
    *l_out = lsum;
    return acc;
  }
  return lsum > 0.0f ? acc / lsum : 0.0f;
}

// tcgen05 decode of the 4-bit page modes at head_dim 128 (kvq_decode_umma.cu):
// whether a cache and query shape take it, its resident CTAs per SM, the pages
// one split may hold, and the launch (decode only; the caller adds the combine).
bool umma_decode_eligible(const kvq_cache* c, int num_q_heads, int num_queries);
int umma_resident_ctas(const kvq_cache* c, int num_q_heads, int num_queries);
int umma_max_pages_per_split();
cudaError_t launch_umma_decode(const kvq_cache* c, const DecodeArgs& a, cudaStream_t stream);

// KVarN decode + combine (kvq_decode_kvarn.cu).
cudaError_t launch_kvarn_decode(const DecodeArgs& a, cudaStream_t stream);
int kvarn_resident_ctas();  // resident KVarN decode CTAs per SM (occupancy query)

}  // namespace kvq
