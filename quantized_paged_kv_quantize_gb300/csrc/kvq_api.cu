// kvq_api.cu -- the C ABI of libkvq (see include/kvq.h): argument validation,
// the pool header, the TMA tensor map of the pool, decode planning, launches.
// Every argument error is caught here, before any device work is enqueued.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace {

thread_local char g_err[512] = "";

kvq_status fail(kvq_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_mode(int m) {
  return m == KVQ_FP8_PER_TENSOR || m == KVQ_INT8_PER_TOKEN_HEAD || m == KVQ_FP8_PER_TOKEN_HEAD || m == KVQ_NVFP4 ||
         m == KVQ_INT4_PER_TOKEN_HEAD || m == KVQ_NVFP4_4OVER6 || m == KVQ_KVARN_K4V2_G128;
}

kvq_status check_config(const kvq_cache_config* cfg) {
  if (!cfg) return fail(KVQ_ERR_INVALID_ARG, "config is NULL");
  if (!valid_mode(cfg->mode)) return fail(KVQ_ERR_UNSUPPORTED, "unknown mode %d", cfg->mode);
  if (cfg->io_dtype != KVQ_F16 && cfg->io_dtype != KVQ_F32)
    return fail(KVQ_ERR_UNSUPPORTED, "io_dtype %d is not f16 or f32", cfg->io_dtype);
  if (cfg->num_pages <= 0 || cfg->num_kv_heads <= 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_pages and num_kv_heads must be positive");
  if (cfg->mode == KVQ_KVARN_K4V2_G128) {
    if (cfg->page_size != 128 || cfg->head_dim != 128)
      return fail(KVQ_ERR_UNSUPPORTED, "kvarn_k4v2_g128 needs page_size 128 and head_dim 128 (got %d, %d)",
                  cfg->page_size, cfg->head_dim);
  } else {
    if (cfg->page_size != 16)
      return fail(KVQ_ERR_UNSUPPORTED, "mode %d needs page_size 16 (got %d)", cfg->mode, cfg->page_size);
    if (cfg->head_dim != 32 && cfg->head_dim != 128)
      return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d unsupported (32 or 128)", cfg->head_dim);
  }
  return KVQ_OK;
}

size_t pool_bytes(const kvq_cache_config* c) {
  return kvq::kHeaderBytes +
         (size_t)c->num_pages * c->num_kv_heads * kvq::block_bytes(c->mode, c->page_size, c->head_dim);
}

kvq_status check_cache(const kvq_cache* c) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  return KVQ_OK;
}

// Argument checks shared by every decode entry point (each checks the cache
// mode itself first), in this order: sizes, the GQA group, max_seq_len against the block table, the
// output dtype, the softmax scale, then (only when there is work) the device
// pointers and their alignment.  `tail` is checked when `need_tail` is set
// (KVarN open tiles).  Returns KVQ_OK with *empty set when num_seqs is 0.
kvq_status check_decode_args(const kvq_cache* cache, const void* q, const int32_t* block_table, int max_pages,
                             const int32_t* seq_lens, int num_seqs, int num_q_heads, int max_seq_len,
                             float softmax_scale, const void* out, int out_dtype, bool need_tail,
                             const void* tail, bool* empty) {
  *empty = false;
  kvq_status s = check_cache(cache);
  if (s) return s;
  const kvq_cache_config& c = cache->cfg;
  if (num_seqs < 0 || max_pages < 0 || max_seq_len < 0) return fail(KVQ_ERR_INVALID_ARG, "negative size");
  if (num_q_heads <= 0 || num_q_heads % c.num_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                c.num_kv_heads);
  if (num_q_heads / c.num_kv_heads > 8)
    return fail(KVQ_ERR_UNSUPPORTED, "GQA group %d > 8", num_q_heads / c.num_kv_heads);
  if ((long long)max_seq_len > (long long)max_pages * c.page_size)
    return fail(KVQ_ERR_INVALID_ARG, "max_seq_len %d exceeds max_pages * page_size", max_seq_len);
  if (out_dtype != KVQ_F16 && out_dtype != KVQ_F32) return fail(KVQ_ERR_UNSUPPORTED, "out_dtype %d", out_dtype);
  if (!(softmax_scale > 0.0f) || softmax_scale > 3.0e38f)
    return fail(KVQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (num_seqs == 0) {
    *empty = true;
    return KVQ_OK;
  }
  if (!q || !block_table || !seq_lens || !out || (need_tail && !tail))
    return fail(KVQ_ERR_INVALID_ARG, need_tail ? "NULL q, table, lens, tail or out" : "NULL q, table, lens or out");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (need_tail && !aligned(tail, 16)))
    return fail(KVQ_ERR_INVALID_ARG, need_tail ? "q, tail and out must be 16-byte aligned"
                                               : "q and out must be 16-byte aligned");
  return KVQ_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

namespace kvq {
int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}
}  // namespace kvq

extern "C" {

const char* kvq_last_error(void) { return g_err; }

int kvq_version(void) { return 1; }

int kvq_debug_build(void) { return KVQ_DEBUG ? 1 : 0; }

kvq_status kvq_debug_bounds_selftest(kvq_cache* cache, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (!KVQ_DEBUG) return fail(KVQ_ERR_UNSUPPORTED, "a release build has no store checks (build with -DKVQ_DEBUG=1)");
  cudaError_t e = kvq::launch_bounds_selftest(cache->base, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return KVQ_OK;
}

kvq_status kvq_cache_bytes(const kvq_cache_config* cfg, size_t* bytes) {
  kvq_status s = check_config(cfg);
  if (s) return s;
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = pool_bytes(cfg);
  return KVQ_OK;
}

kvq_status kvq_cache_block_bytes(const kvq_cache_config* cfg, size_t* bytes) {
  kvq_status s = check_config(cfg);
  if (s) return s;
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = kvq::block_bytes(cfg->mode, cfg->page_size, cfg->head_dim);
  return KVQ_OK;
}

kvq_status kvq_cache_alloc(const kvq_cache_config* cfg, void* dev_buf, size_t bytes, kvq_cache** out) {
  kvq_status s = check_config(cfg);
  if (s) return s;
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!dev_buf) return fail(KVQ_ERR_INVALID_ARG, "dev_buf is NULL");
  if (!aligned(dev_buf, 256)) return fail(KVQ_ERR_INVALID_ARG, "dev_buf must be 256-byte aligned");
  const size_t need = pool_bytes(cfg);
  if (bytes < need) return fail(KVQ_ERR_CAPACITY, "pool needs %zu bytes, got %zu", need, bytes);

  kvq_cache* c = new (std::nothrow) kvq_cache();
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "out of host memory");
  c->cfg = *cfg;
  c->base = static_cast<uint8_t*>(dev_buf);
  c->bytes = bytes;
  c->block_bytes = kvq::block_bytes(cfg->mode, cfg->page_size, cfg->head_dim);
  c->row_bytes = 0;
  c->rows_per_block = 0;
  memset(&c->tmap, 0, sizeof c->tmap);

  // The decode kernels of modes 1-4 at head_dim 128 stage pages with a tiled
  // TMA copy: the pool seen as rows of 128 (1-byte codes) or 64 (4-bit codes) bytes,
  // one box = one (page, kv head) block, hardware-swizzled in shared memory.
  if (cfg->mode != KVQ_KVARN_K4V2_G128 && cfg->head_dim == 128) {
    const bool four_bit = cfg->mode == KVQ_NVFP4 || cfg->mode == KVQ_NVFP4_4OVER6 ||
                          cfg->mode == KVQ_INT4_PER_TOKEN_HEAD;
    const int rw = four_bit ? 64 : 128;
    const unsigned long long rows = need / rw;
    const int rpb = static_cast<int>(c->block_bytes / rw);
    if (rows >= (1ull << 31)) {
      delete c;
      return fail(KVQ_ERR_CAPACITY, "pool too large for 32-bit TMA row coordinates");
    }
    auto enc = tensor_map_encoder();
    if (!enc) {
      delete c;
      return fail(KVQ_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (no CUDA driver?)");
    }
    cuuint64_t dims[2] = {(cuuint64_t)rw, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)rw};
    cuuint32_t box[2] = {(cuuint32_t)rw, (cuuint32_t)rpb};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&c->tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dev_buf, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     rw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      delete c;
      return fail(KVQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    c->row_bytes = rw;
    c->rows_per_block = rpb;
  }

  unsigned char hdr[kvq::kHeaderBytes];
  memset(hdr, 0, sizeof hdr);
  const uint32_t magic = 0x3151564Bu, version = 1;
  const float one = 1.0f;
  memcpy(hdr + 0, &magic, 4);
  memcpy(hdr + 4, &version, 4);
  memcpy(hdr + 8, &cfg->mode, 4);
  memcpy(hdr + kvq::kHdrKScaleOffset, &one, 4);
  memcpy(hdr + kvq::kHdrVScaleOffset, &one, 4);
  memcpy(hdr + 24, &cfg->num_pages, 4);
  memcpy(hdr + 28, &cfg->page_size, 4);
  memcpy(hdr + 32, &cfg->num_kv_heads, 4);
  memcpy(hdr + 36, &cfg->head_dim, 4);
  cudaError_t e = cudaMemcpy(dev_buf, hdr, sizeof hdr, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "writing the pool header");
  }
  *out = c;
  return KVQ_OK;
}

kvq_status kvq_cache_free(kvq_cache* cache) {
  delete cache;
  return KVQ_OK;
}

kvq_status kvq_cache_set_tensor_scales(kvq_cache* cache, float k_scale, float v_scale, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || k_scale > 3.0e38f || v_scale > 3.0e38f)
    return fail(KVQ_ERR_INVALID_ARG, "scales must be finite and > 0");
  float sc[2] = {k_scale, v_scale};
  // pageable source: the copy is staged before this call returns, so `sc` may go out of scope
  cudaError_t e = cudaMemcpyAsync(cache->base + kvq::kHdrKScaleOffset, sc, sizeof sc, cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "setting tensor scales");
  return KVQ_OK;
}

kvq_status kvq_tensor_amax(const void* x, int dtype, size_t n, float* dev_out, void* stream) {
  if (dtype != KVQ_F16 && dtype != KVQ_F32) return fail(KVQ_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (!dev_out || (!x && n)) return fail(KVQ_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(x, 16) || !aligned(dev_out, 4)) return fail(KVQ_ERR_INVALID_ARG, "x must be 16-byte aligned");
  cudaError_t e = kvq::launch_amax(x, dtype, n, dev_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "amax launch");
  return KVQ_OK;
}

kvq_status kvq_cache_set_tensor_scales_from_amax(kvq_cache* cache, const float* dev_amax_k,
                                                 const float* dev_amax_v, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (!dev_amax_k || !dev_amax_v) return fail(KVQ_ERR_INVALID_ARG, "NULL amax pointer");
  if (cache->cfg.mode != KVQ_FP8_PER_TENSOR && cache->cfg.mode != KVQ_NVFP4 && cache->cfg.mode != KVQ_NVFP4_4OVER6)
    return fail(KVQ_ERR_MODE_MISMATCH, "mode %d has no per-tensor scale", cache->cfg.mode);
  const float div = cache->cfg.mode == KVQ_FP8_PER_TENSOR ? 448.0f : 2688.0f;
  cudaError_t e =
      kvq::launch_scales_from_amax(cache->base, dev_amax_k, dev_amax_v, div, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scale launch");
  return KVQ_OK;
}

kvq_status kvq_cache_read_errors(kvq_cache* cache, uint32_t* flags, int clear, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (!flags) return fail(KVQ_ERR_INVALID_ARG, "flags is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, cache->base + kvq::kHdrErrOffset, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(cache->base + kvq::kHdrErrOffset, 0, 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
  *flags = v;
  return KVQ_OK;
}

kvq_status kvq_quantize_write(kvq_cache* cache, const void* k, const void* v, const int32_t* slot_mapping,
                              int num_tokens, int mode, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (mode != cache->cfg.mode)
    return fail(KVQ_ERR_MODE_MISMATCH, "write mode %d but the cache holds mode %d", mode, cache->cfg.mode);
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return KVQ_OK;
  if (!k || !v || !slot_mapping) return fail(KVQ_ERR_INVALID_ARG, "NULL k, v or slot_mapping");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 4))
    return fail(KVQ_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  if (mode == KVQ_KVARN_K4V2_G128 && num_tokens % 128 != 0)
    return fail(KVQ_ERR_UNSUPPORTED, "kvarn_k4v2_g128 writes whole 128-token tiles (num_tokens %d)", num_tokens);
  cudaError_t e = kvq::launch_write(cache, k, v, slot_mapping, num_tokens, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "write launch");
  return KVQ_OK;
}

kvq_status kvq_tensor_error_stats(const kvq_cache* cache, const void* k, const void* v, const int32_t* slot_mapping,
                                  int num_tokens, kvq_error_stats* dev_stats, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  if (!dev_stats || !aligned(dev_stats, 8)) return fail(KVQ_ERR_INVALID_ARG, "dev_stats must be a non-NULL, 8-byte aligned device array");
  if (num_tokens > 0 && (!k || !v || !slot_mapping)) return fail(KVQ_ERR_INVALID_ARG, "NULL k, v or slot_mapping");
  if (num_tokens > 0 && (!aligned(k, 4) || !aligned(v, 4) || !aligned(slot_mapping, 4)))
    return fail(KVQ_ERR_INVALID_ARG, "k, v and slot_mapping must be 4-byte aligned");
  cudaError_t e = kvq::launch_error_stats(cache, k, v, slot_mapping, num_tokens, dev_stats,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "error statistics launch");
  return KVQ_OK;
}

kvq_status kvq_decode_plan(const kvq_cache* cache, int num_seqs, int num_q_heads, int max_seq_len, int* num_splits,
                           int* tokens_per_split, size_t* workspace_bytes) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (num_seqs < 0 || num_q_heads <= 0 || max_seq_len < 0)
    return fail(KVQ_ERR_INVALID_ARG, "bad sizes (num_seqs %d, num_q_heads %d, max_seq_len %d)", num_seqs,
                num_q_heads, max_seq_len);
  kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len);
  if (num_splits) *num_splits = p.num_splits;
  if (tokens_per_split) *tokens_per_split = p.tokens_per_split;
  if (workspace_bytes) *workspace_bytes = p.workspace_bytes;
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_bytes(const kvq_cache* cache, int num_seqs, int num_q_heads, int max_seq_len,
                                      size_t* bytes) {
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  return kvq_decode_plan(cache, num_seqs, num_q_heads, max_seq_len, nullptr, nullptr, bytes);
}

kvq_status kvq_decode_attention(const kvq_cache* cache, const void* q, const int32_t* block_table, int max_pages,
                                const int32_t* seq_lens, int num_seqs, int num_q_heads, int max_seq_len, int mode,
                                float softmax_scale, void* out, int out_dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (cache && mode != cache->cfg.mode)
    return fail(KVQ_ERR_MODE_MISMATCH, "decode mode %d but the cache holds mode %d", mode, cache->cfg.mode);
  bool empty = false;
  kvq_status s = check_decode_args(cache, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads, max_seq_len,
                                   softmax_scale, out, out_dtype, false, nullptr, &empty);
  if (s || empty) return s;
  kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len);
  if (p.workspace_bytes > 0) {
    if (!workspace) return fail(KVQ_ERR_CAPACITY, "workspace of %zu bytes required", p.workspace_bytes);
    if (workspace_bytes < p.workspace_bytes)
      return fail(KVQ_ERR_CAPACITY, "workspace needs %zu bytes, got %zu", p.workspace_bytes, workspace_bytes);
    if (!aligned(workspace, 16)) return fail(KVQ_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  }
  cudaError_t e = kvq::launch_decode(cache, p, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads,
                                     max_seq_len, softmax_scale, out, out_dtype, workspace,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KVQ_OK;
}

// ---- multi-query decode
kvq_status kvq_decode_multi_plan(const kvq_cache* cache, int num_seqs, int num_queries, int num_q_heads,
                                 int max_seq_len, int* num_splits, int* tokens_per_split, size_t* workspace_bytes) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (num_seqs < 0 || num_queries < 1 || num_q_heads <= 0 || max_seq_len < 0)
    return fail(KVQ_ERR_INVALID_ARG, "bad sizes (num_seqs %d, num_queries %d, num_q_heads %d, max_seq_len %d)",
                num_seqs, num_queries, num_q_heads, max_seq_len);
  if (num_q_heads % cache->cfg.num_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                cache->cfg.num_kv_heads);
  const kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len, num_queries);
  if (num_splits) *num_splits = p.num_splits;
  if (tokens_per_split) *tokens_per_split = p.tokens_per_split;
  if (workspace_bytes) *workspace_bytes = p.workspace_bytes;
  return KVQ_OK;
}

kvq_status kvq_decode_multi_workspace_bytes(const kvq_cache* cache, int num_seqs, int num_queries, int num_q_heads,
                                            int max_seq_len, size_t* bytes) {
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  return kvq_decode_multi_plan(cache, num_seqs, num_queries, num_q_heads, max_seq_len, nullptr, nullptr, bytes);
}

kvq_status kvq_decode_attention_multi(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                      int max_pages, const int32_t* seq_lens, int num_seqs, int num_queries,
                                      int num_q_heads, int max_seq_len, int mode, float softmax_scale, void* out,
                                      int out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (cache && mode != cache->cfg.mode)
    return fail(KVQ_ERR_MODE_MISMATCH, "decode mode %d but the cache holds mode %d", mode, cache->cfg.mode);
  if (num_queries < 1) return fail(KVQ_ERR_INVALID_ARG, "num_queries < 1");
  if ((long long)num_seqs * num_queries > 65535)
    return fail(KVQ_ERR_UNSUPPORTED, "num_seqs * num_queries = %lld > 65535", (long long)num_seqs * num_queries);
  bool empty = false;
  kvq_status s = check_decode_args(cache, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads, max_seq_len,
                                   softmax_scale, out, out_dtype, false, nullptr, &empty);
  if (s || empty) return s;
  const kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len, num_queries);
  if (p.workspace_bytes > 0) {
    if (!workspace || workspace_bytes < p.workspace_bytes)
      return fail(KVQ_ERR_CAPACITY, "workspace needs %zu bytes, got %zu", p.workspace_bytes,
                  workspace ? workspace_bytes : 0);
    if (!aligned(workspace, 16)) return fail(KVQ_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  }
  cudaError_t e = kvq::launch_decode(cache, p, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads,
                                     max_seq_len, softmax_scale, out, out_dtype, workspace,
                                     static_cast<cudaStream_t>(stream), nullptr, num_queries);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KVQ_OK;
}

// ---- KVarN open tiles
kvq_status kvq_kvarn_tail_bytes(const kvq_cache* cache, int num_seqs, size_t* bytes) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  if (cache->cfg.mode != KVQ_KVARN_K4V2_G128)
    return fail(KVQ_ERR_MODE_MISMATCH, "mode %d has no open tiles (KVarN only)", cache->cfg.mode);
  if (num_seqs < 0) return fail(KVQ_ERR_INVALID_ARG, "num_seqs < 0");
  const size_t esz = cache->cfg.io_dtype == KVQ_F16 ? 2 : 4;
  *bytes = (size_t)2 * num_seqs * 128 * cache->cfg.num_kv_heads * cache->cfg.head_dim * esz;
  return KVQ_OK;
}

kvq_status kvq_kvarn_append(kvq_cache* cache, const void* k, const void* v, const int32_t* slot_mapping,
                            const int32_t* seq_ids, int num_tokens, void* tail, int num_seqs, void* stream) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (cache->cfg.mode != KVQ_KVARN_K4V2_G128)
    return fail(KVQ_ERR_MODE_MISMATCH, "kvq_kvarn_append needs a KVarN cache (mode %d)", cache->cfg.mode);
  if (num_tokens < 0 || num_seqs < 0) return fail(KVQ_ERR_INVALID_ARG, "negative size");
  if (num_tokens == 0) return KVQ_OK;
  if (!k || !v || !slot_mapping || !seq_ids || !tail)
    return fail(KVQ_ERR_INVALID_ARG, "NULL k, v, slot_mapping, seq_ids or tail");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(tail, 16) || !aligned(slot_mapping, 4) || !aligned(seq_ids, 4))
    return fail(KVQ_ERR_INVALID_ARG, "k, v and tail must be 16-byte aligned");
  cudaError_t e = kvq::launch_kvarn_append(cache, k, v, slot_mapping, seq_ids, num_tokens, tail, num_seqs,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return KVQ_OK;
}

kvq_status kvq_kvarn_decode_workspace_bytes(const kvq_cache* cache, int num_seqs, int num_q_heads, int max_seq_len,
                                            size_t* bytes) {
  kvq_status s = check_cache(cache);
  if (s) return s;
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  if (cache->cfg.mode != KVQ_KVARN_K4V2_G128)
    return fail(KVQ_ERR_MODE_MISMATCH, "mode %d has no open tiles (KVarN only)", cache->cfg.mode);
  if (num_seqs < 0 || num_q_heads <= 0 || max_seq_len < 0)
    return fail(KVQ_ERR_INVALID_ARG, "bad sizes (num_seqs %d, num_q_heads %d, max_seq_len %d)", num_seqs,
                num_q_heads, max_seq_len);
  const kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len);
  *bytes = (size_t)num_seqs * num_q_heads * p.num_splits * (cache->cfg.head_dim + 2) * sizeof(float);
  return KVQ_OK;
}

kvq_status kvq_kvarn_decode_attention(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                      int max_pages, const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                      int max_seq_len, float softmax_scale, const void* tail, void* out,
                                      int out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (cache && cache->cfg.mode != KVQ_KVARN_K4V2_G128)
    return fail(KVQ_ERR_MODE_MISMATCH, "kvq_kvarn_decode_attention needs a KVarN cache (mode %d)", cache->cfg.mode);
  bool empty = false;
  kvq_status s = check_decode_args(cache, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads, max_seq_len,
                                   softmax_scale, out, out_dtype, true, tail, &empty);
  if (s || empty) return s;
  const kvq_cache_config& c = cache->cfg;
  const kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len);
  const size_t need = (size_t)num_seqs * num_q_heads * p.num_splits * (c.head_dim + 2) * sizeof(float);
  if (!workspace || workspace_bytes < need)
    return fail(KVQ_ERR_CAPACITY, "workspace needs %zu bytes, got %zu", need, workspace ? workspace_bytes : 0);
  if (!aligned(workspace, 16)) return fail(KVQ_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  cudaError_t e = kvq::launch_decode(cache, p, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads,
                                     max_seq_len, softmax_scale, out, out_dtype, workspace,
                                     static_cast<cudaStream_t>(stream), tail);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KVQ_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode.  Some callers cannot allocate device memory at the
// point where they decode: inference loops that sized and froze their memory
// pool up front, or hosts embedding the library with no device allocator of
// their own (no torch, no cudaMalloc in their process model).
// For them the split-KV scratch that kvq_decode_attention takes as a caller
// buffer lives instead in this fixed, library-owned device array.  Every GPU
// that loads the library keeps this array for the life of the process.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's
// name in host code is only a host-side handle, never a device address, so it
// is resolved once per device (with that device current) and cached.
kvq_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(KVQ_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the decode scratch");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_cache* cache, const void* q,
                                                   const int32_t* block_table, int max_pages,
                                                   const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                                   int max_seq_len, int mode, float softmax_scale, void* out,
                                                   int out_dtype, void* stream) {
  if (cache && mode != cache->cfg.mode)
    return fail(KVQ_ERR_MODE_MISMATCH, "decode mode %d but the cache holds mode %d", mode, cache->cfg.mode);
  bool empty = false;
  kvq_status s = check_decode_args(cache, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads, max_seq_len,
                                   softmax_scale, out, out_dtype, false, nullptr, &empty);
  if (s || empty) return s;
  kvq::DecodePlan p = kvq::plan_decode(cache, num_seqs, num_q_heads, max_seq_len);
  if (p.workspace_bytes > (size_t)KVQ_NOALLOC_SCRATCH_BYTES)
    return fail(KVQ_ERR_CAPACITY,
                "this decode needs %zu bytes of split scratch but the built-in scratch holds %zu; "
                "use kvq_decode_attention with a caller workspace",
                p.workspace_bytes, (size_t)KVQ_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (p.workspace_bytes > 0) {
    s = noalloc_scratch(&scratch);
    if (s) return s;
  }
  // Every scratch entry the combine step reads is written earlier in the same
  // call, so nothing needs clearing between calls.
  cudaError_t e = kvq::launch_decode(cache, p, q, block_table, max_pages, seq_lens, num_seqs, num_q_heads,
                                     max_seq_len, softmax_scale, out, out_dtype, scratch,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KVQ_OK;
}
