// kvq_internal.h -- host-side definitions shared by the libkvq translation
// units: the cache descriptor behind the opaque kvq_cache handle, the decode
// plan, and the kernel launchers each .cu file provides.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"

struct kvq_cache {
  kvq_cache_config cfg;
  uint8_t* base;        // device pool (header at byte 0)
  size_t bytes;         // bytes the caller provided
  size_t block_bytes;   // bytes of one (page, kv head) block
  int row_bytes;        // width of a page row as seen by the decode TMA (0: no tensor map)
  int rows_per_block;   // block_bytes / row_bytes
  CUtensorMap tmap;  // 2-D view of the pool as rows of row_bytes (64-byte aligned type)
};

namespace kvq {

struct DecodePlan {
  int num_splits;        // KV splits per (sequence, kv head)
  int tokens_per_split;  // multiple of the page size
  size_t workspace_bytes;
  // the splits of each query row run as one thread-block cluster and merge
  // through distributed shared memory (no combine kernel, workspace unused)
  bool cluster_merge = false;
};

int num_sms();

cudaError_t launch_write(const kvq_cache* c, const void* k, const void* v, const int32_t* slots,
                         int num_tokens, cudaStream_t stream);
cudaError_t launch_kvarn_append(const kvq_cache* c, const void* k, const void* v, const int32_t* slots,
                                const int32_t* seq_ids, int num_tokens, void* tail, int num_seqs,
                                cudaStream_t stream);
// Debug builds: one thread stores a byte just past a one-byte span inside the
// pool header (byte 40); the check must skip it and set KVQ_DEVERR_BOUNDS.
cudaError_t launch_bounds_selftest(uint8_t* pool, cudaStream_t stream);
cudaError_t launch_error_stats(const kvq_cache* c, const void* k, const void* v, const int32_t* slots, int num_tokens,
                               kvq_error_stats* out, cudaStream_t stream);
cudaError_t launch_amax(const void* x, int dtype, size_t n, float* out, cudaStream_t stream);
cudaError_t launch_scales_from_amax(uint8_t* pool, const float* amax_k, const float* amax_v, float div,
                                    cudaStream_t stream);

// num_seqs counts sequences; each has num_queries query rows (multi-query decode).
DecodePlan plan_decode(const kvq_cache* c, int num_seqs, int num_q_heads, int max_seq_len, int num_queries = 1);
cudaError_t launch_decode(const kvq_cache* c, const DecodePlan& plan, const void* q, const int32_t* block_table,
                          int max_pages, const int32_t* seq_lens, int num_seqs, int num_q_heads,
                          int max_seq_len, float softmax_scale, void* out, int out_dtype, void* workspace,
                          cudaStream_t stream, const void* kvarn_tail = nullptr, int num_queries = 1);

}  // namespace kvq
