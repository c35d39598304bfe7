/*
 * kvq.h -- C ABI of libkvq: quantize-on-write into a paged KV cache and paged
 * decode attention that reads the packed low-bit cache and folds
 * dequantization into its load path.  One process, one NVIDIA GB300 GPU
 * (sm_103a).
 *
 * Sources of the operations (web pages, by title and section):
 *  [P1] "KV Cache 量化深度解析：Per-Tensor、Per-Token-Head 与 NVFP4":
 *       sec. 二 (the KVQuantMode enum: NONE, FP8_PER_TENSOR, INT8/FP8
 *       PER_TOKEN_HEAD, NVFP4), sec. 2.1, 2.2, 2.3.
 *  [P2] "KVarN：华为推出的原生 vLLM KV-cache 量化后端，打破性能与精度的权衡":
 *       技术原理 (tile, Hadamard rotation, variance normalisation, asymmetric
 *       RTN), 配置与部署 (preset kvarn_k4v2_g128), 注意事项 (tile = page = 128).
 *  [P3] "KV Cache 量化 · LLM Glossary": s = max|x|/127, q = clip(round(x/s)),
 *       dequantize while loading inside the attention kernel.
 *  [P4] "KV 量化" (rustineverything.app): 写和读 (the write call takes the
 *       cache dtype and the k/v scales, the read multiplies by the descale;
 *       FP8 stored as uint8 bit patterns), per-token-head and NVFP4 scales
 *       stored inside the page next to the data.
 *  [P5] "NVFP4 KV Cache：Blackwell 上的 4-bit 缓存量化": two-level scaling,
 *       KV write/read paths, attention A = softmax(QK^T/sqrt(d)), O = AV;
 *       an unsupported combination is an immediate error, not a silent
 *       fallback; "用一组数直观看缩放的作用" (the nvfp4_4over6 mode picks a
 *       max/6 or max/4 block scale by reconstruction error).
 *  [P4] also names int4_per_token_head: head_size/2 bytes of data plus one
 *       fp32 scale per token and kv head.
 *
 * Conventions
 *  - Every call returns a kvq_status; KVQ_OK is 0.  On error,
 *    kvq_last_error() returns a message (thread-local, valid until the next
 *    call on the same thread).  Argument errors are detected on the host
 *    before anything is launched.
 *  - Pointers named dev_* or documented as device pointers are CUDA device
 *    memory owned by the caller.  The library never allocates device memory:
 *    the cache pool and the decode workspace are caller buffers (the one
 *    library-owned buffer is the fixed scratch array described at
 *    kvq_decode_attention_noalloc).  A kvq_cache handle owns only a small
 *    host-side descriptor.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All device
 *    work is enqueued on it asynchronously, unless a call says otherwise.
 *  - There is no fallback path: an unsupported combination of mode, head_dim,
 *    page_size or dtype returns KVQ_ERR_UNSUPPORTED.
 *  - Errors that only the device can see (a slot or page id out of range, a
 *    KVarN write that is not whole tiles, a seq_len above its bound) never
 *    fault: the offending token or tile is skipped and a bit is set in the
 *    cache's device error word; kvq_cache_read_errors() fetches it.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int kvq_status;
#define KVQ_OK 0
#define KVQ_ERR_INVALID_ARG 1   /* null pointer, negative size, misaligned buffer, ... */
#define KVQ_ERR_UNSUPPORTED 2   /* mode / head_dim / page_size / dtype combination */
#define KVQ_ERR_MODE_MISMATCH 3 /* call mode differs from the cache's mode */
#define KVQ_ERR_CAPACITY 4      /* buffer too small for the layout or the plan */
#define KVQ_ERR_CUDA 5          /* a CUDA runtime/driver call failed */
#define KVQ_ERR_DEVICE_CHECK 6  /* the device error word is non-zero */

/* Quantization modes ([P1] sec. 二 enum values, plus the KVarN preset of [P2]). */
typedef enum {
  KVQ_FP8_PER_TENSOR = 1,      /* E4M3 payload, one fp32 scale per side (K, V) */
  KVQ_INT8_PER_TOKEN_HEAD = 2, /* int8 payload, fp32 scale per token x kv head, s = max|x|/127 */
  KVQ_FP8_PER_TOKEN_HEAD = 3,  /* E4M3 payload, fp32 scale per token x kv head, s = max|x|/448 */
  KVQ_NVFP4 = 4,               /* E2M1 payload, E4M3 scale per 16 values, fp32 global scale */
  KVQ_INT4_PER_TOKEN_HEAD = 5, /* signed 4-bit payload, fp32 scale per token x kv head, s = max|x|/7 */
  KVQ_NVFP4_4OVER6 = 6,        /* NVFP4 storage; each block scale is max/6 or max/4, by error */
  KVQ_KVARN_K4V2_G128 = 16     /* 4-bit keys, 2-bit values, 128-token tiles */
} kvq_mode;

typedef enum { KVQ_F16 = 0, KVQ_F32 = 1 } kvq_dtype;

/* Device error bits (kvq_cache_read_errors). */
#define KVQ_DEVERR_SLOT_RANGE 0x1u   /* a write slot >= num_pages * page_size */
#define KVQ_DEVERR_PAGE_RANGE 0x2u   /* a block_table entry outside [0, num_pages) */
#define KVQ_DEVERR_PARTIAL_TILE 0x4u /* KVarN: a write or a sequence that is not whole tiles, or an
                                        append carrying rows of two tiles of one sequence */
#define KVQ_DEVERR_SEQ_LEN 0x8u      /* a seq_len above max_seq_len or max_pages * page_size */
#define KVQ_DEVERR_TIMEOUT 0x10u     /* a bounded wait on a copy ran out (work skipped) */
#define KVQ_DEVERR_SEQ_ID 0x20u      /* kvq_kvarn_append: a seq_id outside [0, num_seqs) */
#define KVQ_DEVERR_BOUNDS 0x40u      /* debug build only: a store fell outside the buffer its
                                        arguments describe (skipped); see kvq_debug_build */

typedef struct {
  int32_t num_pages;    /* pages in the pool */
  int32_t page_size;    /* tokens per page: 16 (modes 1-4) or 128 (KVarN) */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* D: 32 or 128 (modes 1-4), 128 (KVarN) */
  int32_t mode;         /* kvq_mode */
  int32_t io_dtype;     /* kvq_dtype of the K/V written and of the decode query */
} kvq_cache_config;

typedef struct kvq_cache kvq_cache;

/* Pool layout (little-endian, version 1).  The pool is a 256-byte header
 * followed by one block per (page, kv head), page-major:
 *   block(p, h) at byte 256 + (p * num_kv_heads + h) * block_bytes.
 * Token t of page p is row t of that block.  Per mode (P = page_size, D = head_dim):
 *   FP8 per-tensor : K[P][D] e4m3 | V[P][D] e4m3                    (2PD bytes)
 *   INT8 / FP8 PTH : K[P][D] | V[P][D] | K scale[P] f32 | V scale[P] f32
 *   NVFP4, 4over6  : K[P][D/2] | V[P/2][D] | K s_b[P][D/16] e4m3 | V s_b[P][D/16] e4m3
 *   INT4 PTH       : K[P][D/2] | V[P/2][D] | K scale[P] f32 | V scale[P] f32
 *   KVarN (P=D=128): K[128][64] u4 | V[128][32] u2 |
 *                    K scale[D] zero[D] c[D] r[P] f32 | V scale[P] zero[P] r[P] c[D] f32
 * 4-bit codes: NVFP4 K (E2M1) the even head_dim index in the low nibble;
 * NVFP4 V byte [k][d] holds channel d of tokens 2k (low nibble) and 2k+1 --
 * the pairing decode's tensor-core fragments take, with no nibble shuffling.
 * INT4 (two's complement) in 32-bit little-endian words, nibble k = bits
 * 4k..4k+3: a K row word m holds channel 8m + 2k in nibble k < 4 and
 * 8m + 2(k-4) + 1 in nibble k >= 4; a V pair row [k] word m holds channel
 * 4m + k of token 2k' = 2k in nibble k < 4 and channel 4m + k - 4 of token
 * 2k + 1 in nibble k >= 4 -- the orders one lop3 turns into f16 pairs.
 * 2-bit codes: element 4i+j in bits 2j..2j+1 of byte i.  The header holds, at byte 16 and
 * 20, the per-tensor K and V scales (FP8 per-tensor s; NVFP4 s_t), and at
 * byte 12 the device error word.  This is the same content as the in-page
 * layouts of [P4] (data plus one fp32 scale per token-head; head_size/2 bytes
 * of FP4 then head_size/16 bytes of E4M3 block scales), with each kind of
 * field gathered into its own 16-byte-aligned sub-array. */

const char* kvq_last_error(void);
int kvq_version(void); /* layout/ABI version, currently 1 */

/* 1 when the library was built with -DKVQ_DEBUG=1, else 0.  In such a build
 * every global store of every kernel first checks that its bytes lie inside
 * the buffer its arguments describe (the pool, the tail buffer, the output,
 * the workspace); a store that does not is skipped and KVQ_DEVERR_BOUNDS is
 * set in the cache's error word.  It stands in for a memory checker: an
 * indexing fault shows up as a flag instead of a corrupted neighbour.  A
 * release build checks nothing and never sets KVQ_DEVERR_BOUNDS. */
int kvq_debug_build(void);

/* Debug builds only (KVQ_ERR_UNSUPPORTED otherwise): one kernel tries a store
 * one byte past the end of the pool's header span, which lies inside the
 * pool's memory, and so must set KVQ_DEVERR_BOUNDS and leave the byte as it
 * was.  Lets a test see that the checks are live.  Enqueued on `stream`. */
kvq_status kvq_debug_bounds_selftest(kvq_cache* cache, void* stream);

/* Bytes of the pool for `cfg` (header included), and of one (page, kv head)
 * block.  No device work. */
kvq_status kvq_cache_bytes(const kvq_cache_config* cfg, size_t* bytes);
kvq_status kvq_cache_block_bytes(const kvq_cache_config* cfg, size_t* bytes);

/* Bind a cache descriptor to the caller's device buffer `dev_buf` (at least
 * kvq_cache_bytes bytes, 256-byte aligned).  Writes the header (scales = 1.0,
 * error word = 0) synchronously; page contents are left as they are.
 * `*out` is freed with kvq_cache_free, which never touches device memory. */
kvq_status kvq_cache_alloc(const kvq_cache_config* cfg, void* dev_buf, size_t bytes, kvq_cache** out);
kvq_status kvq_cache_free(kvq_cache* cache);

/* Per-tensor scales ([P1] sec. 2.1 K_fp8 = K/scale; [P5] s_t), written into
 * the header on `stream`.  Used by KVQ_FP8_PER_TENSOR (s) and the two NVFP4
 * modes (s_t); other modes ignore them.  Scales must be finite and > 0. */
kvq_status kvq_cache_set_tensor_scales(kvq_cache* cache, float k_scale, float v_scale, void* stream);

/* amax = max |x| over n elements of `x` (device, dtype kvq_dtype), written
 * to the device float *dev_out (overwritten, not accumulated).  Exact. */
kvq_status kvq_tensor_amax(const void* x, int dtype, size_t n, float* dev_out, void* stream);

/* Set the header's scales from device amax values without a host round trip:
 * FP8 per-tensor s = amax/448, NVFP4 (both modes) s_t = amax/(448*6); an amax of 0 gives
 * 1.0.  Both pointers are device floats (e.g. from kvq_tensor_amax). */
kvq_status kvq_cache_set_tensor_scales_from_amax(kvq_cache* cache, const float* dev_amax_k,
                                                 const float* dev_amax_v, void* stream);

/* Copy the device error word to *flags (synchronises `stream`); if `clear`,
 * reset it to 0 afterwards. */
kvq_status kvq_cache_read_errors(kvq_cache* cache, uint32_t* flags, int clear, void* stream);

/* Quantize-on-write ([P4] 写和读; [P1] sec. 2.1-2.3; [P2] 技术原理).
 *  k, v          device [num_tokens][num_kv_heads][head_dim], io_dtype of the cache
 *  slot_mapping  device int32 [num_tokens]: slot = page * page_size + row;
 *                a negative slot skips the token; a slot past the pool skips it
 *                and sets KVQ_DEVERR_SLOT_RANGE.
 *  mode          must equal the cache's mode (else KVQ_ERR_MODE_MISMATCH).
 * Per mode: FP8 per-tensor q = E4M3(x/s) with the header scale; INT8/FP8
 * per-token-head s = max(max|x|, 1e-8)/127 (or /448), q = clip(rint(x/s)) (or
 * E4M3(x/s)); INT4 per-token-head s = max(max|x|, 1e-8)/7, q = clip(rint(x/s),
 * -7, 7); NVFP4 s_b = E4M3(max_block|x| / (6 s_t)), q = E2M1(x/(s_t s_b));
 * NVFP4 4over6: the same block coded with s_b = E4M3(max_block|x| / (4 s_t))
 * as well, keeping the coding whose fp32 sum of squared reconstruction errors
 * (x - s_t s_b q)^2, summed as a pairwise tree of neighbours, is smaller
 * (max/6 on a tie);
 * KVarN: num_tokens must be a multiple of 128 and every 128 consecutive tokens
 * must fill one page in order (slot_mapping[128i + j] = 128 page + j); a tile
 * that does not is skipped with KVQ_DEVERR_PARTIAL_TILE.  All divisions are
 * IEEE round-to-nearest; results are bit-identical to the specification. */
kvq_status kvq_quantize_write(kvq_cache* cache, const void* k, const void* v,
                              const int32_t* slot_mapping, int num_tokens, int mode, void* stream);

/* Decode plan: how many KV splits per (sequence, kv head), the tokens per
 * split, and the workspace bytes kvq_decode_attention needs for these sizes
 * (0 when a single split suffices, and 0 when the splits of each query row
 * merge on chip: 2 to 8 splits of the one-query kernel whose CTAs are all
 * resident at once run as one thread-block cluster per row, so that no split
 * partial goes through memory and no combine kernel is launched).
 * max_seq_len is a host-side upper bound of every seq_len. */
kvq_status kvq_decode_plan(const kvq_cache* cache, int num_seqs, int num_q_heads, int max_seq_len,
                           int* num_splits, int* tokens_per_split, size_t* workspace_bytes);
kvq_status kvq_decode_workspace_bytes(const kvq_cache* cache, int num_seqs, int num_q_heads,
                                      int max_seq_len, size_t* bytes);

/* Paged decode attention over the packed cache ([P5] "K 与 V 的量化误差..."
 * A = softmax(QK^T/sqrt(d)), O = AV, one query per sequence; [P3]/[P5]:
 * dequantization happens in the kernel's load path, no dequantized copy of
 * the cache is made).
 *  q            device [num_seqs][num_q_heads][head_dim], io_dtype of the cache
 *  block_table  device int32 [num_seqs][max_pages]: page ids of each sequence
 *  seq_lens     device int32 [num_seqs]; 0 gives a zero output row
 *  max_seq_len  host upper bound of seq_lens (<= max_pages * page_size)
 *  softmax_scale  usually 1/sqrt(head_dim)
 *  out          device [num_seqs][num_q_heads][head_dim], dtype out_dtype
 *  workspace    device scratch of >= the planned bytes (may be NULL if 0)
 * GQA: query head h reads kv head h / (num_q_heads / num_kv_heads), which
 * must divide evenly with a group of at most 8.  KVarN: every seq_len must be
 * a multiple of 128 (whole tiles), the query is rotated by the same
 * normalised Hadamard transform and the output rotated back. */
kvq_status kvq_decode_attention(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                int max_pages, const int32_t* seq_lens, int num_seqs,
                                int num_q_heads, int max_seq_len, int mode, float softmax_scale,
                                void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Multi-query decode: num_queries queries per sequence, as in speculative
 * decoding or a short prefill chunk, over the same packed pages ([P5] "K 与 V
 * 的量化误差进入 attention 的位置不同": A = softmax(QK^T/sqrt(d) + M), O = AV,
 * with M the causal mask).  q and out are [num_seqs][num_queries][num_q_heads]
 * [head_dim]; query i of sequence b stands at position seq_len_b - num_queries
 * + i and attends to tokens 0 .. seq_len_b - num_queries + i (none, output 0,
 * when that is negative).  Other arguments and rules are those of
 * kvq_decode_attention; num_seqs * num_queries <= 65535.  KVQ_KVARN_K4V2_G128
 * reads whole tiles only (every seq_len a multiple of 128, no open tile); a
 * query's causal prefix may end inside the last tile, whose later tokens it
 * does not see.  NVFP4 (and 4over6) and INT4 at head_dim 128 with
 * group * num_queries <= 64 read each page once for all the sequence's
 * queries (tensor-core columns = queries x heads); the other modes run each
 * query as one row of the decode grid over its causal prefix, the rows of a
 * sequence side by side so that the pages they share are mostly served from
 * L2.  Plan and workspace: kvq_decode_multi_plan /
 * kvq_decode_multi_workspace_bytes. */
kvq_status kvq_decode_multi_plan(const kvq_cache* cache, int num_seqs, int num_queries, int num_q_heads,
                                 int max_seq_len, int* num_splits, int* tokens_per_split, size_t* workspace_bytes);
kvq_status kvq_decode_multi_workspace_bytes(const kvq_cache* cache, int num_seqs, int num_queries,
                                            int num_q_heads, int max_seq_len, size_t* bytes);
kvq_status kvq_decode_attention_multi(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                      int max_pages, const int32_t* seq_lens, int num_seqs, int num_queries,
                                      int num_q_heads, int max_seq_len, int mode, float softmax_scale,
                                      void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* ---- KVarN open tiles ---------------------------------------------------
 * [P2] 注意事项: a KVarN tile is exactly one 128-token page, and the backend
 * keeps a small fixed decode workspace.  A sequence's last, incomplete tile is
 * therefore held raw in a caller-owned tail buffer until its 128th token
 * arrives, when it is quantized into its page; decode reads the quantized
 * tiles plus the raw tail rows.
 *
 * Tail buffer (device, caller-owned, io_dtype): K rows [num_seqs][128][Hkv][D]
 * followed by V rows of the same shape; row r of sequence b holds token
 * 128 * floor(seq_len_b / 128) + r of that sequence, as written. */
kvq_status kvq_kvarn_tail_bytes(const kvq_cache* cache, int num_seqs, size_t* bytes);

/* Append tokens to their sequences' open tiles.  Token i (k, v [num_tokens][Hkv][D])
 * belongs to sequence seq_ids[i] at slot slot_mapping[i] = 128 * page + r: it is
 * copied to row r of that sequence's tail, and if r == 127 the tile is complete
 * and the sequence's 128 tail rows are quantized into `page` exactly as a
 * whole-tile kvq_quantize_write would.  Within one call a sequence's tokens
 * must belong to one tile (a decode step appends one token per sequence; a
 * prefill writes its whole tiles with kvq_quantize_write and appends the rest);
 * a tile completed by a call that also carries rows of another tile of the
 * same sequence is not written and sets KVQ_DEVERR_PARTIAL_TILE (its rows may
 * already be overwritten in the tail).  A negative
 * slot skips the token; a slot past the pool (KVQ_DEVERR_SLOT_RANGE) or a
 * seq_id outside [0, num_seqs) (KVQ_DEVERR_SEQ_ID) skips it and flags it.
 * Cache mode must be KVQ_KVARN_K4V2_G128; `tail` is 16-byte aligned and at
 * least kvq_kvarn_tail_bytes(num_seqs). */
kvq_status kvq_kvarn_append(kvq_cache* cache, const void* k, const void* v, const int32_t* slot_mapping,
                            const int32_t* seq_ids, int num_tokens, void* tail, int num_seqs, void* stream);

/* KVarN decode over whole tiles plus each sequence's open tile: any seq_len;
 * its first seq_len - seq_len % 128 tokens are read from the quantized pages
 * (as kvq_decode_attention does) and the last seq_len % 128 from rows 0.. of
 * the sequence's tail (raw, in the input domain).  The tail must hold
 * num_seqs sequences.  Workspace: kvq_kvarn_decode_workspace_bytes (never 0:
 * the tail is merged with the tiles' partial results by a second kernel). */
kvq_status kvq_kvarn_decode_workspace_bytes(const kvq_cache* cache, int num_seqs, int num_q_heads,
                                            int max_seq_len, size_t* bytes);
kvq_status kvq_kvarn_decode_attention(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                      int max_pages, const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                      int max_seq_len, float softmax_scale, const void* tail, void* out,
                                      int out_dtype, void* workspace, size_t workspace_bytes, void* stream);

/* ---- Tensor-level quantization error ([P5] "量化误差该怎样测", 张量层: MSE and
 * normalised MSE, max absolute error, cosine similarity, zero ratio,
 * clipping/saturation ratio, scale distribution, by head; K and V counted
 * separately).  For each token i with slot_mapping[i] >= 0 and each kv head,
 * the row the pool holds at that slot is dequantized and compared with the
 * row k[i] (v[i]) it was written from (KVarN rows are rotated back to the
 * input domain first).  dev_stats is a device array [2][num_kv_heads]
 * (index side * num_kv_heads + head, side 0 = K), zeroed by the call and then
 * accumulated; derived ratios are the caller's (e.g. NMSE = sum_sq_err /
 * sum_sq_ref, cosine = dot / sqrt(sum_sq_ref * sum_sq_deq)).  A slot past the
 * pool is skipped (KVQ_DEVERR_SLOT_RANGE).  Rows must have been written
 * (KVarN: whole tiles).  Diagnostic, not on the decode path. */
typedef struct {
  double count;           /* values compared */
  double sum_sq_err;      /* sum (x^ - x)^2 */
  double sum_sq_ref;      /* sum x^2 */
  double sum_sq_deq;      /* sum x^^2 */
  double dot;             /* sum x x^ */
  double max_abs_err;     /* max |x^ - x| */
  double zeros;           /* x^ == 0 */
  double saturated;       /* code at the largest magnitude of its grid (KVarN: the largest code) */
  double clipped;         /* saturated and |x| beyond |x^| by more than half the grid's last step
                             (INT8, INT4: s/2; E4M3: 16 s; NVFP4: one s_t s_b; KVarN: never) */
  double scale_hist[64];  /* stored scales by floor(log2 s) + 32, clamped to [0, 63]: per-token-head
                             and KVarN value scales once per row, NVFP4 block scales, KVarN key
                             scales once per tile (at its row 0), the per-tensor scale once per row */
} kvq_error_stats;
kvq_status kvq_tensor_error_stats(const kvq_cache* cache, const void* k, const void* v, const int32_t* slot_mapping,
                                  int num_tokens, kvq_error_stats* dev_stats, void* stream);

/* Allocation-free variant of kvq_decode_attention.  (No counterpart on the
 * source pages: this is an interface for callers, not part of the method.)
 * It is for callers that cannot allocate device memory when they decode --
 * for example code running inside a memory pool that was sized and frozen in
 * advance, or a host process embedding the library without any device
 * allocator of its own -- and so cannot provide the split-KV workspace.
 * Arguments and results are those of kvq_decode_attention minus the
 * workspace: the split partials go to a scratch array built into the library,
 * KVQ_NOALLOC_SCRATCH_BYTES bytes of device memory that every GPU loading the
 * library holds until the process exits.
 *  - A decode whose plan (kvq_decode_plan) needs more scratch than that is
 *    rejected with KVQ_ERR_CAPACITY before anything is launched.
 *  - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *    library routine.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - All calls share the one array and it keeps the last call's contents;
 *    calls whose kernels overlap on the GPU (different streams, or other
 *    host threads) race on it and must be serialised by the caller.
 *  - Each call writes every scratch entry it reads, so nothing has to be
 *    cleared between calls. */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)
kvq_status kvq_decode_attention_noalloc(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                        int max_pages, const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                        int max_seq_len, int mode, float softmax_scale, void* out,
                                        int out_dtype, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
