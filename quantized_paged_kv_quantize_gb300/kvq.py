"""Thin Python binding of libkvq (include/kvq.h) -- argument marshalling only.

Every function keeps the C name.  Device buffers are passed as torch CUDA
tensors (their data pointers are handed to the C ABI); torch serves only as
the allocator of device memory and the source of the current CUDA stream.  All
computation runs in the library's kernels.  If the shared library cannot be
loaded this module raises at import time: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
ERRORS = {1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_MODE_MISMATCH",
          4: "KVQ_ERR_CAPACITY", 5: "KVQ_ERR_CUDA", 6: "KVQ_ERR_DEVICE_CHECK"}
MODES = {
    "fp8_per_tensor": 1,
    "int8_per_token_head": 2,
    "fp8_per_token_head": 3,
    "nvfp4": 4,
    "int4_per_token_head": 5,
    "nvfp4_4over6": 6,
    "kvarn_k4v2_g128": 16,
}
KVQ_F16, KVQ_F32 = 0, 1
DEVERR = {0x1: "SLOT_RANGE", 0x2: "PAGE_RANGE", 0x4: "PARTIAL_TILE", 0x8: "SEQ_LEN", 0x10: "TIMEOUT",
          0x20: "SEQ_ID"}

EXPORTED = [
    "kvq_last_error", "kvq_version", "kvq_cache_bytes", "kvq_cache_block_bytes", "kvq_cache_alloc",
    "kvq_cache_free", "kvq_cache_set_tensor_scales", "kvq_tensor_amax",
    "kvq_cache_set_tensor_scales_from_amax", "kvq_cache_read_errors", "kvq_quantize_write",
    "kvq_decode_plan", "kvq_decode_workspace_bytes", "kvq_decode_attention", "kvq_decode_attention_noalloc",
    "kvq_kvarn_tail_bytes", "kvq_kvarn_append", "kvq_kvarn_decode_workspace_bytes", "kvq_kvarn_decode_attention",
    "kvq_decode_multi_plan", "kvq_decode_multi_workspace_bytes", "kvq_decode_attention_multi",
    "kvq_debug_build", "kvq_debug_bounds_selftest", "kvq_tensor_error_stats",
]


class KVQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{ERRORS.get(status, status)}: {msg}")
        self.status = status


class CacheConfig(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("io_dtype", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvq.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    cfgp = ctypes.POINTER(CacheConfig)
    sig = {
        "kvq_last_error": (ctypes.c_char_p, []),
        "kvq_version": (i32, []),
        "kvq_debug_build": (i32, []),
        "kvq_debug_bounds_selftest": (i32, [vp, vp]),
        "kvq_tensor_error_stats": (i32, [vp, vp, vp, vp, i32, vp, vp]),
        "kvq_cache_bytes": (i32, [cfgp, ctypes.POINTER(sz)]),
        "kvq_cache_block_bytes": (i32, [cfgp, ctypes.POINTER(sz)]),
        "kvq_cache_alloc": (i32, [cfgp, vp, sz, ctypes.POINTER(vp)]),
        "kvq_cache_free": (i32, [vp]),
        "kvq_cache_set_tensor_scales": (i32, [vp, f32, f32, vp]),
        "kvq_tensor_amax": (i32, [vp, i32, sz, vp, vp]),
        "kvq_cache_set_tensor_scales_from_amax": (i32, [vp, vp, vp, vp]),
        "kvq_cache_read_errors": (i32, [vp, ctypes.POINTER(ctypes.c_uint32), i32, vp]),
        "kvq_quantize_write": (i32, [vp, vp, vp, vp, i32, i32, vp]),
        "kvq_decode_plan": (i32, [vp, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                  ctypes.POINTER(sz)]),
        "kvq_decode_workspace_bytes": (i32, [vp, i32, i32, i32, ctypes.POINTER(sz)]),
        "kvq_decode_attention": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, f32, vp, i32, vp, sz, vp]),
        "kvq_decode_attention_noalloc": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, f32, vp, i32, vp]),
        "kvq_kvarn_tail_bytes": (i32, [vp, i32, ctypes.POINTER(sz)]),
        "kvq_decode_multi_plan": (i32, [vp, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                        ctypes.POINTER(sz)]),
        "kvq_decode_multi_workspace_bytes": (i32, [vp, i32, i32, i32, i32, ctypes.POINTER(sz)]),
        "kvq_decode_attention_multi": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, vp, i32, vp, sz,
                                             vp]),
        "kvq_kvarn_append": (i32, [vp, vp, vp, vp, vp, i32, vp, i32, vp]),
        "kvq_kvarn_decode_workspace_bytes": (i32, [vp, i32, i32, i32, ctypes.POINTER(sz)]),
        "kvq_kvarn_decode_attention": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, f32, vp, vp, i32, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


_lib = _load()


def lib():
    return _lib


def _check(status: int):
    if status != KVQ_OK:
        raise KVQError(status, _lib.kvq_last_error().decode(errors="replace"))


def _mode(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(dt) -> int:
    if dt in (torch.float16, "f16", KVQ_F16):
        return KVQ_F16
    if dt in (torch.float32, "f32", KVQ_F32):
        return KVQ_F32
    raise ValueError(f"unsupported dtype {dt}")


def make_config(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int, mode,
                io_dtype=KVQ_F16) -> CacheConfig:
    return CacheConfig(num_pages, page_size, num_kv_heads, head_dim, _mode(mode), _dtype_code(io_dtype))


def kvq_version() -> int:
    return _lib.kvq_version()


def kvq_debug_build() -> bool:
    """True when libkvq was built with -DKVQ_DEBUG=1 (store checks in every kernel)."""
    return bool(_lib.kvq_debug_build())


def kvq_debug_bounds_selftest(cache: "KVCache", stream=None):
    _check(_lib.kvq_debug_bounds_selftest(cache.handle, _stream(stream)))


# kvq_error_stats: nine fp64 sums and a 64-bin fp64 histogram per (side, kv head)
ERROR_STATS_FIELDS = ["count", "sum_sq_err", "sum_sq_ref", "sum_sq_deq", "dot", "max_abs_err", "zeros", "saturated",
                      "clipped"]
ERROR_STATS_DOUBLES = len(ERROR_STATS_FIELDS) + 64


def kvq_tensor_error_stats(cache: "KVCache", k, v, slot_mapping, stats: torch.Tensor, num_tokens: Optional[int] = None,
                           stream=None):
    """stats: float64 CUDA tensor [2, num_kv_heads, ERROR_STATS_DOUBLES], overwritten."""
    n = k.shape[0] if num_tokens is None else num_tokens
    assert stats.dtype == torch.float64 and stats.numel() >= 2 * cache.cfg.num_kv_heads * ERROR_STATS_DOUBLES
    _check(_lib.kvq_tensor_error_stats(cache.handle, _ptr(k), _ptr(v), _ptr(slot_mapping), n, _ptr(stats),
                                       _stream(stream)))


def kvq_cache_bytes(cfg: CacheConfig) -> int:
    out = ctypes.c_size_t()
    _check(_lib.kvq_cache_bytes(ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def kvq_cache_block_bytes(cfg: CacheConfig) -> int:
    out = ctypes.c_size_t()
    _check(_lib.kvq_cache_block_bytes(ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


class KVCache:
    """A cache descriptor bound to a caller-owned device pool (a uint8 tensor)."""

    def __init__(self, cfg: CacheConfig, pool: torch.Tensor, handle: int):
        self.cfg = cfg
        self.pool = pool
        self.handle = handle

    @property
    def mode(self) -> int:
        return self.cfg.mode

    def free(self):
        if self.handle:
            _lib.kvq_cache_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def kvq_cache_alloc(cfg: CacheConfig, pool: torch.Tensor) -> KVCache:
    h = ctypes.c_void_p()
    _check(_lib.kvq_cache_alloc(ctypes.byref(cfg), _ptr(pool), pool.numel() * pool.element_size(),
                                ctypes.byref(h)))
    return KVCache(cfg, pool, h.value)


def kvq_cache_free(cache: KVCache):
    cache.free()


def kvq_cache_set_tensor_scales(cache: KVCache, k_scale: float, v_scale: float, stream=None):
    _check(_lib.kvq_cache_set_tensor_scales(cache.handle, k_scale, v_scale, _stream(stream)))


def kvq_tensor_amax(x: torch.Tensor, out: torch.Tensor, stream=None):
    _check(_lib.kvq_tensor_amax(_ptr(x), _dtype_code(x.dtype), x.numel(), _ptr(out), _stream(stream)))


def kvq_cache_set_tensor_scales_from_amax(cache: KVCache, amax_k: torch.Tensor, amax_v: torch.Tensor,
                                          stream=None):
    _check(_lib.kvq_cache_set_tensor_scales_from_amax(cache.handle, _ptr(amax_k), _ptr(amax_v),
                                                      _stream(stream)))


def kvq_cache_read_errors(cache: KVCache, clear: bool = True, stream=None) -> int:
    flags = ctypes.c_uint32()
    _check(_lib.kvq_cache_read_errors(cache.handle, ctypes.byref(flags), int(clear), _stream(stream)))
    return flags.value


def kvq_quantize_write(cache: KVCache, k, v, slot_mapping, mode=None, num_tokens: Optional[int] = None,
                       stream=None):
    n = num_tokens if num_tokens is not None else int(slot_mapping.numel())
    _check(_lib.kvq_quantize_write(cache.handle, _ptr(k), _ptr(v), _ptr(slot_mapping), n,
                                   cache.mode if mode is None else _mode(mode), _stream(stream)))


def kvq_decode_plan(cache: KVCache, num_seqs: int, num_q_heads: int, max_seq_len: int):
    ns, tps, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _check(_lib.kvq_decode_plan(cache.handle, num_seqs, num_q_heads, max_seq_len, ctypes.byref(ns),
                                ctypes.byref(tps), ctypes.byref(ws)))
    return ns.value, tps.value, ws.value


def kvq_decode_workspace_bytes(cache: KVCache, num_seqs: int, num_q_heads: int, max_seq_len: int) -> int:
    ws = ctypes.c_size_t()
    _check(_lib.kvq_decode_workspace_bytes(cache.handle, num_seqs, num_q_heads, max_seq_len, ctypes.byref(ws)))
    return ws.value


def kvq_decode_attention(cache: KVCache, q, block_table, seq_lens, out, *, max_seq_len: int,
                         num_seqs: Optional[int] = None, num_q_heads: Optional[int] = None,
                         max_pages: Optional[int] = None, softmax_scale: Optional[float] = None,
                         mode=None, out_dtype=None, workspace=None, workspace_bytes: Optional[int] = None,
                         stream=None):
    B = num_seqs if num_seqs is not None else q.shape[0]
    Hq = num_q_heads if num_q_heads is not None else q.shape[1]
    mp = max_pages if max_pages is not None else block_table.shape[1]
    sm = softmax_scale if softmax_scale is not None else cache.cfg.head_dim ** -0.5
    od = _dtype_code(out.dtype) if out_dtype is None else _dtype_code(out_dtype)
    wb = workspace_bytes if workspace_bytes is not None else (
        0 if workspace is None else workspace.numel() * workspace.element_size())
    _check(_lib.kvq_decode_attention(cache.handle, _ptr(q), _ptr(block_table), mp, _ptr(seq_lens), B, Hq,
                                     max_seq_len, cache.mode if mode is None else _mode(mode), sm, _ptr(out),
                                     od, _ptr(workspace), wb, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 << 20


def kvq_decode_attention_noalloc(cache: KVCache, q, block_table, seq_lens, out, *, max_seq_len: int,
                                 num_seqs: Optional[int] = None, num_q_heads: Optional[int] = None,
                                 max_pages: Optional[int] = None, softmax_scale: Optional[float] = None,
                                 mode=None, out_dtype=None, stream=None):
    """kvq_decode_attention for callers that cannot allocate device memory: the
    split scratch is the library's own fixed array (NOALLOC_SCRATCH_BYTES), shared
    by all calls, so calls must not overlap on the GPU."""
    B = num_seqs if num_seqs is not None else q.shape[0]
    Hq = num_q_heads if num_q_heads is not None else q.shape[1]
    mp = max_pages if max_pages is not None else block_table.shape[1]
    sm = softmax_scale if softmax_scale is not None else cache.cfg.head_dim ** -0.5
    od = _dtype_code(out.dtype) if out_dtype is None else _dtype_code(out_dtype)
    _check(_lib.kvq_decode_attention_noalloc(cache.handle, _ptr(q), _ptr(block_table), mp, _ptr(seq_lens), B,
                                             Hq, max_seq_len, cache.mode if mode is None else _mode(mode), sm,
                                             _ptr(out), od, _stream(stream)))


# ---- multi-query decode
def kvq_decode_multi_plan(cache: KVCache, num_seqs: int, num_queries: int, num_q_heads: int, max_seq_len: int):
    ns, tps, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _check(_lib.kvq_decode_multi_plan(cache.handle, num_seqs, num_queries, num_q_heads, max_seq_len, ctypes.byref(ns),
                                      ctypes.byref(tps), ctypes.byref(ws)))
    return ns.value, tps.value, ws.value


def kvq_decode_multi_workspace_bytes(cache: KVCache, num_seqs: int, num_queries: int, num_q_heads: int,
                                     max_seq_len: int) -> int:
    ws = ctypes.c_size_t()
    _check(_lib.kvq_decode_multi_workspace_bytes(cache.handle, num_seqs, num_queries, num_q_heads, max_seq_len,
                                                 ctypes.byref(ws)))
    return ws.value


def kvq_decode_attention_multi(cache: KVCache, q, block_table, seq_lens, out, *, max_seq_len: int,
                               workspace=None, softmax_scale: Optional[float] = None, mode=None,
                               out_dtype=None, workspace_bytes: Optional[int] = None, stream=None):
    """q, out [num_seqs][num_queries][Hq][D]: query i of sequence b attends causally
    to tokens 0 .. seq_len_b - num_queries + i."""
    B, nq, Hq = q.shape[0], q.shape[1], q.shape[2]
    sm = softmax_scale if softmax_scale is not None else cache.cfg.head_dim ** -0.5
    od = _dtype_code(out.dtype) if out_dtype is None else _dtype_code(out_dtype)
    wb = workspace_bytes if workspace_bytes is not None else (
        0 if workspace is None else workspace.numel() * workspace.element_size())
    _check(_lib.kvq_decode_attention_multi(cache.handle, _ptr(q), _ptr(block_table), block_table.shape[1],
                                           _ptr(seq_lens), B, nq, Hq, max_seq_len,
                                           cache.mode if mode is None else _mode(mode), sm, _ptr(out), od,
                                           _ptr(workspace), wb, _stream(stream)))


# ---- KVarN open tiles
def kvq_kvarn_tail_bytes(cache: KVCache, num_seqs: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.kvq_kvarn_tail_bytes(cache.handle, num_seqs, ctypes.byref(b)))
    return b.value


def kvq_kvarn_append(cache: KVCache, k, v, slot_mapping, seq_ids, tail, num_seqs: int,
                     num_tokens: Optional[int] = None, stream=None):
    """Copy tokens into their sequences' open tiles (the tail buffer); a token that
    fills row 127 of its tile has the tile quantized into its page."""
    n = num_tokens if num_tokens is not None else int(slot_mapping.numel())
    _check(_lib.kvq_kvarn_append(cache.handle, _ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(seq_ids), n,
                                 _ptr(tail), num_seqs, _stream(stream)))


def kvq_kvarn_decode_workspace_bytes(cache: KVCache, num_seqs: int, num_q_heads: int, max_seq_len: int) -> int:
    ws = ctypes.c_size_t()
    _check(_lib.kvq_kvarn_decode_workspace_bytes(cache.handle, num_seqs, num_q_heads, max_seq_len,
                                                 ctypes.byref(ws)))
    return ws.value


def kvq_kvarn_decode_attention(cache: KVCache, q, block_table, seq_lens, tail, out, *, max_seq_len: int,
                               workspace, num_seqs: Optional[int] = None, num_q_heads: Optional[int] = None,
                               max_pages: Optional[int] = None, softmax_scale: Optional[float] = None,
                               out_dtype=None, workspace_bytes: Optional[int] = None, stream=None):
    """KVarN decode over the quantized whole tiles plus each sequence's open tile."""
    B = num_seqs if num_seqs is not None else q.shape[0]
    Hq = num_q_heads if num_q_heads is not None else q.shape[1]
    mp = max_pages if max_pages is not None else block_table.shape[1]
    sm = softmax_scale if softmax_scale is not None else cache.cfg.head_dim ** -0.5
    od = _dtype_code(out.dtype) if out_dtype is None else _dtype_code(out_dtype)
    wb = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    _check(_lib.kvq_kvarn_decode_attention(cache.handle, _ptr(q), _ptr(block_table), mp, _ptr(seq_lens), B, Hq,
                                           max_seq_len, sm, _ptr(tail), _ptr(out), od, _ptr(workspace), wb,
                                           _stream(stream)))
