"""Python face of the plain C oracle (``kvq_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only users.  The product library never
imports, links or runs anything in this folder, and this folder never imports
the product.

The C source is compiled with gcc on first use (``-O2 -ffp-contract=off``, no
fast-math: every fp32 operation is individually rounded, no fused
multiply-add), into ``oracle/libkvq_oracle.so``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_HDR = os.path.join(_HERE, "kvq_oracle.h")
_LIB = os.path.join(_HERE, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

MODES = {
    "fp8_per_tensor": 1,
    "int8_per_token_head": 2,
    "fp8_per_token_head": 3,
    "nvfp4": 4,
    "int4_per_token_head": 5,
    "nvfp4_4over6": 6,
    "kvarn_k4v2_g128": 16,
}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (skipped when the library is up to date)."""
    with _lock:
        fresh = os.path.exists(_LIB) and all(
            os.path.getmtime(_LIB) >= os.path.getmtime(p) for p in (_SRC, _HDR))
        if force or not fresh:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                   "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i8p = ctypes.POINTER(ctypes.c_int8)
        sig = {
            "kvqo_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "kvqo_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "kvqo_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "kvqo_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "kvqo_int8_encode": (ctypes.c_int, [ctypes.c_float]),
            "kvqo_int4_encode": (ctypes.c_int, [ctypes.c_float]),
            "kvqo_fp8_tensor_scale": (ctypes.c_float, [ctypes.c_float]),
            "kvqo_nvfp4_tensor_scale": (ctypes.c_float, [ctypes.c_float]),
            "kvqo_amax": (ctypes.c_float, [f32p, ctypes.c_size_t]),
            "kvqo_quant_row_fp8_pt": (None, [f32p, ctypes.c_int, ctypes.c_float, u8p]),
            "kvqo_quant_row_int8_pth": (None, [f32p, ctypes.c_int, i8p, f32p]),
            "kvqo_quant_row_fp8_pth": (None, [f32p, ctypes.c_int, u8p, f32p]),
            "kvqo_quant_row_nvfp4": (None, [f32p, ctypes.c_int, ctypes.c_float, u8p, u8p]),
            "kvqo_quant_row_int4_pth": (None, [f32p, ctypes.c_int, u8p, f32p]),
            "kvqo_quant_row_nvfp4_4over6": (None, [f32p, ctypes.c_int, ctypes.c_float, u8p, u8p, u8p]),
            "kvqo_nvfp4_block_sse": (ctypes.c_float, [f32p, u8p, ctypes.c_float]),
            "kvqo_inv_sqrt128": (ctypes.c_float, []),
            "kvqo_fwht128_f32": (None, [f32p]),
            "kvqo_sum128": (ctypes.c_float, [f32p]),
            "kvqo_kvarn_normalize": (None, [f32p, f32p, f32p, ctypes.c_int]),
            "kvqo_kvarn_tile": (None, [f32p, ctypes.c_int, u8p, f32p, f32p, f32p, f32p]),
            "kvqo_hadamard_f64": (None, [f64p, ctypes.c_int]),
            "kvqo_header_bytes": (ctypes.c_size_t, []),
            "kvqo_block_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
            "kvqo_pool_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
            "kvqo_write": (ctypes.c_int, [ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, f32p, f32p, i32p, ctypes.c_int,
                                          ctypes.c_float, ctypes.c_float]),
            "kvqo_dequant_row": (ctypes.c_int, [ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                                ctypes.c_float, ctypes.c_int64, ctypes.c_int,
                                                ctypes.c_int, f64p]),
            "kvqo_decode_kvarn_tail": (ctypes.c_int, [u8p, ctypes.c_int, ctypes.c_int, f32p, i32p, ctypes.c_int,
                                                      i32p, ctypes.c_int, ctypes.c_int, ctypes.c_double, f32p,
                                                      f32p, i32p, ctypes.c_int, f64p]),
            "kvqo_decode": (ctypes.c_int, [ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                           ctypes.c_float, f32p, i32p, ctypes.c_int, i32p,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_double, i32p,
                                           ctypes.c_int, f64p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ct))


def mode_id(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


# ---- codecs -----------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return lib().kvqo_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    return lib().kvqo_e4m3_encode(float(v))


def e2m1_decode(code: int) -> float:
    return lib().kvqo_e2m1_decode(int(code) & 0xF)


def e2m1_encode(v: float) -> int:
    return lib().kvqo_e2m1_encode(float(v))


def int8_encode(v: float) -> int:
    return lib().kvqo_int8_encode(float(v))


def int4_encode(v: float) -> int:
    return lib().kvqo_int4_encode(float(v))


def fp8_tensor_scale(amax: float) -> float:
    return lib().kvqo_fp8_tensor_scale(float(amax))


def nvfp4_tensor_scale(amax: float) -> float:
    return lib().kvqo_nvfp4_tensor_scale(float(amax))


def amax(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return lib().kvqo_amax(_p(x, ctypes.c_float), x.size)


def tensor_scale(mode, amax_value: float) -> float:
    m = mode_id(mode)
    if m == 1:
        return fp8_tensor_scale(amax_value)
    if m in (4, 6):
        return nvfp4_tensor_scale(amax_value)
    return 1.0


# ---- rows ---------------------------------------------------------------------
def quant_row(mode, x: np.ndarray, tensor_scale_value: float = 1.0):
    """Quantize one D-vector; returns (payload bytes, scale bytes)."""
    m = mode_id(mode)
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.size
    L = lib()
    if m == 1:
        q = np.zeros(D, np.uint8)
        L.kvqo_quant_row_fp8_pt(_p(x, ctypes.c_float), D, tensor_scale_value, _p(q, ctypes.c_uint8))
        return q, np.zeros(0, np.uint8)
    if m in (2, 3):
        q = np.zeros(D, np.uint8)
        s = np.zeros(1, np.float32)
        fn = L.kvqo_quant_row_int8_pth if m == 2 else L.kvqo_quant_row_fp8_pth
        if m == 2:
            fn(_p(x, ctypes.c_float), D, _p(q.view(np.int8), ctypes.c_int8), _p(s, ctypes.c_float))
        else:
            fn(_p(x, ctypes.c_float), D, _p(q, ctypes.c_uint8), _p(s, ctypes.c_float))
        return q, s.view(np.uint8)
    if m == 4:
        q = np.zeros(D // 2, np.uint8)
        bs = np.zeros(D // 16, np.uint8)
        L.kvqo_quant_row_nvfp4(_p(x, ctypes.c_float), D, tensor_scale_value, _p(q, ctypes.c_uint8),
                               _p(bs, ctypes.c_uint8))
        return q, bs
    if m == 5:
        q = np.zeros(D // 2, np.uint8)
        s = np.zeros(1, np.float32)
        L.kvqo_quant_row_int4_pth(_p(x, ctypes.c_float), D, _p(q, ctypes.c_uint8), _p(s, ctypes.c_float))
        return q, s.view(np.uint8)
    if m == 6:
        q, bs, _ = nvfp4_4over6_row(x, tensor_scale_value)
        return q, bs
    raise ValueError(f"no row quantizer for mode {mode}")


def nvfp4_4over6_row(x: np.ndarray, s_t: float):
    """nvfp4_4over6 coding of one D-vector: (packed codes, block scales, the
    choice per block: 6 for the max/6 scale, 4 for the max/4 scale)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.size
    q = np.zeros(D // 2, np.uint8)
    bs = np.zeros(D // 16, np.uint8)
    ch = np.zeros(D // 16, np.uint8)
    lib().kvqo_quant_row_nvfp4_4over6(_p(x, ctypes.c_float), D, s_t, _p(q, ctypes.c_uint8),
                                      _p(bs, ctypes.c_uint8), _p(ch, ctypes.c_uint8))
    return q, bs, ch


def nvfp4_block_sse(x: np.ndarray, codes: np.ndarray, den: float) -> float:
    """The fp32 squared reconstruction error the 4over6 choice compares."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    assert x.size == 16 and c.size == 16
    return lib().kvqo_nvfp4_block_sse(_p(x, ctypes.c_float), _p(c, ctypes.c_uint8), den)


# ---- KVarN --------------------------------------------------------------------
def inv_sqrt128() -> float:
    return lib().kvqo_inv_sqrt128()


def fwht128_f32(x: np.ndarray) -> np.ndarray:
    y = np.array(x, dtype=np.float32).copy()
    assert y.size == 128
    lib().kvqo_fwht128_f32(_p(y, ctypes.c_float))
    return y


def sum128(x: np.ndarray) -> float:
    y = np.ascontiguousarray(x, dtype=np.float32)
    assert y.size == 128
    return lib().kvqo_sum128(_p(y, ctypes.c_float))


def kvarn_normalize(Y: np.ndarray, steps: int = 8):
    Y = np.array(Y, dtype=np.float32).copy()
    r = np.zeros(128, np.float32)
    c = np.zeros(128, np.float32)
    lib().kvqo_kvarn_normalize(_p(Y, ctypes.c_float), _p(r, ctypes.c_float), _p(c, ctypes.c_float), steps)
    return Y, r, c


def kvarn_tile(X: np.ndarray, is_value: bool):
    X = np.ascontiguousarray(X, dtype=np.float32)
    assert X.shape == (128, 128)
    codes = np.zeros((128, 128), np.uint8)
    scale, zero, r, c = (np.zeros(128, np.float32) for _ in range(4))
    lib().kvqo_kvarn_tile(_p(X, ctypes.c_float), int(bool(is_value)), _p(codes, ctypes.c_uint8),
                          _p(scale, ctypes.c_float), _p(zero, ctypes.c_float), _p(r, ctypes.c_float),
                          _p(c, ctypes.c_float))
    return codes, scale, zero, r, c


def hadamard_f64(x: np.ndarray) -> np.ndarray:
    y = np.array(x, dtype=np.float64).copy()
    lib().kvqo_hadamard_f64(_p(y, ctypes.c_double), y.size)
    return y


# ---- pool -----------------------------------------------------------------------
def header_bytes() -> int:
    return lib().kvqo_header_bytes()


def block_bytes(mode, page_size: int, head_dim: int) -> int:
    return lib().kvqo_block_bytes(mode_id(mode), page_size, head_dim)


def pool_bytes(mode, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return lib().kvqo_pool_bytes(mode_id(mode), num_pages, page_size, num_kv_heads, head_dim)


def write(mode, pool: np.ndarray, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int,
          k: np.ndarray, v: np.ndarray, slots: np.ndarray, k_scale: float = 1.0,
          v_scale: float = 1.0) -> int:
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    rc = lib().kvqo_write(mode_id(mode), _p(pool, ctypes.c_uint8), num_pages, page_size, num_kv_heads,
                          head_dim, _p(k, ctypes.c_float), _p(v, ctypes.c_float),
                          _p(slots, ctypes.c_int32), len(slots), k_scale, v_scale)
    if rc < 0:
        raise ValueError("oracle write rejected its arguments")
    return rc


def dequant_row(mode, pool, num_pages, page_size, num_kv_heads, head_dim, k_scale, v_scale,
                slot: int, h: int, side: int) -> np.ndarray:
    out = np.zeros(head_dim, np.float64)
    rc = lib().kvqo_dequant_row(mode_id(mode), _p(pool, ctypes.c_uint8), num_pages, page_size,
                                num_kv_heads, head_dim, k_scale, v_scale, int(slot), h, side,
                                _p(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("bad dequant_row arguments")
    return out


def decode(mode, pool: np.ndarray, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int,
           q: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray, softmax_scale: float,
           k_scale: float = 1.0, v_scale: float = 1.0,
           rows: Optional[Sequence[int]] = None) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    B, Hq, D = q.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    rr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    rc = lib().kvqo_decode(mode_id(mode), _p(pool, ctypes.c_uint8), num_pages, page_size, num_kv_heads,
                           head_dim, k_scale, v_scale, _p(q, ctypes.c_float), _p(bt, ctypes.c_int32),
                           bt.shape[1], _p(sl, ctypes.c_int32), B, Hq, softmax_scale,
                           None if rr is None else _p(rr, ctypes.c_int32),
                           0 if rr is None else len(rr), _p(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments")
    return out


def decode_kvarn_tail(pool: np.ndarray, num_pages: int, num_kv_heads: int, q: np.ndarray,
                      block_table: np.ndarray, seq_lens: np.ndarray, softmax_scale: float,
                      tail_k: np.ndarray, tail_v: np.ndarray,
                      rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """KVarN decode over quantized whole tiles plus each sequence's raw open
    tile (tail_k / tail_v [num_seqs][128][Hkv][128]); fp64 output [B][Hq][128]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    B, Hq, D = q.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    tk = np.ascontiguousarray(tail_k, dtype=np.float32)
    tv = np.ascontiguousarray(tail_v, dtype=np.float32)
    assert tk.shape == (B, 128, num_kv_heads, D) and tv.shape == tk.shape
    out = np.zeros((B, Hq, D), np.float64)
    rr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    rc = lib().kvqo_decode_kvarn_tail(_p(pool, ctypes.c_uint8), num_pages, num_kv_heads, _p(q, ctypes.c_float),
                                      _p(bt, ctypes.c_int32), bt.shape[1], _p(sl, ctypes.c_int32), B, Hq,
                                      softmax_scale, _p(tk, ctypes.c_float), _p(tv, ctypes.c_float),
                                      None if rr is None else _p(rr, ctypes.c_int32),
                                      0 if rr is None else len(rr), _p(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments")
    return out


def decode_multi(mode, pool: np.ndarray, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int,
                 q: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray, softmax_scale: float,
                 k_scale: float = 1.0, v_scale: float = 1.0,
                 rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Several queries per sequence under the causal mask of A = softmax(QK^T/sqrt(d) + M) V:
    q [B][nq][Hq][D]; query i of sequence b stands at position seq_len_b - nq + i and
    sees tokens 0 .. seq_len_b - nq + i (none if that is negative).  Written as the
    plain decode of B * nq sequences, query (b, i) reading sequence b's pages up to
    its own causal length; fp64 output [B][nq][Hq][D] (rows: flat (b*nq + i)*Hq + h
    indices to compute, the others left 0)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    B, nq, Hq, D = q.shape
    lens = np.asarray(seq_lens, np.int64)
    rows_len = np.maximum(lens[:, None] - (nq - 1 - np.arange(nq))[None, :], 0).astype(np.int32).reshape(-1)
    bt = np.repeat(np.ascontiguousarray(block_table, dtype=np.int32), nq, axis=0)
    out = decode(mode, pool, num_pages, page_size, num_kv_heads, head_dim, q.reshape(B * nq, Hq, D), bt,
                 rows_len, softmax_scale, k_scale, v_scale, rows=rows)
    return out.reshape(B, nq, Hq, D)
