"""Shared test helpers: build GPU caches through the C ABI and the same caches
through the oracle, from the same seeded inputs (workloads.py)."""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as wl

MODE_NAMES = ["fp8_per_tensor", "int8_per_token_head", "fp8_per_token_head", "nvfp4", "int4_per_token_head",
              "nvfp4_4over6", "kvarn_k4v2_g128"]
TENSOR_SCALED = {"fp8_per_tensor", "nvfp4", "nvfp4_4over6"}
FILL = 0xCD  # untouched bytes of both pools
GUARD = 4096        # canary bytes on each side of every device buffer a kernel writes
GUARD_BYTE = 0xA5
_guarded = []       # (raw tensor, payload bytes, name) of the buffers handed out since the last check


def guarded(shape, dtype, fill=None, name="buffer") -> torch.Tensor:
    """A CUDA tensor with GUARD canary bytes before and after it (the pool,
    an output, a workspace, a tail buffer): a kernel store that strays past
    its buffer changes a canary, which check_guards() reports after the test."""
    shape = (shape,) if isinstance(shape, int) else tuple(shape)
    esz = torch.empty((), dtype=dtype).element_size()
    n = 1
    for x in shape:
        n *= int(x)
    raw = torch.full((2 * GUARD + n * esz,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
    view = raw[GUARD:GUARD + n * esz].view(dtype).view(shape)
    if fill is not None:
        view.fill_(fill)
    _guarded.append((raw, n * esz, name))
    return view


def check_guards():
    """Every canary band still holds GUARD_BYTE (then forget the buffers)."""
    bad = []
    for raw, n, name in _guarded:
        lo, hi = raw[:GUARD], raw[GUARD + n:]
        if bool((lo != GUARD_BYTE).any()) or bool((hi != GUARD_BYTE).any()):
            bad.append(name)
    _guarded.clear()
    assert not bad, f"canary bytes overwritten next to: {bad}"


def kvq():
    from quantized_paged_kv_quantize_gb300 import kvq as _k
    return _k


def torch_dtype(w: wl.Workload):
    return torch.float16 if w.io_dtype == "f16" else torch.float32


@dataclass
class Case:
    w: wl.Workload
    lay: wl.PagedLayout
    k: np.ndarray          # [N, Hkv, D] io dtype
    v: np.ndarray
    slots: np.ndarray      # [N] int32
    q: np.ndarray          # [B, Hq, D] io dtype
    k_scale: float = 1.0   # oracle tensor scales (from the oracle's amax)
    v_scale: float = 1.0


def make_case(w: wl.Workload, lens: Sequence[int], slack_pages: int = 1) -> Case:
    lay = wl.paged_layout(w, np.asarray(lens, np.int32), slack_pages=slack_pages)
    ks, vs, ss = [], [], []
    for b, n in enumerate(lens):
        k, v = wl.gen_kv_seq(w, b, int(n))
        ks.append(k); vs.append(v); ss.append(wl.slots_for_seq(w, lay, b))
    k = np.concatenate(ks) if ks else np.zeros((0, w.num_kv_heads, w.head_dim), w.np_dtype)
    v = np.concatenate(vs) if vs else np.zeros_like(k)
    slots = np.concatenate(ss) if ss else np.zeros(0, np.int32)
    q = wl.gen_q(w, len(lens))
    c = Case(w, lay, k, v, slots.astype(np.int32), q)
    if w.mode in TENSOR_SCALED:
        c.k_scale = oracle.tensor_scale(w.mode, oracle.amax(k.astype(np.float32)))
        c.v_scale = oracle.tensor_scale(w.mode, oracle.amax(v.astype(np.float32)))
    return c


def oracle_pool(c: Case, k=None, v=None, slots=None) -> np.ndarray:
    w = c.w
    pool = np.full(oracle.pool_bytes(w.mode, c.lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim),
                   FILL, np.uint8)
    oracle.write(w.mode, pool, c.lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim,
                 (c.k if k is None else k).astype(np.float32), (c.v if v is None else v).astype(np.float32),
                 c.slots if slots is None else slots, c.k_scale, c.v_scale)
    return pool


def config(c: Case):
    w = c.w
    return kvq().make_config(c.lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim, w.mode,
                             torch_dtype(w))


def gpu_cache(c: Case, fill: int = FILL):
    K = kvq()
    cfg = config(c)
    pool = guarded(K.kvq_cache_bytes(cfg), torch.uint8, fill=fill, name="pool")
    return K.kvq_cache_alloc(cfg, pool)


def gpu_calibrate(cache, k_dev: torch.Tensor, v_dev: torch.Tensor):
    """Per-tensor scales from device amax (FP8 per-tensor, NVFP4)."""
    K = kvq()
    amax = torch.zeros(2, dtype=torch.float32, device="cuda")
    K.kvq_tensor_amax(k_dev, amax[0:1])
    K.kvq_tensor_amax(v_dev, amax[1:2])
    K.kvq_cache_set_tensor_scales_from_amax(cache, amax[0:1], amax[1:2])
    return amax


def header_scales(cache) -> tuple:
    h = cache.pool[:24].cpu().numpy()
    return float(h[16:20].view(np.float32)[0]), float(h[20:24].view(np.float32)[0])


def gpu_decode(cache, c: Case, q_dev=None, out_dtype=torch.float32, max_seq_len=None, bt=None, lens=None):
    K = kvq()
    w = c.w
    B = len(c.lay.seq_lens)
    msl = int(c.lay.seq_lens.max()) if max_seq_len is None and B else (max_seq_len or 0)
    q_dev = torch.from_numpy(c.q).cuda() if q_dev is None else q_dev
    bt_dev = torch.from_numpy(c.lay.block_table if bt is None else bt).cuda()
    sl_dev = torch.from_numpy(c.lay.seq_lens if lens is None else np.asarray(lens, np.int32)).cuda()
    out = guarded((B, w.num_q_heads, w.head_dim), out_dtype, fill=float("nan"), name="out")
    ns, tps, wsb = K.kvq_decode_plan(cache, B, w.num_q_heads, msl)
    ws = guarded(max(wsb // 4, 1), torch.float32, name="workspace")
    K.kvq_decode_attention(cache, q_dev, bt_dev, sl_dev, out, max_seq_len=msl, workspace=ws)
    torch.cuda.synchronize()
    return out, (ns, tps, wsb)


def oracle_decode(c: Case, pool: np.ndarray, rows=None, bt=None, lens=None) -> np.ndarray:
    w = c.w
    return oracle.decode(w.mode, pool, c.lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim,
                         c.q.astype(np.float32), c.lay.block_table if bt is None else bt,
                         c.lay.seq_lens if lens is None else np.asarray(lens, np.int32),
                         1.0 / math.sqrt(w.head_dim), c.k_scale, c.v_scale, rows=rows)


def check_attention(gpu: torch.Tensor, ref: np.ndarray, rows: Optional[np.ndarray] = None, tol: float = 2e-3):
    """Attention parity: fp32 outputs within tol of the fp64 oracle; fp16 outputs
    within tol of fp16(oracle) or within one fp16 ulp of it."""
    g = gpu.float().cpu().numpy().astype(np.float64)
    B, Hq, D = ref.shape
    if rows is not None:
        g = g.reshape(B * Hq, D)[rows]
        ref = ref.reshape(B * Hq, D)[rows]
    assert np.isfinite(g).all(), "non-finite output"
    if gpu.dtype == torch.float32:
        err = np.abs(g - ref)
        assert err.max() <= tol, f"max abs err {err.max():.3e} > {tol}"
        return float(err.max())
    r16 = ref.astype(np.float16).astype(np.float64)
    ulp = np.abs(np.spacing(ref.astype(np.float16)).astype(np.float64))
    err = np.abs(g - r16)
    bad = (err > tol) & (err > ulp)
    assert not bad.any(), f"{bad.sum()} fp16 outputs off by more than max(tol, 1 ulp); worst {err.max():.3e}"
    return float(err.max())
