"""Seeded synthetic workloads for the quantized paged KV-cache hot path.

This module only draws inputs: it holds none of the quantization or attention
arithmetic.  Both the CUDA path (through the tests and ``bench.py``) and the
CPU oracle take their K/V/q tensors, sequence lengths, block tables and slot
mappings from here, so the two sides see identical bytes.

Recipe (the same for every workload):

* every random stream is ``numpy.random.PCG64`` seeded with
  ``SeedSequence([workload seed, stream tag, index])``; the tags are listed in
  ``_TAG``;
* K, V and q are standard normal draws in float32, scaled where the workload
  plants outliers, then rounded once to the workload's I/O dtype (float16, or
  float32 for the tiny INT8 case);
* sequence ``b`` owns ``ceil(seq_len_b / page_size)`` pages; page ids are a
  seeded random permutation of ``[0, num_pages)``, so a sequence's pages are
  scattered over the pool;
* token ``i`` of sequence ``b`` lives at slot ``block_table[b][i // P] * P + i % P``.

The workload shapes follow the pages the method comes from: the fake-quant
experiment on "KV Cache 量化 · LLM Glossary" (B=2, H=4, T=16, D=32, fp32), and
GQA decode shapes with head_dim 128 (8 KV heads) for the per-tensor FP8,
per-token-head INT8/FP8, NVFP4 and KVarN k4v2 modes.  Outliers model the
attention-sink tokens named in "KV Cache 量化深度解析" section 2.1, outlier
tokens (per-token-head motivation, section 2.2) and outlier channels (NVFP4
block scales, KVarN rotation).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterator, List, Optional, Tuple

import numpy as np

_TAG = {
    "k": 1,
    "v": 2,
    "q": 3,
    "outlier_tokens": 4,
    "outlier_channels": 5,
    "seq_lens": 6,
    "pages": 7,
}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str                 # fp8_per_tensor | int8_per_token_head | fp8_per_token_head | nvfp4 | kvarn_k4v2_g128
    num_seqs: int             # B
    num_q_heads: int          # Hq
    num_kv_heads: int         # Hkv
    head_dim: int             # D
    page_size: int            # P
    io_dtype: str             # "f16" or "f32"
    seed: int
    seq_len: Optional[int] = None                  # every sequence has this length
    seq_len_range: Optional[Tuple[int, int]] = None  # or uniform integers in [lo, hi]
    sink_tokens: int = 0          # first tokens of every sequence scaled by sink_gain
    sink_gain: float = 1.0
    outlier_token_frac: float = 0.0   # fraction of tokens per sequence scaled by token_gain
    token_gain: float = 1.0
    outlier_channels: int = 0         # number of (kv head, dim) channels scaled by channel_gain
    channels_per_head: bool = False   # if True, outlier_channels is per kv head
    channel_gain: float = 1.0
    num_queries: int = 1              # queries per sequence per decode step (causal; >1: speculative decoding)
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def np_dtype(self):
        return np.float16 if self.io_dtype == "f16" else np.float32

    def with_mode(self, mode: str) -> "Workload":
        return dataclasses.replace(self, mode=mode, name=f"{self.name}:{mode}")

    def scaled(self, **kw) -> "Workload":
        """A smaller copy with the same structure (for oracle-sized parity)."""
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "int8_pth_tiny": Workload(
        name="int8_pth_tiny", mode="int8_per_token_head", num_seqs=2, num_q_heads=4,
        num_kv_heads=4, head_dim=32, page_size=16, io_dtype="f32", seed=1001, seq_len=16,
        description="INT8 per-token-head, B=2 Hq=Hkv=4 T=16 D=32, fp32 K,V,q ~ N(0,1)"),
    "fp8_pt_b16_s4096": Workload(
        name="fp8_pt_b16_s4096", mode="fp8_per_tensor", num_seqs=16, num_q_heads=32,
        num_kv_heads=8, head_dim=128, page_size=16, io_dtype="f16", seed=1002, seq_len=4096,
        sink_tokens=4, sink_gain=20.0,
        description="FP8-E4M3 per-tensor, GQA 32/8, D=128, fp16, B=16 x 4096, page 16, "
                    "first 4 tokens x20, scale = global amax/448"),
    "pth_b64_u1k_32k": Workload(
        name="pth_b64_u1k_32k", mode="int8_per_token_head", num_seqs=64, num_q_heads=64,
        num_kv_heads=8, head_dim=128, page_size=16, io_dtype="f16", seed=1003,
        seq_len_range=(1024, 32768), outlier_token_frac=0.01, token_gain=30.0,
        description="INT8 / FP8 per-token-head, GQA 64/8, D=128, fp16, B=64, seq U[1024,32768], "
                    "page 16, 1% of tokens x30"),
    "nvfp4_b32_s32768": Workload(
        name="nvfp4_b32_s32768", mode="nvfp4", num_seqs=32, num_q_heads=64, num_kv_heads=8,
        head_dim=128, page_size=16, io_dtype="f16", seed=1004, seq_len=32768,
        outlier_channels=20, channel_gain=10.0,
        description="NVFP4 (E2M1 + E4M3 per 16 + FP32 global), GQA 64/8, D=128, fp16, "
                    "B=32 x 32768, page 16, 2% of (head,dim) channels x10"),
    "kvarn_b16_s16384": Workload(
        name="kvarn_b16_s16384", mode="kvarn_k4v2_g128", num_seqs=16, num_q_heads=64,
        num_kv_heads=8, head_dim=128, page_size=128, io_dtype="f16", seed=1005, seq_len=16384,
        outlier_channels=4, channels_per_head=True, channel_gain=15.0,
        description="KVarN k4v2 g128, GQA 64/8, D=128, fp16, B=16 x 16384, 128-token tiles, "
                    "4 channels per kv head x15"),
}


def _rng(w: Workload, tag: str, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAG[tag], index])))


def seq_lens(w: Workload) -> np.ndarray:
    if w.seq_len is not None:
        return np.full(w.num_seqs, w.seq_len, dtype=np.int32)
    lo, hi = w.seq_len_range
    return _rng(w, "seq_lens").integers(lo, hi, size=w.num_seqs, endpoint=True).astype(np.int32)


@dataclasses.dataclass
class PagedLayout:
    seq_lens: np.ndarray        # [B] int32
    num_pages: int
    block_table: np.ndarray     # [B, max_pages] int32, -1 where unused
    token_offset: np.ndarray    # [B+1] int64: first global token index of each sequence

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]

    @property
    def num_tokens(self) -> int:
        return int(self.token_offset[-1])


def paged_layout(w: Workload, lens: Optional[np.ndarray] = None, slack_pages: int = 0) -> PagedLayout:
    lens = seq_lens(w) if lens is None else np.asarray(lens, dtype=np.int32)
    P = w.page_size
    npages = [(int(n) + P - 1) // P for n in lens]
    total = sum(npages) + slack_pages
    perm = _rng(w, "pages").permutation(total).astype(np.int32)
    max_pages = max(1, max(npages) if npages else 1)
    bt = np.full((len(lens), max_pages), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens.astype(np.int64))
    return PagedLayout(seq_lens=lens, num_pages=total, block_table=bt, token_offset=off)


def slots_for_seq(w: Workload, lay: PagedLayout, b: int, start: int = 0,
                  stop: Optional[int] = None) -> np.ndarray:
    """Slot ids of tokens [start, stop) of sequence b."""
    stop = int(lay.seq_lens[b]) if stop is None else stop
    P = w.page_size
    i = np.arange(start, stop, dtype=np.int64)
    return (lay.block_table[b, i // P].astype(np.int64) * P + i % P).astype(np.int32)


def slot_mapping(w: Workload, lay: PagedLayout) -> np.ndarray:
    """Slots of every token of every sequence, in global token order."""
    return np.concatenate([slots_for_seq(w, lay, b) for b in range(len(lay.seq_lens))]) \
        if len(lay.seq_lens) else np.zeros(0, np.int32)


def _outlier_channel_mask(w: Workload) -> Optional[np.ndarray]:
    if w.outlier_channels <= 0:
        return None
    rng = _rng(w, "outlier_channels")
    gain = np.ones((w.num_kv_heads, w.head_dim), dtype=np.float32)
    if w.channels_per_head:
        for h in range(w.num_kv_heads):
            d = rng.choice(w.head_dim, size=w.outlier_channels, replace=False)
            gain[h, d] = w.channel_gain
    else:
        flat = rng.choice(w.num_kv_heads * w.head_dim, size=w.outlier_channels, replace=False)
        gain.reshape(-1)[flat] = w.channel_gain
    return gain


def outlier_tokens(w: Workload, b: int, n: int) -> np.ndarray:
    if w.outlier_token_frac <= 0 or n == 0:
        return np.zeros(0, dtype=np.int64)
    cnt = max(1, int(round(w.outlier_token_frac * n)))
    return np.sort(_rng(w, "outlier_tokens", b).choice(n, size=cnt, replace=False))


def gen_kv_seq(w: Workload, b: int, n: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """K and V of sequence b: [n, Hkv, D] in the workload's I/O dtype."""
    if n is None:
        n = int(seq_lens(w)[b])
    shape = (n, w.num_kv_heads, w.head_dim)
    out = []
    chan = _outlier_channel_mask(w)
    toks = outlier_tokens(w, b, n)
    for tag in ("k", "v"):
        x = _rng(w, tag, b).standard_normal(shape, dtype=np.float32)
        if w.sink_tokens:
            x[: w.sink_tokens] *= np.float32(w.sink_gain)
        if len(toks):
            x[toks] *= np.float32(w.token_gain)
        if chan is not None:
            x *= chan[None]
        out.append(x.astype(w.np_dtype))
    return out[0], out[1]


def gen_q(w: Workload, num_seqs: Optional[int] = None) -> np.ndarray:
    B = w.num_seqs if num_seqs is None else num_seqs
    x = _rng(w, "q").standard_normal((B, w.num_q_heads, w.head_dim), dtype=np.float32)
    return x.astype(w.np_dtype)


def iter_kv_chunks(w: Workload, lay: PagedLayout, max_tokens: int = 1 << 20
                   ) -> Iterator[Tuple[np.ndarray, np.ndarray, np.ndarray]]:
    """Yield (K, V, slots) for whole sequences, about max_tokens tokens at a time."""
    ks: List[np.ndarray] = []
    vs: List[np.ndarray] = []
    ss: List[np.ndarray] = []
    cnt = 0
    for b in range(len(lay.seq_lens)):
        k, v = gen_kv_seq(w, b, int(lay.seq_lens[b]))
        ks.append(k); vs.append(v); ss.append(slots_for_seq(w, lay, b))
        cnt += len(k)
        if cnt >= max_tokens:
            yield np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)
            ks, vs, ss, cnt = [], [], [], 0
    if ks:
        yield np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)


def last_token_step(w: Workload, lay: PagedLayout) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The decode-step append: the last token of every sequence (K, V, slot).

    The values are the same rows the bulk fill wrote, so re-writing them is
    idempotent and the cache stays consistent step after step.
    """
    ks, vs, ss = [], [], []
    for b in range(len(lay.seq_lens)):
        n = int(lay.seq_lens[b])
        if n == 0:
            continue
        k, v = gen_kv_seq(w, b, n)
        ks.append(k[-1:]); vs.append(v[-1:]); ss.append(slots_for_seq(w, lay, b, n - 1, n))
    return np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)


def decode_bytes(w: Workload, lens: np.ndarray, bytes_per_token_head: float, scale_bytes: int) -> int:
    """Algorithmic bytes of one decode pass: packed K/V (+ in-page scales) of every
    token, the per-tensor scales, q in and out."""
    esz = 2 if w.io_dtype == "f16" else 4
    kv = int(round(float(np.sum(lens.astype(np.int64))) * w.num_kv_heads * bytes_per_token_head))
    return kv + scale_bytes + 2 * w.num_seqs * w.num_queries * w.num_q_heads * w.head_dim * esz


def describe(w: Workload) -> dict:
    lens = seq_lens(w)
    return {
        "workload": w.name,
        "mode": w.mode,
        "B": w.num_seqs,
        "Hq": w.num_q_heads,
        "Hkv": w.num_kv_heads,
        "D": w.head_dim,
        "page_size": w.page_size,
        "io_dtype": w.io_dtype,
        "tokens": int(np.sum(lens.astype(np.int64))),
        "max_seq_len": int(lens.max()) if len(lens) else 0,
    }
