"""Benchmark of the quantized paged KV-cache hot path on GB300.

One step = one decode step of a workload: quantize-on-write of each
sequence's newest token into its page, then paged decode attention of every
sequence over its whole packed history (the split-KV combine included).  The
bulk fill of the cache (per-tensor scale calibration + quantize-write of every
token) runs once before the timed steps and is timed on its own (``write``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--suite all|none|NAME,NAME..] [--impl ours|reference]

Prints one JSON line (rank 0).  Its headline (``value``, ``roofline``,
``e2e``, ...) is the ``--workload`` (default: the 32K-context NVFP4
configuration); ``workloads`` holds the same decode / write / step
measurements for every other configuration of the suite, each timed the same
way, one after another, each freed before the next.  Under torchrun each rank
runs its own replica (the path has no data exchange; weak scaling).  Inputs
are seeded synthetic tensors from workloads.py; the decode working set (the
packed cache) is larger than L2 for the large workloads, and for smaller ones
L2 is flushed between timed steps.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "decode-attn HBM GB/s (packed KV+scales) & % of peak; quantize-write GB/s"
DEFAULT_WORKLOAD = "nvfp4_b32_s32768"
L2_BYTES = 129 * 2 ** 20
BYTES_PER_TOKEN_HEAD = {"fp8_per_tensor": 256, "int8_per_token_head": 264, "fp8_per_token_head": 264,
                        "nvfp4": 144, "int4_per_token_head": 136, "nvfp4_4over6": 144, "kvarn_k4v2_g128": 128}
TENSOR_SCALED = ("fp8_per_tensor", "nvfp4", "nvfp4_4over6")
# mode variants of a workload: the same shapes and inputs, another quantization mode
VARIANTS = {
    "pth_b64_u1k_32k:fp8": ("pth_b64_u1k_32k", "fp8_per_token_head"),
    "pth_b64_u1k_32k:int4": ("pth_b64_u1k_32k", "int4_per_token_head"),
    "nvfp4_b32_s32768:4over6": ("nvfp4_b32_s32768", "nvfp4_4over6"),
}
# speculative-decoding shape: 4 causal queries per sequence over the same pages
SPEC_VARIANTS = {"nvfp4_b32_s32768:spec4": ("nvfp4_b32_s32768", 4), "kvarn_b16_s16384:spec4": ("kvarn_b16_s16384", 4)}
# every configuration the default run measures, grouped so that the variants of
# one base reuse its K/V inputs on the device
SUITE = ["nvfp4_b32_s32768", "nvfp4_b32_s32768:4over6", "nvfp4_b32_s32768:spec4",
         "pth_b64_u1k_32k", "pth_b64_u1k_32k:fp8", "pth_b64_u1k_32k:int4",
         "fp8_pt_b16_s4096", "kvarn_b16_s16384", "kvarn_b16_s16384:spec4", "int8_pth_tiny"]


def workload_by_name(name: str) -> wl.Workload:
    import dataclasses
    if name in VARIANTS:
        base, mode = VARIANTS[name]
        return dataclasses.replace(wl.WORKLOADS[base].with_mode(mode), name=name)
    if name in SPEC_VARIANTS:
        base, nq = SPEC_VARIANTS[name]
        return dataclasses.replace(wl.WORKLOADS[base], num_queries=nq, name=name)
    return wl.WORKLOADS[name]


def base_of(name: str) -> str:
    return name.split("[")[0].split(":")[0]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def bytes_per_token_head(w: wl.Workload) -> float:
    """Packed bytes of one token and kv head, K + V, payload and in-page scales
    (BYTES_PER_TOKEN_HEAD holds them at head_dim 128)."""
    D, P = w.head_dim, w.page_size
    return {"fp8_per_tensor": 2 * D, "int8_per_token_head": 2 * D + 8, "fp8_per_token_head": 2 * D + 8,
            "nvfp4": D + D / 8, "nvfp4_4over6": D + D / 8, "int4_per_token_head": D + 8,
            "kvarn_k4v2_g128": (P * D * 3 / 4 + 4 * (3 * D + P) + 4 * (3 * P + D)) / P}[w.mode]


def decode_bytes(w: wl.Workload, lens: np.ndarray) -> int:
    scale_bytes = 8 if w.mode in TENSOR_SCALED else 0
    return wl.decode_bytes(w, lens, bytes_per_token_head(w), scale_bytes)


def write_bytes(w: wl.Workload, ntok: int) -> int:
    esz = 2 if w.io_dtype == "f16" else 4
    return int(ntok * w.num_kv_heads * (2 * w.head_dim * esz + bytes_per_token_head(w)) + 4 * ntok)


def cache_pool_bytes(w: wl.Workload, lay: wl.PagedLayout) -> int:
    """Bytes of the packed pool: the 256-byte header and one block of
    page_size x (bytes per token and kv head) per (page, kv head)."""
    return 256 + int(lay.num_pages * w.num_kv_heads * w.page_size * bytes_per_token_head(w))


def l2_policy(w: wl.Workload, lay: wl.PagedLayout) -> str:
    cb = cache_pool_bytes(w, lay)
    if cb >= 2 * L2_BYTES:
        return "inputs larger than L2 (%.2f GB packed cache)" % (cb / 1e9)
    return ("L2 flushed before each timed step (256 MiB written, then 256 MiB read so that no dirty "
            "line is written back inside the timed region)")


def config_of(w: wl.Workload, lay: wl.PagedLayout = None) -> dict:
    """The workload's description, identical in both arms of the bench."""
    lay = wl.paged_layout(w) if lay is None else lay
    return {
        "workload": w.name, "mode": w.mode, "B": w.num_seqs, "Hq": w.num_q_heads,
        "Hkv": w.num_kv_heads, "D": w.head_dim, "page_size": w.page_size,
        "seq_len": w.seq_len if w.seq_len else list(w.seq_len_range),
        "io_dtype": w.io_dtype,
        "step": "quantize-write of 1 new token/seq + decode attention" if w.num_queries == 1 else
                f"quantize-write of {w.num_queries} new tokens/seq + causal decode of "
                f"{w.num_queries} queries/seq",
        "queries_per_seq": w.num_queries,
        "l2": l2_policy(w, lay),
    }


# --------------------------------------------------------------------------- GPU side
def _host_kv_chunks(w: wl.Workload, lens: np.ndarray, window: int = 16):
    """(b, K_b, V_b) for every sequence in order, drawn on a pool of host
    threads (numpy's generators release the GIL), at most `window` sequences
    ahead of the consumer."""
    from concurrent.futures import ThreadPoolExecutor
    nthreads = max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        pending = {}
        nxt = 0
        for b in range(len(lens)):
            while nxt < len(lens) and nxt < b + window:
                pending[nxt] = ex.submit(wl.gen_kv_seq, w, nxt, int(lens[nxt]))
                nxt += 1
            k, v = pending.pop(b).result()
            yield b, k, v


class GpuWorkload:
    """The workload resident on one GPU: full K/V, the packed cache, q, tables.
    `kv` = (K, V) device tensors of another workload with the same inputs (a
    mode variant of the same base) are reused instead of drawn again."""

    def __init__(self, w: wl.Workload, device="cuda", keep_host: bool = False, kv=None):
        import torch
        from quantized_paged_kv_quantize_gb300 import kvq
        self.kvq = kvq
        self.w = w
        self.dev = device
        self.lay = wl.paged_layout(w)
        lens = self.lay.seq_lens
        N = self.lay.num_tokens
        tdt = torch.float16 if w.io_dtype == "f16" else torch.float32
        self.tdt = tdt
        self.slots = torch.from_numpy(wl.slot_mapping(w, self.lay)).to(device)
        self.host = [] if keep_host else None
        if kv is not None and not keep_host:
            self.K, self.V = kv
            assert tuple(self.K.shape) == (N, w.num_kv_heads, w.head_dim) and self.K.dtype == tdt
        else:
            self.K = torch.empty((N, w.num_kv_heads, w.head_dim), dtype=tdt, device=device)
            self.V = torch.empty_like(self.K)
            off = 0
            pin_k = torch.empty((int(lens.max()), w.num_kv_heads, w.head_dim), dtype=tdt).pin_memory()
            pin_v = torch.empty_like(pin_k)
            for b, k, v in _host_kv_chunks(w, lens):
                n = len(k)
                pin_k[:n].copy_(torch.from_numpy(k))
                pin_v[:n].copy_(torch.from_numpy(v))
                self.K[off:off + n].copy_(pin_k[:n], non_blocking=True)
                self.V[off:off + n].copy_(pin_v[:n], non_blocking=True)
                torch.cuda.synchronize()
                if keep_host:
                    self.host.append((k, v))
                off += n
        nq = w.num_queries
        q = wl.gen_q(w, w.num_seqs * nq)
        self.q = torch.from_numpy(q.reshape(w.num_seqs, nq, w.num_q_heads, w.head_dim) if nq > 1 else q).to(device)
        self.block_table = torch.from_numpy(self.lay.block_table).to(device)
        self.seq_lens = torch.from_numpy(lens).to(device)
        self.max_seq_len = int(lens.max())
        self.cfg = kvq.make_config(self.lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim, w.mode, tdt)
        self.pool = torch.zeros(kvq.kvq_cache_bytes(self.cfg), dtype=torch.uint8, device=device)
        assert self.pool.numel() == cache_pool_bytes(w, self.lay)
        self.cache = kvq.kvq_cache_alloc(self.cfg, self.pool)
        if nq > 1:
            ns, tps, wsb = kvq.kvq_decode_multi_plan(self.cache, w.num_seqs, nq, w.num_q_heads, self.max_seq_len)
        else:
            ns, tps, wsb = kvq.kvq_decode_plan(self.cache, w.num_seqs, w.num_q_heads, self.max_seq_len)
        self.plan = (ns, tps, wsb)
        self.ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device=device)
        self.out = torch.empty(tuple(self.q.shape), dtype=tdt, device=device)
        self.amax = torch.zeros(2, dtype=torch.float32, device=device)
        # the decode step's append: the newest token of every sequence (the newest
        # nq tokens when nq queries are verified per step)
        ends = self.lay.token_offset[1:].astype(np.int64)
        last = np.concatenate([np.arange(max(e - min(nq, int(n)), 0), e) for e, n in zip(ends, lens) if n > 0])
        idx = torch.from_numpy(last).to(device)
        self.step_k = self.K.index_select(0, idx).contiguous()
        self.step_v = self.V.index_select(0, idx).contiguous()
        self.step_slots = self.slots.index_select(0, idx).contiguous()
        if w.mode == "kvarn_k4v2_g128":  # whole tiles only: the step re-writes each sequence's last tile
            tiles = []
            for b in range(len(lens)):
                e = int(self.lay.token_offset[b + 1])
                tiles.append(np.arange(e - 128, e))
            tidx = torch.from_numpy(np.concatenate(tiles)).to(device)
            self.step_k = self.K.index_select(0, tidx).contiguous()
            self.step_v = self.V.index_select(0, tidx).contiguous()
            self.step_slots = self.slots.index_select(0, tidx).contiguous()

    def calibrate(self):
        if self.w.mode in TENSOR_SCALED:
            self.kvq.kvq_tensor_amax(self.K, self.amax[0:1])
            self.kvq.kvq_tensor_amax(self.V, self.amax[1:2])
            self.kvq.kvq_cache_set_tensor_scales_from_amax(self.cache, self.amax[0:1], self.amax[1:2])

    def fill(self):
        self.kvq.kvq_quantize_write(self.cache, self.K, self.V, self.slots)

    def write_step(self):
        self.kvq.kvq_quantize_write(self.cache, self.step_k, self.step_v, self.step_slots)

    def decode(self, out=None, q=None):
        q = self.q if q is None else q
        out = self.out if out is None else out
        if self.w.num_queries > 1:
            self.kvq.kvq_decode_attention_multi(self.cache, q, self.block_table, self.seq_lens, out,
                                                max_seq_len=self.max_seq_len, workspace=self.ws)
        else:
            self.kvq.kvq_decode_attention(self.cache, q, self.block_table, self.seq_lens, out,
                                          max_seq_len=self.max_seq_len, workspace=self.ws)

    def launches_per_step(self) -> int:
        # write + decode, + the split combine when the split partials go through
        # memory (the plan then asks for workspace; splits merged inside a
        # thread-block cluster need none and launch no combine)
        return 1 + 1 + (1 if self.plan[2] > 0 else 0)

    def split_merge(self) -> str:
        if self.plan[0] <= 1:
            return ""
        return " + its split combine" if self.plan[2] > 0 else " (splits merged in a thread-block cluster)"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int, device=None) -> float:
    """Max over ranks (the slowest rank sets the time)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(buf):
    """Evict L2 before a timed step: write a buffer larger than L2, then read a
    second one, so that the lines the write left dirty are written back here
    and not inside the timed region (they would add ~L2-size bytes of HBM
    writes to a decode that reads little more than that)."""
    wr, rd = buf
    wr.zero_()
    rd.sum()


# --------------------------------------------------------------------------- recorded DRAM traffic
CSRC = os.path.join(ROOT, "quantized_paged_kv_quantize_gb300", "csrc")
KERNEL_SOURCES = {
    "decode_kernel": ["kvq_decode.cu", "kvq_device.cuh", "kvq_internal.h", "../_build.py"],
    "kvarn_decode_kernel": ["kvq_decode_kvarn.cu", "kvq_device.cuh", "kvq_internal.h", "../_build.py"],
    "umma_decode_kernel": ["kvq_decode_umma.cu", "kvq_device.cuh", "kvq_internal.h", "../_build.py"],
}


def decode_kernel_of(w: wl.Workload) -> str:
    """The decode kernel the library runs for the workload: the KVarN kernel, the
    tcgen05 kernel (4-bit modes at head_dim 128 with several queries per sequence
    and at most 64 query rows x heads per kv head), else the mma.sync kernel."""
    if w.mode == "kvarn_k4v2_g128":
        return "kvarn_decode_kernel"
    if (w.mode in ("nvfp4", "nvfp4_4over6", "int4_per_token_head") and w.head_dim == 128 and w.page_size == 16
            and w.num_queries >= 2 and w.group * w.num_queries <= 64):
        return "umma_decode_kernel"
    return "decode_kernel"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


def kernel_sources_hash(kernel: str) -> str:
    """sha256 of the sources a decode kernel is built from (its file, the shared
    device header and the build flags), to tell whether a recorded capture still
    describes the kernel that runs."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str, kv_tokens: int):
    """DRAM bytes (read + write) per launch of the kernel on this workload, from the
    ncu capture recorded in profiles/traffic.txt, scaled from the capture's cached
    tokens to kv_tokens; None when there is no record or the kernel's sources have
    changed since it was taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    want = kernel_sources_hash(kernel)
    for line in open(TRAFFIC_FILE):
        f = line.split()
        if len(f) == 5 and not line.startswith("#") and f[0] == workload and f[1] == kernel and f[4] == want:
            return int(round(float(f[3]) * kv_tokens / float(f[2])))
    return None


def measure(gw: GpuWorkload, args, dev, ws: int, full: bool, sampler=None) -> dict:
    """Bulk write, then W warm-up and K timed decode steps of one resident
    workload (CUDA events on the launching stream; L2 flushed before every step
    when the packed cache is under 2 x L2).  With `full`, also the end-to-end
    pass through the C ABI with host buffers.  Times are the max over ranks."""
    import torch
    w = gw.w
    stream = torch.cuda.current_stream(dev)
    lens = gw.lay.seq_lens
    dbytes = decode_bytes(w, lens)
    n_step_tok = int(gw.step_slots.numel())
    step_bytes = dbytes + write_bytes(w, n_step_tok)

    # ---- bulk fill (timed once): a0 calibration, then quantize-write of every token
    torch.cuda.synchronize()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record(stream)
    gw.calibrate()
    e1.record(stream)
    gw.fill()
    e2.record(stream)
    torch.cuda.synchronize()
    calib_ms, fill_ms = e0.elapsed_time(e1), e1.elapsed_time(e2)
    # repeat the fill a few times for a steadier write number (idempotent)
    reps = 3
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(reps):
        gw.fill()
    f1.record(stream)
    torch.cuda.synchronize()
    fill_ms = min(fill_ms, f0.elapsed_time(f1) / reps)
    flags = gw.kvq.kvq_cache_read_errors(gw.cache)
    if flags:
        raise RuntimeError(f"{w.name}: device error word after fill: {flags:#x}")
    wbytes = write_bytes(w, gw.lay.num_tokens)
    diag = tensor_diagnostics(gw)

    flush = None
    if gw.pool.numel() < 2 * L2_BYTES:
        flush = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev),
                 torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev))

    for _ in range(args.warmup):
        if flush is not None:
            flush_l2(flush)
        gw.write_step()
        gw.decode()
    torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush is not None:
            flush_l2(flush)
        starts[i].record(stream)
        gw.write_step()
        mids[i].record(stream)
        gw.decode()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler is not None else None
    step_ms = [x.elapsed_time(y) for x, y in zip(starts, ends)]
    dec_ms = [x.elapsed_time(y) for x, y in zip(mids, ends)]
    total_ms = reduce_max(float(np.sum(step_ms)), ws, dev)
    dec_total = reduce_max(float(np.sum(dec_ms)), ws, dev)
    ms_per_step = total_ms / args.steps
    dec_avg = dec_total / args.steps
    peak, peak_kind = measured_peaks()
    dec_gbs = dbytes / (dec_avg * 1e-3) / 1e9
    dec_kernel = decode_kernel_of(w)
    traffic = recorded_traffic(w.name.split("[")[0], dec_kernel, int(lens.sum()))
    tokens_heads = float(np.sum(lens.astype(np.int64))) * w.num_q_heads * w.num_queries
    res = {
        "config": config_of(w, gw.lay),
        "step": {"ms": round(ms_per_step, 5), "gbs": round(ws * step_bytes / (ms_per_step * 1e-3) / 1e9, 2),
                 "bytes": step_bytes},
        "decode": {"gbs": round(dec_gbs, 2), "us": round(dec_avg * 1e3, 2),
                   "frac_of_peak": round(dec_gbs / peak, 4), "algorithmic_bytes": dbytes,
                   "tokens_heads_per_s": tokens_heads / (dec_avg * 1e-3),
                   "splits": gw.plan[0], "tokens_per_split": gw.plan[1]},
        "write": {"bulk_gbs": round(wbytes / (fill_ms * 1e-3) / 1e9, 2), "bulk_ms": round(fill_ms, 4),
                  "bulk_bytes": wbytes, "tokens_heads_per_s": gw.lay.num_tokens * w.num_kv_heads / (fill_ms * 1e-3),
                  "calibrate_ms": round(calib_ms, 4) if w.mode in TENSOR_SCALED else None},
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "kernel": dec_kernel, "peak_kind": peak_kind,
                     "timed": dec_kernel + gw.split_merge()},
        "gpu_launches": gw.launches_per_step() * args.steps,
        "clocks": clocks,
        "diagnostics": diag,
    }
    if not full:
        return res

    # ---- end to end through the C ABI with host buffers (copies inside the timed region).
    # The step's inputs (q, the new tokens' K and V, their slots) sit in one pinned
    # staging buffer at 256-byte aligned offsets and go to the device in one copy.
    parts = [gw.q.cpu(), gw.step_k.cpu(), gw.step_v.cpu(), gw.step_slots.cpu()]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        stage_h[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        views.append(stage_d[o:o + n].view(t.dtype).view(t.shape))
    q_d, k_d, v_d, s_d = views
    out_h = torch.empty(gw.out.shape, dtype=gw.out.dtype).pin_memory()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        if flush is not None:
            flush_l2(flush)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        stage_d.copy_(stage_h, non_blocking=True)
        gw.kvq.kvq_quantize_write(gw.cache, k_d, v_d, s_d)
        gw.decode(q=q_d)
        out_h.copy_(gw.out, non_blocking=True)
        t1.record(stream)
        t1.synchronize()
        if i >= args.warmup:
            e2e_ms.append(t0.elapsed_time(t1))
    e2e_tot = reduce_max(float(np.sum(e2e_ms)), ws, dev)
    res["e2e"] = {"value": round(ws * step_bytes / (e2e_tot / args.steps * 1e-3) / 1e9, 2), "unit": "GB/s",
                  "h2d_bytes_per_step": total,
                  "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}
    flags = gw.kvq.kvq_cache_read_errors(gw.cache)
    if flags:
        raise RuntimeError(f"{w.name}: device error word after the timed steps: {flags:#x}")
    return res


DIAG_TOKENS = 16384  # tokens the tensor-level diagnostics cover (whole KVarN tiles: a multiple of 128)


def tensor_diagnostics(gw: GpuWorkload) -> dict:
    """Tensor-level error of the filled cache against its inputs (kvq_tensor_error_stats),
    K and V apart: the ratios the NVFP4 page lists under 张量层, plus the worst head.
    The first DIAG_TOKENS tokens (every one for smaller caches): the statistics are
    fp64 sums, slow on this GPU's fp64 units, and a sample of that size fixes them
    to a few digits."""
    import torch
    K = gw.kvq
    Hkv = gw.w.num_kv_heads
    n = min(int(gw.K.shape[0]), DIAG_TOKENS)
    stats = torch.zeros((2, Hkv, K.ERROR_STATS_DOUBLES), dtype=torch.float64, device=gw.dev)
    K.kvq_tensor_error_stats(gw.cache, gw.K[:n], gw.V[:n], gw.slots[:n], stats)
    st = stats.cpu().numpy()
    out = {"tokens": n}
    for side, name in enumerate(("K", "V")):
        f = {k: st[side, :, i] for i, k in enumerate(K.ERROR_STATS_FIELDS)}
        n, se, sr, sd, dot = (float(f[k].sum()) for k in ("count", "sum_sq_err", "sum_sq_ref", "sum_sq_deq", "dot"))
        head_nmse = f["sum_sq_err"] / np.maximum(f["sum_sq_ref"], 1e-300)
        hist = st[side, :, len(K.ERROR_STATS_FIELDS):].sum(axis=0)
        out[name] = {
            "mse": se / n, "nmse": se / sr, "cosine": dot / math.sqrt(sr * sd),
            "max_abs_err": float(f["max_abs_err"].max()), "zero_ratio": float(f["zeros"].sum()) / n,
            "saturation_ratio": float(f["saturated"].sum()) / n, "clipping_ratio": float(f["clipped"].sum()) / n,
            "worst_head_nmse": float(head_nmse.max()), "worst_head": int(head_nmse.argmax()),
            "scale_log2_hist": {str(b - 32): int(c) for b, c in enumerate(hist) if c},
        }
    return out


def suite_names(args) -> list:
    if args.suite == "none":
        return []
    names = SUITE if args.suite == "all" else [n for n in args.suite.split(",") if n]
    for n in names:
        workload_by_name(n)  # unknown names fail here, before any GPU work
    return [n for n in names if n != args.workload]


def run_ours(args, w: wl.Workload):
    import torch
    import torch.distributed as dist
    ws, rank, local = _dist()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    # the headline workload first: its line carries the contract keys
    gw = GpuWorkload(w, dev)
    head = measure(gw, args, dev, ws, full=True,
                   sampler=ClockSampler(dev.index if dev.index is not None else 0))
    kv = (base_of(w.name), gw.K, gw.V) if args.num_seqs is None else None
    del gw
    # then every other configuration of the suite, one at a time; mode variants
    # of a base reuse its K/V on the device
    others = {}
    for name in suite_names(args):
        wk = workload_by_name(name)
        if kv is not None and kv[0] != base_of(name):
            kv = None
            torch.cuda.empty_cache()
        try:
            g = GpuWorkload(wk, dev, kv=None if kv is None else kv[1:])
            others[name] = measure(g, args, dev, ws, full=False)
            kv = (base_of(name), g.K, g.V)
            del g
        except Exception as e:  # reported in the line; the headline stands on its own
            print(f"bench: {name} failed: {e!r}", file=sys.stderr, flush=True)
            others[name] = {"error": repr(e)}
            kv = None
        torch.cuda.empty_cache()
    del kv
    torch.cuda.empty_cache()

    result = None
    if rank == 0:
        cpu = cpu_baseline(w, args.cpu_seconds) if not args.no_cpu_baseline else None
        result = {
            "metric": METRIC,
            "value": head["step"]["gbs"],
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["step"]["ms"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16 x f16 -> f32 tensor-core math on dequantized codes (u8 storage)",
            "data": "synthetic",
            "config": head["config"],
            "decode": head["decode"],
            "write": head["write"],
            "roofline": head["roofline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "cpu_baseline": cpu,
            "diagnostics": head["diagnostics"],
            "workloads": {n: ({k: r[k] for k in ("config", "step", "decode", "write", "roofline", "gpu_launches",
                                                 "diagnostics")}
                              if "error" not in r else r) for n, r in others.items()},
        }
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


# --------------------------------------------------------------------------- oracle side
_ORACLE_POOLS = {}


def _oracle_seq_pool(w: wl.Workload, b: int):
    """The oracle's own packed pages of sequence b (built once, not timed)."""
    import oracle
    key = (w.name, b)
    if key not in _ORACLE_POOLS:
        n = int(wl.seq_lens(w)[b])
        k, v = wl.gen_kv_seq(w, b, n)
        P = w.page_size
        npg = (n + P - 1) // P
        ks = vs = 1.0
        if w.mode in TENSOR_SCALED:
            ks = oracle.tensor_scale(w.mode, oracle.amax(k.astype(np.float32)))
            vs = oracle.tensor_scale(w.mode, oracle.amax(v.astype(np.float32)))
        pool = np.zeros(oracle.pool_bytes(w.mode, npg, P, w.num_kv_heads, w.head_dim), np.uint8)
        idx = np.arange(n)
        oracle.write(w.mode, pool, npg, P, w.num_kv_heads, w.head_dim, k.astype(np.float32),
                     v.astype(np.float32), (idx // P * P + idx % P).astype(np.int32), ks, vs)
        _ORACLE_POOLS[key] = (pool, npg, n, ks, vs)
    return _ORACLE_POOLS[key]


def oracle_sample(w: wl.Workload, seconds: float, start: int = 0):
    """Time the oracle (as it stands, one thread) on decode work units of the
    workload: one unit = one (sequence, kv head) group, i.e. the G query heads
    that share those pages.  Runs units until `seconds` are spent.
    Returns (algorithmic bytes, seconds, units, next start)."""
    import oracle
    G = w.group
    esz = 2 if w.io_dtype == "f16" else 4
    nq = w.num_queries
    q_all = wl.gen_q(w, w.num_seqs * nq).astype(np.float32)
    done_bytes, spent, units, u = 0, 0.0, 0, start
    while nq > 1:  # one unit = one (sequence, kv head) group: its G query heads, every query
        b, kvh = (u // w.num_kv_heads) % w.num_seqs, u % w.num_kv_heads
        pool, npg, n, ks, vs = _oracle_seq_pool(w, b)
        qb = q_all[b * nq:(b + 1) * nq].reshape(1, nq, w.num_q_heads, w.head_dim)
        rows = (np.arange(nq)[:, None] * w.num_q_heads + kvh * G + np.arange(G)[None, :]).reshape(-1)
        t0 = time.perf_counter()
        oracle.decode_multi(w.mode, pool, npg, w.page_size, w.num_kv_heads, w.head_dim, qb,
                            np.arange(npg, dtype=np.int32)[None], np.array([n], np.int32),
                            1.0 / math.sqrt(w.head_dim), ks, vs, rows=rows)
        spent += time.perf_counter() - t0
        done_bytes += int(n * bytes_per_token_head(w)) + 2 * nq * G * w.head_dim * esz
        units += 1
        u += 1
        if spent >= seconds:
            return done_bytes, spent, units, u
    while True:
        b, kvh = (u // w.num_kv_heads) % w.num_seqs, u % w.num_kv_heads
        pool, npg, n, ks, vs = _oracle_seq_pool(w, b)
        rows = np.arange(G, dtype=np.int32) + kvh * G
        t0 = time.perf_counter()
        oracle.decode(w.mode, pool, npg, w.page_size, w.num_kv_heads, w.head_dim, q_all[b:b + 1],
                      np.arange(npg, dtype=np.int32)[None], np.array([n], np.int32),
                      1.0 / math.sqrt(w.head_dim), ks, vs, rows=rows)
        spent += time.perf_counter() - t0
        done_bytes += int(n * bytes_per_token_head(w)) + 2 * G * w.head_dim * esz
        units += 1
        u += 1
        if spent >= seconds:
            return done_bytes, spent, units, u


def cpu_baseline(w: wl.Workload, seconds: float):
    import oracle
    oracle.build()
    nb, sec, units, _ = oracle_sample(w, seconds)
    return {"value": round(nb / sec / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": (f"{units} (sequence, kv head) groups of {w.name} decoded by the single-threaded C oracle "
                       f"(each: all {w.group} query heads over the full sequence), {sec:.1f} s")
            if w.num_queries == 1 else
            (f"{units} (sequence, kv head) groups of {w.name} decoded by the single-threaded C oracle (each: "
             f"all {w.group} query heads, {w.num_queries} causal queries over the full sequence), {sec:.1f} s")}


def run_reference(args, w: wl.Workload):
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    u = 0
    for _ in range(args.warmup):
        _, _, _, u = oracle_sample(w, 0.0, u)
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, s, _, u = oracle_sample(w, 0.0, u)
        tot_b += b
        tot_s += s
    val = tot_b / tot_s / 1e9
    return {
        "metric": METRIC, "value": round(val, 6), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention from stored codes (oracle)",
        "data": "synthetic", "impl": "reference",
        "config": config_of(w),
        "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: one (sequence, kv head) group of {w.name} decoded by the "
                                   f"single-threaded C oracle"},
        "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(wl.WORKLOADS) + sorted(VARIANTS) + sorted(SPEC_VARIANTS))
    ap.add_argument("--suite", default="all",
                    help="the other configurations measured after the headline one: 'all' (default), "
                         "'none', or a comma-separated list of workload names")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="shrink the batch (same shapes otherwise), e.g. to size an ncu capture; "
                         "implies --suite none")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    w = workload_by_name(args.workload)
    if args.num_seqs is not None:
        import dataclasses
        w = dataclasses.replace(w, num_seqs=args.num_seqs, name=f"{w.name}[B={args.num_seqs}]")
        args.suite = "none"
    res = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
