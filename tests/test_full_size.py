"""Parity at the workloads' full sizes, in the launch configuration bench.py
times: the same bulk quantize-write, the same decode plan.  The oracle
recomputes sampled sequences one by one (their page blocks byte-exact, their
decode rows within the attention tolerance); properties that hold at any size
are checked on every output."""
import math

import numpy as np
import pytest
import torch

import bench
import oracle
import workloads as wl
from _helpers import check_attention, guarded

pytestmark = pytest.mark.gpu

CASES = [
    ("fp8_pt_b16_s4096", None, [0, 15]),
    ("pth_b64_u1k_32k", None, None),            # shortest and longest sequence
    ("pth_b64_u1k_32k", "fp8_per_token_head", None),
    ("nvfp4_b32_s32768", None, [5]),
    ("pth_b64_u1k_32k", "int4_per_token_head", None),
    ("nvfp4_b32_s32768", "nvfp4_4over6", [7]),
    ("kvarn_b16_s16384", None, [3]),
]


def _workload(name, mode):
    w = wl.WORKLOADS[name]
    return w.with_mode(mode) if mode else w


@pytest.mark.parametrize("name,mode,sample", CASES)
def test_full_size_sampled_parity(name, mode, sample):
    w = _workload(name, mode)
    gw = bench.GpuWorkload(w, keep_host=True)
    gw.calibrate()
    gw.fill()
    for _ in range(3):                       # the timed step: append + decode
        gw.write_step()
        gw.decode()
    out16 = gw.out.clone()
    out32 = guarded(tuple(gw.out.shape), torch.float32, name="out")
    gw.decode(out32)
    torch.cuda.synchronize()
    assert gw.kvq.kvq_cache_read_errors(gw.cache) == 0
    assert torch.isfinite(out16.float()).all() and torch.isfinite(out32).all()

    lens = gw.lay.seq_lens
    if sample is None:
        sample = [int(np.argmin(lens)), int(np.argmax(lens))]
    P, Hkv, D = w.page_size, w.num_kv_heads, w.head_dim
    ks = vs = 1.0
    if w.mode in ("fp8_per_tensor", "nvfp4", "nvfp4_4over6"):
        ak = max(oracle.amax(k.astype(np.float32)) for k, _ in gw.host)
        av = max(oracle.amax(v.astype(np.float32)) for _, v in gw.host)
        ks, vs = oracle.tensor_scale(w.mode, ak), oracle.tensor_scale(w.mode, av)
        hdr = gw.pool[:24].cpu().numpy()
        assert hdr[16:20].view(np.float32)[0] == np.float32(ks)
        assert hdr[20:24].view(np.float32)[0] == np.float32(vs)
    blk = oracle.block_bytes(w.mode, P, D)
    pool_gpu = gw.pool.cpu().numpy()
    q = wl.gen_q(w).astype(np.float32)
    for b in sample:
        n = int(lens[b])
        k, v = gw.host[b]
        npg = (n + P - 1) // P
        pool = np.zeros(oracle.pool_bytes(w.mode, npg, P, Hkv, D), np.uint8)
        idx = np.arange(n)
        assert oracle.write(w.mode, pool, npg, P, Hkv, D, k.astype(np.float32), v.astype(np.float32),
                            idx.astype(np.int32), ks, vs) == 0
        for j in range(npg):                 # every page block of the sequence, byte-exact
            pid = int(gw.lay.block_table[b, j])
            for h in range(Hkv):
                g0 = 256 + (pid * Hkv + h) * blk
                o0 = 256 + (j * Hkv + h) * blk
                assert np.array_equal(pool_gpu[g0:g0 + blk], pool[o0:o0 + blk]), (b, j, h)
        ref = oracle.decode(w.mode, pool, npg, P, Hkv, D, q[b:b + 1], np.arange(npg, dtype=np.int32)[None],
                            np.array([n], np.int32), 1.0 / math.sqrt(D), ks, vs)
        check_attention(out16[b:b + 1], ref)
        check_attention(out32[b:b + 1], ref)


def test_full_size_spec_decode_sampled_parity():
    """The 4-queries-per-sequence NVFP4 workload (B=32 x 32768) in the launch
    configuration bench.py times; sequence 9's pages byte-exact and its query
    rows of kv heads 0 and 5 (all 4 queries, 8 heads each) against the oracle."""
    import dataclasses
    base, nq = bench.SPEC_VARIANTS["nvfp4_b32_s32768:spec4"]
    w = dataclasses.replace(wl.WORKLOADS[base], num_queries=nq, name="nvfp4_b32_s32768:spec4")
    gw = bench.GpuWorkload(w, keep_host=True)
    gw.calibrate()
    gw.fill()
    for _ in range(3):
        gw.write_step()
        gw.decode()
    out32 = guarded(tuple(gw.out.shape), torch.float32, name="out")
    gw.decode(out32)
    torch.cuda.synchronize()
    assert gw.kvq.kvq_cache_read_errors(gw.cache) == 0
    assert torch.isfinite(out32).all() and torch.isfinite(gw.out.float()).all()
    b, P, Hkv, D, Hq, G = 9, w.page_size, w.num_kv_heads, w.head_dim, w.num_q_heads, w.group
    k, v = gw.host[b]
    n = len(k)
    ak = max(oracle.amax(x.astype(np.float32)) for x, _ in gw.host)
    av = max(oracle.amax(y.astype(np.float32)) for _, y in gw.host)
    ks, vs = oracle.tensor_scale(w.mode, ak), oracle.tensor_scale(w.mode, av)
    npg = (n + P - 1) // P
    pool = np.zeros(oracle.pool_bytes(w.mode, npg, P, Hkv, D), np.uint8)
    assert oracle.write(w.mode, pool, npg, P, Hkv, D, k.astype(np.float32), v.astype(np.float32),
                        np.arange(n, dtype=np.int32), ks, vs) == 0
    blk = oracle.block_bytes(w.mode, P, D)
    pool_gpu = gw.pool.cpu().numpy()
    for j in range(npg):
        pid = int(gw.lay.block_table[b, j])
        for h in range(Hkv):
            g0, o0 = 256 + (pid * Hkv + h) * blk, 256 + (j * Hkv + h) * blk
            assert np.array_equal(pool_gpu[g0:g0 + blk], pool[o0:o0 + blk]), (j, h)
    q = gw.q[b:b + 1].float().cpu().numpy()                         # [1][nq][Hq][D]
    rows = [i * Hq + kvh * G + h for kvh in (0, 5) for i in range(nq) for h in range(G)]
    ref = oracle.decode_multi(w.mode, pool, npg, P, Hkv, D, q, np.arange(npg, dtype=np.int32)[None],
                              np.array([n], np.int32), 1.0 / math.sqrt(D), ks, vs, rows=rows)
    check_attention(out32[b:b + 1].reshape(1, nq * Hq, D), ref.reshape(1, nq * Hq, D), rows=np.array(rows))
    check_attention(gw.out[b:b + 1].reshape(1, nq * Hq, D), ref.reshape(1, nq * Hq, D), rows=np.array(rows))
