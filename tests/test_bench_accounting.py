"""bench.py's algorithmic byte counts, tied to the oracle's page layout (CPU):
the bytes per token and kv head it charges a decode are the page block's
bytes per token, and a decode pass reads every cached token once plus the
per-tensor scales, and moves each query row in and out once."""
import dataclasses
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads as wl  # noqa: E402


@pytest.mark.parametrize("mode", sorted(bench.BYTES_PER_TOKEN_HEAD))
@pytest.mark.parametrize("D", [32, 128])
def test_bytes_per_token_head_is_the_page_layout(mode, D):
    P = 128 if mode == "kvarn_k4v2_g128" else 16
    if P == 128 and D != 128:
        pytest.skip("KVarN has head_dim 128 only")
    w = dataclasses.replace(wl.WORKLOADS["pth_b64_u1k_32k"].with_mode(mode), head_dim=D, page_size=P)
    assert bench.bytes_per_token_head(w) * P == oracle.block_bytes(mode, P, D)
    if D == 128:
        assert bench.BYTES_PER_TOKEN_HEAD[mode] * P == oracle.block_bytes(mode, P, 128)


def test_tiny_config_bytes_are_the_pages_fake_quant_bytes():
    """The [P3] experiment's shape (B=2, H=4, T=16, D=32): 8192 B of int8 K+V
    and 1024 B of fp32 scales, plus q and out (fp32)."""
    w = wl.WORKLOADS["int8_pth_tiny"]
    lens = wl.seq_lens(w)
    assert bench.decode_bytes(w, lens) == 8192 + 1024 + 2 * 2 * 4 * 32 * 4
    lay = wl.paged_layout(w)
    assert bench.cache_pool_bytes(w, lay) == oracle.pool_bytes(w.mode, lay.num_pages, 16, 4, 32)


@pytest.mark.parametrize("nq", [1, 4])
@pytest.mark.parametrize("mode", ["nvfp4", "int8_per_token_head", "fp8_per_tensor", "int4_per_token_head"])
def test_decode_bytes(mode, nq):
    w = dataclasses.replace(wl.WORKLOADS["pth_b64_u1k_32k"].with_mode(mode), num_seqs=5, num_queries=nq)
    lens = np.array([1, 16, 17, 1000, 32768], np.int32)
    esz = 2
    kv = int(lens.sum()) * w.num_kv_heads * oracle.block_bytes(mode, 16, 128) // 16
    scales = 8 if mode in bench.TENSOR_SCALED else 0
    qo = 2 * w.num_seqs * nq * w.num_q_heads * w.head_dim * esz
    assert bench.decode_bytes(w, lens) == kv + scales + qo


def test_write_bytes():
    w = wl.WORKLOADS["nvfp4_b32_s32768"]
    n = 1000
    packed = oracle.block_bytes("nvfp4", 16, 128) // 16          # bytes per token and kv head, K + V
    assert bench.write_bytes(w, n) == n * w.num_kv_heads * (2 * 128 * 2 + packed) + 4 * n
