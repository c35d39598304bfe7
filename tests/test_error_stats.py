"""Tensor-level quantization error (kvq_tensor_error_stats) against the same
quantities computed in numpy from the oracle's dequantization of the oracle's
own pool ("NVFP4 KV Cache…", 量化误差该怎样测, 张量层: MSE / normalised MSE,
max absolute error, cosine similarity, zero ratio, clipping and saturation,
scale distribution, per head, K and V apart)."""
import math

import numpy as np
import pytest
import torch

import oracle
from _helpers import gpu_cache, guarded, kvq, make_case, oracle_pool
from test_parity import small_workload

pytestmark = pytest.mark.gpu

FIELDS = ["count", "sum_sq_err", "sum_sq_ref", "sum_sq_deq", "dot", "max_abs_err", "zeros", "saturated", "clipped"]


def _gpu_stats(cache, c):
    K = kvq()
    stats = guarded((2, c.w.num_kv_heads, K.ERROR_STATS_DOUBLES), torch.float64, name="stats")
    K.kvq_tensor_error_stats(cache, torch.from_numpy(c.k).cuda(), torch.from_numpy(c.v).cuda(),
                             torch.from_numpy(c.slots).cuda(), stats)
    torch.cuda.synchronize()
    return stats.cpu().numpy()


def _oracle_rows(c, pool):
    """Dequantized rows [side][head][token][D] in the input domain (fp64)."""
    w = c.w
    H = None
    if w.mode == "kvarn_k4v2_g128":
        from scipy.linalg import hadamard
        H = hadamard(128).astype(np.float64) / math.sqrt(128)
    N = len(c.slots)
    out = np.zeros((2, w.num_kv_heads, N, w.head_dim))
    for i, s in enumerate(c.slots):
        for h in range(w.num_kv_heads):
            for side in range(2):
                r = oracle.dequant_row(w.mode, pool, c.lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim,
                                       c.k_scale, c.v_scale, int(s), h, side)
                out[side, h, i] = r @ H if H is not None else r
    return out


@pytest.mark.parametrize("mode,D,io", [("int8_per_token_head", 128, "f16"), ("fp8_per_token_head", 128, "f16"),
                                       ("fp8_per_tensor", 128, "f16"), ("nvfp4", 128, "f16"),
                                       ("nvfp4_4over6", 128, "f16"), ("int4_per_token_head", 128, "f16"),
                                       ("int8_per_token_head", 32, "f32"), ("kvarn_k4v2_g128", 128, "f16")])
def test_error_sums_match_the_oracle(mode, D, io):
    lens = [128, 256] if mode == "kvarn_k4v2_g128" else [17, 40, 3]
    c = make_case(small_workload(mode, D=D, io=io), lens, slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    cache.pool[256:].copy_(torch.from_numpy(pool[256:]).cuda())
    kvq().kvq_cache_set_tensor_scales(cache, c.k_scale, c.v_scale)
    got = _gpu_stats(cache, c)
    deq = _oracle_rows(c, pool)
    x = np.stack([c.k.astype(np.float64).transpose(1, 0, 2), c.v.astype(np.float64).transpose(1, 0, 2)])
    rtol = 2e-4 if mode == "kvarn_k4v2_g128" else 2e-6   # fp32 rows (and a fp32 rotation) on the GPU
    for side in range(2):
        for h in range(c.w.num_kv_heads):
            g = dict(zip(FIELDS, got[side, h, :9]))
            xr, xh = x[side, h], deq[side, h]
            e = xh - xr
            assert g["count"] == xr.size
            assert g["sum_sq_err"] == pytest.approx(float((e * e).sum()), rel=10 * rtol, abs=1e-9)
            assert g["sum_sq_ref"] == pytest.approx(float((xr * xr).sum()), rel=1e-9)
            assert g["sum_sq_deq"] == pytest.approx(float((xh * xh).sum()), rel=rtol)
            assert g["dot"] == pytest.approx(float((xr * xh).sum()), rel=rtol)
            assert g["max_abs_err"] == pytest.approx(float(np.abs(e).max()), rel=50 * rtol, abs=1e-6)
            if mode != "kvarn_k4v2_g128":
                assert g["zeros"] == float((xh == 0).sum())
            nmse = g["sum_sq_err"] / g["sum_sq_ref"]
            cosine = g["dot"] / math.sqrt(g["sum_sq_ref"] * g["sum_sq_deq"])
            assert 0 <= nmse < 0.25 and cosine > 0.9      # a sane quantizer, K and V alike


def test_per_token_head_saturation_and_scale_histogram():
    """INT8 per-token-head: each row's largest magnitude maps to +-127
    (saturated, never clipped), and the histogram holds each row's stored
    scale at floor(log2 s) + 32."""
    c = make_case(small_workload("int8_per_token_head", D=128, io="f16"), [20, 7], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    cache.pool[256:].copy_(torch.from_numpy(pool[256:]).cuda())
    got = _gpu_stats(cache, c)
    w = c.w
    x = [c.k.astype(np.float32), c.v.astype(np.float32)]
    for side in range(2):
        for h in range(w.num_kv_heads):
            want = np.zeros(64)
            sat = 0
            for row in x[side][:, h, :]:
                q, s = oracle.quant_row("int8_per_token_head", row)
                sat += int((np.abs(q.view(np.int8).astype(np.int32)) == 127).sum())
                s = float(s.view(np.float32)[0])
                want[min(max(math.floor(math.log2(s)) + 32, 0), 63)] += 1
            assert sat >= len(x[side]) and got[side, h, 7] == sat   # saturated: at least each row's max
            assert got[side, h, 8] == 0                              # clipped: never
            assert np.array_equal(got[side, h, 9:], want)


def test_fp8_per_tensor_clipping_is_counted():
    """A per-tensor scale four times too small: every |x / s| past 448 + 16
    (half the last step of the E4M3 grid) is clipped, and saturated too."""
    c = make_case(small_workload("fp8_per_tensor", D=128, io="f16"), [33, 60], slack_pages=1)
    c.k_scale = c.k_scale / 4
    c.v_scale = c.v_scale / 4
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    cache.pool[256:].copy_(torch.from_numpy(pool[256:]).cuda())
    kvq().kvq_cache_set_tensor_scales(cache, c.k_scale, c.v_scale)
    got = _gpu_stats(cache, c)
    for side, (x, s) in enumerate([(c.k, c.k_scale), (c.v, c.v_scale)]):
        for h in range(c.w.num_kv_heads):
            r = np.abs(x[:, h, :].astype(np.float64))
            top = float(np.float32(448.0) * np.float32(s))   # the dequantized top value, rounded as fp32
            clipped = ((r - top) > 16.0 * float(np.float32(s))).sum()
            assert clipped > 0 and got[side, h, 8] == clipped
            assert got[side, h, 7] >= clipped
