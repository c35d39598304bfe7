"""The allocation-free decode entry point, kvq_decode_attention_noalloc.

It serves callers that cannot allocate device memory when they decode (a
memory pool sized and frozen in advance, or a host embedding the library with
no device allocator): the split scratch is the library's own fixed array.  This
file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process."""
import math

import numpy as np
import pytest
import torch

import oracle
from _helpers import check_attention, guarded, kvq, make_case, gpu_cache, oracle_pool
from test_parity import small_workload

pytestmark = pytest.mark.gpu


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("mode,D,io", [("nvfp4", 128, "f16"), ("int8_per_token_head", 32, "f32"),
                                       ("kvarn_k4v2_g128", 128, "f16")])
def test_noalloc_matches_workspace_entry_point_twice(mode, D, io):
    """Two calls in a row with different queries.  The built-in scratch and a
    caller workspace run the same kernels on the same plan, so the outputs must
    be bit-identical (a stale partial left in the scratch by the first call
    would show here); both are also checked against the oracle."""
    K = kvq()
    lens = [128, 256, 640, 2048] if mode == "kvarn_k4v2_g128" else [17, 100, 333, 1000, 2500]
    c = make_case(small_workload(mode, D=D, io=io), lens, slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    cache.pool[256:].copy_(torch.from_numpy(pool[256:]).cuda())
    K.kvq_cache_set_tensor_scales(cache, c.k_scale, c.v_scale)
    B, Hq, Dh = c.q.shape
    msl = int(max(lens))
    ns, tps, wsb = K.kvq_decode_plan(cache, B, Hq, msl)
    assert ns > 1 and 0 < wsb <= K.NOALLOC_SCRATCH_BYTES   # the scratch is really used
    bt, sl = _dev(c.lay.block_table), _dev(c.lay.seq_lens)
    ws = guarded(wsb // 4, torch.float32, name="workspace")
    rng = np.random.default_rng(3)
    for call in range(2):   # the second call finds the first call's partials in the scratch
        q_np = (c.q.astype(np.float32) * (1.0 + 0.5 * call) + rng.standard_normal(c.q.shape) * 0.1).astype(c.q.dtype)
        q = _dev(q_np)
        ref = guarded((B, Hq, Dh), torch.float32, fill=float("nan"), name="out (workspace entry point)")
        out = guarded((B, Hq, Dh), torch.float32, fill=float("nan"), name="out (allocation-free entry point)")
        K.kvq_decode_attention(cache, q, bt, sl, ref, max_seq_len=msl, workspace=ws)
        K.kvq_decode_attention_noalloc(cache, q, bt, sl, out, max_seq_len=msl)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: max abs difference {(out - ref).abs().max().item():.3e}"
        want = oracle.decode(mode, pool, c.lay.num_pages, c.w.page_size, c.w.num_kv_heads, c.w.head_dim,
                             q_np.astype(np.float32), c.lay.block_table, c.lay.seq_lens, 1.0 / math.sqrt(Dh),
                             c.k_scale, c.v_scale)
        check_attention(out, want)
        check_attention(ref, want)
    assert K.kvq_cache_read_errors(cache) == 0


def test_noalloc_rejects_plans_larger_than_its_scratch():
    K = kvq()
    cfg = K.make_config(4096, 16, 8, 128, "int8_per_token_head")
    pool = torch.zeros(K.kvq_cache_bytes(cfg), dtype=torch.uint8, device="cuda")
    cache = K.kvq_cache_alloc(cfg, pool)
    B, Hq, msl = 512, 64, 32768
    _, _, wsb = K.kvq_decode_plan(cache, B, Hq, msl)
    assert wsb > K.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, Hq, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    bt = torch.zeros((B, msl // 16), dtype=torch.int32, device="cuda")
    sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
    with pytest.raises(K.KVQError) as e:
        K.kvq_decode_attention_noalloc(cache, q, bt, sl, out, max_seq_len=msl)
    assert e.value.status == 4 and "scratch" in str(e.value)
