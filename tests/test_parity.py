"""GPU parity of libkvq against the CPU oracle, through the C ABI.

Quantize-on-write: pool bytes and scales bit-exact.  Decode attention: fp32
outputs within 2e-3 max-abs of the fp64 oracle; fp16 outputs within 2e-3 of
fp16(oracle) or one fp16 ulp of it.  Sizes here finish on the oracle in
seconds but span several pages, several KV splits and ragged tails."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import (guarded, FILL, TENSOR_SCALED, check_attention, gpu_cache, gpu_calibrate, gpu_decode, header_scales,
                      kvq, make_case, oracle_decode, oracle_pool)

pytestmark = pytest.mark.gpu

MODES4 = ["fp8_per_tensor", "int8_per_token_head", "fp8_per_token_head", "nvfp4", "int4_per_token_head",
          "nvfp4_4over6"]
FOUR_BIT = ["nvfp4", "nvfp4_4over6", "int4_per_token_head"]
LENS = [1, 15, 16, 17, 100, 333, 1000, 2500]
KVARN_LENS = [128, 256, 640]


def small_workload(mode, D=128, Hq=16, Hkv=2, io="f16", seed=7):
    """Small shapes with the outlier structure of the mode's full-size workload."""
    P = 128 if mode == "kvarn_k4v2_g128" else 16
    extra = {
        "fp8_per_tensor": dict(sink_tokens=4, sink_gain=20.0),
        "int8_per_token_head": dict(outlier_token_frac=0.01, token_gain=30.0),
        "fp8_per_token_head": dict(outlier_token_frac=0.01, token_gain=30.0),
        "nvfp4": dict(outlier_channels=3, channels_per_head=True, channel_gain=10.0),
        "nvfp4_4over6": dict(outlier_channels=3, channels_per_head=True, channel_gain=10.0),
        "int4_per_token_head": dict(outlier_token_frac=0.01, token_gain=30.0),
        "kvarn_k4v2_g128": dict(outlier_channels=4, channels_per_head=True, channel_gain=15.0),
    }[mode]
    return wl.Workload(name=f"small_{mode}_{D}_{io}", mode=mode, num_seqs=1, num_q_heads=Hq, num_kv_heads=Hkv,
                       head_dim=D, page_size=P, io_dtype=io, seed=seed, seq_len_range=(1, 1), **extra)


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _upload_oracle_pool(cache, pool_np, c):
    cache.pool[256:].copy_(torch.from_numpy(pool_np[256:]).cuda())
    kvq().kvq_cache_set_tensor_scales(cache, c.k_scale, c.v_scale)


# ------------------------------------------------------------------ write
@pytest.mark.parametrize("D,io", [(128, "f16"), (32, "f32"), (32, "f16"), (128, "f32")])
@pytest.mark.parametrize("mode", MODES4)
def test_write_bit_exact(mode, D, io):
    K = kvq()
    c = make_case(small_workload(mode, D=D, io=io), LENS[:6], slack_pages=2)
    slots = c.slots.copy()
    slots[3] = -1                                    # skipped token
    slots[7] = c.lay.num_pages * 16 + 5              # out of range: skipped and flagged
    cache = gpu_cache(c)
    kd, vd = _dev(c.k), _dev(c.v)
    if mode in TENSOR_SCALED:
        gpu_calibrate(cache, kd, vd)
        ks, vs = header_scales(cache)
        assert np.float32(ks) == np.float32(c.k_scale) and np.float32(vs) == np.float32(c.v_scale)
    K.kvq_quantize_write(cache, kd, vd, _dev(slots))
    flags = K.kvq_cache_read_errors(cache)
    assert flags == 0x1, hex(flags)
    got = cache.pool.cpu().numpy()
    ref = oracle_pool(c, slots=slots)
    diff = np.flatnonzero(got[256:] != ref[256:])
    assert diff.size == 0, f"{diff.size} bytes differ, first at pool offset {256 + diff[0]}"


@pytest.mark.parametrize("io", ["f16", "f32"])
@pytest.mark.parametrize("order", ["reversed", "random", "split_calls", "one_by_one"])
@pytest.mark.parametrize("mode", FOUR_BIT)
def test_write_4bit_values_any_batch_order(mode, order, io):
    """4-bit values share a byte between tokens 2k and 2k+1: written as whole
    pairs when the two tokens are neighbours in the batch, else nibble by
    nibble.  Any batch order, split over any number of calls, must give the
    oracle's bytes."""
    K = kvq()
    c = make_case(small_workload(mode, io=io), [1, 15, 16, 17, 100, 333], slack_pages=2)
    cache = gpu_cache(c)
    kd, vd = _dev(c.k), _dev(c.v)
    if mode in TENSOR_SCALED:
        gpu_calibrate(cache, kd, vd)
    n = len(c.slots)
    rng = np.random.default_rng(11)
    if order == "reversed":
        calls = [np.arange(n)[::-1]]
    elif order == "random":
        calls = [rng.permutation(n)]
    elif order == "split_calls":               # every other token, then the rest, in two calls
        calls = [np.arange(0, n, 2), np.arange(1, n, 2)]
    else:
        calls = [np.array([i]) for i in rng.permutation(n)[:40]] + [np.arange(n)]
    for idx in calls:
        idx = np.ascontiguousarray(idx)
        K.kvq_quantize_write(cache, _dev(c.k[idx]), _dev(c.v[idx]), _dev(c.slots[idx]))
    assert K.kvq_cache_read_errors(cache) == 0
    got = cache.pool.cpu().numpy()
    ref = oracle_pool(c)
    diff = np.flatnonzero(got[256:] != ref[256:])
    assert diff.size == 0, f"{diff.size} bytes differ, first at pool offset {256 + diff[0]}"


@pytest.mark.parametrize("io", ["f16", "f32"])
def test_write_kvarn_bit_exact(io):
    K = kvq()
    c = make_case(small_workload("kvarn_k4v2_g128", io=io), KVARN_LENS, slack_pages=1)
    cache = gpu_cache(c)
    K.kvq_quantize_write(cache, _dev(c.k), _dev(c.v), _dev(c.slots))
    assert K.kvq_cache_read_errors(cache) == 0
    got = cache.pool.cpu().numpy()
    ref = oracle_pool(c)
    diff = np.flatnonzero(got[256:] != ref[256:])
    assert diff.size == 0, f"{diff.size} bytes differ, first at pool offset {256 + diff[0]}"


def test_write_kvarn_degenerate_tiles():
    """Tiles whose normalisation steps meet std < 1e-8 (left unchanged) and
    whose rounding meets zero ranges (all codes 0): an all-zero tile, a tile of
    one constant, a tile whose tokens are all equal, and one constant channel."""
    K = kvq()
    c = make_case(small_workload("kvarn_k4v2_g128"), [512], slack_pages=1)
    k, v = c.k.copy(), c.v.copy()
    k[0:128] = 0
    v[0:128] = 0
    k[128:256] = np.asarray(0.75, k.dtype)
    v[128:256] = np.asarray(-1.5, v.dtype)
    k[256:384] = k[256:257]                 # every token of the tile equal
    v[256:384] = v[256:257]
    k[384:512, :, 5] = np.asarray(2.0, k.dtype)   # one constant channel
    v[384:512, :, 7] = np.asarray(-3.0, v.dtype)
    cache = gpu_cache(c)
    K.kvq_quantize_write(cache, _dev(k), _dev(v), _dev(c.slots))
    assert K.kvq_cache_read_errors(cache) == 0
    got = cache.pool.cpu().numpy()
    ref = oracle_pool(c, k=k, v=v)
    diff = np.flatnonzero(got[256:] != ref[256:])
    assert diff.size == 0, f"{diff.size} bytes differ, first at pool offset {256 + diff[0]}"


def test_write_kvarn_partial_tile_is_flagged_and_skipped():
    K = kvq()
    c = make_case(small_workload("kvarn_k4v2_g128"), [256], slack_pages=1)
    slots = c.slots.copy()
    slots[128:] = slots[128:] + 1                      # second tile no longer fills a page in order
    slots[-1] = slots[128] - 1
    cache = gpu_cache(c)
    K.kvq_quantize_write(cache, _dev(c.k), _dev(c.v), _dev(slots))
    assert K.kvq_cache_read_errors(cache) == 0x4
    got = cache.pool.cpu().numpy()
    ref = oracle_pool(c, slots=slots)
    assert (got[256:] == ref[256:]).all()


def test_write_conversion_edge_values():
    """E4M3 and E2M1 ties, signed zeros, tiny values and saturation go through the
    hardware conversions exactly as the format definitions say."""
    K = kvq()
    pos = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (pos[1:] + pos[:-1]) / 2
    vals = np.concatenate([pos, mids, -pos, -mids, [0.0, -0.0, 1e-8, -1e-8, 500.0, -500.0, 6e4, -6e4]])
    vals = vals.astype(np.float16)
    D = 128
    n = (len(vals) + D - 1) // D
    row = np.zeros(n * D, np.float16)
    row[:len(vals)] = vals
    x = row.reshape(n, 1, D)
    w = wl.Workload(name="edge", mode="fp8_per_tensor", num_seqs=1, num_q_heads=1, num_kv_heads=1, head_dim=D,
                    page_size=16, io_dtype="f16", seed=1, seq_len=n)
    for mode, ks in (("fp8_per_tensor", 1.0), ("nvfp4", 1.0), ("fp8_per_token_head", None),
                     ("int8_per_token_head", None), ("nvfp4_4over6", 1.0), ("int4_per_token_head", None)):
        wm = w.with_mode(mode)
        lay = wl.paged_layout(wm, np.array([n], np.int32))
        c = make_case(wm, [n])
        c.k, c.v = x, (x * np.float16(0.75)).astype(np.float16)
        c.slots = wl.slots_for_seq(wm, lay, 0)
        c.lay = lay
        c.k_scale = c.v_scale = 1.0
        cache = gpu_cache(c)
        K.kvq_cache_set_tensor_scales(cache, 1.0, 1.0)
        K.kvq_quantize_write(cache, _dev(c.k), _dev(c.v), _dev(c.slots))
        got = cache.pool.cpu().numpy()
        ref = oracle_pool(c)
        assert (got[256:] == ref[256:]).all(), mode
    # E2M1 ties: with s_t = 1 a block whose max is 6 has s_b = 1 and x/(s_t s_b) = x;
    # INT4 ties: a row whose max is 7 has s = 1 and x/s = x
    ties = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -5.0, 0.0, -0.0, 0.1, -0.1],
                    np.float16)
    ties4 = np.array([7.0, 0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, -0.5, -1.5, -2.5, -6.5, 0.0, -0.0, 6.9, -7.0],
                     np.float16)
    for mode, t in (("nvfp4", ties), ("nvfp4_4over6", ties), ("int4_per_token_head", ties4)):
        xt = np.tile(t, D // 16).reshape(1, 1, D)
        xt = np.repeat(xt, 16, axis=0)
        wm = w.with_mode(mode)
        lay = wl.paged_layout(wm, np.array([16], np.int32))
        c = make_case(wm, [16])
        c.k, c.v, c.lay = xt, xt, lay
        c.slots = wl.slots_for_seq(wm, lay, 0)
        c.k_scale = c.v_scale = 1.0
        cache = gpu_cache(c)
        K.kvq_cache_set_tensor_scales(cache, 1.0, 1.0)
        K.kvq_quantize_write(cache, _dev(c.k), _dev(c.v), _dev(c.slots))
        got = cache.pool.cpu().numpy()
        assert (got[256:] == oracle_pool(c)[256:]).all(), mode


def test_write_4over6_uses_both_scales():
    """The 4over6 write matches the oracle and really differs from plain NVFP4:
    a sizeable share of blocks keep the max/4 scale."""
    K = kvq()
    c = make_case(small_workload("nvfp4_4over6"), [16, 100, 333], slack_pages=1)
    cache = gpu_cache(c)
    kd, vd = _dev(c.k), _dev(c.v)
    gpu_calibrate(cache, kd, vd)
    K.kvq_quantize_write(cache, kd, vd, _dev(c.slots))
    got = cache.pool.cpu().numpy()
    assert (got[256:] == oracle_pool(c)[256:]).all()
    n4 = n = 0
    for t in range(0, len(c.slots), 7):
        for x, s_t in ((c.k[t, 0], c.k_scale), (c.v[t, 0], c.v_scale)):
            _, _, ch = oracle.nvfp4_4over6_row(x.astype(np.float32), s_t)
            n4 += int((ch == 4).sum())
            n += ch.size
    assert 0.1 < n4 / n < 0.9, n4 / n


def test_tensor_amax_exact():
    K = kvq()
    rng = np.random.default_rng(0)
    for n in (1, 7, 8, 1000, 123457):
        x = (rng.standard_normal(n) * 50).astype(np.float16)
        out = torch.zeros(1, dtype=torch.float32, device="cuda")
        K.kvq_tensor_amax(_dev(x), out)
        assert out.item() == np.abs(x.astype(np.float32)).max()
        xf = x.astype(np.float32)
        K.kvq_tensor_amax(_dev(xf), out)
        assert out.item() == np.abs(xf).max()


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("D,io,Hq,Hkv", [(128, "f16", 16, 2), (128, "f16", 8, 2), (32, "f32", 4, 4),
                                         (32, "f16", 16, 2), (128, "f32", 8, 1)])
@pytest.mark.parametrize("mode", MODES4)
def test_decode_parity(mode, D, io, Hq, Hkv, out_dtype):
    c = make_case(small_workload(mode, D=D, io=io, Hq=Hq, Hkv=Hkv), LENS + [0], slack_pages=2)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    out, plan = gpu_decode(cache, c, out_dtype=out_dtype)
    assert plan[0] > 1, "the case should exercise several KV splits"
    ref = oracle_decode(c, pool)
    check_attention(out, ref)
    assert kvq().kvq_cache_read_errors(cache) == 0


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("nseq", [40, 76])
@pytest.mark.parametrize("mode", MODES4)
def test_decode_cluster_merge_parity(mode, nseq, out_dtype):
    """Enough sequences that 2 to 8 splits fill one wave of CTAs: the splits
    of each row then run as one thread-block cluster and merge on chip, and
    the plan asks for no workspace (40 sequences: 7 splits, 76: 4 splits at 4
    CTAs per SM).  Ragged lengths leave the later splits of short rows empty;
    a zero-length row gives zeros."""
    rng = np.random.default_rng(nseq)
    lens = [int(x) for x in rng.integers(1, 2501, size=nseq - 3)] + [0, 2500, 16]
    c = make_case(small_workload(mode), lens, slack_pages=2)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    out, plan = gpu_decode(cache, c, out_dtype=out_dtype)
    assert 2 <= plan[0] <= 8 and plan[2] == 0, f"plan {plan}: the case should merge its splits in a cluster"
    check_attention(out, oracle_decode(c, pool))
    assert (out[nseq - 3] == 0).all()
    assert kvq().kvq_cache_read_errors(cache) == 0


@pytest.mark.parametrize("mode", MODES4)
def test_decode_empty_and_single_token(mode):
    c = make_case(small_workload(mode), [0, 1, 16, 0, 2], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    out, _ = gpu_decode(cache, c)
    ref = oracle_decode(c, pool)
    check_attention(out, ref)
    assert (out[0] == 0).all() and (out[3] == 0).all()


@pytest.mark.parametrize("mode", ["int8_per_token_head", "nvfp4", "int4_per_token_head"])
def test_decode_bad_page_and_long_seq_are_flagged(mode):
    K = kvq()
    c = make_case(small_workload(mode), [300, 200], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    bt = c.lay.block_table.copy()
    bt[0, 3] = 10 ** 6                                   # out-of-range page id: its tokens drop out
    out, _ = gpu_decode(cache, c, bt=bt)
    assert K.kvq_cache_read_errors(cache) == 0x2
    check_attention(out, oracle_decode(c, pool, bt=bt))
    out2, _ = gpu_decode(cache, c, max_seq_len=256)      # seq 0 (300 tokens) exceeds the bound
    assert K.kvq_cache_read_errors(cache) & 0x8
    check_attention(out2, oracle_decode(c, pool, lens=np.array([256, 200], np.int32)))


def test_decode_tiny_config_end_to_end():
    """The tiny INT8 per-token-head workload (fp32 K, V, q; D=32; B=2; T=16)
    through write + decode on the GPU, against the oracle's write + decode."""
    K = kvq()
    w = wl.WORKLOADS["int8_pth_tiny"]
    c = make_case(w, list(wl.seq_lens(w)))
    cache = gpu_cache(c)
    K.kvq_quantize_write(cache, _dev(c.k), _dev(c.v), _dev(c.slots))
    pool = oracle_pool(c)
    assert (cache.pool.cpu().numpy()[256:] == pool[256:]).all()
    out, plan = gpu_decode(cache, c)
    check_attention(out, oracle_decode(c, pool))


def test_mode_mismatch_and_unsupported():
    K = kvq()
    c = make_case(small_workload("nvfp4"), [16])
    cache = gpu_cache(c)
    with pytest.raises(K.KVQError) as e:
        K.kvq_quantize_write(cache, _dev(c.k), _dev(c.v), _dev(c.slots), mode="fp8_per_tensor")
    assert e.value.status == 3
    out = torch.empty((1, 16, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(K.KVQError) as e:
        K.kvq_decode_attention(cache, _dev(c.q), _dev(c.lay.block_table), _dev(c.lay.seq_lens), out,
                               max_seq_len=16, mode="int8_per_token_head")
    assert e.value.status == 3


# ------------------------------------------------------------------ KVarN decode
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("Hq,Hkv,io", [(16, 2, "f16"), (8, 2, "f16"), (2, 2, "f16"), (8, 1, "f32")])
def test_decode_kvarn_parity(Hq, Hkv, io, out_dtype):
    c = make_case(small_workload("kvarn_k4v2_g128", Hq=Hq, Hkv=Hkv, io=io), KVARN_LENS + [0, 2048],
                  slack_pages=2)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    out, plan = gpu_decode(cache, c, out_dtype=out_dtype)
    assert plan[0] > 1
    check_attention(out, oracle_decode(c, pool))
    assert kvq().kvq_cache_read_errors(cache) == 0


def test_decode_kvarn_single_split_and_partial_tile():
    K = kvq()
    c = make_case(small_workload("kvarn_k4v2_g128"), [128, 0], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    out, plan = gpu_decode(cache, c)
    assert plan[0] == 1
    check_attention(out, oracle_decode(c, pool))
    # a sequence that ends inside a tile: only whole tiles are read, and it is flagged
    c2 = make_case(small_workload("kvarn_k4v2_g128"), [256, 0], slack_pages=1)
    pool2 = oracle_pool(c2)
    cache2 = gpu_cache(c2)
    _upload_oracle_pool(cache2, pool2, c2)
    out2, _ = gpu_decode(cache2, c2, lens=np.array([200, 0], np.int32), max_seq_len=256)
    assert K.kvq_cache_read_errors(cache2) & 0x4
    check_attention(out2, oracle_decode(c2, pool2, lens=np.array([128, 0], np.int32)))


# ------------------------------------------------------------------ multi-query decode
@pytest.mark.parametrize("nq,out_dtype", [(2, torch.float32), (4, torch.float16), (7, torch.float32)])
@pytest.mark.parametrize("mode", MODES4)
def test_decode_multi_query_parity(mode, nq, out_dtype):
    """nq queries per sequence under the causal mask, against the oracle; the
    last query row of each sequence equals the plain decode of that query."""
    K = kvq()
    c = make_case(small_workload(mode), [3, 16, 100, 1000, 2500], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    B, Hq, D = len(c.lay.seq_lens), c.w.num_q_heads, c.w.head_dim
    rng = np.random.default_rng(nq)
    q = rng.standard_normal((B, nq, Hq, D)).astype(c.w.np_dtype)
    msl = int(c.lay.seq_lens.max())
    wsb = K.kvq_decode_multi_workspace_bytes(cache, B, nq, Hq, msl)
    ws = guarded(max(wsb // 4, 1), torch.float32, name="workspace")
    out = guarded((B, nq, Hq, D), out_dtype, fill=float("nan"), name="out")
    K.kvq_decode_attention_multi(cache, _dev(q), _dev(c.lay.block_table), _dev(c.lay.seq_lens), out,
                                 max_seq_len=msl, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.decode_multi(c.w.mode, pool, c.lay.num_pages, c.w.page_size, c.w.num_kv_heads, D,
                              q.astype(np.float32), c.lay.block_table, c.lay.seq_lens, 1.0 / math.sqrt(D),
                              c.k_scale, c.v_scale)
    check_attention(out.reshape(B * nq, Hq, D), ref.reshape(B * nq, Hq, D))
    assert (out[0, :max(nq - 3, 0)] == 0).all()          # sequence of 3 tokens: queries before it see nothing
    one = torch.empty((B, Hq, D), dtype=out_dtype, device="cuda")
    ws1 = torch.empty(max(K.kvq_decode_workspace_bytes(cache, B, Hq, msl) // 4, 1), dtype=torch.float32,
                      device="cuda")
    K.kvq_decode_attention(cache, _dev(np.ascontiguousarray(q[:, -1])), _dev(c.lay.block_table),
                           _dev(c.lay.seq_lens), one, max_seq_len=msl, workspace=ws1)
    torch.cuda.synchronize()
    check_attention(one, ref[:, -1])
    assert K.kvq_cache_read_errors(cache) == 0


@pytest.mark.parametrize("nq,Hq,io,out_dtype", [(2, 16, "f16", torch.float32), (5, 16, "f16", torch.float16),
                                                (3, 8, "f32", torch.float32)])
def test_decode_multi_query_kvarn_parity(nq, Hq, io, out_dtype):
    """KVarN, nq causal queries per sequence over whole tiles: the earlier
    queries' prefixes end inside the last tile (tokens 124..127 of a 128-token
    sequence with nq = 5), across split boundaries (2048 tokens), and the last
    query row equals the plain decode of that query."""
    K = kvq()
    c = make_case(small_workload("kvarn_k4v2_g128", Hq=Hq, io=io), [128, 256, 0, 2048, 640], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    B, D = len(c.lay.seq_lens), c.w.head_dim
    q = np.random.default_rng(nq).standard_normal((B, nq, Hq, D)).astype(c.w.np_dtype)
    msl = int(c.lay.seq_lens.max())
    ns, _, wsb = K.kvq_decode_multi_plan(cache, B, nq, Hq, msl)
    assert ns > 1
    ws = guarded(max(wsb // 4, 1), torch.float32, name="workspace")
    out = guarded((B, nq, Hq, D), out_dtype, fill=float("nan"), name="out")
    K.kvq_decode_attention_multi(cache, _dev(q), _dev(c.lay.block_table), _dev(c.lay.seq_lens), out,
                                 max_seq_len=msl, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.decode_multi(c.w.mode, pool, c.lay.num_pages, c.w.page_size, c.w.num_kv_heads, D,
                              q.astype(np.float32), c.lay.block_table, c.lay.seq_lens, 1.0 / math.sqrt(D))
    check_attention(out.reshape(B * nq, Hq, D), ref.reshape(B * nq, Hq, D))
    assert (out[2] == 0).all()                            # the empty sequence
    assert K.kvq_cache_read_errors(cache) == 0
    one = torch.empty((B, Hq, D), dtype=out_dtype, device="cuda")
    ws1 = torch.empty(max(K.kvq_decode_workspace_bytes(cache, B, Hq, msl) // 4, 1), dtype=torch.float32,
                      device="cuda")
    K.kvq_decode_attention(cache, _dev(np.ascontiguousarray(q[:, -1])), _dev(c.lay.block_table),
                           _dev(c.lay.seq_lens), one, max_seq_len=msl, workspace=ws1)
    torch.cuda.synchronize()
    check_attention(one, ref[:, -1])


@pytest.mark.parametrize("mode,nq,Hkv", [("nvfp4", 4, 2), ("nvfp4_4over6", 3, 2), ("int8_per_token_head", 4, 2),
                                         ("nvfp4", 2, 8)])
def test_decode_multi_query_one_split(mode, nq, Hkv):
    """Short sequences (one KV split: outputs written by the decode kernel
    itself), empty ones and ones shorter than the query count."""
    K = kvq()
    c = make_case(small_workload(mode, Hq=16, Hkv=Hkv), [0, 1, 3, 16, 40, 64], slack_pages=1)
    pool = oracle_pool(c)
    cache = gpu_cache(c)
    _upload_oracle_pool(cache, pool, c)
    B, Hq, D = len(c.lay.seq_lens), c.w.num_q_heads, c.w.head_dim
    q = np.random.default_rng(3).standard_normal((B, nq, Hq, D)).astype(c.w.np_dtype)
    msl = int(c.lay.seq_lens.max())
    wsb = K.kvq_decode_multi_workspace_bytes(cache, B, nq, Hq, msl)
    ws = guarded(max(wsb // 4, 1), torch.float32, name="workspace")
    out = guarded((B, nq, Hq, D), torch.float32, fill=float("nan"), name="out")
    K.kvq_decode_attention_multi(cache, _dev(q), _dev(c.lay.block_table), _dev(c.lay.seq_lens), out,
                                 max_seq_len=msl, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.decode_multi(c.w.mode, pool, c.lay.num_pages, c.w.page_size, c.w.num_kv_heads, D,
                              q.astype(np.float32), c.lay.block_table, c.lay.seq_lens, 1.0 / math.sqrt(D),
                              c.k_scale, c.v_scale)
    check_attention(out.reshape(B * nq, Hq, D), ref.reshape(B * nq, Hq, D))
    assert (out[0] == 0).all()
    assert K.kvq_cache_read_errors(cache) == 0
