"""KVarN open tiles on the GPU, through the C ABI, against the oracle.

A sequence's whole tiles are quantized into pages (kvq_quantize_write or, when
a tile fills up, kvq_kvarn_append); the rows of its incomplete last tile live
raw in the tail buffer.  Checked: the tail rows are the appended inputs, bit
for bit; a tile completed by appends is byte-identical to the oracle's
quantization of those 128 tokens; decode over tiles + tail is within the
attention tolerance of the oracle's fp64 attention over the same tokens."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import check_attention, guarded, kvq

pytestmark = pytest.mark.gpu

P, D = 128, 128


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class Seqs:
    """Sequences of the given lengths with their pages, inputs and the oracle's pool."""

    def __init__(self, lens, Hq=16, Hkv=2, io="f16", seed=31, slack_pages=2):
        self.w = wl.Workload(name="tail", mode="kvarn_k4v2_g128", num_seqs=len(lens), num_q_heads=Hq,
                             num_kv_heads=Hkv, head_dim=D, page_size=P, io_dtype=io, seed=seed,
                             seq_len_range=(1, 1), outlier_channels=4, channels_per_head=True, channel_gain=15.0)
        self.lens = np.asarray(lens, np.int32)
        cap = np.maximum(self.lens + 130, 1).astype(np.int32)      # room to append past the end
        self.lay = wl.paged_layout(self.w, cap, slack_pages=slack_pages)
        self.kv = [wl.gen_kv_seq(self.w, b, int(cap[b])) for b in range(len(lens))]
        self.q = wl.gen_q(self.w)
        K = kvq()
        tdt = torch.float16 if io == "f16" else torch.float32
        self.cfg = K.make_config(self.lay.num_pages, P, Hkv, D, "kvarn_k4v2_g128", tdt)
        self.pool = guarded(K.kvq_cache_bytes(self.cfg), torch.uint8, fill=0xCD, name="pool")
        self.cache = K.kvq_cache_alloc(self.cfg, self.pool)
        B = len(lens)
        self.tail = guarded(K.kvq_kvarn_tail_bytes(self.cache, B), torch.uint8, fill=0, name="tail")
        self.ref_pool = np.full(oracle.pool_bytes("kvarn_k4v2_g128", self.lay.num_pages, P, Hkv, D), 0xCD, np.uint8)
        self.tail_np = np.zeros((2, B, P, Hkv, D), self.w.np_dtype)

    def slot(self, b, t):
        return int(self.lay.block_table[b, t // P]) * P + t % P

    def write_whole_tiles(self, b, t0, t1):
        """Tokens [t0, t1) of sequence b, whole tiles, through kvq_quantize_write."""
        k, v = self.kv[b]
        slots = np.array([self.slot(b, t) for t in range(t0, t1)], np.int32)
        kvq().kvq_quantize_write(self.cache, _dev(k[t0:t1]), _dev(v[t0:t1]), _dev(slots))
        oracle.write("kvarn_k4v2_g128", self.ref_pool, self.lay.num_pages, P, self.w.num_kv_heads, D,
                     k[t0:t1].astype(np.float32), v[t0:t1].astype(np.float32), slots)

    def append(self, items):
        """One kvq_kvarn_append call for (b, t) tokens; the oracle side copies the
        rows into its tail and quantizes every tile the call completes."""
        ks = np.stack([self.kv[b][0][t] for b, t in items])
        vs = np.stack([self.kv[b][1][t] for b, t in items])
        slots = np.array([self.slot(b, t) for b, t in items], np.int32)
        seqs = np.array([b for b, _ in items], np.int32)
        kvq().kvq_kvarn_append(self.cache, _dev(ks), _dev(vs), _dev(slots), _dev(seqs), self.tail,
                               len(self.lens))
        for (b, t), kk, vv in zip(items, ks, vs):
            self.tail_np[0, b, t % P], self.tail_np[1, b, t % P] = kk, vv
        for b, t in items:
            if t % P == P - 1:
                tile = np.arange(t - P + 1, t + 1)
                oracle.write("kvarn_k4v2_g128", self.ref_pool, self.lay.num_pages, P, self.w.num_kv_heads, D,
                             self.tail_np[0, b].astype(np.float32), self.tail_np[1, b].astype(np.float32),
                             np.array([self.slot(b, x) for x in tile], np.int32))

    def check_pool_and_tail(self):
        got = self.pool.cpu().numpy()
        diff = np.flatnonzero(got[256:] != self.ref_pool[256:])
        assert diff.size == 0, f"{diff.size} pool bytes differ, first at {256 + diff[0]}"
        B = len(self.lens)
        t = self.tail.cpu().numpy().view(self.w.np_dtype).reshape(2, B, P, self.w.num_kv_heads, D)
        for b, n in enumerate(self.lens):
            r = int(n) % P
            assert np.array_equal(t[:, b, :r].view(np.uint8), self.tail_np[:, b, :r].view(np.uint8)), b

    def decode(self, lens, out_dtype=torch.float32):
        K = kvq()
        B, Hq = len(lens), self.w.num_q_heads
        msl = int(max(lens)) if len(lens) else 0
        ws = guarded(max(K.kvq_kvarn_decode_workspace_bytes(self.cache, B, Hq, msl) // 4, 1), torch.float32,
                     name="workspace")
        out = guarded((B, Hq, D), out_dtype, fill=float("nan"), name="out")
        K.kvq_kvarn_decode_attention(self.cache, _dev(self.q), _dev(self.lay.block_table),
                                     _dev(np.asarray(lens, np.int32)), self.tail, out, max_seq_len=msl,
                                     workspace=ws)
        torch.cuda.synchronize()
        ref = oracle.decode_kvarn_tail(self.ref_pool, self.lay.num_pages, self.w.num_kv_heads,
                                       self.q.astype(np.float32), self.lay.block_table, np.asarray(lens, np.int32),
                                       1.0 / math.sqrt(D), self.tail_np[0].astype(np.float32),
                                       self.tail_np[1].astype(np.float32))
        check_attention(out, ref)
        return out


def _fill(s: Seqs):
    """Whole tiles by kvq_quantize_write, the rest of each sequence by appends
    (one token per sequence per call, as decode steps append)."""
    for b, n in enumerate(s.lens):
        nf = int(n) - int(n) % P
        if nf:
            s.write_whole_tiles(b, 0, nf)
    rest = [[(b, t) for t in range(int(n) - int(n) % P, int(n))] for b, n in enumerate(s.lens)]
    for step in range(max(len(r) for r in rest)):
        s.append([r[step] for r in rest if step < len(r)])


@pytest.mark.parametrize("io,out_dtype", [("f16", torch.float32), ("f16", torch.float16), ("f32", torch.float32)])
def test_tail_decode_parity(io, out_dtype):
    s = Seqs([0, 1, 100, 127, 128, 200, 383, 1000], io=io)
    _fill(s)
    s.check_pool_and_tail()
    assert kvq().kvq_cache_read_errors(s.cache) == 0
    out = s.decode(s.lens, out_dtype)
    assert (out[0] == 0).all()


def test_tail_decode_many_splits_and_single_split():
    """Long sequences (several KV splits each) and a batch short enough for
    one split, both merged with their tails."""
    s = Seqs([5000, 3000 + 77], Hq=8, Hkv=1)
    _fill(s)
    K = kvq()
    ns, _, _ = K.kvq_decode_plan(s.cache, 2, 8, 5000)
    assert ns > 1
    s.decode(s.lens)
    # enough (sequence, kv head) units to fill the GPU with one split each
    s2 = Seqs([130, 129, 255, 200] * 160, Hq=4, Hkv=2, seed=5)
    _fill(s2)
    ns2, _, _ = K.kvq_decode_plan(s2.cache, 640, 4, 255)
    assert ns2 == 1
    s2.decode(s2.lens)


def test_append_completes_tiles_and_starts_the_next():
    """Appends that fill a tile quantize it into its page (byte-exact with the
    oracle); the next tile's first rows then start in the tail."""
    s = Seqs([120, 250, 3], Hq=8, Hkv=2)
    _fill(s)
    s.check_pool_and_tail()
    # finish every open tile: 8, 6 and 125 more tokens, in chunks of up to 8 tokens per sequence
    todo = [list(range(int(n), (int(n) // P + 1) * P)) for n in s.lens]
    while any(todo):
        items = []
        for b, r in enumerate(todo):
            items += [(b, t) for t in r[:8]]
            del r[:8]
        s.append(items)
    lens = np.array([(int(n) // P + 1) * P for n in s.lens], np.int32)
    s.lens = lens
    s.check_pool_and_tail()
    s.decode(lens)                                   # whole tiles only, empty tails
    # the next tile: 1, 2 and 3 tokens
    s.append([(b, int(lens[b]) + j) for b in range(3) for j in range(b + 1)])
    s.lens = lens + np.array([1, 2, 3], np.int32)
    s.check_pool_and_tail()
    s.decode(s.lens, torch.float16)
    assert kvq().kvq_cache_read_errors(s.cache) == 0


def test_append_flags_bad_sequence_ids_and_slots():
    K = kvq()
    s = Seqs([10, 10], Hq=8, Hkv=2)
    k, v = s.kv[0]
    slots = np.array([s.slot(0, 10), s.slot(0, 11), s.lay.num_pages * P + 3, -1], np.int32)
    seqs = np.array([0, 7, 0, 1], np.int32)                       # seq id 7 >= 2: flagged
    K.kvq_kvarn_append(s.cache, _dev(k[10:14]), _dev(v[10:14]), _dev(slots), _dev(seqs), s.tail, 2)
    assert K.kvq_cache_read_errors(s.cache) == 0x20 | 0x1
    t = s.tail.cpu().numpy().view(s.w.np_dtype).reshape(2, 2, P, 2, D)
    assert np.array_equal(t[0, 0, 10].view(np.uint16), k[10].view(np.uint16))   # the good token landed
    assert not t[:, 0, 11].any() and not t[:, 1].any()                          # the others did not
    with pytest.raises(K.KVQError) as e:                                        # not a KVarN cache
        cfg = K.make_config(4, 16, 2, 128, "nvfp4", torch.float16)
        pool = torch.zeros(K.kvq_cache_bytes(cfg), dtype=torch.uint8, device="cuda")
        K.kvq_kvarn_tail_bytes(K.kvq_cache_alloc(cfg, pool), 2)
    assert e.value.status == 3


def test_append_across_two_tiles_of_a_sequence_is_flagged():
    """One call carrying rows 126, 127 of a sequence's tile and row 0 of its
    next tile breaks the one-tile-per-call rule: the tile is not written (its
    page keeps the fill bytes) and KVQ_DEVERR_PARTIAL_TILE is set; another
    sequence completing its tile in the same call is written normally."""
    K = kvq()
    s = Seqs([126, 126], Hq=8, Hkv=2)
    _fill(s)
    assert K.kvq_cache_read_errors(s.cache) == 0
    s.append([(1, 126), (1, 127)])                      # sequence 1: a clean completion
    k0, v0 = s.kv[0]
    items = [(0, 126), (0, 127), (0, 128)]              # sequence 0: crosses into its next tile
    ks = np.stack([k0[t] for _, t in items])
    vs = np.stack([v0[t] for _, t in items])
    slots = np.array([s.slot(0, t) for _, t in items], np.int32)
    K.kvq_kvarn_append(s.cache, _dev(ks), _dev(vs), _dev(slots), _dev(np.zeros(3, np.int32)), s.tail, 2)
    assert K.kvq_cache_read_errors(s.cache) == 0x4
    blk = oracle.block_bytes("kvarn_k4v2_g128", P, D)
    page0 = int(s.lay.block_table[0, 0])
    got = s.pool.cpu().numpy()
    for h in range(2):
        o0 = 256 + (page0 * 2 + h) * blk
        assert (got[o0:o0 + blk] == 0xCD).all()        # sequence 0's tile was not written
    s.lens = np.array([126, 128], np.int32)             # sequence 1's tile matches the oracle
    page1 = int(s.lay.block_table[1, 0])
    for h in range(2):
        o1 = 256 + (page1 * 2 + h) * blk
        assert np.array_equal(got[o1:o1 + blk], s.ref_pool[o1:o1 + blk])



def test_append_completion_with_an_out_of_range_slot_alongside():
    """A call that completes a sequence's tile and also carries a token of the
    same sequence whose slot lies past the pool: that token is skipped and
    flagged (KVQ_DEVERR_SLOT_RANGE) and overwrites nothing, so the tile is still
    complete and is quantized (byte-identical to the oracle); no partial-tile
    flag is raised."""
    K = kvq()
    s = Seqs([126], Hq=8, Hkv=2)
    _fill(s)
    assert K.kvq_cache_read_errors(s.cache) == 0
    k0, v0 = s.kv[0]
    ks = np.stack([k0[126], k0[127], k0[128]])
    vs = np.stack([v0[126], v0[127], v0[128]])
    slots = np.array([s.slot(0, 126), s.slot(0, 127), s.lay.num_pages * P + 5], np.int32)
    K.kvq_kvarn_append(s.cache, _dev(ks), _dev(vs), _dev(slots), _dev(np.zeros(3, np.int32)), s.tail, 1)
    assert K.kvq_cache_read_errors(s.cache) == 0x1
    for t in (126, 127):
        s.tail_np[0, 0, t], s.tail_np[1, 0, t] = k0[t], v0[t]
    oracle.write("kvarn_k4v2_g128", s.ref_pool, s.lay.num_pages, P, s.w.num_kv_heads, D,
                 s.tail_np[0, 0].astype(np.float32), s.tail_np[1, 0].astype(np.float32),
                 np.array([s.slot(0, x) for x in range(P)], np.int32))
    s.lens = np.array([128], np.int32)
    s.check_pool_and_tail()
    s.decode(s.lens)
