"""Pins of the CPU oracle to facts that do not come from the oracle itself:
values the pages print, format definitions, closed forms, invariants, library
routines (torch's float8 cast, scipy's Hadamard matrix, torch SDPA) and brute
force on tiny inputs.  CPU only."""
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(path):
    out = {}
    for line in open(os.path.join(GOLDEN, path)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        for tok in line.split():
            if "=" in tok:
                k, v = tok.split("=")
                out[k] = float(v)
    return out


# --------------------------------------------------------------------------- E2M1
def test_e2m1_value_set_matches_page():
    vals = [float(x) for line in open(os.path.join(GOLDEN, "e2m1_values.txt"))
            if not line.startswith("#") for x in line.split()]
    dec = [oracle.e2m1_decode(c) for c in range(16)]
    assert dec[:8] == vals
    assert dec[8:] == [-v for v in vals]
    assert math.copysign(1.0, dec[8]) == -1.0  # 0x8 is negative zero


def test_e2m1_encoder_ties_and_saturation():
    # round-to-nearest-even on the E2M1 grid: a tie picks the even-mantissa code
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             6.0: 6.0, 7.0: 6.0, 1e9: 6.0, 0.2: 0.0, 0.3: 0.5, 4.9: 4.0, 5.1: 6.0}
    for x, want in cases.items():
        assert oracle.e2m1_decode(oracle.e2m1_encode(x)) == want, x
        assert oracle.e2m1_decode(oracle.e2m1_encode(-x)) == -want, x
    assert oracle.e2m1_encode(-0.0) == 0x8
    assert oracle.e2m1_encode(-0.1) == 0x8


def test_e2m1_encoder_is_nearest_on_dense_sweep():
    grid = np.array([oracle.e2m1_decode(c) for c in range(8)])
    xs = np.concatenate([np.arange(-8 * 64, 8 * 64 + 1) / 64.0,
                         np.random.default_rng(7).uniform(-7, 7, 3000)]).astype(np.float32)
    for x in xs:
        c = oracle.e2m1_encode(float(x))
        got = oracle.e2m1_decode(c)
        a = min(abs(float(x)), 6.0)
        dist = np.abs(grid - a)
        assert abs(abs(got) - a) == dist.min(), x
        ties = np.flatnonzero(dist == dist.min())
        if len(ties) == 2:           # exact midpoint: even code
            assert (c & 7) % 2 == 0, x
        if x != 0:
            assert (c >> 3) == (1 if x < 0 else 0)


# --------------------------------------------------------------------------- E4M3
def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    same = (ref == got) | (np.isnan(ref) & np.isnan(got))
    assert same.all()
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_float8_in_range():
    rng = np.random.default_rng(11)
    pos = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)     # every tie
    xs = np.concatenate([mids, -mids, rng.uniform(-448, 448, 20000),
                         rng.standard_normal(20000) * 1e-2, rng.standard_normal(2000) * 1e-4]
                        ).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert (ref == got).all()


def test_e4m3_saturation_and_sign_of_zero():
    for x in (448.0, 460.0, 464.0, 500.0, 1e30):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0 ** -12) == 0x80
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00      # tie between 0 and 2^-9: even (zero)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02   # 1.5 x 2^-9 ties to 2 x 2^-9
    assert oracle.e4m3_encode(3 * 2.0 ** -11) == 0x01   # 0.75 x 2^-9 is nearest to 2^-9


# --------------------------------------------------------------------------- INT8
def test_int8_encoder_half_even_and_clip():
    assert [oracle.int8_encode(x) for x in (0.5, 1.5, 2.5, -0.5, -1.5, 126.5, 127.4, 200.0, -200.0)] \
        == [0, 2, 2, 0, -2, 126, 127, 127, -127]


def test_int8_pth_row_properties():
    rng = np.random.default_rng(3)
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.uniform(1e-3, 50)).astype(np.float32)
        q, sb = oracle.quant_row("int8_per_token_head", x)
        s = float(sb.view(np.float32)[0])
        q = q.view(np.int8).astype(np.float64)
        amax = np.abs(x).max()
        assert s == np.float32(np.float32(amax) / np.float32(127.0))
        assert np.abs(q).max() == 127 and np.abs(q).max() <= 127
        err = np.abs(q * s - x)
        assert err.max() <= s / 2 * (1 + 1e-6) + 1e-12
    q, sb = oracle.quant_row("int8_per_token_head", np.zeros(32, np.float32))
    assert (q == 0).all() and sb.view(np.float32)[0] == np.float32(np.float32(1e-8) / np.float32(127))


# --------------------------------------------------------------------------- INT4
def test_int4_encoder_half_even_and_clip():
    assert [oracle.int4_encode(x) for x in (0.5, 1.5, 2.5, -2.5, -0.5, 6.5, 7.4, 7.6, 100.0, -100.0)] \
        == [0, 2, 2, -2, 0, 6, 7, 7, 7, -7]


def _nibbles(q):
    """Packed bytes -> signed 4-bit codes (even index from the low nibble)."""
    n = np.stack([q & 15, q >> 4], 1).reshape(-1).astype(np.int64)
    return np.where(n >= 8, n - 16, n)


def test_int4_pth_row_properties():
    """s = fp32(max|x|)/7; codes are numpy's half-even round of the fp32
    quotient, clipped to +-7; the row max maps to +-7; error <= s/2."""
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.uniform(1e-3, 50)).astype(np.float32)
        q, sb = oracle.quant_row("int4_per_token_head", x)
        s = np.float32(sb.view(np.float32)[0])
        assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(7.0))
        codes = _nibbles(q)
        ref = np.clip(np.round(x / s), -7, 7).astype(np.int64)   # fp32 quotient, half-even
        assert np.array_equal(codes, ref)
        assert np.abs(codes).max() == 7
        assert np.abs(codes * np.float64(s) - x).max() <= float(s) / 2 * (1 + 1e-6) + 1e-12
    q, sb = oracle.quant_row("int4_per_token_head", np.zeros(32, np.float32))
    assert (q == 0).all() and sb.view(np.float32)[0] == np.float32(np.float32(1e-8) / np.float32(7))


def test_int4_pth_page_bytes():
    """The page's per-token-head content formula: int4 keeps head_size/2 bytes
    of data per side plus the two fp32 scales."""
    g = _kv("per_token_head_bytes.txt")
    P, D = 16, int(g["head_size"])
    assert oracle.block_bytes("int8_per_token_head", P, D) == P * g["int8_bytes"]
    assert oracle.block_bytes("int4_per_token_head", P, D) == P * g["int4_bytes"]


def test_fake_quant_bytes_and_ratio():
    """The page's printed byte counts and ratio, from the oracle's page layout."""
    g = _kv("fake_quant_int8.txt")
    B, H, T, D = int(g["B"]), int(g["H"]), int(g["T"]), int(g["D"])
    P = 16
    blk = oracle.block_bytes("int8_per_token_head", P, D)
    n_blocks = B * H * (T // P)
    payload = 2 * P * D * n_blocks
    scales = (blk - 2 * P * D) * n_blocks
    assert payload == g["int8_payload_bytes"]
    assert scales == g["scale_metadata_bytes"]
    fp16 = 2 * (B * H * T * D) * 2
    assert fp16 == g["fp16_payload_bytes"]
    assert round(fp16 / (blk * n_blocks), 3) == g["effective_compression_ratio"]


def test_fake_quant_replay_bounds():
    """Replay of the page's experiment (torch CPU RNG, seed 137, draw order q, k, v).
    The printed errors are not reproduced by the CPU generator (the page's device is
    unstated), so the pin is the listing's own tolerance and the s/2 bound."""
    g = _kv("fake_quant_int8.txt")
    torch.manual_seed(137)
    b, h, t, d = 2, 4, 16, 32
    q = torch.randn(b, h, 1, d, dtype=torch.float32)
    k = torch.randn(b, h, t, d, dtype=torch.float32)
    v = torch.randn_like(k)

    def fq(x):
        rows = x.reshape(-1, d).numpy()
        out = np.zeros_like(rows, dtype=np.float64)
        for i, r in enumerate(rows):
            qq, sb = oracle.quant_row("int8_per_token_head", r)
            out[i] = qq.view(np.int8) * float(sb.view(np.float32)[0])
        return torch.from_numpy(out.reshape(x.shape))

    kh, vh = fq(k), fq(v)
    assert (kh - k.double()).abs().max() <= g["listing_atol"]
    assert (vh - v.double()).abs().max() <= g["listing_atol"]
    ref = torch.softmax(q.double() @ k.double().transpose(-2, -1) / math.sqrt(d), -1) @ v.double()
    qa = torch.softmax(q.double() @ kh.transpose(-2, -1) / math.sqrt(d), -1) @ vh
    err = (qa - ref).abs().max().item()
    assert err <= g["listing_atol"]
    assert 0.1 * g["attention_max_abs_error"] < err < 10 * g["attention_max_abs_error"]


# --------------------------------------------------------------------------- FP8 PT / PTH
def test_fp8_pth_row_against_torch_cast():
    rng = np.random.default_rng(5)
    for _ in range(100):
        x = (rng.standard_normal(128) * rng.uniform(1e-2, 30)).astype(np.float32)
        q, sb = oracle.quant_row("fp8_per_token_head", x)
        s = sb.view(np.float32)[0]
        assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(448.0))
        y = torch.from_numpy((x / s).astype(np.float32))   # |x/s| <= 448 (+ rounding)
        ref = y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert (ref == q).all()
        assert np.abs(q & 0x7F).max() == 0x7E   # the row max maps to 448


def test_fp8_per_tensor_scale_and_row():
    assert oracle.fp8_tensor_scale(448.0) == 1.0
    assert oracle.fp8_tensor_scale(0.0) == 1.0          # all-zero tensor keeps the default 1.0
    x = np.array([0.0, -0.0, 1.0, -3.5, 100.0, 104.0, 896.0, 1e6], np.float32)
    q, _ = oracle.quant_row("fp8_per_tensor", x, 2.0)
    ref = torch.from_numpy(np.clip(x / np.float32(2.0), -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert list(q) == ref.tolist()
    assert oracle.e4m3_decode(q[4]) == 48.0             # 50 ties between 48 and 52: even mantissa
    assert q[6] == 0x7E and q[7] == 0x7E                # 448 and saturation


# --------------------------------------------------------------------------- NVFP4
def test_nvfp4_format_arithmetic():
    g = _kv("nvfp4_format.txt")
    P, D = 16, 128
    blk = oracle.block_bytes("nvfp4", P, D)
    bits = blk * 8 / (2 * P * D)
    assert bits == g["bits_per_value"]
    assert blk // (2 * P) == 72                     # bytes per token-head per side
    assert round(16 / bits, 2) == g["ratio_vs_bf16"]
    assert round(8 / bits, 2) == g["ratio_vs_fp8"]
    assert round(bits / 16, 2) == g["fraction_of_fp16"]


def test_per_token_head_scale_counts():
    g = _kv("nvfp4_format.txt")
    P, D, Hkv = 16, 128, 8
    per_token_head = (oracle.block_bytes("int8_per_token_head", P, D) - 2 * P * D) // (4 * P)
    assert per_token_head == 2                   # one K scale and one V scale
    assert 32768 * Hkv * per_token_head == g["scales_32k"]
    assert 131072 * Hkv * per_token_head == g["scales_128k"]
    # FP16 -> FP8 halves the bytes per token per layer: GQA 8 x 128 is 4 KB in FP16
    assert oracle.block_bytes("fp8_per_tensor", P, D) // P * Hkv == 4096 // 2


def _int4_words(codes_k, codes_e, codes_o):
    """INT4 storage words written out from the layout text: a K row word m holds
    channels 8m, 8m+2, 8m+4, 8m+6 in nibbles 0-3 and 8m+1, .., 8m+7 in nibbles
    4-7; a V pair-row word m holds channels 4m..4m+3 of the even token in
    nibbles 0-3 and of the odd token in nibbles 4-7."""
    D = codes_k.size
    kw = np.zeros(D // 8, np.uint32)
    for m in range(D // 8):
        for k in range(8):
            ch = 8 * m + (2 * k if k < 4 else 2 * (k - 4) + 1)
            kw[m] |= np.uint32(int(codes_k[ch]) << (4 * k))
    vw = np.zeros(D // 4, np.uint32)
    for m in range(D // 4):
        for k in range(8):
            src = codes_e if k < 4 else codes_o
            vw[m] |= np.uint32(int(src[4 * m + k % 4]) << (4 * k))
    return kw, vw


@pytest.mark.parametrize("mode", ["nvfp4", "nvfp4_4over6", "int4_per_token_head"])
def test_4bit_value_bytes_pair_tokens(mode):
    """The pool's 4-bit value payload pairs tokens: a V row of D bytes holds
    the codes of tokens 2k and 2k+1 (NVFP4: byte d holds channel d of token 2k
    in the low nibble and of 2k+1 in the high one; INT4: the word order of the
    layout text), each the code quant_row gives for that token alone; keys and
    scales stay per token; the bytes do not depend on the order the tokens are
    written in."""
    P, Hkv, D = 16, 1, 128
    rng = np.random.default_rng(5)
    k = rng.standard_normal((P, Hkv, D)).astype(np.float32)
    v = (rng.standard_normal((P, Hkv, D)) * 3).astype(np.float32)
    ks = oracle.tensor_scale(mode, oracle.amax(k))
    vs = oracle.tensor_scale(mode, oracle.amax(v))
    pool = np.zeros(oracle.pool_bytes(mode, 1, P, Hkv, D), np.uint8)
    assert oracle.write(mode, pool, 1, P, Hkv, D, k, v, np.arange(P, dtype=np.int32), ks, vs) == 0
    perm = rng.permutation(P)
    pool2 = np.zeros_like(pool)
    assert oracle.write(mode, pool2, 1, P, Hkv, D, k[perm], v[perm], perm.astype(np.int32), ks, vs) == 0
    assert np.array_equal(pool, pool2)
    blk = pool[256:]
    vpay, kbs = P * D // 2, P * D
    sw = 4 if mode == "int4_per_token_head" else D // 16     # scale bytes per token and side
    vbs = kbs + P * sw

    def codes_of(q):
        c = np.empty(D, np.uint8)
        c[0::2], c[1::2] = q & 15, q >> 4
        return c
    for t in range(P):
        qk, bk = oracle.quant_row(mode, k[t, 0], ks)
        qv, bv = oracle.quant_row(mode, v[t, 0], vs)
        assert np.array_equal(blk[kbs + t * sw:kbs + (t + 1) * sw], bk)             # K scale(s)
        assert np.array_equal(blk[vbs + t * sw:vbs + (t + 1) * sw], bv)             # V scale(s)
        pair = blk[vpay + (t // 2) * D:vpay + (t // 2 + 1) * D]
        if mode == "int4_per_token_head":
            qv2, _ = oracle.quant_row(mode, v[t ^ 1, 0], vs)                   # the pair's other token
            kw, vw = _int4_words(codes_of(qk), *((codes_of(qv), codes_of(qv2)) if t % 2 == 0
                                                 else (codes_of(qv2), codes_of(qv))))
            assert np.array_equal(blk[t * D // 2:(t + 1) * D // 2].view("<u4"), kw)        # K row t
            assert np.array_equal(pair.view("<u4"), vw)                                    # V pair row
        else:
            assert np.array_equal(blk[t * D // 2:(t + 1) * D // 2], qk)                 # K row t
            assert np.array_equal((pair >> (4 * (t & 1))) & 15, codes_of(qv))           # V nibbles of token t


def test_nvfp4_two_block_worked_example():
    """Two blocks, one in [-0.7, 0.7], one in [-5.5, 5.5], each get their own scale
    and both map their max to (about) 6 and use many grid points."""
    x = np.concatenate([np.linspace(-0.7, 0.7, 16), np.linspace(-5.5, 5.5, 16)]).astype(np.float32)
    st = oracle.nvfp4_tensor_scale(oracle.amax(x))
    q, bs = oracle.quant_row("nvfp4", x, st)
    codes = np.stack([q & 15, q >> 4], 1).reshape(-1)
    for blk in range(2):
        c = codes[16 * blk:16 * blk + 16]
        mags = c & 7
        assert mags.max() == 7                    # block max maps to 6
        assert len(set(mags.tolist())) >= 6       # the block uses the grid
        sb = oracle.e4m3_decode(bs[blk])
        den = np.float32(np.float32(st) * np.float32(sb))
        xh = np.array([oracle.e2m1_decode(int(cc)) for cc in c]) * float(den)
        err = np.abs(xh - x[16 * blk:16 * blk + 16])
        assert err.max() <= float(den) * 1.0 + max(0.0, np.abs(x[16 * blk:16 * blk + 16]).max() - 6 * float(den)) + 1e-6
    assert bs[0] != bs[1]


def test_nvfp4_error_bound_random():
    rng = np.random.default_rng(9)
    for _ in range(50):
        x = (rng.standard_normal(128) * rng.uniform(0.1, 20)).astype(np.float32)
        st = oracle.nvfp4_tensor_scale(oracle.amax(x) * rng.uniform(1.0, 3.0))
        q, bs = oracle.quant_row("nvfp4", x, st)
        codes = np.stack([q & 15, q >> 4], 1).reshape(-1)
        for b in range(8):
            sb = oracle.e4m3_decode(bs[b])
            den = float(np.float32(np.float32(st) * np.float32(sb)))
            seg = x[16 * b:16 * b + 16].astype(np.float64)
            xh = np.array([oracle.e2m1_decode(int(c)) for c in codes[16 * b:16 * b + 16]]) * den
            # half the widest E2M1 gap (4 -> 6) times the block denominator, plus clipping
            assert np.abs(xh - seg).max() <= den + max(0.0, np.abs(seg).max() - 6 * den) + 1e-7


# --------------------------------------------------------------------------- NVFP4 4over6
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_brute(y: float) -> int:
    """Nearest E2M1 code by search over the value set; a tie takes the even code."""
    a = min(abs(y), 6.0)
    d = np.abs(_E2M1_GRID - a)
    best = np.flatnonzero(d == d.min())
    mag = int(best[0] if len(best) == 1 or best[0] % 2 == 0 else best[1])
    return mag | (8 if math.copysign(1.0, y) < 0 else 0)


def _e4m3_torch(v: np.float32) -> int:
    """E4M3 code of a non-negative fp32 by torch's float8 cast (saturated at 448)."""
    v = min(float(v), 448.0)
    return int(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def _candidate(xb: np.ndarray, st: np.float32, c: float):
    """One 4over6 candidate of a 16-value block, computed apart from the oracle:
    torch's E4M3 cast for the block scale, a search over the E2M1 value set for
    the codes, and the fp64 squared error of the reconstruction."""
    amax = np.float32(np.abs(xb).max())
    sb = _e4m3_torch(np.float32(amax / np.float32(np.float32(c) * st)))
    sbf = np.float32(oracle.e4m3_decode(sb))
    den = np.float32(st * sbf)
    codes = [0] * 16 if sbf == 0 else [_e2m1_brute(float(np.float32(v / den))) for v in xb]
    xh = np.array([oracle.e2m1_decode(cc) for cc in codes]) * float(den)
    return sb, codes, float(np.sum((xh - xb.astype(np.float64)) ** 2)), den


def test_nvfp4_4over6_isolated_outlier_worked_example():
    """The page's case for 4over6: one outlier sets the block max and the other
    15 values lose precision under the max/6 scale.  Block: one 6.0 and fifteen
    2.5 with s_t = 2^-8, so s_b = 256 (max/6, divisor 1) or 384 (max/4, divisor
    1.5), both exact in E4M3.  max/6: 2.5 -> 2 (tie to even), squared error
    15 * 0.25 = 3.75.  max/4: 6 -> 4 (exact), 2.5 / 1.5 -> 1.5 (reconstructs
    2.25), squared error 15 * 0.0625 = 0.9375.  max/4 wins."""
    x = np.array([6.0] + [2.5] * 15, np.float32)
    st = 2.0 ** -8
    q, bs, ch = oracle.nvfp4_4over6_row(np.tile(x, 8), st)
    assert (ch == 4).all()
    assert oracle.e4m3_decode(bs[0]) == 384.0
    codes = np.stack([q & 15, q >> 4], 1).reshape(-1)[:16]
    assert codes[0] == 0b110 and (codes[1:] == 0b011).all()        # 4.0 and 1.5
    c6 = [0b111] + [0b100] * 15                                     # 6.0 and 2.0 (tie 2.5 -> 2)
    assert oracle.nvfp4_block_sse(x, np.array(c6, np.uint8), 1.0) == 3.75
    assert oracle.nvfp4_block_sse(x, codes.astype(np.uint8), 1.5) == 0.9375
    # the plain NVFP4 mode keeps the max/6 coding of the same block
    qn, bn = oracle.quant_row("nvfp4", np.tile(x, 8), st)
    assert oracle.e4m3_decode(bn[0]) == 256.0
    assert list(np.stack([qn & 15, qn >> 4], 1).reshape(-1)[:16]) == c6


def test_nvfp4_4over6_grid_blocks():
    """A block on the max/6 grid reconstructs exactly under max/6 and keeps it;
    a block on the max/4 grid reconstructs exactly only under max/4."""
    st = 2.0 ** -8                                                  # divisors 1 and 1.5 as above
    on6 = np.array([6, -4, 3, 2, 1.5, 1, 0.5, 0, -6, 4, -3, -2, -1.5, -1, -0.5, 0], np.float32)
    on4 = (np.array([4, -3, 2, 1.5, 1, 0.5, 0, -4, 3, -2, -1.5, -1, -0.5, 0, 4, 3], np.float32) * 1.5)
    for blk, want in ((on6, 6), (on4, 4)):
        q, bs, ch = oracle.nvfp4_4over6_row(np.tile(blk, 8), st)
        assert (ch == want).all()
        den = float(np.float32(st) * np.float32(oracle.e4m3_decode(bs[0])))
        codes = np.stack([q & 15, q >> 4], 1).reshape(-1)[:16]
        assert np.array_equal(np.array([oracle.e2m1_decode(c) for c in codes]) * den, blk.astype(np.float64))


def test_nvfp4_4over6_matches_brute_force():
    """Random blocks (normal, with and without an outlier): the oracle's block
    scale, codes and choice equal an independent computation of both
    candidates wherever their fp64 errors are not within rounding of a tie, and
    the chosen reconstruction is never worse than max/6 beyond rounding."""
    rng = np.random.default_rng(21)
    n4 = n6 = 0
    for trial in range(300):
        x = rng.standard_normal(128).astype(np.float32) * np.float32(rng.uniform(0.05, 30))
        if trial % 2:
            x[rng.integers(0, 128, 4)] *= np.float32(rng.uniform(3, 12))
        st = np.float32(oracle.nvfp4_tensor_scale(oracle.amax(x) * rng.uniform(1.0, 2.0)))
        q, bs, ch = oracle.nvfp4_4over6_row(x, float(st))
        codes = np.stack([q & 15, q >> 4], 1).reshape(-1)
        for b in range(8):
            xb = x[16 * b:16 * b + 16]
            sb6, c6, e6, _ = _candidate(xb, st, 6.0)
            sb4, c4, e4, _ = _candidate(xb, st, 4.0)
            got = list(codes[16 * b:16 * b + 16])
            if ch[b] == 6:
                assert (bs[b], got) == (sb6, c6)
                n6 += 1
            else:
                assert (bs[b], got) == (sb4, c4)
                n4 += 1
            if abs(e4 - e6) > 1e-5 * max(e4, e6):
                assert ch[b] == (4 if e4 < e6 else 6), (trial, b, e4, e6)
            chosen = e4 if ch[b] == 4 else e6
            assert chosen <= e6 * (1 + 1e-5) + 1e-30
    assert n4 > 100 and n6 > 100                                    # both choices exercised


# --------------------------------------------------------------------------- KVarN
def test_inv_sqrt128_is_correctly_rounded():
    getcontext().prec = 60
    exact = Decimal(1) / Decimal(128).sqrt()
    f = np.float32(float(exact))
    lo = np.nextafter(f, np.float32(0))
    hi = np.nextafter(f, np.float32(1))
    assert abs(Decimal(float(f)) - exact) <= abs(Decimal(float(lo)) - exact)
    assert abs(Decimal(float(f)) - exact) <= abs(Decimal(float(hi)) - exact)
    assert np.float32(oracle.inv_sqrt128()) == f


def test_fwht_matches_sylvester_matrix_and_is_orthogonal():
    from scipy.linalg import hadamard
    H = hadamard(128).astype(np.float64) / math.sqrt(128)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    assert np.allclose(oracle.hadamard_f64(x), H @ x, atol=1e-12)
    assert np.allclose(oracle.hadamard_f64(oracle.hadamard_f64(x)), x, atol=1e-12)
    xf = x.astype(np.float32)
    yf = oracle.fwht128_f32(xf)
    assert np.allclose(yf, H @ xf.astype(np.float64), rtol=0, atol=2e-6 * np.abs(xf).max() * 4)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert abs(oracle.hadamard_f64(q) @ oracle.hadamard_f64(k) - q @ k) < 1e-12
    qf, kf = q.astype(np.float32), k.astype(np.float32)
    assert abs(float(oracle.fwht128_f32(qf).astype(np.float64) @ oracle.fwht128_f32(kf))
               - float(qf.astype(np.float64) @ kf)) < 1e-4


def test_sum128_tree_order():
    v = np.arange(128, dtype=np.float32)
    assert oracle.sum128(v) == 127 * 128 / 2
    v = np.zeros(128, np.float32)
    v[0], v[64], v[32] = 2.0 ** 24, 1.0, 1.0
    # pairwise tree: (2^24 + 1) rounds to 2^24 twice; a running sum would give 2^24 + 2
    assert oracle.sum128(v) == 2.0 ** 24


def test_normalization_invariants():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((128, 128)).astype(np.float32)
    X[:, [3, 77]] *= 15
    Y, r, c = oracle.kvarn_normalize(X, 8)
    assert (r > 0).all() and (c > 0).all()
    col_std = Y.astype(np.float64).std(axis=0)
    assert np.allclose(col_std, 1.0, atol=1e-5)     # last step is per channel
    recon = r[:, None].astype(np.float64) * c[None, :] * Y
    assert np.allclose(recon, X, rtol=1e-5, atol=1e-5)
    Y7, r7, c7 = oracle.kvarn_normalize(X, 7)
    assert np.allclose(Y7.astype(np.float64).std(axis=1), 1.0, atol=1e-5)   # last step per token
    Y1, r1, c1 = oracle.kvarn_normalize(X, 1)
    assert np.all(c1 == 1.0)
    assert np.allclose(r1, X.astype(np.float64).std(axis=1), rtol=1e-5)      # first step is per token
    # a constant token (std 0) is left as is
    Z = X.copy()
    Z[5] = 0.25
    Yz, rz, cz = oracle.kvarn_normalize(Z, 1)
    assert rz[5] == 1.0 and np.all(Yz[5] == 0.25)


@pytest.mark.parametrize("is_value", [False, True])
def test_kvarn_tile_rtn(is_value):
    from scipy.linalg import hadamard
    rng = np.random.default_rng(4 + is_value)
    X = rng.standard_normal((128, 128)).astype(np.float32)
    X[:, [1, 50, 90, 127]] *= 15
    codes, scale, zero, r, c = oracle.kvarn_tile(X, is_value)
    steps = 3 if is_value else 15
    assert codes.max() <= steps
    # rebuild the normalised tile from its definition and check each code
    Yrot = np.stack([oracle.fwht128_f32(row) for row in X])
    Y, r2, c2 = oracle.kvarn_normalize(Yrot, 8)
    assert np.array_equal(r, r2) and np.array_equal(c, c2)
    axis = 1 if is_value else 0      # V: per token over channels; K: per channel over tokens
    assert np.array_equal(zero, Y.min(axis=axis))
    amin = Y.argmin(axis=axis)
    amax = Y.argmax(axis=axis)
    idx = np.arange(128)
    if is_value:
        assert (codes[idx, amin] == 0).all() and (codes[idx, amax] == steps).all()
        sc = scale[:, None]; z = zero[:, None]
    else:
        assert (codes[amin, idx] == 0).all() and (codes[amax, idx] == steps).all()
        sc = scale[None, :]; z = zero[None, :]
    yhat = sc.astype(np.float64) * codes + z
    assert np.all(np.abs(yhat - Y) <= sc / 2 * (1 + 1e-5) + 1e-6)
    # back to the original domain: x^ = H (r c y^) is close to x
    H = hadamard(128).astype(np.float64) / math.sqrt(128)
    xhat = (r[:, None].astype(np.float64) * c[None, :] * yhat) @ H
    rel = np.linalg.norm(xhat - X) / np.linalg.norm(X)
    assert rel < (0.15 if not is_value else 0.5)


@pytest.mark.parametrize("side", [0, 1])
def test_kvarn_pool_round_trip(side):
    """The KVarN page layout and the oracle's dequantization of it.  Tiles are
    written through the pool writer and every stored row is read back:
    (1) each element equals r_t c_d (scale q + zero) built from the tile
    quantizer's own outputs, with the key scale and zero per channel and the
    value scale and zero per token ("KVarN…", 技术原理: keys per channel, values
    per token), so a swap of the metadata fields, of their axes, or of the K
    and V metadata fails; (2) against the input rotated by scipy's Hadamard
    matrix (not the oracle's transform), every element stays within the RTN
    bound r_t c_d scale / 2 (plus fp32 rounding of the rotation and of the
    normalisation)."""
    from scipy.linalg import hadamard
    rng = np.random.default_rng(31 + side)
    Hkv, P, D, num_pages, page = 2, 128, 128, 3, 2
    k = rng.standard_normal((P, Hkv, D)).astype(np.float32)
    v = (rng.standard_normal((P, Hkv, D)) * 0.5 + 0.2).astype(np.float32)
    k[:, :, [5, 64]] *= 15
    v[:, 1, [7, 100]] *= 15
    pool = np.zeros(oracle.pool_bytes("kvarn_k4v2_g128", num_pages, P, Hkv, D), np.uint8)
    slots = (page * P + np.arange(P)).astype(np.int32)
    assert oracle.write("kvarn_k4v2_g128", pool, num_pages, P, Hkv, D, k, v, slots) == 0
    H = hadamard(128).astype(np.float64) / math.sqrt(128)
    steps = 3 if side else 15
    for h in range(Hkv):
        X = (v if side else k)[:, h]
        codes, scale, zero, r, c = oracle.kvarn_tile(X, bool(side))
        got = np.stack([oracle.dequant_row("kvarn_k4v2_g128", pool, num_pages, P, Hkv, D, 1.0, 1.0,
                                           page * P + t, h, side) for t in range(P)])
        sc = scale[:, None] if side else scale[None, :]
        z = zero[:, None] if side else zero[None, :]
        rc = r[:, None].astype(np.float64) * c[None, :]
        want = rc * (sc.astype(np.float64) * codes + z)
        assert np.array_equal(got, want)
        assert codes.max() == steps and codes.min() == 0
        Yrot = X.astype(np.float64) @ H                 # the rotated tile, fp64
        bound = rc * sc / 2 * (1 + 1e-5) + 2e-5 * np.abs(Yrot) + 1e-6
        assert np.all(np.abs(got - Yrot) <= bound)
    # the other side's metadata was written too, and differs (K and V use their own)
    other = np.stack([oracle.dequant_row("kvarn_k4v2_g128", pool, num_pages, P, Hkv, D, 1.0, 1.0,
                                         page * P + t, 0, 1 - side) for t in range(P)])
    Xo = (k if side else v)[:, 0].astype(np.float64) @ H
    assert np.abs(other - Xo).max() < 0.5 * np.abs(Xo).max()


@pytest.mark.parametrize("side", [0, 1])
def test_kvarn_constant_tile_round_trips_exactly(side):
    """A tile of one constant: the rotation leaves one non-zero channel, every
    std step meets zero spread on one axis, and the asymmetric RTN codes it
    with no error, so rotating the stored tile back gives the constant."""
    from scipy.linalg import hadamard
    Hkv, P, D = 1, 128, 128
    x = np.full((P, Hkv, D), 0.8125, np.float32)
    pool = np.zeros(oracle.pool_bytes("kvarn_k4v2_g128", 1, P, Hkv, D), np.uint8)
    assert oracle.write("kvarn_k4v2_g128", pool, 1, P, Hkv, D, x, x, np.arange(P, dtype=np.int32)) == 0
    H = hadamard(128).astype(np.float64) / math.sqrt(128)
    got = np.stack([oracle.dequant_row("kvarn_k4v2_g128", pool, 1, P, Hkv, D, 1.0, 1.0, t, 0, side)
                    for t in range(P)]) @ H
    assert np.allclose(got, 0.8125, rtol=0, atol=1e-6)


def test_nvfp4_tensor_scale_maps_the_tensor_max_to_the_top_of_both_grids():
    """The NVFP4 global scale s_t = amax / (448 * 6) ("NVFP4 KV Cache…",
    双层缩放 with the block max mapped to about 6, 用一组数直观看缩放的作用): the
    block holding the tensor's largest magnitude gets the largest finite E4M3
    block scale, 448 (byte 0x7E), its largest element gets E2M1 magnitude 6
    (code 7, sign kept), and no block scale exceeds 448.  A divisor of 448 or 6
    instead of 2688 fails all three."""
    rng = np.random.default_rng(17)
    for trial in range(300):
        D, rows = 128, 4
        x = (rng.standard_normal((rows, D)) * 10.0 ** rng.uniform(-4, 4)).astype(np.float32)
        x[rng.integers(rows), rng.integers(D)] *= rng.uniform(1, 30)
        st = oracle.nvfp4_tensor_scale(oracle.amax(x))
        i, j = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        for row in range(rows):
            q, bs = oracle.quant_row("nvfp4", x[row], st)
            assert (bs & 0x7F).max() <= 0x7E and not (bs & 0x80).any()
            if row == i:
                assert bs[j // 16] == 0x7E, (trial, hex(int(bs[j // 16])))
                code = (q[j // 2] >> (4 * (j & 1))) & 15
                assert code & 7 == 7 and (code >> 3) == (x[i, j] < 0)
                assert abs(oracle.e2m1_decode(int(code)) * 448.0 * st - x[i, j]) <= 1e-6 * abs(x[i, j])


# --------------------------------------------------------------------------- pool + attention
def _fill(mode, w, lay, k, v, slots, ks=1.0, vs=1.0):
    pool = np.zeros(oracle.pool_bytes(mode, lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim), np.uint8)
    bad = oracle.write(mode, pool, lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim, k, v, slots, ks, vs)
    assert bad == 0
    return pool


def _dequant_seq(mode, w, lay, pool, b, ks=1.0, vs=1.0):
    n = int(lay.seq_lens[b])
    K = np.zeros((w.num_kv_heads, n, w.head_dim))
    V = np.zeros_like(K)
    for t in range(n):
        slot = int(lay.block_table[b, t // w.page_size]) * w.page_size + t % w.page_size
        for h in range(w.num_kv_heads):
            K[h, t] = oracle.dequant_row(mode, pool, lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim, ks, vs, slot, h, 0)
            V[h, t] = oracle.dequant_row(mode, pool, lay.num_pages, w.page_size, w.num_kv_heads, w.head_dim, ks, vs, slot, h, 1)
    return K, V


MODES_SMALL = ["fp8_per_tensor", "int8_per_token_head", "fp8_per_token_head", "nvfp4", "int4_per_token_head",
               "nvfp4_4over6"]


@pytest.mark.parametrize("mode", MODES_SMALL + ["kvarn_k4v2_g128"])
def test_decode_matches_torch_sdpa(mode):
    from scipy.linalg import hadamard
    P = 128 if mode == "kvarn_k4v2_g128" else 16
    lens = [256, 128] if P == 128 else [37, 16, 1, 50]
    w = wl.Workload(name="t", mode=mode, num_seqs=len(lens), num_q_heads=8, num_kv_heads=2,
                    head_dim=128, page_size=P, io_dtype="f16", seed=42, seq_len_range=(1, 1))
    lay = wl.paged_layout(w, np.array(lens, np.int32), slack_pages=2)
    ks_, vs_, ss_ = [], [], []
    for b in range(len(lens)):
        k, v = wl.gen_kv_seq(w, b, lens[b])
        ks_.append(k); vs_.append(v); ss_.append(wl.slots_for_seq(w, lay, b))
    k, v, slots = np.concatenate(ks_), np.concatenate(vs_), np.concatenate(ss_)
    kscale = oracle.tensor_scale(mode, oracle.amax(k.astype(np.float32)))
    vscale = oracle.tensor_scale(mode, oracle.amax(v.astype(np.float32)))
    pool = _fill(mode, w, lay, k, v, slots, kscale, vscale)
    q = wl.gen_q(w).astype(np.float32)
    sm = 1 / math.sqrt(w.head_dim)
    out = oracle.decode(mode, pool, lay.num_pages, P, w.num_kv_heads, w.head_dim, q, lay.block_table,
                        lay.seq_lens, sm, kscale, vscale)
    H = hadamard(128).astype(np.float64) / math.sqrt(128)
    G = w.group
    for b in range(len(lens)):
        K, V = _dequant_seq(mode, w, lay, pool, b, kscale, vscale)
        if mode == "kvarn_k4v2_g128":          # stored in the rotated domain: rotate back
            K, V = K @ H, V @ H
        for hq in range(w.num_q_heads):
            qq = torch.from_numpy(q[b, hq].astype(np.float64))[None, None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq, torch.from_numpy(K[hq // G])[None, None], torch.from_numpy(V[hq // G])[None, None],
                scale=sm)[0, 0, 0].numpy()
            assert np.allclose(out[b, hq], ref, rtol=1e-9, atol=1e-9), (b, hq)
        # dequantised values stay close to the inputs (sanity of the round trip)
        if mode != "kvarn_k4v2_g128":
            x = k[wl.paged_layout(w, np.array(lens)).token_offset[b]:][:lens[b]].astype(np.float64)
            assert np.abs(K.transpose(1, 0, 2) - x).max() <= 0.5 * np.abs(x).max()


def test_kvarn_tail_decode_matches_torch_sdpa():
    """KVarN with open tiles: sequences of 0, 1, 100, 128, 200 and 383 tokens,
    whole tiles quantized, the rest raw in the tail.  Against torch SDPA in fp64
    over [scipy-Hadamard-rotated dequantized tiles; raw tail rows], and equal to
    the whole-tile decode when no tail row is used."""
    from scipy.linalg import hadamard
    lens = np.array([0, 1, 100, 128, 200, 383], np.int32)
    mode, P, D, Hkv, Hq = "kvarn_k4v2_g128", 128, 128, 2, 8
    full = (lens // P) * P
    w = wl.Workload(name="t", mode=mode, num_seqs=len(lens), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                    page_size=P, io_dtype="f32", seed=77, seq_len_range=(1, 1))
    lay = wl.paged_layout(w, np.maximum(lens, 1).astype(np.int32), slack_pages=1)
    tail_k = np.zeros((len(lens), P, Hkv, D), np.float32)
    tail_v = np.zeros_like(tail_k)
    pool = np.zeros(oracle.pool_bytes(mode, lay.num_pages, P, Hkv, D), np.uint8)
    seqs = []
    for b, n in enumerate(lens):
        k, v = wl.gen_kv_seq(w, b, int(n))
        seqs.append((k.astype(np.float64), v.astype(np.float64)))
        nf = int(full[b])
        if nf:
            slots = wl.slots_for_seq(w, lay, b)[:nf]
            assert oracle.write(mode, pool, lay.num_pages, P, Hkv, D, k[:nf], v[:nf], slots) == 0
        tail_k[b, :n - nf], tail_v[b, :n - nf] = k[nf:], v[nf:]
    q = wl.gen_q(w).astype(np.float32)
    sm = 1 / math.sqrt(D)
    out = oracle.decode_kvarn_tail(pool, lay.num_pages, Hkv, q, lay.block_table, lens, sm, tail_k, tail_v)
    H = hadamard(D).astype(np.float64) / math.sqrt(D)
    for b, n in enumerate(lens):
        if n == 0:
            assert (out[b] == 0).all()
            continue
        nf = int(full[b])
        K = np.zeros((Hkv, n, D))
        V = np.zeros_like(K)
        for t in range(n):
            for h in range(Hkv):
                if t < nf:
                    slot = int(lay.block_table[b, t // P]) * P + t % P
                    K[h, t] = oracle.dequant_row(mode, pool, lay.num_pages, P, Hkv, D, 1.0, 1.0, slot, h, 0) @ H
                    V[h, t] = oracle.dequant_row(mode, pool, lay.num_pages, P, Hkv, D, 1.0, 1.0, slot, h, 1) @ H
                else:
                    K[h, t], V[h, t] = seqs[b][0][t, h], seqs[b][1][t, h]
        for hq in range(Hq):
            qq = torch.from_numpy(q[b, hq].astype(np.float64))[None, None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq, torch.from_numpy(K[hq // (Hq // Hkv)])[None, None],
                torch.from_numpy(V[hq // (Hq // Hkv)])[None, None], scale=sm)[0, 0, 0].numpy()
            assert np.allclose(out[b, hq], ref, rtol=1e-9, atol=1e-9), (b, hq)
    whole = np.array([l for l in lens if l % P == 0 and l > 0])
    rows = [b * Hq + h for b in range(len(lens)) if lens[b] % P == 0 and lens[b] > 0 for h in range(Hq)]
    ref_whole = oracle.decode(mode, pool, lay.num_pages, P, Hkv, D, q, lay.block_table, lens, sm, rows=rows)
    assert whole.size and np.allclose(out.reshape(-1, D)[rows], ref_whole.reshape(-1, D)[rows], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["int8_per_token_head", "nvfp4"])
def test_decode_multi_matches_masked_sdpa(mode):
    """Several queries per sequence: torch SDPA in fp64 with an explicit causal
    mask (query i of nq stands at position n - nq + i) over the dequantized
    K/V; nq = 1 is the plain decode; a query before the first token gets 0."""
    lens = [37, 16, 3, 50]
    nq = 4
    w = wl.Workload(name="t", mode=mode, num_seqs=len(lens), num_q_heads=8, num_kv_heads=2,
                    head_dim=128, page_size=16, io_dtype="f16", seed=43, seq_len_range=(1, 1))
    lay = wl.paged_layout(w, np.array(lens, np.int32), slack_pages=1)
    ks_, vs_, ss_ = [], [], []
    for b in range(len(lens)):
        k, v = wl.gen_kv_seq(w, b, lens[b])
        ks_.append(k); vs_.append(v); ss_.append(wl.slots_for_seq(w, lay, b))
    k, v, slots = np.concatenate(ks_), np.concatenate(vs_), np.concatenate(ss_)
    kscale = oracle.tensor_scale(mode, oracle.amax(k.astype(np.float32)))
    vscale = oracle.tensor_scale(mode, oracle.amax(v.astype(np.float32)))
    pool = _fill(mode, w, lay, k, v, slots, kscale, vscale)
    rng = np.random.default_rng(8)
    q = rng.standard_normal((len(lens), nq, 8, 128)).astype(np.float32)
    sm = 1 / math.sqrt(128)
    out = oracle.decode_multi(mode, pool, lay.num_pages, 16, 2, 128, q, lay.block_table, lay.seq_lens, sm,
                              kscale, vscale)
    for b, n in enumerate(lens):
        K, V = _dequant_seq(mode, w, lay, pool, b, kscale, vscale)
        pos = n - nq + np.arange(nq)                                    # query positions
        allowed = np.arange(n)[None, :] <= pos[:, None]                 # causal mask [nq][n]
        for hq in range(8):
            qq = torch.from_numpy(q[b, :, hq].astype(np.float64))[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq, torch.from_numpy(K[hq // 4])[None, None], torch.from_numpy(V[hq // 4])[None, None],
                attn_mask=torch.from_numpy(allowed)[None, None], scale=sm)[0, 0].numpy()
            for i in range(nq):
                if pos[i] < 0:
                    assert (out[b, i, hq] == 0).all()
                else:
                    assert np.allclose(out[b, i, hq], ref[i], rtol=1e-9, atol=1e-9), (b, i, hq)
    one = oracle.decode_multi(mode, pool, lay.num_pages, 16, 2, 128, q[:, -1:], lay.block_table, lay.seq_lens, sm,
                              kscale, vscale)
    plain = oracle.decode(mode, pool, lay.num_pages, 16, 2, 128, q[:, -1], lay.block_table, lay.seq_lens, sm,
                          kscale, vscale)
    assert np.array_equal(one[:, 0], plain)


def test_decode_special_cases():
    w = wl.Workload(name="t", mode="int8_per_token_head", num_seqs=3, num_q_heads=4, num_kv_heads=2,
                    head_dim=32, page_size=16, io_dtype="f32", seed=5, seq_len_range=(1, 1))
    lens = np.array([20, 1, 0], np.int32)
    lay = wl.paged_layout(w, lens, slack_pages=1)
    n = int(lens.sum())
    rng = np.random.default_rng(0)
    k = np.tile(rng.standard_normal((1, 2, 32)).astype(np.float32), (n, 1, 1))  # all keys equal
    v = rng.standard_normal((n, 2, 32)).astype(np.float32)
    slots = wl.slot_mapping(w, lay)
    pool = _fill("int8_per_token_head", w, lay, k, v, slots)
    q = rng.standard_normal((3, 4, 32)).astype(np.float32)
    out = oracle.decode("int8_per_token_head", pool, lay.num_pages, 16, 2, 32, q, lay.block_table,
                        lay.seq_lens, 1 / math.sqrt(32))
    K, V = _dequant_seq("int8_per_token_head", w, lay, pool, 0)
    for hq in range(4):
        assert np.allclose(out[0, hq], V[hq // 2].mean(0), atol=1e-12)    # uniform attention
    K1, V1 = _dequant_seq("int8_per_token_head", w, lay, pool, 1)
    for hq in range(4):
        assert np.allclose(out[1, hq], V1[hq // 2, 0], atol=1e-12)        # one token: o = v
    assert (out[2] == 0).all()                                            # empty sequence
    # a page id out of range drops that page's tokens only
    bt = lay.block_table.copy()
    bt[0, 1] = 10 ** 6
    out2 = oracle.decode("int8_per_token_head", pool, lay.num_pages, 16, 2, 32, q, bt, lay.seq_lens,
                         1 / math.sqrt(32))
    assert np.allclose(out2[0, 0], V[0, :16].mean(0), atol=1e-12)


def test_write_skips_negative_and_counts_out_of_range_slots():
    pool = np.zeros(oracle.pool_bytes("int8_per_token_head", 2, 16, 1, 32), np.uint8)
    k = np.ones((3, 1, 32), np.float32)
    bad = oracle.write("int8_per_token_head", pool, 2, 16, 1, 32, k, k, np.array([-1, 40, 5], np.int32))
    assert bad == 1
    blk = oracle.block_bytes("int8_per_token_head", 16, 32)
    body = pool[oracle.header_bytes():].reshape(2, blk)
    assert (body[0, 5 * 32:6 * 32].view(np.int8) == 127).all()
    assert body[1].sum() == 0 and body[0, :5 * 32].sum() == 0


def test_kvarn_write_requires_whole_tiles():
    pool = np.zeros(oracle.pool_bytes("kvarn_k4v2_g128", 2, 128, 1, 128), np.uint8)
    x = np.random.default_rng(0).standard_normal((128, 1, 128)).astype(np.float32)
    good = np.arange(128, 256, dtype=np.int32)
    assert oracle.write("kvarn_k4v2_g128", pool, 2, 128, 1, 128, x, x, good) == 0
    shifted = np.arange(1, 129, dtype=np.int32)
    assert oracle.write("kvarn_k4v2_g128", pool, 2, 128, 1, 128, x, x, shifted) == 128
    with pytest.raises(ValueError):
        oracle.write("kvarn_k4v2_g128", pool, 2, 128, 1, 128, x[:64], x[:64], good[:64])
