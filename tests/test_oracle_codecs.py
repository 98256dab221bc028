"""Pins for the oracle's codecs (CPU only).

Each codec is tied to something other than itself: PyTorch's own float8_e4m3fn
and bfloat16 conversions (library routines), brute-force nearest-value search,
exhaustive code tables and the byte counts the pages print.
"""

import numpy as np
import pytest
import torch

from oracle import codecs


def _torch_e4m3_bits(x):
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = codecs.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert ours[0x38] == 1.0 and ours[0xB8] == -1.0


def test_e4m3_encode_matches_torch_rne():
    # every representable value, every midpoint between neighbours (ties), and random points
    pos = codecs.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    rs = np.random.default_rng(7)
    rnd = rs.uniform(-447.9, 447.9, 200000)
    tiny = rs.uniform(-2.0 ** -5, 2.0 ** -5, 50000)
    x = np.concatenate([pos, -pos, mids, -mids, rnd, tiny, [0.0, -0.0]]).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    assert np.array_equal(codecs.e4m3_encode(x), _torch_e4m3_bits(x))


def test_e4m3_encode_saturates():
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e6, -500.0, 3e38], np.float32)
    out = codecs.e4m3_encode(x)
    assert list(out) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E]


def test_e2m1_tables_and_brute_force():
    vals = codecs.e2m1_decode(np.arange(16))
    assert list(vals[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(vals[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    rs = np.random.default_rng(3)
    x = np.concatenate([rs.uniform(0, 7, 20000), np.arange(0, 7.01, 0.125)])
    enc = codecs.e2m1_encode(x.astype(np.float32)) & 7
    for xi, ci in zip(x, enc):
        if xi >= 6:
            assert ci == 7
            continue
        d = np.abs(grid - xi)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert ci == want, (xi, ci, want)
    # e2m1 midpoints: each rounds to the even neighbour
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    assert list(codecs.e2m1_decode(codecs.e2m1_encode(ties))) == [0, 1, 1, 2, 2, 4, 4]


def test_e8m0_exponent_brute_force():
    rs = np.random.default_rng(11)
    a = np.concatenate([rs.uniform(0, 1, 3000) * np.exp2(rs.integers(-140, 120, 3000)),
                        448.0 * np.exp2(np.arange(-130, 120, dtype=np.float64)),
                        np.nextafter(448.0, 1e9) * np.exp2(np.arange(-120, 110, dtype=np.float64)),
                        [0.0, 1e-45, 3e38]]).astype(np.float32)
    got = codecs.e8m0_exponent(a)
    for ai, gi in zip(a.astype(np.float64), got):
        if ai == 0:
            assert gi == 0
            continue
        want = next(e for e in range(-127, 128) if ai <= 448.0 * 2.0 ** e) \
            if ai > 448.0 * 2.0 ** -127 else -127
        assert gi == want, (ai, gi, want)


def test_bf16_matches_torch():
    rs = np.random.default_rng(5)
    x = np.concatenate([rs.standard_normal(100000) * np.exp2(rs.integers(-60, 60, 100000)),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codecs.bf16_encode(x), ref)
    assert np.array_equal(codecs.bf16_decode(ref), torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_fp8_rows_roundtrip_and_scale_choice():
    rs = np.random.default_rng(1)
    x = (rs.standard_normal((300, 512)) * np.exp2(rs.integers(-20, 20, (300, 1)))).astype(np.float32)
    x[0] = 0.0
    x[1, :32] = 0.0
    b = codecs.encode_rows(x, codecs.FMT_FP8)
    assert b.shape == (300, 528)
    dec = codecs.decode_rows(b, codecs.FMT_FP8, 512)
    scale = codecs.e8m0_decode(b[:, 512:]).repeat(32, axis=1)
    # RNE to 3 mantissa bits: |err| <= 2^-4 |x| for normals, <= 2^-10 * scale below 2^-6 * scale
    err = np.abs(dec - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, scale * 2.0 ** -10) * (1 + 1e-12))
    # the scale is the smallest power of two that fits: block amax / scale in (224, 448]
    amax = np.abs(x.reshape(300, 16, 32)).max(-1)
    ratio = amax / codecs.e8m0_decode(b[:, 512:])
    nz = amax > 0
    assert np.all((ratio[nz] > 224) & (ratio[nz] <= 448))
    assert np.all(b[:, 512:][~nz] == 127)


def test_fp4_rows_roundtrip():
    rs = np.random.default_rng(2)
    x = rs.standard_normal((200, 512)).astype(np.float32)
    x[0] = 0.0
    b = codecs.encode_rows(x, codecs.FMT_FP4)
    assert b.shape == (200, 288)
    dec = codecs.decode_rows(b, codecs.FMT_FP4, 512)
    s = codecs.e4m3_decode(b[:, 256:]).repeat(16, axis=1)
    # e2m1 spacing is at most 2 * s, so RNE error <= s; plus the saturation of a rounded scale
    amax = np.abs(x.reshape(200, 32, 16)).max(-1).repeat(16, axis=1)
    assert np.all(np.abs(dec - x) <= np.maximum(s, amax - 6 * s) + 1e-12)
    assert np.all(dec[0] == 0)
    # channel 2i is the low nibble
    one = np.zeros((1, 512), np.float32)
    one[0, 0] = 6.0
    one[0, 3] = -3.0
    p, sc = codecs.fp4_encode(one)
    assert p[0, 0] == 0x07 and p[0, 1] == 0xD0


def test_pagesplit_roundtrip():
    rs = np.random.default_rng(4)
    x = (rs.standard_normal((128, 128)) * np.exp2(rs.integers(-10, 10, (128, 1)))).astype(np.float32)
    x[3] = 0.0
    pages = codecs.encode_pagesplit(x)
    assert pages.shape == (2, 64 * 132)
    dec = codecs.decode_pagesplit(pages, 128)
    # same codes as the block-128 FP8 rule, the scale kept as an fp32 power of two
    c, e = codecs.fp8_encode(x, block=128)
    assert np.array_equal(dec, codecs.e4m3_decode(c) * codecs.e8m0_decode(e))
    sc = np.ascontiguousarray(pages[:, 64 * 128:]).view(np.float32).reshape(-1)
    assert np.array_equal(np.log2(sc), np.round(np.log2(sc)))
    amax = np.abs(x).max(-1)
    nz = amax > 0
    assert np.all((amax[nz] / sc[nz] > 224) & (amax[nz] / sc[nz] <= 448)) and sc[3] == 1.0


def test_byte_layouts(golden):
    g = golden["byte_layouts"]
    assert codecs.row_bytes(codecs.FMT_FP8, 512) == g["fp8_row"] == g["fp8_data"] + g["fp8_scales"]
    assert codecs.row_bytes(codecs.FMT_FP4, 512) == g["fp4_row"]
    assert codecs.row_bytes(codecs.FMT_BF16, 512) == 1024
    assert codecs.row_bytes(codecs.FMT_FP8_PAGESPLIT, 128) == 132


def test_v41_global_kv_decomposition(golden):
    # 890 B/token is not itemised on the pages; one consistent decomposition (derived):
    # (3 encoder copies merged 2:1 + 1 decoder copy) x (FP4 main row + FP4 128-d index key
    # with one e8m0 scale per 32)
    g = golden["v41_global_kv"]
    copies = g["encoder_copies"] / g["encoder_merge"] + g["decoder_copies"] / g["decoder_merge"]
    fp4_index_key = codecs.row_bytes(codecs.FMT_FP4H_PAGESPLIT, 128)   # 64 code bytes + 4 scale bytes
    assert copies * (codecs.row_bytes(codecs.FMT_FP4, 512) + fp4_index_key) == g["bytes_per_token"]


def test_fp4_scale_is_rne_e4m3_of_amax_over_six():
    """The FP4 block scale ("DeepSeek-V4.1-Flash" diagram: an E4M3 scale per 16
    channels) is read as RNE_e4m3(fp32(amax / 6)).  Pinned against PyTorch's own
    float8_e4m3fn cast of the same fp32 quotient: every e4m3 value, every midpoint
    between neighbours (ties go to the even code, so a rounding-up rule fails here)
    and random amax values."""
    vals = codecs.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    # values and midpoints times 6 are exact in fp32, and so are their quotients by 6
    exact = np.concatenate([vals, mids]) * 6.0
    assert np.all(exact.astype(np.float32).astype(np.float64) == exact)
    rs = np.random.default_rng(17)
    amax = np.concatenate([exact, rs.uniform(2.0 ** -9, 2640.0, 4000),
                           6.0 * np.exp2(rs.uniform(-9, 8.7, 4000))]).astype(np.float32)
    x = np.zeros((len(amax), 16), np.float32)
    x[:, 3] = amax
    x[:, 7] = -amax * np.float32(0.5)
    _, s_code = codecs.fp4_encode(x)
    want = _torch_e4m3_bits((amax / np.float32(6.0)).astype(np.float32))
    assert np.array_equal(s_code[:, 0], want)
    # the midpoints, alone: the even neighbour (an upward rounding would take the odd one)
    mid_amax = (mids * 6.0).astype(np.float32)
    xm = np.zeros((len(mids), 16), np.float32)
    xm[:, 0] = mid_amax
    _, mcode = codecs.fp4_encode(xm)
    assert np.all(mcode[:, 0] % 2 == 0)
