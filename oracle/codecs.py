"""Cache-row codecs (oracle side).  TEST INFRASTRUCTURE ONLY.

Formats fixed by the pages:

* FP8 latent, 528 bytes per 512-d token: 512 float8_e4m3 values over all 512
  dims (the 64 RoPE dims are quantised too), then 16 float8_e8m0 scales, one
  per 32 values.  ("DeepSeek-V4-Flash" model record, serviceability join,
  engine kernel constraint (2): the FlashMLA decode-kernel cache layout.)
* FP4 latent, 288 bytes per 512-d token: E2M1 values with one E4M3 scale per
  16 channels ("DeepSeek-V4.1-Flash - KV-Cache-Compressed Inference" diagram,
  "The four compression axes"; the same FlashMLA record gives 288 B/token).
* bf16 rows (the unquantised case of the tiny configuration).

Readings where the pages are silent:

* e8m0 scale: the smallest power of two 2^e with amax <= 448 * 2^e (rounded
  up, so no value saturates); byte = e + 127, e clamped to [-127, 127]; an
  all-zero block stores byte 127 (scale 1).
* value codes: round-to-nearest-even with saturation to the largest finite
  magnitude (448 for e4m3, 6 for e2m1); the sign bit of the input is kept,
  also when the magnitude rounds to zero; NaN codes are never produced.
* FP4 scale: s = RNE_e4m3(amax / 6) (fp32 division); a zero scale zeroes the
  whole block.  Channel 2i sits in the low nibble of byte i.
* FP8 index keys (128-d): 128 e4m3 codes and one scale for the whole key,
  stored as the fp32 value of its power of two - 132 bytes per key, the size
  of the V3.2 index key - with the same rounding rules (the block is the 128
  values); in a 64-row page all 64 data rows come first, then the 64 fp32
  scales ("page-split"), so the data rows form one dense 8 KiB tile.
* Query rows of the FP8 indexer are coded with the same rule, one scale per
  head (block 128).
* FP4 index keys ("DeepSeek-V4 deep dive", section 5.2: the indexer's keys and
  queries go through a Hadamard rotation and then FP4 rounding with block size
  32; "DeepSeek-V4.1 Flash", section 10.4: MXFP4, E2M1 values sharing a scale per
  1 x 32): the 128-d key is rotated by H / sqrt(128) (H the Sylvester Hadamard
  matrix), then coded as 128 e2m1 values with one e8m0 scale per 32 - 64 + 4 = 68
  bytes.  The scale follows the FP8 rule with 6 in place of 448: the smallest
  power of two 2^e with amax <= 6 * 2^e (nothing saturates).  Page-split like the
  FP8 keys: in a 64-row page the 64 rows of 64 code bytes come first, then the 64
  rows of 4 scale bytes.  The rotation's fp32 rendering (the order fixed so that
  the codes are reproducible bit for bit) is the fast Walsh-Hadamard butterfly
  with strides 1, 2, 4, ..., 64, each (a, b) -> (a + b, a - b) rounded to fp32,
  then one multiplication by fp32(1 / sqrt(128)).

Everything here is elementwise numpy on exactly representable values; fp32
steps are done in np.float32 (IEEE, round-to-nearest-even).
"""

import numpy as np

E4M3_MAX = 448.0
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


# ----------------------------------------------------------------------------
# scalar code <-> value
# ----------------------------------------------------------------------------

def e4m3_decode(codes):
    """float8_e4m3 (bias 7, no infinities, S.1111.111 = NaN) -> float64."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 7
    mag = np.where(exp == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.exp2(exp - 7.0))
    val = np.where(sign == 1, -mag, mag)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(y):
    """Round finite values to float8_e4m3 codes (RNE, saturating at +-448)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    sign = np.signbit(y).astype(np.int64)
    # subnormal binade and zero: multiples of 2^-9 below 2^-6
    sub_q = np.rint(np.minimum(a, 1.0) * 512.0).astype(np.int64)   # 0..8 (8 == 2^-6, carries into exp 1)
    # normal: a = f * 2^E with f in [1, 2)
    m, ex = np.frexp(np.where(a > 0, a, 1.0))            # a = m * 2^ex, m in [0.5, 1)
    E = ex - 1
    frac = np.where(a > 0, a / np.exp2(E.astype(np.float64)), 1.0)
    q = np.rint((frac - 1.0) * 8.0).astype(np.int64)     # 0..8
    carry = q == 8
    E = np.where(carry, E + 1, E)
    q = np.where(carry, 0, q)
    norm_code = ((E + 7) << 3) | q
    mag = np.where(a < 2.0 ** -6, sub_q, norm_code)
    mag = np.where(a >= E4M3_MAX, 0x7E, np.minimum(mag, 0x7E))
    return ((sign << 7) | mag).astype(np.uint8)


def e2m1_decode(codes):
    """float4_e2m1 nibble -> float64 (0, .5, 1, 1.5, 2, 3, 4, 6 with a sign bit)."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    mag = E2M1_VALUES[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e2m1_encode(y):
    """Round finite values to e2m1 nibbles (RNE on the e2m1 grid, saturating at 6)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    sign = np.signbit(y).astype(np.int64)
    # the grid has step 0.5 below 2, step 1 in [2, 4), step 2 in [4, 6]
    lo = np.rint(a * 2.0)                 # codes 0..4
    mid = np.rint(a) + 2.0                # 2 -> code 4, 3 -> 5, 4 -> 6
    hi = np.rint(a / 2.0) + 4.0           # 4 -> code 6, 6 -> 7
    mag = np.where(a < 2.0, lo, np.where(a < 4.0, mid, hi))
    mag = np.where(a >= 6.0, 7, np.minimum(mag, 7)).astype(np.int64)
    return ((sign << 3) | mag).astype(np.uint8)


def e8m0_exponent(amax):
    """Scale exponent e of a block: the smallest integer with amax <= 448 * 2^e.

    amax is a non-negative fp32 value.  Returns int64 e in [-127, 127]; amax == 0
    returns 0 (scale byte 127).
    """
    a = np.asarray(amax, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.int64)
    biased = bits >> 23
    mant = bits & 0x7FFFFF
    # a = 1.mant * 2^(biased-127); 448 = 1.75 * 2^8; 1.75 <-> mantissa field 0x600000
    e = np.where(mant <= 0x600000, biased - 127 - 8, biased - 127 - 7)
    e = np.where(biased == 0, -127, e)              # fp32 subnormal amax: clamp
    e = np.clip(e, -127, 127)
    return np.where(a == 0, 0, e).astype(np.int64)


def e8m0_decode(byte):
    """e8m0 scale byte -> 2^(byte-127) as float64 (255 would be NaN; never written)."""
    return np.exp2(np.asarray(byte).astype(np.float64) - 127.0)


def bf16_encode(x):
    """fp32 -> bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_decode(bits):
    """bf16 bit patterns -> float64."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# block-scaled row codecs
# ----------------------------------------------------------------------------

def _pow2_f32(e):
    """2^e as float32, exact for e in [-149, 127]."""
    return np.ldexp(np.float32(1.0), np.asarray(e, dtype=np.int64)).astype(np.float32)


def fp8_encode(x, block=32):
    """x [..., D] float32 -> (codes uint8 [..., D], scale bytes uint8 [..., D/block])."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    xb = x.reshape(x.shape[:-1] + (D // block, block))
    amax = np.max(np.abs(xb), axis=-1)
    e = e8m0_exponent(amax)
    y = (xb * _pow2_f32(-e)[..., None]).astype(np.float32)     # exact power-of-two scaling
    codes = e4m3_encode(y).reshape(x.shape)
    return codes, (e + 127).astype(np.uint8)


def fp8_decode(codes, scales, block=32):
    """Inverse of fp8_encode (exact) -> float64 [..., D]."""
    codes = np.asarray(codes)
    D = codes.shape[-1]
    v = e4m3_decode(codes).reshape(codes.shape[:-1] + (D // block, block))
    v = v * e8m0_decode(scales)[..., None]
    return v.reshape(codes.shape)


def fp4_encode(x, block=16):
    """x [..., D] float32 -> (packed uint8 [..., D/2], e4m3 scale codes uint8 [..., D/block])."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    xb = x.reshape(x.shape[:-1] + (D // block, block))
    amax = np.max(np.abs(xb), axis=-1)
    s_code = e4m3_encode((amax / np.float32(6.0)).astype(np.float32))
    s_val = e4m3_decode(s_code).astype(np.float32)
    safe = np.where(s_val > 0, s_val, np.float32(1.0)).astype(np.float32)
    y = (xb / safe[..., None]).astype(np.float32)
    nib = e2m1_encode(y).astype(np.uint8)
    nib = np.where((s_val > 0)[..., None], nib, 0).astype(np.uint8)
    nib = nib.reshape(x.shape)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    return packed, s_code


def fp4_decode(packed, scales, block=16):
    """Inverse of fp4_encode -> float64 [..., D]."""
    packed = np.asarray(packed)
    lo = e2m1_decode(packed & 0xF)
    hi = e2m1_decode(packed >> 4)
    v = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))
    D = v.shape[-1]
    v = v.reshape(v.shape[:-1] + (D // block, block)) * e4m3_decode(scales)[..., None]
    return v.reshape(v.shape[:-2] + (D,))


# ----------------------------------------------------------------------------
# whole cache rows (bytes) and pages
# ----------------------------------------------------------------------------

FMT_BF16 = 0
FMT_FP8 = 1            # e4m3 data then e8m0 per 32, inline per row
FMT_FP4 = 2            # packed e2m1 data then e4m3 per 16, inline per row
FMT_FP8_PAGESPLIT = 3  # index keys: e4m3 codes + one fp32 power-of-two scale per row, page-split
FMT_FP4H_PAGESPLIT = 4  # index keys: Hadamard-rotated, e2m1 codes + e8m0 per 32, page-split

PAGE_ROWS = 64


def row_bytes(fmt, dim):
    if fmt == FMT_BF16:
        return 2 * dim
    if fmt == FMT_FP8:
        return dim + dim // 32
    if fmt == FMT_FP8_PAGESPLIT:
        return dim + 4
    if fmt == FMT_FP4:
        return dim // 2 + dim // 16
    if fmt == FMT_FP4H_PAGESPLIT:
        return dim // 2 + dim // 32
    raise ValueError(fmt)


def encode_rows(x, fmt):
    """x [n, D] float32 -> bytes [n, row_bytes] for the inline formats."""
    x = np.asarray(x, dtype=np.float32)
    if fmt == FMT_BF16:
        return bf16_encode(x).view(np.uint8).reshape(x.shape[0], -1)
    if fmt == FMT_FP8:
        c, s = fp8_encode(x)
        return np.concatenate([c, s], axis=-1)
    if fmt == FMT_FP4:
        p, s = fp4_encode(x)
        return np.concatenate([p, s], axis=-1)
    raise ValueError(fmt)


def decode_rows(b, fmt, dim):
    """bytes [n, row_bytes] of an inline format -> float64 [n, dim]."""
    b = np.asarray(b, dtype=np.uint8)
    if fmt == FMT_BF16:
        return bf16_decode(np.ascontiguousarray(b).view(np.uint16))
    if fmt == FMT_FP8:
        return fp8_decode(b[:, :dim], b[:, dim:])
    if fmt == FMT_FP4:
        return fp4_decode(b[:, :dim // 2], b[:, dim // 2:])
    raise ValueError(fmt)


def encode_pagesplit(x):
    """Index keys x [64*p, D] float32 -> bytes [p, 64*(D + 4)]: per page 64 rows of e4m3
    codes (one power-of-two scale per row), then the 64 scales as fp32."""
    x = np.asarray(x, dtype=np.float32)
    n, D = x.shape
    assert n % PAGE_ROWS == 0
    c, e = fp8_encode(x, block=D)                       # e: scale bytes [n, 1]
    scale = _pow2_f32(e[:, 0].astype(np.int64) - 127)    # exact powers of two
    p = n // PAGE_ROWS
    return np.concatenate([c.reshape(p, -1), scale.view(np.uint8).reshape(p, -1)], axis=-1)


def decode_pagesplit(pages, dim):
    """bytes [p, 64*(D + 4)] -> float64 [64*p, D]."""
    pages = np.asarray(pages, dtype=np.uint8)
    p = pages.shape[0]
    c = pages[:, :PAGE_ROWS * dim].reshape(p * PAGE_ROWS, dim)
    sc = np.ascontiguousarray(pages[:, PAGE_ROWS * dim:PAGE_ROWS * (dim + 4)]).view(np.float32).reshape(-1)
    return e4m3_decode(c) * sc.astype(np.float64)[:, None]


def encode_q_perhead(q):
    """Indexer queries [..., H, 128] float32 -> (codes [..., H, 128], e8m0 bytes [..., H]).

    One scale per head (block 128); same rounding rules as the cache codes.
    """
    c, s = fp8_encode(q, block=q.shape[-1])
    return c, s[..., 0]


# ----------------------------------------------------------------------------
# FP4 index keys: Hadamard rotation, e2m1 + e8m0 per 32
# ----------------------------------------------------------------------------

def hadamard_matrix(n):
    """Sylvester Hadamard matrix: H[i, j] = (-1)^popcount(i & j), n a power of two."""
    i = np.arange(n)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pop = np.zeros_like(bits)
    while np.any(bits):
        pop += bits & 1
        bits >>= 1
    return np.where(pop % 2 == 0, 1.0, -1.0)


def hadamard_fp64(x):
    """The rotation by definition: y = H x / sqrt(n) along the last axis (fp64)."""
    x = np.asarray(x, np.float64)
    n = x.shape[-1]
    return x @ hadamard_matrix(n).T / np.sqrt(n)


def hadamard_contract(x):
    """fp32 rendering of the rotation in the fixed order: butterflies of stride 1, 2,
    ..., n/2 on the pairs (i, i + h) with i & h == 0, each (a, b) -> (a + b, a - b)
    rounded to fp32, then a multiplication by fp32(1 / sqrt(n))."""
    y = np.array(x, dtype=np.float32, copy=True)
    n = y.shape[-1]
    h = 1
    while h < n:
        idx = np.arange(n)
        lo = idx[(idx & h) == 0]
        a = y[..., lo].copy()
        b = y[..., lo + h].copy()
        y[..., lo] = (a + b).astype(np.float32)
        y[..., lo + h] = (a - b).astype(np.float32)
        h *= 2
    return (y * np.float32(1.0 / np.sqrt(float(n)))).astype(np.float32)


def e8m0_exponent_fp4(amax):
    """Scale exponent of an FP4 block: the smallest integer e with amax <= 6 * 2^e.

    amax is a non-negative fp32 value; 6 = 1.5 * 2^2.  Returns int64 e in
    [-127, 127]; amax == 0 returns 0 (scale byte 127).
    """
    a = np.asarray(amax, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.int64)
    biased = bits >> 23
    mant = bits & 0x7FFFFF
    e = np.where(mant <= 0x400000, biased - 127 - 2, biased - 127 - 1)
    e = np.where(biased == 0, -127, e)              # fp32 subnormal amax: clamp
    e = np.clip(e, -127, 127)
    return np.where(a == 0, 0, e).astype(np.int64)


def fp4b32_encode(x, block=32):
    """x [..., D] float32 -> (packed e2m1 uint8 [..., D/2], e8m0 scale bytes uint8 [..., D/block]).

    Channel 2i sits in the low nibble of byte i."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    xb = x.reshape(x.shape[:-1] + (D // block, block))
    e = e8m0_exponent_fp4(np.max(np.abs(xb), axis=-1))
    y = (xb * _pow2_f32(-e)[..., None]).astype(np.float32)     # exact power-of-two scaling
    nib = e2m1_encode(y).astype(np.uint8).reshape(x.shape)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


def fp4b32_decode(packed, scales, block=32):
    """Inverse of fp4b32_encode (exact) -> float64 [..., D]."""
    packed = np.asarray(packed)
    lo = e2m1_decode(packed & 0xF)
    hi = e2m1_decode(packed >> 4)
    v = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))
    D = v.shape[-1]
    v = v.reshape(v.shape[:-1] + (D // block, block)) * e8m0_decode(scales)[..., None]
    return v.reshape(v.shape[:-2] + (D,))


def encode_fp4h_pagesplit(x):
    """Index keys x [64*p, 128] float32 (not yet rotated) -> bytes [p, 64*68]: per page
    64 rows of 64 code bytes, then 64 rows of 4 scale bytes."""
    x = np.asarray(x, dtype=np.float32)
    n, D = x.shape
    assert n % PAGE_ROWS == 0
    c, s = fp4b32_encode(hadamard_contract(x))
    p = n // PAGE_ROWS
    return np.concatenate([c.reshape(p, -1), s.reshape(p, -1)], axis=-1)


def decode_fp4h_pagesplit(pages, dim):
    """bytes [p, 64*(D/2 + D/32)] -> the rotated key values, float64 [64*p, D]."""
    pages = np.asarray(pages, dtype=np.uint8)
    p = pages.shape[0]
    cb = dim // 2
    c = pages[:, :PAGE_ROWS * cb].reshape(p * PAGE_ROWS, cb)
    s = pages[:, PAGE_ROWS * cb:PAGE_ROWS * (cb + dim // 32)].reshape(p * PAGE_ROWS, dim // 32)
    return fp4b32_decode(c, s)


def encode_q_fp4h(q):
    """Indexer queries [..., H, 128] float32 -> (packed codes [..., H, 64], e8m0 bytes [..., H, 4]):
    rotated like the keys, then coded with one scale per 32."""
    return fp4b32_encode(hadamard_contract(q))
