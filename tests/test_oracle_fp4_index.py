"""Pins for the oracle's FP4 index keys (CPU only): the Hadamard rotation, the e2m1 +
e8m0-per-32 codec, the 68-byte page-split layout and the BF16-score selection
("DeepSeek-V4 deep dive", section 5.2; "DeepSeek-V4.1 Flash", section 10.4).

Each is tied to something other than itself: SciPy's Hadamard matrix (a library
routine), orthogonality and dot-product invariance, exact integer butterflies, the
scale rule's boundary cases, brute-force nearest-value search and full sorts.
"""

import numpy as np
import pytest

from oracle import codecs, indexer

scipy_linalg = pytest.importorskip("scipy.linalg")


def test_hadamard_matrix_is_sylvester():
    for n in (2, 8, 32, 128):
        assert np.array_equal(codecs.hadamard_matrix(n), scipy_linalg.hadamard(n).astype(np.float64))


def test_hadamard_rotation_orthogonal_and_dot_products_unchanged():
    H = codecs.hadamard_matrix(128)
    assert np.array_equal(H @ H.T, 128.0 * np.eye(128))
    rs = np.random.default_rng(3)
    x = rs.standard_normal((64, 128))
    y = rs.standard_normal((64, 128))
    hx, hy = codecs.hadamard_fp64(x), codecs.hadamard_fp64(y)
    np.testing.assert_allclose(np.sum(hx * hy, axis=1), np.sum(x * y, axis=1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(hx, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # an involution up to the scale: rotating twice gives the input back
    np.testing.assert_allclose(codecs.hadamard_fp64(hx), x, rtol=1e-12, atol=1e-12)


def test_hadamard_contract_against_the_definition():
    rs = np.random.default_rng(4)
    x = rs.standard_normal((256, 128)).astype(np.float32)
    got = codecs.hadamard_contract(x).astype(np.float64)
    ref = codecs.hadamard_fp64(x.astype(np.float64))
    # 7 rounded butterfly stages and one rounded product: a few ulps of the l1 mass
    bound = 16 * 2.0 ** -24 * np.sum(np.abs(x), axis=1, keepdims=True) / np.sqrt(128)
    assert np.all(np.abs(got - ref) <= bound)
    # integer inputs: the butterflies are exact, so only the final product rounds
    xi = rs.integers(-1000, 1001, (64, 128)).astype(np.float32)
    yint = xi.astype(np.float64) @ codecs.hadamard_matrix(128).T          # exact integers
    c32 = float(np.float32(1.0 / np.sqrt(128.0)))
    assert np.array_equal(codecs.hadamard_contract(xi), (yint * c32).astype(np.float32))


def test_fp4b32_scale_rule_boundaries():
    for e in (-20, -3, 0, 1, 7, 40):
        s = 2.0 ** e
        x = np.zeros((1, 32), np.float32)
        x[0, 5] = 6 * s                      # exactly 6 * 2^e: scale e, code 7
        c, b = codecs.fp4b32_encode(x)
        assert b[0, 0] == e + 127 and (c[0, 2] >> 4) == 7     # channel 5: high nibble of byte 2
        x[0, 5] = np.nextafter(np.float32(6 * s), np.float32(np.inf))   # just above: e + 1
        c, b = codecs.fp4b32_encode(x)
        assert b[0, 0] == e + 128
        x[0, 5] = np.nextafter(np.float32(3 * s), np.float32(np.inf))   # just above 3 * 2^e: still e
        c, b = codecs.fp4b32_encode(x)
        assert b[0, 0] == e + 127
    z = np.zeros((1, 32), np.float32)
    z[0, 1] = -0.0
    c, b = codecs.fp4b32_encode(z)
    assert b[0, 0] == 127 and c[0, 0] == 0x80          # -0 keeps its sign bit (code 8)
    rs = np.random.default_rng(5)
    x = (rs.standard_normal((500, 128)) * np.exp2(rs.integers(-30, 30, (500, 1)))).astype(np.float32)
    c, b = codecs.fp4b32_encode(x)
    e = b.astype(np.int64) - 127
    amax = np.max(np.abs(x.reshape(500, 4, 32)), axis=-1).astype(np.float64)
    assert np.all(amax <= 6 * np.exp2(e)) and np.all(amax > 3 * np.exp2(e))   # the smallest such e


def test_fp4b32_codes_are_nearest_grid_values_ties_to_even():
    rs = np.random.default_rng(6)
    grid = codecs.E2M1_VALUES
    x = rs.standard_normal((300, 128)).astype(np.float32)
    # plant ties: midpoints between neighbouring grid values at the block's scale
    x[:, 0] = 6.0
    x[:, 1] = 0.25
    x[:, 2] = 2.5
    x[:, 3] = -5.0
    c, b = codecs.fp4b32_encode(x)
    got = codecs.fp4b32_decode(c, b)
    s = np.repeat(codecs.e8m0_decode(b), 32, axis=1)
    y = x.astype(np.float64) / s
    dist = np.abs(np.abs(y)[..., None] - grid)
    best = np.argmin(dist, axis=-1)
    tie = np.sum(dist == dist.min(axis=-1, keepdims=True), axis=-1) > 1
    # ties: the even code (e2m1 codes 0..7 index the grid; "even" = mantissa bit 0)
    up = np.minimum(best + 1, 7)
    best = np.where(tie & (best % 2 == 1), up, best)
    ref = np.sign(y) * grid[best] * s
    assert np.array_equal(np.abs(got), np.abs(ref))
    assert np.all((got == 0) | (np.sign(got) == np.sign(x)))


def test_fp4h_row_bytes_and_page_layout():
    assert codecs.row_bytes(codecs.FMT_FP4H_PAGESPLIT, 128) == 68
    rs = np.random.default_rng(8)
    x = rs.standard_normal((128, 128)).astype(np.float32)
    pages = codecs.encode_fp4h_pagesplit(x)
    assert pages.shape == (2, 64 * 68)
    c, s = codecs.fp4b32_encode(codecs.hadamard_contract(x))
    assert np.array_equal(pages[1, :4096].reshape(64, 64), c[64:])
    assert np.array_equal(pages[1, 4096:].reshape(64, 4), s[64:])
    np.testing.assert_array_equal(codecs.decode_fp4h_pagesplit(pages, 128), codecs.fp4b32_decode(c, s))


def test_fp4_scores_from_rotated_operands_equal_the_unrotated_ones():
    # the rotation of both sides leaves every score unchanged (before rounding)
    rs = np.random.default_rng(9)
    q = rs.standard_normal((16, 128))
    k = rs.standard_normal((200, 128))
    w = rs.standard_normal(16)
    np.testing.assert_allclose(indexer.scores_fp64(codecs.hadamard_fp64(q), w, codecs.hadamard_fp64(k)),
                               indexer.scores_fp64(q, w, k), rtol=1e-11, atol=1e-11)


def test_fp4_selection_is_a_full_sort_of_bf16_scores():
    rs = np.random.default_rng(10)
    for n, k in ((5, 8), (40, 8), (300, 64), (1000, 512)):
        q = rs.standard_normal((8, 128)).astype(np.float32)
        w = rs.standard_normal(8).astype(np.float32)
        keys = rs.standard_normal((((n + 63) // 64) * 64, 128)).astype(np.float32)
        k_hat = codecs.decode_fp4h_pagesplit(codecs.encode_fp4h_pagesplit(keys), 128)
        topk, Ib, I = indexer.index_topk_fp4(q, w, k_hat, 4 * n + 3, 4, k)
        # brute force: sort by (bf16 score desc, index asc), keep min(k, n), ascending
        order = sorted(range(n), key=lambda j: (-Ib[j], j))[:min(k, n)]
        want = np.full(k, -1)
        want[:len(order)] = sorted(order)
        assert np.array_equal(topk, want)
        assert np.array_equal(Ib, codecs.bf16_decode(codecs.bf16_encode(I.astype(np.float32))))


def test_fp4_bf16_ties_go_to_the_smaller_entry():
    # two keys whose scores differ in fp64 but are equal in bf16: with room for one,
    # the smaller entry is kept
    q = np.zeros((1, 128), np.float32)
    q[0, 0] = 1.0
    w = np.ones(1, np.float32)
    base = np.zeros((64, 128), np.float32)
    base[:, 0] = 0.01
    k_hat = codecs.decode_fp4h_pagesplit(codecs.encode_fp4h_pagesplit(base), 128)
    qh = indexer.quantize_queries_fp4(q)
    I = indexer.scores_fp64(qh, w, k_hat)
    # perturb entry 9 upwards by less than half a bf16 step of its score, entry 3 stays
    k_hat = k_hat.copy()
    step = np.abs(I[9]) * 2.0 ** -10
    dot_unit = float(np.dot(qh[0], qh[0]))
    k_hat[9] = k_hat[9] + qh[0] * (step / dot_unit)
    topk, Ib, I2 = indexer.index_topk_fp4(q, w, k_hat, 4 * 64, 4, 1)
    assert I2[9] > I2[3] and Ib[9] == Ib[3]
    assert topk[0] == 0      # all 64 tie in bf16: the smallest index wins
