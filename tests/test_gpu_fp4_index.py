"""GPU parity: FP4 index keys ("DeepSeek-V4 deep dive", section 5.2) - the rotated
e2m1 + e8m0-per-32 keys and queries scored by the block-scaled tensor-core product,
BF16 scores, top-k - against the oracle."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from oracle import codecs, indexer

from cases import HostPaged, bf16_values, check_topk_fp4, cuda

pytestmark = pytest.mark.gpu

FP4H = codecs.FMT_FP4H_PAGESPLIT


def _run(q_t, w, cache, ctx, ratio, k, max_ctx):
    dev = cache.to_device()
    idx, sc = cskv.index_topk(q_t.cuda(), cuda(w), dev, cuda(np.asarray(ctx, np.int32)), ratio, k, max_ctx)
    assert cskv.device_status() == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("Hi", [64, 16, 1])
def test_random_fp4_keys(Hi):
    ratio, k = 4, 512
    ctx = [4 * 7000 + 1, 4 * 513, 4 * 512, 4 * 129 + 3, 4 * 20001, 0]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(40 + Hi)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(FP4H, 128, [max(1, x) for x in n], seed=41)
    for b, nb in enumerate(n):
        cache.fill(b, (rs.standard_normal((max(1, nb), 128)) * np.exp2(rs.integers(-8, 8, (max(1, nb), 1)))).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    swaps = 0
    for b, nb in enumerate(n):
        if nb == 0:
            assert np.all(idx[b] == -1)
            continue
        swaps += check_topk_fp4(idx[b], sc[b], q_v[b], w[b], cache.decoded[b], nb, k)
    assert swaps <= 4


def _lsb_exponent(v):
    """Exponent of the lowest set bit over the nonzero values (all are dyadic)."""
    v = np.abs(np.asarray(v, np.float64))
    v = v[v != 0]
    mant, ex = np.frexp(v)
    bits = np.round(mant * 2.0 ** 53).astype(np.int64)
    tz = np.array([(int(b) & -int(b)).bit_length() - 1 for b in bits])
    return int(np.min(ex - 53 + tz))


def _exact_safe(qh, w, kh):
    """Every product q * k * w is a multiple of 2^u (u from the operands' lowest bits); if
    every score's l1 mass stays below 2^(24 + u), every partial sum in any order is an
    exactly representable fp32 value."""
    u = _lsb_exponent(kh) + _lsb_exponent(qh) + _lsb_exponent(w)
    mass = np.abs(kh) @ (np.abs(qh).T @ np.abs(np.asarray(w, np.float64)))
    return bool(np.all(mass < 2.0 ** (24 + u)))


def test_integer_inputs_exact():
    """Small-integer keys and queries, weights 1/2: the rotation and the FP4 codes are
    reproduced bit for bit, every fp32 partial sum of every score is exact (checked), so
    the bf16 scores and the selected sets must equal the oracle's exactly."""
    ratio, k, Hi = 4, 256, 4
    ctx = [4 * 3000 + 3, 4 * 700, 4 * 300 + 1]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(50)
    q = rs.integers(-2, 3, (len(ctx), Hi, 128)).astype(np.float32)
    w = np.full((len(ctx), Hi), 0.5, np.float32)
    cache = HostPaged(FP4H, 128, n, seed=51)
    for b, nb in enumerate(n):
        cache.fill(b, rs.integers(-2, 3, (nb, 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    for b, nb in enumerate(n):
        qh = indexer.quantize_queries_fp4(q_v[b])
        assert _exact_safe(qh, w[b], cache.decoded[b][:nb]), "inputs not exact in fp32"
        topk, Ib, I = indexer.index_topk_fp4(q_v[b], w[b], cache.decoded[b], ctx[b], ratio, k)
        assert np.array_equal(idx[b], topk), b
        m = min(k, nb)
        assert np.array_equal(sc[b, :m].astype(np.float64), Ib[topk[:m]])


def test_bf16_ties_resolved_to_smaller_entries():
    """Many keys share one bf16 score (equal codes): the selection keeps the smallest
    entries among them, as the oracle does."""
    ratio, k, Hi = 4, 64, 8
    nb = 1000
    rs = np.random.default_rng(52)
    base = rs.standard_normal((1, 128)).astype(np.float32)
    keys = np.repeat(base, nb, axis=0)
    keys[::7] = rs.standard_normal((len(keys[::7]), 128)).astype(np.float32)
    q = rs.standard_normal((1, Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (1, Hi)).astype(np.float32)
    cache = HostPaged(FP4H, 128, [nb], seed=53)
    cache.fill(0, keys)
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, [4 * nb], ratio, k, 4 * nb)
    assert check_topk_fp4(idx[0], sc[0], q_v[0], w[0], cache.decoded[0], nb, k) == 0
