"""Failure handling on the GPU without a fault: an index outside its table or pool is
skipped and reported (CSKV_ERR_BOUNDS), a bounded wait that runs out ends its kernel with
CSKV_ERR_TIMEOUT, and in both cases the context stays usable (the next calls are exact)."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from oracle import codecs, indexer

from cases import HostPaged, bf16_values, check_topk, cuda, swa_ring

pytestmark = pytest.mark.gpu

ERR_TIMEOUT, ERR_BOUNDS = 4, 5


def _index_case(seed=51):
    ratio, k, Hi = 4, 64, 8
    ctx = [4 * 900 + 1, 4 * 300, 4 * 1500]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(seed)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=seed + 1)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((nb, 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    return dict(ratio=ratio, k=k, ctx=ctx, n=n, w=w, cache=cache, q_t=q_t, q_v=q_v)


def _run_index(c, cache_dev):
    return cskv.index_topk(c["q_t"].cuda(), cuda(c["w"]), cache_dev, cuda(np.asarray(c["ctx"], np.int32)),
                           c["ratio"], c["k"], max(c["ctx"]))


def _check_index(c, idx, sc, skip=()):
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    for b, nb in enumerate(c["n"]):
        if b in skip:
            continue
        check_topk(idx[b], sc[b], indexer.quantize_queries(c["q_v"][b]), c["w"][b], c["cache"].decoded[b], nb, c["k"])


def test_page_outside_the_pool_is_skipped_and_reported():
    c = _index_case()
    assert cskv.device_status() == 0
    bad = c["cache"].block_table.copy()
    bad[1, 2] = c["cache"].num_pages + 7          # request 1's third page: outside the pool
    dev = cskv.PagedCache(cuda(c["cache"].pool), cuda(bad), codecs.FMT_FP8_PAGESPLIT, 128)
    idx, sc = _run_index(c, dev)
    assert cskv.device_status() == ERR_BOUNDS
    _check_index(c, idx, sc, skip=(1,))           # the other requests are exact
    assert cskv.device_status() == 0              # the status was taken (cleared) above
    # the same call on the good table is exact and clean
    idx, sc = _run_index(c, c["cache"].to_device())
    assert cskv.device_status() == 0
    _check_index(c, idx, sc)


def test_attention_row_outside_the_pool_is_skipped_and_reported():
    rs = np.random.default_rng(52)
    ctx = [4 * 700, 4 * 300 + 2]
    n = [x // 4 for x in ctx]
    cache = HostPaged(codecs.FMT_FP8, 512, n, seed=53)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((nb, 512)).astype(np.float32))
    swa_b, _ = swa_ring(rs.standard_normal((2, 128, 512)).astype(np.float32), codecs.FMT_FP8)
    q_t, _ = bf16_values(rs.standard_normal((2, 16, 512)).astype(np.float32))
    topk = np.stack([rs.choice(nb, 64, replace=False) for nb in n]).astype(np.int32)
    bad = cache.block_table.copy()
    bad[0, 0] = -9                                 # a page id below 0
    dev = cskv.PagedCache(cuda(cache.pool), cuda(bad), codecs.FMT_FP8, 512)
    cs = cskv.rope_table(np.asarray(ctx) - 1)
    args = (q_t.cuda(), None, cuda(swa_b), codecs.FMT_FP8, cuda(np.asarray(ctx, np.int32)), cuda(topk), 64, 4,
            max(ctx), None, 512 ** -0.5, cuda(cs))
    out_bad = cskv.sparse_decode_attn(args[0], dev, *args[2:])
    assert cskv.device_status() == ERR_BOUNDS
    out_good = cskv.sparse_decode_attn(args[0], cache.to_device(), *args[2:])
    assert cskv.device_status() == 0
    # request 1 never touches the bad page: its output is unchanged
    assert torch.equal(out_bad[1], out_good[1])
    assert torch.isfinite(out_bad.float()).all()


def test_bounded_waits_give_up_and_the_context_stays_usable():
    """A spin limit far below the time a key page takes to arrive: the indexer's waits
    give up, its blocks drain their copies, free their tensor memory and return, and the
    status reads CSKV_ERR_TIMEOUT; with the default limit the next call is exact."""
    c = _index_case(seed=54)
    dev = c["cache"].to_device()
    assert cskv.device_status() == 0
    try:
        cskv.set_spin_limit(64)
        _run_index(c, dev)
        assert cskv.device_status() == ERR_TIMEOUT
    finally:
        cskv.set_spin_limit(0)                     # back to the default
    idx, sc = _run_index(c, dev)
    assert cskv.device_status() == 0
    _check_index(c, idx, sc)
