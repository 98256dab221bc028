"""GPU parity: lightning indexer + top-k against the oracle."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from compressed_sparse_attention_kv_gb300 import synth
from oracle import codecs, indexer

from cases import HostPaged, bf16_values, check_topk, cuda, swa_ring

pytestmark = pytest.mark.gpu


def _run(q_t, w, cache, ctx, ratio, k, max_ctx):
    dev = cache.to_device()
    idx, sc = cskv.index_topk(q_t.cuda(), cuda(w), dev, cuda(np.asarray(ctx, np.int32)), ratio, k, max_ctx)
    assert cskv.device_status() == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


def test_integer_inputs_exact_with_ties():
    """Integer-valued q, k, w: every fp32 partial sum is exact, so the selected sets
    (with their tie-breaks to the smaller index) must equal the oracle's exactly."""
    ratio, k, Hi = 4, 512, 64
    ctx = [4 * 1000 + 3, 4 * 5000, 4 * 300 + 1, 4 * 777 + 2]
    n = [c // ratio for c in ctx]
    q, _, w = synth.integer_index_inputs(11, len(ctx), Hi, 1)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=5)
    keys = []
    for b, nb in enumerate(n):
        _, kk, _ = synth.integer_index_inputs(100 + b, 1, 1, nb)
        cache.fill(b, kk)
        keys.append(cache.decoded[b])
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    for b, nb in enumerate(n):
        q_hat = indexer.quantize_queries(q_v[b])
        I = indexer.scores_fp64(q_hat, w[b], keys[b])
        ref = indexer.select_topk(I, k)
        assert np.array_equal(idx[b], ref), b
        m = min(k, nb)
        assert np.array_equal(sc[b, :m].astype(np.float64), I[ref[:m]])
        assert np.all(np.isneginf(sc[b, m:]))


@pytest.mark.parametrize("Hi", [64, 16, 4])
def test_random_fp8_keys(Hi):
    ratio, k = 4, 512
    ctx = [4 * 7000 + 1, 4 * 513, 4 * 512, 4 * 129 + 3, 4 * 20001]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(Hi)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=6)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((nb, 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    swaps = 0
    for b, nb in enumerate(n):
        swaps += check_topk(idx[b], sc[b], indexer.quantize_queries(q_v[b]), w[b], cache.decoded[b], nb, k)
    assert swaps <= 1


def test_bf16_keys_and_negative_weights():
    ratio, k, Hi = 4, 64, 8
    ctx = [4 * 1024, 4 * 50 + 2, 4 * 3000 + 1]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(3)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(-1, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(codecs.FMT_BF16, 128, n, seed=7)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((nb, 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    for b, nb in enumerate(n):
        check_topk(idx[b], sc[b], q_v[b].astype(np.float64), w[b], cache.decoded[b], nb, k)


def test_empty_and_tiny_contexts():
    ratio, k, Hi = 4, 16, 4
    ctx = [0, 3, 4, 4 * 16, 4 * 17]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(4)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, [max(1, x) for x in n], seed=8)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((max(1, nb), 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    assert np.all(idx[0] == -1) and np.all(idx[1] == -1)
    assert idx[2, 0] == 0 and np.all(idx[2, 1:] == -1)
    assert np.array_equal(idx[3], np.arange(16))
    check_topk(idx[4], sc[4], indexer.quantize_queries(q_v[4]), w[4], cache.decoded[4], n[4], k)


def test_csa_1m_full_size_sampled():
    """The 1M-context workload (batch 8, 262,144 FP8 keys per request, 64 heads,
    top-512) in the bench's launch configuration; two requests checked in full."""
    wl = synth.workload("csa_1m")
    n = int(wl.n_entries[0])
    bt, num_pages = synth.page_tables(wl, "index")
    pb = 64 * 132
    pool = torch.zeros((num_pages, pb), dtype=torch.uint8, device="cuda")
    dev = cskv.PagedCache(pool, cuda(bt), codecs.FMT_FP8_PAGESPLIT, 128)
    ppr = int(wl.pages_per_req()[0])
    for b in range(wl.B):
        vals = synth.request_values(wl, b, "index")
        rows = np.arange(ppr * 64, dtype=np.int32)
        cskv.encode_rows(cuda(vals), dev, req=cuda(np.full(rows.shape, b, np.int32)), row=cuda(rows))
    _, q_idx, w, _ = synth.queries(wl)
    q_t, q_v = bf16_values(q_idx)
    ctx = wl.ctx_len.astype(np.int32)
    idx, sc = cskv.index_topk(q_t.cuda(), cuda(w), dev, cuda(ctx), wl.ratio, wl.k, wl.max_ctx)
    assert cskv.device_status() == 0
    idx = idx.cpu().numpy()
    sc = sc.cpu().numpy()
    for b in (0, 5):
        vals = synth.request_values(wl, b, "index")
        k_hat = codecs.decode_pagesplit(codecs.encode_pagesplit(vals), 128)
        check_topk(idx[b], sc[b], indexer.quantize_queries(q_v[b]), w[b], k_hat, n, wl.k)


def test_many_empty_requests_share_a_block():
    """Twenty empty requests in a row all belong to one block's selection work (more than
    that block's work list holds), then requests of 125, 0, 175 and 0 entries."""
    ratio, k, Hi = 4, 16, 4
    ctx = [0] * 20 + [4 * 125 + 1, 2, 4 * 175, 3]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(12)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, [max(1, x) for x in n], seed=13)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((max(1, nb), 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    for b, nb in enumerate(n):
        if nb == 0:
            assert np.all(idx[b] == -1), b
        else:
            check_topk(idx[b], sc[b], indexer.quantize_queries(q_v[b]), w[b], cache.decoded[b], nb, k)


@pytest.mark.parametrize("Hi,k", [(1, 2048), (64, 2048), (3, 1)])
def test_extreme_k_and_heads(Hi, k):
    """The largest selection (k = 2048), a single indexer head, and k = 1."""
    ratio = 4
    ctx = [4 * 9000 + 3, 4 * 2048, 4 * 2047 + 1, 4 * 5000]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(60 + Hi + k)
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=61)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((nb, 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    swaps = 0
    for b, nb in enumerate(n):
        swaps += check_topk(idx[b], sc[b], indexer.quantize_queries(q_v[b]), w[b], cache.decoded[b], nb, k)
    assert swaps <= 1


@pytest.mark.parametrize("fmt", [codecs.FMT_FP8_PAGESPLIT, codecs.FMT_BF16])
def test_large_ragged_batch(fmt):
    """A batch of 700 requests (the large-batch prologue; for FP8 keys also the scheduler
    that counts the tiles handed out): empty, tiny and long contexts mixed, most requests
    shorter than one 128-entry tile, a few hundred times longer."""
    ratio, k, Hi = 4, 64, 8
    rs = np.random.default_rng(70 + fmt)
    n = rs.choice([0, 1, 5, 63, 64, 65, 127, 128, 129, 300, 1000], size=700).tolist()
    for b in rs.choice(700, 6, replace=False):
        n[b] = int(rs.integers(20000, 40000))
    ctx = [ratio * nb + int(rs.integers(0, ratio)) for nb in n]
    q = rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32)
    w = rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32)
    cache = HostPaged(fmt, 128, [max(1, x) for x in n], seed=71)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((max(1, nb), 128)).astype(np.float32))
    q_t, q_v = bf16_values(q)
    idx, sc = _run(q_t, w, cache, ctx, ratio, k, max(ctx))
    swaps = 0
    for b, nb in enumerate(n):
        if nb == 0:
            assert np.all(idx[b] == -1), b
            continue
        q_hat = indexer.quantize_queries(q_v[b]) if fmt == codecs.FMT_FP8_PAGESPLIT else q_v[b].astype(np.float64)
        swaps += check_topk(idx[b], sc[b], q_hat, w[b], cache.decoded[b][:nb], nb, k)
    assert swaps <= 2


def test_results_are_identical_run_to_run():
    """Dynamic tile scheduling and atomic histograms leave no trace in the results: two
    runs of the indexer and the attention give the same bits (each score is one thread's
    fixed-order sum, the counts are order-free, partials are merged in tile order)."""
    ratio, k, Hi, H = 4, 512, 64, 64
    ctx = [4 * 60000 + 1, 4 * 41000, 4 * 9000 + 3, 4 * 70000 + 2, 4 * 513, 4 * 30000]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(80)
    keys = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=81)
    main = HostPaged(codecs.FMT_FP8, 512, n, seed=82)
    for b, nb in enumerate(n):
        keys.fill(b, rs.standard_normal((nb, 128)).astype(np.float32))
        main.fill(b, rs.standard_normal((nb, 512)).astype(np.float32))
    qi_t, _ = bf16_values(rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32))
    q_t, _ = bf16_values(rs.standard_normal((len(ctx), H, 512)).astype(np.float32))
    w = cuda(rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32))
    swa = cuda(swa_ring(rs.standard_normal((len(ctx), 128, 512)).astype(np.float32), codecs.FMT_FP8)[0])
    sink = cuda(rs.standard_normal(H).astype(np.float32))
    ctx_d = cuda(np.asarray(ctx, np.int32))
    cs = cuda(cskv.rope_table(np.asarray(ctx) - 1))
    kd, md = keys.to_device(), main.to_device()
    runs = []
    for _ in range(3):
        idx, sc = cskv.index_topk(qi_t.cuda(), w, kd, ctx_d, ratio, k, max(ctx))
        out = cskv.sparse_decode_attn(q_t.cuda(), md, swa, codecs.FMT_FP8, ctx_d, idx, k, ratio, max(ctx), sink,
                                      512 ** -0.5, cs)
        runs.append((idx.clone(), sc.clone(), out.clone()))
    assert cskv.device_status() == 0
    for idx, sc, out in runs[1:]:
        assert torch.equal(idx, runs[0][0])
        assert torch.equal(sc.view(torch.int32), runs[0][1].view(torch.int32))
        assert torch.equal(out.view(torch.int16), runs[0][2].view(torch.int16))
