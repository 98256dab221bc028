"""GPU parity for the V4.1 CSA2 variant ("DeepSeek-V4.1 Flash", section 1.1; the
architecture diagram's encoder and decoder CSA2 blocks).

The encoder merges 2 adjacent positions into one entry (ratio 2), the decoder keeps
one entry per position (ratio 1); neither compressor has an overlap or a slot bias.
Several layers share one global KV and one top-512 (Full / Reindex / Reuse).  The
chain runs as it does in a decode step: the main-KV and index-key compressors write
the paged caches (one launch), the indexer selects over those keys, and every layer's
attention reads the shared cache with the shared selection, all on the device.  The
oracle recomputes each stage from the same bf16 inputs.
"""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from oracle import attention as o_attn, codecs, compress as o_comp, indexer, rope as o_rope

from cases import HostPaged, PAGE, bf16_values, check_attention, check_topk, cuda, swa_ring

pytestmark = pytest.mark.gpu

SCALE = 512 ** -0.5
CHUNK = 256     # entries per full compressor chunk
K = 512


def _layout(ratio, chunks, tail, extra):
    n = [c * CHUNK + tail for c in chunks]
    ctx = np.array([ratio * nb + e for nb, e in zip(n, extra)], np.int32)
    return n, ctx


def _jobs(ratio, dim, chunks, tail, rs):
    """bf16 inputs of the two compressor jobs that fill one cache: full chunks
    (sequence = one chunk of one request) and the common-length tails."""
    B = len(chunks)
    seqs = [(b, c * CHUNK) for b in range(B) for c in range(chunks[b])]
    jobs = []
    for T_ent, sq in ((CHUNK, seqs), (tail, [(b, chunks[b] * CHUNK) for b in range(B)])):
        S, T = len(sq), T_ent * ratio
        kv_t, kv_v = bf16_values(rs.standard_normal((S, T, 1, dim)).astype(np.float32))
        g_t, g_v = bf16_values((1.5 * rs.standard_normal((S, T, 1, dim))).astype(np.float32))
        req = np.array([b for b, _ in sq], np.int32)
        first = np.array([f for _, f in sq], np.int32)
        pos = [(f + np.arange(T_ent)) * ratio for f in first]
        jobs.append(dict(kv=(kv_t, kv_v), gate=(g_t, g_v), req=req, first=first, pos=pos, n=T_ent))
    return jobs


def _oracle_entries(jobs, ratio, dim, nw, n):
    """Entries [n_b, dim] of every request, by the oracle's fp32 contract."""
    out = [np.zeros((nb, dim), np.float32) for nb in n]
    ape = np.zeros((ratio, dim), np.float32)
    for j in jobs:
        for s in range(len(j["req"])):
            e = o_comp.compress_contract(j["kv"][1][s], j["gate"][1][s], ape, ratio, False, norm_w=nw,
                                         eps=1e-6, rope_cs=o_rope.table(j["pos"][s]))
            f = int(j["first"][s])
            out[int(j["req"][s])][f:f + j["n"]] = e
    return out


def _device_job(j, ratio, nw, dev):
    return dict(kv=j["kv"][0].cuda(), gate=j["gate"][0].cuda(), ape=None, ratio=ratio, overlap=0, out=dev,
                req=cuda(j["req"]), first_entry=cuda(j["first"]), norm_w=cuda(nw), eps=1e-6,
                rope_cs=cuda(np.stack([cskv.rope_table(p) for p in j["pos"]])))


def _rows_equal(host, got_pool, b, n):
    """Request b's first n rows of a device pool image equal the oracle-coded host pool."""
    rb = codecs.row_bytes(host.fmt, host.dim)
    for p in range((n + PAGE - 1) // PAGE):
        pg = host.block_table[b, p]
        m = min(PAGE, n - p * PAGE)
        want, got = host.pool[pg], got_pool[pg]
        if host.fmt == codecs.FMT_FP8_PAGESPLIT:
            d = host.dim
            ok = (np.array_equal(got[:m * d], want[:m * d])
                  and np.array_equal(got[PAGE * d:PAGE * d + 4 * m], want[PAGE * d:PAGE * d + 4 * m]))
        else:
            ok = np.array_equal(got[:m * rb], want[:m * rb])
        if not ok:
            return False
    return True


@pytest.mark.parametrize("ratio,chunks,tail,extra", [
    (2, [3, 1, 6], 45, [1, 0, 1]),      # encoder CSA2: 2 positions per entry
    (1, [2, 0, 5], 45, [0, 0, 0]),      # decoder CSA2: one entry per position
])
def test_csa2_decode_chain(ratio, chunks, tail, extra):
    rs = np.random.default_rng(100 + ratio)
    B, H, Hi = len(chunks), 64, 64
    n, ctx = _layout(ratio, chunks, tail, extra)
    max_ctx = int(ctx.max())
    nw_main = rs.uniform(0.5, 1.5, 512).astype(np.float32)
    nw_idx = rs.uniform(0.5, 1.5, 128).astype(np.float32)
    jobs_main = _jobs(ratio, 512, chunks, tail, rs)
    jobs_idx = _jobs(ratio, 128, chunks, tail, rs)

    # ---- compress: main KV (MXFP4, 288 B/entry) and index keys, one launch
    host_main = HostPaged(codecs.FMT_FP4, 512, n, seed=7)
    host_idx = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=8)
    dev_main = cskv.PagedCache(torch.zeros((host_main.num_pages, host_main.page_bytes), dtype=torch.uint8,
                                           device="cuda"), cuda(host_main.block_table), codecs.FMT_FP4, 512)
    dev_idx = cskv.PagedCache(torch.zeros((host_idx.num_pages, host_idx.page_bytes), dtype=torch.uint8,
                                          device="cuda"), cuda(host_idx.block_table),
                              codecs.FMT_FP8_PAGESPLIT, 128)
    cskv.compress_many([_device_job(j, ratio, nw_main, dev_main) for j in jobs_main if len(j["req"])] +
                       [_device_job(j, ratio, nw_idx, dev_idx) for j in jobs_idx if len(j["req"])])
    assert cskv.device_status() == 0
    ent_main = _oracle_entries(jobs_main, ratio, 512, nw_main, n)
    ent_idx = _oracle_entries(jobs_idx, ratio, 128, nw_idx, n)
    for b in range(B):
        host_main.fill(b, ent_main[b])
        host_idx.fill(b, ent_idx[b])
    got_main = dev_main.pool.cpu().numpy()
    got_idx = dev_idx.pool.cpu().numpy()
    for b in range(B):
        assert _rows_equal(host_main, got_main, b, n[b]), ("main", b)
        assert _rows_equal(host_idx, got_idx, b, n[b]), ("index", b)

    # ---- layers: Full (own indexer call), Reindex (another indexer call), then two Reuse
    ctx_d = cuda(ctx)
    cs = cskv.rope_table(ctx - 1)
    topk_dev, topk_ref = None, None
    for layer, mode in enumerate(("full", "reindex", "reuse", "reuse")):
        if mode != "reuse":
            q_idx = rs.standard_normal((B, Hi, 128)).astype(np.float32)
            w = rs.uniform(0, 1, (B, Hi)).astype(np.float32)
            qi_t, qi_v = bf16_values(q_idx)
            topk_dev, sc = cskv.index_topk(qi_t.cuda(), cuda(w), dev_idx, ctx_d, ratio, K, max_ctx)
            assert cskv.device_status() == 0
            got_idx_sel = topk_dev.cpu().numpy()
            sc = sc.cpu().numpy()
            topk_ref = np.full((B, K), -1, np.int32)
            for b in range(B):
                q_hat = indexer.quantize_queries(qi_v[b])
                swaps = check_topk(got_idx_sel[b], sc[b], q_hat, w[b], host_idx.decoded[b], n[b], K)
                assert swaps == 0, (layer, b, swaps)       # no near-tie with these seeds
                topk_ref[b] = indexer.select_topk(indexer.scores_fp64(q_hat, w[b], host_idx.decoded[b]), K)
        q_t, q_v = bf16_values(rs.standard_normal((B, H, 512)).astype(np.float32))
        sink = rs.standard_normal(H).astype(np.float32)
        swa_b, swa_dec = swa_ring(rs.standard_normal((B, 128, 512)).astype(np.float32), codecs.FMT_FP8)
        out = cskv.sparse_decode_attn(q_t.cuda(), dev_main, cuda(swa_b), codecs.FMT_FP8, ctx_d, topk_dev, K,
                                      ratio, max_ctx, cuda(sink), SCALE, cuda(cs))
        assert cskv.device_status() == 0
        got = out.float().cpu().numpy()
        for b in range(B):
            ref = o_attn.request_attention(q_v[b], int(ctx[b]), ratio, swa_dec[b], host_main.decoded[b],
                                           topk_ref[b], sink, SCALE)
            check_attention(got[b], ref, fp4=True)


def test_csa2_ratio2_compress_matches_ratio2_with_zero_bias_table():
    """No slot bias (a null table) writes the same bytes as an explicit zero table."""
    rs = np.random.default_rng(5)
    jobs = _jobs(2, 512, [2], 10, rs)
    nw = rs.uniform(0.5, 1.5, 512).astype(np.float32)
    pools = []
    for ape in (None, torch.zeros((2, 512), dtype=torch.float32, device="cuda")):
        host = HostPaged(codecs.FMT_FP8, 512, [2 * CHUNK + 10], seed=3)
        dev = cskv.PagedCache(torch.zeros((host.num_pages, host.page_bytes), dtype=torch.uint8, device="cuda"),
                              cuda(host.block_table), codecs.FMT_FP8, 512)
        js = [_device_job(j, 2, nw, dev) for j in jobs]
        for j in js:
            j["ape"] = ape
        cskv.compress_many(js)
        assert cskv.device_status() == 0
        pools.append(dev.pool)
    assert torch.equal(pools[0], pools[1])
