"""GPU parity on the named workloads themselves: the tiny CSA layer end to end (compress,
index, attend; the oracle finishes it in seconds), and the 1M-context and mixed-batch MXFP4
decode layers at full size, every request's selection and attention output against the
oracle - also through the fused decode step the benchmark times."""

import concurrent.futures

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from compressed_sparse_attention_kv_gb300 import synth
from oracle import attention as o_attn, codecs, compress as o_comp, indexer, rope as o_rope

from cases import bf16_values, check_attention, check_topk, check_topk_fp4, cuda, swa_ring

pytestmark = pytest.mark.gpu

SCALE = 512 ** -0.5


def _page_bytes(fmt, dim):
    return (64 * codecs.row_bytes(fmt, dim) + 15) // 16 * 16


def _build_lane(wl, lane, fmt, dim):
    """Device cache of one lane of a (possibly ragged) workload, coded on the GPU from the
    seeded values, request by request."""
    bt, num_pages = synth.page_tables(wl, lane)
    cache = cskv.PagedCache(torch.zeros((num_pages, _page_bytes(fmt, dim)), dtype=torch.uint8, device="cuda"),
                            cuda(bt), fmt, dim)
    f = synth.index_page_values if lane == "index" else synth.main_page_values
    ppr = wl.pages_per_req()
    with concurrent.futures.ThreadPoolExecutor(max_workers=16) as ex:
        for b in range(wl.B):
            pages = list(ex.map(lambda p: f(wl, b, p), range(int(ppr[b]))))
            vals = torch.from_numpy(np.concatenate(pages)).cuda()
            rows = torch.arange(vals.shape[0], dtype=torch.int32, device="cuda")
            cskv.encode_rows(vals, cache, req=torch.full_like(rows, b), row=rows)
            del vals
    return cache


def _oracle_keys(wl, b):
    """The oracle's decoded index keys of request b (coded by the oracle's codecs; FP4
    keys come out rotated)."""
    vals = synth.request_values(wl, b, "index")
    n = int(wl.n_entries[b])
    if wl.key_fmt == codecs.FMT_FP4H_PAGESPLIT:
        return codecs.decode_fp4h_pagesplit(codecs.encode_fp4h_pagesplit(vals), 128)[:n]
    return codecs.decode_pagesplit(codecs.encode_pagesplit(vals), 128)[:n]


def _check_selection(wl, b, got, qi, w, k_hat, n, ctx):
    """The GPU's selection of request b against the oracle; returns the oracle's selection."""
    if wl.key_fmt == codecs.FMT_FP4H_PAGESPLIT:
        assert check_topk_fp4(got, None, qi, w, k_hat, n, wl.k) == 0, b
        return indexer.index_topk_fp4(qi, w, k_hat, ctx, wl.ratio, wl.k)[0]
    q_hat = indexer.quantize_queries(qi)
    assert check_topk(got, None, q_hat, w, k_hat, n, wl.k) == 0, b
    return indexer.select_topk(indexer.scores_fp64(q_hat, w, k_hat), wl.k)


def _oracle_entries(wl, b, rows, fmt):
    """Decoded main entries of request b at the given rows (others zero): [n_b, 512]."""
    n = int(wl.n_entries[b])
    out = np.zeros((n, 512))
    pages = synth.request_values(wl, b, "main", rows=rows)
    for p, v in pages.items():
        dec = codecs.decode_rows(codecs.encode_rows(v, fmt), fmt, 512)
        lo = p * 64
        hi = min(n, lo + 64)
        out[lo:hi] = dec[:hi - lo]
    return out


def _full_size(name, sample):
    wl = synth.workload(name)
    keys = _build_lane(wl, "index", wl.key_fmt, 128)
    main = _build_lane(wl, "main", wl.main_fmt, 512)
    swa_vals = np.stack([synth.swa_values(wl, b) for b in range(wl.B)])
    swa_b, swa_dec = swa_ring(swa_vals, wl.swa_fmt)
    q, q_idx, w, sink = synth.queries(wl)
    q_t, q_v = bf16_values(q)
    qi_t, qi_v = bf16_values(q_idx)
    ctx = wl.ctx_len.astype(np.int32)
    topk, _ = cskv.index_topk(qi_t.cuda(), cuda(w), keys, cuda(ctx), wl.ratio, wl.k, wl.max_ctx, want_scores=False)
    out = cskv.sparse_decode_attn(q_t.cuda(), main, cuda(swa_b), wl.swa_fmt, cuda(ctx), topk, wl.k, wl.ratio,
                                  wl.max_ctx, cuda(sink), SCALE, cuda(cskv.rope_table(ctx - 1)))
    assert cskv.device_status() == 0
    topk = topk.cpu().numpy()
    got = out.float().cpu().numpy()
    for b in sample:
        n = int(wl.n_entries[b])
        k_hat = _oracle_keys(wl, b)
        sel = _check_selection(wl, b, topk[b], qi_v[b], w[b], k_hat, n, int(ctx[b]))
        ent = _oracle_entries(wl, b, sel[sel >= 0], wl.main_fmt)
        ref = o_attn.request_attention(q_v[b], int(ctx[b]), wl.ratio, swa_dec[b], ent, sel, sink, SCALE)
        check_attention(got[b], ref, fp4=wl.main_fmt == synth.FMT_FP4)


def test_csa_1m_full_size_every_request():
    """Batch 8 at 1,048,576 tokens: the selection and the attention output of every
    request against the oracle."""
    _full_size("csa_1m", range(8))


def test_csa_fp4_keys_full_size_every_request():
    """The 1M-context batch with FP4 index keys (rotated, e2m1 + e8m0 per 32, BF16
    scores): every request's selection and attention output against the oracle."""
    _full_size("csa_fp4", range(8))


def test_mixed_mxfp4_full_size_every_request():
    """Batch 64 with contexts from 32,768 to 524,288 tokens, MXFP4 main entries: the
    selection and the attention output of every request against the oracle."""
    _full_size("mixed_mxfp4", range(64))


def test_csa_1m_fused_decode_step_every_request():
    """The same batch through one cskv_decode_layer call (device buffers): the indexer's
    prep, the compressor writing every request's newest main entry and index key, the
    score kernel overlapping it, the attention starting per request on its ready flag.
    Every request's selection and output against the oracle, which codes the same
    newest entries itself."""
    wl = synth.workload("csa_1m")
    keys = _build_lane(wl, "index", synth.FMT_FP8_PAGESPLIT, 128)
    main = _build_lane(wl, "main", wl.main_fmt, 512)
    swa_vals = np.stack([synth.swa_values(wl, b) for b in range(wl.B)])
    swa_b, swa_dec = swa_ring(swa_vals, wl.swa_fmt)
    q, q_idx, w, sink = synth.queries(wl)
    q_t, q_v = bf16_values(q)
    qi_t, qi_v = bf16_values(q_idx)
    ctx = wl.ctx_len.astype(np.int32)
    r, B = wl.ratio, wl.B
    n = (ctx // r).astype(np.int64)
    first = (n - 1).astype(np.int32)
    lanes = {}
    for lane, dim, il in (("main", 512, False), ("index", 128, True)):
        kv, gate, pkv, pgate = [], [], [], []
        for b in range(B):
            a_, g_ = synth.compressor_tokens(wl.seed, r, r, True, dim, index_lane=il, seq=b)
            pa, pg = synth.compressor_prev(wl.seed, r, dim, index_lane=il, seq=b)
            kv.append(a_); gate.append(g_); pkv.append(pa); pgate.append(pg)
        ape, nw = synth.compressor_params(wl.seed, r, True, dim, index_lane=il)
        lanes[lane] = dict(kv=bf16_values(np.stack(kv)), gate=bf16_values(np.stack(gate)),
                           pkv=bf16_values(np.stack(pkv)), pgate=bf16_values(np.stack(pgate)), ape=ape, nw=nw)
    ecs = cskv.rope_table((first.astype(np.int64) * r)[:, None])
    jobs = []
    for lane, cache in (("main", main), ("index", keys)):
        L_ = lanes[lane]
        jobs.append(dict(kv=L_["kv"][0].cuda(), gate=L_["gate"][0].cuda(), ape=cuda(L_["ape"]), ratio=r, overlap=True,
                         out=cache, req=cuda(np.arange(B, dtype=np.int32)), first_entry=cuda(first),
                         prev_kv=L_["pkv"][0].cuda(), prev_gate=L_["pgate"][0].cuda(), norm_w=cuda(L_["nw"]),
                         rope_cs=cuda(ecs)))
    out, topk = cskv.decode_layer(jobs, qi_t.cuda(), cuda(w), keys, q_t.cuda(), main, cuda(swa_b), wl.swa_fmt,
                                  cuda(ctx), wl.k, r, wl.max_ctx, cuda(sink), SCALE, cuda(cskv.rope_table(ctx - 1)))
    assert cskv.device_status() == 0
    topk = topk.cpu().numpy()
    got = out.float().cpu().numpy()
    for b in range(B):
        nb = int(n[b])
        cs = o_rope.table(np.array([int(first[b]) * r]))
        ents = {}
        for lane in ("main", "index"):
            L_ = lanes[lane]
            ents[lane] = o_comp.compress_contract(L_["kv"][1][b], L_["gate"][1][b], L_["ape"], r, True,
                                                  prev_kv=L_["pkv"][1][b], prev_gate=L_["pgate"][1][b],
                                                  norm_w=L_["nw"], eps=1e-6, rope_cs=cs)[0]
        k_hat = _oracle_keys(wl, b)
        k_hat[nb - 1] = codecs.decode_pagesplit(codecs.encode_pagesplit(np.tile(ents["index"], (64, 1))), 128)[0]
        q_hat = indexer.quantize_queries(qi_v[b])
        assert check_topk(topk[b], None, q_hat, w[b], k_hat, nb, wl.k) == 0, b
        sel = indexer.select_topk(indexer.scores_fp64(q_hat, w[b], k_hat), wl.k)
        ent = _oracle_entries(wl, b, sel[sel >= 0], wl.main_fmt)
        ent[nb - 1] = codecs.decode_rows(codecs.encode_rows(ents["main"][None], wl.main_fmt), wl.main_fmt, 512)[0]
        ref = o_attn.request_attention(q_v[b], int(ctx[b]), r, swa_dec[b], ent, sel, sink, SCALE)
        check_attention(got[b], ref, fp4=wl.main_fmt == synth.FMT_FP4)


def test_tiny_csa_end_to_end():
    """The tiny CSA layer: 4,096 tokens compressed (ratio 4, overlap) into bf16 main entries
    and index keys, 4 indexer heads select 512 of the 1,024 entries, 16 heads attend."""
    wl = synth.workload("tiny_csa")
    T, r, n = 4096, 4, 1024
    outs = {}
    for lane, dim, idx_lane in (("main", 512, False), ("index", 128, True)):
        kv, gate = synth.compressor_tokens(wl.seed, T, r, True, dim, index_lane=idx_lane)
        ape, nw = synth.compressor_params(wl.seed, r, True, dim, index_lane=idx_lane)
        kv_t, kv_v = bf16_values(kv)
        g_t, g_v = bf16_values(gate)
        dev = cskv.PagedCache(torch.zeros((n // 64, 64 * dim * 2), dtype=torch.uint8, device="cuda"),
                              cuda(np.arange(n // 64, dtype=np.int32)[None]), codecs.FMT_BF16, dim)
        cskv.compress(kv_t[None].cuda(), g_t[None].cuda(), cuda(ape), r, 1, dev, cuda(np.array([0], np.int32)),
                      cuda(np.array([0], np.int32)), norm_w=cuda(nw), eps=1e-6,
                      rope_cs=cuda(cskv.rope_table(np.arange(n) * r)[None]))
        ents = o_comp.compress_contract(kv_v, g_v, ape, r, True, norm_w=nw, eps=1e-6,
                                        rope_cs=o_rope.table(np.arange(n) * r))
        want = codecs.encode_rows(ents, codecs.FMT_BF16)
        got = dev.pool.cpu().numpy()[:, :64 * want.shape[1]].reshape(n, -1)
        assert np.array_equal(got, want), lane
        outs[lane] = (dev, codecs.decode_rows(want, codecs.FMT_BF16, dim))
    swa_b, swa_dec = swa_ring(synth.swa_values(wl, 0)[None], codecs.FMT_BF16)
    q, q_idx, w, sink = synth.queries(wl)
    q_t, q_v = bf16_values(q)
    qi_t, qi_v = bf16_values(q_idx)
    ctx = np.array([T], np.int32)
    topk, sc = cskv.index_topk(qi_t.cuda(), cuda(w), outs["index"][0], cuda(ctx), r, wl.k, T)
    out = cskv.sparse_decode_attn(q_t.cuda(), outs["main"][0], cuda(swa_b), codecs.FMT_BF16, cuda(ctx), topk,
                                  wl.k, r, T, cuda(sink), SCALE, cuda(cskv.rope_table(ctx - 1)))
    assert cskv.device_status() == 0
    k_hat = outs["index"][1]
    q_hat = qi_v[0].astype(np.float64)          # bf16 keys: the queries are used as given
    assert check_topk(topk.cpu().numpy()[0], sc.cpu().numpy()[0], q_hat, w[0], k_hat, n, wl.k) == 0
    sel = indexer.select_topk(indexer.scores_fp64(q_hat, w[0], k_hat), wl.k)
    ref = o_attn.request_attention(q_v[0], T, r, swa_dec[0], outs["main"][1], sel, sink, SCALE)
    check_attention(out.float().cpu().numpy()[0], ref)
