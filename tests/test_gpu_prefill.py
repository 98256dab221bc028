"""GPU parity for prefill ("DeepSeek-V4 deep dive", section 5.3: the prefill buffer [raw rows
of the prompt ; its compressed entries], window indices below 0 masked): many queries of two
prompts, each with its own causal window and its own top-k from the indexer, against the
oracle query by query."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from oracle import attention as o_attn, codecs, indexer

from cases import HostPaged, bf16_values, check_attention, check_topk, cuda

pytestmark = pytest.mark.gpu

SCALE = 512 ** -0.5


@pytest.mark.parametrize("main_fmt,win_fmt", [(codecs.FMT_FP8, codecs.FMT_FP8), (codecs.FMT_FP4, codecs.FMT_BF16)])
def test_prefill_queries_of_two_prompts(main_fmt, win_fmt):
    rs = np.random.default_rng(41 + main_fmt)
    ratio, k, H, Hi = 4, 64, 16, 8
    L = [1000, 701]                                   # prompt lengths (raw tokens)
    n = [x // ratio for x in L]                       # compressed entries of each prompt
    raw = HostPaged(win_fmt, 512, L, seed=1)          # the raw rows by position (the window's source)
    main = HostPaged(main_fmt, 512, n, seed=2)
    keys = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=3)
    for b in range(2):
        raw.fill(b, rs.standard_normal((L[b], 512)).astype(np.float32))
        main.fill(b, rs.standard_normal((n[b], 512)).astype(np.float32))
        keys.fill(b, rs.standard_normal((n[b], 128)).astype(np.float32))
    # queries: both prompts, positions from the first token on (window partly below 0)
    pos = []
    for b in range(2):
        p = np.concatenate([[0, 1, 3, 4, 126, 127, 128, 255, L[b] - 1], rs.choice(L[b], 60, replace=False)])
        pos += [(b, int(t)) for t in p]
    T = len(pos)
    req_of = np.array([b for b, _ in pos], np.int32)
    pos1 = np.array([t + 1 for _, t in pos], np.int32)
    q_t, q_v = bf16_values(rs.standard_normal((T, H, 512)).astype(np.float32))
    qi_t, qi_v = bf16_values(rs.standard_normal((T, Hi, 128)).astype(np.float32))
    w = rs.uniform(0, 1, (T, Hi)).astype(np.float32)
    sink = rs.standard_normal(H).astype(np.float32)
    max_ctx = max(L)
    # the indexer with one row per query: each query's row of the block table is its prompt's
    kdev = keys.to_device()
    kq = cskv.PagedCache(kdev.pool, cuda(keys.block_table[req_of]), kdev.fmt, kdev.dim)
    topk, sc = cskv.index_topk(qi_t.cuda(), cuda(w), kq, cuda(pos1), ratio, k, max_ctx)
    out = cskv.sparse_prefill_attn(q_t.cuda(), main.to_device(), raw.to_device(), cuda(pos1), topk, k, ratio,
                                   max_ctx, cuda(sink), SCALE, cuda(cskv.rope_table(pos1 - 1)), req_of=cuda(req_of))
    assert cskv.device_status() == 0
    topk = topk.cpu().numpy()
    sc = sc.cpu().numpy()
    got = out.float().cpu().numpy()
    for i, (b, t) in enumerate(pos):
        nv = (t + 1) // ratio
        q_hat = indexer.quantize_queries(qi_v[i])
        assert check_topk(topk[i], sc[i], q_hat, w[i], keys.decoded[b], nv, k) == 0, i
        sel = indexer.select_topk(indexer.scores_fp64(q_hat, w[i], keys.decoded[b][:nv]), k)
        ring = np.zeros((128, 512))
        for p in range(max(0, t - 127), t + 1):
            ring[p % 128] = raw.decoded[b][p]
        ref = o_attn.request_attention(q_v[i], t + 1, ratio, ring, main.decoded[b], sel, sink, SCALE)
        check_attention(got[i], ref, fp4=main_fmt == codecs.FMT_FP4)


def test_hca_prefill_reads_every_visible_entry():
    """HCA prefill (ratio 128, no selection): each query attends its causal window and
    every entry complete before it (j < floor((t + 1) / 128))."""
    rs = np.random.default_rng(45)
    ratio, H = 128, 16
    L = [128 * 9 + 40]
    n = [L[0] // ratio]
    raw = HostPaged(codecs.FMT_FP8, 512, L, seed=4)
    main = HostPaged(codecs.FMT_FP8, 512, n, seed=5)
    raw.fill(0, rs.standard_normal((L[0], 512)).astype(np.float32))
    main.fill(0, rs.standard_normal((n[0], 512)).astype(np.float32))
    pos = np.array([0, 100, 127, 128, 255, 256, 700, L[0] - 1], np.int64)
    T = len(pos)
    pos1 = (pos + 1).astype(np.int32)
    q_t, q_v = bf16_values(rs.standard_normal((T, H, 512)).astype(np.float32))
    sink = rs.standard_normal(H).astype(np.float32)
    out = cskv.sparse_prefill_attn(q_t.cuda(), main.to_device(), raw.to_device(), cuda(pos1), None, 0, ratio,
                                   L[0], cuda(sink), SCALE, cuda(cskv.rope_table(pos)),
                                   req_of=cuda(np.zeros(T, np.int32)))
    assert cskv.device_status() == 0
    got = out.float().cpu().numpy()
    for i, t in enumerate(pos):
        ring = np.zeros((128, 512))
        for p in range(max(0, int(t) - 127), int(t) + 1):
            ring[p % 128] = raw.decoded[0][p]
        ref = o_attn.request_attention(q_v[i], int(t) + 1, ratio, ring, main.decoded[0], None, sink, SCALE)
        check_attention(got[i], ref)
