"""GPU parity: shared-KV sparse decode attention against the fp64 oracle on the same coded bytes."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from compressed_sparse_attention_kv_gb300 import synth
from oracle import attention as o_attn, codecs

from cases import HostPaged, bf16_values, check_attention, cuda, swa_ring

pytestmark = pytest.mark.gpu

SCALE = 512 ** -0.5


def _case(ctx, ratio, k, H, main_fmt, swa_fmt, with_sink, seed, topk_mode="random"):
    rs = np.random.default_rng(seed)
    B = len(ctx)
    n = [c // ratio for c in ctx]
    cache = HostPaged(main_fmt, 512, [max(1, x) for x in n], seed=seed + 1)
    for b in range(B):
        cache.fill(b, rs.standard_normal((max(1, n[b]), 512)).astype(np.float32))
    swa_b, swa_dec = swa_ring(rs.standard_normal((B, 128, 512)).astype(np.float32), swa_fmt)
    q = rs.standard_normal((B, H, 512)).astype(np.float32)
    q_t, q_v = bf16_values(q)
    sink = rs.standard_normal(H).astype(np.float32) if with_sink else None
    topk = None
    if k is not None:
        topk = np.full((B, k), -1, np.int32)
        for b in range(B):
            m = min(k, n[b])
            if m == 0:
                continue
            if topk_mode == "random":
                ids = rs.choice(n[b], size=m, replace=False)
                ids[: m // 8] = ids[m // 8: 2 * (m // 8)]           # duplicates kept
                pos = rs.permutation(k)[:m]                            # -1 holes anywhere
                topk[b, pos] = ids
            else:
                topk[b, :m] = np.arange(m)
    cs = cskv.rope_table(np.asarray(ctx) - 1)
    return dict(cache=cache, swa=swa_b, swa_dec=swa_dec, q=(q_t, q_v), sink=sink, topk=topk, cs=cs,
                ctx=np.asarray(ctx, np.int32), n=n)


def _gpu(c, ratio, k, swa_fmt, max_ctx):
    dev = c["cache"].to_device()
    out = cskv.sparse_decode_attn(
        c["q"][0].cuda(), dev, cuda(c["swa"]), swa_fmt, cuda(c["ctx"]),
        None if c["topk"] is None else cuda(c["topk"]), k or 0, ratio, max_ctx,
        None if c["sink"] is None else cuda(c["sink"]), SCALE, cuda(c["cs"]))
    assert cskv.device_status() == 0
    return out.float().cpu().numpy()


def _oracle(c, b, ratio):
    return o_attn.request_attention(c["q"][1][b], int(c["ctx"][b]), ratio, c["swa_dec"][b],
                                    c["cache"].decoded[b], None if c["topk"] is None else c["topk"][b],
                                    c["sink"], SCALE)


@pytest.mark.parametrize("main_fmt,swa_fmt", [(codecs.FMT_FP8, codecs.FMT_FP8), (codecs.FMT_FP4, codecs.FMT_FP8),
                                              (codecs.FMT_BF16, codecs.FMT_BF16)])
@pytest.mark.parametrize("H,with_sink", [(64, True), (16, False), (128, True), (40, True)])
def test_csa_attention(main_fmt, swa_fmt, H, with_sink):
    ctx = [4 * 1500 + 2, 100, 4 * 513, 127, 128, 4 * 9000 + 3]
    k = 512
    c = _case(ctx, 4, k, H, main_fmt, swa_fmt, with_sink, seed=H + main_fmt)
    got = _gpu(c, 4, k, swa_fmt, max(ctx))
    for b in range(len(ctx)):
        check_attention(got[b], _oracle(c, b, 4), fp4=main_fmt == codecs.FMT_FP4)


@pytest.mark.parametrize("with_sink", [True, False])
def test_hca_attention(with_sink):
    ctx = [131072, 1000, 128 * 77 + 5, 129, 5]
    c = _case(ctx, 128, None, 64, codecs.FMT_FP8, codecs.FMT_FP8, with_sink, seed=9)
    got = _gpu(c, 128, None, codecs.FMT_FP8, max(ctx))
    for b in range(len(ctx)):
        check_attention(got[b], _oracle(c, b, 128))


def test_all_minus_one_is_window_only():
    ctx = [4 * 2000]
    c = _case(ctx, 4, 256, 64, codecs.FMT_FP8, codecs.FMT_FP8, True, seed=10)
    c["topk"][:] = -1
    got = _gpu(c, 4, 256, codecs.FMT_FP8, ctx[0])
    check_attention(got[0], _oracle(c, 0, 4))


def test_hca_128k_full_size_sampled():
    """The HCA workload at full size (batch 32, 1,024 FP8 entries + 128 window rows
    per request, 64 heads); four requests checked against the oracle."""
    wl = synth.workload("hca_128k")
    bt, num_pages = synth.page_tables(wl, "main")
    pb = 64 * 528
    dev = cskv.PagedCache(torch.zeros((num_pages, pb), dtype=torch.uint8, device="cuda"), cuda(bt),
                          codecs.FMT_FP8, 512)
    ppr = int(wl.pages_per_req()[0])
    for b in range(wl.B):
        vals = synth.request_values(wl, b, "main")
        rows = np.arange(ppr * 64, dtype=np.int32)
        cskv.encode_rows(cuda(vals), dev, req=cuda(np.full(rows.shape, b, np.int32)), row=cuda(rows))
    swa_vals = np.stack([synth.swa_values(wl, b) for b in range(wl.B)])
    swa_b, swa_dec = swa_ring(swa_vals, codecs.FMT_FP8)
    q, _, _, sink = synth.queries(wl)
    q_t, q_v = bf16_values(q)
    ctx = wl.ctx_len.astype(np.int32)
    cs = cskv.rope_table(ctx - 1)
    out = cskv.sparse_decode_attn(q_t.cuda(), dev, cuda(swa_b), codecs.FMT_FP8, cuda(ctx), None, 0,
                                  wl.ratio, wl.max_ctx, cuda(sink), SCALE, cuda(cs))
    assert cskv.device_status() == 0
    got = out.float().cpu().numpy()
    for b in (0, 7, 19, 31):
        vals = synth.request_values(wl, b, "main")
        dec = codecs.decode_rows(codecs.encode_rows(vals, codecs.FMT_FP8), codecs.FMT_FP8, 512)
        ref = o_attn.request_attention(q_v[b], int(ctx[b]), wl.ratio, swa_dec[b], dec, None, sink, SCALE)
        check_attention(got[b], ref)


def test_largest_selection_k2048():
    """k = 2048: seventeen 128-key tiles per request, merged by the combine kernel."""
    ctx = [4 * 3000 + 1, 4 * 2048, 4 * 100 + 3]
    k = 2048
    c = _case(ctx, 4, k, 64, codecs.FMT_FP8, codecs.FMT_FP8, True, seed=70)
    got = _gpu(c, 4, k, codecs.FMT_FP8, max(ctx))
    for b in range(len(ctx)):
        check_attention(got[b], _oracle(c, b, 4))
