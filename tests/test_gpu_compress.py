"""GPU parity: row coder and compressor, bit-exact against the oracle (fp32 contract + codecs)."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from compressed_sparse_attention_kv_gb300 import synth
from oracle import codecs, compress as o_comp, rope as o_rope

from cases import HostPaged, bf16_values, cuda, page_bytes_of

pytestmark = pytest.mark.gpu

FMTS = [(codecs.FMT_FP8, 512), (codecs.FMT_FP4, 512), (codecs.FMT_BF16, 512),
        (codecs.FMT_FP8_PAGESPLIT, 128), (codecs.FMT_FP8, 128), (codecs.FMT_BF16, 128),
        (codecs.FMT_FP4, 128), (codecs.FMT_FP4H_PAGESPLIT, 128)]


def _edge_rows(dim, rs):
    rows = [np.zeros(dim), -np.zeros(dim), np.full(dim, 1e-40), np.full(dim, -3e-39),
            np.full(dim, 1e30), np.full(dim, -2.5e-3)]
    # e4m3 / e2m1 rounding ties at a fixed scale: block amax 448 -> scale 1
    t = np.tile(np.array([448.0, 0.0009765625 * 3, 1.0625, 2.25, 13.0, 0.5, 0.25 * 3, 5.0]), dim // 8)
    rows.append(t)
    rows.append(-t)
    # FP4 ties: amax 6 -> scale 1, values at e2m1 midpoints
    f = np.tile(np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), dim // 8)
    rows.append(f)
    rows.append(rs.standard_normal(dim) * 1e-20)
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("fmt,dim", FMTS)
def test_encode_rows_bit_exact(fmt, dim):
    rs = np.random.default_rng(fmt * 7 + dim)
    n = 640
    x = (rs.standard_normal((n, dim)) * np.exp2(rs.integers(-30, 30, (n, 1)))).astype(np.float32)
    e = _edge_rows(dim, rs)
    x[:len(e)] = e
    pb = page_bytes_of(fmt, dim)
    dst = cskv.PagedCache(torch.zeros((n // 64, pb), dtype=torch.uint8, device="cuda"), None, fmt, dim)
    cskv.encode_rows(cuda(x), dst)
    got = dst.pool.cpu().numpy()
    if fmt == codecs.FMT_FP8_PAGESPLIT:
        want = codecs.encode_pagesplit(x)
        assert np.array_equal(got[:, :want.shape[1]], want)
    elif fmt == codecs.FMT_FP4H_PAGESPLIT:
        want = codecs.encode_fp4h_pagesplit(x)   # rotated, then coded
        bad = np.flatnonzero(np.any(got[:, :want.shape[1]] != want, axis=1))
        assert bad.size == 0, bad
    else:
        rows = codecs.encode_rows(x, fmt)
        rb = rows.shape[1]
        assert np.array_equal(got[:, :64 * rb].reshape(n, rb), rows)
    # bf16 source gives the same codes as its fp32 values
    xb, xv = bf16_values(x)
    dst2 = cskv.PagedCache(torch.zeros_like(dst.pool), None, fmt, dim)
    cskv.encode_rows(xb.cuda(), dst2)
    dst3 = cskv.PagedCache(torch.zeros_like(dst.pool), None, fmt, dim)
    cskv.encode_rows(cuda(xv), dst3)
    assert torch.equal(dst2.pool, dst3.pool)
    assert cskv.device_status() == 0


def _compress_case(ratio, overlap, dim, fmt, S=2, entries=96, seed=0):
    coff = 2 if overlap else 1
    T = ratio * entries
    rs = np.random.default_rng(seed)
    kv = rs.standard_normal((S, T, coff, dim)).astype(np.float32)
    gate = (1.5 * rs.standard_normal((S, T, coff, dim))).astype(np.float32)
    ape = (0.5 * rs.standard_normal((ratio, coff * dim))).astype(np.float32)
    nw = rs.uniform(0.5, 1.5, dim).astype(np.float32)
    prev_kv = rs.standard_normal((S, ratio, 2, dim)).astype(np.float32)
    prev_gate = rs.standard_normal((S, ratio, 2, dim)).astype(np.float32)
    kv_t, kv_v = bf16_values(kv)
    g_t, g_v = bf16_values(gate)
    pk_t, pk_v = bf16_values(prev_kv)
    pg_t, pg_v = bf16_values(prev_gate)
    first = np.array([37, 0] + [5] * (S - 2), np.int32)[:S]
    req = np.array([1, 0] + list(range(2, S)), np.int32)[:S]
    rows_per_req = [0] * S
    for s in range(S):
        rows_per_req[req[s]] = max(rows_per_req[req[s]], int(first[s]) + entries)
    cache = HostPaged(fmt, dim, rows_per_req, seed=seed + 1)
    pos = [(first[s] + np.arange(entries)) * ratio for s in range(S)]
    cs = np.stack([o_rope.table(p) for p in pos])
    return dict(T=T, kv=(kv_t, kv_v), gate=(g_t, g_v), ape=ape, nw=nw, prev=((pk_t, pk_v), (pg_t, pg_v)),
                first=first, req=req, cache=cache, cs=cs, entries=entries)


@pytest.mark.parametrize("ratio,overlap,dim,fmt,use_prev", [
    (4, 1, 512, codecs.FMT_FP8, True), (4, 1, 512, codecs.FMT_FP4, False),
    (4, 1, 512, codecs.FMT_BF16, True), (4, 1, 128, codecs.FMT_FP8_PAGESPLIT, True),
    (4, 1, 128, codecs.FMT_FP8_PAGESPLIT, False), (4, 1, 128, codecs.FMT_BF16, False),
    (4, 1, 128, codecs.FMT_FP4H_PAGESPLIT, True), (4, 1, 128, codecs.FMT_FP4H_PAGESPLIT, False),
    (128, 0, 512, codecs.FMT_FP8, False), (128, 0, 512, codecs.FMT_FP4, False),
    (4, 0, 512, codecs.FMT_FP8, False)])
def test_compress_bit_exact(ratio, overlap, dim, fmt, use_prev):
    c = _compress_case(ratio, overlap, dim, fmt, entries=96 if ratio == 4 else 5)
    cache = c["cache"]
    dev = cache.to_device()
    # the product's RoPE table helper reproduces the oracle's table bit for bit
    for s in range(2):
        assert np.array_equal(cskv.rope_table((c["first"][s] + np.arange(c["entries"])) * ratio), c["cs"][s])
    pk, pg = c["prev"]
    cskv.compress(c["kv"][0].cuda(), c["gate"][0].cuda(), cuda(c["ape"]), ratio, overlap, dev,
                  cuda(c["req"]), cuda(c["first"]),
                  prev_kv=pk[0].cuda() if use_prev and overlap else None,
                  prev_gate=pg[0].cuda() if use_prev and overlap else None,
                  norm_w=cuda(c["nw"]), eps=1e-6, rope_cs=cuda(c["cs"]))
    assert cskv.device_status() == 0
    pool = dev.pool.cpu().numpy()
    for s in range(2):
        ents = o_comp.compress_contract(
            c["kv"][1][s], c["gate"][1][s], c["ape"], ratio, bool(overlap),
            prev_kv=pk[1][s] if use_prev and overlap else None,
            prev_gate=pg[1][s] if use_prev and overlap else None,
            norm_w=c["nw"], eps=1e-6, rope_cs=c["cs"][s])
        b = int(c["req"][s])
        e0 = int(c["first"][s])
        rb = codecs.row_bytes(fmt, dim)
        for i in range(c["entries"]):
            e = e0 + i
            page = pool[cache.block_table[b, e // 64]]
            slot = e % 64
            if fmt == codecs.FMT_FP8_PAGESPLIT:
                cd, e = codecs.fp8_encode(ents[i:i + 1], block=dim)
                got_d = page[slot * dim:(slot + 1) * dim]
                got_s = page[64 * dim + slot * 4:64 * dim + (slot + 1) * 4].view(np.float32)[0]
                assert np.array_equal(got_d, cd[0]) and got_s == codecs.e8m0_decode(e[0, 0]), (s, i)
            elif fmt == codecs.FMT_FP4H_PAGESPLIT:
                cd, sb = codecs.fp4b32_encode(codecs.hadamard_contract(ents[i:i + 1]))
                got_d = page[slot * 64:(slot + 1) * 64]
                got_s = page[64 * 64 + slot * 4:64 * 64 + (slot + 1) * 4]
                assert np.array_equal(got_d, cd[0]) and np.array_equal(got_s, sb[0]), (s, i)
            else:
                want = codecs.encode_rows(ents[i:i + 1], fmt)[0]
                assert np.array_equal(page[slot * rb:(slot + 1) * rb], want), (s, i)


@pytest.mark.parametrize("ratio,fmt", [(4, codecs.FMT_FP8), (128, codecs.FMT_FP4), (4, codecs.FMT_BF16)])
def test_compressor_full_chunk_bit_exact(ratio, fmt):
    """The 65,536-token compressor workload, every byte compared."""
    overlap = ratio == 4
    T = 65536
    kv, gate = synth.compressor_tokens(3, T, ratio, overlap, 512)
    ape, nw = synth.compressor_params(3, ratio, overlap, 512)
    kv_t, kv_v = bf16_values(kv)
    g_t, g_v = bf16_values(gate)
    n = T // ratio
    cs = cskv.rope_table(np.arange(n) * ratio)
    pb = page_bytes_of(fmt, 512)
    pages = (n + 63) // 64
    dst = cskv.PagedCache(torch.zeros((pages, pb), dtype=torch.uint8, device="cuda"),
                          cuda(np.arange(pages, dtype=np.int32)[None]), fmt, 512)
    cskv.compress(kv_t[None].cuda(), g_t[None].cuda(), cuda(ape), ratio, overlap, dst,
                  cuda(np.array([0], np.int32)), cuda(np.array([0], np.int32)), norm_w=cuda(nw),
                  eps=1e-6, rope_cs=cuda(cs[None]))
    assert cskv.device_status() == 0
    ents = o_comp.compress_contract(kv_v, g_v, ape, ratio, overlap, norm_w=nw, eps=1e-6,
                                    rope_cs=o_rope.table(np.arange(n) * ratio))
    rows = codecs.encode_rows(ents, fmt)
    rb = rows.shape[1]
    got = dst.pool.cpu().numpy()[:, :64 * rb].reshape(-1, rb)[:n]
    bad = np.flatnonzero(np.any(got != rows, axis=1))
    assert bad.size == 0, "rows differ: %s" % bad[:10]


def _job(c, ratio, overlap, dev, use_prev):
    pk, pg = c["prev"]
    return dict(kv=c["kv"][0].cuda(), gate=c["gate"][0].cuda(), ape=cuda(c["ape"]), ratio=ratio,
                overlap=overlap, out=dev, req=cuda(c["req"]), first_entry=cuda(c["first"]),
                prev_kv=pk[0].cuda() if use_prev and overlap else None,
                prev_gate=pg[0].cuda() if use_prev and overlap else None,
                norm_w=cuda(c["nw"]), eps=1e-6, rope_cs=cuda(c["cs"]))


def test_compress_many_equals_separate_calls():
    """Three jobs of different widths, ratios and formats in one launch write exactly the
    bytes three separate compress calls write (the decode step compresses the main and
    the index-key entry together)."""
    specs = [(4, 1, 512, codecs.FMT_FP8, True, 96), (4, 1, 128, codecs.FMT_FP8_PAGESPLIT, False, 96),
             (128, 0, 512, codecs.FMT_FP4, False, 5), (4, 1, 128, codecs.FMT_FP4H_PAGESPLIT, True, 96)]
    cases = [_compress_case(r, o, d, f, entries=e, seed=10 + i) for i, (r, o, d, f, _, e) in enumerate(specs)]
    sep = [c["cache"].to_device() for c in cases]
    many = [c["cache"].to_device() for c in cases]
    for c, dev, (r, o, d, f, up, e) in zip(cases, sep, specs):
        j = _job(c, r, o, dev, up)
        cskv.compress(j.pop("kv"), j.pop("gate"), j.pop("ape"), j.pop("ratio"), j.pop("overlap"), j.pop("out"),
                      j.pop("req"), j.pop("first_entry"), **j)
    cskv.compress_many([_job(c, r, o, dev, up) for c, dev, (r, o, d, f, up, e) in zip(cases, many, specs)])
    assert cskv.device_status() == 0
    for a, b in zip(sep, many):
        assert torch.equal(a.pool, b.pool)
