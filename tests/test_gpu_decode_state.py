"""GPU parity: one decode step's state update (cskv_decode_append) against the oracle's
state ring, step after step: the main and index-key compressors of a CSA layer (ratio 4,
overlap), an HCA compressor (ratio 128), a CSA2 compressor (ratio 2, no slot bias) and the
128-slot window, five requests at different positions, some steps without a token."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from oracle import codecs, decode_state, rope

from cases import HostPaged, PAGE, bf16_values, cuda

pytestmark = pytest.mark.gpu

STARTS = [0, 3, 126, 1021, 65530]
STEPS = 140
SKIP = {2: range(50, 60)}     # request 2 has no token in these steps

SPECS = [  # name, ratio, overlap, dim, format, slot bias, window ring rows
    ("main", 4, 1, 512, codecs.FMT_FP8, True, 0),
    ("index", 4, 1, 128, codecs.FMT_FP8_PAGESPLIT, True, 0),
    ("hca", 128, 0, 512, codecs.FMT_FP8, True, 0),
    ("csa2", 2, 0, 512, codecs.FMT_FP4, False, 0),
    ("window", 1, 0, 512, codecs.FMT_FP8, False, 128),
    ("index_fp4", 4, 1, 128, codecs.FMT_FP4H_PAGESPLIT, True, 0),
]


def _row_bytes(pool, cache, b, row):
    pg = pool[cache.block_table[b, row // PAGE]]
    slot = row % PAGE
    if cache.fmt == codecs.FMT_FP8_PAGESPLIT:
        d = cache.dim
        return pg[slot * d:(slot + 1) * d], pg[PAGE * d + 4 * slot:PAGE * d + 4 * slot + 4]
    if cache.fmt == codecs.FMT_FP4H_PAGESPLIT:
        h = cache.dim // 2
        return pg[slot * h:(slot + 1) * h], pg[PAGE * h + 4 * slot:PAGE * h + 4 * slot + 4]
    rb = codecs.row_bytes(cache.fmt, cache.dim)
    return pg[slot * rb:(slot + 1) * rb], None


def _want_bytes(entry, fmt, dim):
    if fmt == codecs.FMT_FP8_PAGESPLIT:
        cd, e = codecs.fp8_encode(entry[None], block=dim)
        return cd[0], np.array([codecs.e8m0_decode(e[0, 0])], np.float32).view(np.uint8)
    if fmt == codecs.FMT_FP4H_PAGESPLIT:
        cd, sb = codecs.fp4b32_encode(codecs.hadamard_contract(entry[None]))
        return cd[0], sb[0]
    return codecs.encode_rows(entry[None], fmt)[0], None


def test_decode_steps_match_the_oracle():
    B = len(STARTS)
    rs = np.random.default_rng(7)
    steps_taken = [STEPS - len(SKIP.get(b, ())) for b in range(B)]
    final = [STARTS[b] + steps_taken[b] - 1 for b in range(B)]
    jobs = []
    for name, r, ov, dim, fmt, with_ape, ring in SPECS:
        coff = 2 if ov else 1
        rows = [ring] * B if ring else [max(1, (f + 1) // r) for f in final]
        host = HostPaged(fmt, dim, rows, seed=len(jobs) + 3)
        dev = host.to_device()                       # an all-zero pool with the host's block table
        ape = (0.5 * rs.standard_normal((r, coff * dim))).astype(np.float32) if with_ape else None
        nw = rs.uniform(0.5, 1.5, dim).astype(np.float32)
        jobs.append(dict(name=name, r=r, ov=ov, dim=dim, fmt=fmt, ring=ring, coff=coff, host=host, dev=dev,
                         ape=ape, nw=nw, state=cskv.decode_state(B, r, ov, dim) if r > 1 else None,
                         ostate=[decode_state.CompressorState(r, ov, dim) for _ in range(B)] if r > 1 else None,
                         want={}))
    nxt = list(STARTS)
    for t in range(STEPS):
        pos = np.array([-1 if t in SKIP.get(b, ()) else nxt[b] for b in range(B)], np.int32)
        djobs = []
        for j in jobs:
            r, dim, coff = j["r"], j["dim"], j["coff"]
            kv_t, kv_v = bf16_values(rs.standard_normal((B, coff, dim)).astype(np.float32))
            g_t, g_v = bf16_values((1.5 * rs.standard_normal((B, coff, dim))).astype(np.float32))
            wpos = np.where(pos >= 0, pos + 1 - r, 0) if r > 1 else np.maximum(pos, 0)
            djobs.append(dict(kv=kv_t.cuda(), gate=g_t.cuda() if r > 1 else None, state=j["state"], ratio=r,
                              overlap=j["ov"], out=j["dev"], ape=None if j["ape"] is None else cuda(j["ape"]),
                              norm_w=cuda(j["nw"]), eps=1e-6, ring_rows=j["ring"],
                              rope_cs=cuda(cskv.rope_table(wpos, yarn=cskv.YARN_V4))))
            ape0 = j["ape"] if j["ape"] is not None else np.zeros((r, coff * dim), np.float32)
            for b in range(B):
                p = int(pos[b])
                if p < 0:
                    continue
                if r > 1:
                    out = j["ostate"][b].push(p, kv_v[b], g_v[b], ape0, norm_w=j["nw"], yarn=rope.YARN_V4)
                    if out is not None:
                        j["want"][(b, out[0])] = out[1]
                else:
                    slot, row = decode_state.window_row(kv_v[b, 0], p, norm_w=j["nw"], yarn=rope.YARN_V4)
                    j["want"][(b, slot)] = row
        cskv.decode_append(djobs, cuda(pos))
        for b in range(B):
            if pos[b] >= 0:
                nxt[b] += 1
    assert cskv.device_status() == 0
    for j in jobs:
        pool = j["dev"].pool.cpu().numpy()
        assert j["want"], j["name"]
        for (b, row), e in sorted(j["want"].items()):
            got, got_s = _row_bytes(pool, j["host"], b, row)
            want, want_s = _want_bytes(e, j["fmt"], j["dim"])
            assert np.array_equal(got, want), (j["name"], b, row)
            if want_s is not None:
                assert np.array_equal(got_s, want_s), (j["name"], b, row)
        if j["state"] is not None:
            sk = j["state"][0].float().cpu().numpy()
            sg = j["state"][1].float().cpu().numpy()
            for b in range(B):
                assert np.array_equal(sk[b], j["ostate"][b].kv), (j["name"], b)
                assert np.array_equal(sg[b], j["ostate"][b].gate), (j["name"], b)
    # every request crossed a block boundary of every compressor, the window wrapped
    assert {b for b, _ in jobs[2]["want"]} == set(range(B))
    assert len(jobs[4]["want"]) == B * 128
