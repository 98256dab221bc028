"""GPU parity for one layer's decode step in one call (cskv_decode_layer), host memory in
and host memory out: the step's inputs copied from a pinned host buffer into a device
buffer the call's tensors view, the completed blocks' entries written to the caches
("DeepSeek-V4 deep dive", section 4.1), the indexer's top-k (section 5.2; none for HCA,
section 6.1), the attention (sections 3.4 and 5.3), and the output copied back to the
host.  The oracle recomputes every stage from the same bf16 inputs."""

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from oracle import attention as o_attn, codecs, compress as o_comp, indexer, rope as o_rope

from cases import check_topk_fp4, HostPaged, bf16_values, check_attention, check_topk, cuda, swa_ring

pytestmark = pytest.mark.gpu

SCALE = 512 ** -0.5


def _stage(items, pinned=True):
    """Host tensors packed into one host buffer (256-byte aligned parts; page-locked unless
    pinned is False) and an uninitialised device buffer of the same size; returns
    (h_in, d_in, device views)."""
    offs, tot = [], 0
    for t in items.values():
        offs.append(tot)
        tot = (tot + t.numel() * t.element_size() + 255) // 256 * 256
    h = torch.empty(tot, dtype=torch.uint8, pin_memory=pinned)
    d = torch.empty(tot, dtype=torch.uint8, device="cuda")
    views = {}
    for (name, t), o in zip(items.items(), offs):
        nb = t.numel() * t.element_size()
        h[o:o + nb].view(t.dtype).view(t.shape).copy_(t)
        views[name] = d[o:o + nb].view(t.dtype).view(t.shape)
    return h, d, views


def _block_inputs(rs, B, ratio, overlap, dim):
    """bf16 tokens of each request's completed block (and, with overlap, the block before)."""
    coff = 2 if overlap else 1
    kv = bf16_values(rs.standard_normal((B, ratio, coff, dim)).astype(np.float32))
    gate = bf16_values((1.5 * rs.standard_normal((B, ratio, coff, dim))).astype(np.float32))
    prev = None
    if overlap:
        prev = (bf16_values(rs.standard_normal((B, ratio, 2, dim)).astype(np.float32)),
                bf16_values(rs.standard_normal((B, ratio, 2, dim)).astype(np.float32)))
    ape = (0.5 * rs.standard_normal((ratio, coff * dim))).astype(np.float32)
    nw = rs.uniform(0.5, 1.5, dim).astype(np.float32)
    return dict(kv=kv, gate=gate, prev=prev, ape=ape, nw=nw, overlap=overlap)


def _oracle_entry(blk, b, ratio, e):
    """The oracle's entry e of request b from its completed block (fp32 contract)."""
    prev = blk["prev"]
    return o_comp.compress_contract(blk["kv"][1][b], blk["gate"][1][b], blk["ape"], ratio, blk["overlap"],
                                    prev_kv=prev[0][1][b] if prev else None,
                                    prev_gate=prev[1][1][b] if prev else None,
                                    norm_w=blk["nw"], eps=1e-6, rope_cs=o_rope.table([e * ratio]))[0]


def _caches(rs, fmt, dim, n, seed):
    """Device cache holding every entry but each request's last (zero there: this step
    writes it) and the oracle's host copy; returns (host, device, values)."""
    host = HostPaged(fmt, dim, n, seed=seed)
    vals = []
    for b, nb in enumerate(n):
        v = rs.standard_normal((nb, dim)).astype(np.float32)
        v[nb - 1] = 0.0
        host.fill(b, v)
        vals.append(v)
    return host, host.to_device(), vals


@pytest.mark.parametrize("main_fmt,key_fmt", [(codecs.FMT_FP8, codecs.FMT_FP8_PAGESPLIT),
                                               (codecs.FMT_FP4, codecs.FMT_FP8_PAGESPLIT),
                                               (codecs.FMT_FP8, codecs.FMT_FP4H_PAGESPLIT)])
def test_csa_layer_step_host_to_host(main_fmt, key_fmt):
    rs = np.random.default_rng(61 + main_fmt)
    ratio, k, H, Hi = 4, 512, 64, 64
    n = [300, 1029, 64]                       # entries after this step (the last one is new)
    B = len(n)
    ctx = np.array([ratio * x for x in n], np.int32)
    max_ctx = int(ctx.max())
    host_main, dev_main, main_vals = _caches(rs, main_fmt, 512, n, seed=11)
    host_idx, dev_idx, idx_vals = _caches(rs, key_fmt, 128, n, seed=12)
    blk_m = _block_inputs(rs, B, ratio, True, 512)
    blk_i = _block_inputs(rs, B, ratio, True, 128)
    q_t, q_v = bf16_values(rs.standard_normal((B, H, 512)).astype(np.float32))
    qi_t, qi_v = bf16_values(rs.standard_normal((B, Hi, 128)).astype(np.float32))
    w = rs.uniform(0, 1, (B, Hi)).astype(np.float32)
    sink = rs.standard_normal(H).astype(np.float32)
    swa_b, swa_dec = swa_ring(rs.standard_normal((B, 128, 512)).astype(np.float32), codecs.FMT_FP8)
    first = np.array([x - 1 for x in n], np.int32)
    h_in, d_in, v = _stage({
        "kv": blk_m["kv"][0], "gate": blk_m["gate"][0], "pkv": blk_m["prev"][0][0], "pgate": blk_m["prev"][1][0],
        "ikv": blk_i["kv"][0], "igate": blk_i["gate"][0], "ipkv": blk_i["prev"][0][0],
        "ipgate": blk_i["prev"][1][0], "q": q_t, "q_idx": qi_t, "w": torch.from_numpy(w),
        "ctx": torch.from_numpy(ctx), "first": torch.from_numpy(first),
        "req": torch.arange(B, dtype=torch.int32),
        "ecs": torch.from_numpy(cskv.rope_table(first[:, None] * ratio)),
        "qcs": torch.from_numpy(cskv.rope_table(ctx - 1))})
    jobs = [dict(kv=v["kv"], gate=v["gate"], ape=cuda(blk_m["ape"]), ratio=ratio, overlap=True, out=dev_main,
                 req=v["req"], first_entry=v["first"], prev_kv=v["pkv"], prev_gate=v["pgate"],
                 norm_w=cuda(blk_m["nw"]), rope_cs=v["ecs"]),
            dict(kv=v["ikv"], gate=v["igate"], ape=cuda(blk_i["ape"]), ratio=ratio, overlap=True, out=dev_idx,
                 req=v["req"], first_entry=v["first"], prev_kv=v["ipkv"], prev_gate=v["ipgate"],
                 norm_w=cuda(blk_i["nw"]), rope_cs=v["ecs"])]
    h_out = torch.empty((B, H, 512), dtype=torch.bfloat16, pin_memory=True)
    pools0 = dev_main.pool.clone(), dev_idx.pool.clone()   # before the step writes its entries
    out, topk = cskv.decode_layer(jobs, v["q_idx"], v["w"], dev_idx, v["q"], dev_main, cuda(swa_b), codecs.FMT_FP8,
                                  v["ctx"], k, ratio, max_ctx, cuda(sink), SCALE, v["qcs"],
                                  h_in=h_in, d_in=d_in, h_out=h_out)
    torch.cuda.synchronize()
    assert cskv.device_status() == 0
    assert torch.equal(h_out, out.cpu())
    # the same step with the attention queries and the compressor's per-step inputs left
    # in pinned host memory (read in place): the same selection and the same output bits
    # (the step's compressor writes the same entries again; the caches are checked below)
    q_pin = q_t.clone().pin_memory()
    pin = {kk: v[kk].cpu().pin_memory() for kk in ("kv", "gate", "pkv", "pgate", "ikv", "igate", "ipkv", "ipgate",
                                                    "ecs")}
    jobs_pin = [dict(j, kv=pin[a], gate=pin[g], prev_kv=pin[pa], prev_gate=pin[pg], rope_cs=pin["ecs"])
                for j, (a, g, pa, pg) in zip(jobs, (("kv", "gate", "pkv", "pgate"), ("ikv", "igate", "ipkv", "ipgate")))]
    h_out2 = torch.empty((B, H, 512), dtype=torch.bfloat16, pin_memory=True)
    dev_main.pool.copy_(pools0[0])   # the step's entries must be written again
    dev_idx.pool.copy_(pools0[1])
    _, topk2 = cskv.decode_layer(jobs_pin, v["q_idx"], v["w"], dev_idx, q_pin, dev_main, cuda(swa_b), codecs.FMT_FP8,
                                 v["ctx"], k, ratio, max_ctx, cuda(sink), SCALE, v["qcs"],
                                 h_in=h_in, d_in=d_in, h_out=h_out2)
    torch.cuda.synchronize()
    assert cskv.device_status() == 0
    assert torch.equal(topk2, topk)
    assert torch.equal(h_out2, h_out)
    # the caches now hold the oracle's entries, bit for bit
    for b in range(B):
        main_vals[b][n[b] - 1] = _oracle_entry(blk_m, b, ratio, n[b] - 1)
        idx_vals[b][n[b] - 1] = _oracle_entry(blk_i, b, ratio, n[b] - 1)
        host_main.fill(b, main_vals[b])
        host_idx.fill(b, idx_vals[b])
    assert np.array_equal(dev_main.pool.cpu().numpy(), host_main.pool)
    assert np.array_equal(dev_idx.pool.cpu().numpy(), host_idx.pool)
    topk = topk.cpu().numpy()
    got = h_out.float().numpy()
    for b in range(B):
        if key_fmt == codecs.FMT_FP4H_PAGESPLIT:
            assert check_topk_fp4(topk[b], None, qi_v[b], w[b], host_idx.decoded[b], n[b], k) == 0, b
            sel = indexer.index_topk_fp4(qi_v[b], w[b], host_idx.decoded[b], int(ctx[b]), ratio, k)[0]
        else:
            q_hat = indexer.quantize_queries(qi_v[b])
            assert check_topk(topk[b], None, q_hat, w[b], host_idx.decoded[b], n[b], k) == 0, b
            sel = indexer.select_topk(indexer.scores_fp64(q_hat, w[b], host_idx.decoded[b]), k)
        ref = o_attn.request_attention(q_v[b], int(ctx[b]), ratio, swa_dec[b], host_main.decoded[b], sel, sink,
                                       SCALE)
        check_attention(got[b], ref, fp4=main_fmt == codecs.FMT_FP4)


@pytest.mark.parametrize("pinned", [True, False])
def test_hca_layer_steps_with_and_without_a_completed_block(pinned):
    """HCA (ratio 128, no indexer): a step that completes each request's last entry, then
    a step five tokens later that completes none (no compressor job), which copies back
    only the first request's output.  Page-locked host buffers are read by the library's
    copy kernel and a whole page-locked output is written by the attention's last kernel
    (a part of one by the copy kernel); pageable buffers go through the copy engine."""
    rs = np.random.default_rng(67)
    ratio, H = 128, 16
    n = [9, 3]
    B = len(n)
    host_main, dev_main, main_vals = _caches(rs, codecs.FMT_FP8, 512, n, seed=13)
    blk = _block_inputs(rs, B, ratio, False, 512)
    sink = rs.standard_normal(H).astype(np.float32)
    swa_b, swa_dec = swa_ring(rs.standard_normal((B, 128, 512)).astype(np.float32), codecs.FMT_FP8)
    first = np.array([x - 1 for x in n], np.int32)
    for b in range(B):
        main_vals[b][n[b] - 1] = _oracle_entry(blk, b, ratio, n[b] - 1)
        host_main.fill(b, main_vals[b])
    for extra, with_job in ((0, True), (5, False)):
        ctx = np.array([ratio * x + extra for x in n], np.int32)
        q_t, q_v = bf16_values(rs.standard_normal((B, H, 512)).astype(np.float32))
        items = {"q": q_t, "ctx": torch.from_numpy(ctx), "qcs": torch.from_numpy(cskv.rope_table(ctx - 1))}
        if with_job:
            items.update({"kv": blk["kv"][0], "gate": blk["gate"][0], "first": torch.from_numpy(first),
                          "req": torch.arange(B, dtype=torch.int32),
                          "ecs": torch.from_numpy(cskv.rope_table(first[:, None] * ratio))})
        h_in, d_in, v = _stage(items, pinned)
        jobs = []
        if with_job:
            jobs = [dict(kv=v["kv"], gate=v["gate"], ape=cuda(blk["ape"]), ratio=ratio, overlap=False,
                         out=dev_main, req=v["req"], first_entry=v["first"], norm_w=cuda(blk["nw"]),
                         rope_cs=v["ecs"])]
        nout = B if with_job else 1
        h_out = torch.empty((nout, H, 512), dtype=torch.bfloat16, pin_memory=pinned)
        out, topk = cskv.decode_layer(jobs, None, None, None, v["q"], dev_main, cuda(swa_b), codecs.FMT_FP8,
                                      v["ctx"], 0, ratio, int(ctx.max()), cuda(sink), SCALE, v["qcs"],
                                      h_in=h_in, d_in=d_in, h_out=h_out)
        torch.cuda.synchronize()
        assert cskv.device_status() == 0
        assert topk is None
        assert np.array_equal(dev_main.pool.cpu().numpy(), host_main.pool)
        assert torch.equal(h_out, out[:nout].cpu())
        got = h_out.float().numpy()
        for b in range(nout):
            ref = o_attn.request_attention(q_v[b], int(ctx[b]), ratio, swa_dec[b], host_main.decoded[b], None,
                                           sink, SCALE)
            check_attention(got[b], ref)


def test_captured_layer_step_reads_the_host_buffers_at_every_replay():
    """The call captured once into a CUDA graph (as a serving loop, or the benchmark, runs
    it): each replay copies the host buffer's current contents in and writes the current
    output back, so new queries written into the same pinned buffer give new results."""
    rs = np.random.default_rng(73)
    ratio, H = 128, 16
    n = [6, 2, 4]
    B = len(n)
    host_main, dev_main, _ = _caches(rs, codecs.FMT_FP8, 512, n, seed=14)
    sink = rs.standard_normal(H).astype(np.float32)
    swa_b, swa_dec = swa_ring(rs.standard_normal((B, 128, 512)).astype(np.float32), codecs.FMT_FP8)
    ctx = np.array([ratio * x + 7 for x in n], np.int32)           # no block completes: no compressor job
    q0_t, _ = bf16_values(rs.standard_normal((B, H, 512)).astype(np.float32))
    h_in, d_in, v = _stage({"q": q0_t, "ctx": torch.from_numpy(ctx),
                            "qcs": torch.from_numpy(cskv.rope_table(ctx - 1))})
    h_out = torch.empty((B, H, 512), dtype=torch.bfloat16, pin_memory=True)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cskv.sparse_decode_attn_workspace_size(B, H, int(ctx.max()), ratio, 0), dtype=torch.uint8,
                     device="cuda")

    swa_d, sink_d = cuda(swa_b), cuda(sink)   # device copies made before the capture

    def call():
        cskv.decode_layer([], None, None, None, v["q"], dev_main, swa_d, codecs.FMT_FP8, v["ctx"], 0, ratio,
                          int(ctx.max()), sink_d, SCALE, v["qcs"], out=out, attn_workspace=ws,
                          h_in=h_in, d_in=d_in, h_out=h_out)

    call()                                        # outside the capture first
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    torch.cuda.synchronize()
    q_view = h_in[:q0_t.numel() * 2].view(torch.bfloat16).view(q0_t.shape)   # "q" is the first part
    for rep in range(3):
        q_t, q_v = bf16_values(rs.standard_normal((B, H, 512)).astype(np.float32))
        q_view.copy_(q_t)
        h_out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert cskv.device_status() == 0
        got = h_out.float().numpy()
        for b in range(B):
            ref = o_attn.request_attention(q_v[b], int(ctx[b]), ratio, swa_dec[b], host_main.decoded[b], None,
                                           sink, SCALE)
            check_attention(got[b], ref)
