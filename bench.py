#!/usr/bin/env python
"""Decode-attention benchmark: queries/s per layer at 1M context on one GB300.

One step = one decode token through one CSA layer for a batch of 8 requests at
1,048,576 tokens (262,144 compressed entries each), i.e. every row of the hot path,
run by one cskv_decode_layer call (device buffers; the kernels overlap):
  1. compress the block that the new token completes (main 512-d entry -> FP8-528,
     index 128-d key -> FP8-132),
  2. index_topk: score all 262,144 FP8 keys per request with 64 indexer heads, keep 512,
  3. sparse_decode_attn: 64 heads over 128 window rows + 512 selected FP8 entries,
     one softmax with the sink, inverse RoPE.
Caches are resident in HBM before timing; the L2 is flushed (512 MB write) between
timed steps, outside the timed region.  Inputs are seeded synthetic data.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl cskv|reference]

--impl reference times the CPU oracle (the test oracle, not tuned) on the same workload,
one query per step.  Under torchrun each rank runs an independent replica (the path
shards by request; no collective); rank 0 prints one JSON line.
"""

import argparse
import concurrent.futures
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from compressed_sparse_attention_kv_gb300 import synth  # noqa: E402

METRIC = "decode attn queries/s per layer at 1M ctx; KV-read GB/s and % of HBM/FP8 roofline"
MIXED_METRIC = "mixed-batch MXFP4 CSA decode: queries/s per layer (batch 64, contexts 32K-512K)"
FP4_METRIC = "decode attn queries/s per layer at 1M ctx with FP4 index keys (68 B, BF16 scores)"
WORKLOAD = "csa_1m"
L2_FLUSH_BYTES = 512 << 20


def workload_desc(wl):
    if wl.name == "mixed_mxfp4":
        return ("Mixed-batch MXFP4 CSA decode: batch %d, contexts %d..%d tokens (U{32768..524288}, seed 4; "
                "%d entries in all) at ratio %d, paged 64-row blocks shuffled in a pool, indexer %d heads x 128 "
                "FP8 keys (132 B), top-%d, %d query heads x 512 over MXFP4-288 entries (E2M1 + E4M3 per 16) + "
                "FP8 window 128, sink; per step: compress the completed block (main + index key), index_topk, "
                "sparse_decode_attn" % (wl.B, int(wl.ctx_len.min()), int(wl.ctx_len.max()),
                                        int(wl.n_entries.sum()), wl.ratio, wl.Hi, wl.k, wl.H))
    keys = ("FP4 keys (68 B: Hadamard-rotated e2m1 + e8m0 per 32, BF16 scores)"
            if wl.key_fmt == synth.FMT_FP4H_PAGESPLIT else "FP8 keys (132 B)")
    return (("CSA decode at 1M context: batch %d, %d tokens -> %d entries at ratio %d, indexer %d heads "
             "x 128 " + keys + " w~U(0,1), top-%d, %d query heads x 512 over FP8-528 entries "
            "+ FP8 window 128, sink; per step: compress the completed block (main + index key), "
            "index_topk, sparse_decode_attn") % (wl.B, int(wl.ctx_len[0]), int(wl.n_entries[0]), wl.ratio,
                                                wl.Hi, wl.k, wl.H))


def step_inputs(wl):
    """Per-step inputs (host arrays): queries and the completed block for both compressors."""
    q, q_idx, w, sink = synth.queries(wl)
    kv, gate, pkv, pgate, ikv, igate, ipkv, ipgate = ([] for _ in range(8))
    for b in range(wl.B):
        a, g = synth.compressor_tokens(wl.seed, wl.ratio, wl.ratio, True, 512, seq=b)
        pa, pg = synth.compressor_prev(wl.seed, wl.ratio, 512, seq=b)
        ia, ig = synth.compressor_tokens(wl.seed, wl.ratio, wl.ratio, True, 128, index_lane=True, seq=b)
        ipa, ipg = synth.compressor_prev(wl.seed, wl.ratio, 128, index_lane=True, seq=b)
        kv.append(a); gate.append(g); pkv.append(pa); pgate.append(pg)
        ikv.append(ia); igate.append(ig); ipkv.append(ipa); ipgate.append(ipg)
    ape, nw = synth.compressor_params(wl.seed, wl.ratio, True, 512)
    iape, inw = synth.compressor_params(wl.seed, wl.ratio, True, 128, index_lane=True)
    st = lambda x: np.ascontiguousarray(np.stack(x))  # noqa: E731
    return dict(q=q, q_idx=q_idx, w=w, sink=sink, kv=st(kv), gate=st(gate), pkv=st(pkv), pgate=st(pgate),
                ikv=st(ikv), igate=st(igate), ipkv=st(ipkv), ipgate=st(ipgate), ape=ape, nw=nw, iape=iape,
                inw=inw)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 50 ms; stop() keeps those taken between mark("t0") and
    mark("t1") (the timed region), or all of them if the region was too short to hold one."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        self.gpu_id = gpu_id
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 9]

        def when(r):
            try:
                return datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None and when(r) is not None
                  and self.t0 <= when(r) <= self.t1]
        window = "timed region" if inside else "around the timed region"
        rows = inside or rows
        sm = [float(r[2].split()[0]) for r in rows if r[2].split()[0].replace(".", "").isdigit()]
        mx = [float(r[3].split()[0]) for r in rows if r[3].split()[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].strip().lower() == "active"})
        loaded = [s for s in sm if mx and s >= 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "window": window}


# ----------------------------------------------------------------------------- GPU arm

def live_events(torch):
    """Two timing events whose CUDA handles exist (torch creates them on first record)."""
    evs = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    return evs


def gen_parallel(fn, items, threads=16):
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def build_caches(wl, torch, cskv):
    """Resident caches: index keys and main entries (the workload's formats), window ring (FP8-528)."""
    dev = "cuda"
    bt_i, np_i = synth.page_tables(wl, "index")
    bt_m, np_m = synth.page_tables(wl, "main")
    krb = cskv.row_bytes(wl.key_fmt, 128)
    keys = cskv.PagedCache(torch.zeros((np_i, (64 * krb + 15) // 16 * 16), dtype=torch.uint8, device=dev),
                           torch.from_numpy(bt_i).to(dev), wl.key_fmt, 128)
    mrb = cskv.row_bytes(wl.main_fmt, 512)
    main = cskv.PagedCache(torch.zeros((np_m, (64 * mrb + 15) // 16 * 16), dtype=torch.uint8, device=dev),
                           torch.from_numpy(bt_m).to(dev), wl.main_fmt, 512)
    pprs = wl.pages_per_req()
    for lane, cache, dim in (("index", keys, 128), ("main", main, 512)):
        f = synth.index_page_values if lane == "index" else synth.main_page_values
        for b in range(wl.B):
            ppr = int(pprs[b])
            rows = torch.arange(ppr * 64, dtype=torch.int32, device=dev)
            pages = gen_parallel(lambda p: f(wl, b, p), range(ppr))
            vals = torch.from_numpy(np.concatenate(pages)).to(dev)
            cskv.encode_rows(vals, cache, req=torch.full_like(rows, b), row=rows)
            del vals
    swa_vals = torch.from_numpy(np.stack([synth.swa_values(wl, b) for b in range(wl.B)])).to(dev)
    swa = torch.zeros((wl.B, 128, 528), dtype=torch.uint8, device=dev)
    swa_c = cskv.PagedCache(swa.view(wl.B * 2, 64 * 528), None, cskv.FMT_FP8, 512)
    cskv.encode_rows(swa_vals.reshape(-1, 512), swa_c)
    torch.cuda.synchronize()
    return keys, main, swa


def max_over_ranks(values, world, device="cpu"):
    """Per-rank timings -> their maxima over the ranks (every rank gets them); the job's
    time is the slowest replica's."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world, per_rank_batch, ms):
    """Whole-job queries/s: every replica processes its batch in the (slowest) step time."""
    return world * per_rank_batch / (ms * 1e-3)


def run_gpu(args, rank, world, workload=WORKLOAD):
    import torch
    import compressed_sparse_attention_kv_gb300 as cskv
    from compressed_sparse_attention_kv_gb300 import _lib

    _lib.lib()
    dev = "cuda"
    wl = synth.workload(workload)
    B, H, Hi, k, r = wl.B, wl.H, wl.Hi, wl.k, wl.ratio
    L = wl.max_ctx
    n_b = wl.n_entries.astype(np.int64)
    t_setup = time.time()
    keys, main, swa = build_caches(wl, torch, cskv)
    inp = step_inputs(wl)

    # ---- static device buffers (graph-capture safe) and pinned host copies of the step inputs
    bf = torch.bfloat16
    host = {
        "q_idx": torch.from_numpy(inp["q_idx"]).to(bf), "w": torch.from_numpy(inp["w"]),
        "qcs": torch.from_numpy(cskv.rope_table(wl.ctx_len - 1)),
        "ctx": torch.from_numpy(wl.ctx_len.astype(np.int32)),
        "first": torch.from_numpy((n_b - 1).astype(np.int32)),
        "q": torch.from_numpy(inp["q"]).to(bf),
        # from here on the compressor's per-step inputs, which the end-to-end leg leaves in place
        "kv": torch.from_numpy(inp["kv"]).to(bf),
        "gate": torch.from_numpy(inp["gate"]).to(bf), "pkv": torch.from_numpy(inp["pkv"]).to(bf),
        "pgate": torch.from_numpy(inp["pgate"]).to(bf), "ikv": torch.from_numpy(inp["ikv"]).to(bf),
        "igate": torch.from_numpy(inp["igate"]).to(bf), "ipkv": torch.from_numpy(inp["ipkv"]).to(bf),
        "ipgate": torch.from_numpy(inp["ipgate"]).to(bf),
        "ecs": torch.from_numpy(cskv.rope_table(((n_b - 1) * r)[:, None])),
    }
    # the step's inputs live in one pinned host buffer and one device buffer (views at
    # 256-byte offsets), so that the end-to-end leg moves them with a single copy of a
    # prefix; what follows the prefix it leaves in place: the compressor's inputs (read
    # by the compressor, which runs beside the score kernel) and, when the batch's
    # attention tiles all fit on the GPU, the attention queries (read before each tile
    # waits for its selection)
    offs, tot = {}, 0
    for kk, v in host.items():
        offs[kk] = tot
        tot = (tot + v.numel() * v.element_size() + 255) // 256 * 256
    host_buf = torch.empty(tot, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(tot, dtype=torch.uint8, device=dev)

    def view(buf, kk, like):
        nb = like.numel() * like.element_size()
        return buf[offs[kk]:offs[kk] + nb].view(like.dtype).view(like.shape)

    for kk, v in host.items():
        view(host_buf, kk, v).copy_(v.contiguous())
    d = {kk: view(dev_buf, kk, v) for kk, v in host.items()}
    dev_buf.copy_(host_buf)
    req = torch.arange(B, dtype=torch.int32, device=dev)
    ape, nw = torch.from_numpy(inp["ape"]).to(dev), torch.from_numpy(inp["nw"]).to(dev)
    iape, inw = torch.from_numpy(inp["iape"]).to(dev), torch.from_numpy(inp["inw"]).to(dev)
    sink = torch.from_numpy(inp["sink"]).to(dev)
    topk = torch.empty((B, k), dtype=torch.int32, device=dev)
    out = torch.empty((B, H, 512), dtype=bf, device=dev)
    ws_i = torch.empty(cskv.index_topk_workspace_size(B, L, r, Hi, k), dtype=torch.uint8, device=dev)
    ws_a = torch.empty(cskv.sparse_decode_attn_workspace_size(B, H, L, r, k), dtype=torch.uint8, device=dev)
    out_host = torch.empty_like(out, device="cpu").pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # the completed block's entry of both caches (main, index keys), one launch
    jobs = [dict(kv=d["kv"], gate=d["gate"], ape=ape, ratio=r, overlap=True, out=main, req=req,
                 first_entry=d["first"], prev_kv=d["pkv"], prev_gate=d["pgate"], norm_w=nw, rope_cs=d["ecs"]),
            dict(kv=d["ikv"], gate=d["igate"], ape=iape, ratio=r, overlap=True, out=keys, req=req,
                 first_entry=d["first"], prev_kv=d["ipkv"], prev_gate=d["ipgate"], norm_w=inw,
                 rope_cs=d["ecs"])]

    def step():
        # one cskv_decode_layer call without host buffers: the indexer's query prep, the
        # compressor (both caches), the score kernel (selection included), attention tiles, combine
        cskv.decode_layer(jobs, d["q_idx"], d["w"], keys, d["q"], main, swa, wl.swa_fmt, d["ctx"], k, r, L, sink,
                          cskv.DEFAULT_SCALE, d["qcs"], topk_idx=topk, out=out, index_workspace=ws_i,
                          attn_workspace=ws_a)

    launches_per_step = 1 + 2 + 2   # query prep, compressor, score/select, attention tiles, combine
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = cskv.device_status()
    if status != 0:
        raise RuntimeError("device status %d after warm-up" % status)

    graph = None
    if not args.no_graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        ev_sb, ev_se = live_events(torch)
        graph = torch.cuda.CUDAGraph()
        # armed outside the capture (it creates the library's timing branch stream),
        # turned off inside it (that joins the branch into the captured step)
        cskv.set_timing_events(ev_sb, ev_se)
        with torch.cuda.graph(graph):
            step()
            cskv.set_timing_events(None, None)
    setup_s = time.time() - t_setup

    def run_once():
        if graph is not None:
            graph.replay()
        else:
            step()

    for _ in range(args.warmup):
        flush.zero_()
        run_once()
    torch.cuda.synchronize()

    # ---- timed region: K steps, L2 flushed before each (outside the events)
    clk = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
    clk.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    score_ms = []
    if graph is None:
        ev_sb, ev_se = live_events(torch)
        cskv.set_timing_events(ev_sb, ev_se)
    wall0 = time.time()
    clk.mark("t0")
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record()
        run_once()
        evs[i][1].record()
        evs[i][1].synchronize()
        ev_se.synchronize()
        score_ms.append(ev_sb.elapsed_time(ev_se))
    torch.cuda.synchronize()
    clk.mark("t1")
    wall = time.time() - wall0
    if world > 1:
        torch.distributed.barrier()
    cskv.set_timing_events(None, None)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    clocks = clk.stop()
    status = cskv.device_status()
    if status != 0:
        raise RuntimeError("device status %d after timing" % status)

    # ---- end to end through the C ABI with host buffers: one cskv_decode_layer call copies
    # the step's inputs in (one pinned buffer), runs the step's five kernels and copies the
    # output out; captured once into a CUDA graph like the device-resident step
    e2e_ms = []
    h2d = tot
    d2h = out.numel() * out.element_size()

    # The attention queries stay in pinned memory (read in place by the attention, before
    # each tile waits for its selection) when the batch's attention tiles all fit on the
    # GPU at once; a larger batch's later tiles would wait on the host link, so its
    # queries are copied in with the rest.
    tiles = 1 + (k + 127) // 128
    q_in_place = B * tiles * ((wl.H + 31) // 32) <= torch.cuda.get_device_properties(dev).multi_processor_count
    h_in = host_buf[:offs["q"]] if q_in_place else host_buf[:offs["kv"]]
    q_arg = view(host_buf, "q", host["q"]) if q_in_place else d["q"]
    hv = {kk: view(host_buf, kk, host[kk]) for kk in ("kv", "gate", "pkv", "pgate", "ikv", "igate", "ipkv", "ipgate",
                                                      "ecs")}
    jobs_e2e = [dict(jobs[0], kv=hv["kv"], gate=hv["gate"], prev_kv=hv["pkv"], prev_gate=hv["pgate"], rope_cs=hv["ecs"]),
                dict(jobs[1], kv=hv["ikv"], gate=hv["igate"], prev_kv=hv["ipkv"], prev_gate=hv["ipgate"],
                     rope_cs=hv["ecs"])]

    def layer_call():
        cskv.decode_layer(jobs_e2e, d["q_idx"], d["w"], keys, q_arg, main, swa, wl.swa_fmt, d["ctx"], k, r, L, sink,
                          cskv.DEFAULT_SCALE, d["qcs"], topk_idx=topk, out=out, index_workspace=ws_i,
                          attn_workspace=ws_a, h_in=h_in, d_in=dev_buf, h_out=out_host)

    layer_call()
    torch.cuda.synchronize()
    e2e_run = layer_call
    if not args.no_graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer_call()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            layer_call()
        e2e_run = g_e2e.replay
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        e2e_run()
        e1.record()
        e1.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    status = cskv.device_status()
    if status != 0:
        raise RuntimeError("device status %d after the end-to-end leg" % status)

    mean_ms, e2e_mean = max_over_ranks([statistics.mean(step_ms), statistics.mean(e2e_ms)], world, dev)

    # ---- roofline of the dominant kernel (the indexer score pass): bytes it must read
    fp4_keys = wl.key_fmt == synth.FMT_FP4H_PAGESPLIT
    algo_bytes = cskv.row_bytes(wl.key_fmt, 128) * int(wl.n_entries.sum())
    score_mean = statistics.mean(score_ms)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    achieved = algo_bytes / (score_mean * 1e-3) / 1e9
    traffic = profiled_traffic() if workload == WORKLOAD else None   # the capture is of the csa_1m launch
    path_bytes = algo_bytes + B * (512 * cskv.row_bytes(wl.main_fmt, 512) + 128 * 528 + 2 * H * 512 * 2
                                   + Hi * 128 * 2)

    res = {
        "metric": METRIC if workload == WORKLOAD else (FP4_METRIC if fp4_keys else MIXED_METRIC),
        "value": job_throughput(world, B, mean_ms),
        "unit": "queries/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": mean_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e2m1 block-scaled (indexer MMA)" if fp4_keys else "e4m3 (indexer MMA)")
                 + " + bf16 (attention MMA), fp32 accumulate",
        "data": "synthetic (seeded N(0,1) caches and queries, U(0,1) head weights)",
        "config": {"workload": workload_desc(wl), "batch_per_gpu": B, "context": L,
                   "l2": "flushed before every timed step (512 MB write, outside the timed region); "
                         "inputs (%d MB of index keys) also exceed L2" % (algo_bytes // 1000000),
                   "timing": "CUDA events per step around a CUDA-graph replay" if graph else "CUDA events per step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"kernel": ("index_score_kernel (FP4 keys, tcgen05 kind::mxf4 block-scaled MMA)" if fp4_keys
                                else "index_score_kernel (FP8 keys, tcgen05 e4m3 MMA)"), "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
                     "algorithmic_bytes_per_launch": algo_bytes, "ms_per_launch": score_mean,
                     "traffic": traffic},
        "kv_read_gbs": path_bytes / (mean_ms * 1e-3) / 1e9,
        "step_frac_of_hbm_roofline": (path_bytes / (peak * 1e9)) / (mean_ms * 1e-3),
        "e2e": {"value": job_throughput(world, B, e2e_mean), "unit": "queries/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "call": "cskv_decode_layer (pinned host buffers in and out; the compressor's "
                "inputs%s read in place from pinned memory)" % (" and the attention queries" if q_in_place else ""),
                "ms_per_step": e2e_mean},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
        "setup_s": setup_s,
    }
    return res


def profiled_traffic():
    """DRAM bytes per score-kernel launch from the committed ncu summary, if the kernel
    source is unchanged since that capture (else None)."""
    src = os.path.join(ROOT, "compressed_sparse_attention_kv_gb300", "csrc", "index_topk.cu")
    summ = os.path.join(ROOT, "profiles", "index_score_csa_1m.json")
    try:
        with open(src, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
        with open(summ) as f:
            p = json.load(f)
    except OSError:
        return None
    if p.get("source_sha256_16") != h:
        return None
    return p.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- oracle arm

class OracleRunner:
    """The CPU oracle on the same workload: one query (one request) per step, from the coded bytes."""

    def __init__(self, wl, requests):
        from oracle import codecs
        self.wl = wl
        self.inp = step_inputs(wl)
        self.req = list(requests)
        self.keys, self.main_pages, self.swa = {}, {}, {}
        self.fp4 = wl.key_fmt == codecs.FMT_FP4H_PAGESPLIT
        for b in self.req:
            vals = synth.request_values(wl, b, "index")
            self.keys[b] = codecs.encode_fp4h_pagesplit(vals) if self.fp4 else codecs.encode_pagesplit(vals)
            self.swa[b] = codecs.encode_rows(synth.swa_values(wl, b), wl.swa_fmt)
            # cache preparation (untimed): code the main pages this request's selection reads
            ent, ik = self._compress(b)
            top = self._topk(b, ik)
            pages = sorted(set(int(j) // 64 for j in top if j >= 0))
            self.main_pages[b] = {p: codecs.encode_rows(synth.main_page_values(wl, b, p), wl.main_fmt)
                                  for p in pages}

    @staticmethod
    def _bf(x):
        from oracle import codecs
        return codecs.bf16_decode(codecs.bf16_encode(x)).astype(np.float32)

    def _compress(self, b):
        """The completed block's main entry and index key (fp32 contract)."""
        from oracle import compress, rope
        wl, inp, bf = self.wl, self.inp, self._bf
        r = wl.ratio
        n = int(wl.n_entries[b])
        cs = rope.table(np.array([(n - 1) * r]))
        ent = compress.compress_contract(bf(inp["kv"][b]), bf(inp["gate"][b]), inp["ape"], r, True,
                                         prev_kv=bf(inp["pkv"][b]), prev_gate=bf(inp["pgate"][b]),
                                         norm_w=inp["nw"], rope_cs=cs)
        ik = compress.compress_contract(bf(inp["ikv"][b]), bf(inp["igate"][b]), inp["iape"], r, True,
                                        prev_kv=bf(inp["ipkv"][b]), prev_gate=bf(inp["ipgate"][b]),
                                        norm_w=inp["inw"], rope_cs=cs)
        return ent, ik

    def _topk(self, b, ik):
        from oracle import codecs, indexer
        wl, inp = self.wl, self.inp
        n = int(wl.n_entries[b])
        if self.fp4:
            k_hat = codecs.decode_fp4h_pagesplit(self.keys[b], 128)
            k_hat[n - 1] = codecs.fp4b32_decode(*codecs.fp4b32_encode(codecs.hadamard_contract(ik)))[0]
            return indexer.index_topk_fp4(self._bf(inp["q_idx"][b]), inp["w"][b], k_hat, int(wl.ctx_len[b]),
                                          wl.ratio, wl.k)[0]
        k_hat = codecs.decode_pagesplit(self.keys[b], 128)
        k_hat[n - 1] = codecs.fp8_decode(*codecs.fp8_encode(ik, block=128), block=128)[0]   # one scale per key
        top, _ = indexer.index_topk(self._bf(inp["q_idx"][b]), inp["w"][b], k_hat, int(wl.ctx_len[b]),
                                    wl.ratio, wl.k, True)
        return top

    def query(self, b):
        """compress (main + index key of the completed block), index_topk, attention for request b."""
        from oracle import attention, codecs
        wl, inp = self.wl, self.inp
        n = int(wl.n_entries[b])
        ent, ik = self._compress(b)
        top = self._topk(b, ik)
        pages = self.main_pages[b]
        mf = wl.main_fmt
        ent_row = codecs.decode_rows(codecs.encode_rows(ent, mf), mf, 512)[0]

        def rows(ids):
            out = np.empty((len(ids), 512))
            for i, j in enumerate(ids):
                j = int(j)
                if j == n - 1:
                    out[i] = ent_row
                else:
                    out[i] = codecs.decode_rows(pages[j // 64][j % 64:j % 64 + 1], mf, 512)[0]
            return out

        swa_dec = codecs.decode_rows(self.swa[b], wl.swa_fmt, 512)
        return attention.request_attention(self._bf(inp["q"][b]), int(wl.ctx_len[b]), wl.ratio, swa_dec, rows,
                                           top, inp["sink"], 512 ** -0.5)


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    wl = synth.workload(WORKLOAD)
    nreq = min(wl.B, max(1, args.steps))
    runner = OracleRunner(wl, range(nreq))
    for i in range(args.warmup):
        runner.query(i % nreq)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        runner.query(i % nreq)
        times.append(time.perf_counter() - t0)
    per = statistics.mean(times)
    value = 1.0 / per
    sample = "one 1M-context query (one request of the batch) per step, %d distinct requests" % nreq
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (f32 for the compressor contract)",
        "data": "synthetic", "config": {"workload": workload_desc(wl)},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


ONE_CORE_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                 "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def _bf32(x):
    from oracle import codecs
    return codecs.bf16_decode(codecs.bf16_encode(x)).astype(np.float32)


def oracle_sample(mode):
    """The oracle timed on a bounded sample of a mode's workload (set-up untimed).
    Returns dict(value, unit, higher_is_better, sample)."""
    from oracle import attention, codecs, compress, indexer, rope
    if mode in ("decode", "mixed", "csa_fp4"):
        wl = synth.workload({"decode": WORKLOAD, "mixed": "mixed_mxfp4", "csa_fp4": "csa_fp4"}[mode])
        reqs = [0, 1]
        runner = OracleRunner(wl, reqs)
        t0 = time.perf_counter()
        for b in reqs:
            runner.query(b)
        dt = (time.perf_counter() - t0) / len(reqs)
        ctx = ", ".join("%d" % int(wl.ctx_len[b]) for b in reqs)
        return dict(value=1.0 / dt, unit="queries/s", higher_is_better=True,
                    sample="requests 0 and 1 of the batch (contexts %s tokens): compress the completed block "
                           "(main entry + index key), index_topk over every visible key, attention; numpy" % ctx)
    if mode == "tiny":
        wl = synth.workload("tiny_csa")
        T, r, n = 4096, 4, 1024
        lanes = {}
        for lane, dim, il in (("main", 512, False), ("index", 128, True)):
            kv, gate = synth.compressor_tokens(wl.seed, T, r, True, dim, index_lane=il)
            ape, nw = synth.compressor_params(wl.seed, r, True, dim, index_lane=il)
            kv, gate = _bf32(kv), _bf32(gate)
            ents = compress.compress_contract(kv, gate, ape, r, True, norm_w=nw, rope_cs=rope.table(np.arange(n) * r))
            lanes[lane] = (kv, gate, ape, nw, codecs.encode_rows(ents, codecs.FMT_BF16))
        q, q_idx, w, sink = synth.queries(wl)
        swa = codecs.encode_rows(synth.swa_values(wl, 0), codecs.FMT_BF16)

        def step():
            rows = {}
            for lane, dim in (("main", 512), ("index", 128)):
                kv, gate, ape, nw, cache = lanes[lane]
                e = compress.compress_contract(kv[-4:], gate[-4:], ape, r, True, prev_kv=kv[-8:-4], prev_gate=gate[-8:-4],
                                               norm_w=nw, rope_cs=rope.table(np.array([(n - 1) * r])))
                c = cache.copy()
                c[n - 1] = codecs.encode_rows(e, codecs.FMT_BF16)[0]
                rows[lane] = codecs.decode_rows(c, codecs.FMT_BF16, dim)
            top, _ = indexer.index_topk(_bf32(q_idx[0]), w[0], rows["index"], T, r, wl.k, False)
            return attention.request_attention(_bf32(q[0]), T, r, codecs.decode_rows(swa, codecs.FMT_BF16, 512),
                                               rows["main"], top, sink, 512 ** -0.5)
        step()
        reps = 3
        t0 = time.perf_counter()
        for _ in range(reps):
            step()
        dt = (time.perf_counter() - t0) / reps
        return dict(value=dt * 1e6, unit="us", higher_is_better=False,
                    sample="the whole step of the one request, 3 repetitions (compress main entry + index key, "
                           "index_topk over 1024 bf16 keys, attention over 128 + 512 bf16 rows); numpy")
    if mode == "hca":
        wl = synth.workload("hca_128k")
        reqs = [0, 1]
        data = {}
        for b in reqs:
            main = codecs.encode_rows(synth.request_values(wl, b, "main"), codecs.FMT_FP8)
            data[b] = (main, codecs.encode_rows(synth.swa_values(wl, b), codecs.FMT_FP8))
        q, _, _, sink = synth.queries(wl)
        t0 = time.perf_counter()
        for b in reqs:
            main, swa = data[b]
            attention.request_attention(_bf32(q[b]), int(wl.ctx_len[b]), wl.ratio,
                                        codecs.decode_rows(swa, codecs.FMT_FP8, 512),
                                        codecs.decode_rows(main, codecs.FMT_FP8, 512), None, sink, 512 ** -0.5)
        dt = (time.perf_counter() - t0) / len(reqs)
        return dict(value=1.0 / dt, unit="queries/s", higher_is_better=True,
                    sample="requests 0 and 1: decode of the 1,024 FP8 entries and 128 window rows, attention over "
                           "all of them with 64 heads; numpy")
    if mode.startswith("compress"):
        _, r, fmt = mode.split(":")
        r, fmt = int(r), int(fmt)
        overlap = r == 4
        T = 2048 if r == 4 else 8192
        kv, gate = synth.compressor_tokens(3, T, r, overlap, 512)
        ape, nw = synth.compressor_params(3, r, overlap, 512)
        kv, gate = _bf32(kv), _bf32(gate)
        cs = rope.table(np.arange(T // r) * r)
        t0 = time.perf_counter()
        ents = compress.compress_contract(kv, gate, ape, r, overlap, norm_w=nw, rope_cs=cs)
        codecs.encode_rows(ents, fmt)
        dt = time.perf_counter() - t0
        return dict(value=T / dt, unit="tokens/s", higher_is_better=True,
                    sample="the first %d tokens of the chunk (%d entries), fp32 contract + coding; numpy" % (T, T // r))
    raise ValueError(mode)


def cpu_baseline(mode="decode"):
    """The oracle on a bounded sample of the mode's workload: on every host core (this
    process, BLAS threads as numpy starts them) and on one core (a child process pinned to
    one CPU, every BLAS / OpenMP thread count set to 1)."""
    allc = oracle_sample(mode)
    res = {"value": allc["value"], "unit": allc["unit"], "cores": cores_used(), "kind": "oracle",
           "sample": allc["sample"]}
    env = dict(os.environ)
    for v in ONE_CORE_VARS:
        env[v] = "1"
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", mode, "--one-core"],
                             env=env, capture_output=True, text=True, timeout=600)
        one = json.loads(out.stdout.strip().splitlines()[-1])
        res["one_core"] = {"value": one["value"], "unit": one["unit"], "cores": 1}
    except Exception as e:  # the all-cores figure stands on its own
        res["one_core"] = {"value": None, "error": repr(e)[:200]}
    return res


def cpu_baseline_sample():
    return cpu_baseline("decode")


# ----------------------------------------------------------------------------- next-row modes
# Measurements of the rows built beyond the decode step (each prints its own JSON line;
# the default mode above is the benchmark).

def _graph_timed(torch, step, steps, warmup, flush, timing=None):
    """CUDA-event times (ms) of a captured step, the L2 flushed (outside the events) before
    each replay; timing = (cskv, ev_b, ev_e) records the score kernel live."""
    for _ in range(max(1, warmup)):
        step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    if timing:
        timing[0].set_timing_events(timing[1], timing[2])
    with torch.cuda.graph(graph):
        step()
        if timing:
            timing[0].set_timing_events(None, None)
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    clk = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
    clk.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    inner = []
    clk.mark("t0")
    for e0, e1 in evs:
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
        e1.synchronize()
        if timing:
            timing[2].synchronize()
            inner.append(timing[1].elapsed_time(timing[2]))
    torch.cuda.synchronize()
    clk.mark("t1")
    return [a.elapsed_time(b) for a, b in evs], inner, clk.stop()


def _lane(torch, cskv, wl, lane, fmt, dim, fill=True):
    """A paged cache of one lane of a workload, coded on the GPU from the seeded values."""
    bt, num_pages = synth.page_tables(wl, lane)
    rb = cskv.row_bytes(fmt, dim)
    cache = cskv.PagedCache(torch.zeros((num_pages, (64 * rb + 15) // 16 * 16), dtype=torch.uint8, device="cuda"),
                            torch.from_numpy(bt).cuda(), fmt, dim)
    if fill:
        f = synth.index_page_values if lane == "index" else synth.main_page_values
        ppr = wl.pages_per_req()
        for b in range(wl.B):
            vals = torch.from_numpy(np.concatenate(gen_parallel(lambda p: f(wl, b, p), range(int(ppr[b]))))).cuda()
            rows = torch.arange(vals.shape[0], dtype=torch.int32, device="cuda")
            cskv.encode_rows(vals, cache, req=torch.full_like(rows, b), row=rows)
            del vals
    return cache


def _ring(torch, cskv, wl, fmt):
    """The window rings as a paged cache (two 64-row pages per request), coded from the seeded values."""
    rb = cskv.row_bytes(fmt, 512)
    pool = torch.zeros((2 * wl.B, 64 * rb), dtype=torch.uint8, device="cuda")
    bt = torch.arange(2 * wl.B, dtype=torch.int32, device="cuda").view(wl.B, 2)
    ring = cskv.PagedCache(pool, bt, fmt, 512)
    vals = torch.from_numpy(np.stack([synth.swa_values(wl, b) for b in range(wl.B)])).cuda().reshape(-1, 512)
    rows = torch.arange(128, dtype=torch.int32, device="cuda").repeat(wl.B)
    req = torch.arange(wl.B, dtype=torch.int32, device="cuda").repeat_interleave(128)
    cskv.encode_rows(vals, ring, req=req, row=rows)
    return ring, pool


def _line(mode, metric, value, unit, ms, hib, config, roofline, clocks, launches, args):
    return {"mode": mode, "metric": metric, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": hib, "data": "synthetic",
            "config": config, "roofline": roofline, "clocks": clocks, "gpu_launches": launches}


def run_next_row(args):
    import torch
    import compressed_sparse_attention_kv_gb300 as cskv
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    psrc = "measured" if "hbm_gbs" in peaks else "fallback"
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    dev = "cuda"
    if args.mode == "csa2":
        # V4.1's CSA2 at 1M context, m = 2: the step updates the state (main and index
        # compressors without overlap or slot bias, the window), selects once and attends
        # in two layers that share the selection (Full, then Reuse)
        L, r, B, k, H, Hi = 1 << 20, 2, 8, 512, 64, 64
        wl = synth.custom_workload("csa2_1m", 5, [L] * B, r, k, H, Hi, synth.FMT_FP4, synth.FMT_FP8,
                                   synth.FMT_FP8_PAGESPLIT)
        keys = _lane(torch, cskv, wl, "index", cskv.FMT_FP8_PAGESPLIT, 128)
        main = _lane(torch, cskv, wl, "main", cskv.FMT_FP4, 512)
        ring, ring_pool = _ring(torch, cskv, wl, cskv.FMT_FP8)
        q, q_idx, w, sink = synth.queries(wl)
        bf = torch.bfloat16
        q = torch.from_numpy(q).to(bf).cuda()
        q2 = torch.roll(q, 1, dims=1).contiguous()            # the Reuse layer's own queries
        q_idx, w, sink = torch.from_numpy(q_idx).to(bf).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(sink).cuda()
        pos = torch.full((B,), L - 1, dtype=torch.int32, device=dev)
        ctx = torch.full((B,), L, dtype=torch.int32, device=dev)
        g = torch.Generator().manual_seed(5)
        tok = lambda c, d: torch.randn((B, c, d), generator=g).to(bf).cuda()   # noqa: E731
        nw = torch.from_numpy(synth.compressor_params(5, r, False, 512)[1]).cuda()
        inw = torch.from_numpy(synth.compressor_params(5, r, False, 128, index_lane=True)[1]).cuda()
        st_m, st_i = cskv.decode_state(B, r, 0, 512), cskv.decode_state(B, r, 0, 128)
        cs_e = torch.from_numpy(cskv.rope_table(np.full(B, L - r), yarn=cskv.YARN_V4)).cuda()
        cs_q = torch.from_numpy(cskv.rope_table(np.full(B, L - 1), yarn=cskv.YARN_V4)).cuda()
        jobs = [dict(kv=tok(1, 512), gate=tok(1, 512), state=st_m, ratio=r, overlap=0, out=main, norm_w=nw,
                     rope_cs=cs_e),
                dict(kv=tok(1, 128), gate=tok(1, 128), state=st_i, ratio=r, overlap=0, out=keys, norm_w=inw,
                     rope_cs=cs_e),
                dict(kv=tok(1, 512), gate=None, state=None, ratio=1, overlap=0, out=ring, norm_w=nw,
                     rope_cs=cs_q, ring_rows=128)]
        topk = torch.empty((B, k), dtype=torch.int32, device=dev)
        ws_i = torch.empty(cskv.index_topk_workspace_size(B, L, r, Hi, k), dtype=torch.uint8, device=dev)
        ws_a = torch.empty(cskv.sparse_decode_attn_workspace_size(B, H, L, r, k), dtype=torch.uint8, device=dev)
        out1, out2 = torch.empty_like(q), torch.empty_like(q)
        swa = ring_pool.view(B, 128, -1)

        def step():
            cskv.decode_append(jobs, pos)
            cskv.index_topk(q_idx, w, keys, ctx, r, k, L, topk_idx=topk, workspace=ws_i, want_scores=False)
            cskv.sparse_decode_attn(q, main, swa, cskv.FMT_FP8, ctx, topk, k, r, L, sink, cskv.DEFAULT_SCALE,
                                    cs_q, out=out1, workspace=ws_a)
            cskv.sparse_decode_attn(q2, main, swa, cskv.FMT_FP8, ctx, topk, k, r, L, sink, cskv.DEFAULT_SCALE,
                                    cs_q, out=out2, workspace=ws_a)

        evb, eve = live_events(torch)
        ms, inner, clocks = _graph_timed(torch, step, args.steps, args.warmup, flush, (cskv, evb, eve))
        st = cskv.device_status()
        assert st == 0, st
        m = statistics.mean(ms)
        sm_ = statistics.mean(inner)
        algo = 132 * B * (L // r)
        ach = algo / (sm_ * 1e-3) / 1e9
        return _line("csa2", "CSA2 (m=2) decode step at 1M context: queries/s (one Full + one Reuse layer)",
                     B / (m * 1e-3), "queries/s", m, True,
                     {"workload": "CSA2 m=2 at 1M context: batch 8, 1048576 tokens -> 524288 entries, 64 indexer "
                                  "heads x 128 FP8 keys (132 B), top-512 shared by two layers, 64 heads x 512 over "
                                  "MXFP4-288 entries + FP8 window; per step: decode_append (main, index key, window), "
                                  "index_topk, two sparse_decode_attn", "l2": "flushed before every step"},
                     {"kernel": "index_score_kernel", "bound": "hbm", "achieved": ach, "peak": peak,
                      "unit": "GB/s", "frac": ach / peak, "peak_source": psrc, "algorithmic_bytes_per_launch": algo,
                      "ms_per_launch": sm_, "traffic": None}, clocks, 1 + 2 + 2 + 2, args)
    if args.mode == "state":
        # one CSA layer's decode-state update for the 1M-context batch: every request's new
        # token completes a block (the costliest step: ring write, pooling, shift, window)
        wl = synth.workload(WORKLOAD)
        B, r, L = wl.B, wl.ratio, int(wl.ctx_len[0])
        keys = _lane(torch, cskv, wl, "index", cskv.FMT_FP8_PAGESPLIT, 128, fill=False)
        main = _lane(torch, cskv, wl, "main", cskv.FMT_FP8, 512, fill=False)
        ring, _ = _ring(torch, cskv, wl, cskv.FMT_FP8)
        bf = torch.bfloat16
        g = torch.Generator().manual_seed(6)
        tok = lambda c, d: torch.randn((B, c, d), generator=g).to(bf).cuda()   # noqa: E731
        ape, nw = (torch.from_numpy(x).cuda() for x in synth.compressor_params(wl.seed, r, True, 512))
        iape, inw = (torch.from_numpy(x).cuda() for x in synth.compressor_params(wl.seed, r, True, 128, True))
        pos = torch.full((B,), L - 1, dtype=torch.int32, device=dev)
        cs_e = torch.from_numpy(cskv.rope_table(np.full(B, L - r), yarn=cskv.YARN_V4)).cuda()
        cs_q = torch.from_numpy(cskv.rope_table(np.full(B, L - 1), yarn=cskv.YARN_V4)).cuda()
        jobs = [dict(kv=tok(2, 512), gate=tok(2, 512), state=cskv.decode_state(B, r, 1, 512), ratio=r, overlap=1,
                     out=main, ape=ape, norm_w=nw, rope_cs=cs_e),
                dict(kv=tok(2, 128), gate=tok(2, 128), state=cskv.decode_state(B, r, 1, 128), ratio=r, overlap=1,
                     out=keys, ape=iape, norm_w=inw, rope_cs=cs_e),
                dict(kv=tok(1, 512), gate=None, state=None, ratio=1, overlap=0, out=ring, norm_w=nw, rope_cs=cs_q,
                     ring_rows=128)]

        def step():
            cskv.decode_append(jobs, pos)

        ms, _, clocks = _graph_timed(torch, step, args.steps, args.warmup, flush)
        assert cskv.device_status() == 0
        m = statistics.mean(ms)
        # bytes the step must move: the new tokens, the rings read and shifted, the rows written
        per_req = (2 * 2 * 512 * 2 + 2 * 2 * 128 * 2 + 512 * 2          # new kv / gate tokens, window token
                   + 2 * (8 * 2 * 512 * 2 + 8 * 2 * 128 * 2)            # rings read (kv, gate)
                   + 2 * (4 * 2 * 512 * 2 + 4 * 2 * 128 * 2) * 2        # shift: read + write
                   + 4 * 1024 + 4 * 256                                 # slot biases
                   + 528 + 132 + 528)                                   # rows written
        algo = B * per_req
        ach = algo / (m * 1e-3) / 1e9
        return _line("state", "decode-step state update of a CSA layer (batch 8, every request completes a block): "
                     "us per step", m * 1e3, "us", m, False,
                     {"workload": "csa_1m batch 8 at position 1048575: main (ratio 4, overlap, FP8-528) and index-key "
                                  "(128-d, FP8-132) compressor state rings, window ring write; one decode_append launch",
                      "l2": "flushed before every step"},
                     {"kernel": "decode_append_kernel", "bound": "latency", "achieved": ach, "peak": peak,
                      "unit": "GB/s", "frac": ach / peak, "peak_source": psrc, "algorithmic_bytes_per_launch": algo,
                      "ms_per_launch": m, "traffic": None}, clocks, 1, args)
    # prefill: the last 2,048 queries of an 8,192-token prompt (one chunk), each with its
    # own selection (indexer rows per query) and causal window
    Lp, r, k, H, Hi, T = 8192, 4, 512, 64, 64, 2048
    wl = synth.custom_workload("prefill_8k", 6, [Lp], r, k, H, Hi, synth.FMT_FP8, synth.FMT_FP8,
                               synth.FMT_FP8_PAGESPLIT)
    keys = _lane(torch, cskv, wl, "index", cskv.FMT_FP8_PAGESPLIT, 128)
    main = _lane(torch, cskv, wl, "main", cskv.FMT_FP8, 512)
    rawwl = synth.custom_workload("prefill_8k_raw", 7, [Lp], 1, k, H, Hi, synth.FMT_FP8, synth.FMT_FP8,
                                  synth.FMT_FP8)
    raw = _lane(torch, cskv, rawwl, "main", cskv.FMT_FP8, 512)
    rs = np.random.default_rng(8)
    bf = torch.bfloat16
    q = torch.from_numpy(rs.standard_normal((T, H, 512)).astype(np.float32)).to(bf).cuda()
    q_idx = torch.from_numpy(rs.standard_normal((T, Hi, 128)).astype(np.float32)).to(bf).cuda()
    w = torch.from_numpy(rs.uniform(0, 1, (T, Hi)).astype(np.float32)).cuda()
    sink = torch.from_numpy(rs.standard_normal(H).astype(np.float32)).cuda()
    posn = np.arange(Lp - T, Lp)
    pos1 = torch.from_numpy((posn + 1).astype(np.int32)).cuda()
    cs = torch.from_numpy(cskv.rope_table(posn)).cuda()
    kq = cskv.PagedCache(keys.pool, keys.block_table[torch.zeros(T, dtype=torch.long, device=dev)].contiguous(),
                         keys.fmt, keys.dim)
    topk = torch.empty((T, k), dtype=torch.int32, device=dev)
    ws_i = torch.empty(cskv.index_topk_workspace_size(T, Lp, r, Hi, k), dtype=torch.uint8, device=dev)
    ws_a = torch.empty(cskv.sparse_decode_attn_workspace_size(T, H, Lp, r, k), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    req_of = torch.zeros(T, dtype=torch.int32, device=dev)   # every query belongs to the one prompt

    def step():
        cskv.index_topk(q_idx, w, kq, pos1, r, k, Lp, topk_idx=topk, workspace=ws_i, want_scores=False)
        cskv.sparse_prefill_attn(q, main, raw, pos1, topk, k, r, Lp, sink, cskv.DEFAULT_SCALE, cs, req_of=req_of,
                                 out=out, workspace=ws_a)

    ms, _, clocks = _graph_timed(torch, step, args.steps, args.warmup, flush)
    st = cskv.device_status()
    assert st == 0, st
    m = statistics.mean(ms)
    # bytes a prefill chunk must move at least: the queries in, the outputs out, the prompt's
    # raw rows, entries and index keys once, the indexer queries
    algo = T * H * 512 * 2 * 2 + Lp * 528 + (Lp // r) * (528 + 132) + T * Hi * 128 * 2
    ach = algo / (m * 1e-3) / 1e9
    return _line("prefill", "prefill chunk: prompt queries/s (2,048 queries of an 8,192-token prompt)",
                 T / (m * 1e-3), "queries/s", m, True,
                 {"workload": "prefill of an 8192-token prompt, last 2048 positions: ratio 4 (2048 entries), 64 "
                              "indexer heads x 128 FP8 keys, top-512 per query, 64 heads x 512 over FP8-528 entries "
                              "+ FP8 raw window rows; per step: index_topk (one row per query), sparse_prefill_attn",
                  "l2": "flushed before every step"},
                 {"kernel": "whole step", "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                  "frac": ach / peak, "peak_source": psrc, "algorithmic_bytes_per_launch": algo,
                  "ms_per_launch": m, "traffic": None}, clocks, 2 + 2, args)


# ----------------------------------------------------------------------------- the other configurations
# The tiny CSA layer, the HCA layer at 128K, the compressor's 65,536-token chunk and the
# mixed-batch MXFP4 layer (the last through run_gpu, the decode step's own path).  Each
# prints a JSON line of its own with the roofline of its step, the oracle's CPU figure and
# the clocks; they are measurements of the other named workloads, not the benchmark.

def _peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk["hbm_gbs"], "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def run_config_mode(args):
    import torch
    import compressed_sparse_attention_kv_gb300 as cskv
    peak, psrc = _peak()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    bf = torch.bfloat16
    dev = "cuda"

    def roof(kernel, algo, ms, bound="hbm"):
        ach = algo / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": bound, "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "peak_source": psrc, "algorithmic_bytes_per_launch": algo, "ms_per_launch": ms, "traffic": None}

    def finish(line, mode):
        if not args.no_cpu_baseline:
            try:
                line["cpu_baseline"] = cpu_baseline(mode)
            except Exception as e:
                line["cpu_baseline"] = {"value": None, "error": repr(e)[:200]}
        return line

    if args.mode == "tiny":
        wl = synth.workload("tiny_csa")
        T, r, n, k, H, Hi = 4096, 4, 1024, wl.k, wl.H, wl.Hi
        zero = torch.zeros(1, dtype=torch.int32, device=dev)
        caches, jobs = {}, []
        for lane, dim, il in (("main", 512, False), ("index", 128, True)):
            kv, gate = synth.compressor_tokens(wl.seed, T, r, True, dim, index_lane=il)
            ape, nw = synth.compressor_params(wl.seed, r, True, dim, index_lane=il)
            kv_t = torch.from_numpy(kv).to(bf)[None].to(dev)
            g_t = torch.from_numpy(gate).to(bf)[None].to(dev)
            ape_t, nw_t = torch.from_numpy(ape).to(dev), torch.from_numpy(nw).to(dev)
            cache = cskv.PagedCache(torch.zeros((n // 64, 64 * dim * 2), dtype=torch.uint8, device=dev),
                                    torch.arange(n // 64, dtype=torch.int32, device=dev)[None], cskv.FMT_BF16, dim)
            cskv.compress(kv_t, g_t, ape_t, r, True, cache, zero, zero, norm_w=nw_t,
                          rope_cs=torch.from_numpy(cskv.rope_table(np.arange(n) * r)[None]).to(dev))
            caches[lane] = cache
            # the step's completed block: the last 4 tokens, with the 4 before them as the previous block
            jobs.append(dict(kv=kv_t[:, -4:].contiguous(), gate=g_t[:, -4:].contiguous(), ape=ape_t, ratio=r,
                             overlap=True, out=cache, req=zero,
                             first_entry=torch.full((1,), n - 1, dtype=torch.int32, device=dev),
                             prev_kv=kv_t[:, -8:-4].contiguous(), prev_gate=g_t[:, -8:-4].contiguous(), norm_w=nw_t,
                             rope_cs=torch.from_numpy(cskv.rope_table(np.array([[(n - 1) * r]]))).to(dev)))
        q, q_idx, w, sink = synth.queries(wl)
        q = torch.from_numpy(q).to(bf).to(dev)
        q_idx = torch.from_numpy(q_idx).to(bf).to(dev)
        w, sink = torch.from_numpy(w).to(dev), torch.from_numpy(sink).to(dev)
        swa = torch.zeros((1, 128, 1024), dtype=torch.uint8, device=dev)
        cskv.encode_rows(torch.from_numpy(synth.swa_values(wl, 0)).to(dev),
                         cskv.PagedCache(swa.view(2, 64 * 1024), None, cskv.FMT_BF16, 512))
        ctx = torch.full((1,), T, dtype=torch.int32, device=dev)
        qcs = torch.from_numpy(cskv.rope_table(np.array([T - 1]))).to(dev)
        topk = torch.empty((1, k), dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws_i = torch.empty(cskv.index_topk_workspace_size(1, T, r, Hi, k), dtype=torch.uint8, device=dev)
        ws_a = torch.empty(cskv.sparse_decode_attn_workspace_size(1, H, T, r, k), dtype=torch.uint8, device=dev)

        def step():
            cskv.compress_many(jobs)
            cskv.index_topk(q_idx, w, caches["index"], ctx, r, k, T, topk_idx=topk, workspace=ws_i, want_scores=False)
            cskv.sparse_decode_attn(q, caches["main"], swa, cskv.FMT_BF16, ctx, topk, k, r, T, sink,
                                    cskv.DEFAULT_SCALE, qcs, out=out, workspace=ws_a)

        ms, _, clocks = _graph_timed(torch, step, args.steps, args.warmup, flush)
        assert cskv.device_status() == 0
        m = statistics.mean(ms)
        # bytes the step must move: the completed block's tokens (2 lanes, 8 slots x 2 halves x kv+gate),
        # the index keys, the 640 bf16 rows attended, queries and output
        algo = (8 * 2 * 2 * (512 + 128) * 2 + n * 256 + 640 * 1024 + 2 * H * 512 * 2 + Hi * 128 * 2)
        line = _line("tiny", "tiny CSA decode layer (batch 1, 4096 tokens): step latency", m * 1e3, "us", m, False,
                     {"workload": "Tiny CSA decode layer: batch 1, context 4096 tokens, ratio 4 (1024 entries), "
                                  "top-512, 16 query heads x 512 (last 64 RoPE, theta 160000), 4 indexer heads x "
                                  "128, SWA 128, bf16 KV and queries N(0,1), gate logits N(0,1), seed 0; caches "
                                  "compressed from the 4096 tokens; per step: compress the completed block "
                                  "(main + index key), index_topk, sparse_decode_attn",
                      "l2": "flushed before every step (the workload is L2-sized)"},
                     roof("whole step", algo, m, bound="latency"), clocks, 1 + 2 + 2, args)
        return finish(line, "tiny")

    if args.mode == "hca":
        wl = synth.workload("hca_128k")
        B, r, H, L = wl.B, wl.ratio, wl.H, wl.max_ctx
        n = L // r
        main = _lane(torch, cskv, wl, "main", cskv.FMT_FP8, 512)
        swa = torch.zeros((B, 128, 528), dtype=torch.uint8, device=dev)
        cskv.encode_rows(torch.from_numpy(np.stack([synth.swa_values(wl, b) for b in range(B)])).to(dev).reshape(-1, 512),
                         cskv.PagedCache(swa.view(B * 2, 64 * 528), None, cskv.FMT_FP8, 512))
        q, _, _, sink = synth.queries(wl)
        q = torch.from_numpy(q).to(bf).to(dev)
        sink = torch.from_numpy(sink).to(dev)
        ctx = torch.from_numpy(wl.ctx_len.astype(np.int32)).to(dev)
        qcs = torch.from_numpy(cskv.rope_table(wl.ctx_len - 1)).to(dev)
        out = torch.empty_like(q)
        ws_a = torch.empty(cskv.sparse_decode_attn_workspace_size(B, H, L, r, 0), dtype=torch.uint8, device=dev)

        def step():
            cskv.sparse_decode_attn(q, main, swa, cskv.FMT_FP8, ctx, None, 0, r, L, sink, cskv.DEFAULT_SCALE, qcs,
                                    out=out, workspace=ws_a)

        ms, _, clocks = _graph_timed(torch, step, args.steps, args.warmup, flush)
        assert cskv.device_status() == 0
        m = statistics.mean(ms)
        per_q = (n + 128) * 528 + 2 * H * 512 * 2      # every visible entry and the window, query in, output out
        line = _line("hca", "HCA decode layer at 128K context: queries/s per layer (batch 32)", B / (m * 1e-3),
                     "queries/s", m, True,
                     {"workload": "HCA decode layer: batch 32, context 131072 (1024 entries at ratio 128, all read) "
                                  "+ SWA 128, 64 query heads x 512, KV FP8 e4m3 + e8m0 per 32 values (528 B/token), "
                                  "values N(0,1), shuffled 64-row pages, sink; per step: sparse_decode_attn over "
                                  "every visible entry",
                      "l2": "flushed before every step (the 23.7 MB working set would otherwise sit in L2)"},
                     roof("attn_tile_kernel + attn_combine_kernel", B * per_q, m), clocks, 2, args)
        return finish(line, "hca")

    if args.mode == "compress":
        T = 65536
        lines = []
        for r, overlap in ((4, True), (128, False)):
            coff = 2 if overlap else 1
            kv, gate = synth.compressor_tokens(3, T, r, overlap, 512)
            ape, nw = synth.compressor_params(3, r, overlap, 512)
            kv_t = torch.from_numpy(kv).to(bf)[None].to(dev)
            g_t = torch.from_numpy(gate).to(bf)[None].to(dev)
            ape_t, nw_t = torch.from_numpy(ape).to(dev), torch.from_numpy(nw).to(dev)
            n = T // r
            cs = torch.from_numpy(cskv.rope_table(np.arange(n) * r)[None]).to(dev)
            zero = torch.zeros(1, dtype=torch.int32, device=dev)
            for fmt, fname in ((cskv.FMT_FP8, "FP8-528"), (cskv.FMT_FP4, "MXFP4-288")):
                pages = (n + 63) // 64
                out = cskv.PagedCache.allocate(pages, fmt, 512,
                                               block_table=torch.randperm(pages, dtype=torch.int32).to(dev)[None])

                def step():
                    cskv.compress(kv_t, g_t, ape_t, r, overlap, out, zero, zero, norm_w=nw_t, rope_cs=cs)

                ms, _, clocks = _graph_timed(torch, step, args.steps, args.warmup, flush)
                assert cskv.device_status() == 0
                m = statistics.mean(ms)
                rb = cskv.row_bytes(fmt, 512)
                algo = T * coff * 512 * 2 * 2 + n * rb + r * coff * 512 * 4 + n * 64 * 4 + 512 * 4
                line = _line("compress", "compressor throughput: tokens/s (65,536-token chunk, ratio %d -> %s)"
                             % (r, fname), T / (m * 1e-3), "tokens/s", m, True,
                             {"workload": "Compressor throughput: 65536-token chunk of 512-dim bf16 kv + gate "
                                          "(N(0,1), seed 3), slot bias 0.5 N(0,1), RMSNorm weight U(0.5, 1.5), "
                                          "ratio %d%s, RoPE at each entry's first token, coded %s into shuffled "
                                          "64-row pages; one cskv_compress launch"
                                          % (r, " with overlap (coff 2)" if overlap else "", fname),
                              "l2": "flushed before every step; the %d MB read exceeds L2 at ratio 4"
                                    % (T * coff * 512 * 4 // 1000000)},
                             roof("compress_kernel<512>", algo, m), clocks, 1, args)
                lines.append(finish(line, "compress:%d:%d" % (r, fmt)))
        return lines
    raise ValueError(args.mode)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 1000 for the GPU decode benchmark, so that the clock samples "
                         "fall inside the timed region; 50 for the oracle arm and the other modes)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cskv", "reference"], default="cskv")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["decode", "tiny", "hca", "compress", "mixed", "csa_fp4", "csa2", "state",
                                       "prefill"],
                    default="decode",
                    help="decode: the benchmark (1M context); tiny / hca / compress / mixed: the other named "
                         "workloads; csa2 / state / prefill: the rows built beyond the decode step")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--one-core", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample is not None:
        # child of cpu_baseline(): the oracle's sample on one core (thread counts come from the environment)
        if args.one_core and hasattr(os, "sched_setaffinity"):
            os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})
        print(json.dumps(oracle_sample(args.oracle_sample)))
        return
    args.warmup = max(3, args.warmup)
    if args.steps is None:
        args.steps = 1000 if (args.impl == "cskv" and args.mode in ("decode", "mixed", "csa_fp4")) else 50
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if args.mode in ("tiny", "hca", "compress"):
        if rank == 0:
            res = run_config_mode(args)
            for line in (res if isinstance(res, list) else [res]):
                print(json.dumps(line))
        return
    if args.mode in ("mixed", "csa_fp4"):
        res = run_gpu(args, 0, 1, workload="mixed_mxfp4" if args.mode == "mixed" else "csa_fp4")
        res["mode"] = args.mode
        if not args.no_cpu_baseline:
            try:
                res["cpu_baseline"] = cpu_baseline(args.mode)
            except Exception as e:
                res["cpu_baseline"] = {"value": None, "error": repr(e)[:200]}
        print(json.dumps(res))
        return
    if args.mode != "decode":
        if rank == 0:
            print(json.dumps(run_next_row(args)))
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    res = run_gpu(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            try:
                res["cpu_baseline"] = cpu_baseline_sample()
            except Exception as e:  # report the GPU line even if the CPU leg fails
                res["cpu_baseline"] = {"value": None, "error": repr(e)[:200]}
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
