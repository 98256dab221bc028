"""cskv_index_topk_noalloc, the indexer entry point that allocates nothing.

Some callers cannot allocate device memory (code running under CUDA-graph
stream capture, plugins whose host owns all device memory, threads that must
not block on the driver); this entry point takes its scratch from a fixed
array inside the library.  It must give exactly what cskv_index_topk gives
with a caller-provided workspace, call after call.  The file sorts last so
that a run that stops at the first failure has run every other test first.
"""

import ctypes

import numpy as np
import pytest
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from compressed_sparse_attention_kv_gb300 import _lib
from oracle import codecs

from cases import HostPaged, bf16_values, cuda

pytestmark = pytest.mark.gpu

NOALLOC_LIMIT = 32 << 20   # CSKV_NOALLOC_SCRATCH_BYTES


def _noalloc(q, w, keys, ctx, B, Hi, ratio, k, max_ctx, idx, score):
    return _lib.lib().cskv_index_topk_noalloc(q.data_ptr(), w.data_ptr(), keys.desc(), ctx.data_ptr(), B, Hi,
                                              ratio, k, max_ctx, idx.data_ptr(), score.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_twice():
    ratio, k, Hi = 4, 512, 64
    ctx = [4 * 9000 + 1, 4 * 300, 4 * 20000 + 3]
    n = [c // ratio for c in ctx]
    rs = np.random.default_rng(21)
    cache = HostPaged(codecs.FMT_FP8_PAGESPLIT, 128, n, seed=22)
    for b, nb in enumerate(n):
        cache.fill(b, rs.standard_normal((nb, 128)).astype(np.float32))
    keys = cache.to_device()
    q_t, _ = bf16_values(rs.standard_normal((len(ctx), Hi, 128)).astype(np.float32))
    q = q_t.cuda()
    w = cuda(rs.uniform(0, 1, (len(ctx), Hi)).astype(np.float32))
    ctx_d = cuda(np.asarray(ctx, np.int32))
    ref_idx, ref_sc = cskv.index_topk(q, w, keys, ctx_d, ratio, k, max(ctx))
    assert cskv.device_status() == 0
    for _ in range(2):   # two calls in a row share the library's scratch array
        idx = torch.full((len(ctx), k), 7, dtype=torch.int32, device="cuda")
        sc = torch.zeros((len(ctx), k), dtype=torch.float32, device="cuda")
        st = _noalloc(q, w, keys, ctx_d, len(ctx), Hi, ratio, k, max(ctx), idx, sc)
        assert st == 0, cskv.CskvError(st, "cskv_index_topk_noalloc")
        assert cskv.device_status() == 0
        assert torch.equal(idx, ref_idx)
        assert torch.equal(sc, ref_sc)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ratio, k, Hi, B = 4, 512, 64, 8
    max_ctx = 1 << 24          # 4M entries per request: the workspace would not fit
    assert cskv.index_topk_workspace_size(B, max_ctx, ratio, Hi, k) > NOALLOC_LIMIT
    keys = cskv.PagedCache(torch.zeros((4, 64 * 132), dtype=torch.uint8, device="cuda"),
                           torch.zeros((B, 4), dtype=torch.int32, device="cuda"), cskv.FMT_FP8_PAGESPLIT, 128)
    q = torch.zeros((B, Hi, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((B, Hi), dtype=torch.float32, device="cuda")
    ctx = torch.ones(B, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, k), dtype=torch.float32, device="cuda")
    assert _noalloc(q, w, keys, ctx, B, Hi, ratio, k, max_ctx, idx, sc) == 1


def _limit_sizes(B, ratio, Hi, k):
    """The largest max_ctx_len whose workspace fits the scratch array, and the smallest
    one that does not (the workspace grows in steps of 128 entries)."""
    def ws(c):
        return cskv.index_topk_workspace_size(B, c, ratio, Hi, k)
    lo, hi = ratio, ratio * (1 << 24)
    assert ws(lo) <= NOALLOC_LIMIT < ws(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if ws(mid) <= NOALLOC_LIMIT:
            lo = mid
        else:
            hi = mid
    return lo, hi


def test_noalloc_at_the_edge_of_its_scratch():
    """One request whose workspace is just under the 32 MiB array (the array's top end
    in use) gives the workspace entry point's bits, twice in a row; one context step
    further the call is rejected before anything is launched."""
    ratio, k, Hi, B = 4, 512, 64, 1
    under, over = _limit_sizes(B, ratio, Hi, k)
    assert cskv.index_topk_workspace_size(B, under, ratio, Hi, k) > NOALLOC_LIMIT - (1 << 16)
    n = under // ratio
    pages = (n + 63) // 64
    g = torch.Generator(device="cuda").manual_seed(31)
    keys = cskv.PagedCache(torch.zeros((pages, 64 * 132), dtype=torch.uint8, device="cuda"),
                           torch.randperm(pages, generator=g, device="cuda").to(torch.int32)[None].contiguous(),
                           cskv.FMT_FP8_PAGESPLIT, 128)
    step = 1 << 18
    for r0 in range(0, pages * 64, step):
        rows = torch.arange(r0, min(r0 + step, pages * 64), dtype=torch.int32, device="cuda")
        vals = torch.randn((rows.numel(), 128), generator=g, device="cuda")
        cskv.encode_rows(vals, keys, req=torch.zeros_like(rows), row=rows)
    q = torch.randn((B, Hi, 128), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.rand((B, Hi), generator=g, device="cuda")
    ctx = torch.full((B,), under, dtype=torch.int32, device="cuda")
    ref_idx, ref_sc = cskv.index_topk(q, w, keys, ctx, ratio, k, under)
    assert cskv.device_status() == 0
    for _ in range(2):
        idx = torch.full((B, k), 7, dtype=torch.int32, device="cuda")
        sc = torch.zeros((B, k), dtype=torch.float32, device="cuda")
        st = _noalloc(q, w, keys, ctx, B, Hi, ratio, k, under, idx, sc)
        assert st == 0, cskv.CskvError(st, "cskv_index_topk_noalloc")
        assert cskv.device_status() == 0
        assert torch.equal(idx, ref_idx)
        assert torch.equal(sc, ref_sc)
    assert cskv.index_topk_workspace_size(B, over, ratio, Hi, k) > NOALLOC_LIMIT
    idx = torch.full((B, k), 7, dtype=torch.int32, device="cuda")
    sc = torch.zeros((B, k), dtype=torch.float32, device="cuda")
    assert _noalloc(q, w, keys, ctx, B, Hi, ratio, k, over, idx, sc) == 1
    assert cskv.device_status() == 0
    assert torch.all(idx == 7)                  # nothing was launched
