"""compressed_sparse_attention_kv_gb300: DeepSeek-V4-style compressed-KV decode attention on GB300.

Thin Python binding over libcskv.so (include/cskv.h).  Every function here only
marshals arguments: torch tensors provide device memory and the current CUDA
stream; all arithmetic of the decode path runs in the library's sm_103a
kernels.  There is no CPU fallback: calling into the library without it being
built raises.

Calls (same names as the C ABI, without the ``cskv_`` prefix):

    compress(...)            gated per-channel pooling compressor -> cache rows
    compress_many(...)       several compressor jobs in one launch
    decode_append(...)       one decode step's compressor state ring and window update
    index_topk(...)          lightning-indexer scores + top-k selection
    sparse_decode_attn(...)  shared-KV attention over window + compressed entries
    sparse_prefill_attn(...) the same attention for many prompt queries
    decode_layer(...)        one layer's decode step, host buffers in and out
    encode_rows(...)         code rows of values into a cache format
"""

import ctypes
import math

import numpy as np

from . import _lib

FMT_BF16 = 0
FMT_FP8 = 1
FMT_FP4 = 2
FMT_FP8_PAGESPLIT = 3
FMT_FP4H_PAGESPLIT = 4
PAGE_ROWS = 64
WINDOW = 128

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device timeout",
           5: "device bounds"}


class CskvError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, _STATUS.get(status, "?"), status))


def _check(status, what):
    if status != 0:
        raise CskvError(status, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t, dtype, name, device=True):
    import torch
    if t is None:
        return
    if device and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def row_bytes(fmt, dim):
    return int(_lib.lib().cskv_row_bytes(fmt, dim))


def version():
    return int(_lib.lib().cskv_version())


def device_status(stream=None):
    """Synchronise the stream and return (and clear) the library's sticky device status."""
    return int(_lib.lib().cskv_device_status(_stream(stream)))


def set_spin_limit(cycles):
    _lib.lib().cskv_set_spin_limit(int(cycles))


def set_timing_events(begin, end):
    """Record torch.cuda.Event `begin`/`end` around every later indexer score kernel (None, None: off)."""
    if begin is None or end is None:
        _lib.lib().cskv_set_timing_events(None, None)
    else:
        _lib.lib().cskv_set_timing_events(begin.cuda_event, end.cuda_event)


class PagedCache:
    """A paged cache: `pool` uint8 [num_pages, page_bytes] on the GPU and an int32
    block table [batch, max_pages] (or None for a flat array of rows)."""

    def __init__(self, pool, block_table, fmt, dim):
        import torch
        _need(pool, torch.uint8, "pool")
        _need(block_table, torch.int32, "block_table")
        self.pool = pool
        self.block_table = block_table
        self.fmt = int(fmt)
        self.dim = int(dim)

    @classmethod
    def allocate(cls, num_pages, fmt, dim, block_table=None, device="cuda"):
        import torch
        rb = row_bytes(fmt, dim)
        page = PAGE_ROWS * rb
        page = (page + 15) // 16 * 16
        pool = torch.zeros((num_pages, page), dtype=torch.uint8, device=device)
        return cls(pool, block_table, fmt, dim)

    def desc(self):
        return _lib.Paged(self.pool.data_ptr(),
                          None if self.block_table is None else self.block_table.data_ptr(),
                          self.pool.shape[1], self.pool.shape[0],
                          0 if self.block_table is None else self.block_table.shape[1],
                          self.fmt, self.dim)


# YaRN of the compressed layers: 65,536 original positions stretched 16-fold, betas 32 / 1
YARN_V4 = dict(factor=16.0, original=65536, beta_fast=32.0, beta_slow=1.0)


def rope_table(positions, theta=160000.0, rope_dim=64, yarn=None):
    """float32 [..., 32, 2] (cos, sin) of every position, from cskv_rope_table (host code in
    the library): plain frequencies theta^(-2k/64), or with yarn (a dict like YARN_V4) the
    YaRN blend over the pair index."""
    if rope_dim != 64:
        raise ValueError("the kernels rotate 64 dims")
    pos = np.ascontiguousarray(np.asarray(positions), dtype=np.int64)
    out = np.empty(pos.shape + (32, 2), dtype=np.float32)
    y = yarn or {}
    st = _lib.lib().cskv_rope_table(pos.ctypes.data, int(pos.size), float(theta), float(y.get("factor", 1.0)),
                                    float(y.get("original", 1.0)), float(y.get("beta_fast", 1.0)),
                                    float(y.get("beta_slow", 1.0)), out.ctypes.data)
    _check(st, "cskv_rope_table")
    return out


def encode_rows(src, dst, req=None, row=None, stream=None):
    """Code rows of src (fp32 or bf16 [n, dim]) into the cache dst (rows row[i] of request req[i])."""
    import torch
    if src.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("src must be float32 or bfloat16")
    _need(src, None, "src")
    _need(req, torch.int32, "req")
    _need(row, torch.int32, "row")
    n, dim = src.shape
    st = _lib.lib().cskv_encode_rows(src.data_ptr(), int(src.dtype == torch.bfloat16), n, dim,
                                     _ptr(req), _ptr(row), dst.desc(), _stream(stream))
    _check(st, "cskv_encode_rows")


def compress(kv, gate, ape, ratio, overlap, out, req, first_entry, prev_kv=None, prev_gate=None,
             norm_w=None, eps=1e-6, rope_cs=None, stream=None):
    """Gated per-channel pooling of S sequences of T tokens (kv, gate: bf16 [S, T, coff, dim]);
    ape None = no slot bias (the V4.1 compressor)."""
    import torch
    for t, n in ((kv, "kv"), (gate, "gate"), (prev_kv, "prev_kv"), (prev_gate, "prev_gate")):
        _need(t, torch.bfloat16, n)
    for t, n in ((ape, "ape"), (norm_w, "norm_w"), (rope_cs, "rope_cs")):
        _need(t, torch.float32, n)
    _need(req, torch.int32, "req")
    _need(first_entry, torch.int32, "first_entry")
    S, T, coff, dim = kv.shape
    st = _lib.lib().cskv_compress(kv.data_ptr(), gate.data_ptr(), _ptr(prev_kv), _ptr(prev_gate),
                                  _ptr(ape), _ptr(norm_w), float(eps), _ptr(rope_cs),
                                  S, T, int(ratio), int(bool(overlap)), dim, req.data_ptr(),
                                  first_entry.data_ptr(), out.desc(), _stream(stream))
    _check(st, "cskv_compress")


def compress_many(jobs, stream=None):
    """Several compressor jobs in one launch.  Each job is a dict of compress()'s
    arguments (kv, gate, ape, ratio, overlap, out, req, first_entry and, optionally,
    prev_kv, prev_gate, norm_w, eps, rope_cs); same results as separate calls."""
    arr = _compress_jobs(jobs)
    st = _lib.lib().cskv_compress_many(arr, len(jobs), _stream(stream))
    _check(st, "cskv_compress_many")


def _compress_jobs(jobs, host_inputs=False):
    """ctypes array of struct cskv_compress_job for compress()-style job dicts.  With
    host_inputs (decode_layer), kv, gate, prev_kv, prev_gate and rope_cs may be pinned
    host tensors (read in place by the compressor)."""
    import torch

    def need_in(t, dtype, name):
        _need(t, dtype, name, device=not host_inputs)
        if t is not None and not t.is_cuda and not t.is_pinned():
            raise ValueError("%s must be a CUDA tensor or a pinned host tensor" % name)

    arr = (_lib.CompressJob * max(1, len(jobs)))()
    for i, j in enumerate(jobs):
        kv, gate = j["kv"], j["gate"]
        for t, n in ((kv, "kv"), (gate, "gate"), (j.get("prev_kv"), "prev_kv"), (j.get("prev_gate"), "prev_gate")):
            need_in(t, torch.bfloat16, n)
        need_in(j.get("rope_cs"), torch.float32, "rope_cs")
        for t, n in ((j.get("ape"), "ape"), (j.get("norm_w"), "norm_w")):
            _need(t, torch.float32, n)
        _need(j["req"], torch.int32, "req")
        _need(j["first_entry"], torch.int32, "first_entry")
        S, T, coff, dim = kv.shape
        arr[i] = _lib.CompressJob(kv.data_ptr(), gate.data_ptr(), _ptr(j.get("prev_kv")), _ptr(j.get("prev_gate")),
                                  _ptr(j.get("ape")), _ptr(j.get("norm_w")), float(j.get("eps", 1e-6)),
                                  _ptr(j.get("rope_cs")), S, T, int(j["ratio"]), int(bool(j["overlap"])), dim,
                                  j["req"].data_ptr(), j["first_entry"].data_ptr(), j["out"].desc())
    return arr


def decode_state(B, ratio, overlap, dim, device="cuda"):
    """A fresh per-request compressor state ring for decode_append: (state_kv, state_gate),
    bf16 [B, nblk * ratio, coff, dim] (nblk = coff = 2 with overlap, else 1), kv 0 and gate -inf."""
    import torch
    nblk = 2 if overlap else 1
    coff = 2 if overlap else 1
    shape = (B, nblk * ratio, coff, dim)
    return (torch.zeros(shape, dtype=torch.bfloat16, device=device),
            torch.full(shape, float("-inf"), dtype=torch.bfloat16, device=device))


def decode_append(jobs, pos, stream=None):
    """One decode step's state update.  Each job is a dict: kv, gate (bf16 [B, coff, dim]; gate
    may be None at ratio 1), state (the (state_kv, state_gate) pair of decode_state; None at
    ratio 1), ratio, overlap, out (PagedCache), and optionally ape, norm_w, eps, rope_cs
    (fp32 [B, 32, 2] at the position each request writes), ring_rows.  pos: int32 [B]
    positions of the new tokens (< 0: no token)."""
    import torch
    _need(pos, torch.int32, "pos")
    arr = (_lib.DecodeJob * len(jobs))()
    for i, j in enumerate(jobs):
        kv = j["kv"]
        _need(kv, torch.bfloat16, "kv")
        _need(j.get("gate"), torch.bfloat16, "gate")
        st = j.get("state")
        sk, sg = (st if st is not None else (None, None))
        _need(sk, torch.bfloat16, "state_kv")
        _need(sg, torch.bfloat16, "state_gate")
        for t, n in ((j.get("ape"), "ape"), (j.get("norm_w"), "norm_w"), (j.get("rope_cs"), "rope_cs")):
            _need(t, torch.float32, n)
        arr[i] = _lib.DecodeJob(kv.data_ptr(), _ptr(j.get("gate")), _ptr(sk), _ptr(sg), _ptr(j.get("ape")),
                                _ptr(j.get("norm_w")), float(j.get("eps", 1e-6)), _ptr(j.get("rope_cs")),
                                int(j["ratio"]), int(bool(j.get("overlap", 0))), int(kv.shape[-1]),
                                int(j.get("ring_rows", 0)), j["out"].desc())
    st = _lib.lib().cskv_decode_append(arr, len(jobs), pos.data_ptr(), int(pos.shape[0]), _stream(stream))
    _check(st, "cskv_decode_append")


def index_topk_workspace_size(B, max_ctx_len, ratio, Hi, k):
    return int(_lib.lib().cskv_index_topk_workspace_size(B, max_ctx_len, ratio, Hi, k))


def index_topk(q_idx, w, keys, ctx_len, ratio, k, max_ctx_len, topk_idx=None, topk_score=None,
               workspace=None, want_scores=True, stream=None):
    """Lightning-indexer top-k; returns (topk_idx int32 [B, k], topk_score fp32 [B, k] or None)."""
    import torch
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(w, torch.float32, "w")
    _need(ctx_len, torch.int32, "ctx_len")
    B, Hi, _ = q_idx.shape
    dev = q_idx.device
    if topk_idx is None:
        topk_idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    if topk_score is None and want_scores:
        topk_score = torch.empty((B, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(index_topk_workspace_size(B, max_ctx_len, ratio, Hi, k),
                                dtype=torch.uint8, device=dev)
    st = _lib.lib().cskv_index_topk(q_idx.data_ptr(), w.data_ptr(), keys.desc(), ctx_len.data_ptr(),
                                    B, Hi, int(ratio), int(k), int(max_ctx_len), topk_idx.data_ptr(),
                                    _ptr(topk_score), workspace.data_ptr(), workspace.numel(),
                                    _stream(stream))
    _check(st, "cskv_index_topk")
    return topk_idx, topk_score


def sparse_decode_attn_workspace_size(B, H, max_ctx_len, ratio, k):
    return int(_lib.lib().cskv_sparse_decode_attn_workspace_size(B, H, max_ctx_len, ratio, k))


def sparse_decode_attn(q, main_kv, swa, swa_fmt, ctx_len, topk_idx, k, ratio, max_ctx_len, sink,
                       softmax_scale, q_rope_cs, out=None, workspace=None, stream=None):
    """Shared-KV decode attention; returns out bf16 [B, H, 512]."""
    import torch
    _need(q, torch.bfloat16, "q")
    _need(swa, torch.uint8, "swa")
    _need(ctx_len, torch.int32, "ctx_len")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(sink, torch.float32, "sink")
    _need(q_rope_cs, torch.float32, "q_rope_cs")
    B, H, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    kk = int(k) if topk_idx is not None else 0
    if workspace is None:
        workspace = torch.empty(sparse_decode_attn_workspace_size(B, H, max_ctx_len, ratio, kk),
                                dtype=torch.uint8, device=q.device)
    st = _lib.lib().cskv_sparse_decode_attn(q.data_ptr(), main_kv.desc(), swa.data_ptr(), int(swa_fmt),
                                            ctx_len.data_ptr(), _ptr(topk_idx), kk, int(ratio),
                                            int(max_ctx_len), _ptr(sink), float(softmax_scale),
                                            q_rope_cs.data_ptr(), B, H, out.data_ptr(),
                                            workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(st, "cskv_sparse_decode_attn")
    return out


def sparse_prefill_attn(q, main_kv, window, pos1, topk_idx, k, ratio, max_ctx_len, sink, softmax_scale,
                        q_rope_cs, req_of=None, out=None, workspace=None, stream=None):
    """The attention of many prompt queries; query i of request req_of[i] sits at position
    pos1[i] - 1 and reads its window from `window` (raw rows by position).  Returns out
    bf16 [T, H, 512]."""
    import torch
    _need(q, torch.bfloat16, "q")
    _need(pos1, torch.int32, "pos1")
    _need(req_of, torch.int32, "req_of")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(sink, torch.float32, "sink")
    _need(q_rope_cs, torch.float32, "q_rope_cs")
    T, H, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    kk = int(k) if topk_idx is not None else 0
    if workspace is None:
        workspace = torch.empty(sparse_decode_attn_workspace_size(T, H, max_ctx_len, ratio, kk),
                                dtype=torch.uint8, device=q.device)
    st = _lib.lib().cskv_sparse_prefill_attn(q.data_ptr(), main_kv.desc(), window.desc(), _ptr(req_of),
                                             pos1.data_ptr(), _ptr(topk_idx), kk, int(ratio), int(max_ctx_len),
                                             _ptr(sink), float(softmax_scale), q_rope_cs.data_ptr(), T, H,
                                             out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                             _stream(stream))
    _check(st, "cskv_sparse_prefill_attn")
    return out


def decode_layer(jobs, q_idx, w, keys, q, main_kv, swa, swa_fmt, ctx_len, k, ratio, max_ctx_len, sink,
                 softmax_scale, q_rope_cs, topk_idx=None, out=None, index_workspace=None, attn_workspace=None,
                 h_in=None, d_in=None, h_out=None, stream=None):
    """One decode step of one layer in one call (cskv_decode_layer): h_in (host uint8) is
    copied into d_in (device uint8, which the other tensors may view), then compress_many(jobs)
    (jobs may be empty), index_topk (skipped when q_idx is None: HCA) and sparse_decode_attn
    run, and out is copied into h_out (host, out's dtype and size or less) last.  Host
    buffers should be pinned; q, and the jobs' kv, gate, prev_kv, prev_gate and
    rope_cs, may be pinned host tensors (read in place by the attention and the
    compressor).  Returns (out, topk_idx); h_out holds the output once the stream has
    synchronised."""
    import torch
    for t, dt, n in ((q_idx, torch.bfloat16, "q_idx"), (w, torch.float32, "w"),
                     (swa, torch.uint8, "swa"), (ctx_len, torch.int32, "ctx_len"), (sink, torch.float32, "sink"),
                     (q_rope_cs, torch.float32, "q_rope_cs"), (d_in, torch.uint8, "d_in")):
        _need(t, dt, n)
    _need(q, torch.bfloat16, "q", device=False)
    if not q.is_cuda and not q.is_pinned():
        raise ValueError("q must be a CUDA tensor or a pinned host tensor")
    _need(h_in, torch.uint8, "h_in", device=False)
    _need(h_out, None, "h_out", device=False)
    for t, n in ((h_in, "h_in"), (h_out, "h_out")):
        if t is not None and t.is_cuda:
            raise ValueError("%s must be a host tensor" % n)
    if h_in is not None and (d_in is None or d_in.numel() < h_in.numel()):
        raise ValueError("d_in must be a device buffer at least as large as h_in")
    B, H, _ = q.shape
    dev = ctx_len.device
    csa = q_idx is not None
    Hi = q_idx.shape[1] if csa else 0
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    if csa and topk_idx is None:
        topk_idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    if csa and index_workspace is None:
        index_workspace = torch.empty(index_topk_workspace_size(B, max_ctx_len, ratio, Hi, k), dtype=torch.uint8,
                                      device=dev)
    kk = int(k) if csa else 0
    if attn_workspace is None:
        attn_workspace = torch.empty(sparse_decode_attn_workspace_size(B, H, max_ctx_len, ratio, kk),
                                     dtype=torch.uint8, device=dev)
    arr = _compress_jobs(jobs, host_inputs=True)
    empty = _lib.Paged(None, None, 0, 0, 0, 0, 128)
    a = _lib.DecodeLayerArgs(
        ctypes.cast(arr, ctypes.POINTER(_lib.CompressJob)) if jobs else None, len(jobs), _ptr(q_idx), _ptr(w), keys.desc() if csa else empty, Hi, kk,
        _ptr(topk_idx) if csa else None, _ptr(index_workspace) if csa else None,
        index_workspace.numel() if csa else 0, q.data_ptr(), main_kv.desc(), swa.data_ptr(), int(swa_fmt),
        ctx_len.data_ptr(), int(ratio), int(max_ctx_len), _ptr(sink), float(softmax_scale), q_rope_cs.data_ptr(),
        B, H, out.data_ptr(), attn_workspace.data_ptr(), attn_workspace.numel(),
        _ptr(h_in), _ptr(d_in), h_in.numel() if h_in is not None else 0,
        _ptr(h_out), h_out.numel() * h_out.element_size() if h_out is not None else 0)
    st = _lib.lib().cskv_decode_layer(ctypes.byref(a), _stream(stream))
    _check(st, "cskv_decode_layer")
    return out, topk_idx


DEFAULT_SCALE = 1.0 / math.sqrt(512.0)
