"""The C-ABI library: it builds, loads without a GPU, exports every symbol include/cskv.h
declares, and rejects bad arguments on the host before any launch (CPU only)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_kv_gb300 import build, _lib
    build.build()
    return _lib.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "cskv.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"CSKV_API\s+[\w\s\*]+?\b(cskv_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    from compressed_sparse_attention_kv_gb300 import _lib
    names = _declared()
    assert len(names) == 18
    assert sorted(_lib.SIGNATURES) == names


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    out = os.popen("nm -D --defined-only %s" % os.path.join(ROOT, "compressed_sparse_attention_kv_gb300",
                                                             "libcskv.so")).read()
    exported = set(re.findall(r"\bT (cskv_\w+)", out))
    assert exported == set(_declared())


def test_row_bytes_and_status(lib):
    assert lib.cskv_row_bytes(1, 512) == 528
    assert lib.cskv_row_bytes(2, 512) == 288
    assert lib.cskv_row_bytes(0, 512) == 1024
    assert lib.cskv_row_bytes(3, 128) == 132
    assert lib.cskv_row_bytes(1, 100) == 0
    assert lib.cskv_status_string(0) == b"ok"
    assert lib.cskv_version() >= 100


def test_workspace_sizes(lib):
    small = lib.cskv_index_topk_workspace_size(1, 4096, 4, 4, 512)
    big = lib.cskv_index_topk_workspace_size(8, 1 << 20, 4, 64, 512)
    assert 0 < small < big
    # scores + candidates dominate: 12 bytes per visible entry
    assert big >= 8 * (1 << 18) * 12
    # bf16 partials (O / l) of every (request, tile, head) plus fp32 (m, l)
    assert lib.cskv_sparse_decode_attn_workspace_size(8, 64, 1 << 20, 4, 512) >= 8 * 5 * 64 * (512 * 2 + 8)
    assert lib.cskv_index_topk_workspace_size(0, 10, 4, 4, 4) == 0


def test_invalid_arguments_launch_nothing(lib):
    from compressed_sparse_attention_kv_gb300._lib import Paged
    bad = Paged(None, None, 0, 0, 0, 1, 512)
    # null required pointers / bad sizes -> CSKV_ERR_INVALID (1), checked before any CUDA call
    assert lib.cskv_compress(None, None, None, None, None, None, 1e-6, None, 1, 4, 4, 1, 512,
                             None, None, bad, None) == 1
    fake = ctypes.c_void_p(4096)
    good = Paged(4096, None, 64 * 528, 4, 0, 1, 512)
    assert lib.cskv_compress(fake, fake, None, None, fake, None, 1e-6, None, 1, 6, 4, 1, 512,
                             fake, fake, good, None) == 1                      # T % ratio != 0
    assert lib.cskv_compress(fake, fake, None, None, fake, None, 1e-6, None, 1, 128, 128, 1, 512,
                             fake, fake, good, None) == 1                      # overlap needs ratio <= 8
    assert lib.cskv_compress(fake, fake, None, None, fake, None, -1.0, None, 1, 8, 4, 1, 512,
                             fake, fake, good, None) == 1                      # eps < 0
    assert lib.cskv_compress_many(None, 1, None) == 1                          # no jobs
    from compressed_sparse_attention_kv_gb300._lib import CompressJob
    jobs = (CompressJob * 5)()
    assert lib.cskv_compress_many(jobs, 5, None) == 1                          # more than 4 jobs
    jobs[0] = CompressJob(4096, 4096, None, None, 4096, None, 1e-6, None, 1, 6, 4, 1, 512, 4096, 4096, good)
    assert lib.cskv_compress_many(jobs, 1, None) == 1                          # T % ratio != 0
    from compressed_sparse_attention_kv_gb300._lib import DecodeJob
    dj = (DecodeJob * 9)()
    assert lib.cskv_decode_append(dj, 9, fake, 2, None) == 1                     # more than 8 jobs
    dj[0] = DecodeJob(4096, 4096, None, None, None, None, 1e-6, None, 4, 1, 512, 0, good)
    assert lib.cskv_decode_append(dj, 1, fake, 2, None) == 1                     # ratio 4 without a state ring
    dj[0] = DecodeJob(4096, None, 4096, 4096, None, None, 1e-6, None, 4, 1, 512, 0, good)
    assert lib.cskv_decode_append(dj, 1, fake, 2, None) == 1                     # ratio 4 without a gate
    dj[0] = DecodeJob(4096, 4096, 4096, 4096, None, None, 1e-6, None, 4, 1, 512, 128, good)
    assert lib.cskv_decode_append(dj, 1, fake, 2, None) == 1                     # a ring needs ratio 1
    dj[0] = DecodeJob(4096, None, None, None, None, None, 1e-6, None, 1, 1, 512, 128, good)
    assert lib.cskv_decode_append(dj, 1, fake, 2, None) == 1                     # overlap needs ratio 2..8
    dj[0] = DecodeJob(4096, None, None, None, None, None, 1e-6, None, 1, 0, 512, 128, good)
    assert lib.cskv_decode_append(dj, 1, None, 2, None) == 1                     # no positions
    assert lib.cskv_decode_append(dj, 1, None, 0, None) == 0                     # empty batch: nothing to do
    keys = Paged(4096, 4096, 64 * 132, 4, 4, 3, 128)
    assert lib.cskv_index_topk(fake, fake, keys, fake, 1, 65, 4, 512, 4096, fake, None, fake, 1 << 30,
                               None) == 2                                       # > 64 heads
    assert lib.cskv_index_topk(fake, fake, keys, fake, 1, 4, 4, 4096, 4096, fake, None, fake, 1 << 30,
                               None) == 1                                       # k > 2048
    assert lib.cskv_index_topk(fake, fake, keys, fake, 1, 4, 4, 512, 4096, fake, None, fake, 16,
                               None) == 1                                       # workspace too small
    main = Paged(4096, 4096, 64 * 528, 4, 4, 3, 512)                           # page-split is not a main format
    assert lib.cskv_sparse_decode_attn(fake, main, fake, 1, fake, None, 0, 128, 4096, None, 0.04, fake,
                                       1, 64, fake, fake, 1 << 30, None) == 1
    main = Paged(4096, 4096, 64 * 528, 4, 4, 1, 512)
    assert lib.cskv_sparse_decode_attn(fake, main, fake, 2, fake, None, 0, 128, 4096, None, 0.04, fake,
                                       1, 64, fake, fake, 1 << 30, None) == 1    # FP4 window not allowed
    assert lib.cskv_sparse_decode_attn(fake, main, fake, 1, fake, None, 0, 128, 4096, None, 0.04, fake,
                                       1, 129, fake, fake, 1 << 30, None) == 1   # H > 128
    # the layer step checks every stage before it enqueues anything
    from compressed_sparse_attention_kv_gb300._lib import DecodeLayerArgs
    assert lib.cskv_decode_layer(None, None) == 1
    la = DecodeLayerArgs()
    la.q, la.main_kv, la.swa, la.swa_fmt, la.ctx_len = 4096, main, 4096, 1, 4096
    la.ratio, la.max_ctx_len, la.softmax_scale, la.q_rope_cs, la.B, la.H = 128, 4096, 0.04, 4096, 1, 64
    la.out, la.attn_workspace, la.attn_workspace_bytes = 4096, 4096, 1 << 30
    la.njobs = 5
    assert lib.cskv_decode_layer(ctypes.byref(la), None) == 1                  # more than 4 jobs
    la.njobs = 1
    assert lib.cskv_decode_layer(ctypes.byref(la), None) == 1                  # jobs NULL
    la.njobs = 0
    la.H = 129
    assert lib.cskv_decode_layer(ctypes.byref(la), None) == 1                  # the attention's H > 128
    la.H = 64
    la.q_idx, la.w, la.keys, la.Hi, la.k, la.topk_idx = 4096, 4096, keys, 65, 512, 4096
    la.index_workspace, la.index_workspace_bytes = 4096, 1 << 30
    assert lib.cskv_decode_layer(ctypes.byref(la), None) == 2                  # the indexer's > 64 heads
    la.Hi = 4
    la.in_bytes = 1024
    assert lib.cskv_decode_layer(ctypes.byref(la), None) == 1                  # input bytes without buffers
    la.in_bytes, la.h_out, la.out_bytes = 0, 4096, 64 * 512 * 2 + 2
    assert lib.cskv_decode_layer(ctypes.byref(la), None) == 1                  # more bytes out than the output


def test_binding_refuses_without_library(tmp_path, monkeypatch):
    from compressed_sparse_attention_kv_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()


def test_binding_refuses_host_tensors_for_device_arguments(lib):
    """No silent CPU path: caches and every entry point's device arguments must be CUDA
    tensors, and the binding says so before anything reaches the library."""
    import torch
    import compressed_sparse_attention_kv_gb300 as cskv
    with pytest.raises(ValueError, match="CUDA tensor"):
        cskv.PagedCache(torch.zeros((1, 64 * 132), dtype=torch.uint8), torch.zeros((1, 1), dtype=torch.int32),
                        cskv.FMT_FP8_PAGESPLIT, 128)
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16)
    w = torch.zeros((1, 4), dtype=torch.float32)
    ctx = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cskv.index_topk(q, w, None, ctx, 4, 1, 4)
    qa = torch.zeros((1, 16, 512), dtype=torch.bfloat16)
    swa = torch.zeros((1, 128, 528), dtype=torch.uint8)
    cs = torch.zeros((1, 32, 2), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cskv.sparse_decode_attn(qa, None, swa, cskv.FMT_FP8, ctx, None, 0, 128, 4, None, 0.04, cs)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cskv.decode_layer([], None, None, None, qa, None, swa, cskv.FMT_FP8, ctx, 0, 128, 4, None, 0.04, cs)


def test_rope_table_is_host_code_and_checks_its_arguments(lib):
    """cskv_rope_table runs on the host (no GPU here) and rejects bad arguments."""
    import numpy as np
    pos = np.array([0, 1, 1 << 20], dtype=np.int64)
    out = np.zeros((3, 32, 2), dtype=np.float32)
    assert lib.cskv_rope_table(pos.ctypes.data, 3, 160000.0, 1.0, 1.0, 1.0, 1.0, out.ctypes.data) == 0
    assert out[0, :, 0].tolist() == [1.0] * 32 and out[0, :, 1].tolist() == [0.0] * 32
    assert lib.cskv_rope_table(None, 3, 160000.0, 1.0, 1.0, 1.0, 1.0, out.ctypes.data) == 1
    assert lib.cskv_rope_table(pos.ctypes.data, -1, 160000.0, 1.0, 1.0, 1.0, 1.0, out.ctypes.data) == 1
    assert lib.cskv_rope_table(pos.ctypes.data, 3, 1.0, 1.0, 1.0, 1.0, 1.0, out.ctypes.data) == 1
    assert lib.cskv_rope_table(pos.ctypes.data, 3, 160000.0, 16.0, 0.0, 32.0, 1.0, out.ctypes.data) == 1
    assert lib.cskv_rope_table(None, 0, 160000.0, 1.0, 1.0, 1.0, 1.0, None) == 0
