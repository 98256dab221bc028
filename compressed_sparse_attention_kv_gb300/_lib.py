"""ctypes view of libcskv.so (the C ABI declared in include/cskv.h)."""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcskv.so")

c_int32 = ctypes.c_int32
c_int64 = ctypes.c_int64
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p
c_float = ctypes.c_float


class Paged(ctypes.Structure):
    """struct cskv_paged."""
    _fields_ = [
        ("pool", c_void_p),
        ("block_table", c_void_p),
        ("page_bytes", c_int64),
        ("num_pages", c_int32),
        ("max_pages", c_int32),
        ("fmt", c_int32),
        ("dim", c_int32),
    ]


class CompressJob(ctypes.Structure):
    """struct cskv_compress_job (the arguments of one cskv_compress call)."""
    _fields_ = [
        ("kv", c_void_p),
        ("gate", c_void_p),
        ("prev_kv", c_void_p),
        ("prev_gate", c_void_p),
        ("ape", c_void_p),
        ("norm_w", c_void_p),
        ("eps", c_float),
        ("rope_cs", c_void_p),
        ("S", c_int32),
        ("T", c_int32),
        ("ratio", c_int32),
        ("overlap", c_int32),
        ("dim", c_int32),
        ("req", c_void_p),
        ("first_entry", c_void_p),
        ("out", Paged),
    ]


class DecodeJob(ctypes.Structure):
    """struct cskv_decode_job (one compressor, or the window, of a decode step)."""
    _fields_ = [
        ("kv", c_void_p),
        ("gate", c_void_p),
        ("state_kv", c_void_p),
        ("state_gate", c_void_p),
        ("ape", c_void_p),
        ("norm_w", c_void_p),
        ("eps", c_float),
        ("rope_cs", c_void_p),
        ("ratio", c_int32),
        ("overlap", c_int32),
        ("dim", c_int32),
        ("ring_rows", c_int32),
        ("out", Paged),
    ]


class DecodeLayerArgs(ctypes.Structure):
    """struct cskv_decode_layer_args (one decode step of one layer, host to host)."""
    _fields_ = [
        ("jobs", ctypes.POINTER(CompressJob)),
        ("njobs", c_int32),
        ("q_idx", c_void_p),
        ("w", c_void_p),
        ("keys", Paged),
        ("Hi", c_int32),
        ("k", c_int32),
        ("topk_idx", c_void_p),
        ("index_workspace", c_void_p),
        ("index_workspace_bytes", c_size_t),
        ("q", c_void_p),
        ("main_kv", Paged),
        ("swa", c_void_p),
        ("swa_fmt", c_int32),
        ("ctx_len", c_void_p),
        ("ratio", c_int32),
        ("max_ctx_len", c_int32),
        ("sink", c_void_p),
        ("softmax_scale", c_float),
        ("q_rope_cs", c_void_p),
        ("B", c_int32),
        ("H", c_int32),
        ("out", c_void_p),
        ("attn_workspace", c_void_p),
        ("attn_workspace_bytes", c_size_t),
        ("h_in", c_void_p),
        ("d_in", c_void_p),
        ("in_bytes", c_size_t),
        ("h_out", c_void_p),
        ("out_bytes", c_size_t),
    ]


# name -> (restype, argtypes); every symbol include/cskv.h declares
SIGNATURES = {
    "cskv_row_bytes": (c_size_t, [c_int32, c_int32]),
    "cskv_status_string": (ctypes.c_char_p, [c_int32]),
    "cskv_version": (c_int32, []),
    "cskv_device_status": (c_int32, [c_void_p]),
    "cskv_set_spin_limit": (None, [ctypes.c_uint64]),
    "cskv_set_timing_events": (None, [c_void_p, c_void_p]),
    "cskv_rope_table": (c_int32, [c_void_p, c_int32, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                  ctypes.c_double, ctypes.c_double, c_void_p]),
    "cskv_encode_rows": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, Paged,
                                   c_void_p]),
    "cskv_compress": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_float,
                                c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p,
                                c_void_p, Paged, c_void_p]),
    "cskv_compress_many": (c_int32, [ctypes.POINTER(CompressJob), c_int32, c_void_p]),
    "cskv_decode_append": (c_int32, [ctypes.POINTER(DecodeJob), c_int32, c_void_p, c_int32, c_void_p]),
    "cskv_index_topk_workspace_size": (c_size_t, [c_int32, c_int32, c_int32, c_int32, c_int32]),
    "cskv_index_topk": (c_int32, [c_void_p, c_void_p, Paged, c_void_p, c_int32, c_int32, c_int32,
                                  c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "cskv_index_topk_noalloc": (c_int32, [c_void_p, c_void_p, Paged, c_void_p, c_int32, c_int32, c_int32,
                                          c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "cskv_sparse_decode_attn_workspace_size": (c_size_t, [c_int32, c_int32, c_int32, c_int32, c_int32]),
    "cskv_sparse_decode_attn": (c_int32, [c_void_p, Paged, c_void_p, c_int32, c_void_p, c_void_p,
                                          c_int32, c_int32, c_int32, c_void_p, c_float, c_void_p,
                                          c_int32, c_int32, c_void_p, c_void_p, c_size_t, c_void_p]),
    "cskv_sparse_prefill_attn": (c_int32, [c_void_p, Paged, Paged, c_void_p, c_void_p, c_void_p, c_int32,
                                           c_int32, c_int32, c_void_p, c_float, c_void_p, c_int32, c_int32,
                                           c_void_p, c_void_p, c_size_t, c_void_p]),
    "cskv_decode_layer": (c_int32, [ctypes.POINTER(DecodeLayerArgs), c_void_p]),
}

_lib = None


def lib():
    """The loaded library; raises if libcskv.so has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libcskv.so is missing at %s: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback for the decode path)" % LIB_PATH)
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib
