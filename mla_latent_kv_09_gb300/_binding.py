"""ctypes binding of libmla_decode.so: the C ABI of include/mla_decode.h.

Argument marshalling only.  Functions keep the C names and take either raw
integers (device pointers, sizes) or torch tensors, whose data pointers are
passed through.  Every step of the computation runs in the CUDA library;
there is no fallback: if the library cannot be loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libmla_decode.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE = 5
MLA_ERR_BAD_TABLE = 6
MLA_ERR_BAD_INDEX = 7
MLA_ERR_TIMEOUT = 8
MLA_ERR_VALUE_RANGE = 9

MLA_FLAG_CAUSAL = 1
MLA_FLAG_OUT_FP32 = 2
MLA_FLAG_VALIDATE = 4
MLA_FLAG_BF16_PV = 8
MLA_FLAG_KV_FP8 = 16

# every symbol the headers in include/ declare: name -> (restype, argtypes)
_c_int, _c_size, _vp, _i64, _f32, _uint = (ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p,
                                           ctypes.c_int64, ctypes.c_float, ctypes.c_uint)
SIGNATURES = {
    "mla_default_num_units": (_c_int, [_c_int, ctypes.POINTER(_c_int)]),
    "mla_decode_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "mla_decode_plan": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
    "mla_decode_plan_host": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "mla_decode": (_c_int, [_vp, _vp, _i64, _vp, _i64, _vp, _c_int, _c_int, _c_int, _f32, _vp, _c_int,
                            _uint, _c_int, _vp, _c_size, _vp, _vp, _vp]),
    "mla_combine": (_c_int, [_vp, _c_size, _c_int, _c_int, _c_int, _uint, _c_int, _vp, _vp, _vp]),
    "mla_workspace_status": (_c_int, [_vp, _vp]),
    "mla_selftest_wait_timeout": (_c_int, [_vp, _c_size, _vp]),
    "mla_decode_noalloc": (_c_int, [_vp, _vp, _i64, _vp, _i64, _vp, _c_int, _c_int, _c_int, _f32, _vp, _c_int,
                                    _uint, _vp, _vp, _vp]),
    "mla_noalloc_status": (_c_int, [_vp]),
    "mla_noalloc_workspace": (_c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_c_size)]),
    "mla_status_string": (ctypes.c_char_p, [_c_int]),
    "mla_absorb_q": (_c_int, [_vp, _vp, _i64, _vp, _c_int, _c_int, _vp, _i64, _vp, _vp]),
    "mla_absorb_o": (_c_int, [_vp, _i64, _vp, _c_int, _c_int, _vp, _i64, _vp, _vp]),
    "mla_indexer_scores": (_c_int, [_vp, _vp, _vp, _i64, _vp, _i64, _vp, _c_int, _c_int, _uint, _c_int, _vp, _i64,
                                    _vp, _vp]),
    "mla_topk": (_c_int, [_vp, _i64, _vp, _c_int, _c_int, _uint, _c_int, _c_int, _vp, _vp, _vp]),
}

_lib = None


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


def load(path: str = LIB_PATH):
    """Load the shared library (once) and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with mla_latent_kv_09_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(fn: str, rc: int):
    if rc != MLA_OK:
        raise MlaError(fn, rc)


def status_string(status: int) -> str:
    return load().mla_status_string(int(status)).decode()


def mla_status_string(status: int) -> str:
    return status_string(status)


def mla_default_num_units(s_q: int) -> int:
    err = ctypes.c_int(0)
    u = load().mla_default_num_units(int(s_q), ctypes.byref(err))
    _check("mla_default_num_units", err.value)
    return u


def mla_decode_workspace_size(batch: int, s_q: int, num_heads: int = 128, num_units: int = 0) -> int:
    n = load().mla_decode_workspace_size(int(batch), int(s_q), int(num_heads), int(num_units))
    if n == 0:
        raise MlaError("mla_decode_workspace_size", MLA_ERR_INVALID_ARG)
    return n


def mla_decode_plan(cache_lens, batch: int, s_q: int, topk: int, num_units: int, workspace,
                    ws_bytes: int, stream=None) -> None:
    _check("mla_decode_plan", load().mla_decode_plan(
        _ptr(cache_lens), int(batch), int(s_q), int(topk), int(num_units), _ptr(workspace),
        int(ws_bytes), _stream(stream)))


def mla_decode_plan_host(cache_lens, s_q: int, topk: int, num_units: int):
    """Host-side partition: returns (unit_meta [U,5], req_meta [B,4]) as numpy int32."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(cache_lens, dtype=np.int32))
    B = lens.size
    um = np.zeros((num_units, 5), np.int32)
    rm = np.zeros((B, 4), np.int32)
    rc = load().mla_decode_plan_host(lens.ctypes.data, B, int(s_q), int(topk), int(num_units),
                                     um.ctypes.data, rm.ctypes.data)
    _check("mla_decode_plan_host", rc)
    return um, rm


def mla_decode(q, kv_cache, num_pages: int, block_table, bt_stride: int, cache_lens, batch: int,
               s_q: int, num_heads: int, softmax_scale: float, topk_idx, topk: int, flags: int,
               num_units: int, workspace, ws_bytes: int, out, lse, stream=None) -> None:
    _check("mla_decode", load().mla_decode(
        _ptr(q), _ptr(kv_cache), int(num_pages), _ptr(block_table), int(bt_stride), _ptr(cache_lens),
        int(batch), int(s_q), int(num_heads), float(softmax_scale), _ptr(topk_idx), int(topk),
        int(flags), int(num_units), _ptr(workspace), int(ws_bytes), _ptr(out), _ptr(lse),
        _stream(stream)))


def mla_combine(workspace, ws_bytes: int, batch: int, s_q: int, num_heads: int, flags: int,
                num_units: int, out, lse, stream=None) -> None:
    _check("mla_combine", load().mla_combine(
        _ptr(workspace), int(ws_bytes), int(batch), int(s_q), int(num_heads), int(flags),
        int(num_units), _ptr(out), _ptr(lse), _stream(stream)))


def mla_decode_noalloc(q, kv_cache, num_pages: int, block_table, bt_stride: int, cache_lens, batch: int,
                       s_q: int, num_heads: int, softmax_scale: float, topk_idx, topk: int, flags: int,
                       out, lse, stream=None) -> None:
    """The decode step with the library's built-in workspace (allocates nothing)."""
    _check("mla_decode_noalloc", load().mla_decode_noalloc(
        _ptr(q), _ptr(kv_cache), int(num_pages), _ptr(block_table), int(bt_stride), _ptr(cache_lens),
        int(batch), int(s_q), int(num_heads), float(softmax_scale), _ptr(topk_idx), int(topk), int(flags),
        _ptr(out), _ptr(lse), _stream(stream)))


def mla_workspace_status(workspace, stream=None) -> int:
    return load().mla_workspace_status(_ptr(workspace), _stream(stream))


def mla_selftest_wait_timeout(workspace, ws_bytes: int, stream=None) -> None:
    _check("mla_selftest_wait_timeout",
           load().mla_selftest_wait_timeout(_ptr(workspace), int(ws_bytes), _stream(stream)))


def mla_noalloc_status(stream=None) -> int:
    """Status word of mla_decode_noalloc's built-in workspace (synchronises the stream)."""
    return load().mla_noalloc_status(_stream(stream))


def mla_noalloc_workspace():
    """(device address, bytes) of mla_decode_noalloc's built-in workspace on the current device."""
    ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check("mla_noalloc_workspace", load().mla_noalloc_workspace(ctypes.byref(ptr), ctypes.byref(n)))
    return ptr.value, n.value


def mla_absorb_q(q_nope, q_pe, q_stride: int, w_uk, num_tokens: int, num_heads: int, out, out_stride: int,
                 status, stream=None) -> None:
    _check("mla_absorb_q", load().mla_absorb_q(
        _ptr(q_nope), _ptr(q_pe), int(q_stride), _ptr(w_uk), int(num_tokens), int(num_heads), _ptr(out),
        int(out_stride), _ptr(status), _stream(stream)))


def mla_absorb_o(o, o_stride: int, w_uv, num_tokens: int, num_heads: int, out, out_stride: int, status,
                 stream=None) -> None:
    _check("mla_absorb_o", load().mla_absorb_o(
        _ptr(o), int(o_stride), _ptr(w_uv), int(num_tokens), int(num_heads), _ptr(out), int(out_stride),
        _ptr(status), _stream(stream)))


def mla_indexer_scores(q_idx, w_idx, k_idx_cache, num_pages: int, block_table, bt_stride: int, cache_lens,
                       batch: int, s_q: int, flags: int, max_len: int, scores, scores_stride: int, status,
                       stream=None) -> None:
    _check("mla_indexer_scores", load().mla_indexer_scores(
        _ptr(q_idx), _ptr(w_idx), _ptr(k_idx_cache), int(num_pages), _ptr(block_table), int(bt_stride),
        _ptr(cache_lens), int(batch), int(s_q), int(flags), int(max_len), _ptr(scores), int(scores_stride),
        _ptr(status), _stream(stream)))


def mla_topk(scores, scores_stride: int, cache_lens, batch: int, s_q: int, flags: int, max_len: int, topk: int,
             out_idx, status, stream=None) -> None:
    _check("mla_topk", load().mla_topk(
        _ptr(scores), int(scores_stride), _ptr(cache_lens), int(batch), int(s_q), int(flags), int(max_len),
        int(topk), _ptr(out_idx), _ptr(status), _stream(stream)))
