"""ctypes binding of the lat_attn C ABI (include/lat_attn.h).

Argument marshalling only: every function forwards to the CUDA library under the same
name and argument order.  Pointer arguments accept a torch tensor (its data_ptr), an int
address or None (NULL); ``stream`` accepts a torch.cuda.Stream, an int handle or None
(torch's current stream when CUDA is up, else the legacy default stream).  A non-OK
status raises LatError.  There is no CPU fallback: if the library is not built, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblat_attn.so")

LAT_F32, LAT_BF16 = 0, 1
STATUS_NAMES = {0: "LAT_OK", 1: "LAT_ERR_INVALID_ARG", 2: "LAT_ERR_UNSUPPORTED",
                3: "LAT_ERR_WORKSPACE", 4: "LAT_ERR_CUDA", 5: "LAT_ERR_BOUNDS",
                6: "LAT_ERR_TIMEOUT"}
(LAT_OK, LAT_ERR_INVALID_ARG, LAT_ERR_UNSUPPORTED, LAT_ERR_WORKSPACE, LAT_ERR_CUDA,
 LAT_ERR_BOUNDS, LAT_ERR_TIMEOUT) = range(7)


class LatError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS_NAMES.get(status, str(status))))


_lock = threading.Lock()
_lib = None

_P, _I64, _I32, _F32, _SZ, _U64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64)
_SIGNATURES = {
    "lat_status_string": (ctypes.c_char_p, [_I32]),
    "lat_attn_prefill": (_I32, [_I32, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _P,
                                _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P]),
    "lat_attn_prefill_cached": (_I32, [_I32, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I64, _P,
                                       _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P,
                                       _P]),
    "lat_attn_prefill_softcap": (_I32, [_I32, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _P,
                                        _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F32,
                                        _F32, _P, _P]),
    "lat_attn_decode_softcap": (_I32, [_I32, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I32, _P,
                                       _I64, _P, _I32, _I32, _I32, _I32, _I32, _F32, _F32, _P,
                                       _SZ, _P, _P]),
    "lat_attn_decode_ring": (_I32, [_I32, _P, _I64, _P, _P, _I64, _I64, _I64, _I32, _P, _I32,
                                    _P, _I64, _P, _I32, _I32, _I32, _I32, _I32, _F32, _P, _SZ,
                                    _P, _P]),
    "lat_kv_append_ring": (_I32, [_I32, _P, _P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _I32,
                                  _I32, _I32, _I32, _P, _P]),
    "lat_qkv_norm_rope_append": (_I32, [_I32, _P, _I64, _P, _P, _F32, ctypes.c_double, _I32,
                                        _P, _I64, _P, _P, _I64, _I64, _I64, _I32, _P, _I32,
                                        _I32, _I32, _I32, _I32, _P, _P]),
    "lat_attn_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "lat_attn_decode": (_I32, [_I32, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I32, _P, _I64,
                               _P, _I32, _I32, _I32, _I32, _I32, _F32, _P, _SZ, _P, _P]),
    "lat_attn_decode_static": (_I32, [_I32, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I32, _P,
                                      _I64, _P, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P]),
    "lat_kv_append": (_I32, [_I32, _P, _P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _I32,
                             _I32, _I32, _I32, _P, _P]),
    "lat_test_prefill_timeout": (_I32, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _I32, _I32,
                                        _I32, _I32, _I32, _U64, _P, _P]),
    "lat_test_decode_timeout": (_I32, [_P, _I64, _P, _P, _I64, _I64, _I64, _P, _I32, _P, _I64,
                                       _I32, _I32, _I32, _I32, _P, _SZ, _U64, _P, _P]),
    "lat_test_capped_scores": (_I32, [_P, _I64, _F32, _F32, _P, _P]),
}


def library(path: str = LIB_PATH) -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError("lat_attn CUDA library missing at %s; build it with "
                                   "`python -m gqa_attention_lat_gb300.build`" % path)
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_initialized() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str):
    if st != LAT_OK:
        raise LatError(st, where)


def lat_status_string(status: int) -> str:
    return library().lat_status_string(status).decode()


def lat_attn_prefill(dt, q, q_rs, k, k_rs, v, v_rs, out, out_rs, lse, batch, seq_len, kv_len,
                     n_heads, n_kv_heads, head_dim, causal, window, scale, status=None,
                     stream=None):
    _check(library().lat_attn_prefill(
        dt, _ptr(q), q_rs, _ptr(k), k_rs, _ptr(v), v_rs, _ptr(out), out_rs, _ptr(lse), batch,
        seq_len, kv_len, n_heads, n_kv_heads, head_dim, int(bool(causal)), window, scale,
        _ptr(status), _stream(stream)), "lat_attn_prefill")


def lat_attn_prefill_softcap(dt, q, q_rs, k, k_rs, v, v_rs, out, out_rs, lse, batch, seq_len,
                             kv_len, n_heads, n_kv_heads, head_dim, causal, window, scale,
                             softcap, status=None, stream=None):
    _check(library().lat_attn_prefill_softcap(
        dt, _ptr(q), q_rs, _ptr(k), k_rs, _ptr(v), v_rs, _ptr(out), out_rs, _ptr(lse), batch,
        seq_len, kv_len, n_heads, n_kv_heads, head_dim, int(bool(causal)), window, scale,
        softcap, _ptr(status), _stream(stream)), "lat_attn_prefill_softcap")


def lat_attn_decode_softcap(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                            cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch,
                            n_heads, n_kv_heads, head_dim, window, scale, softcap, workspace,
                            workspace_bytes, status=None, stream=None):
    _check(library().lat_attn_decode_softcap(
        dt, _ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride,
        cache_seq_stride, _ptr(kv_lens), max_kv_len, _ptr(out), out_rs, _ptr(lse), batch,
        n_heads, n_kv_heads, head_dim, window, scale, softcap, _ptr(workspace),
        workspace_bytes, _ptr(status), _stream(stream)), "lat_attn_decode_softcap")


def lat_attn_decode_ring(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                         cache_seq_stride, ring_capacity, kv_lens, max_kv_len, out, out_rs, lse,
                         batch, n_heads, n_kv_heads, head_dim, window, scale, workspace,
                         workspace_bytes, status=None, stream=None):
    _check(library().lat_attn_decode_ring(
        dt, _ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride,
        cache_seq_stride, ring_capacity, _ptr(kv_lens), max_kv_len, _ptr(out), out_rs,
        _ptr(lse), batch, n_heads, n_kv_heads, head_dim, window, scale, _ptr(workspace),
        workspace_bytes, _ptr(status), _stream(stream)), "lat_attn_decode_ring")


def lat_kv_append_ring(dt, k_cache, v_cache, cache_rs, cache_head_stride, cache_seq_stride,
                       ring_capacity, k_new, v_new, new_rs, pos, n_new, batch, n_kv_heads,
                       head_dim, status=None, stream=None):
    _check(library().lat_kv_append_ring(
        dt, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride, cache_seq_stride,
        ring_capacity, _ptr(k_new), _ptr(v_new), new_rs, _ptr(pos), n_new, batch, n_kv_heads,
        head_dim, _ptr(status), _stream(stream)), "lat_kv_append_ring")


def lat_qkv_norm_rope_append(dt, qkv, qkv_rs, q_norm_w, k_norm_w, eps, rope_base, v_unit_norm,
                             q_out, q_out_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                             cache_seq_stride, capacity, pos, n_new, batch, n_heads, n_kv_heads,
                             head_dim, status=None, stream=None):
    _check(library().lat_qkv_norm_rope_append(
        dt, _ptr(qkv), qkv_rs, _ptr(q_norm_w), _ptr(k_norm_w), eps, rope_base,
        int(bool(v_unit_norm)), _ptr(q_out), q_out_rs, _ptr(k_cache), _ptr(v_cache), cache_rs,
        cache_head_stride, cache_seq_stride, capacity, _ptr(pos), n_new, batch, n_heads,
        n_kv_heads, head_dim, _ptr(status), _stream(stream)), "lat_qkv_norm_rope_append")


def lat_attn_prefill_cached(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                            cache_seq_stride, out, out_rs, lse, batch, seq_len, kv_len, n_heads,
                            n_kv_heads, head_dim, causal, window, scale, status=None,
                            stream=None):
    _check(library().lat_attn_prefill_cached(
        dt, _ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride,
        cache_seq_stride, _ptr(out), out_rs, _ptr(lse), batch, seq_len, kv_len, n_heads,
        n_kv_heads, head_dim, int(bool(causal)), window, scale, _ptr(status), _stream(stream)),
        "lat_attn_prefill_cached")


def lat_attn_decode_workspace_size(dt, batch, n_heads, n_kv_heads, head_dim, max_kv_len) -> int:
    return library().lat_attn_decode_workspace_size(dt, batch, n_heads, n_kv_heads, head_dim,
                                                    max_kv_len)


def lat_attn_decode(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                    cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch, n_heads,
                    n_kv_heads, head_dim, window, scale, workspace, workspace_bytes,
                    status=None, stream=None):
    _check(library().lat_attn_decode(
        dt, _ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride,
        cache_seq_stride, _ptr(kv_lens), max_kv_len, _ptr(out), out_rs, _ptr(lse), batch,
        n_heads, n_kv_heads, head_dim, window, scale, _ptr(workspace), workspace_bytes,
        _ptr(status), _stream(stream)), "lat_attn_decode")


def lat_attn_decode_static(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                           cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch,
                           n_heads, n_kv_heads, head_dim, window, scale, status=None,
                           stream=None):
    """lat_attn_decode with the library's own fixed device scratch (no workspace)."""
    _check(library().lat_attn_decode_static(
        dt, _ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride,
        cache_seq_stride, _ptr(kv_lens), max_kv_len, _ptr(out), out_rs, _ptr(lse), batch,
        n_heads, n_kv_heads, head_dim, window, scale, _ptr(status), _stream(stream)),
        "lat_attn_decode_static")


def lat_kv_append(dt, k_cache, v_cache, cache_rs, cache_head_stride, cache_seq_stride,
                  capacity, k_new, v_new, new_rs, pos, n_new, batch, n_kv_heads, head_dim,
                  status=None, stream=None):
    _check(library().lat_kv_append(
        dt, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride, cache_seq_stride,
        capacity, _ptr(k_new), _ptr(v_new), new_rs, _ptr(pos), n_new, batch, n_kv_heads,
        head_dim, _ptr(status), _stream(stream)), "lat_kv_append")


def lat_test_prefill_timeout(q, q_rs, k, k_rs, v, v_rs, out, out_rs, batch, seq_len, n_heads,
                             n_kv_heads, head_dim, timeout_ns, status, stream=None):
    _check(library().lat_test_prefill_timeout(
        _ptr(q), q_rs, _ptr(k), k_rs, _ptr(v), v_rs, _ptr(out), out_rs, batch, seq_len,
        n_heads, n_kv_heads, head_dim, timeout_ns, _ptr(status), _stream(stream)),
        "lat_test_prefill_timeout")


def lat_test_decode_timeout(q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                            cache_seq_stride, kv_lens, max_kv_len, out, out_rs, batch, n_heads,
                            n_kv_heads, head_dim, workspace, workspace_bytes, timeout_ns, status,
                            stream=None):
    _check(library().lat_test_decode_timeout(
        _ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), cache_rs, cache_head_stride,
        cache_seq_stride, _ptr(kv_lens), max_kv_len, _ptr(out), out_rs, batch, n_heads,
        n_kv_heads, head_dim, _ptr(workspace), workspace_bytes, timeout_ns, _ptr(status),
        _stream(stream)), "lat_test_decode_timeout")


def lat_test_capped_scores(raw, n, scale, softcap, out, stream=None):
    _check(library().lat_test_capped_scores(_ptr(raw), n, scale, softcap, _ptr(out),
                                            _stream(stream)), "lat_test_capped_scores")
