"""Python face of the fp64 attention oracle (TEST INFRASTRUCTURE, not product code).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this module.  It shares nothing with the CUDA library: the arithmetic lives
in ``attention_oracle.c`` (plain double-precision loops) and this file only marshals
numpy arrays into it.

Functions
---------
prefill(q, k, v, causal, window, scale, rows=None, threads=None, softcap=0.0)
    The attention definition for every query row (or a subset of rows).
decode(q, k_cache, v_cache, kv_lens, window, scale, softcap=0.0)
    A decode step is the prefill definition with one query row whose position is the
    last cached key (query length 1, key length kv_len): the hf2q "Current Inference
    Path" page, section 3, runs the decode step as attention at seq_len 1 over the
    KV cache right after the cache append.
kv_append(k_cache, v_cache, k_new, v_new, pos)
    The in-place cache append of the same page (section 1, the in-place
    ``--kv-cache-kernel`` mode; section 3, "KV cache append"): rows
    ``pos[b] .. pos[b]+n_new-1`` of sequence b take the new rows.  A plain copy.
kv_append_ring(k_cache, v_cache, k_new, v_new, pos)
    The same copy into a ring cache of ``cap`` rows: position p goes to row p % cap.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_library(src: str, out: str) -> str:
    """gcc, IEEE double, no FMA contraction (the same bits on x86 and Arm)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
        "-shared", "-pthread", src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build_library(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_library(SOURCE, _LIB)
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor: take its values, exactly
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class Oracle:
    """The oracle functions bound to one compiled copy of ``attention_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        fn = lib.oracle_attention_rows
        fn.restype = ctypes.c_int
        P = ctypes.POINTER(ctypes.c_double)
        fn.argtypes = [P, P, P, P, P] + [ctypes.c_int] * 8 + [
            ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
            ctypes.c_int]
        self._fn = fn

    def prefill(self, q, k, v, *, causal: bool, window: int, scale: float, rows=None,
                threads=None, softcap: float = 0.0):
        """Softmax attention by definition, in double precision (scores capped as
        softcap * tanh(s / softcap) when softcap > 0).

        q: [B, S, Hq, D]; k, v: [B, L, Hkv, D].  Returns (out, lse) with out
        [B, S, Hq, D] and lse [B, S, Hq] when ``rows`` is None, else out [n, Hq, D] and
        lse [n, Hq] for the flattened query rows ``rows`` (row r = b*S + i).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, S, Hq, D = q.shape
        Bk, L, Hkv, Dk = k.shape
        if v.shape != k.shape or Bk != B or Dk != D:
            raise ValueError("shape mismatch: q %s k %s v %s" % (q.shape, k.shape, v.shape))
        if rows is None:
            n_out, rows_ptr = B * S, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
            n_out = rows_arr.size
            rows_ptr = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        out = np.zeros((n_out, Hq, D), dtype=np.float64)
        lse = np.zeros((n_out, Hq), dtype=np.float64)
        P = ctypes.POINTER(ctypes.c_double)
        rc = self._fn(
            q.ctypes.data_as(P), k.ctypes.data_as(P), v.ctypes.data_as(P),
            out.ctypes.data_as(P), lse.ctypes.data_as(P),
            B, S, L, Hq, Hkv, D, int(bool(causal)), int(window), float(scale), float(softcap),
            rows_ptr, int(n_out) if rows is not None else 0,
            int(threads) if threads else default_threads())
        if rc != 0:
            raise ValueError("oracle_attention_rows failed with code %d" % rc)
        if rows is None:
            return out.reshape(B, S, Hq, D), lse.reshape(B, S, Hq)
        return out, lse

    def decode(self, q, k_cache, v_cache, kv_lens, *, window: int, scale: float,
               threads=None, softcap: float = 0.0):
        """One decode step per sequence: q [B, Hq, D], caches [B, cap, Hkv, D].

        Sequence b attends to its first kv_lens[b] cached keys from query position
        kv_lens[b] - 1 (the prefill definition with S = 1, L = kv_lens[b]).
        Returns out [B, Hq, D], lse [B, Hq].
        """
        q = _f64(q)
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D), dtype=np.float64)
        lse = np.zeros((B, Hq), dtype=np.float64)
        for b in range(B):
            n = int(kv_lens[b])
            # only the visible prefix of each cache is converted (slots past n are unused)
            kb, vb = _f64(k_cache[b, :n]), _f64(v_cache[b, :n])
            o, l = self.prefill(q[b][None, None], kb[None], vb[None],
                                causal=True, window=window, scale=scale, threads=threads,
                                softcap=softcap)
            out[b], lse[b] = o[0, 0], l[0, 0]
        return out, lse


def _get() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build_library())
    return _default


def prefill(q, k, v, *, causal, window, scale, rows=None, threads=None, softcap=0.0):
    return _get().prefill(q, k, v, causal=causal, window=window, scale=scale, rows=rows,
                          threads=threads, softcap=softcap)


def decode(q, k_cache, v_cache, kv_lens, *, window, scale, threads=None, softcap=0.0):
    return _get().decode(q, k_cache, v_cache, kv_lens, window=window, scale=scale,
                         threads=threads, softcap=softcap)


def kv_append(k_cache, v_cache, k_new, v_new, pos):
    """Copy new rows into the caches: cache[b, pos[b] + t] = new[b, t].

    k_cache, v_cache: [B, cap, Hkv, D]; k_new, v_new: [B, n_new, Hkv, D].
    Returns fresh arrays; raises IndexError when a row would fall outside [0, cap).
    """
    kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    k_new, v_new = np.asarray(k_new), np.asarray(v_new)
    B, cap = kc.shape[:2]
    n_new = k_new.shape[1]
    for b in range(B):
        p = int(pos[b])
        if p < 0 or p + n_new > cap:
            raise IndexError("append rows [%d, %d) outside capacity %d" % (p, p + n_new, cap))
        kc[b, p:p + n_new] = k_new[b]
        vc[b, p:p + n_new] = v_new[b]
    return kc, vc


def kv_append_ring(k_cache, v_cache, k_new, v_new, pos):
    """The same copy into a ring cache that keeps only its last ``cap`` positions, as a
    sliding-window layer does (hf2q "Current Inference Path", section 2 step 1: window
    1024; hf2q target architecture, section 3.3: per-layer caches): position p lives in
    row p % cap, so new row t of sequence b lands in row (pos[b] + t) % cap.

    k_cache, v_cache: [B, cap, Hkv, D]; k_new, v_new: [B, n_new, Hkv, D], n_new <= cap.
    Returns fresh arrays; raises IndexError for a negative position.
    """
    kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    k_new, v_new = np.asarray(k_new), np.asarray(v_new)
    B, cap = kc.shape[:2]
    n_new = k_new.shape[1]
    if n_new > cap:
        raise IndexError("%d new rows do not fit a ring of %d" % (n_new, cap))
    for b in range(B):
        p = int(pos[b])
        if p < 0:
            raise IndexError("negative position %d" % p)
        for t in range(n_new):
            kc[b, (p + t) % cap] = k_new[b, t]
            vc[b, (p + t) % cap] = v_new[b, t]
    return kc, vc
