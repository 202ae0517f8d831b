"""fp64 CPU oracle for causal GQA prefill, single-query decode and kv_append.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links or
calls it, and it imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over independent (head, row) problems).  This module compiles it with gcc on
first use and wraps it with ctypes; it adds no arithmetic of its own.

Sources: the web pages "aprender-gpu 0.32.0 -- prefill_fused.rs" (fused causal
prefill, module doc and ``build_ptx``) and "honeycrisp kernels/attention.rs"
(Metal decode ``kmain``, sliding window, KV_APPEND templates).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u32p = ctypes.POINTER(ctypes.c_uint32)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP,
    no fast-math so the fp64 arithmetic keeps its written order)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_prefill_causal.restype = ctypes.c_int
            lib.oracle_prefill_causal.argtypes = [
                _f32p, _f32p, _f32p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_double,
                _u32p, ctypes.c_uint32, _f64p, _f64p, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [
                _f32p, _f32p, _f32p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_double,
                _f64p, _f64p, ctypes.c_int]
            lib.oracle_kv_append.restype = ctypes.c_int
            lib.oracle_kv_append.argtypes = [
                _f32p, _f32p, _f32p, _f32p, ctypes.c_uint32, ctypes.c_uint32,
                ctypes.c_uint32, ctypes.c_uint32]
            lib.oracle_decode_append.restype = ctypes.c_int
            lib.oracle_decode_append.argtypes = [
                _f32p, _f32p, _f32p, _f32p, _f32p, _f32p, _f32p, ctypes.c_uint32,
                ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                ctypes.c_uint32, ctypes.c_uint32, ctypes.c_double, _f64p, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle uses by default on this host."""
    return int(_load().oracle_max_threads())


def _as_f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle inputs are fp32 tensors, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def prefill_causal(q, k, v, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                   kv_stride, scale=None, rows=None, return_weights=False,
                   nthreads=0):
    """Causal GQA prefill in fp64.  q: [m, q_stride] fp32; k, v: [m, kv_stride].

    Returns O as float64 [n_rows, num_q_heads, head_dim] (all rows when
    ``rows`` is None); with ``return_weights`` also the materialised softmax
    weights [n_rows, num_q_heads, m].  ``scale`` defaults to 1/sqrt(head_dim),
    the constant the prefill page bakes in.
    """
    lib = _load()
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    if m > 0 and (q.size < (m - 1) * q_stride + num_q_heads * head_dim
                  or k.size < (m - 1) * kv_stride + num_kv_heads * head_dim
                  or v.size < (m - 1) * kv_stride + num_kv_heads * head_dim):
        raise ValueError("input smaller than its last row's end")
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    if rows is None:
        rows_arr, n_rows, rows_p = None, m, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.uint32))
        n_rows, rows_p = rows_arr.size, _ptr(rows_arr, _u32p)
    out = np.empty((n_rows, num_q_heads, head_dim), dtype=np.float64)
    w = np.empty((n_rows, num_q_heads, m), dtype=np.float64) if return_weights else None
    rc = lib.oracle_prefill_causal(
        _ptr(q, _f32p), _ptr(k, _f32p), _ptr(v, _f32p), m, num_q_heads, num_kv_heads,
        head_dim, q_stride, kv_stride, float(scale), rows_p, n_rows,
        _ptr(out, _f64p), _ptr(w, _f64p) if w is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_prefill_causal rejected its arguments")
    return (out, w) if return_weights else out


def decode(q, k_cache, v_cache, num_heads, kv_heads, head_dim, max_seq, total_seq,
           window=0, scale=None, return_weights=False, nthreads=0):
    """Single-query GQA decode in fp64.  q: [num_heads, head_dim];
    caches: [kv_heads, max_seq, head_dim].  Returns out [num_heads, head_dim]
    float64 (and the weights [num_heads, total_seq] when asked)."""
    lib = _load()
    q, kc, vc = _as_f32(q), _as_f32(k_cache), _as_f32(v_cache)
    if kc.size < kv_heads * max_seq * head_dim or vc.size < kv_heads * max_seq * head_dim:
        raise ValueError("cache smaller than kv_heads * max_seq * head_dim")
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    out = np.empty((num_heads, head_dim), dtype=np.float64)
    w = np.empty((num_heads, max(total_seq, 1)), dtype=np.float64) if return_weights else None
    rc = lib.oracle_decode(
        _ptr(q, _f32p), _ptr(kc, _f32p), _ptr(vc, _f32p), num_heads, kv_heads, head_dim,
        max_seq, total_seq, window, float(scale), _ptr(out, _f64p),
        _ptr(w, _f64p) if w is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return (out, w) if return_weights else out


def kv_append(k_src, v_src, k_cache, v_cache, kv_heads, head_dim, max_seq, position):
    """In-place cache append on fp32 numpy arrays (v_src/v_cache may be None)."""
    lib = _load()
    ks = _as_f32(k_src)
    if not (isinstance(k_cache, np.ndarray) and k_cache.flags.c_contiguous
            and k_cache.dtype == np.float32):
        raise TypeError("k_cache must be a C-contiguous fp32 numpy array")
    vs = _as_f32(v_src) if v_src is not None else None
    if v_cache is not None and not (isinstance(v_cache, np.ndarray)
                                    and v_cache.flags.c_contiguous
                                    and v_cache.dtype == np.float32):
        raise TypeError("v_cache must be a C-contiguous fp32 numpy array")
    rc = lib.oracle_kv_append(
        _ptr(ks, _f32p), _ptr(vs, _f32p) if vs is not None else None,
        _ptr(k_cache, _f32p), _ptr(v_cache, _f32p) if v_cache is not None else None,
        kv_heads, head_dim, max_seq, position)
    if rc != 0:
        raise ValueError("oracle_kv_append rejected its arguments")


def decode_append(q, k_new, v_new, k_cache, v_cache, num_heads, kv_heads, head_dim, max_seq,
                  total_seq, position, window=0, scale=None, rope_cos=None, rope_sin=None,
                  nthreads=0):
    """Fused (RoPE +) append + decode in fp64; updates the fp32 numpy caches
    in place and returns out [num_heads, head_dim] float64."""
    lib = _load()
    q, kn, vn = _as_f32(q), _as_f32(k_new), _as_f32(v_new)
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.flags.c_contiguous and c.dtype == np.float32):
            raise TypeError("caches must be C-contiguous fp32 numpy arrays")
    cs = _as_f32(rope_cos) if rope_cos is not None else None
    sn = _as_f32(rope_sin) if rope_sin is not None else None
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    out = np.empty((num_heads, head_dim), dtype=np.float64)
    rc = lib.oracle_decode_append(
        _ptr(q, _f32p), _ptr(kn, _f32p), _ptr(vn, _f32p),
        _ptr(cs, _f32p) if cs is not None else None, _ptr(sn, _f32p) if sn is not None else None,
        _ptr(k_cache, _f32p), _ptr(v_cache, _f32p), num_heads, kv_heads, head_dim, max_seq,
        total_seq, position, window, float(scale), _ptr(out, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_append rejected its arguments")
    return out
