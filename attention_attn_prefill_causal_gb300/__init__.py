"""Python binding of libattn (include/attn.h): grouped-query causal prefill
attention, single-query decode attention and the K/V cache append on one
GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libattn.so``.  Tensors are torch CUDA tensors (fp32, 16-byte
aligned); plain integers are accepted as raw device pointers.  The functions
carry the C names and argument order; a workspace is allocated with torch
when the caller passes none.  The five calls that launch kernels convert
their arguments in the small C extension ``_calls`` (a decode step is a few
microseconds of GPU work, and ctypes' per-argument conversion is a visible
part of that on the host); sizes must be non-negative and below 2^32.  The
other calls go through ctypes.  ``lib`` stays available for direct ctypes
calls.  There is no CPU fallback: importing this package fails loudly when
the library or the extension has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA",
    "ATTN_ERR_TIMEOUT", "ATTN_ERR_RANGE", "ATTN_PREC_FP32", "ATTN_PREC_FP16", "ATTN_PREC_BF16",
    "ATTN_PREC_TF32",
    "AttnError", "lib", "library_path", "attn_prefill_causal", "attn_prefill_workspace_size",
    "attn_decode", "attn_decode_workspace_size", "attn_decode_append", "attn_decode_noalloc",
    "kv_append", "attn_status_string",
    "attn_last_error_string", "attn_get_device_status", "attn_selftest_wait_timeout",
    "exported_symbols",
]

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA = 0, 1, 2, 3
ATTN_ERR_TIMEOUT, ATTN_ERR_RANGE = 4, 5
ATTN_PREC_FP32, ATTN_PREC_FP16, ATTN_PREC_BF16, ATTN_PREC_TF32 = 0, 1, 2, 3

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libattn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "attn.h")

if not os.path.exists(library_path):
    raise ImportError(
        f"libattn.so is not built ({library_path}); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` first")

lib = ctypes.CDLL(library_path)

_u32, _f32, _sz, _vp, _i = ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
_SIGS = {
    "attn_prefill_causal": (_i, [_vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32, _u32, _u32, _f32, _i,
                                 _vp, _sz, _vp]),
    "attn_prefill_workspace_size": (_sz, [_u32, _u32, _u32, _u32, _i]),
    "attn_decode": (_i, [_vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32, _u32, _u32, _f32, _vp, _sz,
                         _vp]),
    "attn_decode_workspace_size": (_sz, [_u32, _u32, _u32, _u32, _u32]),
    "attn_decode_append": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32,
                                _u32, _u32, _u32, _f32, _vp, _sz, _vp]),
    "attn_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32, _u32, _u32, _f32,
                                 _vp]),
    "kv_append": (_i, [_vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32, _vp]),
    "attn_status_string": (ctypes.c_char_p, [_i]),
    "attn_last_error_string": (ctypes.c_char_p, []),
    "attn_get_device_status": (_i, []),
    "attn_selftest_wait_timeout": (_i, [_u32]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype, _fn.argtypes = _res, _args

try:
    from . import _calls
except ImportError as _e:
    raise ImportError(
        f"the _calls extension is not built next to {library_path} ({_e}); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` first") from _e
_calls.bind(*(ctypes.cast(getattr(lib, _n), ctypes.c_void_p).value
              for _n in ("attn_prefill_causal", "attn_decode", "attn_decode_append",
                         "attn_decode_noalloc", "kv_append")))


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib.attn_status_string(status).decode()
        extra = lib.attn_last_error_string().decode()
        super().__init__(f"{where}: {msg}" + (f" ({extra})" if extra and status == ATTN_ERR_CUDA else ""))
        self.status = status


def exported_symbols() -> list[str]:
    """Function names declared in include/attn.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?([a-z_0-9]+)\(", text, re.M)))


def _current_stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, where: str, check: bool) -> int:
    if check and status != ATTN_OK:
        raise AttnError(status, where)
    return status


def _workspace(nbytes: int, like, workspace):
    """The caller's workspace, or a new device buffer of nbytes.  Neither
    entry point reads workspace bytes it has not written in the same call,
    so the buffer is left uninitialised."""
    if workspace is not None or nbytes == 0:
        return workspace
    import torch
    dev = like.device if getattr(like, "is_cuda", False) else torch.device(
        "cuda", torch.cuda.current_device())
    return torch.empty(nbytes, dtype=torch.uint8, device=dev)


def _workspace_args(workspace, workspace_bytes, size_fn, like):
    """(workspace, bytes) for a call: the caller's buffer and its size (the
    size query runs only when the library must allocate or the size is not
    known), or a new device buffer of the size the call needs."""
    if workspace is None:
        need = size_fn()
        workspace = _workspace(need, like, None)
        return workspace, need
    if workspace_bytes is None:
        workspace_bytes = (workspace.numel() * workspace.element_size()
                           if hasattr(workspace, "numel") else size_fn())
    return workspace, workspace_bytes


def attn_prefill_workspace_size(m, num_q_heads, num_kv_heads, head_dim, precision=ATTN_PREC_FP16):
    return int(lib.attn_prefill_workspace_size(m, num_q_heads, num_kv_heads, head_dim, precision))


def attn_decode_workspace_size(num_heads, kv_heads, head_dim, total_seq, window=0):
    return int(lib.attn_decode_workspace_size(num_heads, kv_heads, head_dim, total_seq, window))


def attn_prefill_causal(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride, kv_stride,
                        scale=0.0, precision=ATTN_PREC_FP16, workspace=None, workspace_bytes=None,
                        stream=None, check=True):
    """Causal GQA prefill (C: attn_prefill_causal).  q/o: [m, q_stride] fp32,
    k/v: [m, kv_stride] fp32.  Returns the status (raises when ``check``)."""
    if workspace is None or workspace_bytes is None:
        workspace, workspace_bytes = _workspace_args(
            workspace, workspace_bytes,
            lambda: attn_prefill_workspace_size(m, num_q_heads, num_kv_heads, head_dim,
                                                precision), q)
    st = _calls.attn_prefill_causal(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                                    kv_stride, scale, precision, workspace, workspace_bytes,
                                    _current_stream() if stream is None else stream)
    return _check(st, "attn_prefill_causal", check)


def attn_decode(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim, max_seq, total_seq,
                window=0, scale=0.0, workspace=None, workspace_bytes=None, stream=None, check=True):
    """Single-query GQA decode (C: attn_decode).  q/out: [num_heads, head_dim];
    caches: [kv_heads, max_seq, head_dim].  Returns the status."""
    if workspace is None or workspace_bytes is None:
        workspace, workspace_bytes = _workspace_args(
            workspace, workspace_bytes,
            lambda: attn_decode_workspace_size(num_heads, kv_heads, head_dim, total_seq, window),
            k_cache)
    st = _calls.attn_decode(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim, max_seq,
                            total_seq, window, scale, workspace, workspace_bytes,
                            _current_stream() if stream is None else stream)
    return _check(st, "attn_decode", check)


def attn_decode_append(q, k_new, v_new, k_cache, v_cache, out, num_heads, kv_heads, head_dim,
                       max_seq, total_seq, position, window=0, scale=0.0, rope_cos=None,
                       rope_sin=None, workspace=None, workspace_bytes=None, stream=None,
                       check=True):
    """Fused (RoPE +) append + decode (C: attn_decode_append)."""
    if workspace is None or workspace_bytes is None:
        workspace, workspace_bytes = _workspace_args(
            workspace, workspace_bytes,
            lambda: attn_decode_workspace_size(num_heads, kv_heads, head_dim, total_seq, window),
            k_cache)
    st = _calls.attn_decode_append(q, k_new, v_new, rope_cos, rope_sin, k_cache, v_cache, out,
                                   num_heads, kv_heads, head_dim, max_seq, total_seq, position,
                                   window, scale, workspace, workspace_bytes,
                                   _current_stream() if stream is None else stream)
    return _check(st, "attn_decode_append", check)


def attn_decode_noalloc(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim, max_seq,
                        total_seq, window=0, scale=0.0, stream=None, check=True):
    """attn_decode with the library's fixed scratch instead of a workspace
    (C: attn_decode_noalloc).  For callers that cannot allocate."""
    st = _calls.attn_decode_noalloc(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim,
                                    max_seq, total_seq, window, scale,
                                    _current_stream() if stream is None else stream)
    return _check(st, "attn_decode_noalloc", check)


def kv_append(k_src, v_src, k_cache, v_cache, kv_heads, head_dim, max_seq, position, stream=None,
              check=True):
    """Write one K row and one V row at ``position`` (C: kv_append)."""
    st = _calls.kv_append(k_src, v_src, k_cache, v_cache, kv_heads, head_dim, max_seq, position,
                          _current_stream() if stream is None else stream)
    return _check(st, "kv_append", check)


def attn_status_string(status: int) -> str:
    return lib.attn_status_string(status).decode()


def attn_last_error_string() -> str:
    return lib.attn_last_error_string().decode()


def attn_get_device_status() -> int:
    return int(lib.attn_get_device_status())


def attn_selftest_wait_timeout(limit_us: int = 1000) -> int:
    return int(lib.attn_selftest_wait_timeout(limit_us))
