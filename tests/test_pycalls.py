"""The C extension `_calls` that the Python binding uses for the five calls
that launch kernels: it must hand libattn exactly what the ctypes binding
hands it.  Every call here is rejected by the library's host-side checks
(null or misaligned pointers, bad sizes, a missing workspace) or is the
empty prefill, so nothing reaches a device even where one is present (the
base argument sets are never called unmodified); the status codes from both
bindings must agree.  Conversion errors (negative or 32-bit-overflowing
sizes, wrong argument counts, objects without data_ptr) raise before the
library is called."""
import ctypes

import pytest
import torch

import __graft_entry__

FAKE = 0x10000  # 16-byte aligned, non-null, never dereferenced (every call below is rejected)


@pytest.fixture(scope="module")
def attn():
    __graft_entry__.build()
    import attention_attn_prefill_causal_gb300 as a
    return a


class _Stream:
    """Stands in for a torch stream: only its cuda_stream attribute is read."""
    cuda_stream = 0


class _Tensor:
    """Stands in for a tensor: only data_ptr() is called."""
    def __init__(self, p):
        self.p = p

    def data_ptr(self):
        return self.p


PREFILL = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, m=16, hq=12, hkv=2, d=128, qs=1536, kvs=256,
               scale=0.0, prec=0, ws=None, wsb=0)
DECODE = dict(q=FAKE, kc=FAKE, vc=FAKE, out=FAKE, hq=12, hkv=2, d=128, S=4096, T=4096, W=0,
              scale=0.0, ws=None, wsb=0)
APPEND = dict(q=FAKE, kn=FAKE, vn=FAKE, cos=None, sin=None, kc=FAKE, vc=FAKE, out=FAKE, hq=12,
              hkv=2, d=128, S=4096, T=4096, pos=4095, W=0, scale=0.0, ws=None, wsb=0)
NOALLOC = dict(q=FAKE, kc=FAKE, vc=FAKE, out=FAKE, hq=8192, hkv=8192, d=128, S=1, T=1, W=0,
               scale=0.0)
KVAPP = dict(ks=FAKE, vs=FAKE, kc=FAKE, vc=FAKE, hkv=2, d=128, S=4096, pos=5)

CASES = [
    ("attn_prefill_causal", PREFILL, dict(q=0)),
    ("attn_prefill_causal", PREFILL, dict(d=48)),
    ("attn_prefill_causal", PREFILL, dict(hkv=5)),
    ("attn_prefill_causal", PREFILL, dict(q=FAKE + 4)),
    ("attn_prefill_causal", PREFILL, dict(scale=-1.0)),
    ("attn_prefill_causal", PREFILL, dict(prec=7)),
    ("attn_prefill_causal", PREFILL, dict(prec=1, d=32)),
    ("attn_prefill_causal", PREFILL, dict(prec=3)),
    ("attn_prefill_causal", PREFILL, dict(m=0)),
    ("attn_decode", DECODE, dict(out=0)),
    ("attn_decode", DECODE, dict(T=0)),
    ("attn_decode", DECODE, dict(T=5000)),
    ("attn_decode", DECODE, dict(d=96)),
    ("attn_decode", DECODE, dict()),                 # no workspace
    ("attn_decode_append", APPEND, dict(kn=0)),
    ("attn_decode_append", APPEND, dict(cos=FAKE)),  # cos without sin
    ("attn_decode_append", APPEND, dict(pos=4096)),
    ("attn_decode_append", APPEND, dict(vn=FAKE + 8)),
    ("attn_decode_append", APPEND, dict()),          # no workspace
    ("attn_decode_noalloc", NOALLOC, dict(out=0)),
    ("attn_decode_noalloc", NOALLOC, dict(hkv=5000)),
    ("attn_decode_noalloc", NOALLOC, dict()),        # partials exceed the fixed scratch
    ("kv_append", KVAPP, dict(pos=4096)),
    ("kv_append", KVAPP, dict(vs=None)),
    ("kv_append", KVAPP, dict(d=30)),
]


def _args(base, kw, stream):
    a = dict(base)
    a.update(kw)
    return list(a.values()) + [stream]


@pytest.mark.parametrize("name,base,kw", CASES)
def test_extension_and_ctypes_return_the_same_status(attn, name, base, kw):
    args = _args(base, kw, None)
    expect = getattr(attn.lib, name)(*args)
    assert expect != attn.ATTN_OK or kw.get("m") == 0
    # raw ints and a None stream in ctypes; the extension takes the stream
    # as an int, as an object with cuda_stream, and pointers as objects
    assert getattr(attn._calls, name)(*_args(base, kw, 0)) == expect
    assert getattr(attn._calls, name)(*_args(base, kw, _Stream())) == expect
    wrapped = [(_Tensor(v) if isinstance(v, int) and v >= FAKE and i < 8 else v)
               for i, v in enumerate(_args(base, kw, 0))]
    assert getattr(attn._calls, name)(*wrapped) == expect


def test_public_functions_use_the_extension(attn):
    """The public functions accept tensors and ints alike and return the
    library's status (check=False)."""
    q = torch.empty(16, 1536)
    st = attn.attn_prefill_causal(q, q, q, 0, 16, 12, 2, 128, 1536, 256,
                                  precision=attn.ATTN_PREC_FP32, stream=0, check=False)
    assert st == attn.ATTN_ERR_INVALID_ARG                      # null output
    st = attn.attn_decode(0, FAKE, FAKE, FAKE, 12, 2, 128, 4096, 4096, workspace=FAKE,
                          workspace_bytes=1 << 20, stream=_Stream(), check=False)
    assert st == attn.ATTN_ERR_INVALID_ARG
    with pytest.raises(attn.AttnError):
        attn.kv_append(FAKE, FAKE, FAKE, FAKE, 2, 128, 4096, 4096, stream=0)


@pytest.mark.parametrize("bad,exc", [(-1, OverflowError), (1 << 32, OverflowError),
                                     (2.5, TypeError), ("16", TypeError)])
def test_sizes_are_checked_before_the_call(attn, bad, exc):
    a = dict(PREFILL)
    a["m"] = bad
    with pytest.raises(exc):
        attn._calls.attn_prefill_causal(*a.values(), 0)


def test_argument_count_and_pointer_objects_are_checked(attn):
    with pytest.raises(TypeError):
        attn._calls.attn_decode(*DECODE.values())              # stream missing
    with pytest.raises(TypeError):
        attn._calls.kv_append(*KVAPP.values(), 0, 0)
    a = dict(KVAPP)
    a["ks"] = object()                                         # no data_ptr()
    with pytest.raises(AttributeError):
        attn._calls.kv_append(*a.values(), 0)
    a["ks"] = _Tensor(-5)                                      # not an address
    with pytest.raises(OverflowError):
        attn._calls.kv_append(*a.values(), 0)
    with pytest.raises(AttributeError):
        attn._calls.kv_append(*KVAPP.values(), object())      # no cuda_stream


def test_extension_is_bound_to_the_loaded_library(attn):
    """bind() got the addresses of the functions in the libattn.so that
    ctypes loaded, so both bindings share one copy of the library."""
    addr = ctypes.cast(attn.lib.kv_append, ctypes.c_void_p).value
    assert addr
    with pytest.raises(ValueError):
        attn._calls.bind(0, 0, 0, 0, 0)
    # re-binding the same addresses keeps the module working
    attn._calls.bind(*(ctypes.cast(getattr(attn.lib, n), ctypes.c_void_p).value
                       for n in ("attn_prefill_causal", "attn_decode", "attn_decode_append",
                                 "attn_decode_noalloc", "kv_append")))
    a = dict(KVAPP, pos=4096)                                  # rejected: position >= max_seq
    assert attn._calls.kv_append(*a.values(), 0) == attn.ATTN_ERR_INVALID_ARG
