"""The C-ABI library builds, loads without a GPU, exports every function its
header declares, and rejects bad arguments on the host (no device work)."""
import ctypes
import re
import subprocess

import pytest

import __graft_entry__


@pytest.fixture(scope="module")
def attn():
    __graft_entry__.build()
    import attention_attn_prefill_causal_gb300 as a
    return a


def _declared_functions(header_text):
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?([a-z_0-9]+)\(",
                                 header_text, re.M)))


def test_header_declares_the_three_entry_points(attn):
    names = _declared_functions(open(attn.HEADER).read())
    for n in ("attn_prefill_causal", "attn_decode", "kv_append"):
        assert n in names
    assert names == attn.exported_symbols()


def test_library_exports_every_declared_symbol(attn):
    names = attn.exported_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(attn.lib, n), f"libattn.so does not export {n}"
    out = subprocess.run(["nm", "-D", "--defined-only", attn.library_path],
                         capture_output=True, text=True, check=True).stdout
    dyn = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in names if n not in dyn]
    assert not missing, f"not exported with C linkage: {missing}"


def test_library_has_no_driver_link_dependency(attn):
    """The library resolves the driver at run time, so it loads on a host
    without libcuda (this container)."""
    out = subprocess.run(["readelf", "-d", attn.library_path], capture_output=True, text=True,
                         check=True).stdout
    assert "libcuda.so" not in out
    assert "libtorch" not in out


def test_status_strings(attn):
    for code in range(6):
        assert attn.attn_status_string(code)
    assert attn.attn_status_string(0) == "ok"
    assert attn.attn_status_string(99) == "unknown status"


def test_workspace_sizes_are_pure_functions(attn):
    assert attn.attn_prefill_workspace_size(2048, 12, 2, 128, attn.ATTN_PREC_FP32) == 0
    ws = attn.attn_prefill_workspace_size(2048, 12, 2, 128, attn.ATTN_PREC_FP16)
    assert ws >= 2 * 2048 * (2 * 128) * 2       # fp16 K and V
    assert ws == attn.attn_prefill_workspace_size(2048, 12, 2, 128, attn.ATTN_PREC_FP16)
    wt = attn.attn_prefill_workspace_size(2048, 12, 2, 128, attn.ATTN_PREC_TF32)
    assert wt >= 2 * 2048 * (2 * 128) * 4       # TF32-rounded K and transposed V, fp32
    assert wt == attn.attn_prefill_workspace_size(2048, 12, 2, 128, attn.ATTN_PREC_TF32)
    # V^T rows are padded to a multiple of 4 keys (16-byte TMA row pitch)
    assert attn.attn_prefill_workspace_size(1001, 4, 2, 64, attn.ATTN_PREC_TF32) >= \
        1001 * 128 * 4 + 128 * 1004 * 4
    d = attn.attn_decode_workspace_size(12, 2, 128, 4096, 0)
    assert d > 12 * 128 * 4
    # a window shrinks the live range, so the workspace cannot grow
    assert attn.attn_decode_workspace_size(32, 8, 128, 32768, 4096) <= \
        attn.attn_decode_workspace_size(32, 8, 128, 32768, 0)


FAKE = 0x10000  # a 16-byte aligned non-null value; never dereferenced (rejected first)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), 1),                                   # null pointer
    (dict(head_dim=48), 1),                           # head_dim % 32 != 0 (page: assert)
    (dict(num_kv_heads=0), 1),
    (dict(num_q_heads=12, num_kv_heads=5), 1),        # not a divisor
    (dict(q_stride=100), 1),                          # q_stride < Hq*D
    (dict(kv_stride=252), 1),                         # kv_stride < Hkv*D
    (dict(q=FAKE + 4), 1),                            # misaligned pointer
    (dict(scale=-1.0), 1),
    (dict(precision=7), 1),
    (dict(precision=1, head_dim=32), 2),              # tensor path: head_dim 64/128 only
    (dict(precision=1), 1),                           # tensor path without workspace
    (dict(precision=3, head_dim=32), 2),              # TF32 path: head_dim 64/128 only
    (dict(precision=3), 1),                           # TF32 path without workspace
    (dict(precision=4), 1),
    (dict(precision=0, head_dim=96, q_stride=1152, kv_stride=192), 2),
    (dict(m=0), 0),                                   # empty prefill: no-op
])
def test_prefill_rejects_bad_arguments(attn, kw, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, m=16, num_q_heads=12, num_kv_heads=2, head_dim=128,
             q_stride=1536, kv_stride=256, scale=0.0, precision=0)
    a.update(kw)
    st = attn.lib.attn_prefill_causal(a["q"], a["k"], a["v"], a["o"], a["m"], a["num_q_heads"],
                                      a["num_kv_heads"], a["head_dim"], a["q_stride"],
                                      a["kv_stride"], a["scale"], a["precision"], None, 0, None)
    if expect == 0 and kw.get("m") == 0:
        assert st == 0
    else:
        assert st == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(out=0), 1),
    (dict(total_seq=0), 1),                # no softmax over an empty row
    (dict(total_seq=5000), 1),             # beyond max_seq
    (dict(kv_heads=5), 1),
    (dict(head_dim=40), 1),
    (dict(head_dim=96), 2),
    (dict(workspace=None), 1),             # too small / missing workspace
])
def test_decode_rejects_bad_arguments(attn, kw, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, num_heads=12, kv_heads=2, head_dim=128,
             max_seq=4096, total_seq=4096, window=0, scale=0.0, workspace=None)
    a.update(kw)
    st = attn.lib.attn_decode(a["q"], a["k"], a["v"], a["out"], a["num_heads"], a["kv_heads"],
                              a["head_dim"], a["max_seq"], a["total_seq"], a["window"], a["scale"],
                              a["workspace"], 0, None)
    assert st == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(out=0), 1),                      # null output, at sizes beyond the scratch
    (dict(q=FAKE + 4), 1),                 # misaligned, at sizes beyond the scratch
    (dict(kv_heads=5000), 1),              # does not divide num_heads
    (dict(total_seq=0), 1),
    (dict(head_dim=96), 2),                # valid, outside the compiled head_dims
    (dict(), 2),                           # well-formed, but its partials exceed the scratch
])
def test_decode_noalloc_checks_arguments_before_its_scratch_size(attn, kw, expect):
    """The no-workspace decode validates its arguments exactly as attn_decode
    does before it looks at its fixed scratch size, so a malformed call is
    reported as INVALID_ARG whatever its sizes (no device work is launched
    for a rejected call)."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, num_heads=8192, kv_heads=8192, head_dim=128,
             max_seq=1, total_seq=1, window=0, scale=0.0)
    a.update(kw)
    st = attn.lib.attn_decode_noalloc(a["q"], a["k"], a["v"], a["out"], a["num_heads"],
                                      a["kv_heads"], a["head_dim"], a["max_seq"], a["total_seq"],
                                      a["window"], a["scale"], None)
    assert st == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(position=4096), 1),              # position >= max_seq
    (dict(v_src=None), 1),                 # v_src and v_cache must both be given or both null
    (dict(k_src=0), 1),
    (dict(head_dim=30), 1),
])
def test_kv_append_rejects_bad_arguments(attn, kw, expect):
    a = dict(k_src=FAKE, v_src=FAKE, k_cache=FAKE, v_cache=FAKE, kv_heads=2, head_dim=128,
             max_seq=4096, position=5)
    a.update(kw)
    st = attn.lib.kv_append(a["k_src"], a["v_src"], a["k_cache"], a["v_cache"], a["kv_heads"],
                            a["head_dim"], a["max_seq"], a["position"], None)
    assert st == expect


@pytest.mark.parametrize("hq,hkv,d,T,W", [(12, 2, 128, 4096, 0), (32, 8, 128, 32768, 4096),
                                          (4, 1, 32, 1, 0), (64, 8, 64, 100000, 0)])
def test_decode_workspace_has_room_for_staged_inputs(attn, hq, hkv, d, T, W):
    """A decode call with host-resident step inputs copies q, k_new, v_new and
    the RoPE tables ((hq + 2 hkv + 1) * head_dim floats) into its workspace,
    after the partials (one (max, sum) pair and head_dim floats per query head
    and chunk): the size covers both, whatever the chunk count."""
    ws = attn.attn_decode_workspace_size(hq, hkv, d, T, W)
    stage = (hq + 2 * hkv + 1) * d * 4
    assert ws >= stage + hq * (d + 2) * 4
    assert ws % 256 == 0
