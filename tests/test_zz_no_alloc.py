"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some users of this library cannot give it a workspace: an inference engine
that reserved every free byte of HBM for its own pools, or a plugin interface
that only passes input and output pointers.  attn_decode_noalloc serves them
with a fixed scratch array compiled into libattn.  This test calls it through
the C ABI twice in a row (different shapes, so the second call runs on the
first call's leftovers in the shared array), on NaN-poisoned outputs with
canary bands on both sides, and checks each output against the fp64 oracle
and against the workspace entry point attn_decode, within the fp32
tolerances of the other GPU tests.  It lives in its own file, collected last,
and passes both alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity_utils import FP32_ABS, FP32_REL, compare, guarded_empty, guards_intact

pytestmark = pytest.mark.gpu


def _decode_both(attn, shape):
    q, kc, vc, _, _ = workloads.shape_inputs(shape)
    dq, dk, dv = q.cuda(), kc.cuda(), vc.cuda()
    h, d = shape.num_heads, shape.head_dim
    ref_buf, ref = guarded_empty(h * d)
    attn.attn_decode(dq, dk, dv, ref, h, shape.kv_heads, d, shape.max_seq, shape.total_seq,
                     window=shape.window)
    buf, out = guarded_empty(h * d)
    st = attn.lib.attn_decode_noalloc(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), out.data_ptr(),
                                      h, shape.kv_heads, d, shape.max_seq, shape.total_seq,
                                      shape.window, 0.0,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    torch.cuda.synchronize()
    assert guards_intact(buf) and guards_intact(ref_buf)
    expect = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), h, shape.kv_heads, d,
                           shape.max_seq, shape.total_seq, shape.window)
    return out.view(h, d).cpu().numpy(), ref.view(h, d).cpu().numpy(), expect


def test_noalloc_decode_matches_oracle_and_workspace_decode_twice():
    assert torch.cuda.is_available()
    import attention_attn_prefill_causal_gb300 as attn
    for shape in (workloads.DECODE_32K_WINDOW, workloads.DECODE_4K):
        got, via_workspace, expect = _decode_both(attn, shape)
        amax, rel = compare(got, expect)
        assert amax <= FP32_ABS and rel <= FP32_REL, (shape.name, "oracle", amax, rel)
        amax, rel = compare(got, via_workspace)
        assert amax <= FP32_ABS and rel <= FP32_REL, (shape.name, "attn_decode", amax, rel)
    assert attn.attn_get_device_status() == attn.ATTN_OK


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    import attention_attn_prefill_causal_gb300 as attn
    h, d = 8192, 128          # one split per head: 8192 * 128 * 4 B of partials > 4 MiB
    assert attn.attn_decode_workspace_size(h, h, d, 1, 0) > (4 << 20)
    q = torch.zeros(h, d, device="cuda")
    cache = torch.zeros(h, 1, d, device="cuda")
    out = torch.zeros(h, d, device="cuda")
    st = attn.lib.attn_decode_noalloc(q.data_ptr(), cache.data_ptr(), cache.data_ptr(),
                                      out.data_ptr(), h, h, d, 1, 1, 0, 0.0,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_UNSUPPORTED
    assert "scratch" in attn.attn_last_error_string()
    assert bool((out == 0).all().item())
