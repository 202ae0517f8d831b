"""CUDA-graph capture of every entry point: a call captured once and replayed
must give, bit for bit, what the same call gives eagerly, also after the
input buffers' contents have changed (a graph keeps the pointers and sizes
of the capture, so nothing the library decides may depend on the data).
The no-alloc decode is first called eagerly, as its header asks, so that its
scratch address is known before the capture."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import attention_attn_prefill_causal_gb300 as a
    assert a.attn_get_device_status() == a.ATTN_OK
    return a


def _graph_equals_eager(call, outputs, inputs, refill):
    """call(stream) issues the library call(s); outputs: tensors the calls
    write; inputs: tensors refill() rewrites in place."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    for round_ in range(2):
        if round_:
            refill()
            torch.cuda.synchronize()
        with torch.cuda.stream(s):
            call(s)
        torch.cuda.synchronize()
        eager = [o.clone() for o in outputs]
        for o in outputs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, outputs):
            np.testing.assert_array_equal(b.cpu().numpy(), a.cpu().numpy())
    return g


@pytest.mark.parametrize("prec,m,hq,hkv,d", [(1, 1000, 8, 2, 128), (3, 1000, 8, 2, 128),
                                             (0, 300, 4, 2, 64), (1, 700, 2, 1, 64)])
def test_prefill_in_a_graph(attn, prec, m, hq, hkv, d):
    # (1, 700, 2, 1, 64): a grid below one wave, so the key walk is split and
    # the combine kernel is captured too
    q, k, v = (t.cuda() for t in workloads.prefill_inputs(m, hq * d, hkv * d, seed=71))
    o = torch.empty_like(q)
    ws = torch.empty(attn.attn_prefill_workspace_size(m, hq, hkv, d, prec), dtype=torch.uint8,
                     device="cuda")

    def call(s):
        attn.attn_prefill_causal(q, k, v, o, m, hq, hkv, d, hq * d, hkv * d, precision=prec,
                                 workspace=ws, stream=s)

    def refill():
        q2, k2, v2 = workloads.prefill_inputs(m, hq * d, hkv * d, seed=72)
        q.copy_(q2); k.copy_(k2); v.copy_(v2)
    _graph_equals_eager(call, [o], [q, k, v], refill)
    assert attn.attn_get_device_status() == attn.ATTN_OK


def test_decode_calls_in_a_graph(attn):
    hq, hkv, d, S = 12, 2, 128, 4096
    T, pos = 3000, 2999
    q, kc, vc, kn, vn = (t.cuda() for t in workloads.decode_inputs(hq, hkv, d, S, seed=73,
                                                                    append=True))
    half = d // 2
    ang = torch.arange(half, dtype=torch.float32) * 0.01
    cos, sin = torch.cos(ang).cuda(), torch.sin(ang).cuda()
    out1, out2, out3 = (torch.empty(hq, d, device="cuda") for _ in range(3))
    ws = torch.empty(attn.attn_decode_workspace_size(hq, hkv, d, T, 500), dtype=torch.uint8,
                     device="cuda")
    kc0, vc0 = kc.clone(), vc.clone()
    # the no-alloc entry point learns its scratch address in a first eager call
    attn.attn_decode_noalloc(q, kc, vc, out3, hq, hkv, d, S, T)
    torch.cuda.synchronize()

    def call(s):
        kc.copy_(kc0); vc.copy_(vc0)  # every replay starts from the same caches
        attn.attn_decode(q, kc, vc, out1, hq, hkv, d, S, T, window=500, workspace=ws, stream=s)
        attn.attn_decode_append(q, kn, vn, kc, vc, out2, hq, hkv, d, S, T, pos, window=500,
                                rope_cos=cos, rope_sin=sin, workspace=ws, stream=s)
        attn.kv_append(kn, vn, kc, vc, hkv, d, S, pos + 1, stream=s)
        attn.attn_decode_noalloc(q, kc, vc, out3, hq, hkv, d, S, T + 2, stream=s)

    def refill():
        q2, k2, v2, kn2, vn2 = workloads.decode_inputs(hq, hkv, d, S, seed=74, append=True)
        q.copy_(q2); kn.copy_(kn2); vn.copy_(vn2); kc0.copy_(k2); vc0.copy_(v2)
    _graph_equals_eager(call, [out1, out2, out3, kc, vc], [q, kn, vn, kc0, vc0], refill)
    assert attn.attn_get_device_status() == attn.ATTN_OK
