"""Addresses past element 2^31: the row pitch of these prefills and the extent
of these caches put the elements the kernels read and write beyond index
2^31 of their fp32 buffers (more than 8 GiB), so a 32-bit offset anywhere
on the path would touch the wrong place.  The big buffers are left
uninitialised except for the columns and rows the call reads; the oracle
runs on the same inputs in compact form.  Canary columns beside the heads
(prefill) and the cache rows next to the appended one (decode) must survive.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity_utils import FP32_ABS, FP32_REL, TC_ABS, compare

pytestmark = pytest.mark.gpu

FP32, FP16, TF32 = 0, 1, 3
PITCH = 1 << 22          # floats per row: 16 MiB
CANARY = 12345.678

# prefill: 600 tokens, 104 query heads over 8 KV heads, head_dim 128.  Query-
# tile pairs x heads = 3 x 104 fill two waves of 152 SMs, so the fp16 call
# takes the pair kernel (its last pair has one empty tile); TF32 and fp32
# take the single-tile and CUDA-core kernels.
M, HQ, HKV, D = 600, 104, 8, 128


@pytest.fixture(scope="module")
def attn():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import attention_attn_prefill_causal_gb300 as a
    assert a.attn_get_device_status() == a.ATTN_OK
    return a


@pytest.fixture(scope="module")
def prefill_case():
    q, k, v = workloads.prefill_inputs(M, HQ * D, HKV * D, seed=41)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), M, HQ, HKV, D, HQ * D, HKV * D)
    return q, k, v, ref


def _release():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("prec", [FP32, FP16, TF32])
def test_prefill_rows_past_element_2_31(attn, prefill_case, prec):
    q, k, v, ref = prefill_case
    assert (M - 1) * PITCH > 2 ** 31
    bufs = [torch.empty(M * PITCH, dtype=torch.float32, device="cuda") for _ in range(4)]
    try:
        dq, dk, dv, do = (b.view(M, PITCH) for b in bufs)
        dq[:, :HQ * D] = q.cuda()
        dk[:, :HKV * D] = k.cuda()
        dv[:, :HKV * D] = v.cuda()
        do[:, :HQ * D] = float("nan")
        do[:, HQ * D:HQ * D + 8] = CANARY
        attn.attn_prefill_causal(bufs[0], bufs[1], bufs[2], bufs[3], M, HQ, HKV, D, PITCH, PITCH,
                                 precision=prec)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == attn.ATTN_OK
        assert bool((do[:, HQ * D:HQ * D + 8] == CANARY).all())
        got = do[:, :HQ * D].cpu().numpy().reshape(M, HQ, D)
    finally:
        del bufs
        _release()
    amax, rel = compare(got, ref)
    if prec == FP32:
        assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)
    else:
        assert amax <= TC_ABS, amax


def test_decode_append_cache_rows_past_element_2_31(attn):
    """Fused append + windowed decode on [2, 2^24, 128] caches (16 GiB each):
    KV head 1's rows start at element 2^31.  Only the window's rows are
    written; the decode reads nothing below the window (its -1e4 weight is 0
    in fp32 for these scores), so the oracle's decode over the window's rows
    alone is the same result."""
    hq, hkv, d = 16, 2, 128
    S = 1 << 24
    T, W = S, 4096
    pos = T - 1
    assert hkv * S * d > 2 ** 31 and S * d >= 2 ** 31
    q, kw, vw, kn, vn = workloads.decode_inputs(hq, hkv, d, W, seed=43, append=True)
    out_ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kw.numpy().copy(),
                                   vw.numpy().copy(), hq, hkv, d, W, W, W - 1, window=0)
    kc = torch.empty(hkv * S * d, dtype=torch.float32, device="cuda")
    vc = torch.empty_like(kc)
    try:
        k3, v3 = kc.view(hkv, S, d), vc.view(hkv, S, d)
        k3[:, T - W:T] = kw.cuda()
        v3[:, T - W:T] = vw.cuda()
        out = torch.full((hq, d), float("nan"), device="cuda")
        attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), kc, vc, out, hq, hkv, d, S, T, pos,
                                window=W)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == attn.ATTN_OK
        got = out.cpu().numpy()
        appended_k = k3[:, pos].cpu().numpy()
        appended_v = v3[:, pos].cpu().numpy()
        neighbours = k3[:, pos - 1].cpu().numpy()
    finally:
        del kc, vc
        _release()
    np.testing.assert_array_equal(appended_k, kn.numpy())
    np.testing.assert_array_equal(appended_v, vn.numpy())
    np.testing.assert_array_equal(neighbours, kw.numpy()[:, W - 2])
    amax, rel = compare(got, out_ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)
