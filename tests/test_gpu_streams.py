"""Concurrent calls: two host threads issue prefills and decodes on two CUDA
streams at once, each with its own workspace and outputs.  The library holds
no per-call state outside the caller's buffers (its only globals are cached
device queries and the device status word), and every kernel's arithmetic
order is fixed, so each concurrent result must equal, bit for bit, the same
call made alone."""
import threading

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


def _prefill_job(attn, prec, m=1024, hq=8, hkv=2, d=128, seed=61):
    q, k, v = (t.cuda() for t in workloads.prefill_inputs(m, hq * d, hkv * d, seed))
    ws = torch.empty(attn.attn_prefill_workspace_size(m, hq, hkv, d, prec), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)

    def run(stream):
        attn.attn_prefill_causal(q, k, v, o, m, hq, hkv, d, hq * d, hkv * d, precision=prec,
                                 workspace=ws, stream=stream)
        return o
    return run


def _decode_job(attn, hq=12, hkv=2, d=128, S=4096, window=0, seed=62):
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed)
    q, kc, vc = q.cuda(), kc.cuda(), vc.cuda()
    ws = torch.empty(attn.attn_decode_workspace_size(hq, hkv, d, S, window), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(hq, d, device="cuda")

    def run(stream):
        attn.attn_decode(q, kc, vc, out, hq, hkv, d, S, S, window=window, workspace=ws,
                         stream=stream)
        return out
    return run


def test_concurrent_calls_on_two_streams_equal_the_calls_alone(attn):
    jobs = [[_prefill_job(attn, attn.ATTN_PREC_FP16), _decode_job(attn)],
            [_prefill_job(attn, attn.ATTN_PREC_TF32, seed=63), _decode_job(attn, window=1000, seed=64),
             _prefill_job(attn, attn.ATTN_PREC_FP32, m=300, hq=4, hkv=2, d=64, seed=65)]]
    # each call alone, on the default stream
    alone = []
    for group in jobs:
        res = []
        for job in group:
            res.append(job(torch.cuda.current_stream()).clone())
            torch.cuda.synchronize()
        alone.append(res)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = [[None] * len(g) for g in jobs]
    errors = []

    def worker(i):
        try:
            s = streams[i]
            with torch.cuda.stream(s):
                for rep in range(8):
                    for j, job in enumerate(jobs[i]):
                        out = job(s)
                        if rep == 7:
                            got[i][j] = out.clone()
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    for i, group in enumerate(jobs):
        for j in range(len(group)):
            a, b = alone[i][j].cpu().numpy(), got[i][j].cpu().numpy()
            assert np.isfinite(b).all()
            np.testing.assert_array_equal(b, a, err_msg=f"thread {i}, job {j}")
