"""The tensor-core prefill kernels' abort paths, run for real: a child
process sets the library's device wait limit to 1 us (ATTN_WAIT_LIMIT_US,
read once per process), so a bounded mbarrier wait inside the kernels that
lasts long enough gives up mid-call (a wait checks its clock every 64 polls,
so in practice only the longer waits, such as those of a process's first
calls, run out).  A kernel that gives up must record the timeout in the
device status word, drain its copies and MMAs, free TMEM and exit: every
call must end with status OK or timeout, and the context must stay usable,
which the child checks with the self-test's timeout (always fires) and a
correct exact-mode prefill afterwards.  No fault is provoked: the waits run
out on their own limit."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import attention_attn_prefill_causal_gb300 as attn
    import oracle
    import workloads

    # (tokens, query heads, kv heads, head_dim, mode): the pair kernel (16-bit,
    # pairs x heads at least two waves of SMs), the single-tile kernel in each
    # operand type, and a split single-tile call (partials and combine)
    calls = [(8192, 16, 4, 128, attn.ATTN_PREC_FP16), (8192, 16, 4, 128, attn.ATTN_PREC_BF16),
             (2048, 12, 2, 128, attn.ATTN_PREC_FP16), (2048, 12, 2, 128, attn.ATTN_PREC_TF32),
             (2048, 2, 1, 64, attn.ATTN_PREC_TF32)]
    timeouts = 0
    for m, hq, hkv, d, prec in calls:
        q, k, v = (t.cuda() for t in workloads.prefill_inputs(m, hq * d, hkv * d, seed=5))
        o = torch.zeros_like(q)
        st = attn.attn_prefill_causal(q, k, v, o, m, hq, hkv, d, hq * d, hkv * d,
                                      precision=prec, check=False)
        torch.cuda.synchronize()  # raises if the context was lost
        ds = attn.attn_get_device_status()
        assert st == attn.ATTN_OK, st
        assert ds in (attn.ATTN_OK, attn.ATTN_ERR_TIMEOUT), ds
        timeouts += ds == attn.ATTN_ERR_TIMEOUT
        print(f"m={m} heads={hq}x{hkv} d={d} prec={prec}: device status {ds}", flush=True)
    assert attn.attn_selftest_wait_timeout(1) == attn.ATTN_ERR_TIMEOUT
    # The context still computes: the exact mode has no device waits.
    m, hq, hkv, d = 300, 4, 2, 64
    q, k, v = workloads.prefill_inputs(m, hq * d, hkv * d, seed=6)
    o = torch.empty(m, hq * d, device="cuda")
    attn.attn_prefill_causal(q.cuda(), k.cuda(), v.cuda(), o, m, hq, hkv, d, hq * d, hkv * d,
                             precision=attn.ATTN_PREC_FP32)
    torch.cuda.synchronize()
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, hq * d, hkv * d)
    err = float(np.abs(o.cpu().numpy().reshape(m, hq, d) - ref).max())
    assert err <= 1e-4, err
    assert attn.attn_get_device_status() == attn.ATTN_OK
    print(f"timeouts {timeouts} of {len(calls)}; exact-mode prefill afterwards max abs {err:.2e}",
          flush=True)
""")


def test_prefill_kernels_give_up_cleanly_when_waits_run_out():
    env = dict(os.environ, ATTN_WAIT_LIMIT_US="1")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env,
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert any(line.startswith("timeouts ") for line in r.stdout.splitlines()), r.stdout
