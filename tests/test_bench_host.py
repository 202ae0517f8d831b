"""Host-side logic of bench.py (no GPU): multi-rank aggregation over gloo,
clock-sample parsing, the reference (oracle) arm's JSON line, and the hash
that ties profiled DRAM traffic to the kernel code."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    secs, units = bench.aggregate(1.0 + rank, 10.0 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, secs, units))
    torch.distributed.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    """Whole-job value = units summed over ranks / max time over ranks."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, secs, units in res:
        assert secs == 2.0 and units == 30.0


def test_clock_summary_parsing():
    s = bench.ClockSampler(0)
    s.proc = object()
    now = 1000.0
    s.lines = [(now + 0.1, "2026/12/02 10:00:00.000, 0, 1965, 2070, 900.1, 0x0, Not Active, "
                           "Not Active, Not Active, Active"),
               (now + 0.3, "2026/12/02 10:00:00.200, 0, 1980, 2070, 950.0, 0x0, Not Active, "
                           "Not Active, Not Active, Not Active"),
               (now + 9.0, "2026/12/02 10:00:09.000, 0, 500, 2070, 50.0, 0x0, Not Active, "
                           "Not Active, Not Active, Not Active")]
    out = s.summary(now, now + 0.4)
    assert out["sm_mhz"] == pytest.approx(1972.5)
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 2


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["metric"] == bench.METRIC


def test_traffic_hash_ignores_comments_only():
    """The counters in profiles/traffic.json stay attached to a kernel while
    only its comments or blank space change, and drop when its code does."""
    src = "int f(int x) {  // doubles x\n    return 2 * x; /* the\n  result */\n}\n"
    same = "// header comment\nint f(int x) {\n  return 2 * x;\n}\n"
    changed = "int f(int x) {  // doubles x\n    return 3 * x;\n}\n"
    assert bench.code_text(src) == bench.code_text(same) == "int f(int x) { return 2 * x; }"
    assert bench.code_text(changed) != bench.code_text(src)


@pytest.mark.parametrize("m,hq,hkv,d", [(2048, 12, 2, 128), (16384, 28, 4, 128), (4096, 2, 1, 64),
                                        (300, 4, 2, 128), (1000, 40, 8, 64), (5000, 3, 1, 128)])
def test_prefill_launch_count_follows_the_library_plan(m, hq, hkv, d):
    """bench.py counts a third launch (the combine kernel) exactly when the
    library splits the key walk, which shows in the workspace as chunk
    partials beyond the rounded K and V (both sizes are host arithmetic over
    152 SMs when no GPU is visible)."""
    import attention_attn_prefill_causal_gb300 as attn
    ws16 = attn.attn_prefill_workspace_size(m, hq, hkv, d, attn.ATTN_PREC_FP16)
    operands16 = 2 * (-(-m * hkv * d * 2 // 256) * 256)
    wst = attn.attn_prefill_workspace_size(m, hq, hkv, d, attn.ATTN_PREC_TF32)
    operandst = -(-m * hkv * d * 4 // 256) * 256 + -(-hkv * d * (-(-m // 4) * 4) * 4 // 256) * 256
    launches16 = bench.prefill_launches(m, hq, 152)             # pair or single-tile kernel
    launchest = bench.prefill_launches(m, hq, 152, tf32=True)   # single query tiles
    assert (ws16 > operands16) == (launches16 == 3), (ws16, operands16, launches16)
    assert (wst > operandst) == (launchest == 3), (wst, operandst, launchest)
