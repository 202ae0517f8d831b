"""The C ABI from plain C: tests/c_client/attn_client.c includes only
include/attn.h (and the CUDA runtime for its own buffers), is compiled as C
and linked against libattn.so.  On the CPU it checks the calls that need no
device (status strings, workspace sizes, null-pointer rejection); on a GPU it
runs an exact and an fp16 tensor-core prefill, a decode and a kv_append +
decode on cudaMalloc'd buffers, whose outputs are compared with the oracle
on the same seeded inputs."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import __graft_entry__
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_client", "attn_client.c")
PKG = os.path.join(ROOT, "attention_attn_prefill_causal_gb300")

# sizes fixed in attn_client.c
PM, PHQ, PHKV, PD = 200, 4, 2, 64
DHQ, DHKV, DD, DS = 8, 2, 128, 1000


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    pytest.skip("nvcc not available")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    __graft_entry__.build()
    exe = str(tmp_path_factory.mktemp("c_client") / "attn_client")
    # a .c file goes to the host compiler as C
    subprocess.run([_nvcc(), "-O2", SRC, "-o", exe,
                    "-I", os.path.join(ROOT, "include"), "-L", PKG, "-lattn",
                    "-Xlinker", "-rpath", "-Xlinker", PKG],
                   check=True, capture_output=True, text=True)
    return exe


def test_header_compiles_as_c_and_host_calls_work(client):
    r = subprocess.run([client, "abi"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("abi ok")


@pytest.mark.gpu
def test_c_client_matches_the_oracle(client, tmp_path):
    import oracle
    q, k, v = workloads.prefill_inputs(PM, PHQ * PD, PHKV * PD, seed=51)
    dq, kc, vc, kn, vn = workloads.decode_inputs(DHQ, DHKV, DD, DS, seed=52, append=True)
    for name, t in (("prefill_q", q), ("prefill_k", k), ("prefill_v", v), ("decode_q", dq),
                    ("decode_k", kc), ("decode_v", vc), ("decode_k_new", kn),
                    ("decode_v_new", vn)):
        t.numpy().astype(np.float32).tofile(str(tmp_path / f"{name}.bin"))
    r = subprocess.run([client, "run", str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("run ok")

    def load(name, shape):
        return np.fromfile(str(tmp_path / name), dtype=np.float32).reshape(shape)

    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), PM, PHQ, PHKV, PD, PHQ * PD,
                                PHKV * PD)
    got32 = load("prefill_o_fp32.bin", (PM, PHQ, PD))
    got16 = load("prefill_o_fp16.bin", (PM, PHQ, PD))
    assert np.abs(got32 - ref).max() <= 1e-4
    assert np.abs(got16 - ref).max() <= 3e-3

    ref_dec = oracle.decode(dq.numpy(), kc.numpy(), vc.numpy(), DHQ, DHKV, DD, DS, DS)
    assert np.abs(load("decode_out.bin", (DHQ, DD)) - ref_dec).max() <= 1e-4
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    oracle.kv_append(kn.numpy(), vn.numpy(), kh, vh, DHKV, DD, DS, DS - 1)
    ref_app = oracle.decode(dq.numpy(), kh, vh, DHQ, DHKV, DD, DS, DS)
    assert np.abs(load("decode_out_appended.bin", (DHQ, DD)) - ref_app).max() <= 1e-4
