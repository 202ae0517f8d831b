"""Seeded random-shape parity sweep through the C ABI against the fp64 oracle.

Each case draws its shape from a fixed generator: GQA ratios from 1 to 16,
head_dim 32/64/128, ragged token counts, padded row strides, explicit and
default scales, the four prefill precisions (including token counts that
make the tensor-core path split its key walk), and decode with windows,
ragged lengths, the fused append and RoPE.  Tolerances are the ones the
named tests use: fp32 max abs <= 1e-4 and normwise rel <= 1e-4; fp16 and
tf32 operands max abs <= 3e-3; bf16 operands max abs <= 2.5e-2 (unit roundoff
2^-9 on |V| up to about 4).  The rounding error of a score grows linearly
with the scale (|ds| ~ scale |q| |k| u), so with an explicit scale above the
default 1/sqrt(head_dim) the two operand-rounding bounds are multiplied by
scale * sqrt(head_dim)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity_utils import (FP32_ABS, FP32_REL, TC_ABS, compare, guarded_empty,
                                guards_intact, heads_view, untouched_columns)

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, TF32 = 0, 1, 2, 3
BF16_ABS = 2.5e-2


def _tf32_variants(cases):
    """Every tensor-core case again in the TF32 mode (same shape and inputs;
    case ids offset by 500)."""
    return [(c[0] + 500, TF32) + tuple(c[2:]) for c in cases if c[1] in (FP16, BF16)]


def _prefill_cases(n=28, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        prec = int(rng.choice([FP32, FP16, FP16, BF16]))
        d = int(rng.choice([64, 128])) if prec != FP32 else int(rng.choice([32, 64, 128]))
        hkv = int(rng.choice([1, 2, 3, 4]))
        g = int(rng.choice([1, 2, 3, 4, 6, 8]))
        while hkv * g > 16:
            g //= 2
        hq = hkv * g
        big = rng.random() < 0.3
        m = int(rng.integers(1000, 3001)) if big else int(rng.integers(1, 400))
        q_pad, kv_pad = 4 * int(rng.integers(0, 9)), 4 * int(rng.integers(0, 9))
        mul = float(rng.choice([0.5, 1.0])) if prec != FP32 else float(rng.choice([0.5, 1.0, 2.0]))
        scale = float(rng.choice([0.0, 0.0, 0.05, 0.3]))
        cases.append((i, prec, m, hq, hkv, d, q_pad, kv_pad, mul, scale, big))
    return cases


def _decode_cases(n=32, seed=20261204):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 12, 16]))
        while hkv * g > 64:
            g //= 2
        hq = hkv * g
        d = int(rng.choice([32, 64, 128]))
        S = int(rng.integers(1, 40001))
        T = int(rng.integers(1, S + 1))
        W = 0 if rng.random() < 0.5 else int(rng.integers(1, T + 100))
        fused = bool(rng.random() < 0.5)
        rope = fused and bool(rng.random() < 0.5)
        scale = float(rng.choice([0.0, 0.0, 0.02, 0.2]))
        cases.append((i, hq, hkv, d, S, T, W, fused, rope, scale))
    return cases


def _wide_prefill_cases(n=32, seed=99101):
    """Longer prompts (up to 6000 tokens, up to 32 query heads): more split
    plans and grids of several waves."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        prec = int(rng.choice([FP32, FP16, FP16, FP16, BF16]))
        d = int(rng.choice([64, 128])) if prec != FP32 else int(rng.choice([32, 64, 128]))
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8]))
        while hkv * g > 32:
            g //= 2
        m = int(rng.integers(1, 6001)) if prec != FP32 else int(rng.integers(1, 3001))
        cases.append((100 + i, prec, m, hkv * g, hkv, d, 4 * int(rng.integers(0, 9)),
                      4 * int(rng.integers(0, 9)), float(rng.choice([0.5, 1.0])),
                      float(rng.choice([0.0, 0.0, 0.05])), m > 1200))
    return cases


def _wide_decode_cases(n=32, seed=99102):
    """Caches up to 100000 rows and GQA groups up to 16 (several warp steps,
    the one-step-ahead L2 prefetch, ragged tails)."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        hkv = int(rng.choice([1, 2, 3, 4, 8]))
        g = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16]))
        while hkv * g > 64:
            g //= 2
        d = int(rng.choice([32, 64, 128]))
        S = int(rng.integers(1, 100001))
        T = int(rng.integers(1, S + 1))
        W = 0 if rng.random() < 0.5 else int(rng.integers(1, T + 100))
        fused = bool(rng.random() < 0.5)
        rope = fused and bool(rng.random() < 0.5)
        cases.append((100 + i, hkv * g, hkv, d, S, T, W, fused, rope,
                      float(rng.choice([0.0, 0.02]))))
    return cases


@pytest.fixture(scope="module")
def attn():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import attention_attn_prefill_causal_gb300 as a
    assert a.attn_get_device_status() == a.ATTN_OK
    return a


@pytest.mark.parametrize("case", _prefill_cases() + _wide_prefill_cases()
                         + _tf32_variants(_prefill_cases() + _wide_prefill_cases()),
                         ids=lambda c: f"p{c[0]}")
def test_fuzz_prefill(attn, case):
    i, prec, m, hq, hkv, d, q_pad, kv_pad, mul, scale, big = case
    qs, kvs = hq * d + q_pad, hkv * d + kv_pad
    q, k, v = workloads.prefill_inputs(m, qs, kvs, seed=1000 + i % 500, mul=mul)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    buf, o = guarded_empty(m * qs)
    attn.attn_prefill_causal(dq, dk, dv, o, m, hq, hkv, d, qs, kvs, scale=scale, precision=prec)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf) and untouched_columns(o, m, qs, hq, d)
    rows = workloads.sample_rows(m, 2000 + i, 16, 16, 32) if big else None
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs,
                                scale=scale if scale > 0 else None, rows=rows)
    got = heads_view(o, m, qs, hq, d)
    if rows is not None:
        got = got[rows]
    amax, rel = compare(got, ref)
    if prec == FP32:
        assert amax <= FP32_ABS and rel <= FP32_REL, (case, amax, rel)
    else:
        widen = max(1.0, scale * d ** 0.5)
        assert amax <= (BF16_ABS if prec == BF16 else TC_ABS) * widen, (case, amax)


def _rope_tables(d, seed):
    theta = np.random.default_rng(seed).uniform(-3.0, 3.0, d // 2)
    return np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)


@pytest.mark.parametrize("case", _decode_cases() + _wide_decode_cases(), ids=lambda c: f"d{c[0]}")
def test_fuzz_decode(attn, case):
    i, hq, hkv, d, S, T, W, fused, rope, scale = case
    q, kc, vc, kn, vn = workloads.decode_inputs(hq, hkv, d, S, seed=3000 + i, append=True)
    dk, dv = kc.cuda(), vc.cuda()
    buf, out = guarded_empty(hq * d)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    sc = scale if scale > 0 else None
    if fused:
        pos = T - 1
        cos = sin = None
        if rope:
            cos, sin = _rope_tables(d, i)
        attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), dk, dv, out, hq, hkv, d, S, T,
                                pos, window=W, scale=scale,
                                rope_cos=torch.from_numpy(cos).cuda() if rope else None,
                                rope_sin=torch.from_numpy(sin).cuda() if rope else None)
        ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kh, vh, hq, hkv, d, S, T,
                                   pos, window=W, scale=sc, rope_cos=cos, rope_sin=sin)
    else:
        attn.attn_decode(q.cuda(), dk, dv, out, hq, hkv, d, S, T, window=W, scale=scale)
        ref = oracle.decode(q.numpy(), kh, vh, hq, hkv, d, S, T, W, scale=sc)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf)
    amax, rel = compare(out.view(hq, d).cpu().numpy(), ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (case, amax, rel)
    if fused:
        np.testing.assert_allclose(dk[:, T - 1].cpu().numpy(), kh[:, T - 1], rtol=0, atol=2e-6)
        np.testing.assert_array_equal(dv[:, T - 1].cpu().numpy(), vh[:, T - 1])
