"""Pins for the fp64 CPU oracle (runs without a GPU).

The pages print no attention output values, so the oracle is pinned to what
the mathematics and the pages fix: closed forms, invariants, special cases
that reduce to a library routine, page examples (tests/golden/), and brute
force on tiny inputs.  Each test names the passage it follows and the kind of
mistake in the oracle it would catch.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")


def _rand(shape, seed, mul=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * mul).numpy()


def _packed(m, hq, hkv, d, seed, q_pad=0, kv_pad=0, mul=1.0):
    q_stride, kv_stride = hq * d + q_pad, hkv * d + kv_pad
    q, k, v = workloads.prefill_inputs(m, q_stride, kv_stride, seed, mul)
    return q.numpy(), k.numpy(), v.numpy(), q_stride, kv_stride


def _head(x, row_pitch_cols, h, d):
    """View of head h as [rows, d] from a [rows, pitch] array."""
    return x[:, h * d:(h + 1) * d]


# ---------------------------------------------------------------- special cases

def test_decode_total_seq_one_is_v_row0():
    """honeycrisp attention.rs, kbypass: total_seq = 1 attention writes
    v_cache[kv_h, 0, :].  Catches a wrong normalisation or GQA route."""
    fx = json.load(open(GOLDEN))["total_seq_one"]
    hq, hkv, d, s = 8, 2, 64, 16
    q = _rand((hq, d), 1)
    kc, vc = _rand((hkv, s, d), 2), _rand((hkv, s, d), 3)
    out = oracle.decode(q, kc, vc, hq, hkv, d, s, fx["total_seq"])
    for h in range(hq):
        np.testing.assert_array_equal(out[h], vc[h // (hq // hkv), 0].astype(np.float64))


def test_prefill_row0_is_v_row0():
    """prefill_fused.rs, causal column loop j = 0..=i: row 0 attends only to
    key 0, so O[0, h] = V[0, kv_head(h)] exactly."""
    m, hq, hkv, d = 9, 6, 3, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 7)
    out = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    for h in range(hq):
        g = h // (hq // hkv)
        np.testing.assert_array_equal(out[0, h], v[0, g * d:(g + 1) * d].astype(np.float64))


def test_gqa_routing_page_example():
    """prefill_fused.rs, heads_per_kv doc: 6 query heads per KV head for 12Q/2KV,
    kv_head = head_idx / heads_per_kv (consecutive grouping, not h % kv_heads).
    Distinct constant V per KV head makes the route visible."""
    fx = json.load(open(GOLDEN))["gqa_example"]
    hq, hkv, G = fx["num_q_heads"], fx["num_kv_heads"], fx["heads_per_kv"]
    assert hq // hkv == G
    d, s = 32, 4
    q = _rand((hq, d), 11)
    kc = _rand((hkv, s, d), 12)
    vc = np.stack([np.full((s, d), 10.0 * (g + 1), np.float32) for g in range(hkv)])
    out = oracle.decode(q, kc, vc, hq, hkv, d, s, s)
    got = [int(round(out[h, 0] / 10.0)) - 1 for h in range(hq)]
    assert got == [h // G for h in range(hq)]
    # The same route in prefill (row 3 of a 4-token sequence).
    qp = np.zeros((s, hq * d), np.float32)
    kp = np.zeros((s, hkv * d), np.float32)
    vp = np.concatenate([np.full((s, d), 10.0 * (g + 1), np.float32) for g in range(hkv)], 1)
    outp = oracle.prefill_causal(qp, kp, vp, s, hq, hkv, d, hq * d, hkv * d)
    assert [int(round(outp[3, h, 0] / 10.0)) - 1 for h in range(hq)] == got


def test_two_key_closed_form_weights():
    """Softmax of two scores 0 and ln 3 gives weights 1/4 and 3/4.  Row 1 of a
    causal prefill with scale 1/sqrt(d) (prefill_fused.rs, compile-time scale):
    q = e0 * a, K[0] = 0, K[1] = e0 * b with a*b*scale = ln 3.  V rows one-hot.
    Catches a dropped scale, a wrong sign, exp vs exp2, or a missing normalise."""
    d = 32
    scale = 1.0 / math.sqrt(d)
    a = np.float32(2.0)
    b = np.float32(math.log(3.0) / (scale * 2.0))
    q = np.zeros((2, d), np.float32)
    q[1, 0] = a
    k = np.zeros((2, d), np.float32)
    k[1, 0] = b
    v = np.zeros((2, d), np.float32)
    v[0, 0] = 1.0
    v[1, 1] = 1.0
    out, w = oracle.prefill_causal(q, k, v, 2, 1, 1, d, d, d, return_weights=True)
    s1 = scale * float(a) * float(b)          # the exact score of the fp32 inputs
    w1 = math.exp(s1) / (1.0 + math.exp(s1))
    assert abs(w1 - 0.75) < 1e-6
    np.testing.assert_allclose(w[1, 0], [1.0 - w1, w1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[1, 0, :2], [1.0 - w1, w1], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(out[1, 0, 2:], 0.0)


def test_decode_scale_is_runtime_argument():
    """honeycrisp attention.rs Params.scale is a runtime value: doubling the
    scale squares the two-key weight ratio (e^{2s} vs e^{s})."""
    d = 32
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 1.0
    kc = np.zeros((1, 2, d), np.float32)
    kc[0, 1, 0] = 1.0
    vc = np.zeros((1, 2, d), np.float32)
    vc[0, 0, 0] = 1.0
    vc[0, 1, 1] = 1.0
    for sc in (0.5, 1.0, 2.0):
        out = oracle.decode(q, kc, vc, 1, 1, d, 2, 2, scale=sc)
        assert abs(out[0, 1] / out[0, 0] - math.exp(sc)) < 1e-12


# ---------------------------------------------------------------- invariants

def test_constant_keys_give_mean_of_values():
    """Equal keys give equal scores, so softmax is uniform: row i of a causal
    prefill is the mean of V[0..i]; decode is the mean of V[0..T).  The mean
    is numpy's (a library routine), not the oracle's loop."""
    m, hq, hkv, d = 12, 4, 2, 32
    q, _, v, qs, kvs = _packed(m, hq, hkv, d, 21)
    k = np.tile(_rand((1, kvs), 22), (m, 1))
    out = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    for h in range(hq):
        g = h // (hq // hkv)
        vh = v[:, g * d:(g + 1) * d].astype(np.float64)
        for i in range(m):
            np.testing.assert_allclose(out[i, h], vh[:i + 1].mean(0), rtol=0, atol=1e-13)
    T = 10
    qd = _rand((hq, d), 23)
    kc = np.tile(_rand((hkv, 1, d), 24), (1, 16, 1))
    vc = _rand((hkv, 16, d), 25)
    outd = oracle.decode(qd, kc, vc, hq, hkv, d, 16, T)
    for h in range(hq):
        np.testing.assert_allclose(outd[h], vc[h // 2, :T].astype(np.float64).mean(0),
                                   rtol=0, atol=1e-13)


def test_scale_zero_gives_mean_of_values():
    """scale -> 0 makes every score 0: the output is the mean of the attended V
    rows.  Catches a scale applied after the softmax or to the output."""
    m, hq, hkv, d = 7, 2, 1, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 31)
    out = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs, scale=0.0)
    v64 = v[:, :d].astype(np.float64)
    for i in range(m):
        for h in range(hq):
            np.testing.assert_allclose(out[i, h], v64[:i + 1].mean(0), rtol=0, atol=1e-13)


def test_huge_scale_gives_the_argmax_value_row():
    """With a very large scale the softmax becomes an argmax: each output is
    the V row of the key with the highest score (unique for random inputs).
    Scores reach about 1e5 here, so an oracle that exponentiates without
    subtracting the row max overflows; a scale applied in the wrong place
    picks the wrong row."""
    m, hq, hkv, d = 9, 2, 1, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 57)
    big = 2.0e4
    out = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs, scale=big)
    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    for i in range(m):
        for h in range(hq):
            s = k64[:i + 1, :d] @ q64[i, h * d:(h + 1) * d]
            order = np.sort(s)
            if i > 0:
                assert big * (order[-1] - order[-2]) > 50  # the argmax is decisive
            np.testing.assert_allclose(out[i, h], v64[int(np.argmax(s)), :d], rtol=0, atol=1e-12)
    S = 16
    qd, kc, vc = _rand((hq, d), 58), _rand((hkv, S, d), 59), _rand((hkv, S, d), 60)
    outd = oracle.decode(qd, kc, vc, hq, hkv, d, S, S, 0, scale=big)
    for h in range(hq):
        s = kc[0].astype(np.float64) @ qd[h].astype(np.float64)
        np.testing.assert_allclose(outd[h], vc[0, int(np.argmax(s))], rtol=0, atol=1e-12)


def test_key_shift_invariance():
    """Adding one vector c to every key adds scale*q.c to every score of a query,
    which softmax cancels (shift invariance)."""
    m, hq, hkv, d = 10, 4, 2, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 41)
    c = _rand((1, kvs), 42)
    a = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    b = oracle.prefill_causal(q, (k + c).astype(np.float32), v, m, hq, hkv, d, qs, kvs)
    # k + c is rounded to fp32, so the score shift is only nearly constant.
    np.testing.assert_allclose(a, b, rtol=0, atol=2e-5)


def test_value_affine_map():
    """Softmax weights sum to 1, so V -> V A + b maps O -> O A + b (per head)."""
    m, hq, hkv, d = 8, 2, 2, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 51)
    A = _rand((d, d), 52, 0.2).astype(np.float64)
    bvec = _rand((d,), 53).astype(np.float64)
    out = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    v2 = np.empty_like(v)
    for g in range(hkv):
        v2[:, g * d:(g + 1) * d] = (v[:, g * d:(g + 1) * d].astype(np.float64) @ A + bvec).astype(np.float32)
    out2 = oracle.prefill_causal(q, k, v2, m, hq, hkv, d, qs, kvs)
    np.testing.assert_allclose(out2, out @ A + bvec, rtol=0, atol=5e-6)


def test_weights_are_a_causal_distribution():
    """Materialised prefill weights: nonnegative, zero above the diagonal
    (prefill_fused.rs causal limit j <= i), summing to 1 per row."""
    m, hq, hkv, d = 16, 4, 1, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 61)
    _, w = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs, return_weights=True)
    assert (w >= 0).all()
    for i in range(m):
        assert (w[i, :, i + 1:] == 0).all()
        assert (w[i, :, :i + 1] > 0).all()
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-14)
    qd = _rand((hq, d), 62)
    kc, vc = _rand((hkv, 20, d), 63), _rand((hkv, 20, d), 64)
    _, wd = oracle.decode(qd, kc, vc, hq, hkv, d, 20, 17, return_weights=True)
    np.testing.assert_allclose(wd.sum(-1), 1.0, rtol=0, atol=1e-14)


def test_gqa_equals_mha_with_repeated_kv():
    """GQA with G = Hq/Hkv equals MHA whose KV heads repeat each original head
    G times in order (consecutive grouping)."""
    m, hq, hkv, d = 9, 6, 2, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 71)
    G = hq // hkv
    k_rep = np.concatenate([k[:, (h // G) * d:(h // G + 1) * d] for h in range(hq)], 1)
    v_rep = np.concatenate([v[:, (h // G) * d:(h // G + 1) * d] for h in range(hq)], 1)
    a = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    b = oracle.prefill_causal(q, np.ascontiguousarray(k_rep), np.ascontiguousarray(v_rep),
                              m, hq, hq, d, qs, hq * d)
    np.testing.assert_array_equal(a, b)
    qd = _rand((hq, d), 72)
    kc, vc = _rand((hkv, 12, d), 73), _rand((hkv, 12, d), 74)
    kr, vr = np.repeat(kc, G, axis=0), np.repeat(vc, G, axis=0)
    np.testing.assert_array_equal(oracle.decode(qd, kc, vc, hq, hkv, d, 12, 11),
                                  oracle.decode(qd, kr, vr, hq, hq, d, 12, 11))


def test_prefill_row_equals_decode_prefix():
    """Cross-form: row i of causal prefill equals single-query decode over the
    first i+1 cache rows (prefill_fused.rs algorithm vs honeycrisp kmain)."""
    m, hq, hkv, d = 14, 4, 2, 64
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 81)
    out = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    kc = np.ascontiguousarray(k.reshape(m, hkv, d).transpose(1, 0, 2))
    vc = np.ascontiguousarray(v.reshape(m, hkv, d).transpose(1, 0, 2))
    for i in range(m):
        qi = np.ascontiguousarray(q[i, :hq * d].reshape(hq, d))
        od = oracle.decode(qi, kc, vc, hq, hkv, d, m, i + 1)
        np.testing.assert_allclose(out[i], od, rtol=0, atol=1e-14)


def test_packed_single_buffer_layout():
    """prefill_fused.rs packed layout: Q, K, V read through independent row
    pitches.  One packed [M, (Hq+2Hkv)D] buffer with q = col 0, k = col Hq*D,
    v = col (Hq+Hkv)*D and all strides equal must match tight separate buffers."""
    m, hq, hkv, d = 11, 4, 2, 32
    W = (hq + 2 * hkv) * d
    buf = _rand((m, W), 91)
    q = np.ascontiguousarray(buf[:, :hq * d])
    k = np.ascontiguousarray(buf[:, hq * d:(hq + hkv) * d])
    v = np.ascontiguousarray(buf[:, (hq + hkv) * d:])
    a = oracle.prefill_causal(q, k, v, m, hq, hkv, d, hq * d, hkv * d)
    flat = buf.reshape(-1)
    b = oracle.prefill_causal(flat, flat[hq * d:], flat[(hq + hkv) * d:], m, hq, hkv, d, W, W)
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------- window

def test_window_off_and_at_least_total_seq():
    """honeycrisp kmain window_start: window = 0 is off, and window >= total_seq
    masks nothing."""
    hq, hkv, d, S, T = 4, 2, 32, 40, 33
    q = _rand((hq, d), 101)
    kc, vc = _rand((hkv, S, d), 102), _rand((hkv, S, d), 103)
    base = oracle.decode(q, kc, vc, hq, hkv, d, S, T, window=0)
    for W in (T, T + 1, 1000):
        np.testing.assert_array_equal(oracle.decode(q, kc, vc, hq, hkv, d, S, T, window=W), base)


def test_window_equals_attention_over_last_rows():
    """With N(0,1) data the -1e4 replacement weight e^{-1e4-m} underflows to 0
    in double, so windowed decode equals plain decode over rows
    [T-W, T).  Catches an off-by-one in window_start."""
    hq, hkv, d, S = 8, 2, 64, 64
    q = _rand((hq, d), 111)
    kc, vc = _rand((hkv, S, d), 112), _rand((hkv, S, d), 113)
    for T, W in [(64, 16), (50, 1), (33, 32), (64, 63)]:
        ws = T - W
        ks = np.ascontiguousarray(kc[:, ws:T])
        vs = np.ascontiguousarray(vc[:, ws:T])
        a = oracle.decode(q, kc, vc, hq, hkv, d, S, T, window=W)
        b = oracle.decode(q, ks, vs, hq, hkv, d, W, W)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
        _, w = oracle.decode(q, kc, vc, hq, hkv, d, S, T, window=W, return_weights=True)
        assert (w[:, :ws] == 0).all() and (w[:, ws:] > 0).all()


def test_window_mask_replaces_score_with_minus_1e4():
    """honeycrisp kmain: a masked score is REPLACED by -1e4 (not -inf, not
    -1e4 added).  With one masked row (score -> -1e4) and one live row whose
    score is -1e4 + ln 3, the weights are 1/4 and 3/4."""
    fx = json.load(open(GOLDEN))["window_mask_value"]
    d = 32
    scale = 1.0
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 1.0
    kc = np.zeros((1, 2, d), np.float32)
    kc[0, 0, 0] = 5.0                                  # masked: its own score is ignored
    kc[0, 1, 0] = np.float32(fx["mask_score"] + math.log(3.0))
    vc = np.zeros((1, 2, d), np.float32)
    vc[0, 0, 0] = 1.0
    vc[0, 1, 1] = 1.0
    out = oracle.decode(q, kc, vc, 1, 1, d, 2, 2, window=1, scale=scale)
    delta = float(kc[0, 1, 0]) - fx["mask_score"]      # exact live-minus-mask gap
    w1 = 1.0 / (1.0 + math.exp(-delta))
    np.testing.assert_allclose(out[0, :2], [1.0 - w1, w1], rtol=0, atol=1e-12)
    assert abs(w1 - 0.75) < 1e-3


# ---------------------------------------------------------------- brute force

def _naive_prefill(q, k, v, m, hq, hkv, d, qs, kvs, scale):
    """Pure-Python loops, written independently of the C oracle."""
    G = hq // hkv
    out = np.zeros((m, hq, d))
    for i in range(m):
        for h in range(hq):
            g = h // G
            sc = []
            for j in range(i + 1):
                sc.append(scale * sum(float(q[i, h * d + e]) * float(k[j, g * d + e]) for e in range(d)))
            mx = max(sc)
            ex = [math.exp(s - mx) for s in sc]
            tot = sum(ex)
            for e in range(d):
                out[i, h, e] = sum(ex[j] * float(v[j, g * d + e]) for j in range(i + 1)) / tot
    return out


def test_brute_force_prefill_tiny():
    for (m, hq, hkv, d, seed) in [(1, 1, 1, 32, 1), (5, 2, 1, 32, 2), (8, 4, 2, 32, 3), (3, 3, 3, 32, 4)]:
        q, k, v, qs, kvs = _packed(m, hq, hkv, d, 120 + seed, q_pad=32, kv_pad=32)
        sc = 1.0 / math.sqrt(d)
        np.testing.assert_allclose(oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs),
                                   _naive_prefill(q, k, v, m, hq, hkv, d, qs, kvs, sc),
                                   rtol=0, atol=1e-13)


def test_library_sdpa_prefill_and_decode():
    """torch.nn.functional.scaled_dot_product_attention in float64 on the CPU,
    with an explicit boolean causal / window mask and K/V repeat_interleave(G)."""
    F = torch.nn.functional
    m, hq, hkv, d = 8, 4, 2, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 131)
    G = hq // hkv
    Q = torch.from_numpy(q).double().view(m, hq, d).transpose(0, 1)
    K = torch.from_numpy(k).double().view(m, hkv, d).transpose(0, 1).repeat_interleave(G, 0)
    V = torch.from_numpy(v).double().view(m, hkv, d).transpose(0, 1).repeat_interleave(G, 0)
    mask = torch.ones(m, m, dtype=torch.bool).tril()
    ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask).transpose(0, 1).numpy()
    np.testing.assert_allclose(oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs), ref,
                               rtol=0, atol=1e-13)
    # decode, windowed: positions below T-W are excluded (their weight underflows)
    S, T, W = 8, 7, 4
    qd = _rand((hq, d), 132)
    kc, vc = _rand((hkv, S, d), 133), _rand((hkv, S, d), 134)
    Qd = torch.from_numpy(qd).double().view(hq, 1, d)
    Kd = torch.from_numpy(kc[:, :T]).double().repeat_interleave(G, 0)
    Vd = torch.from_numpy(vc[:, :T]).double().repeat_interleave(G, 0)
    wm = torch.zeros(1, T, dtype=torch.bool)
    wm[:, T - W:] = True
    refd = F.scaled_dot_product_attention(Qd, Kd, Vd, attn_mask=wm).view(hq, d).numpy()
    np.testing.assert_allclose(oracle.decode(qd, kc, vc, hq, hkv, d, S, T, window=W), refd,
                               rtol=0, atol=1e-13)


# ---------------------------------------------------------------- kv_append

def test_kv_append_literal_copy():
    """honeycrisp KV_APPEND_BOTH_TEMPLATE: cache[h, position, d] = src[h, d];
    every other cache element is untouched (bit-exact)."""
    hkv, d, S = 3, 32, 10
    kc, vc = _rand((hkv, S, d), 141), _rand((hkv, S, d), 142)
    ks, vs = _rand((hkv, d), 143), _rand((hkv, d), 144)
    for pos in (0, 4, S - 1):
        k2, v2 = kc.copy(), vc.copy()
        oracle.kv_append(ks, vs, k2, v2, hkv, d, S, pos)
        np.testing.assert_array_equal(k2[:, pos], ks)
        np.testing.assert_array_equal(v2[:, pos], vs)
        keep = [p for p in range(S) if p != pos]
        np.testing.assert_array_equal(k2[:, keep], kc[:, keep])
        np.testing.assert_array_equal(v2[:, keep], vc[:, keep])
    k3 = kc.copy()
    oracle.kv_append(ks, None, k3, None, hkv, d, S, 2)     # single-cache form
    np.testing.assert_array_equal(k3[:, 2], ks)


def test_append_then_decode_sees_new_row():
    """Append at position T-1 then decode with total_seq = T and window 1: only
    the appended row is live, so out = v_new (after the mask's underflow)."""
    hq, hkv, d, S = 4, 2, 32, 16
    q = _rand((hq, d), 151)
    kc, vc = _rand((hkv, S, d), 152), _rand((hkv, S, d), 153)
    kn, vn = _rand((hkv, d), 154), _rand((hkv, d), 155)
    oracle.kv_append(kn, vn, kc, vc, hkv, d, S, S - 1)
    out = oracle.decode(q, kc, vc, hq, hkv, d, S, S, window=1)
    for h in range(hq):
        np.testing.assert_allclose(out[h], vn[h // 2].astype(np.float64), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- arguments

def test_oracle_rejects_undefined_arguments():
    d = 32
    q = np.zeros((2, d), np.float32)
    kc = np.zeros((1, 4, d), np.float32)
    with pytest.raises(ValueError):
        oracle.decode(q, kc, kc, 2, 1, d, 4, 0)           # total_seq = 0: no softmax
    with pytest.raises(ValueError):
        oracle.decode(q, kc, kc, 2, 1, d, 4, 5)           # total_seq > max_seq
    with pytest.raises(ValueError):
        oracle.kv_append(q[:1], q[:1], kc, kc.copy(), 1, d, 4, 4)   # position >= max_seq
    qp = np.zeros((4, 64), np.float32)
    with pytest.raises(ValueError):
        oracle.prefill_causal(qp, qp, qp, 4, 3, 2, 32, 96, 64)      # 3 % 2 != 0
    with pytest.raises(ValueError):
        oracle.prefill_causal(qp, qp, qp, 2, 4, 2, 32, 64, 64)      # q_stride < Hq*D


def test_sampled_rows_match_full():
    """The row-subset entry (used at full sizes) returns exactly the full rows."""
    m, hq, hkv, d = 40, 4, 2, 32
    q, k, v, qs, kvs = _packed(m, hq, hkv, d, 161)
    full = oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs)
    rows = [0, 3, 17, 39]
    np.testing.assert_array_equal(oracle.prefill_causal(q, k, v, m, hq, hkv, d, qs, kvs, rows=rows),
                                  full[rows])


# ---------------------------------------------------------------- fused RoPE + append + decode

def _complex_rotate(x, theta):
    """Rotate-half RoPE written as complex multiplication: pair (x[i], x[i+h])
    is the complex number x[i] + 1j*x[i+h], multiplied by exp(1j*theta[i])."""
    h = x.shape[-1] // 2
    z = (x[..., :h].astype(np.float64) + 1j * x[..., h:].astype(np.float64)) * np.exp(1j * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_decode_append_without_rope_is_append_then_decode():
    """honeycrisp FUSED_ROPE_KV_ATTN_TEMPLATE with no rotation reduces to
    KV_APPEND_BOTH_TEMPLATE followed by kmain."""
    hq, hkv, d, S, T = 8, 2, 64, 40, 33
    q = _rand((hq, d), 201)
    kc, vc = _rand((hkv, S, d), 202), _rand((hkv, S, d), 203)
    kn, vn = _rand((hkv, d), 204), _rand((hkv, d), 205)
    k1, v1 = kc.copy(), vc.copy()
    out = oracle.decode_append(q, kn, vn, k1, v1, hq, hkv, d, S, T, T - 1, window=8)
    k2, v2 = kc.copy(), vc.copy()
    oracle.kv_append(kn, vn, k2, v2, hkv, d, S, T - 1)
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(v1, v2)
    np.testing.assert_array_equal(out, oracle.decode(q, k2, v2, hq, hkv, d, S, T, window=8))


def test_rope_quarter_turn_closed_form():
    """cos = 0, sin = 1 rotates every pair by 90 degrees:
    y[i] = -x[i+h], y[i+h] = x[i] (exact in fp32)."""
    hq, hkv, d, S = 2, 1, 32, 4
    q = _rand((hq, d), 211)
    kc, vc = _rand((hkv, S, d), 212), _rand((hkv, S, d), 213)
    kn, vn = _rand((hkv, d), 214), _rand((hkv, d), 215)
    cos = np.zeros(d // 2, np.float32)
    sin = np.ones(d // 2, np.float32)
    oracle.decode_append(q, kn, vn, kc, vc, hq, hkv, d, S, S, 2, rope_cos=cos, rope_sin=sin)
    np.testing.assert_array_equal(kc[0, 2], np.concatenate([-kn[0, d // 2:], kn[0, :d // 2]]))
    np.testing.assert_array_equal(vc[0, 2], vn[0])


def test_rope_matches_complex_rotation_and_keeps_norms():
    hkv, d, S = 3, 64, 8
    theta = np.random.default_rng(7).uniform(-3, 3, d // 2)
    cos, sin = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    q = _rand((6, d), 221)
    kc, vc = _rand((hkv, S, d), 222), _rand((hkv, S, d), 223)
    kn, vn = _rand((hkv, d), 224), _rand((hkv, d), 225)
    oracle.decode_append(q, kn, vn, kc, vc, 6, hkv, d, S, S, 5, rope_cos=cos, rope_sin=sin)
    # the fp32 tables are not exactly on the unit circle: rotate by their angle
    # and scale by their radius
    th32 = np.arctan2(sin.astype(np.float64), cos.astype(np.float64))
    rad = np.hypot(cos.astype(np.float64), sin.astype(np.float64))
    ref = _complex_rotate(kn, th32) * np.concatenate([rad, rad])
    np.testing.assert_allclose(kc[:, 5], ref, rtol=0, atol=2e-6)
    np.testing.assert_allclose(np.linalg.norm(kc[:, 5].astype(np.float64), axis=1),
                               np.linalg.norm(kn.astype(np.float64), axis=1), rtol=1e-6)


def test_rope_same_angle_leaves_scores_unchanged():
    """Rotating the query and every key by the same angles keeps each q.k
    (RoPE is a rotation): prerotate the old keys with the complex form, append
    a rotated key, and the result equals plain append + decode on the
    unrotated vectors."""
    hq, hkv, d, S, T = 4, 2, 32, 12, 12
    theta = np.random.default_rng(3).uniform(-3, 3, d // 2)
    cos, sin = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    th = np.arctan2(sin.astype(np.float64), cos.astype(np.float64))
    q = _rand((hq, d), 231)
    kc, vc = _rand((hkv, S, d), 232), _rand((hkv, S, d), 233)
    kn, vn = _rand((hkv, d), 234), _rand((hkv, d), 235)
    k_rot = _complex_rotate(kc, th).astype(np.float32)
    v1 = vc.copy()
    got = oracle.decode_append(q, kn, vn, k_rot, v1, hq, hkv, d, S, T, T - 1, rope_cos=cos,
                               rope_sin=sin)
    k_plain = _complex_rotate(_complex_rotate(kc, th).astype(np.float32), -th).astype(np.float32)
    v2 = vc.copy()
    ref = oracle.decode_append(q, kn, vn, k_plain, v2, hq, hkv, d, S, T, T - 1)
    np.testing.assert_allclose(got, ref, rtol=0, atol=5e-5)
