"""GPU parity: every call goes through the C ABI (libattn.so) on cuda:0 and is
compared element by element with the fp64 CPU oracle on the same seeded
inputs.  Tolerances: fp32 CUDA-core paths max abs <= 1e-4 and normwise
relative <= 1e-4; tensor-core (fp16-operand) prefill max abs <= 3e-3.
Output buffers are NaN-poisoned with canary bands on both sides."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity_utils import (FP32_ABS, FP32_REL, TC_ABS, compare, guarded_empty,
                                guards_intact, heads_view, untouched_columns)

pytestmark = pytest.mark.gpu

FP32, FP16, TF32 = 0, 1, 3


@pytest.fixture(scope="module")
def attn():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import attention_attn_prefill_causal_gb300 as a
    assert a.attn_get_device_status() == a.ATTN_OK
    return a


def _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, prec, scale=0.0):
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    buf, o = guarded_empty(m * qs)
    attn.attn_prefill_causal(dq, dk, dv, o, m, hq, hkv, d, qs, kvs, scale=scale, precision=prec)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf)
    assert untouched_columns(o, m, qs, hq, d)
    return heads_view(o, m, qs, hq, d)


def _check_prefill(attn, m, hq, hkv, d, prec, seed, q_pad=0, kv_pad=0, mul=1.0, rows=None):
    qs, kvs = hq * d + q_pad, hkv * d + kv_pad
    q, k, v = workloads.prefill_inputs(m, qs, kvs, seed, mul)
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, prec)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs, rows=rows)
    if rows is not None:
        got = got[rows]
    amax, rel = compare(got, ref)
    if prec == FP32:
        assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)
    else:
        assert amax <= TC_ABS, amax
    return amax, rel


# ------------------------------------------------------------------ named workloads

def test_workload_prefill_small_fp32(attn):
    c = workloads.PREFILL_SMALL
    amax, rel = _check_prefill(attn, c.m, c.num_q_heads, c.num_kv_heads, c.head_dim, FP32, c.seed)
    print(f"{c.name}: max abs {amax:.3e} rel {rel:.3e}")


@pytest.mark.parametrize("prec", [FP16, TF32])
def test_workload_prefill_2k_tensor_core(attn, prec):
    c = workloads.PREFILL_2K
    amax, rel = _check_prefill(attn, c.m, c.num_q_heads, c.num_kv_heads, c.head_dim, prec, c.seed)
    print(f"{c.name} tensor path (precision {prec}): max abs {amax:.3e} rel {rel:.3e}")


def test_workload_prefill_2k_fp32(attn):
    c = workloads.PREFILL_2K
    amax, rel = _check_prefill(attn, c.m, c.num_q_heads, c.num_kv_heads, c.head_dim, FP32, c.seed)
    print(f"{c.name} fp32 path: max abs {amax:.3e} rel {rel:.3e}")


@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_workload_prefill_16k_sampled_rows(attn, prec):
    c = workloads.PREFILL_16K
    rows = workloads.sample_rows(c.m, c.seed)
    q, k, v = workloads.shape_inputs(c)
    got = _run_prefill(attn, q, k, v, c.m, c.num_q_heads, c.num_kv_heads, c.head_dim, c.q_stride,
                       c.kv_stride, prec)
    assert np.isfinite(got).all()
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), c.m, c.num_q_heads,
                                c.num_kv_heads, c.head_dim, c.q_stride, c.kv_stride, rows=rows)
    amax, rel = compare(got[rows], ref)
    print(f"{c.name} prec={prec}: {len(rows)} rows, max abs {amax:.3e} rel {rel:.3e}")
    if prec == FP32:
        assert amax <= FP32_ABS and rel <= FP32_REL
    else:
        assert amax <= TC_ABS


def _run_decode(attn, q, kc, vc, hq, hkv, d, S, T, W, scale=0.0):
    buf, out = guarded_empty(hq * d)
    attn.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), out, hq, hkv, d, S, T, window=W, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf)
    return out.view(hq, d).cpu().numpy()


def test_workload_decode_4k(attn):
    c = workloads.DECODE_4K
    q, kc, vc, _, _ = workloads.shape_inputs(c)
    got = _run_decode(attn, q, kc, vc, c.num_heads, c.kv_heads, c.head_dim, c.max_seq,
                      c.total_seq, c.window)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), c.num_heads, c.kv_heads, c.head_dim,
                        c.max_seq, c.total_seq, c.window)
    amax, rel = compare(got, ref)
    print(f"{c.name}: max abs {amax:.3e} rel {rel:.3e}")
    assert amax <= FP32_ABS and rel <= FP32_REL


def test_workload_append_then_windowed_decode_32k(attn):
    c = workloads.DECODE_32K_WINDOW
    q, kc, vc, kn, vn = workloads.shape_inputs(c)
    dk, dv = kc.cuda(), vc.cuda()
    pos = c.total_seq - 1
    attn.kv_append(kn.cuda(), vn.cuda(), dk, dv, c.kv_heads, c.head_dim, c.max_seq, pos)
    buf, out = guarded_empty(c.num_heads * c.head_dim)
    attn.attn_decode(q.cuda(), dk, dv, out, c.num_heads, c.kv_heads, c.head_dim, c.max_seq,
                     c.total_seq, window=c.window)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    oracle.kv_append(kn.numpy(), vn.numpy(), kh, vh, c.kv_heads, c.head_dim, c.max_seq, pos)
    np.testing.assert_array_equal(dk[:, pos].cpu().numpy(), kh[:, pos])
    np.testing.assert_array_equal(dv[:, pos].cpu().numpy(), vh[:, pos])
    ref = oracle.decode(q.numpy(), kh, vh, c.num_heads, c.kv_heads, c.head_dim, c.max_seq,
                        c.total_seq, c.window)
    amax, rel = compare(out.view(c.num_heads, c.head_dim).cpu().numpy(), ref)
    print(f"{c.name}: max abs {amax:.3e} rel {rel:.3e}")
    assert amax <= FP32_ABS and rel <= FP32_REL


# ------------------------------------------------------------------ prefill edge cases

@pytest.mark.parametrize("m", [1, 2, 31, 127, 128, 129, 255, 256, 257, 300, 511, 640])
@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_prefill_ragged_lengths(attn, m, prec):
    _check_prefill(attn, m, 4, 2, 128, prec, seed=100 + m)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (3, 3), (7, 1), (8, 2), (14, 2)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_prefill_head_configs(attn, hq, hkv, d, prec):
    _check_prefill(attn, 300, hq, hkv, d, prec, seed=hq * 10 + hkv + d)


@pytest.mark.parametrize("d", [32, 64])
def test_prefill_fp32_small_head_dims(attn, d):
    _check_prefill(attn, 200, 6, 2, d, FP32, seed=d)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("m,hq,hkv", [(1000, 40, 8), (1000, 12, 2), (77, 40, 8), (1000, 2, 1)])
def test_prefill_fp32_every_query_block_size(attn, m, hq, hkv, d):
    """The fp32 kernel takes 64-row query blocks when there are at least four
    64-row blocks per SM (640 blocks here, the first case), 32-row blocks
    from one per SM (192, the second) and 16-row blocks below that (the last
    two); ragged tails in each, at every head_dim (the shared-memory layout
    of the weights differs)."""
    _check_prefill(attn, m, hq, hkv, d, FP32, seed=m + hq + d)


@pytest.mark.parametrize("prec", [FP16, TF32])
def test_prefill_long_sequence_sampled_rows(attn, prec):
    """32768 tokens over 2 query heads: query tiles walk up to 256 key tiles
    of 128 keys (512 of 64 keys in the TF32 mode), and the 256 CTAs take more
    than one wave on the SMs."""
    m, hq, hkv, d = 32768, 2, 1, 128
    rows = workloads.sample_rows(m, 321, n_random=128)
    amax, _ = _check_prefill(attn, m, hq, hkv, d, prec, seed=321, rows=rows)
    print(f"prefill m={m}: {len(rows)} rows, max abs {amax:.3e}")


@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_prefill_sharp_softmax(attn, prec):
    """scale 2 on N(0,1) inputs (head_dim 128): scores spread over about
    +-100 in log2 units, so the running max moves past the rescale threshold
    many times and the O rescale path runs often."""
    m, hq, hkv, d = 700, 4, 2, 128
    qs, kvs = hq * d, hkv * d
    q, k, v = workloads.prefill_inputs(m, qs, kvs, 77)
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, prec, scale=2.0)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs, scale=2.0)
    amax, rel = compare(got, ref)
    if prec == FP32:
        assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)
    else:
        # fp16 operand rounding perturbs a score by about scale*|q||k|*2^-11,
        # so the bound of the default scale 1/sqrt(d) grows by scale*sqrt(d).
        assert amax <= TC_ABS * 2.0 * math.sqrt(d), amax


def test_decode_sharp_softmax(attn):
    hq, hkv, d, S = 12, 2, 128, 4096
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=78)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, S, 0, scale=2.0)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, S, 0, scale=2.0)
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)


@pytest.mark.parametrize("prec", [FP16, TF32])
def test_prefill_split_into_many_key_chunks(attn, prec):
    """4096 tokens over 2 query heads leave most SMs idle, so the key walk of
    each query tile is split into chunks of 128-key blocks (nine blocks per
    chunk on 152 SMs): up to 4 chunk partials per row, a full batch of the
    combine.  Sampled rows include the first and last tiles."""
    m, hq, hkv, d = 4096, 2, 1, 64
    rows = workloads.sample_rows(m, 91)
    amax, _ = _check_prefill(attn, m, hq, hkv, d, prec, seed=91, rows=rows)
    print(f"split prefill m={m}: {len(rows)} rows, max abs {amax:.3e}")


@pytest.mark.parametrize("side", [-1, 0])
def test_prefill_fp16_kernel_choice_boundary(attn, side):
    """16-bit calls whose query-tile pairs fill the SMs twice over run the
    pair kernel, smaller ones the single-tile kernel.  16 heads and the
    token count at which pairs x heads reaches 2 x SMs (side 0: the pair
    kernel) or one pair less (side -1: the single-tile kernel), with sampled
    rows checked against the oracle on both sides."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    hq, hkv, d = 16, 4, 128
    pairs = -(-2 * sms // hq) + side
    m = 256 * pairs
    rows = workloads.sample_rows(m, 93 + side, 24, 24, 48)
    amax, _ = _check_prefill(attn, m, hq, hkv, d, FP16, seed=93 + side, rows=rows)
    print(f"fp16 m={m} ({pairs} pairs x {hq} heads, {sms} SMs): {len(rows)} rows, max abs {amax:.3e}")


@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_prefill_padded_strides(attn, prec):
    _check_prefill(attn, 333, 6, 2, 128, prec, seed=7, q_pad=64, kv_pad=128)


@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_stride_padding_is_never_read(attn, prec, d):
    """NaN in the padding columns between rows (past Hq*D in Q, past Hkv*D in
    K and V) must not reach the output: only the heads' columns are read."""
    m, hq, hkv = 333, 6, 2
    qs, kvs = hq * d + 64, hkv * d + 128
    q, k, v = workloads.prefill_inputs(m, qs, kvs, 71)
    q[:, hq * d:] = float("nan")
    k[:, hkv * d:] = float("nan")
    v[:, hkv * d:] = float("nan")
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, prec)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs)
    assert np.isfinite(ref).all() and np.isfinite(got).all()
    amax, rel = compare(got, ref)
    if prec == FP32:
        assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)
    else:
        assert amax <= TC_ABS, amax


@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_prefill_single_packed_buffer(attn, prec):
    """Q, K, V as column slices of one [M, (Hq+2Hkv)D] projection output with
    equal strides (the page's zero-copy packed layout)."""
    m, hq, hkv, d = 260, 4, 2, 128
    W = (hq + 2 * hkv) * d
    g = torch.Generator().manual_seed(55)
    buf = torch.randn(m, W, generator=g)
    dbuf = buf.cuda()
    flat = dbuf.view(-1)
    obuf, o = guarded_empty(m * W)
    attn.attn_prefill_causal(flat, flat[hq * d:], flat[(hq + hkv) * d:], o, m, hq, hkv, d, W, W,
                             precision=prec)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK and guards_intact(obuf)
    got = heads_view(o, m, W, hq, d)
    nb = buf.numpy().reshape(-1)
    ref = oracle.prefill_causal(nb, nb[hq * d:], nb[(hq + hkv) * d:], m, hq, hkv, d, W, W)
    amax, rel = compare(got, ref)
    assert amax <= (FP32_ABS if prec == FP32 else TC_ABS)


@pytest.mark.parametrize("prec", [FP16, TF32, FP32])
def test_prefill_explicit_scale(attn, prec):
    m, hq, hkv, d = 150, 2, 1, 64
    qs, kvs = hq * d, hkv * d
    q, k, v = workloads.prefill_inputs(m, qs, kvs, 9)
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, prec, scale=0.05)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs, scale=0.05)
    amax, _ = compare(got, ref)
    assert amax <= (FP32_ABS if prec == FP32 else TC_ABS)


def test_prefill_rows_beyond_m_untouched(attn):
    """A buffer with extra rows past m keeps them poisoned (no write past m)."""
    m, hq, hkv, d = 130, 2, 2, 128
    qs = hq * d
    q, k, v = workloads.prefill_inputs(m, qs, hkv * d, 3)
    for prec in (FP16, TF32, FP32):
        buf, o = guarded_empty((m + 126) * qs)
        attn.attn_prefill_causal(q.cuda(), k.cuda(), v.cuda(), o, m, hq, hkv, d, qs, hkv * d,
                                 precision=prec)
        torch.cuda.synchronize()
        assert torch.isnan(o[m * qs:]).all().item()
        assert torch.isfinite(o[: m * qs]).all().item()


@pytest.mark.parametrize("where", ["q", "k", "v"])
def test_prefill_tensor_path_rejects_fp16_overflow(attn, where):
    """An input beyond the fp16 range is flagged (ATTN_ERR_RANGE) instead of
    silently producing inf: K and V by the rounding pre-pass, Q by the
    prefill kernel's own rounding of its query tiles."""
    m, hq, hkv, d = 300, 2, 1, 64
    q, k, v = workloads.prefill_inputs(m, hq * d, hkv * d, 4)
    {"q": q, "k": k, "v": v}[where][257, 3] = -1.0e5   # inside the second query-tile pair
    buf, o = guarded_empty(m * hq * d)
    attn.attn_prefill_causal(q.cuda(), k.cuda(), v.cuda(), o, m, hq, hkv, d, hq * d, hkv * d,
                             precision=FP16)
    assert attn.attn_get_device_status() == attn.ATTN_ERR_RANGE
    assert attn.attn_get_device_status() == attn.ATTN_OK  # cleared by the read


# ------------------------------------------------------------------ decode edge cases

@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 100, 1023, 4095, 4096])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_decode_lengths(attn, T, d):
    hq, hkv, S = 8, 2, 4096
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=T + d)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, T, 0)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, 0)
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 4), (8, 1), (12, 1), (16, 2), (24, 2), (32, 8),
                                     (6, 2), (10, 2), (6, 1), (14, 2), (20, 2), (36, 3), (40, 4)])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_decode_gqa_groups(attn, hq, hkv, d):
    """Every head-pass width (1, 2, 4, 6, 8 query heads per CTA), idle head
    slots (groups of 3, 5, 7 and 10), and groups above 8 query heads per KV
    head, which take several CTA head-groups."""
    S, T = 2000, 1777
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=hq * 7 + hkv + d)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, T, 0)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, 0)
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL


@pytest.mark.parametrize("W", [0, 8191])
def test_decode_long_cache(attn, W):
    """131072 cached rows: each warp walks about 27 four-row steps (W = 0),
    or a window ending at the last row that starts inside a chunk."""
    hq, hkv, d, S = 12, 2, 128, 131072
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=131)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, S, W)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, S, W)
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)


@pytest.mark.parametrize("T,W", [(4096, 1), (4096, 7), (4096, 4095), (4096, 4096), (4096, 5000),
                                 (3000, 1024), (33, 32), (2, 1)])
def test_decode_windows(attn, T, W):
    hq, hkv, d, S = 8, 2, 128, 4096
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=T * 3 + W)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, T, W)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, W)
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL


def test_decode_masked_positions_keep_their_minus_1e4_weight(attn):
    """When every live score lies below -1e4 the masked positions (score
    replaced by -1e4) dominate the softmax; the combine then reads the masked
    V rows and reproduces the page's replaced-score result.  Scores of
    magnitude ~1e4 carry an fp32 resolution of ~1e-3 (log2 units), so the
    bound here is 1e-2 rather than the 1e-4 of ordinary inputs."""
    hq, hkv, d, S, T, W = 2, 1, 64, 256, 200, 50
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=77)
    q[:] = 0.0
    q[:, 0] = 1.0
    kc[0, :, 0] = -1.0e4 - 1.0 + torch.linspace(-0.5, 0.5, S)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, T, W, scale=1.0)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, W, scale=1.0)
    amax, _ = compare(got, ref)
    assert amax <= 1e-2, amax
    # the masked rows really carry weight here
    ref_live = oracle.decode(q.numpy(), np.ascontiguousarray(kc.numpy()[:, T - W:T]),
                             np.ascontiguousarray(vc.numpy()[:, T - W:T]), hq, hkv, d, W, W,
                             scale=1.0)
    assert np.abs(ref - ref_live).max() > 0.1


def test_decode_scale_argument(attn):
    hq, hkv, d, S, T = 4, 2, 64, 512, 300
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=5)
    got = _run_decode(attn, q, kc, vc, hq, hkv, d, S, T, 0, scale=0.3)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, 0, scale=0.3)
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL


def test_prefill_rows_match_decode_on_gpu(attn):
    """Cross-form on the GPU: prefill row i equals decode over i+1 cache rows."""
    m, hq, hkv, d = 96, 4, 2, 128
    q, k, v = workloads.prefill_inputs(m, hq * d, hkv * d, 31)
    pre = _run_prefill(attn, q, k, v, m, hq, hkv, d, hq * d, hkv * d, FP32)
    kc = k.view(m, hkv, d).transpose(0, 1).contiguous()
    vc = v.view(m, hkv, d).transpose(0, 1).contiguous()
    for i in (0, 1, 47, 95):
        qi = q[i, : hq * d].view(hq, d).contiguous()
        dec = _run_decode(attn, qi, kc, vc, hq, hkv, d, m, i + 1, 0)
        assert np.abs(dec - pre[i]).max() <= 2 * FP32_ABS


# ------------------------------------------------------------------ kv_append

def test_kv_append_bit_exact(attn):
    hkv, d, S = 4, 128, 64
    g = torch.Generator().manual_seed(3)
    kc, vc = torch.randn(hkv, S, d, generator=g), torch.randn(hkv, S, d, generator=g)
    ks, vs = torch.randn(hkv, d, generator=g), torch.randn(hkv, d, generator=g)
    for pos in (0, 17, S - 1):
        dk, dv = kc.cuda(), vc.cuda()
        attn.kv_append(ks.cuda(), vs.cuda(), dk, dv, hkv, d, S, pos)
        kh, vh = kc.numpy().copy(), vc.numpy().copy()
        oracle.kv_append(ks.numpy(), vs.numpy(), kh, vh, hkv, d, S, pos)
        np.testing.assert_array_equal(dk.cpu().numpy(), kh)
        np.testing.assert_array_equal(dv.cpu().numpy(), vh)
    dk = kc.cuda()
    attn.kv_append(ks.cuda(), None, dk, None, hkv, d, S, 9)
    kh = kc.numpy().copy()
    oracle.kv_append(ks.numpy(), None, kh, None, hkv, d, S, 9)
    np.testing.assert_array_equal(dk.cpu().numpy(), kh)


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_times_out_and_context_survives(attn):
    """A wait on an mbarrier nothing completes gives up after ~1 ms and the
    kernel returns; the status word reports the timeout and the context keeps
    working."""
    assert attn.attn_selftest_wait_timeout(1000) == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_get_device_status() == attn.ATTN_OK
    _check_prefill(attn, 200, 2, 1, 128, FP16, seed=1)


# ------------------------------------------------------------------ fused (RoPE +) append + decode

def _rope_tables(d, seed):
    theta = np.random.default_rng(seed).uniform(-3.0, 3.0, d // 2)
    return np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("hq,hkv,d,S,T,W", [(12, 2, 128, 4096, 4096, 0),
                                            (32, 8, 128, 32768, 32768, 4096),
                                            (8, 8, 64, 300, 257, 0),
                                            (24, 2, 32, 1000, 1000, 100)])
def test_decode_append_matches_oracle(attn, rope, hq, hkv, d, S, T, W):
    q, kc, vc, kn, vn = workloads.decode_inputs(hq, hkv, d, S, seed=hq + d + T, append=True)
    cos = sin = None
    if rope:
        cos, sin = _rope_tables(d, T)
    dk, dv = kc.cuda(), vc.cuda()
    buf, out = guarded_empty(hq * d)
    pos = T - 1
    attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), dk, dv, out, hq, hkv, d, S, T, pos,
                            window=W,
                            rope_cos=torch.from_numpy(cos).cuda() if rope else None,
                            rope_sin=torch.from_numpy(sin).cuda() if rope else None)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK and guards_intact(buf)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kh, vh, hq, hkv, d, S, T, pos,
                               window=W, rope_cos=cos, rope_sin=sin)
    np.testing.assert_allclose(dk[:, pos].cpu().numpy(), kh[:, pos], rtol=0, atol=2e-6)
    np.testing.assert_array_equal(dv[:, pos].cpu().numpy(), vh[:, pos])
    amax, rel = compare(out.view(hq, d).cpu().numpy(), ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("hq,hkv,d,S,T,W", [(12, 2, 128, 4096, 4096, 0),
                                            (32, 8, 64, 9000, 8191, 1000)])
def test_decode_with_host_resident_step_buffers(attn, rope, hq, hkv, d, S, T, W):
    """q, k_new, v_new, the RoPE tables and out in page-locked host memory:
    the kernels read and write them directly.  The result equals the call on
    device copies of the same buffers bit for bit, and the oracle."""
    q, kc, vc, kn, vn = workloads.decode_inputs(hq, hkv, d, S, seed=hq + T, append=True)
    cos = sin = None
    if rope:
        cos, sin = _rope_tables(d, T)
    pos = T - 1
    hq_, hkn, hvn = q.pin_memory(), kn.pin_memory(), vn.pin_memory()
    hcos = torch.from_numpy(cos).pin_memory() if rope else None
    hsin = torch.from_numpy(sin).pin_memory() if rope else None
    hout = torch.full((hq, d), float("nan")).pin_memory()
    dk1, dv1, dk2, dv2 = kc.cuda(), vc.cuda(), kc.cuda(), vc.cuda()
    dout = torch.empty(hq, d, device="cuda")
    attn.attn_decode_append(hq_, hkn, hvn, dk1, dv1, hout, hq, hkv, d, S, T, pos, window=W,
                            rope_cos=hcos, rope_sin=hsin)
    attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), dk2, dv2, dout, hq, hkv, d, S, T,
                            pos, window=W,
                            rope_cos=hcos.cuda() if rope else None,
                            rope_sin=hsin.cuda() if rope else None)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert torch.equal(hout, dout.cpu())
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kh, vh, hq, hkv, d, S, T, pos,
                               window=W, rope_cos=cos, rope_sin=sin)
    amax, rel = compare(hout.numpy(), ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)
    # the plain decode and the separate append take host buffers the same way
    hout2 = torch.full((hq, d), float("nan")).pin_memory()
    attn.kv_append(hkn, hvn, dk2, dv2, hkv, d, S, pos)
    attn.attn_decode(hq_, dk2, dv2, hout2, hq, hkv, d, S, T, window=W)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    if not rope:
        assert (hout2 - hout).abs().max().item() <= 1e-6


def test_decode_append_position_inside_the_cache(attn):
    """An append in the middle of the attended range replaces that row."""
    hq, hkv, d, S, T = 8, 2, 128, 512, 500
    q, kc, vc, kn, vn = workloads.decode_inputs(hq, hkv, d, S, seed=77, append=True)
    dk, dv = kc.cuda(), vc.cuda()
    out = torch.empty(hq, d, device="cuda")
    attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), dk, dv, out, hq, hkv, d, S, T, 123)
    torch.cuda.synchronize()
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kh, vh, hq, hkv, d, S, T, 123)
    amax, rel = compare(out.cpu().numpy(), ref)
    assert amax <= FP32_ABS and rel <= FP32_REL


def test_workload_append_then_streaming_decode_32k(attn):
    """The fused append + decode over a full 32768-row cache (no window),
    268 MB of K/V, as the bench times it: every warp runs many steps with
    the L2 prefetch running ahead of its loads."""
    c = workloads.DECODE_32K_STREAM
    q, kc, vc, kn, vn = workloads.shape_inputs(c)
    dk, dv = kc.cuda(), vc.cuda()
    pos = c.total_seq - 1
    buf, out = guarded_empty(c.num_heads * c.head_dim)
    attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), dk, dv, out, c.num_heads,
                            c.kv_heads, c.head_dim, c.max_seq, c.total_seq, pos,
                            window=c.window)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kh, vh, c.num_heads,
                               c.kv_heads, c.head_dim, c.max_seq, c.total_seq, pos)
    np.testing.assert_array_equal(dk[:, pos].cpu().numpy(), kh[:, pos])
    np.testing.assert_array_equal(dv[:, pos].cpu().numpy(), vh[:, pos])
    amax, rel = compare(out.view(c.num_heads, c.head_dim).cpu().numpy(), ref)
    print(f"{c.name}: max abs {amax:.3e} rel {rel:.3e}")
    assert amax <= FP32_ABS and rel <= FP32_REL


@pytest.mark.parametrize("hq,hkv,d,S,T,W", [
    (12, 2, 128, 4200, 4097, 0),     # one step per warp, ragged tail
    (12, 2, 128, 40000, 33333, 0),   # many steps per warp (L2 prefetch ahead)
    (32, 8, 64, 9000, 8191, 1000),   # window: K rows below its start poisoned too
    (6, 1, 32, 64, 5, 0),
    (8, 8, 128, 300, 1, 0),
])
@pytest.mark.parametrize("fused", [False, True])
def test_decode_rows_outside_the_live_range_are_never_read(attn, hq, hkv, d, S, T, W, fused):
    """Cache rows at or past total_seq are not part of the attention, and the
    keys of rows below the window start are replaced by the -1e4 score: NaN in
    either must not reach the output."""
    q, kc, vc, kn, vn = workloads.decode_inputs(hq, hkv, d, S, seed=T + W, append=True)
    kc[:, T:] = float("nan")
    vc[:, T:] = float("nan")
    ws = T - W if (W > 0 and T > W) else 0
    kc[:, :ws] = float("nan")
    dk, dv = kc.cuda(), vc.cuda()
    buf, out = guarded_empty(hq * d)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    if fused:
        attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), dk, dv, out, hq, hkv, d, S, T,
                                T - 1, window=W)
        ref = oracle.decode_append(q.numpy(), kn.numpy(), vn.numpy(), kh, vh, hq, hkv, d, S, T,
                                   T - 1, window=W)
    else:
        attn.attn_decode(q.cuda(), dk, dv, out, hq, hkv, d, S, T, window=W)
        ref = oracle.decode(q.numpy(), kh, vh, hq, hkv, d, S, T, W)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    assert guards_intact(buf)
    got = out.view(hq, d).cpu().numpy()
    assert np.isfinite(ref).all() and np.isfinite(got).all()
    amax, rel = compare(got, ref)
    assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)


def test_decode_append_equals_unfused_append_then_decode(attn):
    """The fused entry point and kv_append + attn_decode agree to fp32 rounding."""
    c = workloads.DECODE_32K_WINDOW
    q, kc, vc, kn, vn = workloads.shape_inputs(c)
    pos = c.total_seq - 1
    k1, v1, k2, v2 = kc.cuda(), vc.cuda(), kc.cuda(), vc.cuda()
    o1 = torch.empty(c.num_heads, c.head_dim, device="cuda")
    o2 = torch.empty_like(o1)
    attn.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), k1, v1, o1, c.num_heads, c.kv_heads,
                            c.head_dim, c.max_seq, c.total_seq, pos, window=c.window)
    attn.kv_append(kn.cuda(), vn.cuda(), k2, v2, c.kv_heads, c.head_dim, c.max_seq, pos)
    attn.attn_decode(q.cuda(), k2, v2, o2, c.num_heads, c.kv_heads, c.head_dim, c.max_seq,
                     c.total_seq, window=c.window)
    torch.cuda.synchronize()
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert (o1 - o2).abs().max().item() <= 1e-6


def test_decode_waits_for_the_kernel_before_it(attn):
    """Decode launches overlap the previous kernel on the stream (they only
    prefetch until it completes).  Here the kernels right before each decode
    rewrite q and the cache row the decode reads: back-to-back calls on one
    stream must still see the new values."""
    hq, hkv, d, S, T = 12, 2, 128, 4096, 4096
    q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=77)
    q2, kc2, vc2, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=78)
    dq, dk, dv = q.cuda(), kc.cuda(), vc.cuda()
    dq2, dk2, dv2 = q2.cuda(), kc2.cuda(), vc2.cuda()
    outs = [torch.full((hq, d), float("nan"), device="cuda") for _ in range(3)]
    torch.cuda.synchronize()
    attn.attn_decode(dq, dk, dv, outs[0], hq, hkv, d, S, T)
    dq.copy_(dq2)                      # predecessor kernels of the next decode
    dk[:, T - 1].copy_(dk2[:, T - 1])
    dv[:, T - 1].copy_(dv2[:, T - 1])
    attn.attn_decode(dq, dk, dv, outs[1], hq, hkv, d, S, T)
    attn.attn_decode(dq, dk, dv, outs[2], hq, hkv, d, S, T)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    kh[:, T - 1], vh[:, T - 1] = kc2.numpy()[:, T - 1], vc2.numpy()[:, T - 1]
    ref0 = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, 0)
    ref1 = oracle.decode(q2.numpy(), kh, vh, hq, hkv, d, S, T, 0)
    for got, ref in ((outs[0], ref0), (outs[1], ref1), (outs[2], ref1)):
        amax, rel = compare(got.cpu().numpy(), ref)
        assert amax <= FP32_ABS and rel <= FP32_REL


def test_prefill_fp32_waits_for_the_kernel_before_it(attn):
    """The exact-mode prefill launches as a programmatic dependent of the
    previous kernel on the stream.  Here the kernels right before the second
    call rewrite Q, K and V, and the call right after reads the first call's
    output as its Q: every call must see the values of the kernel before it."""
    m, hq, hkv, d = 64, 4, 2, 32
    qs, kvs = 128, 64
    q, k, v = workloads.prefill_inputs(m, qs, kvs, 0)
    q2, k2, v2 = workloads.prefill_inputs(m, qs, kvs, 1)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    outs = [torch.full((m, qs), float("nan"), device="cuda") for _ in range(3)]
    torch.cuda.synchronize()
    attn.attn_prefill_causal(dq, dk, dv, outs[0], m, hq, hkv, d, qs, kvs,
                             precision=attn.ATTN_PREC_FP32)
    dq.copy_(q2.cuda())                # predecessor kernels of the next call
    dk.copy_(k2.cuda())
    dv.copy_(v2.cuda())
    attn.attn_prefill_causal(dq, dk, dv, outs[1], m, hq, hkv, d, qs, kvs,
                             precision=attn.ATTN_PREC_FP32)
    attn.attn_prefill_causal(outs[1], dk, dv, outs[2], m, hq, hkv, d, qs, kvs,
                             precision=attn.ATTN_PREC_FP32)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    ref0 = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs)
    ref1 = oracle.prefill_causal(q2.numpy(), k2.numpy(), v2.numpy(), m, hq, hkv, d, qs, kvs)
    o1 = outs[1].cpu().numpy()
    ref2 = oracle.prefill_causal(o1, k2.numpy(), v2.numpy(), m, hq, hkv, d, qs, kvs)
    for got, ref in ((outs[0], ref0), (outs[1], ref1), (outs[2], ref2)):
        amax, rel = compare(heads_view(got.reshape(-1), m, qs, hq, d), ref)
        assert amax <= FP32_ABS and rel <= FP32_REL, (amax, rel)


@pytest.mark.parametrize("prec", [FP16, TF32])
def test_prefill_tc_waits_for_the_kernels_before_it(attn, prec):
    """The tensor-core prefill chains its kernels as programmatic dependents
    (rounding pre-pass, main kernel staging the caller's Q before it waits
    for the pre-pass, combine), and its pre-pass depends the same way on the
    kernel before the call.  Back-to-back calls where the kernels right
    before a call rewrite K and V, and where a call's Q is the previous
    call's output (written by that call's combine kernel), must see the new
    values."""
    m, hq, hkv, d = 2048, 12, 2, 128    # splits its key walk: the combine runs last
    qs, kvs = hq * d, hkv * d
    q, k, v = workloads.prefill_inputs(m, qs, kvs, 2)
    q2, k2, v2 = workloads.prefill_inputs(m, qs, kvs, 3)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    outs = [torch.full((m, qs), float("nan"), device="cuda") for _ in range(3)]
    torch.cuda.synchronize()
    attn.attn_prefill_causal(dq, dk, dv, outs[0], m, hq, hkv, d, qs, kvs, precision=prec)
    dk.copy_(k2.cuda())                # predecessor kernels of the next call
    dv.copy_(v2.cuda())
    attn.attn_prefill_causal(dq, dk, dv, outs[1], m, hq, hkv, d, qs, kvs, precision=prec)
    attn.attn_prefill_causal(outs[1], dk, dv, outs[2], m, hq, hkv, d, qs, kvs, precision=prec)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_OK
    rows = workloads.sample_rows(m, 5, 16, 16, 48)
    o1 = outs[1].cpu().numpy()
    refs = (oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs, rows=rows),
            oracle.prefill_causal(q.numpy(), k2.numpy(), v2.numpy(), m, hq, hkv, d, qs, kvs, rows=rows),
            oracle.prefill_causal(o1, k2.numpy(), v2.numpy(), m, hq, hkv, d, qs, kvs, rows=rows))
    for got, ref in zip(outs, refs):
        amax, _ = compare(heads_view(got.reshape(-1), m, qs, hq, d)[rows], ref)
        assert amax <= TC_ABS, amax


def test_decode_workspace_reuse(attn):
    """One workspace, never cleared, serves many calls of different shapes."""
    ws = torch.full((8 << 20,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN garbage
    for (hq, hkv, d, S, T, W) in [(12, 2, 128, 4096, 4096, 0), (32, 8, 128, 8192, 8000, 1000),
                                  (12, 2, 128, 4096, 4096, 0), (4, 1, 64, 100, 3, 0),
                                  (64, 8, 128, 20000, 20000, 0)]:
        q, kc, vc, _, _ = workloads.decode_inputs(hq, hkv, d, S, seed=T)
        out = torch.empty(hq, d, device="cuda")
        attn.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), out, hq, hkv, d, S, T, window=W,
                         workspace=ws)
        torch.cuda.synchronize()
        ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), hq, hkv, d, S, T, W)
        amax, rel = compare(out.cpu().numpy(), ref)
        assert amax <= FP32_ABS and rel <= FP32_REL


# ------------------------------------------------------------------ autoregressive loop

@pytest.mark.parametrize("prec", [FP32, FP16, TF32])
def test_autoregressive_steps_match_prefill_rows(attn, prec):
    """Prefill a prompt, then run decode steps that append each new token's
    K/V row and attend to the cache: step t must reproduce row P+t of a causal
    prefill over the whole sequence (honeycrisp KV_APPEND + kmain against
    prefill_fused.rs).  Both sides run on the GPU; the oracle checks them."""
    P, N, hq, hkv, d = 200, 24, 8, 2, 128
    M = P + N
    q, k, v = workloads.prefill_inputs(M, hq * d, hkv * d, seed=901)
    full = _run_prefill(attn, q, k, v, M, hq, hkv, d, hq * d, hkv * d, prec)
    # cache holding the prompt rows
    kc = torch.zeros(hkv, M, d, device="cuda")
    vc = torch.zeros(hkv, M, d, device="cuda")
    kc[:, :P] = k[:P].view(P, hkv, d).transpose(0, 1).cuda()
    vc[:, :P] = v[:P].view(P, hkv, d).transpose(0, 1).cuda()
    out = torch.empty(hq, d, device="cuda")
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), M, hq, hkv, d, hq * d, hkv * d,
                                rows=list(range(P, M)))
    for t in range(N):
        pos = P + t
        qt = q[pos].view(hq, d).cuda()
        kt = k[pos].view(hkv, d).cuda()
        vt = v[pos].view(hkv, d).cuda()
        if t % 2 == 0:   # fused entry point on even steps, separate calls on odd steps
            attn.attn_decode_append(qt, kt, vt, kc, vc, out, hq, hkv, d, M, pos + 1, pos)
        else:
            attn.kv_append(kt, vt, kc, vc, hkv, d, M, pos)
            attn.attn_decode(qt, kc, vc, out, hq, hkv, d, M, pos + 1)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        amax, rel = compare(got, ref[t])
        assert amax <= FP32_ABS and rel <= FP32_REL, (t, amax)
        tol = FP32_ABS if prec == FP32 else TC_ABS
        assert np.abs(got - full[pos]).max() <= tol + FP32_ABS


# ------------------------------------------------------------------ bf16 operand mode

BF16 = 2


@pytest.mark.parametrize("m,hq,hkv,d", [(300, 4, 2, 128), (129, 2, 1, 64)])
def test_prefill_bf16_operands(attn, m, hq, hkv, d):
    """ATTN_PREC_BF16: operands rounded to bf16 (8-bit mantissa, unit roundoff
    2^-9).  Row 0 alone carries |V| * 2^-9 (about 8e-3 for |V| <= 4.2), and
    score rounding adds the same order; bound 2.5e-2.  The fp16 mode meets
    3e-3 on the same inputs."""
    qs, kvs = hq * d, hkv * d
    q, k, v = workloads.prefill_inputs(m, qs, kvs, seed=m + d)
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, BF16)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs)
    amax, _ = compare(got, ref)
    assert amax <= 2.5e-2, amax
    got16 = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, FP16)
    assert compare(got16, ref)[0] <= TC_ABS


def test_prefill_bf16_operands_pair_kernel(attn):
    """The bf16 mode through the query-tile-pair kernel: 16 pairs x 40 heads
    fill two waves of SMs.  Sampled rows against the oracle at the bf16 bound
    (reading 16), and the fp16 mode at 3e-3 on the same inputs."""
    m, hq, hkv, d = 4096, 40, 8, 128
    assert (m // 256) * hq >= 2 * torch.cuda.get_device_properties(0).multi_processor_count
    qs, kvs = hq * d, hkv * d
    q, k, v = workloads.prefill_inputs(m, qs, kvs, seed=77)
    rows = workloads.sample_rows(m, 77, 32, 32, 64)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs, rows=rows)
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, BF16)[rows]
    amax, _ = compare(got, ref)
    assert amax <= 2.5e-2, amax
    got16 = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, FP16)[rows]
    assert compare(got16, ref)[0] <= TC_ABS


# ------------------------------------------------------------------ TF32 operand mode

@pytest.mark.parametrize("d", [64, 128])
def test_prefill_tf32_takes_inputs_beyond_the_fp16_range(attn, d):
    """ATTN_PREC_TF32 keeps fp32's exponent: Q scaled by 1e5 (past fp16's
    65504), K by 1e-5 (below fp16's normal range) and V by 1e5.  The scores
    are those of the unscaled inputs, the output is 1e5 times theirs, and the
    TF32 result meets the tensor-core bound after dividing by 1e5.  The fp16
    mode flags the same inputs with ATTN_ERR_RANGE."""
    m, hq, hkv = 300, 4, 2
    qs, kvs = hq * d, hkv * d
    q, k, v = workloads.prefill_inputs(m, qs, kvs, 202)
    q, k, v = q * 1e5, k * 1e-5, v * 1e5
    got = _run_prefill(attn, q, k, v, m, hq, hkv, d, qs, kvs, TF32)
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), m, hq, hkv, d, qs, kvs)
    amax, _ = compare(got / 1e5, ref / 1e5)
    assert amax <= TC_ABS, amax
    buf, o = guarded_empty(m * qs)
    attn.attn_prefill_causal(q.cuda(), k.cuda(), v.cuda(), o, m, hq, hkv, d, qs, kvs,
                             precision=FP16)
    assert attn.attn_get_device_status() == attn.ATTN_ERR_RANGE
