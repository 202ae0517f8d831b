"""Seeded synthetic inputs for the attention workloads.

This module only draws random tensors and names the workload shapes; it holds
none of the attention arithmetic.  The CPU oracle, the CUDA path, the tests and
the benchmark all take their inputs from here, so that both sides of every
parity check see the very same fp32 values.

Draw recipe (the pages say only "iid N(0,1) from seed s"; this is the reading
taken): a CPU ``torch.Generator`` seeded with ``s`` and ``torch.randn`` in
float32, drawing in this order
  * prefill: Q [M, q_stride], then K [M, kv_stride], then V [M, kv_stride];
  * decode:  q [Hq, D], then K cache [Hkv, S, D], then V cache [Hkv, S, D],
             then (append workloads only) k_new [Hkv, D], then v_new [Hkv, D];
and multiplying every tensor by ``mul`` afterwards (0.5 for the long prefill).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillShape:
    name: str
    m: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_stride: int
    kv_stride: int
    seed: int
    mul: float = 1.0
    tensor_core: bool = False
    kind: str = field(default="prefill")

    @property
    def heads_per_kv(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def flops(self) -> int:
        """Causal FLOPs counted as 2*M*(M+1)*D*Hq (QK^T and PV over the
        M(M+1)/2 attended pairs, 2 FLOPs per multiply-add)."""
        return 2 * self.m * (self.m + 1) * self.head_dim * self.num_q_heads


@dataclass(frozen=True)
class DecodeShape:
    name: str
    num_heads: int
    kv_heads: int
    head_dim: int
    max_seq: int
    total_seq: int
    window: int
    seed: int
    append: bool = False
    mul: float = 1.0
    kind: str = field(default="decode")

    @property
    def window_start(self) -> int:
        return (self.total_seq - self.window
                if (self.window > 0 and self.total_seq > self.window) else 0)

    def kv_bytes_algorithmic(self) -> int:
        """K+V bytes that must be read: the live (unmasked) rows only."""
        return 2 * self.kv_heads * (self.total_seq - self.window_start) * self.head_dim * 4

    def kv_bytes_all_rows(self) -> int:
        """K+V bytes over all total_seq rows: 2*kv_heads*total_seq*head_dim*4."""
        return 2 * self.kv_heads * self.total_seq * self.head_dim * 4


# The five named workloads: small correctness prefill, decode, mid prefill,
# windowed decode after an append, long prefill.
PREFILL_SMALL = PrefillShape("prefill_m64_h4x2_d32", 64, 4, 2, 32, 128, 64, seed=0)
DECODE_4K = DecodeShape("decode_h12x2_d128_t4096", 12, 2, 128, 4096, 4096, 0, seed=1)
PREFILL_2K = PrefillShape("prefill_m2048_h12x2_d128", 2048, 12, 2, 128, 1536, 256, seed=2,
                          tensor_core=True)
DECODE_32K_WINDOW = DecodeShape("append_decode_h32x8_d128_t32768_w4096", 32, 8, 128, 32768,
                                32768, 4096, seed=3, append=True)
PREFILL_16K = PrefillShape("prefill_m16384_h28x4_d128", 16384, 28, 4, 128, 3584, 512, seed=4,
                           mul=0.5, tensor_core=True)
# Decode over a full 32768-row cache with no window: 268 MB of K/V per step,
# more than L2 holds, so every step streams from HBM.
DECODE_32K_STREAM = DecodeShape("append_decode_h32x8_d128_t32768", 32, 8, 128, 32768, 32768, 0,
                                seed=5, append=True)

ALL = [PREFILL_SMALL, DECODE_4K, PREFILL_2K, DECODE_32K_WINDOW, PREFILL_16K]
BY_NAME = {c.name: c for c in ALL}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def prefill_inputs(m, q_stride, kv_stride, seed, mul=1.0):
    """(q, k, v) fp32 CPU tensors of shapes [m, q_stride], [m, kv_stride] x2."""
    g = _gen(seed)
    q = torch.randn(m, q_stride, generator=g, dtype=torch.float32)
    k = torch.randn(m, kv_stride, generator=g, dtype=torch.float32)
    v = torch.randn(m, kv_stride, generator=g, dtype=torch.float32)
    if mul != 1.0:
        q.mul_(mul), k.mul_(mul), v.mul_(mul)
    return q, k, v


def decode_inputs(num_heads, kv_heads, head_dim, max_seq, seed, append=False, mul=1.0):
    """(q, k_cache, v_cache, k_new, v_new) fp32 CPU tensors; k_new/v_new are
    None unless ``append``.  Caches are [kv_heads, max_seq, head_dim]."""
    g = _gen(seed)
    q = torch.randn(num_heads, head_dim, generator=g, dtype=torch.float32)
    kc = torch.randn(kv_heads, max_seq, head_dim, generator=g, dtype=torch.float32)
    vc = torch.randn(kv_heads, max_seq, head_dim, generator=g, dtype=torch.float32)
    kn = vn = None
    if append:
        kn = torch.randn(kv_heads, head_dim, generator=g, dtype=torch.float32)
        vn = torch.randn(kv_heads, head_dim, generator=g, dtype=torch.float32)
    ts = [q, kc, vc] + ([kn, vn] if append else [])
    if mul != 1.0:
        for t in ts:
            t.mul_(mul)
    return q, kc, vc, kn, vn


def shape_inputs(shape):
    """Inputs of a named workload, drawn by the recipe above."""
    if isinstance(shape, PrefillShape):
        return prefill_inputs(shape.m, shape.q_stride, shape.kv_stride, shape.seed, shape.mul)
    return decode_inputs(shape.num_heads, shape.kv_heads, shape.head_dim, shape.max_seq,
                         shape.seed, shape.append, shape.mul)


def sample_rows(m: int, seed: int, n_first=64, n_last=64, n_random=256):
    """A fixed, seeded sample of query rows: the first and last rows and a
    random draw in between (sorted, unique)."""
    g = _gen(seed + 1000)
    rows = set(range(min(n_first, m)))
    rows.update(range(max(0, m - n_last), m))
    if m > 0:
        rows.update(torch.randint(0, m, (n_random,), generator=g).tolist())
    return sorted(rows)
