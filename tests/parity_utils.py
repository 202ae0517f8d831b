"""Shared helpers for the GPU parity tests: run a call through the C ABI on
guard-banded, NaN-poisoned device buffers and compare with the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

# Tolerances (fp32 CUDA-core paths; tensor-core path reported separately).
FP32_ABS = 1e-4
FP32_REL = 1e-4      # normwise: max|gpu - oracle| / max|oracle|
TC_ABS = 3e-3

GUARD = 256          # floats of canary on each side of every output buffer
CANARY = 12345.678


def guarded_empty(n_floats: int, device="cuda"):
    """A NaN-poisoned device buffer of n_floats with canary bands on both
    sides; returns (full_buffer, view_of_payload).  The payload starts at a
    16-byte aligned offset (GUARD floats = 1 KB)."""
    buf = torch.full((n_floats + 2 * GUARD,), CANARY, dtype=torch.float32, device=device)
    buf[GUARD:GUARD + n_floats] = float("nan")
    return buf, buf[GUARD:GUARD + n_floats]


def guards_intact(buf: torch.Tensor) -> bool:
    h = buf.detach().cpu().numpy()
    return bool((h[:GUARD] == np.float32(CANARY)).all() and (h[-GUARD:] == np.float32(CANARY)).all())


def compare(gpu: np.ndarray, ref: np.ndarray):
    """(max abs error, normwise relative error)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), "non-finite values in the GPU output"
    err = np.abs(gpu - ref)
    amax = float(err.max()) if err.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 1.0
    return amax, amax / max(scale, 1e-300)


def heads_view(o_flat: torch.Tensor, m: int, q_stride: int, hq: int, d: int) -> np.ndarray:
    """[m, hq, d] numpy view of the head columns of an [m, q_stride] output."""
    o = o_flat[: m * q_stride].view(m, q_stride)[:, : hq * d]
    return o.detach().cpu().numpy().reshape(m, hq, d)


def untouched_columns(o_flat: torch.Tensor, m: int, q_stride: int, hq: int, d: int) -> bool:
    """Columns past the head columns of each row must keep their NaN poison."""
    if q_stride == hq * d:
        return True
    o = o_flat[: m * q_stride].view(m, q_stride)[:, hq * d:]
    return bool(torch.isnan(o).all().item())
