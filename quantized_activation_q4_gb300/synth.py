"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and lays them out as bytes. It holds none
of the arithmetic of the method (no quantisation, no norm, no dot products), so
the oracle and the CUDA library can both be fed from it without sharing any
computation.

Distributions follow the workloads described for the activation-image pages:
activations ~N(0,1), RMSNorm weights ~N(1,0.1), Q4_0 weights with uniform
nibbles 0..15 and half scales drawn U[0.002, 0.02], router logits ~N(0,1).

Every generator takes an explicit integer seed and uses numpy's Philox
counter-based bit generator, so the same seed gives the same bytes on x86 and
Arm hosts.
"""
from __future__ import annotations

import numpy as np

Q4_0_BLOCK_BYTES = 18  # half d + 16 bytes of nibbles per 32 weights
Q8_0_BLOCK_BYTES = 34  # half d + 32 int8 codes per 32 weights


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(int(seed)))


def activations(seed: int, T: int, K: int, stride: int | None = None) -> np.ndarray:
    """F32 activation rows ~N(0,1); shape [T, stride] with columns >= K left 0."""
    stride = K if stride is None else stride
    out = np.zeros((T, stride), dtype=np.float32)
    out[:, :K] = rng(seed).standard_normal((T, K), dtype=np.float32)
    return out


def norm_weight(seed: int, K: int, mean: float = 1.0, std: float = 0.1) -> np.ndarray:
    """RMSNorm per-channel weight ~N(mean, std), F32."""
    return (mean + std * rng(seed).standard_normal(K)).astype(np.float32)


def half_scales(g: np.random.Generator, shape, lo: float = 0.002, hi: float = 0.02) -> np.ndarray:
    """Scales drawn U[lo, hi] and stored as IEEE half (numpy's own conversion)."""
    return g.uniform(lo, hi, size=shape).astype(np.float16)


def q4_0_weight(seed: int, N: int, K: int) -> np.ndarray:
    """Canonical Q4_0 blocks, uint8 array of shape [N, K/32, 18].

    Block bytes: [d as little-endian half][16 bytes of nibbles]. Nibbles are
    uniform on 0..15; d is U[0.002, 0.02] rounded to half.
    """
    assert K % 32 == 0
    g = rng(seed)
    kb = K // 32
    d = half_scales(g, (N, kb))
    nib = g.integers(0, 256, size=(N, kb, 16), dtype=np.uint8)  # two uniform nibbles per byte
    out = np.empty((N, kb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d.view(np.uint8).reshape(N, kb, 2)
    out[:, :, 2:] = nib
    return out


def q8_0_weight(seed: int, N: int, K: int) -> np.ndarray:
    """Canonical Q8_0 blocks, uint8 array of shape [N, K/32, 34]: [half d][32 int8]."""
    assert K % 32 == 0
    g = rng(seed)
    kb = K // 32
    d = half_scales(g, (N, kb), 0.0002, 0.002)
    q = g.integers(-127, 128, size=(N, kb, 32), dtype=np.int16).astype(np.int8)
    out = np.empty((N, kb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d.view(np.uint8).reshape(N, kb, 2)
    out[:, :, 2:] = q.view(np.uint8)
    return out


def q4_0_identity(N: int, K: int) -> np.ndarray:
    """Q4_0 blocks with d=1, nibble 9 on the diagonal and 8 elsewhere.

    Each row dequantises to a one-hot vector e_n, so W @ x == x[:N] exactly.
    """
    assert K % 32 == 0
    kb = K // 32
    out = np.zeros((N, kb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
    out[:, :, 2:] = 0x88
    for n in range(min(N, K)):
        b, j = divmod(n, 32)
        byte = j % 16
        if j < 16:
            out[n, b, 2 + byte] = (out[n, b, 2 + byte] & 0xF0) | 9
        else:
            out[n, b, 2 + byte] = (out[n, b, 2 + byte] & 0x0F) | (9 << 4)
    return out


def router_logits(seed: int, rows: int, E: int) -> np.ndarray:
    return rng(seed).standard_normal((rows, E), dtype=np.float32)


POISON_CYCLE = (np.float32(np.nan), np.float32(1e30), np.float32(-1e30))


def poison_rows(a: np.ndarray, live: int) -> np.ndarray:
    """Fill rows >= live with NaN, +1e30, -1e30 in turn (padding of a captured bucket)."""
    a = a.copy()
    for r in range(live, a.shape[0]):
        a[r] = POISON_CYCLE[(r - live) % 3]
    return a


def stale_ids(seed: int, rows: int, k: int, E: int) -> np.ndarray:
    """Stale expert picks naming real experts, as left behind by an earlier forward."""
    return rng(seed).integers(0, E, size=(rows, k), dtype=np.int32)
