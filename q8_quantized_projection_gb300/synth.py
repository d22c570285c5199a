"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module only draws random numbers and arranges them into arrays; it holds
none of the projection's arithmetic (no quantiser, no dot product, no norm).
Both the CUDA path and the CPU oracle consume the arrays it returns, so that the
two sides see the same bytes.

Recipe (numpy PCG64 ``default_rng(seed)``):

* Q8_0 weights: int8 quants uniform over [-127, 127]; one fp16 scale per
  32-value block along K, drawn as |N(0, 0.02)| / 127 and rounded to binary16
  by numpy (the ".q" / ".s" planar pair the model-author page declares).
* activations: f32 N(0, 1) rows of length K (the hidden state before the
  producer's RMSNorm).
* RMSNorm gain: 1 + 0.1 N(0, 1) (tests only; the workloads use no gain).
* head: 8 planted rows whose quants are 127 * sign(h_j) of the first eight
  activation rows and whose scales are all 0.02 / 127, so the arg-max of
  activation row m is the planted row m mod 8 by a wide margin.
"""
from __future__ import annotations

import numpy as np

QK = 32  # values per Q8_0 block along K

# Decode-step projections of a d = 4096 Llama-shaped layer (32 q heads,
# 8 kv heads, head dim 128, FFN 14336).
LAYER_D4096 = (
    ("wqkv", 6144, 4096),
    ("wo", 4096, 4096),
    ("gate_up", 28672, 4096),
    ("down", 4096, 14336),
)
HEAD_SHAPE = (128256, 4096)


def rng_for(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def q8_weights(rng: np.random.Generator, n: int, k: int):
    """Return (q int8 [n, k], s uint16 fp16-bits [n, k/32])."""
    if k % QK:
        raise ValueError("K must be a multiple of 32")
    q = rng.integers(-127, 128, size=(n, k), dtype=np.int8)
    s = (np.abs(rng.normal(0.0, 0.02, size=(n, k // QK))) / 127.0).astype(np.float16)
    return q, s.view(np.uint16)


def f32_weights(rng: np.random.Generator, n: int, k: int, sigma: float = 0.02):
    """Dense f32 weights for the pack step, N(0, sigma)."""
    return rng.normal(0.0, sigma, size=(n, k)).astype(np.float32)


def activations(rng: np.random.Generator, rows: int, k: int):
    return rng.standard_normal(size=(rows, k), dtype=np.float32)


def gain(rng: np.random.Generator, k: int):
    return (1.0 + 0.1 * rng.standard_normal(size=(k,))).astype(np.float32)


def head_activations(rng: np.random.Generator, rows: int, k: int):
    """Activation rows for the LM head: rows 0..7 are N(0,1); row m >= 8 is
    row m-8 plus 0.1 N(0,1) noise.  Always draws the eight base rows, so the
    planted head rows exist whatever `rows` is; returns (h [rows, k], base [8, k])."""
    base = rng.standard_normal(size=(8, k), dtype=np.float32)
    out = np.empty((rows, k), dtype=np.float32)
    for m in range(rows):
        if m < 8:
            out[m] = base[m]
        else:
            out[m] = out[m - 8] + np.float32(0.1) * rng.standard_normal(size=(k,), dtype=np.float32)
    return out, base


def planted_positions(rng: np.random.Generator, n: int, count: int = 8):
    """Distinct head rows for the planted winners, always including 0 and n-1."""
    if n < count:
        raise ValueError("head too small for the planted rows")
    pos = [0, n - 1]
    while len(pos) < count:
        p = int(rng.integers(1, n - 1))
        if p not in pos:
            pos.append(p)
    return np.array(pos, dtype=np.int64)


def plant_head_rows(q: np.ndarray, s: np.ndarray, base: np.ndarray, positions: np.ndarray):
    """Write the planted rows in place: quants 127*sign(base_j), scales fp16(0.02/127)."""
    s_planted = np.float16(0.02 / 127.0).view(np.uint16)
    for j, p in enumerate(positions):
        q[p] = np.where(base[j] >= 0, 127, -127).astype(np.int8)
        s[p] = s_planted
    return q, s


def planted_head(seed: int, n: int, k: int, rows: int):
    """A Q8_0 head with 8 planted rows and its activation rows.
    Returns (q, s, h, positions); the winner of row m is positions[m % 8]."""
    rng = rng_for(seed)
    q, s = q8_weights(rng, n, k)
    h, base = head_activations(rng, rows, k)
    pos = planted_positions(rng, n)
    plant_head_rows(q, s, base, pos)
    return q, s, h, pos
