"""Seeded synthetic inputs for the FIFO data plane.

This module only draws random numbers in the shapes the transport pages'
workloads use; it holds none of the transport's arithmetic (no channel
partition, no slot schedule, no reduction).  Both the CPU oracle and the CUDA
path receive the same arrays from here.

Recipe (one `numpy.random.default_rng(seed)` stream per input, drawn in blocks
of ``BLOCK`` values so the multi-GiB inputs never need a second full-size
temporary):

* SIMPLE loopback: ``n`` uniform bytes, seed 0.
* LL sweep: uint32 words uniform over [0, 2**32), seed 1.
* SIMPLE multi-channel: bf16 values N(0, 1), seed 2: fp32 normal draws rounded
  to bf16 by round-to-nearest-even on the bit pattern.
* host-placed FIFO: fp32 uniform [-1, 1), seed 3.
* virtual ring: rank ``r`` draws fp32 uniform [-1, 1) from seed ``10 + r``;
  the int32 variant draws integers in [-1000, 1000] from the same seed.
"""
from __future__ import annotations

import numpy as np

BLOCK = 1 << 22

# Sizes of the five workloads (bytes, slots, slot bytes, channels, ranks).
SIMPLE_LOOPBACK = dict(nbytes=1 << 20, nslots=8, slot_bytes=64 << 10, nchannels=1, seed=0)
LL_SWEEP = dict(sizes=[1 << k for k in range(3, 19)], nslots=8, slot_bytes=32 << 10, nchannels=1, seed=1)
SIMPLE_MULTI = dict(nelems=1 << 29, nslots=8, slot_bytes=512 << 10, nchannels=16, seed=2)
HOST_FIFO = dict(nelems=1 << 26, nslots=8, slot_bytes=1 << 20, nchannels=8, seed=3)
RING = dict(nranks=8, nelems=1 << 26, nslots=8, slot_bytes=512 << 10, nchannels=8, seed_base=10)


def uniform_bytes(n: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    out = np.empty(n, np.uint8)
    for i in range(0, n, BLOCK):
        m = min(BLOCK, n - i)
        out[i:i + m] = rng.integers(0, 256, m, dtype=np.uint8)
    return out


def uniform_u32(nwords: int, seed: int = 1) -> np.ndarray:
    rng = np.random.default_rng(seed)
    out = np.empty(nwords, np.uint32)
    for i in range(0, nwords, BLOCK):
        m = min(BLOCK, nwords - i)
        out[i:i + m] = rng.integers(0, 1 << 32, m, dtype=np.uint32)
    return out


def normal_bf16_bits(nelems: int, seed: int = 2) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws, rounded to nearest even."""
    rng = np.random.default_rng(seed)
    out = np.empty(nelems, np.uint16)
    for i in range(0, nelems, BLOCK):
        m = min(BLOCK, nelems - i)
        u = rng.standard_normal(m, dtype=np.float32).view(np.uint32)
        u = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        out[i:i + m] = (u >> np.uint32(16)).astype(np.uint16)
    return out


def uniform_f32(nelems: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    out = np.empty(nelems, np.float32)
    for i in range(0, nelems, BLOCK):
        m = min(BLOCK, nelems - i)
        out[i:i + m] = rng.uniform(-1.0, 1.0, m).astype(np.float32)
    return out


def uniform_i32(nelems: int, seed: int, lo: int = -1000, hi: int = 1000) -> np.ndarray:
    rng = np.random.default_rng(seed)
    out = np.empty(nelems, np.int32)
    for i in range(0, nelems, BLOCK):
        m = min(BLOCK, nelems - i)
        out[i:i + m] = rng.integers(lo, hi + 1, m, dtype=np.int32)
    return out


def ring_inputs(nranks: int, nelems: int, dtype: str = "f32", seed_base: int = 10) -> list[np.ndarray]:
    if dtype == "f32":
        return [uniform_f32(nelems, seed_base + r) for r in range(nranks)]
    if dtype == "i32":
        return [uniform_i32(nelems, seed_base + r) for r in range(nranks)]
    raise ValueError(dtype)
