"""Seeded synthetic inputs for the Q8_0 product -- shared by the tests, the benchmark and the oracle's callers.

This module draws inputs only; it holds none of the product's arithmetic.  The distributions are the ones the
workloads name:

* activations x: bf16(N(0, 1)), rounded to nearest-even from an fp32 normal draw, returned as uint16 bit patterns;
* values q: int8 uniform on [-127, 127], then one entry of every (32-row block, column) forced to +-127 (random
  position and sign), so the block's amax is 127 * s and the pair (q, s) is its own Q8_0 quantization;
* scales s: fp32(2^u / 127) with u uniform on [-8, -2];
* pad columns N .. Np-1 (Np = N rounded up to a multiple of 32): q = 0 and s = 0.

Host draws use numpy's Philox bit generator; the device draws (for weights too large to make on the host) use a
seeded torch CUDA generator.  The seed of a workload case is 1000 * workload + 10 * m + variant.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32


def padded(n: int) -> int:
    return -(-n // BLOCK) * BLOCK


def case_seed(workload: int, m: int, variant: int = 0) -> int:
    return 1000 * workload + 10 * m + variant


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round fp32 values (finite) to the nearest bf16, ties to even; returns uint16 bit patterns."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(m: int, K: int, seed: int) -> np.ndarray:
    """bf16(N(0,1)) activations [m, K] as uint16 bit patterns."""
    return f32_to_bf16_bits(_rng(seed).standard_normal((m, K), dtype=np.float32))


def weight(K: int, N: int, seed: int):
    """A Q8_0 weight drawn as the workloads describe: (q int8 [K, Np], s float32 [K/32, Np]), pads zero."""
    if K % BLOCK:
        raise ValueError("K must be a whole number of 32-row blocks")
    rng = _rng(seed + 7919)
    nb, Np = K // BLOCK, padded(N)
    q = np.zeros((K, Np), dtype=np.int8)
    s = np.zeros((nb, Np), dtype=np.float32)
    body = rng.integers(-127, 128, size=(K, N), dtype=np.int16).astype(np.int8)
    pos = rng.integers(0, BLOCK, size=(nb, N))
    sign = np.where(rng.integers(0, 2, size=(nb, N)) == 1, 127, -127).astype(np.int8)
    rows = BLOCK * np.arange(nb)[:, None] + pos
    body[rows, np.arange(N)[None, :]] = sign
    q[:, :N] = body
    u = rng.uniform(-8.0, -2.0, size=(nb, N))
    s[:, :N] = (np.exp2(u) / 127.0).astype(np.float32)
    return q, s


def case(m: int, K: int, N: int, seed: int):
    """x bits [m, K], q [K, Np], s [K/32, Np] for one product."""
    return activations(m, K, seed), *weight(K, N, seed)


# ---------------------------------------------------------------------------------------------------------------
# Device draws (torch).  Same distributions; the bits differ from the host draws (a different generator).
# ---------------------------------------------------------------------------------------------------------------

def device_weight(K: int, N: int, seed: int, device="cuda"):
    """(q int8 [K, Np], s float32 [K/32, Np]) drawn on the device with a seeded torch generator; pads zero."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nb, Np = K // BLOCK, padded(N)
    q = torch.zeros((K, Np), dtype=torch.int8, device=device)
    body = torch.randint(-127, 128, (K, N), generator=g, device=device, dtype=torch.int8)
    pos = torch.randint(0, BLOCK, (nb, N), generator=g, device=device)
    sign = torch.randint(0, 2, (nb, N), generator=g, device=device, dtype=torch.int8) * 254 - 127
    rows = (BLOCK * torch.arange(nb, device=device)[:, None] + pos).reshape(-1)
    cols = torch.arange(N, device=device).repeat(nb)
    body[rows, cols] = sign.reshape(-1)
    q[:, :N] = body
    u = torch.rand((nb, N), generator=g, device=device, dtype=torch.float64) * 6.0 - 8.0
    s = torch.zeros((nb, Np), dtype=torch.float32, device=device)
    s[:, :N] = (torch.exp2(u) / 127.0).to(torch.float32)
    return q, s


def device_activations(m: int, K: int, seed: int, device="cuda"):
    """bf16(N(0,1)) activations [m, K] drawn on the device (torch's fp32 -> bf16 cast rounds to nearest-even)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((m, K), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
