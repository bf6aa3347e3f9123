"""Seeded synthetic inputs shaped like a 7B model's prefill GEMMs.

This module only draws random numbers and lays bytes out; it holds none of
the quantization or GEMM arithmetic.  Both the CUDA path and the CPU oracle
consume what it produces, so the same bytes feed both sides.

Recipes (numpy PCG64 streams, one seed per tensor):
  activations  x ~ N(0, 1) float32 [M][K]; optionally round(frac*K) channels,
               picked by a seeded permutation, are multiplied by `scale`
               for every token (the "1% of channels x20" outlier mix).
  q4_K weights [N][K/256][144] bytes: bytes 4..143 of every super-block are
               uniform random bytes, which makes every nibble v ~ U{0..15}
               and every 6-bit sc, m ~ U{0..63}; d and dmin ~ U(lo, hi)
               rounded to fp16 (round to nearest even) and stored little
               endian in bytes 0-1 and 2-3.
"""
from __future__ import annotations

import numpy as np

Q4K_BLOCK_BYTES = 144
QK_K = 256

# Named shapes of the 7B-at-2K-token prefill (M tokens, K in, N out).
SHAPES = {
    "tiny": (128, 512, 256),
    "q_proj": (2048, 4096, 4096),
    "gate_up": (2048, 4096, 11008),
    "down": (2048, 11008, 4096),
}
SWEEP_M = (1, 16, 77, 128, 512, 2047, 8192)

# The 7B prefill linear stack: 32 layers, each with these GEMMs as (name, K, N);
# every (layer, GEMM) has its own weights and its own activations.
STACK_LAYERS = 32
STACK_TOKENS = 2048
STACK_GEMMS = (("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
               ("gate", 4096, 11008), ("up", 4096, 11008), ("down", 11008, 4096))


def stack_seeds(layer: int, g: int):
    """(weight seed, activation seed) of GEMM g of `layer` in the stack."""
    s = 3000 + 7 * layer + g
    return s, 1_000_000 + s


def activations(M: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = rng.permutation(K)[:n_out]
        x[:, ch] *= np.float32(outlier_scale)
    return x


def q4K_weights(N: int, K: int, seed: int, d_lo: float = 1e-3,
                d_hi: float = 1e-2) -> np.ndarray:
    assert K % QK_K == 0
    nsb = K // QK_K
    rng = np.random.Generator(np.random.PCG64(seed))
    blk = rng.integers(0, 256, size=(N, nsb, Q4K_BLOCK_BYTES), dtype=np.uint8)
    d = rng.uniform(d_lo, d_hi, size=(N, nsb)).astype(np.float16)
    dmin = rng.uniform(d_lo, d_hi, size=(N, nsb)).astype(np.float16)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(N, nsb, 2)
    blk[:, :, 2:4] = dmin.view(np.uint8).reshape(N, nsb, 2)
    return blk


Q6K_BLOCK_BYTES = 210


def q6K_weights(N: int, K: int, seed: int, d_lo: float = 1e-4,
                d_hi: float = 1e-3) -> np.ndarray:
    """Customary q6_K super-blocks [N][K/256][210]: uniform random bytes for
    the quant bits (so u = q + 32 ~ U{0..63}) and the int8 scales, fp16 d ~
    U(d_lo, d_hi) in bytes 208-209."""
    assert K % QK_K == 0
    nsb = K // QK_K
    rng = np.random.Generator(np.random.PCG64(seed))
    blk = rng.integers(0, 256, size=(N, nsb, Q6K_BLOCK_BYTES), dtype=np.uint8)
    d = rng.uniform(d_lo, d_hi, size=(N, nsb)).astype(np.float16)
    blk[:, :, 208:210] = d.view(np.uint8).reshape(N, nsb, 2)
    return blk


def torch_q6K_weights(N: int, K: int, seed: int, device, d_lo: float = 1e-4, d_hi: float = 1e-3):
    """Device-side variant of q6K_weights (same recipe, torch Philox stream)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nsb = K // QK_K
    blk = torch.randint(0, 256, (N, nsb, Q6K_BLOCK_BYTES), dtype=torch.uint8, device=device, generator=g)
    d = (torch.rand((N, nsb), device=device, generator=g) * (d_hi - d_lo) + d_lo).half()
    blk[:, :, 208:210] = d.view(torch.uint8).view(N, nsb, 2)
    return blk


def config_inputs(name: str, M: int | None = None):
    """(x, blk, N) for a named workload; seeds fixed per workload."""
    if name == "tiny":
        M0, K, N = SHAPES["tiny"]
        return activations(M0, K, 1000), q4K_weights(N, K, 2000), N
    if name == "q_proj":
        M0, K, N = SHAPES["q_proj"]
        return activations(M0, K, 1001, 0.01), q4K_weights(N, K, 2001), N
    if name == "gate_up":
        M0, K, N = SHAPES["gate_up"]
        return activations(M0, K, 1002, 0.01), q4K_weights(N, K, 2002), N
    if name == "down":
        M0, K, N = SHAPES["down"]
        return activations(M0, K, 1003, 0.01), q4K_weights(N, K, 2003), N
    if name == "sweep":
        assert M is not None
        K, N = 4096, 4096
        return activations(M, K, 1004 + M), q4K_weights(N, K, 2004), N
    raise KeyError(name)


def torch_q4K_weights(N: int, K: int, seed: int, device, d_lo: float = 1e-3,
                      d_hi: float = 1e-2):
    """Device-side variant of q4K_weights (same recipe, torch Philox stream)
    for workloads too large to draw on the host."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nsb = K // QK_K
    blk = torch.randint(0, 256, (N, nsb, Q4K_BLOCK_BYTES), dtype=torch.uint8,
                        device=device, generator=g)
    d = (torch.rand((N, nsb), device=device, generator=g) * (d_hi - d_lo) + d_lo).half()
    dmin = (torch.rand((N, nsb), device=device, generator=g) * (d_hi - d_lo) + d_lo).half()
    blk[:, :, 0:2] = d.view(torch.uint8).view(N, nsb, 2)
    blk[:, :, 2:4] = dmin.view(torch.uint8).view(N, nsb, 2)
    return blk


def torch_activations(M: int, K: int, seed: int, device, outlier_frac: float = 0.0,
                      outlier_scale: float = 20.0):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((M, K), device=device, generator=g, dtype=torch.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = torch.randperm(K, device=device, generator=g)[:n_out]
        x[:, ch] *= outlier_scale
    return x
