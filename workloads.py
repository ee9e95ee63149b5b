"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle
checks.

This module holds no step of the compression method: it only draws random
matrices and activations and rounds them to BF16.  Both the CUDA library's
tests and the oracle's tests take their inputs from here, so that the two
sides see the same bits.

Workloads (the weight shapes are those of the Llama-3.1-8B MLP the Unweight
blog post measures on; its trained weights are not available, so seeded
normal and Student-t matrices stand in for them):

  small      1024 x 1024, N(0, 0.02), seed 0, x ~ N(0,1), batch 1
  gate       14336 x 4096 gate_proj, N(0, 0.02), seed 0, batch 1
  mlp        gate/up 14336 x 4096 and down 4096 x 14336, N(0, 0.02),
             seeds 0/1/2, batches 1, 8, 32
  heavy      4096 x 4096 Student-t (nu = 4) x 0.02, then 0.1% of entries
             x100 and a disjoint 0.01% set to +0.0, batches 1, 16, 64, 256
  model      32 layers x {gate, up, down}, per-layer sigma ~ U[0.01, 0.04]
             (seed 0), matrix seed 3*layer + j, batches 1 .. 256

Rounding to BF16: fp64 samples are cast to fp32, then rounded to nearest
even on the upper 16 bits (every sample here is finite).
"""
from __future__ import annotations

import numpy as np

GATE_SHAPE = (14336, 4096)
DOWN_SHAPE = (4096, 14336)
ACT_SEED_BASE = 1_000_003


def bf16_bits(a) -> np.ndarray:
    """Round finite fp64/fp32 values to BF16 (nearest even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_weights(rows: int, cols: int, sigma: float = 0.02, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal((rows, cols)) * sigma)


def heavy_tailed_weights(rows: int = 4096, cols: int = 4096, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    w = rng.standard_t(4, (rows, cols)) * 0.02
    flat = w.reshape(-1)
    perm = np.random.default_rng(0).permutation(flat.size)
    n_big = int(round(0.001 * flat.size))
    n_zero = int(round(0.0001 * flat.size))
    flat[perm[:n_big]] *= 100.0
    flat[perm[n_big:n_big + n_zero]] = 0.0
    return bf16_bits(w)


def activations(batch: int, cols: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(ACT_SEED_BASE + seed)
    return bf16_bits(rng.standard_normal((batch, cols)))


def all_bf16_patterns() -> np.ndarray:
    """Every one of the 65,536 BF16 bit patterns once, as a 1024 x 64 matrix."""
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(1024, 64)


def model_sigmas(layers: int = 32, seed: int = 0) -> np.ndarray:
    return np.random.default_rng(seed).uniform(0.01, 0.04, layers)


def model_matrix(layer: int, j: int) -> np.ndarray:
    """Matrix j (0 gate, 1 up, 2 down) of layer `layer` of the 32-layer model."""
    sigma = float(model_sigmas()[layer])
    shape = GATE_SHAPE if j < 2 else DOWN_SHAPE
    return normal_weights(shape[0], shape[1], sigma, seed=3 * layer + j)


WORKLOADS = {
    "small": {"shape": (1024, 1024), "sigma": 0.02, "seed": 0, "batches": [1]},
    "gate": {"shape": GATE_SHAPE, "sigma": 0.02, "seed": 0, "batches": [1]},
    "mlp": {"shapes": [GATE_SHAPE, GATE_SHAPE, DOWN_SHAPE], "sigma": 0.02, "seeds": [0, 1, 2],
            "batches": [1, 8, 32]},
    "heavy": {"shape": (4096, 4096), "seed": 0, "batches": [1, 16, 64, 256]},
    "model": {"layers": 32, "batches": [1, 2, 4, 8, 16, 32, 64, 128, 256]},
}


def workload_weights(name: str) -> np.ndarray:
    spec = WORKLOADS[name]
    if name == "heavy":
        return heavy_tailed_weights(*spec["shape"], seed=spec["seed"])
    rows, cols = spec["shape"]
    return normal_weights(rows, cols, spec["sigma"], spec["seed"])
