"""Seeded synthetic BF16 inputs shaped like the workloads the LCT pages describe.

This module holds no codec arithmetic: it draws float64 samples with
``numpy.random.default_rng(seed)``, casts them to float32 and then to BF16 with
round-to-nearest-even (torch's CPU cast, no flush to zero), and returns the raw
BF16 bit patterns as ``numpy.uint16``.  The same arrays feed the CUDA path and
the CPU oracle.

Workloads (sizes and distributions; the pages measure no public dataset for the
codec, so these synthetic tensors stand in for trained weights, optimizer state
and activations):

* ``gauss_block``   65,536 values ~ N(0, 0.02), seed 0: one CLEAN block.
* ``laplace_16m``   2^24 values ~ Laplace(0, 0.01), seed 1, CLEAN.
* ``heavy_64m``     2^26 values ~ Student-t(3) * 1e-3, seed 2; 0.1% of positions
                    multiplied by 1e4 and a further 1% replaced by +-1e-39
                    (BF16 subnormals); MEDIUM.
* ``sgd_162m``      W ~ N(0, 0.02) (seed 3) and M ~ N(0, 1e-3) (seed 4),
                    162,000,000 values each, CLEAN, eta = 1e-3.
* ``momentum_162m`` the ``sgd_162m`` W and M with a dense BF16 gradient
                    g ~ N(0, 1e-4) (seed 6 on odd steps, 7 on even ones),
                    mu = 0.9, eta = 1e-3: SGD with momentum.
* ``adamw_162m``    the ``sgd_162m`` W, a first moment M ~ N(0, 1e-4) (seed 4),
                    a second moment V = |N(0, 1e-8)| (seed 5) and the
                    ``momentum_162m`` gradients; AdamW with lr = 1e-3,
                    betas (0.9, 0.999), eps = 1e-8, weight decay 0.01.
* ``gelu_act``      [8, 4096, 3072] GELU(z), z ~ N(0, 1), seed 5, with 30% of
                    positions set to +0.0; HIGH; scaled by 2^k, k = -4..4.
* ``gelu_act_zero`` the same activations coded with a zero-atom Gaussian(1)
                    model (a point mass of 0.3 at zero).
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = ["bf16_bits", "normal", "laplace", "heavy_tail", "gelu_sparse", "scale_pow2",
           "all_bf16_patterns", "random_bits", "generate", "momentum", "gradient", "second_moment",
           "WORKLOADS"]


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float64/float32 array -> BF16 bit patterns (float32 first, then RNE)."""
    f32 = np.ascontiguousarray(a, dtype=np.float32)
    t = torch.from_numpy(f32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def normal(n: int, sigma: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.normal(0.0, sigma, size=n))


def laplace(n: int, b: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.laplace(0.0, b, size=n))


def heavy_tail(n: int, seed: int = 2, nu: float = 3.0, scale: float = 1e-3,
               outlier_frac: float = 0.001, outlier_mult: float = 1e4,
               tiny_frac: float = 0.01, tiny: float = 1e-39) -> np.ndarray:
    """Student-t(nu)*scale; one permutation picks disjoint position sets: the
    first floor(outlier_frac*n) are multiplied by outlier_mult, the next
    floor(tiny_frac*n) become sign(x)*tiny."""
    rng = np.random.default_rng(seed)
    x = rng.standard_t(nu, size=n) * scale
    perm = rng.permutation(n)
    n_out = int(np.floor(outlier_frac * n))
    n_tiny = int(np.floor(tiny_frac * n))
    x[perm[:n_out]] *= outlier_mult
    idx = perm[n_out:n_out + n_tiny]
    x[idx] = np.sign(x[idx]) * tiny
    return bf16_bits(x)


def gelu_sparse(n: int, seed: int = 5, zero_frac: float = 0.3) -> np.ndarray:
    """GELU(z) = z * Phi(z) (erf form) for z ~ N(0, 1), then a uniformly
    chosen floor(zero_frac*n) positions set to +0.0."""
    from scipy.special import erf
    rng = np.random.default_rng(seed)
    z = rng.normal(0.0, 1.0, size=n)
    x = z * 0.5 * (1.0 + erf(z / np.sqrt(2.0)))
    nz = int(np.floor(zero_frac * n))
    x[rng.choice(n, size=nz, replace=False)] = 0.0
    return bf16_bits(x)


def scale_pow2(h: np.ndarray, k: int) -> np.ndarray:
    """x * 2^k for BF16 bit patterns (exact while no value leaves the normal range)."""
    with np.errstate(over="ignore", invalid="ignore"):  # infinities and NaNs stay what they are
        f = bits_to_f32(h) * np.float32(2.0 ** k)
    return bf16_bits(f)


def random_bits(n: int, seed: int) -> np.ndarray:
    """n uniformly random BF16 bit patterns: exponents spread evenly over all
    256 values, so almost every one falls outside any fitted codebook."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 65536, size=n, dtype=np.uint32).astype(np.uint16)


def all_bf16_patterns(seed: int = 7) -> np.ndarray:
    """Every one of the 65,536 BF16 bit patterns (zeros, subnormals, normals,
    infinities, NaN payloads) in a seeded random order."""
    rng = np.random.default_rng(seed)
    return rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16)


# Workload table: generator, its arguments, the codebook model the user picks
# for it, and the block level.
WORKLOADS = {
    "gauss_block": dict(n=65536, gen="normal", args=dict(sigma=0.02, seed=0),
                        model="gaussian", scale=0.02, shape=0.0, level="CLEAN"),
    "laplace_16m": dict(n=1 << 24, gen="laplace", args=dict(b=0.01, seed=1),
                        model="laplace", scale=0.01, shape=0.0, level="CLEAN"),
    "heavy_64m": dict(n=1 << 26, gen="heavy_tail", args=dict(seed=2),
                      model="powerlaw", scale=1e-3, shape=3.0, level="MEDIUM"),
    "sgd_162m": dict(n=162_000_000, gen="normal", args=dict(sigma=0.02, seed=3),
                     model="gaussian", scale=0.02, shape=0.0, level="CLEAN",
                     momentum=dict(sigma=1e-3, seed=4, model="gaussian", scale=1e-3),
                     eta=1e-3, steps=100),
    "momentum_162m": dict(n=162_000_000, gen="normal", args=dict(sigma=0.02, seed=3),
                          model="gaussian", scale=0.02, shape=0.0, level="CLEAN",
                          momentum=dict(sigma=1e-3, seed=4, model="gaussian", scale=1e-3),
                          gradient=dict(sigma=1e-4, seeds=(6, 7)), eta=1e-3, mu=0.9),
    "adamw_162m": dict(n=162_000_000, gen="normal", args=dict(sigma=0.02, seed=3),
                       model="gaussian", scale=0.02, shape=0.0, level="CLEAN",
                       momentum=dict(sigma=1e-4, seed=4, model="gaussian", scale=1e-4),
                       second=dict(sigma=1e-8, seed=5, model="laplace", scale=1e-8),
                       gradient=dict(sigma=1e-4, seeds=(6, 7)),
                       adamw=dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)),
    "gelu_act": dict(n=8 * 4096 * 3072, gen="gelu_sparse", args=dict(seed=5),
                     model="gaussian", scale=1.0, shape=0.0, level="HIGH",
                     pow2=list(range(-4, 5))),
    "gelu_act_zero": dict(n=8 * 4096 * 3072, gen="gelu_sparse", args=dict(seed=5),
                          model="gaussian", scale=1.0, shape=0.0, zero_frac=0.3, level="HIGH",
                          pow2=list(range(-4, 5))),
}


def generate(name: str, n: int | None = None) -> np.ndarray:
    """The named workload's input (optionally at another size, same recipe)."""
    w = WORKLOADS[name]
    size = w["n"] if n is None else n
    fn = {"normal": normal, "laplace": laplace, "heavy_tail": heavy_tail,
          "gelu_sparse": gelu_sparse}[w["gen"]]
    return fn(size, **w["args"])


def momentum(name: str, n: int | None = None) -> np.ndarray:
    w = WORKLOADS[name]
    m = w["momentum"]
    return normal(w["n"] if n is None else n, m["sigma"], m["seed"])


def gradient(name: str, step: int, n: int | None = None) -> np.ndarray:
    """The dense BF16 gradient of a momentum workload at step 1, 2, ...
    (two seeded draws, alternating)."""
    w = WORKLOADS[name]
    g = w["gradient"]
    return normal(w["n"] if n is None else n, g["sigma"], g["seeds"][(step - 1) % 2])


def second_moment(name: str, n: int | None = None) -> np.ndarray:
    """A non-negative second-moment tensor: |N(0, sigma)| in BF16."""
    w = WORKLOADS[name]
    sm = w["second"]
    rng = np.random.default_rng(sm["seed"])
    return bf16_bits(np.abs(rng.normal(0.0, sm["sigma"], size=w["n"] if n is None else n)))
