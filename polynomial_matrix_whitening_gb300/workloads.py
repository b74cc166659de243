"""Seeded synthetic inputs for the ANVIL bank step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA path (tests, bench) and the CPU oracle
(tests) take their inputs from here, so the two sides see identical bytes.

Shapes follow the three projection banks of anvil.py (modded-nanogpt
track_1_short/optim, `AnvilBank` and the bank comments next to
SPLIT_BADDBMM_MIN_ROWS): qk 256 rows, vo 768 rows, mlp 2816 rows, all with 768
columns, 22 matrices per bank on one GPU.

Every generator is numpy PCG64 (`default_rng`) seeded by a list
``[workload_id, ...]`` so that any array can be regenerated on its own.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Default scalars of the page (anvil.py, the twin-rail constants and ANVIL_MAPS).
RAIL_FAST_BETA = 0.85
RAIL_SLOW_BETA = 0.98
RAIL_FAST_WEIGHT = 0.4385
MOMENTUM = 0.95
FROBENIUS_MARGIN = 1.05
FROBENIUS_EPS = 1e-6

BANK_SHAPES = {"qk": (256, 768), "vo": (768, 768), "mlp": (2816, 768)}
BANK_BATCH = 22


def gaussian(seed, shape, std):
    """N(0, std^2) fp32 array."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape, dtype=np.float64) * std).astype(np.float32)


def _orthonormal(rng, rows, cols):
    """Orthonormal columns from the QR of a Gaussian, signs fixed so diag(R) > 0."""
    q, r = np.linalg.qr(rng.standard_normal((rows, cols)))
    return q * np.sign(np.diag(r))[None, :]


def power_law(seed, g, m, n, exponent=1.5):
    """g matrices U diag(i^-exponent) V^T with random orthonormal U [m,k], V [n,k], k = min(m,n)."""
    rng = np.random.default_rng(seed)
    k = min(m, n)
    sig = np.arange(1, k + 1, dtype=np.float64) ** (-exponent)
    out = np.empty((g, m, n), np.float32)
    for i in range(g):
        u = _orthonormal(rng, m, k)
        v = _orthonormal(rng, n, k)
        out[i] = ((u * sig[None, :]) @ v.T).astype(np.float32)
    return out


def low_rank_plus_noise(seed, g, m, n, rank=32, std=0.02, noise=1e-3):
    """g matrices std * P Q^T / sqrt(rank) + noise * N(0,1), P [m,rank], Q [n,rank] ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    out = np.empty((g, m, n), np.float32)
    for i in range(g):
        p = rng.standard_normal((m, rank))
        q = rng.standard_normal((n, rank))
        e = rng.standard_normal((m, n))
        out[i] = (std * (p @ q.T) / np.sqrt(rank) + noise * e).astype(np.float32)
    return out


def mixed_bank(seed, g, m, n):
    """Matrices [0, g/2) Gaussian N(0, 0.02^2); [g/2, g) rank-32 plus 1e-3 Gaussian noise."""
    half = g // 2
    out = np.empty((g, m, n), np.float32)
    out[:half] = gaussian(list(seed) + [0], (half, m, n), 0.02)
    out[half:] = low_rank_plus_noise(list(seed) + [1], g - half, m, n)
    return out


@dataclass
class Scalars:
    """Per-step scalars of one bank: the Nesterov momentum and the twin-rail knobs."""
    momentum: float = MOMENTUM
    fast_beta: float = RAIL_FAST_BETA
    fast_weight: float = RAIL_FAST_WEIGHT
    slow_beta: float = RAIL_SLOW_BETA


@dataclass
class Bank:
    name: str
    g: int
    m: int
    n: int


@dataclass
class Workload:
    """A seeded multi-step workload: banks, per-step grads and scalars, initial velocities."""
    wid: int
    name: str
    banks: list
    steps: int
    kind: str                       # "gaussian" | "power_law" | "mixed"
    std: float = 0.02
    velocity_std: float = 0.0       # 0 => zero-initialised rails
    fresh_per_step: bool = True
    pool: int = 0                   # >0: grads cycle through a pool of this many draws
    scalars_fn: object = field(default=None, repr=False)

    def scalars(self, step: int) -> Scalars:
        return self.scalars_fn(step) if self.scalars_fn else Scalars()

    def grad(self, bank_index: int, step: int) -> np.ndarray:
        b = self.banks[bank_index]
        if self.pool:
            step = step % self.pool
        elif not self.fresh_per_step:
            step = 0
        seed = [self.wid, bank_index, step]
        if self.kind == "gaussian":
            return gaussian(seed, (b.g, b.m, b.n), self.std)
        if self.kind == "power_law":
            return power_law(seed, b.g, b.m, b.n)
        if self.kind == "mixed":
            return mixed_bank(seed, b.g, b.m, b.n)
        raise ValueError(self.kind)

    def velocity(self, bank_index: int) -> np.ndarray:
        b = self.banks[bank_index]
        if self.velocity_std == 0.0:
            return np.zeros((2, b.g, b.m, b.n), np.float32)
        return gaussian([self.wid, bank_index, 1000], (2, b.g, b.m, b.n), self.velocity_std)


def _pre_engage(step):
    # Before the engage step only the fast rail is read: fast_weight = 1.
    return Scalars(fast_weight=1.0)


def _sweep(step, steps=10):
    # fast_beta swept linearly from 0.6 to 0.85 over the steps (both ends included).
    return Scalars(fast_beta=0.6 + 0.25 * step / (steps - 1), fast_weight=1.0)


def _post_engage(step):
    return Scalars(fast_weight=RAIL_FAST_WEIGHT)


def workloads():
    """The five seeded workloads, keyed by name."""
    qk = Bank("qk", BANK_BATCH, 256, 768)
    vo = Bank("vo", BANK_BATCH, 768, 768)
    mlp = Bank("mlp", BANK_BATCH, 2816, 768)
    return {
        # single wide matrix, one step, pre-engage (fast rail only)
        "single_wide": Workload(1, "single_wide", [Bank("qk", 1, 256, 768)], 1, "gaussian",
                                scalars_fn=_pre_engage),
        # the same, with the printed post-engage fast_weight
        "single_wide_blend": Workload(1, "single_wide_blend", [Bank("qk", 1, 256, 768)], 1,
                                      "gaussian", scalars_fn=_post_engage),
        "qk_bank": Workload(2, "qk_bank", [qk], 10, "gaussian", scalars_fn=_sweep),
        "vo_bank": Workload(3, "vo_bank", [vo], 10, "gaussian", velocity_std=0.01,
                            scalars_fn=_post_engage),
        "mlp_bank": Workload(4, "mlp_bank", [mlp], 10, "power_law", fresh_per_step=False,
                             scalars_fn=_post_engage),
        "full_step": Workload(5, "full_step", [qk, vo, mlp], 100, "mixed", pool=4,
                              scalars_fn=_post_engage),
    }


def random_case(seed, g, m, n, std=0.02, velocity_std=0.01):
    """A small generic case (grad, velocity) for parity tests of odd shapes."""
    grad = gaussian([9000, seed, 0], (g, m, n), std)
    vel = gaussian([9000, seed, 1], (2, g, m, n), velocity_std)
    return grad, vel
