"""Seeded synthetic workloads for the SVDQuant W4A4 linear layer.

This module only draws random numbers and rounds them to the BF16 input format.
It holds none of the layer's arithmetic (no smoothing, SVD, quantisation or
matmul), so that the CPU oracle and the CUDA path can both be fed from it
without sharing any of the method's code.

Workload shapes are the FLUX.1-dev transformer linears the SVDQuant/Nunchaku
pages benchmark on ("Concrete performance gains" and "Performance Benchmarks"
sections of the Nunchaku/Diffusers articles): QKV projection, MLP up and down
projections and the 3072->3072 output projection.  The pages use trained FLUX
weights and real activations; these generators stand in for them with the value
distributions below (Gaussian activations with a few large outlier channels,
Gaussian weights with a low-rank spike, heavy-tailed post-GELU activations).

Draw order per workload (one numpy Generator, fixed order):
  1. outlier channel indices (without replacement)
  2. outlier factors
  3. X
  4. W
  5. spike factors U, V (Gaussian, then orthonormalised by QR)
  6. bias
Values are drawn in float64, then rounded float64 -> float32 -> bfloat16 with
round-to-nearest-even at each step.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    rank: int
    x_kind: str = "gauss_outliers"   # "gauss_outliers" | "abs_student_t3"
    n_outlier: int = 0               # number of outlier channels in X
    outlier_lo: float = 1.0          # outlier factor range (uniform); lo == hi -> fixed
    outlier_hi: float = 1.0
    spike_rank: int = 0              # rank of the additive weight spike
    spike_sigma: float = 0.0         # its singular value
    bias_std: float = 0.1
    seed: int = 0

    @property
    def flops_4bit(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def flops_lowrank(self) -> int:
        return 2 * self.M * self.K * self.rank + 2 * self.M * self.rank * self.N


def _flux(name, M, K, N, rank, **kw) -> Workload:
    n_out = int(round(0.01 * K))
    base = dict(x_kind="gauss_outliers", n_outlier=n_out, outlier_lo=20.0,
                outlier_hi=50.0, spike_rank=8, spike_sigma=5.0)
    base.update(kw)
    return Workload(name, M, K, N, rank, **base)


TINY = Workload("tiny", 64, 256, 256, 16, "gauss_outliers", 4, 30.0, 30.0, 4, 5.0)
QKV = _flux("flux_qkv", 4608, 3072, 9216, 32)
MLP_UP = _flux("flux_mlp_up", 4608, 3072, 12288, 32)
MLP_DOWN = Workload("flux_mlp_down", 4608, 12288, 3072, 32, x_kind="abs_student_t3")
OPROJ_M = [_flux(f"flux_oproj_m{m}", m, 3072, 3072, 32) for m in (256, 1024, 4096, 16384)]
OPROJ_R = [_flux(f"flux_oproj_r{r}", 4096, 3072, 3072, r) for r in (16, 64, 128)]

# AWQ-style W4A16 modulation layers: the conditioning vector (one row per image, two with
# classifier-free guidance) against the adaptive-norm weight that produces the six
# 3072-wide shift / scale / gate vectors of a FLUX double block; rank is unused (0)
MOD = _flux("flux_mod", 1, 3072, 6 * 3072, 0)
MOD_CFG = _flux("flux_mod_cfg", 2, 3072, 6 * 3072, 0)
AWQ_WORKLOADS = [MOD, MOD_CFG]

# every timed point of the FLUX-shaped scope, the headline (MLP up) first
SWEEP = [MLP_UP, QKV, MLP_DOWN, *OPROJ_M, *OPROJ_R]

WORKLOADS: Dict[str, Workload] = {w.name: w for w in [TINY, QKV, MLP_UP, MLP_DOWN, *OPROJ_M, *OPROJ_R, *AWQ_WORKLOADS]}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(w: Workload, **changes) -> Workload:
    """Same value recipe with other sizes (used for small parity cases)."""
    return dataclasses.replace(w, **changes)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE) bit patterns as uint16."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make(w: Workload, seed: int | None = None) -> Dict[str, np.ndarray]:
    """Draw X (M x K), W (N x K) and bias (N) as bfloat16 bit patterns."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    M, K, N = w.M, w.K, w.N
    idx = rng.choice(K, size=w.n_outlier, replace=False) if w.n_outlier else np.zeros(0, np.int64)
    if w.n_outlier:
        if w.outlier_lo == w.outlier_hi:
            fac = np.full(w.n_outlier, w.outlier_lo)
        else:
            fac = rng.uniform(w.outlier_lo, w.outlier_hi, size=w.n_outlier)
    else:
        fac = np.zeros(0)
    if w.x_kind == "gauss_outliers":
        X = rng.standard_normal((M, K))
    elif w.x_kind == "abs_student_t3":
        X = np.abs(rng.standard_t(3.0, size=(M, K)))
    else:
        raise ValueError(w.x_kind)
    if w.n_outlier:
        X[:, idx] *= fac[None, :]
    W = rng.standard_normal((N, K)) * (1.0 / np.sqrt(K))
    if w.spike_rank:
        U, _ = np.linalg.qr(rng.standard_normal((N, w.spike_rank)))
        V, _ = np.linalg.qr(rng.standard_normal((K, w.spike_rank)))
        W += w.spike_sigma * (U @ V.T)
    b = rng.standard_normal(N) * w.bias_std
    return {
        "X": f64_to_bf16_bits(X),
        "W": f64_to_bf16_bits(W),
        "bias": f64_to_bf16_bits(b),
        "outlier_channels": np.sort(idx),
    }


def make_x(w: Workload, M: int, seed: int) -> np.ndarray:
    """Another activation batch of the same recipe (for e2e and flush inputs)."""
    return make(scaled(w, M=M), seed=seed)["X"]


def make_weights(w: Workload, seed: int | None = None) -> Dict[str, np.ndarray]:
    """W (N x K) and bias (N) of the recipe alone, from their own generator (the second layer of
    an MLP pair, whose input is the first layer's activated output, not drawn).  Draw order: W,
    spike factors U, V, bias."""
    rng = np.random.default_rng((w.seed if seed is None else seed, 1))
    N, K = w.N, w.K
    W = rng.standard_normal((N, K)) * (1.0 / np.sqrt(K))
    if w.spike_rank:
        U, _ = np.linalg.qr(rng.standard_normal((N, w.spike_rank)))
        V, _ = np.linalg.qr(rng.standard_normal((K, w.spike_rank)))
        W += w.spike_sigma * (U @ V.T)
    b = rng.standard_normal(N) * w.bias_std
    return {"W": f64_to_bf16_bits(W), "bias": f64_to_bf16_bits(b)}


@dataclasses.dataclass(frozen=True)
class PairWorkload:
    """An MLP pair: up (M x K -> N_up), GELU, down (N_up -> N).  X, W_up and b_up come from
    make(up); W_down and b_down from make_weights(down)."""
    name: str
    up: Workload
    down: Workload

    def __post_init__(self):
        assert self.down.K == self.up.N and self.down.M == self.up.M


# the FLUX transformer block's feed-forward (3072 -> 12288 -> GELU -> 3072)
MLP_PAIR = PairWorkload("flux_mlp_pair", MLP_UP, MLP_DOWN)


def pair(name: str, M: int, K: int, N_up: int, N: int, r_up: int, r_down: int) -> PairWorkload:
    """A smaller pair with the FLUX pair's value recipes."""
    return PairWorkload(name, scaled(MLP_UP, name=name + "_up", M=M, K=K, N=N_up, rank=r_up,
                                     n_outlier=max(1, int(round(0.01 * K)))),
                        scaled(MLP_DOWN, name=name + "_down", M=M, K=N_up, N=N, rank=r_down))


def pair_parity_cases() -> List[PairWorkload]:
    """Small pairs: ragged M and N_up, every supported down rank, one column tile per unit
    (small M) and longer units (M spanning several row blocks)."""
    return [
        pair("pair_tiny", 64, 256, 256, 128, 16, 16),
        pair("pair_ragged", 300, 512, 320, 272, 32, 32),
        pair("pair_r64", 257, 768, 1024, 512, 32, 64),
        pair("pair_r48_small_m", 40, 256, 2048, 256, 16, 48),
        pair("pair_down_r0", 130, 256, 512, 256, 16, 0),
        pair("pair_units", 2560, 256, 4096, 256, 32, 32),
    ]


def parity_cases() -> List[Workload]:
    """Small cases: several tiles of every kernel plus a ragged tail in M."""
    return [
        TINY,
        scaled(QKV, name="qkv_small", M=300, K=512, N=768, rank=32, n_outlier=5),
        scaled(MLP_DOWN, name="down_small", M=130, K=1024, N=512, rank=16),
        scaled(QKV, name="rank64_small", M=257, K=768, N=512, rank=64, n_outlier=8),
        # long K at small M: the split-K activation kernel, K % 256 != 0
        scaled(MLP_DOWN, name="down_split", M=300, K=6464, N=512, rank=32),
    ]
