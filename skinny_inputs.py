"""Seeded synthetic inputs for the skinny BF16 GEMM workloads.

This module is the ONLY code shared by the CUDA path's tests / bench and the
CPU oracle.  It draws random numbers and rounds them to bf16; it holds none of
the GEMM's arithmetic.

Recipe (the same on every machine that runs it):

* draws are fp32 from a CPU ``torch.Generator`` seeded per case;
* values are then rounded once to bf16 with round-to-nearest-even (torch's
  fp32 -> bf16 conversion) and returned as ``uint16`` bit patterns;
* "x100 outliers": a second draw (uniform) picks about 1% of the entries,
  which are multiplied by 100 in fp32 before the single rounding to bf16.

Workloads (sizes, distributions and structure follow the router GEMM and the
decode-projection GEMMs that the pages describe: 256 / 384 experts x 7168
hidden for the MoE router, K = 2880 as the non-tile-aligned K, and the
qkv_a / q_b / eh_proj style projection shapes):

* ``router_small``   M=1, K=7168, N=256, X~N(0,1), W~N(0,0.02^2), seed 0.
* ``dotprod``        M in {1,2,3,4} x (K,N) in {(7168,256),(7168,384),(2880,128)},
                     same distributions, seeds 1..12 (one per case).
* ``splitk``         M in {5,8,12,16} x (K,N) in {(7168,256),(7168,384),(4096,256)},
                     same distributions, seeds 101..112.
* ``projection``     M in {1,2,3,8,16} x (N,K) in {(2112,7168),(24576,1536),(7168,14336)},
                     X~N(0,1), W~U(-1/sqrt(K), 1/sqrt(K)), output stride ldy = N+64,
                     seeds 201..215.
* ``edge``           200 random cases, M in [1,16], N in [1,1024], K in [1,8200],
                     ldw = K (so odd K gives rows that are not 16-byte aligned),
                     ldy in [N, N+67], X and W ~N(0,1) with 1% x100 outliers;
                     case parameters from master seed 4.
* ``pdl_chain``      64 back-to-back calls M=4, K=7168, N=256 (seed 5).
* same-sign operands (``abs_normal``: |N(0,1)|, ``abs_uniform_isqrtk``:
  U(0, 1/sqrt(K))) for the accumulation tests: every product is positive,
  so rounding errors of a long fp32 sum cannot cancel.
* ``midm``           the medium-M decode regime, 17..64 tokens:
                     M in {17,24,32,40,64} x (K,N) in {(7168,256),(4096,384)}
                     (router distributions, seeds 401..410), then
                     M in {17,32,64} x (N,K) in {(2112,7168),(24576,1536)} and
                     M in {17,32} x (N,K) = (7168,14336) (projection
                     distributions, ldy = N+64, seeds 421..428).
* ``midm_edge``      40 random cases, M in [17,64], N in [1,1024],
                     K = 16*[1,512] (the path needs K % 16 == 0), ldy in [N, N+67],
                     X and W ~N(0,1) with 1% x100 outliers; master seed 6.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Iterator

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Case:
    """One GEMM call: shapes, strides, value distribution and seed."""
    name: str
    M: int
    N: int
    K: int
    seed: int
    x_dist: str = "normal"          # "normal" -> N(0,1); "abs_normal" -> |N(0,1)|
    w_dist: str = "normal0.02"      # "normal0.02", "uniform_isqrtk", "normal", "abs_normal",
                                    # "abs_uniform_isqrtk" (U(0, 1/sqrt(K)))
    outliers: bool = False          # 1% of entries x100 (both X and W)
    ldx: int | None = None
    ldw: int | None = None
    ldy: int | None = None

    @property
    def lx(self) -> int:
        return self.K if self.ldx is None else self.ldx

    @property
    def lw(self) -> int:
        return self.K if self.ldw is None else self.ldw

    @property
    def ly(self) -> int:
        return self.N if self.ldy is None else self.ldy

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes the GEMM must move at least once: W, X (bf16) and Y (fp32)."""
        return 2 * self.N * self.K + 2 * self.M * self.K + 4 * self.M * self.N

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _to_bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Round fp32 to bf16 (round-to-nearest-even) and return the bit patterns."""
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _draw(shape: tuple[int, int], dist: str, K: int, outliers: bool,
          g: torch.Generator) -> np.ndarray:
    if dist == "normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "normal0.02":
        v = torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    elif dist == "uniform_isqrtk":
        bound = 1.0 / math.sqrt(max(K, 1))
        v = (torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0) * bound
    elif dist == "abs_normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32).abs()
    elif dist == "abs_uniform_isqrtk":
        v = torch.rand(shape, generator=g, dtype=torch.float32) / math.sqrt(max(K, 1))
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    if outliers:
        pick = torch.rand(shape, generator=g, dtype=torch.float32) < 0.01
        v = torch.where(pick, v * 100.0, v)
    return _to_bf16_bits(v)


def make_inputs(case: Case) -> tuple[np.ndarray, np.ndarray]:
    """Compact bf16 bit patterns ``X [M,K]`` and ``W [N,K]`` for ``case``.

    Strided layouts (``ldx``/``ldw`` > K) are built by the caller from these
    compact arrays so that the values do not depend on the strides."""
    g = torch.Generator().manual_seed(int(case.seed))
    X = _draw((case.M, case.K), case.x_dist, case.K, case.outliers, g)
    W = _draw((case.N, case.K), case.w_dist, case.K, case.outliers, g)
    return X, W


def make_f32_weights(case: Case) -> np.ndarray:
    """fp32 weights ``W [N, K]`` for the fp32-router-weight path: the case's W
    distribution drawn in fp32 and kept at full fp32 precision (no rounding to
    bf16), from the case seed + 7919 so they differ from ``make_inputs``' W."""
    g = torch.Generator().manual_seed(int(case.seed) + 7919)
    shape = (case.N, case.K)
    if case.w_dist == "normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    elif case.w_dist == "normal0.02":
        v = torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    elif case.w_dist == "uniform_isqrtk":
        v = (torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0) / math.sqrt(max(case.K, 1))
    elif case.w_dist == "abs_normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32).abs()
    elif case.w_dist == "abs_uniform_isqrtk":
        v = torch.rand(shape, generator=g, dtype=torch.float32) / math.sqrt(max(case.K, 1))
    else:
        raise ValueError(f"unknown distribution {case.w_dist!r}")
    if case.outliers:
        pick = torch.rand(shape, generator=g, dtype=torch.float32) < 0.01
        v = torch.where(pick, v * 100.0, v)
    return v.numpy().copy()


def embed_rows(a: np.ndarray, ld: int, fill: int = 0) -> np.ndarray:
    """Place a compact ``[R, C]`` array into a flat buffer with row stride ``ld``."""
    R, C = a.shape
    if ld < C:
        raise ValueError("stride smaller than row length")
    out = np.full(max(R, 1) * ld, fill, dtype=a.dtype)
    if R and C:
        out[: R * ld].reshape(R, ld)[:, :C] = a
    return out


# --------------------------------------------------------------------------- workloads

ROUTER_SHAPES_DOT = [(7168, 256), (7168, 384), (2880, 128)]     # (K, N)
ROUTER_SHAPES_SPLIT = [(7168, 256), (7168, 384), (4096, 256)]   # (K, N)
PROJECTION_SHAPES = [(2112, 7168), (24576, 1536), (7168, 14336)]  # (N, K)


def router_small() -> list[Case]:
    return [Case("router_small", M=1, N=256, K=7168, seed=0)]


def dotprod_cases() -> list[Case]:
    out = []
    seed = 1
    for (K, N) in ROUTER_SHAPES_DOT:
        for M in (1, 2, 3, 4):
            out.append(Case(f"dotprod_M{M}_K{K}_N{N}", M=M, N=N, K=K, seed=seed))
            seed += 1
    return out


def splitk_cases() -> list[Case]:
    out = []
    seed = 101
    for (K, N) in ROUTER_SHAPES_SPLIT:
        for M in (5, 8, 12, 16):
            out.append(Case(f"splitk_M{M}_K{K}_N{N}", M=M, N=N, K=K, seed=seed))
            seed += 1
    return out


def projection_cases() -> list[Case]:
    out = []
    seed = 201
    for (N, K) in PROJECTION_SHAPES:
        for M in (1, 2, 3, 8, 16):
            out.append(Case(f"proj_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=seed,
                            w_dist="uniform_isqrtk", ldy=N + 64))
            seed += 1
    return out


def edge_cases(count: int = 200, master_seed: int = 4) -> list[Case]:
    rng = np.random.default_rng(master_seed)
    out = []
    for i in range(count):
        M = int(rng.integers(1, 17))
        N = int(rng.integers(1, 1025))
        K = int(rng.integers(1, 8201))
        ldy = N + int(rng.integers(0, 68))
        seed = int(rng.integers(0, 2**31 - 1))
        out.append(Case(f"edge{i:03d}_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=seed,
                        x_dist="normal", w_dist="normal", outliers=True, ldy=ldy))
    return out


def midm_cases() -> list[Case]:
    out = []
    seed = 401
    for (K, N) in ((7168, 256), (4096, 384)):
        for M in (17, 24, 32, 40, 64):
            out.append(Case(f"midm_M{M}_K{K}_N{N}", M=M, N=N, K=K, seed=seed))
            seed += 1
    seed = 421
    for (N, K), ms in (((2112, 7168), (17, 32, 64)), ((24576, 1536), (17, 32, 64)), ((7168, 14336), (17, 32))):
        for M in ms:
            out.append(Case(f"midm_proj_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=seed,
                            w_dist="uniform_isqrtk", ldy=N + 64))
            seed += 1
    return out


def midm_edge_cases(count: int = 40, master_seed: int = 6) -> list[Case]:
    rng = np.random.default_rng(master_seed)
    out = []
    for i in range(count):
        M = int(rng.integers(17, 65))
        N = int(rng.integers(1, 1025))
        K = 16 * int(rng.integers(1, 513))
        ldy = N + int(rng.integers(0, 68))
        seed = int(rng.integers(0, 2**31 - 1))
        out.append(Case(f"midm_edge{i:02d}_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=seed,
                        x_dist="normal", w_dist="normal", outliers=True, ldy=ldy))
    return out


def pdl_chain_case() -> Case:
    return Case("pdl_chain_M4_K7168_N256", M=4, N=256, K=7168, seed=5)


WORKLOADS = {
    "router_small": router_small,
    "dotprod": dotprod_cases,
    "splitk": splitk_cases,
    "projection": projection_cases,
    "edge": edge_cases,
    "midm": midm_cases,
    "midm_edge": midm_edge_cases,
}


def workload(name: str) -> list[Case]:
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")
    return WORKLOADS[name]()


def iter_all() -> Iterator[Case]:
    for name in WORKLOADS:
        yield from workload(name)
