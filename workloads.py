"""Seeded synthetic inputs for the persistent batched GEMM with custom epilogue.

This module only draws inputs and lays them out in memory.  It holds none of
the GEMM or epilogue arithmetic, and it is the one piece the oracle side and
the CUDA side share.

Draw recipe (the pages give problem shapes but no data; this is the plainest
reading): one ``torch.Generator('cpu').manual_seed(seed)`` per workload; the
tensors are drawn in the order A, B, C, X, each over its logical index order
(A [L][M][K], B [L][N][K], C/X [L][M][N]); values are rounded to the storage
type with ``.to()`` (round to nearest even); only then are they laid out in
the requested major order, so logical values never depend on the layout.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

# ---------------------------------------------------------------- workloads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    L: int
    ab: str                 # "f16" | "bf16" | "e4m3"
    a_mn_major: bool        # A stored M-major (column-major) instead of K-major
    b_mn_major: bool        # B stored N-major instead of K-major
    c: str | None           # C type or None (not supplied)
    d: str
    x: str | None           # X type or None
    y: str | None           # Y type or None (Y not written)
    cd_m_major: bool        # C/D/X/Y stored M-major instead of N-major
    alpha: float
    beta: float
    x_factor: float
    seed: int
    dist: str               # see draw()
    b: str | None = None    # B's type when it differs from A's (fp8 pairs)
    relu: bool = False      # D = max(alpha*AB + beta*C, 0) + x_factor*X
    acc: str = "f32"        # tensor-core accumulator: "f32" or "f16"

    @property
    def b_type(self) -> str:
        return self.b or self.ab

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K * self.L


# The five problem shapes the benchmark description lists, plus the bf16
# 8192^3 GEMM its throughput target names.
WORKLOADS = {
    "int256_f16_f32": Workload("int256_f16_f32", 256, 256, 256, 1, "f16", False, False,
                               "f32", "f32", None, None, False, 1.5, -0.5, 0.0, 0, "int2"),
    "gemm2048_bf16_f32": Workload("gemm2048_bf16_f32", 2048, 2048, 2048, 1, "bf16", False,
                                  False, "f32", "f32", None, None, False, 1.0, 1.0, 0.0, 1,
                                  "uniform1"),
    "efc8192_f16": Workload("efc8192_f16", 8192, 8192, 8192, 1, "f16", False, False, "f16",
                            "f16", "f16", "f16", False, 2.0, 1.0, 3.0, 2, "normal1"),
    "gemm8192_bf16": Workload("gemm8192_bf16", 8192, 8192, 8192, 1, "bf16", False, False,
                              "bf16", "bf16", None, None, False, 1.0, 1.0, 0.0, 5, "normal1"),
    "batched16_bf16_mn": Workload("batched16_bf16_mn", 1024, 1024, 4096, 16, "bf16", True, True,
                                  "bf16", "bf16", None, None, True, 0.5, 0.0, 0.0, 3,
                                  "normal002"),
    "ragged_e4m3_f16": Workload("ragged_e4m3_f16", 3000, 5000, 4096, 1, "e4m3", False, False,
                                "f16", "f16", None, None, False, 0.25, 1.0, 0.0, 4,
                                "e4m3_pm4"),
    # Beyond the listed shapes: E5M2 inputs, and a mixed E4M3 x E5M2 pair with
    # the relu epilogue and an X term.
    "e5m2_4096_f16": Workload("e5m2_4096_f16", 4096, 4096, 4096, 1, "e5m2", False, False,
                              "f16", "f16", None, None, False, 0.25, 1.0, 0.0, 6, "e4m3_pm4"),
    "fp8mix_relu_4096": Workload("fp8mix_relu_4096", 4096, 4096, 4096, 1, "e4m3", False, False,
                                 "f16", "f16", "f16", None, False, 0.25, 1.0, 0.5, 7,
                                 "e4m3_pm4", b="e5m2", relu=True),
    # tf32 inputs (fp32 storage of tf32 values), fp32 C and D
    "tf32_4096_f32": Workload("tf32_4096_f32", 4096, 4096, 4096, 1, "tf32", False, False,
                              "f32", "f32", None, None, False, 1.0, 1.0, 0.0, 8, "normal1"),
    # fp16 accumulation: fp16 inputs with the custom epilogue, and E4M3 inputs
    "f16acc_4096_f16": Workload("f16acc_4096_f16", 4096, 4096, 4096, 1, "f16", False, False,
                                "f16", "f16", "f16", "f16", False, 2.0, 1.0, 3.0, 9, "normal1",
                                acc="f16"),
    "e4m3_f16acc_4096": Workload("e4m3_f16acc_4096", 4096, 4096, 4096, 1, "e4m3", False, False,
                                 "f16", "f16", None, None, False, 0.25, 1.0, 0.0, 10, "e4m3_pm4",
                                 acc="f16"),
}

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
               "e4m3": torch.uint8, "e5m2": torch.uint8, "tf32": torch.float32}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1, "e5m2": 1, "tf32": 4}


def round_to_tf32(v: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to the nearest tf32 value (10 fraction bits, ties to
    even), kept in fp32 storage: the tf32 inputs' storage type."""
    bits = v.contiguous().view(torch.int32)
    lsb = (bits >> 13) & 1
    bits = (bits + 0xFFF + lsb) & ~0x1FFF
    return bits.view(torch.float32)


def e4m3_codes_in_pm4() -> torch.Tensor:
    """The 146 OCP E4M3 bit patterns whose value lies in [-4, 4].

    Selected by bit pattern alone: exponent field <= 8 covers every value
    below 4 (subnormals, both zeros, biased exponents 1..8), and exponent 9
    with a zero mantissa is exactly 4.0."""
    codes = []
    for c in range(256):
        e, f = (c >> 3) & 0xF, c & 0x7
        if e <= 8 or (e == 9 and f == 0):
            codes.append(c)
    return torch.tensor(codes, dtype=torch.uint8)


def e5m2_codes_in_pm4() -> torch.Tensor:
    """The 138 OCP E5M2 bit patterns whose value lies in [-4, 4]: exponent
    field <= 16 (every value below 4, both zeros, subnormals) or exponent 17
    with a zero mantissa (exactly 4.0).  Selected by bit pattern alone."""
    codes = []
    for c in range(256):
        e, f = (c >> 2) & 0x1F, c & 0x3
        if e <= 16 or (e == 17 and f == 0):
            codes.append(c)
    return torch.tensor(codes, dtype=torch.uint8)


def draw(dist: str, shape, gen: torch.Generator, out_dtype: str) -> torch.Tensor:
    """One seeded draw over a logical shape, rounded to `out_dtype` storage."""
    if dist == "int2":         # integers uniform in [-2, 2]
        v = torch.randint(-2, 3, shape, generator=gen).to(torch.float32)
    elif dist == "uniform1":   # uniform [-1, 1)
        v = torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
    elif dist == "normal1":    # N(0, 1)
        v = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif dist == "normal002":  # N(0, sigma=0.02)
        v = torch.randn(shape, generator=gen, dtype=torch.float32) * 0.02
    elif dist == "e4m3_pm4":   # discrete uniform over the fp8 codes in [-4, 4]
        # (146 E4M3 codes or 138 E5M2 codes, by the storage type asked for)
        table = e4m3_codes_in_pm4() if out_dtype == "e4m3" else e5m2_codes_in_pm4()
        idx = torch.randint(0, table.numel(), shape, generator=gen)
        assert out_dtype in ("e4m3", "e5m2")
        return table[idx]
    else:
        raise ValueError(dist)
    if out_dtype == "tf32":
        return round_to_tf32(v)
    return v.to(TORCH_DTYPE[out_dtype])


@dataclasses.dataclass
class Inputs:
    """Logical tensors (CPU, storage dtype): A [L,M,K], B [L,N,K], C/X [L,M,N]."""
    A: torch.Tensor
    B: torch.Tensor
    C: torch.Tensor | None
    X: torch.Tensor | None


def make_inputs(w: Workload, M=None, N=None, K=None, L=None, seed=None) -> Inputs:
    """Draw A, B, C, X for workload `w` (shape and seed overridable)."""
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    L = w.L if L is None else L
    gen = torch.Generator("cpu").manual_seed(w.seed if seed is None else seed)
    A = draw(w.dist, (L, M, K), gen, w.ab)
    B = draw(w.dist, (L, N, K), gen, w.b_type)
    cdist = {"e4m3_pm4": "uniform1"}.get(w.dist, w.dist)
    C = draw(cdist, (L, M, N), gen, w.c) if w.c else None
    X = draw(cdist, (L, M, N), gen, w.x) if w.x else None
    return Inputs(A, B, C, X)


# ---------------------------------------------------------------- layouts


def to_storage(t: torch.Tensor, mn_major: bool) -> torch.Tensor:
    """Lay a logical [L, R, K] (or [L, M, N]) tensor out in memory.

    mn_major=False keeps the last logical dimension contiguous (K-major for
    A/B, N-major for C/D/X/Y); mn_major=True makes the middle one contiguous
    (M- or N-major), i.e. stores [L][K][R]."""
    return (t.transpose(1, 2) if mn_major else t).contiguous()


def from_storage(t: torch.Tensor, mn_major: bool) -> torch.Tensor:
    """Inverse of to_storage: back to the logical [L, R, C] view."""
    return t.transpose(1, 2) if mn_major else t


def storage_view_np(t: torch.Tensor) -> np.ndarray:
    """The raw storage of a CPU tensor as numpy (bit patterns for 16-bit)."""
    t = t.contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.numpy()


# ---------------------------------------------------------------- sampling


def check_entries(M: int, N: int, L: int, tile_m: int, tile_n: int, seed: int,
                  n_random: int = 4096, max_boundaries: int = 8):
    """Entries to compare at full size: `n_random` seeded (m, n, l) triples,
    plus the index sets of full rows and columns at tile boundaries.

    Returns (ms, ns, ls, rows, cols): 1-D random triples, and the lists of
    row and column indices to check in full (each in every batch)."""
    g = np.random.default_rng(seed)
    ms = g.integers(0, M, n_random)
    ns = g.integers(0, N, n_random)
    ls = g.integers(0, L, n_random)

    def boundary(ext, t):
        idx = {0, ext - 1}
        if ext > t:
            idx |= {t - 1, t}
        nb = (ext - 1) // t
        picks = np.unique(np.linspace(1, nb, min(nb, max_boundaries)).astype(int)) if nb else []
        for b in picks:
            for i in (b * t - 1, b * t):
                if 0 <= i < ext:
                    idx.add(int(i))
        last = (ext // t) * t          # first row of the last (partial) tile
        if last < ext:
            idx |= {last, ext - 1}
        return sorted(i for i in idx if 0 <= i < ext)

    return ms, ns, ls, boundary(M, tile_m), boundary(N, tile_n)
