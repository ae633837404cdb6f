"""Seeded synthetic inputs and the workload table.

This module is shared by the tests, ``bench.py`` and ``smoke()``: it is the one
place both the CUDA path and the oracle take their inputs from.  It draws
random numbers and nothing else -- no scale, code or rounding of the method is
computed here; encoding random values into codes is left to each caller (the
oracle's codec in tests, the library's own quantizer or torch's float8
conversion when preparing bench inputs).

Workloads follow the shapes and value distributions of the source pages:

* ``grouped``  -- atrex-bench #002 block_scaled_mm, Input Generation and the
  Shapes table: standard-normal float32 activations and weights, quantized
  per 1 x 128 (activations) and 128 x 128 (weights) blocks.
* ``int8``     -- TensorTonic INT8 per-channel matmul, scaled up: standard-
  normal x and w with about 1% of x rows and w columns set to zero (the page
  allows all-zero rows and columns).
* ``mxfp8`` / ``nvfp4`` -- jax.nn.scaled_matmul with the Blackwell formats:
  E4M3 codes of standard-normal values with UE8M0 exponents uniform in
  [-6, 6] per 32-block; E2M1 codes drawn uniformly over the 16 code points
  with E4M3 scales log-uniform in [2**-4, 2**4] per 16-block.
* ``backward`` -- NKI MXFP8 backward: bfloat16 dY, W, X standard normal, W and
  X multiplied by 0.02.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


# --------------------------------------------------------------------------- #
# Workload table                                                              #
# --------------------------------------------------------------------------- #

@dataclass(frozen=True)
class Grouped:
    m: int
    n: int
    k: int
    group_n: int = 128
    group_k: int = 128


@dataclass(frozen=True)
class Int8Channel:
    B: int
    D_in: int
    D_out: int
    zero_frac: float = 0.01


@dataclass(frozen=True)
class Batched:
    B: int
    M: int
    N: int
    K: int
    fmt: str  # "mxfp8" | "nvfp4"


@dataclass(frozen=True)
class Backward:
    M: int
    N: int
    K: int
    fp8: str = "e5m2"


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    problems: tuple = field(default_factory=tuple)


# The small block_scaled_mm case (m=64, n=k=256) the oracle finishes at once.
GROUPED_SMALL = Workload("block_scaled_mm m=64 n=k=256", 0, (Grouped(64, 256, 256),))
INT8_4096 = Workload("int8 per-channel B=D_in=D_out=4096", 1, (Int8Channel(4096, 4096, 4096),))
# The block_scaled_mm Shapes-table rows taken as the sweep: n=k=2048 rows with
# m = 349, 4533, 65536, 704512 and n=k=4096 rows with m = 237, 4096, 65536, 299520.
GROUPED_SWEEP = Workload(
    "block_scaled_mm sweep n=k=2048 m=349..704512, n=k=4096 m=237..299520", 2,
    tuple(Grouped(m, 2048, 2048) for m in (349, 4533, 65536, 704512))
    + tuple(Grouped(m, 4096, 4096) for m in (237, 4096, 65536, 299520)))
MXFP8_BATCHED = Workload("mxfp8 B=8 M=N=4096 K=8192", 3, (Batched(8, 4096, 4096, 8192, "mxfp8"),))
NVFP4_SQUARE = Workload("nvfp4 B=1 M=N=K=16384", 3, (Batched(1, 16384, 16384, 16384, "nvfp4"),))
# MXFP4 (E2M1 with UE8M0 per 32) at the NVFP4 problem's size; not one of the
# pages' published configurations, measured as the next format.
MXFP4_SQUARE = Workload("mxfp4 B=1 M=N=K=16384", 3, (Batched(1, 16384, 16384, 16384, "mxfp4"),))
BACKWARD = Workload("mxfp8 linear backward M=16384 N=K=8192", 4, (Backward(16384, 8192, 8192),))

WORKLOADS = {w.name: w for w in (GROUPED_SMALL, INT8_4096, GROUPED_SWEEP,
                                 MXFP8_BATCHED, NVFP4_SQUARE, MXFP4_SQUARE, BACKWARD)}


# --------------------------------------------------------------------------- #
# Seeded draws                                                                #
# --------------------------------------------------------------------------- #

def generator(seed: int, stream: int, device="cpu") -> torch.Generator:
    """A torch generator for (workload seed, named stream).  Different streams
    of one workload draw independent numbers."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def randn(shape, seed: int, stream: int, device="cpu", dtype=torch.float32,
          scale: float = 1.0) -> torch.Tensor:
    """Standard-normal draws (times ``scale``) of the given dtype."""
    g = generator(seed, stream, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        t = t * scale
    return t.to(dtype)


def zero_lines(n: int, frac: float, seed: int, stream: int) -> torch.Tensor:
    """Indices of ``round(frac * n)`` distinct lines (rows or columns) chosen
    uniformly at random; at least one when ``frac > 0``."""
    count = max(1 if frac > 0 else 0, int(round(frac * n)))
    g = generator(seed, stream)
    return torch.randperm(n, generator=g)[:count].sort().values


def uniform_int(shape, lo: int, hi: int, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """Integers uniform in [lo, hi] (inclusive), int32."""
    g = generator(seed, stream, device)
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, device=device, dtype=torch.int32)


def random_bytes(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """Uniform random bytes (uint8)."""
    return uniform_int(shape, 0, 255, seed, stream, device).to(torch.uint8)


def log_uniform(shape, lo_exp: float, hi_exp: float, seed: int, stream: int,
                device="cpu") -> torch.Tensor:
    """float32 values 2**u with u uniform in [lo_exp, hi_exp]."""
    g = generator(seed, stream, device)
    u = torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return torch.exp2(lo_exp + (hi_exp - lo_exp) * u)


# Stream ids, so every caller draws the same numbers for the same role.
S_A, S_B, S_A_SCALE, S_B_SCALE, S_X, S_W, S_DY, S_ZERO_ROWS, S_ZERO_COLS = range(9)


def grouped_raw(p: Grouped, seed: int, device="cpu"):
    """Unquantized float32 activations a[m, k] and weights b[n, k]."""
    a = randn((p.m, p.k), seed, S_A * 100 + _shape_tag(p), device)
    b = randn((p.n, p.k), seed, S_B * 100 + _shape_tag(p), device)
    return a, b


def int8_raw(p: Int8Channel, seed: int, device="cpu"):
    """x [B, D_in] and w [D_in, D_out] float32 with zeroed x rows / w columns."""
    x = randn((p.B, p.D_in), seed, S_X, device)
    w = randn((p.D_in, p.D_out), seed, S_W, device)
    x[zero_lines(p.B, p.zero_frac, seed, S_ZERO_ROWS).to(x.device)] = 0
    w[:, zero_lines(p.D_out, p.zero_frac, seed, S_ZERO_COLS).to(w.device)] = 0
    return x, w


def batched_raw(p: Batched, seed: int, device="cpu"):
    """Raw draws for the batched scaled matmul.

    mxfp8: (a_vals, b_vals) standard-normal float32 [B, M|N, K] to be encoded
    to E4M3, and (a_exp, b_exp) int32 exponents uniform in [-6, 6] per
    32-block.  nvfp4: (a_bytes, b_bytes) uniform random bytes [B, M|N, K/2]
    (two E2M1 codes each) and (a_sv, b_sv) float32 scale values log-uniform in
    [2**-4, 2**4] per 16-block, to be encoded to E4M3."""
    if p.fmt == "mxfp8":
        a = randn((p.B, p.M, p.K), seed, S_A, device)
        b = randn((p.B, p.N, p.K), seed, S_B, device)
        ea = uniform_int((p.B, p.M, p.K // 32), -6, 6, seed, S_A_SCALE, device)
        eb = uniform_int((p.B, p.N, p.K // 32), -6, 6, seed, S_B_SCALE, device)
        return a, b, ea, eb
    if p.fmt == "nvfp4":
        a = random_bytes((p.B, p.M, p.K // 2), seed, S_A, device)
        b = random_bytes((p.B, p.N, p.K // 2), seed, S_B, device)
        sa = log_uniform((p.B, p.M, p.K // 16), -4, 4, seed, S_A_SCALE, device)
        sb = log_uniform((p.B, p.N, p.K // 16), -4, 4, seed, S_B_SCALE, device)
        return a, b, sa, sb
    if p.fmt == "mxfp4":  # E2M1 code bytes as for nvfp4, exponents as for mxfp8
        a = random_bytes((p.B, p.M, p.K // 2), seed, S_A, device)
        b = random_bytes((p.B, p.N, p.K // 2), seed, S_B, device)
        ea = uniform_int((p.B, p.M, p.K // 32), -6, 6, seed, S_A_SCALE, device)
        eb = uniform_int((p.B, p.N, p.K // 32), -6, 6, seed, S_B_SCALE, device)
        return a, b, ea, eb
    raise ValueError(p.fmt)


def backward_raw(p: Backward, seed: int, device="cpu"):
    """bfloat16 dY [M, N], W [N, K] (x0.02), X [M, K] (x0.02)."""
    dY = randn((p.M, p.N), seed, S_DY, device, torch.bfloat16)
    W = randn((p.N, p.K), seed, S_W, device, torch.bfloat16, scale=0.02)
    X = randn((p.M, p.K), seed, S_X, device, torch.bfloat16, scale=0.02)
    return dY, W, X


def _shape_tag(p) -> int:
    return (p.m * 31 + p.n * 7 + p.k) % 97
