"""Seeded synthetic inputs for the tests and the benchmark.

This module is the only code the CPU oracle and the CUDA path both use: it
draws random numbers and converts them to 16-bit patterns, and holds none of
the method's arithmetic.  Recipes follow the workloads of "Fast Polynomial
Transcendentals for LLMs" (arXiv 2610.00049): the isolated FP16 sweep of
§4.2 / Table 3 (4,194,304 and 268,435,456 elements), the dense SwiGLU of
B1 and the routed-expert SwiGLU of B4 (§4.3, §5.2.4).

Generator: numpy PCG64 (``default_rng(seed)``), float32 draws, converted to
FP16 by numpy's round-to-nearest cast and to BF16 by torch's
round-to-nearest cast.  Deterministic on every platform.
"""
from __future__ import annotations

import numpy as np

SEED_X, SEED_DY, SEED_G, SEED_U = 0, 1, 2, 3

# sizes (elements)
N_L2 = 4_194_304            # L2-resident isolated sweep (8 MiB per FP16 tensor)
N_HBM = 268_435_456         # HBM-resident isolated sweep (512 MiB per FP16 tensor)
DENSE_ROWS, DENSE_COLS = 8192, 14336
RAGGED_TOKENS, RAGGED_TOPK, RAGGED_EXPERTS, RAGGED_COLS = 16_384, 8, 64, 2048
ZIPF_S = 1.1

CHUNK = 1 << 24


def to_bits(x32: np.ndarray, fmt: str) -> np.ndarray:
    """float32 -> FP16 / BF16 bit patterns (round to nearest even)."""
    if fmt == "f16":
        return x32.astype(np.float16).view(np.uint16)
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def normal(n: int, seed: int, scale: float, fmt: str) -> np.ndarray:
    """n draws of N(0, scale^2) as target-format bits, generated in chunks."""
    rng = np.random.default_rng(seed)
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, CHUNK):
        m = min(CHUNK, n - s)
        out[s:s + m] = to_bits(rng.standard_normal(m, dtype=np.float32) * np.float32(scale), fmt)
    return out


def normal_with_outliers(n: int, seed: int, scale: float, frac: float, lim: float,
                         fmt: str) -> np.ndarray:
    """N(0, scale^2) with a fraction ``frac`` of the elements replaced by
    U[-lim, lim] (the HBM-resident sweep: 1 % in [-40, 40]).  Draw order per
    chunk: normals, then the outlier mask, then the outlier values."""
    rng = np.random.default_rng(seed)
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, CHUNK):
        m = min(CHUNK, n - s)
        x = rng.standard_normal(m, dtype=np.float32) * np.float32(scale)
        mask = rng.random(m, dtype=np.float32) < frac
        x[mask] = rng.uniform(-lim, lim, int(mask.sum())).astype(np.float32)
        out[s:s + m] = to_bits(x, fmt)
    return out


def exhaustive() -> np.ndarray:
    """All 65,536 bit patterns, ascending."""
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def zipf_segment_counts(total: int = RAGGED_TOKENS * RAGGED_TOPK,
                        experts: int = RAGGED_EXPERTS, s: float = ZIPF_S,
                        cap: int = RAGGED_TOKENS) -> np.ndarray:
    """Rows per expert: Zipf(s) weights by rank, capped at ``cap`` (top-k
    routing sends a token to an expert at most once) with the excess
    re-spread proportionally over the uncapped experts, then rounded by
    largest remainder (ties to the lower index).  Sums to ``total``."""
    w = (np.arange(experts, dtype=np.float64) + 1.0) ** (-s)
    share = np.zeros(experts)
    free = np.ones(experts, dtype=bool)
    remaining = float(total)
    while True:
        share[free] = remaining * w[free] / w[free].sum()
        over = free & (share > cap)
        if not over.any():
            break
        share[over] = cap
        free &= ~over
        remaining = total - share[~free].sum()
    counts = np.floor(share).astype(np.int64)
    short = total - int(counts.sum())
    order = sorted(range(experts), key=lambda e: (-(share[e] - counts[e]), e))
    for e in order[:short]:
        counts[e] += 1
    return counts


def segment_offsets(counts: np.ndarray) -> np.ndarray:
    """int32 offsets [0, c0, c0+c1, ...] of length experts + 1."""
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


# ---- named workloads ------------------------------------------------------

def isolated_l2(fmt: str = "f16"):
    """x ~ N(0, 3^2) seed 0, dy ~ N(0, 1) seed 1; 4,194,304 elements."""
    return normal(N_L2, SEED_X, 3.0, fmt), normal(N_L2, SEED_DY, 1.0, fmt)


def isolated_hbm(fmt: str = "f16", n: int = N_HBM):
    """x ~ N(0, 3^2) with 1 % uniform in [-40, 40], seed 0; dy ~ N(0, 1) seed 1."""
    return (normal_with_outliers(n, SEED_X, 3.0, 0.01, 40.0, fmt),
            normal(n, SEED_DY, 1.0, fmt))


def dense_swiglu(fmt: str = "bf16", rows: int = DENSE_ROWS, cols: int = DENSE_COLS):
    """gate, up ~ 2 N(0, 1); dy ~ N(0, 1); [rows, cols] BF16."""
    n = rows * cols
    return (normal(n, SEED_G, 2.0, fmt).reshape(rows, cols),
            normal(n, SEED_U, 2.0, fmt).reshape(rows, cols),
            normal(n, SEED_DY, 1.0, fmt).reshape(rows, cols))


def ragged_swiglu(fmt: str = "bf16", cols: int = RAGGED_COLS):
    """16,384 tokens x top-8 over 64 experts, Zipf(1.1) segments summing to
    131,072 rows; gate, up ~ N(0, 1.5^2); dy ~ N(0, 1)."""
    counts = zipf_segment_counts()
    seg = segment_offsets(counts)
    rows = int(seg[-1])
    n = rows * cols
    return (normal(n, SEED_G, 1.5, fmt).reshape(rows, cols),
            normal(n, SEED_U, 1.5, fmt).reshape(rows, cols),
            normal(n, SEED_DY, 1.0, fmt).reshape(rows, cols), seg)
