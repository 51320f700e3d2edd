"""Seeded synthetic inputs for the partial MXFP8 cast of master weights.

This module is shared by the CPU oracle side (tests) and the CUDA side (tests,
bench). It holds NO arithmetic of the method: it only draws numbers and lays
them out.  BF16 inputs are produced by truncating the low 16 bits of FP32 draws
(a generator choice; the method's own FP32->BF16 rounding is round-to-nearest
and lives separately in the oracle and in the kernels).

The workloads follow the five configurations of the distributed master-weight
cast ("Support row-only MXFP8 distributed master-weight casts", sections
"Changes" and "Bidirectional kernel performance"): the shapes of the timing
table (160x96 .. 16384x6144, FP32 and BF16), partial inputs that start at
offset 17 and hold a quarter of the matrix, fragment boundaries inside a
32-value block, an empty master shard and mixed row-only/bidirectional batches.

Every array is returned as a numpy array: FP32 data as ``float32``, BF16 data
as ``uint16`` bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"


def normal_f32(rng: np.random.Generator, shape, std: float = 0.02) -> np.ndarray:
    """N(0, std) draws as float32 (standard normals drawn in float32, then scaled)."""
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)


def truncate_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of ``x`` by dropping the low 16 mantissa bits (truncation)."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to float32 values."""
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Fragment:
    """A contiguous fragment ``[start, start+length)`` of a flattened rows x cols weight."""

    start: int
    length: int

    @property
    def end(self) -> int:
        return self.start + self.length


@dataclass
class Weight:
    """One weight: full master values (flattened row-major) and its direction set."""

    rows: int
    cols: int
    dtype: str
    data: np.ndarray  # flat, rows*cols elements (float32 or uint16 bf16 bits)
    colwise: bool = True
    fragments: list = field(default_factory=list)

    @property
    def numel(self) -> int:
        return self.rows * self.cols


def cfg1_tiny(seed: int = 0) -> Weight:
    """160x96 FP32 ~ N(0, 0.02), full fragment, bidirectional."""
    rng = np.random.default_rng(seed)
    x = normal_f32(rng, 160 * 96)
    return Weight(160, 96, F32, x, True, [Fragment(0, x.size)])


def cfg2_bf16_outliers(seed: int = 0) -> Weight:
    """1024x1024 BF16 ~ N(0, 0.02) with 0.1% of entries x100 and one all-zero 32x32 tile.

    Draw order: 1,048,576 FP32 normals; then ``rng.choice(n, 1049, replace=False)``
    outlier indices (multiplied by 100 in FP32); then the tile rows 32..63,
    cols 64..95 is set to zero (this makes all-zero 1x32 and 32x1 blocks inside
    the fragment); then truncation to BF16.  Fragment: start 17, a quarter of
    the elements.
    """
    rows = cols = 1024
    n = rows * cols
    rng = np.random.default_rng(seed)
    x = normal_f32(rng, n)
    idx = rng.choice(n, int(round(0.001 * n)), replace=False)
    x[idx] *= np.float32(100.0)
    x2 = x.reshape(rows, cols)
    x2[32:64, 64:96] = 0.0
    return Weight(rows, cols, BF16, truncate_to_bf16_bits(x), True, [Fragment(17, n // 4)])


def cfg3_square(seed: int = 0) -> Weight:
    """4096x4096 FP32 ~ N(0, 0.02); full fragment and the partial (17, n/4) with its complements."""
    rows = cols = 4096
    n = rows * cols
    rng = np.random.default_rng(seed)
    x = normal_f32(rng, n)
    q = n // 4
    frags = [Fragment(0, 17), Fragment(17, q), Fragment(17 + q, n - 17 - q)]
    return Weight(rows, cols, F32, x, True, frags)


def cfg4_headline(seed: int = 0, rows: int = 16384, cols: int = 6144) -> Weight:
    """16384x6144 FP32: per-row scale 10**U(-4, 1) times N(0, 0.02); full fragment.

    Draw order: ``rows`` uniforms for the row scales (float64), then the FP32
    normals; the product is taken in float32.
    """
    rng = np.random.default_rng(seed)
    row_scale = (10.0 ** rng.uniform(-4.0, 1.0, size=rows)).astype(np.float32)
    x = normal_f32(rng, (rows, cols))
    x *= row_scale[:, None]
    return Weight(rows, cols, F32, x.reshape(-1), True, [Fragment(0, rows * cols)])


@dataclass
class ShardedBatch:
    """A batch of weights concatenated into one flat master buffer, split into shards."""

    weights: list  # list[Weight]; .fragments unused
    offsets: list  # flat offset of each weight in the concatenated buffer
    bounds: list   # shard boundaries b0=0 < ... ; shard s = [bounds[s], bounds[s+1])
    flat: np.ndarray

    @property
    def total(self) -> int:
        return int(self.flat.size)

    def shard(self, s: int) -> np.ndarray:
        return self.flat[self.bounds[s]:self.bounds[s + 1]]

    def fragments(self, s: int):
        """(weight index, Fragment, offset of the fragment inside shard s) for every non-empty cut."""
        lo, hi = self.bounds[s], self.bounds[s + 1]
        out = []
        for w, (wt, off) in enumerate(zip(self.weights, self.offsets)):
            a, b = max(lo, off), min(hi, off + wt.numel)
            if a < b:
                out.append((w, Fragment(a - off, b - a), a - lo))
        return out


def cfg5_sharded_batch(seed: int = 0, scale: int = 1) -> ShardedBatch:
    """Mixed batch split into 4 emulated shards.

    Weights in order: W0 8192x8192 bidirectional, then W1..W6 alternating
    4096x4096 / 2048x8192, W1-W3 row-only and W4-W6 bidirectional, all FP32
    ~ N(0, 0.02).  ``scale`` > 1 divides every dimension by ``scale`` (small
    variant for quick tests; 32-value blocks stay whole).

    Shard boundaries: b1 = 32*k + r with k ~ U[n0/64, n0/32) and r ~ U[1, 31]
    (a boundary strictly inside a 32-value block of W0); b2 = b3 = 32*u with u
    ~ U[n0/32, total/32) (an empty shard inside W1..W6); b4 = total.
    """
    dims = [(8192, 8192, True), (4096, 4096, False), (2048, 8192, False), (4096, 4096, False),
            (2048, 8192, True), (4096, 4096, True), (2048, 8192, True)]
    dims = [(r // scale, c // scale, cw) for r, c, cw in dims]
    rng = np.random.default_rng(seed)
    weights, offsets, off = [], [], 0
    for r, c, cw in dims:
        weights.append(Weight(r, c, F32, None, cw))
        offsets.append(off)
        off += r * c
    total = off
    flat = normal_f32(rng, total)
    for wt, o in zip(weights, offsets):
        wt.data = flat[o:o + wt.numel]
    n0 = weights[0].numel
    k = int(rng.integers(n0 // 64, n0 // 32))
    r = int(rng.integers(1, 32))
    b1 = 32 * k + r
    u = int(rng.integers(n0 // 32, total // 32))
    b2 = 32 * u
    bounds = [0, b1, b2, b2, total]
    return ShardedBatch(weights, offsets, bounds, flat)


def cfg_by_name(name: str, seed: int = 0):
    return {"cfg1": cfg1_tiny, "cfg2": cfg2_bf16_outliers, "cfg3": cfg3_square,
            "cfg4": cfg4_headline, "cfg5": cfg5_sharded_batch}[name](seed)
