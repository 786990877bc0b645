"""Seeded random draws used to build every synthetic input.

All normal draws are float32 N(0, 1) from numpy's PCG64 generator, seeded with
a list of integers that names the tensor (so every tensor is reproducible on
its own, independent of the order in which others are drawn).  Large tensors
are drawn in fixed-size chunks on a thread pool; each chunk has its own seed
list, so the result does not depend on the number of threads.

`PooledRows` gives the key/value/query vector of (request, position) as a
pure function of its coordinates, so a request whose cache was dropped and is
later recomputed writes bit-identical values, as a real model would.  The
coordinates are hashed with splitmix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) into a seeded pool of
N(0,1) rows.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

SEED = 127
_CHUNK = 1 << 22  # elements per independently seeded chunk


def _seed_list(*parts) -> list[int]:
    out = []
    for p in parts:
        if isinstance(p, str):
            out.append(int.from_bytes(p.encode()[:8].ljust(8, b"\0"), "little"))
        else:
            out.append(int(p) & 0xFFFFFFFFFFFFFFFF)
    return out


def randn_fp32(shape, *name, dtype=torch.float32, threads: int | None = None) -> torch.Tensor:
    """N(0,1) float32 draws of `shape`, seeded by (SEED, *name), cast to `dtype`.

    The cast to bfloat16 (when asked) rounds each float32 draw to nearest-even.
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = torch.empty(n, dtype=dtype)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    seeds = _seed_list(SEED, *name)

    def fill(i: int) -> None:
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        rng = np.random.default_rng(seeds + [i])
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = torch.from_numpy(x).to(dtype)

    if nchunks <= 1:
        if n:
            fill(0)
    else:
        workers = threads or min(32, os.cpu_count() or 1)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.view(shape)


def uniform_int(lo: int, hi: int, n: int, *name) -> np.ndarray:
    """n integers uniform on the closed range [lo, hi], seeded by (SEED, *name)."""
    rng = np.random.default_rng(_seed_list(SEED, *name))
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64)


def random_block_placement(pool_blocks: int, counts, *name) -> list[np.ndarray]:
    """Scatter requests over a pool: a random permutation of 0..pool_blocks-1 is
    drawn and request r takes the next counts[r] entries, in request order."""
    counts = [int(c) for c in counts]
    total = sum(counts)
    if total > pool_blocks:
        raise ValueError(f"{total} blocks requested from a pool of {pool_blocks}")
    rng = np.random.default_rng(_seed_list(SEED, *name))
    if pool_blocks <= (1 << 24):
        perm = rng.permutation(pool_blocks)[:total]
    else:  # distinct ids without materialising a huge permutation
        perm = rng.choice(pool_blocks, size=total, replace=False)
    out, at = [], 0
    for c in counts:
        out.append(perm[at:at + c].astype(np.int32))
        at += c
    return out


def rope_cos_sin_table(max_position: int, rotary_dim: int, base: float = 500000.0) -> torch.Tensor:
    """A synthetic cos_sin_cache: float32 [max_position, rotary_dim], row p =
    [cos(p w_0) .. cos(p w_{n-1}), sin(p w_0) .. sin(p w_{n-1})] with
    n = rotary_dim / 2 and w_i = base^(-2i / rotary_dim) (the RoFormer angle
    schedule; base 500000 is Llama-3's).  Evaluated in float64, rounded once
    to float32.  Only the table's shape and row layout come from the pages;
    the angles are a plausible input, not part of the method.
    """
    half = rotary_dim // 2
    w = base ** (-2.0 * np.arange(half, dtype=np.float64) / rotary_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * w[None, :]
    return torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


# ---------------------------------------------------------------------------
# counter-hashed row pools
# ---------------------------------------------------------------------------
_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLD = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + _GOLD
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


class PooledRows:
    """Reproducible N(0,1) rows indexed by (stream, a, b), drawn from a pool.

    A pool of `pool_rows` rows of `width` float32 N(0,1) draws is generated
    once (seeded).  The row for (stream, a, b) - e.g. (key, request, position)
    - is pool[splitmix64(seed, stream, a, b) mod pool_rows], so the same
    coordinates always give the same row: a request whose cache was dropped
    and is recomputed writes bit-identical keys and values, as a real model
    would.  Lookups are a vectorised hash and a gather, fast enough for
    thousands of tokens per step.
    """

    def __init__(self, width: int, name: str, pool_rows: int = 1 << 16, dtype=torch.bfloat16):
        self.width = width
        self.pool = randn_fp32((pool_rows, width), name, "pool", dtype=dtype)
        self.n = pool_rows
        self.key = int(_splitmix64(np.array([_seed_list(SEED, name)[1]], dtype=np.uint64))[0])

    def index(self, stream: int, a, b) -> np.ndarray:
        a = np.asarray(a, dtype=np.uint64)
        b = np.asarray(b, dtype=np.uint64)
        with np.errstate(over="ignore"):
            x = (np.uint64(self.key) ^ (np.uint64(stream) << np.uint64(60))
                 ^ (a << np.uint64(32)) ^ b)
            h = _splitmix64(x)
        return (h % np.uint64(self.n)).astype(np.int64)

    def rows(self, stream: int, a, b) -> torch.Tensor:
        return self.pool[torch.from_numpy(self.index(stream, a, b))]
