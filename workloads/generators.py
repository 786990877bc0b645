"""Seeded random draws used to build every synthetic input.

All normal draws are float32 N(0, 1) from numpy's PCG64 generator, seeded with
a list of integers that names the tensor (so every tensor is reproducible on
its own, independent of the order in which others are drawn).  Large tensors
are drawn in fixed-size chunks on a thread pool; each chunk has its own seed
list, so the result does not depend on the number of threads.

`CounterKV` is a counter-based generator: the key/value/query vector of
(request, position) is a pure function of its coordinates, so a request whose
cache was dropped and is later recomputed writes bit-identical values, as a
real model would.  It is splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) feeding the Box-Muller
transform.
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


# ---------------------------------------------------------------------------
# counter-based generator
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


class CounterKV:
    """Deterministic N(0,1) vectors indexed by (stream, request, position).

    stream is 0 for keys, 1 for values and 2 for queries.  `rows(stream, req,
    positions, width)` returns float32 [len(positions), width]; element
    (p, e) depends only on (seed, stream, req, p, e).
    """

    def __init__(self, seed: int = SEED):
        self.seed = np.uint64(seed)

    def rows(self, stream: int, req: int, positions, width: int) -> np.ndarray:
        pos = np.asarray(positions, dtype=np.uint64).reshape(-1, 1)
        half = (width + 1) // 2
        e = np.arange(half, dtype=np.uint64).reshape(1, -1)
        with np.errstate(over="ignore"):
            key = _splitmix64(self.seed ^ (np.uint64(stream) << np.uint64(56))
                              ^ (np.uint64(req) << np.uint64(32)))
            ctr = key + pos * np.uint64(1 << 20) + e
        bits = _splitmix64(ctr)
        # two 32-bit uniforms per 64-bit draw; u1 in (0, 1], u2 in [0, 1)
        u1 = ((bits >> np.uint64(32)).astype(np.float64) + 1.0) / 4294967296.0
        u2 = (bits & np.uint64(0xFFFFFFFF)).astype(np.float64) / 4294967296.0
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty((pos.shape[0], 2 * half), dtype=np.float64)
        z[:, 0::2] = r * np.cos(2.0 * np.pi * u2)
        z[:, 1::2] = r * np.sin(2.0 * np.pi * u2)
        return z[:, :width].astype(np.float32)
