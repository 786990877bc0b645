"""The five synthetic workloads of the paged-attention hot path.

Each builder returns plain host data: per-request lengths, physical block
placements and float tensors drawn by `generators`.  Nothing here computes a
slot, a block count or an attention value.

Shapes follow the pages' example model (Llama 3: 32 query heads, 8 KV heads,
head_dim 128; Llama-3-70B: 64 query heads, 8 KV heads), block_size 16, and
the cache layout [num_blocks, block_size, num_kv_heads, head_dim].

Draw order and seeds: every tensor has its own seed list (127, config name,
tensor name), so the order of draws does not matter.  Integers (context
lengths, block placement) and the N(0,1) query/key/value tensors are drawn from
separate seeded streams; bfloat16 tensors are the float32 draws rounded to
nearest-even.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from .generators import randn_fp32, random_block_placement, uniform_int

BLOCK_SIZE = 16


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class KVHistory:
    """Logical K/V of several requests, concatenated along the token axis.

    key[offsets[r] + p] is the key vector at absolute position p of request r;
    it is the request's own history in position order and never passes
    through the paged layout.
    """
    key: torch.Tensor          # [sum(lengths), num_kv_heads, head_dim]
    value: torch.Tensor        # same
    lengths: np.ndarray        # int64 [R]
    offsets: np.ndarray        # int64 [R]

    def k(self, r: int) -> torch.Tensor:
        o = int(self.offsets[r])
        return self.key[o:o + int(self.lengths[r])]

    def v(self, r: int) -> torch.Tensor:
        o = int(self.offsets[r])
        return self.value[o:o + int(self.lengths[r])]


def _history(name: str, lengths, hkv: int, d: int, dtype) -> KVHistory:
    lengths = np.asarray(lengths, dtype=np.int64)
    offsets = np.zeros_like(lengths)
    if len(lengths) > 1:
        offsets[1:] = np.cumsum(lengths)[:-1]
    n = int(lengths.sum())
    key = randn_fp32((n, hkv, d), name, "key_history", dtype=dtype)
    value = randn_fp32((n, hkv, d), name, "value_history", dtype=dtype)
    return KVHistory(key, value, lengths, offsets)


# ---------------------------------------------------------------------------
# tiny fp32 correctness case
# ---------------------------------------------------------------------------
@dataclass
class TinyCase:
    """Two requests with fixed block tables ([5,8,12] and [3,7]), 40 and 20
    tokens, block_size 16, 16 blocks, 4 query heads, 2 KV heads, head_dim 64.

    q[r] holds one query vector per position of request r, so a decode at
    position p reads q[r][p] and a prefill chunk [a, b) reads q[r][a:b].
    """
    block_tables: list
    num_tokens: list
    num_blocks: int
    block_size: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    q: list
    kv: KVHistory
    dtype: torch.dtype = torch.float32


def tiny_fp32_case(dtype=torch.float32) -> TinyCase:
    name = "tiny"
    h, hkv, d = 4, 2, 64
    num_tokens = [40, 20]
    q = [randn_fp32((n, h, d), name, "query", r, dtype=dtype) for r, n in enumerate(num_tokens)]
    kv = _history(name, num_tokens, hkv, d, dtype)
    return TinyCase([[5, 8, 12], [3, 7]], num_tokens, 16, BLOCK_SIZE, h, hkv, d, q, kv, dtype)


# ---------------------------------------------------------------------------
# configs 2 and 4: decode batches
# ---------------------------------------------------------------------------
@dataclass
class DecodeBatch:
    """R decode requests, one query token each.

    context[r] is the request's KV length after this step's write (its
    seq_len); the query sits at position context[r] - 1, and that position's
    key/value are the new token written this step.
    """
    name: str
    context: np.ndarray           # int64 [R]
    blocks: list                  # per request int32 physical block ids, in logical order
    num_blocks: int               # pool size
    num_heads: int
    num_kv_heads: int
    head_dim: int
    q: torch.Tensor               # [R, H, D]
    kv: KVHistory                 # lengths == context
    block_size: int = BLOCK_SIZE
    dtype: torch.dtype = torch.bfloat16


def _decode_batch(name, context, pool, h, hkv, d, dtype) -> DecodeBatch:
    counts = [_ceil_div(int(c), BLOCK_SIZE) for c in context]
    blocks = random_block_placement(pool, counts, name, "placement")
    q = randn_fp32((len(context), h, d), name, "query", dtype=dtype)
    kv = _history(name, context, hkv, d, dtype)
    return DecodeBatch(name, np.asarray(context, np.int64), blocks, pool, h, hkv, d, q, kv,
                       BLOCK_SIZE, dtype)


def decode_batch_llama8b(num_reqs: int = 64, ctx_lo: int = 128, ctx_hi: int = 4096,
                         pool: int = 65536, dtype=torch.bfloat16) -> DecodeBatch:
    """64 decodes, contexts uniform on [128, 4096], Llama-3-8B heads (32/8/128),
    block ids a random permutation of a 65536-block pool."""
    name = f"decode8b_{num_reqs}_{ctx_lo}_{ctx_hi}"
    context = uniform_int(ctx_lo, ctx_hi, num_reqs, name, "context")
    return _decode_batch(name, context, pool, 32, 8, 128, dtype)


def long_decode_llama70b(num_reqs: int = 8, context: int = 131072, pool: int = 1 << 20,
                         dtype=torch.bfloat16) -> DecodeBatch:
    """8 decodes with 131072-token contexts, Llama-3-70B heads (64/8/128),
    blocks scattered over a 2^20-block pool (2^20 x 64 KiB = 68.7 GB)."""
    name = f"decode70b_{num_reqs}_{context}"
    ctx = np.full(num_reqs, context, dtype=np.int64)
    return _decode_batch(name, ctx, pool, 64, 8, 128, dtype)


# ---------------------------------------------------------------------------
# mixed chunked-prefill step
# ---------------------------------------------------------------------------
@dataclass
class MixedStep:
    """Request 0 is a prefill chunk: query positions [chunk_start, chunk_end) of a
    longer prompt, with chunk_start tokens already computed.  Requests 1..R-1
    are decodes (one query at context-1).

    query_len[r] and num_computed[r] describe the step; seq_len = num_computed
    + query_len.  kv.lengths[r] == seq_len[r]: the last query_len positions are
    the tokens written this step.
    """
    name: str
    query_len: np.ndarray         # int64 [R]
    num_computed: np.ndarray      # int64 [R]
    blocks: list
    num_blocks: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    q: torch.Tensor               # [sum(query_len), H, D], requests in order
    kv: KVHistory
    block_size: int = BLOCK_SIZE
    dtype: torch.dtype = torch.bfloat16
    extra: dict = field(default_factory=dict)


def mixed_chunked_step(num_decodes: int = 256, chunk_start: int = 1536, chunk_end: int = 2048,
                       ctx_lo: int = 256, ctx_hi: int = 8192, pool: int = 131072,
                       h: int = 32, hkv: int = 8, d: int = 128,
                       dtype=torch.bfloat16) -> MixedStep:
    """One 512-token prefill chunk at [1536, 2048) plus 256 decodes with contexts
    uniform on [256, 8192]; Llama-3-8B heads; 131072-block pool, random placement."""
    name = f"mixed_{num_decodes}_{chunk_start}_{chunk_end}_{ctx_lo}_{ctx_hi}_{h}_{hkv}_{d}"
    ctx = uniform_int(ctx_lo, ctx_hi, num_decodes, name, "context")
    query_len = np.concatenate([[chunk_end - chunk_start], np.ones(num_decodes, np.int64)])
    num_computed = np.concatenate([[chunk_start], ctx - 1]).astype(np.int64)
    seq = num_computed + query_len
    counts = [_ceil_div(int(s), BLOCK_SIZE) for s in seq]
    blocks = random_block_placement(pool, counts, name, "placement")
    q = randn_fp32((int(query_len.sum()), h, d), name, "query", dtype=dtype)
    kv = _history(name, seq, hkv, d, dtype)
    return MixedStep(name, query_len.astype(np.int64), num_computed, blocks, pool, h, hkv, d,
                     q, kv, BLOCK_SIZE, dtype)


# ---------------------------------------------------------------------------
# continuous-batching trace parameters
# ---------------------------------------------------------------------------
@dataclass
class TraceSpec:
    steps: int = 300
    arrival_rate: float = 2.0          # Poisson arrivals per scheduler step
    prompt_median: int = 1024          # log-normal median
    prompt_sigma: float = 1.0
    prompt_max: int = 16384
    output_mean: int = 256             # geometric on {1, 2, ...}
    max_num_seqs: int = 256
    max_num_batched_tokens: int = 8192
    chunk_size: int = 512
    max_model_len: int = 32768
    block_size: int = BLOCK_SIZE
    num_blocks: int = 16384            # 262,144 token slots: below the live demand
    num_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    dtype: torch.dtype = torch.bfloat16


def trace_spec(**overrides) -> TraceSpec:
    return TraceSpec(**overrides)
