"""Slot addressing, cache scatter and block accounting, written from the pages.

Sources:
* "AI Infra入门干货总结：大模型是如何高效推理的", section "Paged Attention":
  the cache of one layer is [num_blocks, block_size, num_kv_heads, head_dim];
  block_table[r] lists request r's physical blocks; a token's slot is
  physical_block * block_size + offset_in_block, where the physical block is
  block_table[r][pos // block_size] and the offset is pos % block_size
  (worked example: [5, 8, 12], block_size 16, position 25 -> slot 137).
* "显存与调度" (ch. 32), section "从保留词元到物理块": kappa = 2 L n_kv d_head b_kv
  bytes per token; q_i = ceil(T_i / B); M_i = q_i B kappa; w_i = q_i B - T_i
  with 0 <= w_i < B; and the tail-waste program over lengths [37, 81, 130, 211].
* same page, section "分配是词元计划的一部分": the incremental demand
  delta_q_i = ceil((T_i + s_i) / B) - ceil(T_i / B).
* same page, section "只有数据路径划算时才移动 KV 状态": a transfer of S bytes
  over a path of measured bandwidth beta takes tau >= tau_fixed + S / beta.
* "Chunked Prefill 与 Preemption", section "可运行等价性与成本核算": a swap's
  payload round trip is at least 2 * cached_tokens * kv_bytes_per_token /
  bandwidth.
"""

from __future__ import annotations

import math


# -- slot rule ---------------------------------------------------------------
def slot_index(block_table_row, pos: int, block_size: int) -> int:
    """Slot of absolute position `pos` of a request whose physical blocks are
    `block_table_row` (logical block j -> physical block block_table_row[j])."""
    logical_block = pos // block_size
    physical_block = int(block_table_row[logical_block])
    offset = pos % block_size
    return physical_block * block_size + offset


def slot_mapping(block_table_rows, query_lens, num_computed, block_size: int) -> list[int]:
    """Slots of every token scheduled in a step, requests concatenated in order.

    Request r contributes query_lens[r] tokens at absolute positions
    num_computed[r], num_computed[r] + 1, ...
    """
    out = []
    for r, row in enumerate(block_table_rows):
        for i in range(int(query_lens[r])):
            out.append(slot_index(row, int(num_computed[r]) + i, block_size))
    return out


def write_cache(key_cache, value_cache, key, value, slots) -> None:
    """Naive scatter: token t's key/value rows go to cache[slot // B][slot % B].

    key/value are [T, num_kv_heads, head_dim]; caches are
    [num_blocks, block_size, num_kv_heads, head_dim] and are modified in place.
    A negative slot marks a padding token and is skipped.
    """
    block_size = key_cache.shape[1]
    for t, s in enumerate(slots):
        s = int(s)
        if s < 0:
            continue
        key_cache[s // block_size, s % block_size] = key[t]
        value_cache[s // block_size, s % block_size] = value[t]


# -- block accounting ----------------------------------------------------------
def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """kappa: logical K+V bytes one retained token needs across all layers."""
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem


def blocks_for(tokens: int, block_size: int) -> int:
    """q_i: blocks a request retaining `tokens` positions occupies."""
    return math.ceil(tokens / block_size)


def tail_waste(tokens: int, block_size: int) -> int:
    """w_i: unused token positions in the request's last block."""
    return blocks_for(tokens, block_size) * block_size - tokens


def allocated_bytes(tokens: int, block_size: int, kappa: int) -> int:
    """M_i^alloc: KV bytes allocated to the request."""
    return blocks_for(tokens, block_size) * block_size * kappa


def delta_blocks(held_tokens: int, new_tokens: int, block_size: int) -> int:
    """delta_q_i: blocks to add when a request holding `held_tokens` positions
    is planned `new_tokens` more."""
    return blocks_for(held_tokens + new_tokens, block_size) - blocks_for(held_tokens, block_size)


def tail_waste_table(lengths, block_sizes, declared_max: int):
    """Rows (B, block-table entries, allocated slots, tail waste) and the slots a
    contiguous allocator reserving each request's declared maximum would hold."""
    rows = []
    for b in block_sizes:
        entries = sum(blocks_for(n, b) for n in lengths)
        allocated = entries * b
        rows.append((b, entries, allocated, allocated - sum(lengths)))
    return rows, len(lengths) * declared_max


# -- moving KV state ------------------------------------------------------------
def transfer_lower_bound_s(payload_bytes: int, bandwidth_bytes_per_s: float,
                           fixed_s: float = 0.0) -> float:
    """tau_transfer >= tau_fixed + S / beta."""
    return fixed_s + payload_bytes / bandwidth_bytes_per_s


def swap_roundtrip_s(cached_tokens: int, kv_bytes_per_token: int,
                     bandwidth_bytes_per_s: float) -> float:
    """Payload-only lower bound of swapping a request out and back in."""
    payload = cached_tokens * kv_bytes_per_token
    return 2 * transfer_lower_bound_s(payload, bandwidth_bytes_per_s)
