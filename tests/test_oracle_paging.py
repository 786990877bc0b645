"""Pins of the oracle's slot rule, cache scatter and block accounting."""

import json
import math
import os
import random

import pytest
import torch

from oracle import paging

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_slot_worked_example():
    g = _gold("slot_worked_example.json")
    row, B, pos = g["block_table_row"], g["block_size"], g["position"]
    assert pos // B == g["logical_block"]
    assert row[pos // B] == g["physical_block"]
    assert pos % B == g["block_offset"]
    assert paging.slot_index(row, pos, B) == g["slot"] == 137


def test_block_table_example_is_a_mapping():
    # a request occupying 3 blocks can live in physical blocks 7, 2, 9
    row = _gold("block_table_example.json")["logical_to_physical"]
    B = 16
    slots = [paging.slot_index(row, p, B) for p in range(3 * B)]
    assert slots[:B] == list(range(7 * B, 8 * B))
    assert slots[B:2 * B] == list(range(2 * B, 3 * B))
    assert slots[2 * B:] == list(range(9 * B, 10 * B))


def test_slot_rule_brute_force():
    # enumerate the logical token sequence block by block and compare
    rng = random.Random(127)
    for _ in range(200):
        B = rng.choice([1, 2, 4, 8, 16, 32])
        nblocks = rng.randint(1, 12)
        row = rng.sample(range(64), nblocks)
        logical = []
        for b in row:
            logical += [b * B + o for o in range(B)]
        for pos in range(len(logical)):
            assert paging.slot_index(row, pos, B) == logical[pos]


def test_tiny_config_slots():
    # Request 0 holds 40 tokens in blocks [5, 8, 12]: its decode query is at
    # position 39 -> block 39 // 16 = 2 -> physical 12, offset 7 -> 12*16+7.
    # Request 1 holds 20 tokens in [3, 7]: position 19 -> block 1 -> 7*16+3.
    # A 7-token prefill of request 1 fills positions 0..6 of block 3: 48..54.
    assert paging.slot_index([5, 8, 12], 39, 16) == 199
    assert paging.slot_index([3, 7], 19, 16) == 115
    assert paging.slot_mapping([[3, 7]], [7], [0], 16) == list(range(48, 55))
    # the same prefill in chunks of 3 writes the same slots
    chunks = [paging.slot_mapping([[3, 7]], [b - a], [a], 16) for a, b in [(0, 3), (3, 6), (6, 7)]]
    assert sum(chunks, []) == list(range(48, 55))
    # a mixed step: request 0 decodes while request 1 runs chunk [3, 6)
    assert paging.slot_mapping([[5, 8, 12], [3, 7]], [1, 3], [39, 3], 16) == [199, 51, 52, 53]


def test_write_cache_against_flat_view():
    torch.manual_seed(0)
    NB, B, Hkv, D, T = 6, 4, 2, 8, 9
    kc = torch.zeros(NB, B, Hkv, D)
    vc = torch.zeros(NB, B, Hkv, D)
    key = torch.randn(T, Hkv, D)
    value = torch.randn(T, Hkv, D)
    slots = [3, 0, 23, -1, 7, 12, -5, 19, 1]
    paging.write_cache(kc, vc, key, value, slots)
    flat_k = kc.view(NB * B, Hkv, D)
    flat_v = vc.view(NB * B, Hkv, D)
    touched = set()
    for t, s in enumerate(slots):
        if s >= 0:
            assert torch.equal(flat_k[s], key[t]) and torch.equal(flat_v[s], value[t])
            touched.add(s)
    for s in range(NB * B):
        if s not in touched:
            assert not flat_k[s].any() and not flat_v[s].any()


def _simulate_blocks(length, B):
    """Append tokens one at a time; open a new block when the last is full."""
    blocks, used = 0, B
    for _ in range(length):
        if used == B:
            blocks += 1
            used = 0
        used += 1
    return blocks


def test_tail_waste_table():
    g = _gold("tail_waste_inputs.json")
    rows, contiguous = paging.tail_waste_table(g["lengths"], g["block_sizes"], g["declared_max"])
    total = sum(g["lengths"])                       # 37 + 81 + 130 + 211 = 459
    assert total == 459
    for B, entries, allocated, waste in rows:
        sim = sum(_simulate_blocks(n, B) for n in g["lengths"])
        assert entries == sim
        assert allocated == sim * B
        assert waste == sim * B - total
    # by hand: B=8 -> 5+11+17+27 = 60 entries; B=16 -> 3+6+9+14 = 32;
    # B=32 -> 2+3+5+7 = 17; B=64 -> 1+2+3+4 = 10
    assert rows == [(1, 459, 459, 0), (8, 60, 480, 21), (16, 32, 512, 53),
                    (32, 17, 544, 85), (64, 10, 640, 181)]
    assert contiguous == 4 * 256 == 1024
    # Fig. 32.1: a 32-block pool; contiguous mode reserves 8 blocks (256 slots
    # at B = 32) per request - the whole pool - while paged mode needs 17
    assert contiguous // 32 == 32 and rows[3][1] == 17


def test_w_invariant_and_block_count():
    for B in [1, 2, 4, 8, 16, 32, 64]:
        for n in range(1, 600):
            q = paging.blocks_for(n, B)
            w = paging.tail_waste(n, B)
            assert q == _simulate_blocks(n, B)
            assert 0 <= w < B
            assert paging.allocated_bytes(n, B, 4096) == q * B * 4096


def test_preemption_accounting_example():
    g = _gold("preemption_accounting.json")
    assert paging.blocks_for(g["cached_tokens"], g["block_size"]) == g["released_blocks"] == 2


def test_kappa():
    # one layer of Llama-3-8B in bf16: 2 * 8 KV heads * 128 * 2 bytes
    assert paging.kv_bytes_per_token(1, 8, 128, 2) == 4096
    # a 7B multi-head model (32 layers, 32 KV heads, 128 dims, bf16) gives the
    # 512 KiB per token that "Chunked Prefill 与 Preemption" uses in its example
    assert paging.kv_bytes_per_token(32, 32, 128, 2) == 512 * 1024


@pytest.mark.parametrize("B", [1, 4, 16, 32])
def test_delta_blocks_telescopes(B):
    rng = random.Random(B)
    for _ in range(50):
        held, total = 0, 0
        for _ in range(rng.randint(1, 30)):
            s = rng.randint(0, 3 * B)
            d = paging.delta_blocks(held, s, B)
            assert d >= 0
            total += d
            held += s
            assert total == math.ceil(held / B) == _simulate_blocks(held, B)


def test_tiny_config_alternative_readings():
    """The readings the tiny configuration also runs as extra tests: request 0
    with 40 cached tokens and its decode query at position 40 (slot 200), and
    request 1's last 7 of 20 tokens in chunks (13,16), (16,19), (19,20)."""
    assert paging.slot_index([5, 8, 12], 40, 16) == 12 * 16 + 8 == 200
    rows = [[3, 7]]
    got = [paging.slot_mapping(rows, [e - a], [a], 16) for a, e in [(13, 16), (16, 19), (19, 20)]]
    assert got == [[61, 62, 63], [112, 113, 114], [115]]
