"""Pins of the oracle allocator's prefix sharing ("显存与调度", section
"共享前缀会改变块的所有权", and the allocator tests listed in its section
"同时验证分配器与调度器").

What pins it, besides the conservation law checked after every transition:
* the two tests that section asks for: requests sharing a prefix and
  finishing in every order recycle the shared blocks only after the last
  reference; a different namespace (model version, adapter, position
  handling, modality or tenant) never hits;
* q_live equals the union of the request block sets, computed here from the
  tables directly;
* the matched length equals a brute-force search over every indexed prefix,
  rebuilt token by token from the index's parent links;
* hand-derived block ids for a small scenario (sharing, release, eviction of
  the oldest leaf);
* copy-on-write: the copying request gets a private block, the other holder
  keeps the original, rollback undoes it, and the last writer keeps it.
"""

import itertools
import random

import pytest

from oracle.allocator import NaiveAllocator


def _commit(a, plan):
    assert a.reserve(plan)
    a.commit()


def test_hand_derived_sharing_release_and_eviction():
    a = NaiveAllocator(8, 4)
    A = list(range(1, 11))                      # 10 tokens: blocks 0, 1 full, 2 partial
    assert a.match_prefix(0, 7, A) == 0
    _commit(a, [(0, 10)])
    assert a.table(0) == [0, 1, 2]
    assert len(a.index) == 2                    # only the two full prompt blocks
    Bp = list(range(1, 9)) + [99, 100]          # same first 8 tokens, then diverges
    assert a.match_prefix(1, 7, Bp) == 8
    assert a.table(1) == [0, 1]
    _commit(a, [(1, 2)])
    assert a.table(1) == [0, 1, 3]
    assert a.stats().committed == 4             # |{0,1,2} U {0,1,3}|
    assert a.ref_count(0) == 3 and a.ref_count(2) == 1
    assert a.free_request(0) == 1               # only block 2 is released
    assert a.free_list == [4, 5, 6, 7, 2]
    assert a.free_request(1) == 3
    assert a.free_list == [4, 5, 6, 7, 2, 3] and a.cached == [0, 1]
    assert a.ref_count(0) == 1 and a.ref_count(3) == 0
    # 7 blocks wanted, 6 free + 2 cached: the oldest leaf (block 1) is evicted
    assert a.match_prefix(2, 7, list(range(50, 78))) == 0
    assert a.reserve([(2, 28)])
    assert a.table(2) == [4, 5, 6, 7, 2, 3, 1]
    assert a.cached == [0] and len(a.index) == 1
    assert a.prefix_stats().evictions == 1
    a.rollback()                                # the eviction stands
    assert a.free_list == [4, 5, 6, 7, 2, 3, 1] and a.cached == [0]


@pytest.mark.parametrize("order", list(itertools.permutations(range(3))))
def test_shared_blocks_recycled_after_last_reference(order):
    """Three requests share a 3-block prefix and finish in every order."""
    B = 4
    a = NaiveAllocator(32, B)
    prefix = list(range(100, 112))              # 12 tokens = 3 full blocks
    prompts = [prefix + [r * 10 + k for k in range(5)] for r in range(3)]
    a.match_prefix(0, 1, prompts[0])
    _commit(a, [(0, len(prompts[0]))])
    shared = a.table(0)[:3]
    for r in (1, 2):
        assert a.match_prefix(r, 1, prompts[r]) == 12
        _commit(a, [(r, len(prompts[r]) - 12)])
        assert a.table(r)[:3] == shared
    for k, r in enumerate(order):
        a.free_request(r)
        live = 3 - k - 1
        for b in shared:
            assert a.ref_count(b) == live + 1   # the holders left plus the index
            assert b not in a.free_list
            assert (b in a.cached) == (live == 0)
    # recycled only when the index lets go too (eviction), never before
    big = 32 - len(a.free_list) - len(a.cached) + len(a.free_list) + 1
    a.match_prefix(9, 2, list(range(1000, 1000 + 4 * big)))
    assert a.reserve([(9, 4 * big)])            # needs every free block and one cached
    assert a.prefix_stats().evictions == 1


def test_namespace_and_token_divergence():
    B = 4
    a = NaiveAllocator(64, B)
    p = list(range(40))
    a.match_prefix(0, 5, p)
    _commit(a, [(0, 40)])
    assert a.match_prefix(1, 6, p) == 0         # same tokens, other namespace
    q = list(p)
    q[13] = -1                                  # diverges inside block 3
    assert a.match_prefix(2, 5, q) == 12
    q = list(p)
    q[0] = -1
    assert a.match_prefix(3, 5, q) == 0
    assert a.match_prefix(4, 5, p) == 36        # capped at len - 1 tokens: 9 blocks
    assert a.match_prefix(5, 5, p + [7]) == 40       # 41 tokens: all 10 blocks


def _indexed_prefixes(a):
    """Every indexed prefix, rebuilt from the parent links: (ns, tokens, blocks)."""
    out = []
    for b, key in a.key_of.items():
        chain, cur = [], b
        while cur != -1:
            chain.append(cur)
            cur = a.key_of[cur][1]
        chain.reverse()
        toks = []
        for c in chain:
            toks += list(a.key_of[c][2])
        out.append((key[0], toks, chain))
    return out


def _brute_match(a, ns, tokens):
    B = a.block_size
    cap = (len(tokens) - 1) // B
    best = []
    for pns, toks, chain in _indexed_prefixes(a):
        if pns == ns and len(chain) <= cap and toks == list(tokens[:len(toks)]):
            if len(chain) > len(best):
                best = chain
    return best


@pytest.mark.parametrize("seed", range(6))
def test_random_ops_against_brute_force(seed):
    rng = random.Random(seed)
    B = rng.choice([2, 4])
    a = NaiveAllocator(rng.choice([24, 40]), B)
    bases = [[rng.randrange(3) for _ in range(24)] for _ in range(3)]   # few, similar prompts
    live = {}
    nxt = 0
    for _ in range(400):
        op = rng.random()
        if op < 0.3 and len(live) < 8:
            ns = rng.randrange(2)
            base = rng.choice(bases)
            n = rng.randint(2, 24)
            toks = base[:n] if rng.random() < 0.7 else [rng.randrange(3) for _ in range(n)]
            want = _brute_match(a, ns, toks)
            got = a.match_prefix(nxt, ns, toks)
            assert got == len(want) * B and a.table(nxt) == want
            live[nxt] = len(toks)
            nxt += 1
        elif op < 0.7 and live:
            reqs = rng.sample(sorted(live), rng.randint(1, min(3, len(live))))
            plan = [(r, rng.randint(0, 2 * B)) for r in reqs]
            before = {r: a.table(r) for r in reqs}
            if a.reserve(plan):
                for r, s in plan:
                    t = a.table(r)
                    held = a.held_tokens(r)
                    # the blocks this step writes appear in no other request's
                    # table as this plan leaves it (full blocks are immutable,
                    # shared partial ones are copied first)
                    others = [a.table(o) for o in set(a.tables) | set(reqs) if o != r]
                    for p in range(held, held + s):
                        blk = t[p // B]
                        assert not any(blk in o for o in others)
                        assert blk not in a.key_of
                    assert t[:len(before[r]) - 1] == before[r][:-1] or not before[r]
                if rng.random() < 0.8:
                    a.commit()
                else:
                    a.rollback()
        elif op < 0.8 and live:
            parent = rng.choice(sorted(live))
            if parent in a.tables:
                a.fork(parent, nxt)
                live[nxt] = live[parent]
                nxt += 1
        elif live:
            r = rng.choice(sorted(live))
            a.free_request(r)
            del live[r]
        # the page's q_live: the union of the block sets
        union = set()
        for t in a.tables.values():
            union |= set(t)
        assert a.stats().committed == len(union) <= a.capacity


def test_copy_on_write_of_a_shared_partial_block():
    B = 4
    a = NaiveAllocator(16, B)
    _commit(a, [(0, 6)])                        # blocks 0 (full) and 1 (2 of 4 slots)
    a.fork(0, 1)
    assert a.table(1) == [0, 1] and a.ref_count(1) == 2
    assert a.reserve([(1, 1)])
    assert a.pending_copies() == [(1, 2)]
    assert a.table(1) == [0, 2] and a.table(0) == [0, 1]
    a.rollback()
    assert a.table(1) == [0, 1] and a.free_list[0] == 2
    assert a.reserve([(1, 2)])                  # fills block 2 to 8 tokens
    a.commit()
    assert a.table(1) == [0, 2] and a.ref_count(1) == 1 and a.ref_count(0) == 2
    # both holders write in one plan: the first copies, the last keeps block 1
    a.fork(0, 2)
    assert a.reserve([(2, 1), (0, 1)])
    assert a.pending_copies() == [(1, 3)]
    assert a.table(2) == [0, 3] and a.table(0) == [0, 1]
    a.commit()
    assert a.prefix_stats().cow_copies == 2
    # a full shared block is never copied: new tokens start a new block
    _commit(a, [(0, 1)])                        # block 1 now full (8 tokens)
    a.fork(0, 3)
    assert a.reserve([(3, 1)])
    assert a.pending_copies() == [] and a.table(3)[:2] == a.table(0)[:2]
    a.commit()


def test_recompute_after_release_hits_its_own_blocks():
    """A request released (as on a recompute preemption) and matched again
    gets back its full prompt blocks, if nothing evicted them."""
    B = 4
    a = NaiveAllocator(16, B)
    p = list(range(30))
    a.match_prefix(0, 0, p)
    _commit(a, [(0, 16)])
    _commit(a, [(0, 14)])
    t = a.table(0)
    a.free_request(0)
    assert a.match_prefix(0, 0, p) == 28
    assert a.table(0) == t[:7]
