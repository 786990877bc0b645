"""Pins of the oracle allocator against the reserve / execute / commit protocol
and the conservation law of "显存与调度" (ch. 32), and the allocator tests that
page lists under "同时验证分配器与调度器"."""

import random

import pytest

from oracle.allocator import AllocatorError, NaiveAllocator
from oracle.paging import blocks_for


def test_fresh_pool_fifo_order():
    a = NaiveAllocator(8, 4)
    assert a.reserve([(0, 5), (1, 4)])          # 2 blocks, then 1 block
    assert a.table(0) == [0, 1] and a.table(1) == [2]
    a.commit()
    assert a.free_list == [3, 4, 5, 6, 7]
    a.free_request(0)                            # freed blocks go to the back
    assert a.free_list == [3, 4, 5, 6, 7, 0, 1]
    assert a.reserve([(2, 1)]) and a.table(2) == [3]


def test_reserve_is_all_or_nothing():
    a = NaiveAllocator(4, 16)
    assert a.reserve([(0, 40)])                 # 3 blocks
    a.commit()
    before = list(a.free_list)
    assert not a.reserve([(1, 10), (2, 17)])     # needs 1 + 2 > 1 free
    assert a.free_list == before and a.pending is None
    assert a.stats().alloc_failures == 1


def test_rollback_restores_free_list_exactly():
    a = NaiveAllocator(10, 2)
    assert a.reserve([(0, 3)])
    a.commit()
    a.free_request(0)
    before = list(a.free_list)
    assert a.reserve([(1, 5), (2, 1)])
    a.rollback()
    assert a.free_list == before
    assert a.stats().reserved == 0 and a.stats().committed == 0


def test_cancel_between_reserve_and_commit():
    # "在预留与提交之间取消一个请求，确认所有已预留块都回到内存池"
    a = NaiveAllocator(12, 4)
    assert a.reserve([(0, 8), (1, 4)])
    a.commit()                                   # 0 holds 2 blocks, 1 holds 1
    # 0: 8 -> 12 tokens needs block 3; 1: 4 -> 13 needs 4, 5, 6; 2: 3 needs 7
    assert a.reserve([(0, 4), (1, 9), (2, 3)])
    assert a.table(1) == [2, 4, 5, 6]
    a.free_request(1)                            # cancelled mid-step
    s = a.stats()
    assert s.reserved == 2 and s.committed == 2
    a.commit()
    assert a.table(0) == [0, 1, 3] and a.table(2) == [7]
    # request 1's committed block, then its reserved ones, went to the back
    assert a.free_list == [8, 9, 10, 11, 2, 4, 5, 6]
    assert a.held_tokens(1) == 0


def test_injected_failure_rolls_back_only_uncommitted():
    # "注入执行与传输故障，确认已提交映射始终有效，未提交映射全部回滚"
    a = NaiveAllocator(16, 4)
    assert a.reserve([(0, 10), (1, 3)])
    a.commit()
    committed = {0: a.table(0), 1: a.table(1)}
    for _ in range(5):
        assert a.reserve([(0, 7), (1, 2), (5, 4)])
        a.rollback()                             # execution failed
        assert a.table(0) == committed[0] and a.table(1) == committed[1]
        assert a.held_tokens(0) == 10 and a.held_tokens(5) == 0


def test_exhaustion_is_reported_not_retried():
    a = NaiveAllocator(3, 4)
    assert a.reserve([(0, 12)])
    a.commit()
    for _ in range(3):
        assert not a.reserve([(1, 1)])
    assert a.stats().alloc_failures == 3


def test_state_errors():
    a = NaiveAllocator(3, 4)
    with pytest.raises(AllocatorError):
        a.commit()
    with pytest.raises(AllocatorError):
        a.rollback()
    assert a.reserve([(0, 1)])
    with pytest.raises(AllocatorError):
        a.reserve([(1, 1)])
    a.rollback()
    with pytest.raises(AllocatorError):
        a.reserve([(0, 1), (0, 2)])
    b = NaiveAllocator(10, 4, max_blocks_per_req=2)
    with pytest.raises(AllocatorError):
        b.reserve([(0, 9)])


def test_random_transitions_keep_invariants():
    rng = random.Random(127)
    B = 4
    a = NaiveAllocator(40, B)
    live = set()
    for _ in range(2000):
        op = rng.random()
        if op < 0.55:
            plan = [(r, rng.randint(0, 9)) for r in rng.sample(range(12), rng.randint(1, 4))]
            if a.reserve(plan):
                if rng.random() < 0.8:
                    a.commit()
                    live.update(r for r, _ in plan)
                else:
                    a.rollback()
        elif live:
            r = rng.choice(sorted(live))
            a.free_request(r)
            live.discard(r)
        s = a.stats()
        assert s.free + s.reserved + s.committed == s.capacity
        for r in live:
            t = a.held_tokens(r)
            w = blocks_for(t, B) * B - t
            assert len(a.table(r)) == blocks_for(t, B) and 0 <= w < B
    assert a.stats().peak_used <= 40


def test_growth_telescopes():
    a = NaiveAllocator(100, 16)
    for step in range(300):
        assert a.reserve([(0, 1)])
        a.commit()
        assert len(a.table(0)) == blocks_for(step + 1, 16)
