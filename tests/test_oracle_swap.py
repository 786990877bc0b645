"""Pins of the oracle's swap preemption: the allocator's CPU pool and the
scheduler's swap mode ("vLLM 抢占机制源码精读", sections "Swap 模式" and "Swap-in
恢复流程"; "Chunked Prefill 与 Preemption", section "可运行等价性与成本核算").

What pins it:
* the swap round trip the page prints for its accounting example
  (7 tokens x 512 KiB over 24 GB/s -> about 0.306 ms);
* hand-derived block ids for a swap out and back in;
* can_swap_out / never / later as the page defines them;
* over random runs: a swapped request resumes where it stopped (nothing is
  recomputed), every logical block travels GPU -> CPU -> GPU in table order,
  both pools are conserved, and no request is admitted while one is swapped.
"""

import json
import os
import random

import pytest

from oracle import paging
from oracle.allocator import NaiveAllocator
from oracle.scheduler import FINISHED, SWAPPED, WAITING, NaiveScheduler, SchedConfig

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_swap_roundtrip_printed_on_the_page():
    g = json.load(open(os.path.join(GOLD, "preemption_accounting.json")))
    t = paging.swap_roundtrip_s(g["cached_tokens"], g["kv_bytes_per_token"],
                                g["bandwidth_gb_per_s"] * 1e9)
    assert round(t * 1e3, 3) == g["swap_roundtrip_ms_printed"]
    assert paging.blocks_for(g["cached_tokens"], g["block_size"]) == g["released_blocks"]
    # the bound grows with the fixed cost and the payload, linearly
    assert paging.transfer_lower_bound_s(10, 5.0, 1.0) == 3.0


def test_hand_derived_swap_out_and_in():
    a = NaiveAllocator(8, 4, num_cpu_blocks=4)
    assert a.reserve([(0, 10)])
    a.commit()
    assert a.table(0) == [0, 1, 2]
    pairs, released = a.swap_out(0)
    assert pairs == [(0, 0), (1, 1), (2, 2)] and released == 3
    assert a.free_list == [3, 4, 5, 6, 7, 0, 1, 2] and a.cpu_free == [3]
    assert a.table(0) == [] and a.swapped[0] == ([0, 1, 2], 10)
    assert a.swap_in_status(0) == "ok"
    assert a.swap_in(0) == [(0, 3), (1, 4), (2, 5)]
    assert a.table(0) == [3, 4, 5] and a.held_tokens(0) == 10
    assert a.cpu_free == [3, 0, 1, 2]


def test_cpu_pool_too_small_and_swap_in_statuses():
    a = NaiveAllocator(6, 4, num_cpu_blocks=2)
    assert a.reserve([(0, 12)])
    a.commit()
    before = (list(a.free_list), a.table(0), list(a.cpu_free))
    assert a.swap_out(0) is None                    # 3 blocks, 2 CPU blocks: can_swap_out fails
    assert (list(a.free_list), a.table(0), list(a.cpu_free)) == before
    b = NaiveAllocator(4, 4, num_cpu_blocks=8)
    assert b.reserve([(0, 8)])
    b.commit()
    b.swap_out(0)
    assert b.reserve([(1, 12)])                     # takes 3 of the 4 GPU blocks
    b.commit()
    assert b.swap_in_status(0) == "later"
    b.free_request(1)
    assert b.swap_in_status(0) == "ok"
    # "never": more blocks than the whole pool
    c = NaiveAllocator(4, 4, num_cpu_blocks=8)
    c.swapped[5] = ([0, 1, 2, 3, 4], 20)
    c.cpu_free = [x for x in c.cpu_free if x > 4]
    assert c.swap_in_status(5) == "never"


@pytest.mark.parametrize("seed", range(4))
def test_swap_mode_resumes_without_recompute(seed):
    rng = random.Random(seed)
    c = SchedConfig(max_num_seqs=6, max_num_batched_tokens=24, chunk_size=8, max_model_len=120,
                    block_size=4, num_blocks=rng.choice([12, 16]), max_blocks_per_req=40,
                    preemption_mode="swap", num_cpu_blocks=rng.choice([6, 40]))
    s = NaiveScheduler(c)
    where = {}                     # (rid, logical block) -> ("gpu"|"cpu", id)
    rid, swapped_any = 0, False
    for step in range(300):
        for _ in range(rng.choice([0, 0, 1])):
            s.add_request(rid, rng.randint(1, 30), rng.randint(1, 20))
            rid += 1
        before = {r: (q.num_computed, q.status) for r, q in s.reqs.items()}
        plan = s.step()
        # swapped victims keep num_computed; recomputed ones restart at 0
        for r in plan.swapped_out:
            assert s.reqs[r].status == SWAPPED and s.reqs[r].num_computed == before[r][0]
        by_req = {}
        at = 0
        for r in plan.swapped_out:
            n = len(s.alloc.swapped[r][0])
            by_req[r] = plan.swap_out_pairs[at:at + n]
            at += n
        assert at == len(plan.swap_out_pairs)
        for r, pairs in by_req.items():
            for j, (g, cpu) in enumerate(pairs):
                assert where.get((r, j), ("gpu", g)) == ("gpu", g)
                where[(r, j)] = ("cpu", cpu)
            swapped_any = True
        at = 0
        for r in plan.swapped_in:
            t = s.alloc.table(r)
            n = sum(1 for k in range(len(t)) if (r, k) in where and where[(r, k)][0] == "cpu")
            for j, (cpu, g) in enumerate(plan.swap_in_pairs[at:at + n]):
                assert where[(r, j)] == ("cpu", cpu) and t[j] == g
                where[(r, j)] = ("gpu", g)
            at += n
        assert at == len(plan.swap_in_pairs)
        if s.swapped:
            assert not plan.admitted            # swapped requests are not overtaken
        for r, sb, _ in plan.entries:
            for j, g in enumerate(s.alloc.table(r)):
                where[(r, j)] = ("gpu", g)
        s.finish_step(True)
        for r in list(where):
            if s.reqs[r[0]].status in (FINISHED, WAITING):
                del where[r]
    if c.num_cpu_blocks >= 40:
        assert s.recomputed_tokens == 0         # every preemption was a swap
    assert swapped_any and s.total_preemptions > 0


def _blockless_victim_scenario():
    """Two requests admitted in one step whose execution fails: the rollback
    leaves both RUNNING with no blocks (admissions stand).  In the next step
    one injected slot-check failure (the page's artificial-preemption hook)
    makes the head preempt the tail of RUNNING, which holds no GPU block."""
    c = SchedConfig(max_num_seqs=4, max_num_batched_tokens=64, chunk_size=64,
                    max_model_len=200, block_size=4, num_blocks=8, max_blocks_per_req=50,
                    artificial_preempt_prob=1.0, artificial_preempt_max=1,
                    preemption_mode="swap", num_cpu_blocks=8)
    return c, [(0, 4, 3), (1, 4, 3)]


def test_swap_mode_victim_without_blocks_is_recomputed():
    """A swap-mode victim that holds no GPU block has no KV cache to move to
    the CPU pool and no computed token to lose: it is preempted by recompute
    (back to the front of WAITING), not parked in the SWAPPED queue."""
    c, reqs = _blockless_victim_scenario()
    s = NaiveScheduler(c)
    for rid, n, out in reqs:
        assert s.add_request(rid, n, out)
    p1 = s.step()
    assert p1.admitted == [0, 1]
    s.finish_step(False)                          # rollback: both hold nothing
    assert s.running == [0, 1] and not s.alloc.tables.get(0) and not s.alloc.tables.get(1)
    p2 = s.step()
    assert p2.preempted == [1]
    assert p2.swapped_out == [] and p2.swap_out_pairs == []
    assert s.reqs[1].status == WAITING and s.waiting == [1] and s.swapped == []
    assert s.reqs[1].num_computed == 0 and s.recomputed_tokens == 0
    assert [e[0] for e in p2.entries] == [0]      # the head is scheduled after the preemption
    assert s.alloc.cpu_free == list(range(8))     # nothing went to the CPU pool
    s.finish_step(True)
    s.alloc.check()
