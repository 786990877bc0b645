"""Pins of the oracle scheduler.

No page prints a scheduler trace, so this policy's parity is unpinned by the
pages.  These tests pin it to hand-derived scenarios that follow the
preemption loop of "vLLM 抢占机制源码精读" (tail victims, self-preemption and
break) and the rules of "AI Infra入门干货总结" appendix 4 (free all KV, reset
num_computed_tokens, prepend to WAITING, no admission after a preemption), and
check the invariants of "显存与调度" on a long synthetic trace.
"""

import pytest

from oracle.scheduler import FINISHED, RUNNING, WAITING, NaiveScheduler, SchedConfig
from oracle.paging import blocks_for
from workloads import generate_arrivals, trace_spec


def cfg(**kw):
    base = dict(max_num_seqs=8, max_num_batched_tokens=100, chunk_size=100, max_model_len=1000,
                block_size=4, num_blocks=4, max_blocks_per_req=16)
    base.update(kw)
    return SchedConfig(**base)


def test_victim_is_the_tail_and_no_admission_after_preemption():
    s = NaiveScheduler(cfg(num_blocks=4))
    for r in range(3):
        assert s.add_request(r, 4, 10)
    p = s.step()                     # all three admitted, one block each
    assert p.entries == [(0, 4, 0), (1, 4, 0), (2, 4, 0)] and p.admitted == [0, 1, 2]
    assert [s.alloc.table(r) for r in range(3)] == [[0], [1], [2]]
    s.finish_step(True)              # each samples a token: 5 tokens, 4 computed
    # step 2: request 0 takes the last free block; request 1 finds none, so the
    # tail (request 2) is preempted, its block freed, and request 1 proceeds
    p = s.step()
    assert p.entries == [(0, 1, 4), (1, 1, 4)]
    assert p.preempted == [2] and p.admitted == []
    assert s.alloc.table(0) == [0, 3] and s.alloc.table(1) == [1, 2]
    r2 = s.reqs[2]
    assert (r2.status, r2.num_computed, r2.num_tokens, r2.preemptions) == (WAITING, 0, 5, 1)
    assert s.waiting == [2] and s.running == [0, 1]
    s.finish_step(True)
    # step 3: both fit in their second block; request 2 must recompute all 5
    # tokens (prompt + output so far) and needs 2 blocks, none free: deferred
    p = s.step()
    assert p.entries == [(0, 1, 5), (1, 1, 5)] and p.admitted == [] and p.preempted == []
    assert s.waiting == [2]


def test_self_preemption_stops_the_scan():
    s = NaiveScheduler(cfg(num_blocks=3))
    assert s.add_request(0, 4, 8) and s.add_request(1, 4, 8)
    s.step()
    s.finish_step(True)
    # request 0 takes the only free block; request 1 is the last in the queue
    # and has no victim behind it: it preempts itself
    p = s.step()
    assert p.entries == [(0, 1, 4)] and p.preempted == [1]
    assert s.running == [0] and s.waiting == [1]
    assert s.alloc.table(0) == [0, 2]          # block 1 went to the back of the free list
    assert s.alloc.free_list == [1]


def test_artificial_preemption_blocks_admission():
    s = NaiveScheduler(cfg(num_blocks=16, artificial_preempt_prob=1.0, artificial_preempt_max=1))
    for r in range(3):
        s.add_request(r, 4, 5)
    p = s.step()
    assert p.admitted == [0, 1, 2]
    s.finish_step(True)
    s.add_request(3, 4, 5)
    # the injected failure on request 0 preempts the tail (2); the step then
    # proceeds, and although blocks are plentiful nothing is admitted
    p = s.step()
    assert p.entries == [(0, 1, 4), (1, 1, 4)] and p.preempted == [2] and p.admitted == []
    assert s.waiting == [2, 3] and s.inject_left == 0
    s.finish_step(True)
    p = s.step()
    assert p.entries == [(0, 1, 5), (1, 1, 5), (2, 5, 0), (3, 4, 0)]
    assert p.admitted == [2, 3]


def test_chunking_and_token_budget():
    s = NaiveScheduler(cfg(block_size=16, num_blocks=100, max_num_batched_tokens=600,
                           chunk_size=512, max_blocks_per_req=100, max_model_len=4096))
    assert s.add_request(0, 1000, 2) and s.add_request(1, 300, 1)
    p = s.step()
    # 0: min(1000, 512, 600) = 512 (32 blocks); 1: min(300, 512, 88) = 88 (6)
    assert p.entries == [(0, 512, 0), (1, 88, 0)]
    assert len(s.alloc.table(0)) == 32 and len(s.alloc.table(1)) == 6
    s.finish_step(True)
    p = s.step()
    # 0: min(488, 512, 600) = 488 -> 1000 tokens, 63 blocks; 1: min(212, 512, 112) = 112
    assert p.entries == [(0, 488, 512), (1, 112, 88)]
    assert len(s.alloc.table(0)) == 63 and len(s.alloc.table(1)) == 13
    s.finish_step(True)
    assert s.reqs[0].num_tokens == 1001 and s.reqs[0].outputs == 1
    p = s.step()
    # 0 decodes one token (no new block); 1 finishes its prompt: 100 tokens, 6 blocks
    assert p.entries == [(0, 1, 1000), (1, 100, 200)]
    done = s.finish_step(True)
    assert done == [0, 1]
    assert s.alloc.num_free() == 100 and s.running == []


def test_output_accounting_and_finish():
    s = NaiveScheduler(cfg(num_blocks=8))
    s.add_request(7, 5, 3)
    plans = []
    while s.running or s.waiting:
        plans.append(s.step().entries)
        s.finish_step(True)
    # prefill of 5, then two decodes; the third output ends the request
    assert plans == [[(7, 5, 0)], [(7, 1, 5)], [(7, 1, 6)]]
    assert s.reqs[7].status == FINISHED and s.reqs[7].outputs == 3
    assert s.alloc.num_free() == 8


def test_max_num_seqs_and_rejections():
    s = NaiveScheduler(cfg(num_blocks=64, max_num_seqs=2, max_model_len=20))
    assert s.add_request(0, 4, 4) and s.add_request(1, 4, 4) and s.add_request(2, 4, 4)
    assert not s.add_request(2, 4, 4)         # duplicate id
    assert not s.add_request(3, 20, 1)        # prompt reaches max_model_len
    assert s.add_request(4, 18, 100)          # output clamped to 20 - 18
    assert s.reqs[4].max_output == 2
    p = s.step()
    assert p.admitted == [0, 1] and s.waiting == [2, 4]
    small = NaiveScheduler(cfg(num_blocks=2, max_model_len=100))
    assert not small.add_request(0, 6, 3)     # 9 tokens never fit in 2 blocks of 4


def test_failed_step_rolls_back():
    s = NaiveScheduler(cfg(num_blocks=8))
    s.add_request(0, 6, 4)
    s.step()
    s.finish_step(True)
    free_before = list(s.alloc.free_list)
    p = s.step()
    assert p.entries == [(0, 1, 6)]
    s.finish_step(False)                      # execution failed
    assert s.alloc.free_list == free_before
    assert s.reqs[0].num_computed == 6 and s.reqs[0].num_tokens == 7
    assert s.step().entries == [(0, 1, 6)]


def test_metadata_matches_tables():
    s = NaiveScheduler(cfg(num_blocks=32, block_size=4, chunk_size=6, max_num_batched_tokens=9))
    s.add_request(0, 10, 3)
    s.add_request(1, 3, 2)
    p = s.step()
    qsl, seq, ncs, rows, slots = s.metadata(p)
    assert p.entries == [(0, 6, 0), (1, 3, 0)]
    assert qsl == [0, 6, 9] and seq == [6, 3] and ncs == [0, 0]
    assert rows == [[0, 1], [2]]
    assert slots == [0, 1, 2, 3, 4, 5, 8, 9, 10]


def _run_trace(spec, steps=None, deep_every=25):
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, spec.block_size, spec.num_blocks,
                    max_blocks_per_req=spec.max_model_len // spec.block_size)
    s = NaiveScheduler(c, deep_checks=False)
    arrivals = generate_arrivals(spec)
    by_step = {}
    for a in arrivals:
        by_step.setdefault(a.step, []).append(a)
    stats = {"preempt_steps": 0, "tokens": 0}
    for step in range(steps or spec.steps):
        for a in by_step.get(step, []):
            s.add_request(a.req_id, a.prompt_len, a.max_output)
        p = s.step()
        total = sum(x for _, x, _ in p.entries)
        assert total <= spec.max_num_batched_tokens
        assert len(s.running) <= spec.max_num_seqs
        if p.preempted:
            stats["preempt_steps"] += 1
            assert p.admitted == []
        for rid, n, nc in p.entries:
            assert n >= 1 and n <= spec.chunk_size
            assert len(s.alloc.table(rid)) == blocks_for(nc + n, spec.block_size)
        qsl, seq, ncs, rows, slots = s.metadata(p)
        assert len(slots) == total == qsl[-1]
        assert len(set(slots)) == len(slots)
        st = s.alloc.stats()
        assert st.free + st.reserved + st.committed == st.capacity
        if step % deep_every == 0:
            s.alloc.deep_check()
        s.finish_step(True)
        stats["tokens"] += total
    return s, stats


def test_trace_invariants_and_preemption():
    spec = trace_spec()
    s, stats = _run_trace(spec)
    # the pool is sized so that recompute preemption triggers
    assert s.total_preemptions > 0 and stats["preempt_steps"] > 0
    assert s.recomputed_tokens > 0
    assert stats["tokens"] > 300 * 1000


def test_trace_terminates_when_arrivals_stop():
    spec = trace_spec(steps=40, num_blocks=2048)
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, spec.block_size, spec.num_blocks, 2048)
    s = NaiveScheduler(c, deep_checks=False)
    for a in generate_arrivals(spec):
        s.add_request(a.req_id, a.prompt_len, a.max_output)
    n = 0
    while s.running or s.waiting:
        s.step()
        s.finish_step(True)
        n += 1
        assert n < 100000
    assert all(r.status == FINISHED for r in s.reqs.values() if r.rid in s.finished)
    assert s.alloc.num_free() == 2048
