"""The C++ host path (allocator, scheduler, metadata builder) against the
oracle's independent list-based implementations, compared bit-exactly after
every transition.  CPU only."""

import random

import numpy as np
import pytest

import paged_kv_cache_36_gb300 as pkv
from oracle import paging
from oracle.allocator import NaiveAllocator
from oracle.scheduler import NaiveScheduler, SchedConfig
from tests.host_state import assert_same_state
from workloads import generate_arrivals, generate_prefix_arrivals, trace_spec


def _same_alloc(cpp: pkv.Allocator, ref: NaiveAllocator, ids):
    assert cpp.free_list() == ref.free_list
    for r in ids:
        assert cpp.table(r) == ref.table(r)
        assert cpp.held_tokens(r) == ref.held_tokens(r)
    s, t = cpp.stats(), ref.stats()
    assert (s["capacity"], s["free"], s["reserved"], s["committed"], s["num_requests"],
            s["tail_waste"], s["alloc_failures"], s["peak_used"]) == \
        (t.capacity, t.free, t.reserved, t.committed, t.num_requests, t.tail_waste,
         t.alloc_failures, t.peak_used)
    cpp.check()


@pytest.mark.parametrize("seed", range(4))
def test_allocator_random_ops(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 4, 16])
    nb = rng.choice([8, 33, 100])
    cpp, ref = pkv.Allocator(nb, B, 64), NaiveAllocator(nb, B, 64)
    ids = list(range(10))
    for _ in range(600):
        op = rng.random()
        if op < 0.5:
            plan = [(r, rng.randint(0, 3 * B)) for r in rng.sample(ids, rng.randint(1, 4))]
            a, b = cpp.reserve(plan), ref.reserve(plan)
            assert a == b
            if a:
                if rng.random() < 0.3:      # cancel one planned request mid-step
                    r = rng.choice(plan)[0]
                    assert cpp.free_request(r) == ref.free_request(r)
                if rng.random() < 0.75:
                    cpp.commit(); ref.commit()
                else:
                    cpp.rollback(); ref.rollback()
        else:
            r = rng.choice(ids)
            assert cpp.free_request(r) == ref.free_request(r)
        _same_alloc(cpp, ref, ids)


def test_allocator_state_errors():
    a = pkv.Allocator(4, 4, 16)
    with pytest.raises(pkv.PkvError):
        a.commit()
    assert a.reserve([(0, 4)])
    with pytest.raises(pkv.PkvError):
        a.reserve([(1, 1)])
    a.rollback()
    with pytest.raises(pkv.PkvError):
        a.reserve([(0, 1), (0, 1)])
    assert not a.reserve([(0, 17)])          # 5 blocks from a pool of 4
    assert a.stats()["alloc_failures"] == 1
    b = pkv.Allocator(8, 4, 2)
    with pytest.raises(pkv.PkvError):
        b.reserve([(0, 9)])                  # 3 blocks > the 2-entry row


def test_slot_mapping_builder():
    # the worked example: [5, 8, 12], block_size 16, position 25 -> 137
    out = pkv.build_slot_mapping(np.array([[5, 8, 12]]), [0, 1], [25], 16)
    assert out.tolist() == [137]
    rng = random.Random(3)
    for _ in range(50):
        R = rng.randint(1, 6)
        B = rng.choice([1, 4, 16])
        qlens = [rng.randint(0, 9) for _ in range(R)]
        ncs = [rng.randint(0, 40) for _ in range(R)]
        width = max((nc + ql + B - 1) // B for nc, ql in zip(ncs, qlens)) + 1
        rows = [rng.sample(range(500), width) for _ in range(R)]
        qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
        got = pkv.build_slot_mapping(np.array(rows, np.int32), qsl, ncs, B)
        assert got.tolist() == paging.slot_mapping(rows, qlens, ncs, B)
    with pytest.raises(pkv.PkvError):
        pkv.build_slot_mapping(np.array([[1]]), [0, 1], [16], 16)   # position past the row


def _pair(c: SchedConfig):
    ref = NaiveScheduler(c, deep_checks=False)
    cpp = pkv.Scheduler(c.max_num_seqs, c.max_num_batched_tokens, c.chunk_size, c.max_model_len,
                        c.block_size, c.num_blocks, c.max_blocks_per_req,
                        c.artificial_preempt_prob, c.artificial_preempt_max, c.artificial_seed,
                        c.preemption_mode, c.num_cpu_blocks)
    return cpp, ref


def _compare_step(cpp, ref, arrivals_now, fail_step=False, swap=False, prefix=False):
    """One step of both schedulers: the plan, the step metadata, and the whole
    host state (allocator, requests, queues) with the reservation open and
    again after the commit or rollback."""
    for a in arrivals_now:
        if getattr(a, "tokens", ()):
            assert cpp.add_request(a.req_id, a.prompt_len, a.max_output, a.namespace, a.tokens) == \
                ref.add_request(a.req_id, a.prompt_len, a.max_output, a.namespace, a.tokens)
        else:
            assert cpp.add_request(a.req_id, a.prompt_len, a.max_output) == \
                ref.add_request(a.req_id, a.prompt_len, a.max_output)
    pc = cpp.step()
    pr = ref.step()
    assert pc["entries"] == pr.entries
    assert pc["preempted"] == pr.preempted
    assert pc["admitted"] == pr.admitted
    assert pc["swapped_out"] == pr.swapped_out and pc["swapped_in"] == pr.swapped_in
    assert pc["ignored"] == pr.ignored
    assert pc["swap_out_pairs"] == pr.swap_out_pairs and pc["swap_in_pairs"] == pr.swap_in_pairs
    bt, qsl, seq, nc, slots = cpp.metadata()
    rqsl, rseq, rnc, rrows, rslots = ref.metadata(pr)
    assert qsl.tolist() == rqsl and seq.tolist() == rseq and nc.tolist() == rnc
    assert slots.tolist() == rslots
    for k, row in enumerate(rrows):
        assert bt[k, :len(row)].tolist() == row and (bt[k, len(row):] == -1).all()
    assert_same_state(cpp, ref, swap, prefix)
    fin_c = cpp.finish_step(not fail_step)
    fin_r = ref.finish_step(not fail_step)
    assert fin_c == fin_r
    assert_same_state(cpp, ref, swap, prefix)
    return pc


def test_scheduler_trace_bit_exact():
    spec = trace_spec()
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, spec.block_size, spec.num_blocks,
                    spec.max_model_len // spec.block_size)
    cpp, ref = _pair(c)
    by_step = {}
    for a in generate_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    for step in range(spec.steps):
        _compare_step(cpp, ref, by_step.get(step, []))
    cnt = cpp.counters()
    assert cnt["preemptions"] == ref.total_preemptions > 0
    assert cnt["recomputed_tokens"] == ref.recomputed_tokens


@pytest.mark.parametrize("seed", range(3))
def test_scheduler_small_random_with_faults(seed):
    rng = random.Random(seed)
    c = SchedConfig(max_num_seqs=rng.choice([2, 4, 8]), max_num_batched_tokens=rng.choice([8, 20, 64]),
                    chunk_size=rng.choice([3, 8, 16]), max_model_len=200, block_size=4,
                    num_blocks=rng.choice([12, 24]), max_blocks_per_req=50,
                    artificial_preempt_prob=0.5, artificial_preempt_max=rng.choice([0, 5, 500]),
                    artificial_seed=seed)
    cpp, ref = _pair(c)
    rid = 0
    for step in range(200):
        arrivals = []
        for _ in range(rng.choice([0, 0, 1, 2])):
            arrivals.append(type("A", (), {"req_id": rid, "prompt_len": rng.randint(1, 30),
                                           "max_output": rng.randint(1, 12)})())
            rid += 1
        _compare_step(cpp, ref, arrivals, fail_step=rng.random() < 0.1)
    assert cpp.counters()["inject_left"] == ref.inject_left


def _same_prefix_alloc(cpp: pkv.Allocator, ref: NaiveAllocator, ids):
    _same_alloc(cpp, ref, ids)
    assert cpp.cached_list() == ref.cached
    assert cpp.pending_copies() == ref.pending_copies()
    assert cpp.available() == ref.available()
    p, q = cpp.prefix_stats(), ref.prefix_stats()
    assert (p["lookups"], p["hits"], p["matched_tokens"], p["evictions"], p["cow_copies"],
            p["indexed"], p["shared"], p["cached"]) == \
        (q.lookups, q.hits, q.matched_tokens, q.evictions, q.cow_copies, q.indexed, q.shared,
         len(ref.cached))
    for b in range(ref.capacity):
        assert cpp.ref_count(b) == ref.ref_count(b)


@pytest.mark.parametrize("seed", range(8))
def test_allocator_prefix_sharing_random_ops(seed):
    """Prefix matching, forks, copy-on-write, eviction and the base
    transitions, driven at random through both allocators."""
    rng = random.Random(100 + seed)
    B = rng.choice([2, 4, 16])
    nb = rng.choice([12, 40, 96])
    cpp, ref = pkv.Allocator(nb, B, 64), NaiveAllocator(nb, B, 64)
    bases = [[rng.randrange(4) for _ in range(6 * B)] for _ in range(3)]
    ids, live = [], []
    nxt = 0
    for _ in range(500):
        op = rng.random()
        if op < 0.25 and len(live) < 10:
            ns = rng.randrange(2)
            n = rng.randint(1, 6 * B)
            toks = rng.choice(bases)[:n] if rng.random() < 0.75 else \
                [rng.randrange(4) for _ in range(n)]
            assert cpp.peek_prefix(ns, toks) == (len(ref.peek_prefix(ns, toks)) * B,
                                                 sum(1 for b in ref.peek_prefix(ns, toks)
                                                     if b in ref.cached))
            assert cpp.match_prefix(nxt, ns, toks) == ref.match_prefix(nxt, ns, toks)
            ids.append(nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.65 and live:
            plan = [(r, rng.randint(0, 2 * B)) for r in rng.sample(live, rng.randint(1, min(4, len(live))))]
            a, b = cpp.reserve(plan), ref.reserve(plan)
            assert a == b
            if a:
                _same_prefix_alloc(cpp, ref, ids)
                if rng.random() < 0.2:      # cancel one planned request mid-step
                    r = rng.choice(plan)[0]
                    assert cpp.free_request(r) == ref.free_request(r)
                    live.remove(r)
                if rng.random() < 0.8:
                    cpp.commit(); ref.commit()
                else:
                    cpp.rollback(); ref.rollback()
        elif op < 0.75 and live:
            parent = rng.choice(live)
            if ref.tables.get(parent):
                cpp.fork(parent, nxt)
                ref.fork(parent, nxt)
                ids.append(nxt)
                live.append(nxt)
                nxt += 1
        elif live:
            r = rng.choice(live)
            assert cpp.free_request(r) == ref.free_request(r)
            live.remove(r)
        _same_prefix_alloc(cpp, ref, ids)


def test_scheduler_prefix_trace_bit_exact():
    """The 300-step trace with shared system prompts in two namespaces: the
    C++ scheduler and allocator against the oracle's, step by step, including
    the prefix index's statistics."""
    spec = trace_spec()
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, spec.block_size, spec.num_blocks,
                    spec.max_model_len // spec.block_size)
    cpp, ref = _pair(c)
    by_step = {}
    for a in generate_prefix_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    for step in range(spec.steps):
        _compare_step(cpp, ref, by_step.get(step, []), prefix=True)
        if step % 25 == 0:
            ref.alloc.deep_check()
    q = ref.alloc.prefix_stats()
    assert q.hits > 100 and q.matched_tokens > 100000     # sharing actually happens
    cnt = cpp.counters()
    assert cnt["preemptions"] == ref.total_preemptions
    assert cnt["recomputed_tokens"] == ref.recomputed_tokens


@pytest.mark.parametrize("seed", range(4))
def test_scheduler_swap_mode_small_random_with_faults(seed):
    rng = random.Random(50 + seed)
    c = SchedConfig(max_num_seqs=rng.choice([2, 4, 8]), max_num_batched_tokens=rng.choice([8, 20, 64]),
                    chunk_size=rng.choice([3, 8, 16]), max_model_len=200, block_size=4,
                    num_blocks=rng.choice([12, 24]), max_blocks_per_req=50,
                    artificial_preempt_prob=0.3, artificial_preempt_max=rng.choice([0, 20]),
                    artificial_seed=seed, preemption_mode="swap",
                    num_cpu_blocks=rng.choice([4, 16, 200]))
    cpp, ref = _pair(c)
    rid = 0
    swaps = blockless_victims = 0
    for step in range(250):
        arrivals = []
        for _ in range(rng.choice([0, 0, 1, 2])):
            arrivals.append(type("A", (), {"req_id": rid, "prompt_len": rng.randint(1, 30),
                                           "max_output": rng.randint(1, 12)})())
            rid += 1
        blockless = [r for r in ref.running if not ref.alloc.tables.get(r)]
        pc = _compare_step(cpp, ref, arrivals, fail_step=rng.random() < 0.1, swap=True)
        swaps += len(pc["swapped_out"])
        blockless_victims += sum(1 for r in pc["preempted"] if r in blockless)
    assert swaps > 0
    if seed == 0:
        # victims left without blocks by a rolled-back admission step occur here
        assert blockless_victims > 0
    assert cpp.counters()["recomputed_tokens"] == ref.recomputed_tokens


def test_scheduler_swap_mode_blockless_victim():
    """The swap-mode victim that holds no GPU block (left RUNNING with nothing
    by a rolled-back admission step): both schedulers preempt it by
    recompute, in the same step, with the same state afterwards."""
    from tests.test_oracle_swap import _blockless_victim_scenario
    c, reqs = _blockless_victim_scenario()
    cpp, ref = _pair(c)
    arrivals = [type("A", (), {"req_id": r, "prompt_len": n, "max_output": o})() for r, n, o in reqs]
    _compare_step(cpp, ref, arrivals, fail_step=True, swap=True)
    pc = _compare_step(cpp, ref, [], swap=True)
    assert pc["preempted"] == [1] and pc["swapped_out"] == []
    for _ in range(10):
        _compare_step(cpp, ref, [], swap=True)


def test_scheduler_trace_swap_mode_bit_exact():
    """The 300-step trace with swap preemption and a 4096-block CPU pool."""
    spec = trace_spec()
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, spec.block_size, spec.num_blocks,
                    spec.max_model_len // spec.block_size, preemption_mode="swap",
                    num_cpu_blocks=4096)
    cpp, ref = _pair(c)
    by_step = {}
    for a in generate_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    swaps = swapins = 0
    for step in range(spec.steps):
        pc = _compare_step(cpp, ref, by_step.get(step, []), swap=True)
        swaps += len(pc["swapped_out"])
        swapins += len(pc["swapped_in"])
    assert swaps > 10 and swapins > 10
    cnt = cpp.counters()
    assert cnt["preemptions"] == ref.total_preemptions
    assert cnt["recomputed_tokens"] == ref.recomputed_tokens


@pytest.mark.parametrize("seed", range(4))
def test_allocator_swap_random_ops(seed):
    rng = random.Random(200 + seed)
    B = rng.choice([2, 4])
    nb, ncpu = rng.choice([16, 40]), rng.choice([6, 30])
    cpp = pkv.Allocator(nb, B, 64, num_cpu_blocks=ncpu)
    ref = NaiveAllocator(nb, B, 64, num_cpu_blocks=ncpu)
    bases = [[rng.randrange(3) for _ in range(5 * B)] for _ in range(2)]
    live, swapped, ids = [], [], []
    nxt = 0
    for _ in range(400):
        op = rng.random()
        if op < 0.2 and len(live) < 8:
            toks = rng.choice(bases)[:rng.randint(1, 5 * B)]
            assert cpp.match_prefix(nxt, 0, toks) == ref.match_prefix(nxt, 0, toks)
            live.append(nxt); ids.append(nxt); nxt += 1
        elif op < 0.55 and live:
            plan = [(r, rng.randint(0, 2 * B)) for r in rng.sample(live, rng.randint(1, min(3, len(live))))]
            a, b = cpp.reserve(plan), ref.reserve(plan)
            assert a == b
            if a:
                if rng.random() < 0.8:
                    cpp.commit(); ref.commit()
                else:
                    cpp.rollback(); ref.rollback()
        elif op < 0.7 and live:
            r = rng.choice(live)
            if ref.tables.get(r):
                a, b = cpp.swap_out(r), ref.swap_out(r)
                assert a == b
                if a is not None:
                    live.remove(r); swapped.append(r)
        elif op < 0.85 and swapped:
            r = rng.choice(swapped)
            st = ref.swap_in_status(r)
            assert cpp.swap_in_status(r) == st
            assert cpp.swapped_blocks(r) == (ref.swapped[r][0], ref.swapped[r][1])
            if st == "ok":
                assert cpp.swap_in(r) == ref.swap_in(r)
                swapped.remove(r); live.append(r)
        elif live or swapped:
            r = rng.choice(live + swapped)
            assert cpp.free_request(r) == ref.free_request(r)
            (live if r in live else swapped).remove(r)
        _same_prefix_alloc(cpp, ref, ids)
        assert cpp.cpu_free_list() == ref.cpu_free
