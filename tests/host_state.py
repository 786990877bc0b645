"""Whole-state comparison of the C++ scheduler and allocator with the
oracle's, for use after every step of the trace tests (test plumbing).

What is compared: the free list and (swap mode) the CPU free list in order;
the allocator statistics (q_free, q_reserved, q_live, tail waste, failures,
peak) and, with a prefix index, its statistics and cached list; every known
request's status and counters and the block table and token count of every
request that holds blocks; the RUNNING, WAITING and SWAPPED queues in order;
the scheduler's counters; and the C++ allocator's own consistency check.
"""

from __future__ import annotations

STATUS = {"waiting": 0, "running": 1, "finished": 2, "swapped": 3, "finished_ignored": 4}


def assert_same_alloc_stats(cpp_alloc, ref_alloc):
    s, t = cpp_alloc.stats(), ref_alloc.stats()
    assert (s["capacity"], s["free"], s["reserved"], s["committed"], s["num_requests"],
            s["tail_waste"], s["alloc_failures"], s["peak_used"]) == \
        (t.capacity, t.free, t.reserved, t.committed, t.num_requests, t.tail_waste,
         t.alloc_failures, t.peak_used)


def assert_same_state(cpp, ref, swap: bool = False, prefix: bool = False):
    """cpp: paged_kv_cache_36_gb300.Scheduler; ref: oracle NaiveScheduler."""
    ca, ra = cpp.allocator, ref.alloc
    assert ca.free_list() == ra.free_list
    assert_same_alloc_stats(ca, ra)
    if swap:
        assert ca.cpu_free_list() == ra.cpu_free
        for rid, (blocks, tokens) in ra.swapped.items():
            assert ca.swapped_blocks(rid) == (blocks, tokens)
    if prefix:
        p, q = ca.prefix_stats(), ra.prefix_stats()
        assert (p["lookups"], p["hits"], p["matched_tokens"], p["evictions"], p["cow_copies"],
                p["indexed"], p["shared"], p["cached"]) == \
            (q.lookups, q.hits, q.matched_tokens, q.evictions, q.cow_copies, q.indexed,
             q.shared, len(ra.cached))
        assert ca.cached_list() == ra.cached
    for rid, r in ref.reqs.items():
        st = cpp.request(rid)
        assert st is not None, rid
        assert (st["status"], st["num_tokens"], st["num_computed"], st["outputs"],
                st["preemptions"]) == \
            (STATUS[r.status], r.num_tokens, r.num_computed, r.outputs, r.preemptions), rid
    for rid in ra.tables:
        assert ca.table(rid) == ra.table(rid), rid
        assert ca.held_tokens(rid) == ra.held_tokens(rid), rid
    run, wait = cpp.queues()
    assert run == ref.running and wait == ref.waiting
    assert cpp.swapped_queue() == ref.swapped
    cnt = cpp.counters()
    assert cnt["preemptions"] == ref.total_preemptions
    assert cnt["recomputed_tokens"] == ref.recomputed_tokens
    ca.check()
