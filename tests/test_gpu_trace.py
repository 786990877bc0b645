"""The continuous-batching trace on the GPU: 300 scheduler steps of Poisson
arrivals with log-normal prompts and geometric outputs, token budget 8192,
chunk size 512, max_num_seqs 256, a 16384-block pool (small enough that
recompute preemption triggers), Llama-3-8B head shapes in bf16.

Every step the C++ scheduler and the oracle scheduler are compared
bit-exactly (plan, preemptions, admissions, block tables, slot mapping), and
so is the whole host state with the step's reservation open and again after
its commit: free list, allocator statistics, every request's status and
counters, the tables of every request holding blocks, and the queues.  The
step's tokens go through reshape_and_cache and paged attention on the GPU, and every 10th step the attention output of every request is
compared with the float64 oracle over the request's own logical K/V
history.  K/V rows are a function of (request, position) only, so a
recomputed request rewrites identical values.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle.scheduler import NaiveScheduler, SchedConfig
from tests.gpu_support import compare
from tests.host_state import assert_same_state
from workloads import PooledRows, generate_arrivals, trace_spec

pytestmark = pytest.mark.gpu
# The base trace checks attention every 10th step (the float64 oracle over
# every request of every step would take far longer than the rest of the
# suite); the prefix and swap traces check every 20th step, plus every step
# in which a swapped request comes back.
CHECK_EVERY_BASE = 10
CHECK_EVERY = 20


def test_trace_300_steps():
    import paged_kv_cache_36_gb300 as pkv
    spec = trace_spec()
    H, Hkv, D, B = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    mbpr = spec.max_model_len // B
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, B, spec.num_blocks, mbpr)
    ref = NaiveScheduler(c, deep_checks=False)
    cpp = pkv.Scheduler(c.max_num_seqs, c.max_num_batched_tokens, c.chunk_size, c.max_model_len,
                        B, c.num_blocks, mbpr)
    kv_rows = PooledRows(Hkv * D, "trace_kv")
    q_rows = PooledRows(H * D, "trace_q")
    kc = torch.zeros(spec.num_blocks, B, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ws = pkv.new_workspace(spec.max_num_seqs, H, D)
    hist = {}          # rid -> (keys, values) of positions 0..len-1, host bf16
    by_step = {}
    for a in generate_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    checked = preemptions = 0
    for step in range(spec.steps):
        for a in by_step.get(step, []):
            assert cpp.add_request(a.req_id, a.prompt_len, a.max_output) == \
                ref.add_request(a.req_id, a.prompt_len, a.max_output)
        pc, pr = cpp.step(), ref.step()
        assert pc["entries"] == pr.entries and pc["preempted"] == pr.preempted
        assert pc["admitted"] == pr.admitted
        for rid in pr.preempted:
            hist.pop(rid, None)
            preemptions += 1
        bt, qsl, seq, nc, slots = cpp.metadata()
        rqsl, rseq, rnc, rrows, rslots = ref.metadata(pr)
        assert qsl.tolist() == rqsl and seq.tolist() == rseq and nc.tolist() == rnc
        assert slots.tolist() == rslots
        for k, row in enumerate(rrows):
            assert bt[k, :len(row)].tolist() == row
        assert_same_state(cpp, ref)
        T = int(qsl[-1])
        if T:
            rid_of = np.repeat([e[0] for e in pr.entries], [e[1] for e in pr.entries])
            pos = np.concatenate([np.arange(e[2], e[2] + e[1]) for e in pr.entries])
            kn = kv_rows.rows(0, rid_of, pos).view(T, Hkv, D)
            vn = kv_rows.rows(1, rid_of, pos).view(T, Hkv, D)
            q = q_rows.rows(2, np.full(T, step), np.arange(T)).view(T, H, D)
            at = 0
            for rid, s, ncb in pr.entries:
                if ncb == 0:
                    hist[rid] = (kn[at:at + s].clone(), vn[at:at + s].clone())
                else:
                    k0, v0 = hist[rid]
                    assert k0.shape[0] == ncb
                    hist[rid] = (torch.cat([k0, kn[at:at + s]]), torch.cat([v0, vn[at:at + s]]))
                at += s
            pkv.reshape_and_cache(kn.cuda(), vn.cuda(), kc, vc, torch.from_numpy(slots).cuda())
            out = pkv.paged_attention_varlen(
                q.cuda(), kc, vc, torch.from_numpy(bt).cuda(), torch.from_numpy(qsl).cuda(),
                torch.from_numpy(seq).cuda(), torch.from_numpy(nc).cuda(), 1.0 / math.sqrt(D),
                workspace=ws, max_query_len=pc["max_query_len"])
            if step % CHECK_EVERY_BASE == 0:
                histories = [hist[rid] for rid, _, _ in pr.entries]
                want = oa.paged_attention_varlen(q, histories, qsl, seq, nc, 1.0 / math.sqrt(D))
                compare(out, want, qsl, torch.bfloat16)
                assert pkv.read_error_word(ws) == 0
                checked += 1
        fin_c, fin_r = cpp.finish_step(True), ref.finish_step(True)
        assert fin_c == fin_r
        assert_same_state(cpp, ref)
        for rid in fin_r:
            hist.pop(rid, None)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) == 0
    assert preemptions > 0 and checked >= spec.steps // CHECK_EVERY_BASE - 1


def test_prefix_sharing_trace_300_steps():
    """The trace with shared system prompts (8 prompts, two namespaces): the
    schedulers match prompts against the prefix index, so requests read
    blocks another request wrote.  K/V rows are a function of the content
    that fixes them - (namespace, system prompt, position) inside a shared
    system prompt, (request, position) elsewhere - as a real model's would
    be.  Every CHECK_EVERY-th step up to 24 requests (those starting from a
    matched prefix first) are compared with the float64 oracle over their
    logical histories."""
    import paged_kv_cache_36_gb300 as pkv
    from workloads import generate_prefix_arrivals
    spec = trace_spec()
    H, Hkv, D, B = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    mbpr = spec.max_model_len // B
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, B, spec.num_blocks, mbpr)
    ref = NaiveScheduler(c, deep_checks=False)
    cpp = pkv.Scheduler(c.max_num_seqs, c.max_num_batched_tokens, c.chunk_size, c.max_model_len,
                        B, c.num_blocks, mbpr)
    kv_rows = PooledRows(Hkv * D, "prefix_kv")
    q_rows = PooledRows(H * D, "prefix_q")
    kc = torch.zeros(spec.num_blocks, B, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ws = pkv.new_workspace(spec.max_num_seqs, H, D)
    arrivals = generate_prefix_arrivals(spec)
    info = {a.req_id: a for a in arrivals}
    by_step = {}
    for a in arrivals:
        by_step.setdefault(a.step, []).append(a)

    def content(rid, pos):
        a = info[rid]
        key = np.full(len(pos), rid, dtype=np.int64)
        if a.system >= 0:
            key[pos < a.system_len] = (1 << 20) + a.namespace * 64 + a.system
        return key

    def history(rid, n):
        pos = np.arange(n)
        k = content(rid, pos)
        return kv_rows.rows(0, k, pos).view(n, Hkv, D), kv_rows.rows(1, k, pos).view(n, Hkv, D)

    checked = matched_reqs = 0
    for step in range(spec.steps):
        for a in by_step.get(step, []):
            assert cpp.add_request(a.req_id, a.prompt_len, a.max_output, a.namespace, a.tokens) == \
                ref.add_request(a.req_id, a.prompt_len, a.max_output, a.namespace, a.tokens)
        pc, pr = cpp.step(), ref.step()
        assert pc["entries"] == pr.entries and pc["preempted"] == pr.preempted
        assert pc["admitted"] == pr.admitted
        bt, qsl, seq, nc, slots = cpp.metadata()
        rqsl, rseq, rnc, rrows, rslots = ref.metadata(pr)
        assert qsl.tolist() == rqsl and seq.tolist() == rseq and nc.tolist() == rnc
        assert slots.tolist() == rslots
        for k, row in enumerate(rrows):
            assert bt[k, :len(row)].tolist() == row
        assert_same_state(cpp, ref, prefix=True)
        T = int(qsl[-1])
        if T:
            rid_of = np.repeat([e[0] for e in pr.entries], [e[1] for e in pr.entries])
            pos = np.concatenate([np.arange(e[2], e[2] + e[1]) for e in pr.entries])
            keys = np.concatenate([content(r, np.arange(e2, e2 + s)) for r, s, e2 in pr.entries])
            assert len(keys) == len(pos) == len(rid_of)
            kn = kv_rows.rows(0, keys, pos).view(T, Hkv, D)
            vn = kv_rows.rows(1, keys, pos).view(T, Hkv, D)
            q = q_rows.rows(2, np.full(T, step), np.arange(T)).view(T, H, D)
            pkv.reshape_and_cache(kn.cuda(), vn.cuda(), kc, vc, torch.from_numpy(slots).cuda())
            out = pkv.paged_attention_varlen(
                q.cuda(), kc, vc, torch.from_numpy(bt).cuda(), torch.from_numpy(qsl).cuda(),
                torch.from_numpy(seq).cuda(), torch.from_numpy(nc).cuda(), 1.0 / math.sqrt(D),
                workspace=ws, max_query_len=pc["max_query_len"])
            matched_reqs += sum(1 for r in pr.admitted if ref.reqs[r].num_computed > 0)
            if step % CHECK_EVERY == 0:
                R = len(pr.entries)
                order = sorted(range(R), key=lambda k: (pr.entries[k][2] == 0, k))
                pick = sorted(order[:24])
                histories = [history(pr.entries[k][0], int(seq[k])) if k in pick else None
                             for k in range(R)]
                want = oa.paged_attention_varlen(q, histories, qsl, seq, nc, 1.0 / math.sqrt(D),
                                                 rows=pick)
                compare(out, want, qsl, torch.bfloat16, rows=pick)
                assert pkv.read_error_word(ws) == 0
                checked += 1
        assert cpp.finish_step(True) == ref.finish_step(True)
        assert_same_state(cpp, ref, prefix=True)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) == 0
    st = cpp.allocator.prefix_stats()
    assert st["hits"] > 100 and matched_reqs > 50 and checked >= spec.steps // CHECK_EVERY - 1


def test_swap_preemption_trace_300_steps():
    """The trace with swap preemption: a 2048-block pool in pinned host
    memory receives the victims' blocks (copy_blocks, GPU -> host) and gives
    them back on swap-in (host -> GPU) before the step's kernels; swapped
    requests resume from their restored cache without recomputation, and
    attention over their histories is checked against the oracle."""
    import paged_kv_cache_36_gb300 as pkv
    spec = trace_spec()
    H, Hkv, D, B = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    mbpr = spec.max_model_len // B
    ncpu = 2048
    c = SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                    spec.max_model_len, B, spec.num_blocks, mbpr, preemption_mode="swap",
                    num_cpu_blocks=ncpu)
    ref = NaiveScheduler(c, deep_checks=False)
    cpp = pkv.Scheduler(c.max_num_seqs, c.max_num_batched_tokens, c.chunk_size, c.max_model_len,
                        B, c.num_blocks, mbpr, preemption_mode="swap", num_cpu_blocks=ncpu)
    kv_rows = PooledRows(Hkv * D, "swap_kv")
    q_rows = PooledRows(H * D, "swap_q")
    kc = torch.zeros(spec.num_blocks, B, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    hk = torch.zeros((ncpu, B, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    ws = pkv.new_workspace(spec.max_num_seqs, H, D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = {}
    by_step = {}
    for a in generate_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    checked = swaps_out = swaps_in = resumed_checked = 0
    for step in range(spec.steps):
        for a in by_step.get(step, []):
            assert cpp.add_request(a.req_id, a.prompt_len, a.max_output) == \
                ref.add_request(a.req_id, a.prompt_len, a.max_output)
        pc, pr = cpp.step(), ref.step()
        assert pc["entries"] == pr.entries and pc["preempted"] == pr.preempted
        assert pc["swap_out_pairs"] == pr.swap_out_pairs
        assert pc["swap_in_pairs"] == pr.swap_in_pairs
        for rid in pr.preempted:
            if rid not in pr.swapped_out:
                hist.pop(rid, None)            # recompute fallback: history restarts
        if pr.swap_out_pairs:
            pkv.copy_blocks(kc, vc, hk, hv, torch.tensor(pr.swap_out_pairs, dtype=torch.int32,
                                                         device="cuda"), error_word=err)
            swaps_out += len(pr.swapped_out)
        if pr.swap_in_pairs:
            pkv.copy_blocks(hk, hv, kc, vc, torch.tensor(pr.swap_in_pairs, dtype=torch.int32,
                                                         device="cuda"), error_word=err)
            swaps_in += len(pr.swapped_in)
        bt, qsl, seq, nc, slots = cpp.metadata()
        rqsl, rseq, rnc, rrows, rslots = ref.metadata(pr)
        assert qsl.tolist() == rqsl and seq.tolist() == rseq and nc.tolist() == rnc
        assert slots.tolist() == rslots
        for k, row in enumerate(rrows):
            assert bt[k, :len(row)].tolist() == row
        assert_same_state(cpp, ref, swap=True)
        T = int(qsl[-1])
        if T:
            rid_of = np.repeat([e[0] for e in pr.entries], [e[1] for e in pr.entries])
            pos = np.concatenate([np.arange(e[2], e[2] + e[1]) for e in pr.entries])
            kn = kv_rows.rows(0, rid_of, pos).view(T, Hkv, D)
            vn = kv_rows.rows(1, rid_of, pos).view(T, Hkv, D)
            q = q_rows.rows(2, np.full(T, step), np.arange(T)).view(T, H, D)
            at = 0
            for rid, s, ncb in pr.entries:
                if ncb == 0:
                    hist[rid] = (kn[at:at + s].clone(), vn[at:at + s].clone())
                else:
                    k0, v0 = hist[rid]
                    assert k0.shape[0] == ncb
                    hist[rid] = (torch.cat([k0, kn[at:at + s]]), torch.cat([v0, vn[at:at + s]]))
                at += s
            pkv.reshape_and_cache(kn.cuda(), vn.cuda(), kc, vc, torch.from_numpy(slots).cuda())
            out = pkv.paged_attention_varlen(
                q.cuda(), kc, vc, torch.from_numpy(bt).cuda(), torch.from_numpy(qsl).cuda(),
                torch.from_numpy(seq).cuda(), torch.from_numpy(nc).cuda(), 1.0 / math.sqrt(D),
                workspace=ws, max_query_len=pc["max_query_len"])
            if step % CHECK_EVERY == 0 or pr.swapped_in:
                rows = None
                if step % CHECK_EVERY != 0:   # just the requests restored in this step
                    rows = [k for k, e in enumerate(pr.entries) if e[0] in pr.swapped_in]
                    resumed_checked += len(rows)
                histories = [hist[rid] for rid, _, _ in pr.entries]
                want = oa.paged_attention_varlen(q, histories, qsl, seq, nc, 1.0 / math.sqrt(D),
                                                 rows=rows)
                compare(out, want, qsl, torch.bfloat16, rows=rows)
                assert pkv.read_error_word(ws) == 0
                checked += 1
        fin_c, fin_r = cpp.finish_step(True), ref.finish_step(True)
        assert fin_c == fin_r
        assert_same_state(cpp, ref, swap=True)
        for rid in fin_r:
            hist.pop(rid, None)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) == 0 and err.item() == 0
    assert swaps_out > 10 and swaps_in > 10 and resumed_checked > 10
