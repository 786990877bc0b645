"""Naive continuous-batching scheduler with recompute preemption.

PARITY UNPINNED: no page prints a scheduler trace.  This policy is pinned by
hand-derived scenarios that follow the pages' preemption loop, by invariants,
and by bit-exact agreement with the independently written C++ scheduler.

Sources:
* "AI Infra入门干货总结：大模型是如何高效推理的", section "连续批处理": no
  prefill/decode distinction - each step schedules up to num_tokens -
  num_computed_tokens per request under four limits (max_num_seqs, the token
  budget, max_model_len, free KV blocks).  Appendix 4 ("附4：vLLM调度详细流程"):
  on a block shortfall the lowest-priority RUNNING request is preempted - all
  its KV freed, num_computed_tokens reset to 0, put back at the front of
  WAITING; no WAITING request is admitted in a step that preempted.
* "vLLM 抢占机制源码精读", sections "抢占的触发条件" and "_schedule_running 中
  的抢占循环": the RUNNING queue is FCFS with the head first; while the current
  request cannot get its slots, the tail of the queue is preempted; when no
  other request is left the current one preempts itself and the scan stops.
  "reset_state_for_recompute": the resumed prompt is prompt + outputs so far.
  "人工抢占测试": a test hook makes the slot check fail with probability 0.5,
  at most 500 times.
* "显存与调度", sections "分配是词元计划的一部分" (delta_q_i, feasibility,
  reserve/execute/commit) and "分块预填充共享每轮预算" (sum of decode and chunk
  tokens <= K per step).

Readings where the pages are silent (all stated in the design notes):
* s_i = min(num_tokens - num_computed, chunk_size, remaining budget); several
  prefills may share a step; partially prefilled requests stay in RUNNING.
* A request whose num_computed reaches num_tokens samples one output token:
  if that reaches its output target it finishes and frees its blocks,
  otherwise num_tokens grows by one.
* Victims come from the not-yet-scheduled tail, so the step's budget needs no
  adjustment; a self-preempted request's tokens were never counted.
* Admission (only in a step without preemption): WAITING head first, while
  RUNNING is below max_num_seqs, budget remains and its first chunk's blocks
  fit; the first request that does not fit ends admission.
* New blocks are reserved in plan order (scheduled RUNNING requests in queue
  order, then admitted ones) from the front of the FIFO free list.
* On a failed step the reservation is rolled back and no counter moves;
  admissions and preemptions already made stand.
* add_request clamps the output target to max_model_len - prompt_len and
  rejects a request whose largest footprint exceeds the pool or its block
  table, so no request can loop on self-preemption forever.

Prefix sharing ("显存与调度", sections "共享前缀会改变块的所有权" and "内存压力需要
明确策略"; "Chunked Prefill 与 Preemption": a prefix cache can let a
recomputed request hit part of its prefix):
* a request added with its prompt's token ids (and a namespace) is matched
  against the allocator's prefix index when it is admitted: it starts with
  the matched blocks and num_computed = the matched token count, and its
  full prompt blocks are indexed as they are committed;
* the blocks a step may take are q_free + q_cached (cached prefix blocks are
  evicted on demand); an admitted request's first chunk fits when its new
  blocks plus the cached blocks its match takes out of the cache fit; a
  preemption gives back the blocks no other request holds.

Swap preemption ("vLLM 抢占机制源码精读", sections "Swap 模式", "CPU swap 空间
不足时的处理" and "Swap-in 恢复流程"; "GPT-5 时代大模型推理调度系统深度实战",
section 4.3), with preemption_mode = "swap":
* a victim's blocks are swapped out (GPU -> CPU mapping for the transfer),
  it keeps num_computed and goes RUNNING -> SWAPPED, to the back of the
  swapped queue;
* in a step without preemption the swapped queue is served head first before
  any admission: "never" (more blocks than the pool) finishes the request as
  ignored, "later" or a lack of budget or seats stops the loop; otherwise
  the request is swapped in (CPU -> GPU mapping), becomes RUNNING at the back
  of the running queue and is scheduled in this step.

Readings where those sections are silent:
* when the CPU pool cannot take a victim, the victim is preempted by
  recompute instead (the page's engine aborts; its FIXME suggests failing
  only the request; recompute keeps the request alive);
* a victim that holds no GPU block is preempted by recompute: swap exists to
  keep computed KV blocks, and such a victim (left RUNNING with nothing by a
  rolled-back admission step) has none to keep and no computed token to
  lose;
* WAITING requests are admitted only once no request is left swapped, so
  swapped requests (older) are not overtaken;
* a swapped request's first chunk needs its swapped blocks plus the new
  blocks of s_i = min(num_tokens - num_computed, chunk_size, budget) tokens.
"""

from __future__ import annotations

from dataclasses import dataclass, field

from .allocator import NaiveAllocator
from .paging import blocks_for, delta_blocks

WAITING, RUNNING, FINISHED = "waiting", "running", "finished"
SWAPPED, FINISHED_IGNORED = "swapped", "finished_ignored"
_M64 = (1 << 64) - 1


def splitmix64_next(state: int) -> tuple[int, int]:
    """splitmix64 (Steele, Lea, Flood 2014): returns (new state, output)."""
    state = (state + 0x9E3779B97F4A7C15) & _M64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return state, z ^ (z >> 31)


@dataclass
class SchedConfig:
    max_num_seqs: int
    max_num_batched_tokens: int
    chunk_size: int
    max_model_len: int
    block_size: int
    num_blocks: int
    max_blocks_per_req: int
    artificial_preempt_prob: float = 0.0   # 0 disables the test hook
    artificial_preempt_max: int = 0
    artificial_seed: int = 0
    preemption_mode: str = "recompute"     # or "swap"
    num_cpu_blocks: int = 0                # the CPU pool for swapping


@dataclass
class Request:
    rid: int
    prompt_len: int
    max_output: int
    num_tokens: int
    num_computed: int = 0
    outputs: int = 0
    status: str = WAITING
    preemptions: int = 0
    namespace: int = 0
    tokens: list | None = None    # prompt token ids, for prefix sharing


@dataclass
class StepPlan:
    entries: list = field(default_factory=list)   # (rid, s, num_computed_before)
    preempted: list = field(default_factory=list)  # rids, in preemption order
    admitted: list = field(default_factory=list)   # rids admitted this step
    swapped_out: list = field(default_factory=list)   # victims that went to the CPU pool
    swapped_in: list = field(default_factory=list)    # rids brought back this step
    ignored: list = field(default_factory=list)       # rids finished as ignored
    swap_out_pairs: list = field(default_factory=list)  # (gpu block, cpu block)
    swap_in_pairs: list = field(default_factory=list)   # (cpu block, gpu block)


class NaiveScheduler:
    def __init__(self, cfg: SchedConfig, deep_checks: bool = True):
        self.cfg = cfg
        self.alloc = NaiveAllocator(cfg.num_blocks, cfg.block_size, cfg.max_blocks_per_req,
                                    deep=deep_checks, num_cpu_blocks=cfg.num_cpu_blocks)
        self.reqs: dict[int, Request] = {}
        self.waiting: list[int] = []
        self.running: list[int] = []
        self.swapped: list[int] = []
        self.plan: StepPlan | None = None
        self.rng_state = cfg.artificial_seed & _M64
        self.inject_left = cfg.artificial_preempt_max
        self.finished: list[int] = []
        self.total_preemptions = 0
        self.recomputed_tokens = 0
        self.swapped_out_blocks = 0

    # -- requests ------------------------------------------------------------------
    def add_request(self, rid: int, prompt_len: int, max_output: int, namespace: int = 0,
                    tokens=None) -> bool:
        c = self.cfg
        if rid in self.reqs or prompt_len < 1 or max_output < 1 or prompt_len >= c.max_model_len:
            return False
        if tokens is not None and len(tokens) != prompt_len:
            return False
        max_output = min(max_output, c.max_model_len - prompt_len)
        largest = blocks_for(prompt_len + max_output, c.block_size)
        if largest > c.num_blocks or largest > c.max_blocks_per_req:
            return False
        self.reqs[rid] = Request(rid, prompt_len, max_output, num_tokens=prompt_len,
                                 namespace=namespace,
                                 tokens=None if tokens is None else [int(t) for t in tokens])
        self.waiting.append(rid)
        return True

    # -- one step --------------------------------------------------------------------
    def _uniform(self) -> float:
        self.rng_state, z = splitmix64_next(self.rng_state)
        return (z >> 11) * (1.0 / (1 << 53))

    def _preempt(self, rid: int, plan: StepPlan) -> int:
        """Swap (if configured and the CPU pool has room) or recompute
        preemption; returns the blocks no request holds any more."""
        req = self.reqs[rid]
        if self.cfg.preemption_mode == "swap" and self.alloc.tables.get(rid):
            out = self.alloc.swap_out(rid)
            if out is not None:
                pairs, released = out
                req.status = SWAPPED
                req.preemptions += 1
                self.total_preemptions += 1
                self.swapped_out_blocks += len(pairs)
                self.running.remove(rid)
                self.swapped.append(rid)
                plan.preempted.append(rid)
                plan.swapped_out.append(rid)
                plan.swap_out_pairs += pairs
                return released
        self.recomputed_tokens += req.num_computed
        released = self.alloc.free_request(rid)
        req.num_computed = 0
        req.status = WAITING
        req.preemptions += 1
        self.total_preemptions += 1
        self.running.remove(rid)
        self.waiting.insert(0, rid)
        plan.preempted.append(rid)
        return released

    def step(self) -> StepPlan:
        if self.plan is not None:
            raise RuntimeError("previous step not finished")
        c = self.cfg
        B = c.block_size
        plan = StepPlan()
        budget = c.max_num_batched_tokens
        free = self.alloc.available()
        wanted = []   # (rid, s)

        # RUNNING, head first; victims come from the unscheduled tail
        i = 0
        while i < len(self.running):
            if budget == 0:
                break
            rid = self.running[i]
            req = self.reqs[rid]
            s = min(req.num_tokens - req.num_computed, c.chunk_size, budget)
            need = delta_blocks(self.alloc.held_tokens(rid), s, B)
            scheduled = True
            while True:
                fits = need <= free
                if c.artificial_preempt_prob > 0.0:
                    u = self._uniform()
                    if u < c.artificial_preempt_prob and self.inject_left > 0:
                        self.inject_left -= 1
                        fits = False
                if fits:
                    break
                if i + 1 < len(self.running):
                    free += self._preempt(self.running[-1], plan)
                else:
                    free += self._preempt(rid, plan)
                    scheduled = False
                    break
            if not scheduled:
                break
            wanted.append((rid, s))
            budget -= s
            free -= need
            i += 1

        # SWAPPED, head first, only in a step without preemption
        if not plan.preempted:
            while self.swapped and budget > 0 and len(self.running) < c.max_num_seqs:
                rid = self.swapped[0]
                req = self.reqs[rid]
                status = self.alloc.swap_in_status(rid)
                if status == "never":
                    self.swapped.pop(0)
                    self.alloc.free_request(rid)
                    req.status = FINISHED_IGNORED
                    plan.ignored.append(rid)
                    continue
                cpu_blocks, tokens = self.alloc.swapped[rid]
                s = min(req.num_tokens - req.num_computed, c.chunk_size, budget)
                need = len(cpu_blocks) + delta_blocks(tokens, s, B)
                if need > free:
                    break
                self.swapped.pop(0)
                plan.swap_in_pairs += self.alloc.swap_in(rid)
                req.status = RUNNING
                self.running.append(rid)
                plan.swapped_in.append(rid)
                wanted.append((rid, s))
                budget -= s
                free -= need

        # WAITING, only in a step without preemption and with nothing swapped
        if not plan.preempted and not self.swapped:
            while self.waiting and budget > 0 and len(self.running) < c.max_num_seqs:
                rid = self.waiting[0]
                req = self.reqs[rid]
                matched, from_cache = 0, 0
                prefix = req.tokens is not None and req.num_computed == 0
                if prefix:
                    blocks = self.alloc.peek_prefix(req.namespace, req.tokens)
                    matched = len(blocks) * B
                    from_cache = sum(1 for b in blocks if b in self.alloc.cached)
                s = min(req.num_tokens - max(req.num_computed, matched), c.chunk_size, budget)
                need = delta_blocks(max(self.alloc.held_tokens(rid), matched), s, B)
                if need + from_cache > free:
                    break
                if prefix:
                    req.num_computed = self.alloc.match_prefix(rid, req.namespace, req.tokens)
                self.waiting.pop(0)
                self.running.append(rid)
                req.status = RUNNING
                plan.admitted.append(rid)
                wanted.append((rid, s))
                budget -= s
                free -= need + from_cache

        for rid, s in wanted:
            plan.entries.append((rid, s, self.reqs[rid].num_computed))
        if not self.alloc.reserve(wanted):
            raise RuntimeError("plan does not fit although it was sized to fit")
        self.plan = plan
        return plan

    def finish_step(self, executed_ok: bool) -> list[int]:
        """Commit (or roll back) the open step.  Returns rids finished now."""
        if self.plan is None:
            raise RuntimeError("no open step")
        plan, self.plan = self.plan, None
        if not executed_ok:
            self.alloc.rollback()
            return []
        self.alloc.commit()
        done = []
        for rid, s, _ in plan.entries:
            req = self.reqs[rid]
            req.num_computed += s
            if req.num_computed == req.num_tokens:
                req.outputs += 1
                if req.outputs >= req.max_output:
                    self.alloc.free_request(rid)
                    req.status = FINISHED
                    self.running.remove(rid)
                    self.finished.append(rid)
                    done.append(rid)
                else:
                    req.num_tokens += 1
        return done

    # -- step metadata -----------------------------------------------------------------
    def metadata(self, plan: StepPlan):
        """Host arrays the kernels consume for the open step, requests in plan
        order: query_start_loc [R+1], seq_lens [R], num_computed [R], block table
        rows (committed + reserved blocks), slot_mapping [T]."""
        B = self.cfg.block_size
        qsl, seq_lens, ncs, rows, slots = [0], [], [], [], []
        for rid, s, nc in plan.entries:
            row = self.alloc.table(rid)
            qsl.append(qsl[-1] + s)
            seq_lens.append(nc + s)
            ncs.append(nc)
            rows.append(row)
            for k in range(s):
                p = nc + k
                slots.append(row[p // B] * B + p % B)
        return qsl, seq_lens, ncs, rows, slots
