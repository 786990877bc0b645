"""Naive list-based KV block allocator with reserve / execute / commit.

Sources:
* "显存与调度" (ch. 32), section "分配是词元计划的一部分" and Fig. 32.2: all
  new blocks of a plan are reserved atomically before execution; success
  commits mappings and token state; failure or cancellation rolls the
  uncommitted reservation back; q_free + q_reserved + q_committed = q_capacity
  holds after every transition; a referenced block is never handed out again.
* same page, "从保留词元到物理块": q_i = ceil(T_i / B), w_i = q_i B - T_i.
* "GPT-5 时代大模型推理调度系统深度实战", section 5.3 BlockManager: the free
  list is a vector of block ids; allocation drains from its front and freed
  blocks are pushed on its back.

Readings where the pages are silent:
* rollback puts the reserved blocks back at the front of the free list in
  their original order, so the free list is exactly what it was before the
  reserve;
* freeing a request appends its committed blocks to the back in block-table
  order; a request freed while a reservation is open also releases its
  reserved blocks (after its committed ones), and its entry leaves the plan.
"""

from __future__ import annotations

from dataclasses import dataclass

from .paging import blocks_for, delta_blocks


class AllocatorError(Exception):
    pass


@dataclass
class Stats:
    capacity: int
    free: int
    reserved: int
    committed: int
    num_requests: int        # requests holding at least one committed block
    tail_waste: int          # sum over requests of w_i for their committed tokens
    alloc_failures: int      # reserve calls refused for lack of blocks
    peak_used: int           # max over time of reserved + committed


class NaiveAllocator:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_req: int | None = None,
                 deep: bool = True):
        self.deep = deep
        self.capacity = num_blocks
        self.block_size = block_size
        self.max_blocks_per_req = max_blocks_per_req or num_blocks
        self.free_list: list[int] = list(range(num_blocks))
        self.tables: dict[int, list[int]] = {}   # committed blocks per request
        self.tokens: dict[int, int] = {}         # committed token count T_i
        self.pending: list | None = None         # [(req, s, [new blocks])] while reserved
        self.alloc_failures = 0
        self.peak_used = 0
        self.check()

    # -- queries ---------------------------------------------------------------
    def held_tokens(self, req: int) -> int:
        return self.tokens.get(req, 0)

    def table(self, req: int) -> list[int]:
        """Committed blocks followed by blocks reserved for the open plan."""
        out = list(self.tables.get(req, []))
        for r, _, new in self.pending or []:
            if r == req:
                out += new
        return out

    def num_free(self) -> int:
        return len(self.free_list)

    def stats(self) -> Stats:
        reserved = sum(len(n) for _, _, n in self.pending or [])
        committed = sum(len(t) for t in self.tables.values())
        waste = sum(len(self.tables[r]) * self.block_size - self.tokens[r] for r in self.tables)
        holding = sum(1 for t in self.tables.values() if t)
        return Stats(self.capacity, len(self.free_list), reserved, committed, holding,
                     waste, self.alloc_failures, self.peak_used)

    def check(self) -> None:
        """q_free + q_reserved + q_committed = q_capacity, and q_i = ceil(T_i / B)."""
        s = self.stats()
        if s.free + s.reserved + s.committed != s.capacity:
            raise AllocatorError("conservation violated")
        for r, t in self.tables.items():
            if len(t) != blocks_for(self.tokens[r], self.block_size):
                raise AllocatorError("q_i != ceil(T_i / B)")
        if self.deep:
            self.deep_check()

    def deep_check(self) -> None:
        """Every block id is in exactly one place: free, reserved or committed."""
        seen = list(self.free_list)
        for t in self.tables.values():
            seen += t
        for _, _, n in self.pending or []:
            seen += n
        if sorted(seen) != list(range(self.capacity)):
            raise AllocatorError("a block is lost or referenced twice")

    # -- transitions -------------------------------------------------------------
    def reserve(self, plan) -> bool:
        """plan: [(req, s_i)].  Reserves every new block or none.  Returns False
        (state unchanged) when sum of delta_q_i exceeds the free blocks."""
        if self.pending is not None:
            raise AllocatorError("a reservation is already open")
        reqs = [r for r, _ in plan]
        if len(set(reqs)) != len(reqs):
            raise AllocatorError("request listed twice in one plan")
        need = []
        for r, s in plan:
            if s < 0:
                raise AllocatorError("negative token count")
            held = self.held_tokens(r)
            d = delta_blocks(held, s, self.block_size)
            if blocks_for(held + s, self.block_size) > self.max_blocks_per_req:
                raise AllocatorError("block table capacity exceeded")
            need.append(d)
        if sum(need) > len(self.free_list):
            self.alloc_failures += 1
            return False
        pending = []
        for (r, s), d in zip(plan, need):
            new = []
            for _ in range(d):
                new.append(self.free_list.pop(0))
            pending.append((r, s, new))
        self.pending = pending
        used = self.capacity - len(self.free_list)
        self.peak_used = max(self.peak_used, used)
        self.check()
        return True

    def commit(self) -> None:
        if self.pending is None:
            raise AllocatorError("nothing reserved")
        for r, s, new in self.pending:
            self.tables.setdefault(r, [])
            self.tokens.setdefault(r, 0)
            self.tables[r] += new
            self.tokens[r] += s
        self.pending = None
        self.check()

    def rollback(self) -> None:
        if self.pending is None:
            raise AllocatorError("nothing reserved")
        back = []
        for _, _, new in self.pending:
            back += new
        self.free_list = back + self.free_list
        self.pending = None
        self.check()

    def free_request(self, req: int) -> int:
        """Release every block of `req` (committed, then any reserved ones).
        Returns the number of blocks released."""
        released = []
        if req in self.tables:
            released += self.tables.pop(req)
            self.tokens.pop(req)
        if self.pending is not None:
            keep = []
            for r, s, new in self.pending:
                if r == req:
                    released += new
                else:
                    keep.append((r, s, new))
            self.pending = keep
        self.free_list += released
        self.check()
        return len(released)
