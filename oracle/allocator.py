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

Prefix sharing ("显存与调度", section "共享前缀会改变块的所有权"):
* two requests may share a physical block only when their KV state is
  identical; the cache identity here is (namespace, every token of the prefix
  up to the block's end), where the namespace stands for model version,
  adapter, position handling, cache format, modality and tenant;
* q_live = |union of the requests' block sets| <= q_capacity: a shared block
  counts once;
* r_p counts every active request holding block p plus the prefix index if
  it retains p; a block is recycled only when r_p = 0;
* the prefix index maps compatible token prefixes to blocks and is searched
  for the longest reusable prefix; under memory pressure reusable leaf
  entries without an active owner are evicted (the RadixAttention remark);
* full shared blocks are immutable, a diverging suffix gets its own blocks,
  and a shared block that is still being written is copied first
  (copy-on-write).

Readings where that section is silent:
* the index is block-granular: an entry's key is (namespace, the block it
  extends or -1 at the root, its block_size token ids), so a key names the
  whole prefix exactly, with no hashing;
* only full blocks lying wholly inside a request's registered prompt are
  indexed, at the commit that completes them, and only while the request's
  previous block is itself the indexed one (a prefix computed twice
  concurrently keeps the first copy in the index; the second stays private);
* a match takes at most prompt_len - 1 tokens, so every request computes at
  least its last prompt token;
* a block held by no request but kept by the index is "cached": it sits in a
  list in release order and counts towards neither q_free nor q_live, so
  q_free + q_reserved + q_live + q_cached = q_capacity;
* eviction takes the oldest cached block that no indexed block extends,
  appends it to the back of the free list, and happens inside reserve(), only
  when the plan fits in q_free + q_cached but not in q_free; evictions stand
  after a rollback;
* fork(parent, child) gives the child the parent's committed blocks and token
  count (no prompt registration); when a request is planned new tokens while
  its last block is partial and held by another request too, reserve() takes
  one extra block, the plan's table shows it in place of the shared one, and
  the (source, destination) pair is listed for the device copy that must run
  before the step writes; commit drops the request's hold on the source.  In
  plan order, a request copies only while some other holder of the block has
  not already copied it away in the same plan: the last writer keeps the
  original.

Swapping ("vLLM 抢占机制源码精读", sections "Swap 模式" and "Swap-in 恢复流程";
"GPT-5 时代大模型推理调度系统深度实战", section 4.3):
* swap_out moves a request's KV blocks to a CPU block pool: it needs a free
  CPU block per GPU block (can_swap_out), returns the GPU -> CPU mapping for
  the data transfer, and releases the GPU blocks at once;
* swap_in is the reverse: GPU blocks for every CPU block, the CPU -> GPU
  mapping, and the CPU blocks are released; it is "never" possible when the
  request has more blocks than the GPU pool, "later" when they are not
  available now.

Readings where those sections are silent:
* the CPU pool is a FIFO free list like the GPU one (take from the front,
  release to the back, in block-table order);
* a swapped-out request's GPU blocks are released exactly as free_request
  would (indexed ones become cached) and its prompt registration is
  dropped; swap-in takes fresh, private GPU blocks in table order (evicting
  cached blocks as reserve() would) and restores T_i;
* swap_out and swap_in happen outside a plan (no reservation open) and stand
  whatever later happens to the step.
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
    cached: int = 0          # indexed blocks held by no request (q_cached)


@dataclass
class PrefixStats:
    lookups: int = 0         # match_prefix calls
    hits: int = 0            # calls that matched at least one block
    matched_tokens: int = 0  # tokens served from the index
    evictions: int = 0       # blocks evicted from the index
    cow_copies: int = 0      # copy-on-write block copies committed
    indexed: int = 0         # blocks in the index now
    shared: int = 0          # live blocks held by two or more requests now


class NaiveAllocator:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_req: int | None = None,
                 deep: bool = True, num_cpu_blocks: int = 0):
        self.deep = deep
        self.capacity = num_blocks
        self.block_size = block_size
        self.max_blocks_per_req = max_blocks_per_req or num_blocks
        self.free_list: list[int] = list(range(num_blocks))
        self.tables: dict[int, list[int]] = {}   # committed blocks per request
        self.tokens: dict[int, int] = {}         # committed token count T_i
        # while reserved: [(req, s, [new blocks], cow)], cow = (logical block, src, dst) or None
        self.pending: list | None = None
        self.alloc_failures = 0
        self.peak_used = 0
        # prefix sharing
        self.index: dict[tuple, int] = {}        # (namespace, parent block, tokens) -> block
        self.key_of: dict[int, tuple] = {}       # indexed block -> its key
        self.cached: list[int] = []              # indexed blocks no request holds, release order
        self.prompts: dict[int, tuple] = {}      # req -> (namespace, prompt tokens)
        self.indexed_upto: dict[int, int] = {}   # req -> prompt blocks already settled
        self.pfx = PrefixStats()
        # swapping
        self.cpu_capacity = num_cpu_blocks
        self.cpu_free: list[int] = list(range(num_cpu_blocks))
        self.swapped: dict[int, tuple[list[int], int]] = {}   # req -> (CPU blocks, T_i)
        self.check()

    # -- queries ---------------------------------------------------------------
    def held_tokens(self, req: int) -> int:
        return self.tokens.get(req, 0)

    def table(self, req: int) -> list[int]:
        """Committed blocks (with a copy-on-write destination in place of its
        source) followed by blocks reserved for the open plan."""
        out = list(self.tables.get(req, []))
        for r, _, new, cow in self.pending or []:
            if r == req:
                if cow is not None:
                    out[cow[0]] = cow[2]
                out += new
        return out

    def num_free(self) -> int:
        return len(self.free_list)

    def available(self) -> int:
        """Blocks a plan may take: free ones and cached ones (evictable)."""
        return len(self.free_list) + len(self.cached)

    def holders(self, b: int) -> int:
        """How many requests hold block b in their committed tables."""
        return sum(1 for t in self.tables.values() if b in t)

    def ref_count(self, b: int) -> int:
        """r_p: requests holding b, plus one if the prefix index retains it."""
        return self.holders(b) + (1 if b in self.key_of else 0)

    def live_blocks(self) -> set:
        out = set()
        for t in self.tables.values():
            out |= set(t)
        return out

    def pending_copies(self) -> list[tuple[int, int]]:
        """(source, destination) of every copy-on-write in the open plan."""
        return [(c[1], c[2]) for _, _, _, c in self.pending or [] if c is not None]

    def stats(self) -> Stats:
        reserved = sum(len(n) + (1 if c is not None else 0) for _, _, n, c in self.pending or [])
        committed = len(self.live_blocks())   # q_live: the union, shared blocks once
        waste = sum(len(self.tables[r]) * self.block_size - self.tokens[r] for r in self.tables)
        holding = sum(1 for t in self.tables.values() if t)
        return Stats(self.capacity, len(self.free_list), reserved, committed, holding,
                     waste, self.alloc_failures, self.peak_used, len(self.cached))

    def prefix_stats(self) -> PrefixStats:
        p = PrefixStats(**vars(self.pfx))
        p.indexed = len(self.index)
        count: dict[int, int] = {}
        for t in self.tables.values():
            for b in t:
                count[b] = count.get(b, 0) + 1
        p.shared = sum(1 for c in count.values() if c >= 2)
        return p

    def check(self) -> None:
        """q_free + q_reserved + q_live + q_cached = q_capacity, and q_i = ceil(T_i / B)."""
        s = self.stats()
        if s.free + s.reserved + s.committed + s.cached != s.capacity:
            raise AllocatorError("conservation violated")
        if len(self.cpu_free) + sum(len(c) for c, _ in self.swapped.values()) != self.cpu_capacity:
            raise AllocatorError("CPU pool conservation violated")
        for r, (c, t) in self.swapped.items():
            if r in self.tables or len(c) != blocks_for(t, self.block_size):
                raise AllocatorError("a swapped request is inconsistent")
        for r, t in self.tables.items():
            if len(t) != blocks_for(self.tokens[r], self.block_size):
                raise AllocatorError("q_i != ceil(T_i / B)")
        if self.deep:
            self.deep_check()

    def deep_check(self) -> None:
        """Every block id is in exactly one place (free, cached, reserved or
        live), a request holds a block at most once, and the index is a tree of
        live or cached blocks."""
        live = self.live_blocks()
        for t in self.tables.values():
            if len(set(t)) != len(t):
                raise AllocatorError("a request holds a block twice")
        seen = list(self.free_list) + list(live) + list(self.cached)
        for _, _, n, c in self.pending or []:
            seen += n + ([c[2]] if c is not None else [])
        if sorted(seen) != list(range(self.capacity)):
            raise AllocatorError("a block is lost or referenced twice")
        for b in self.cached:
            if b not in self.key_of or b in live:
                raise AllocatorError("a cached block is unindexed or held")
        for key, b in self.index.items():
            if self.key_of.get(b) != key or not (b in live or b in self.cached):
                raise AllocatorError("index and blocks disagree")
            if key[1] != -1 and key[1] not in self.key_of:
                raise AllocatorError("an indexed block extends an unindexed one")

    # -- prefix index ------------------------------------------------------------
    def peek_prefix(self, namespace: int, tokens) -> list[int]:
        """Blocks of the longest indexed prefix of `tokens` in `namespace`,
        at most len(tokens) - 1 tokens long.  No side effects."""
        B = self.block_size
        out, parent = [], -1
        for j in range((len(tokens) - 1) // B):
            b = self.index.get((namespace, parent, tuple(tokens[j * B:(j + 1) * B])))
            if b is None:
                break
            out.append(b)
            parent = b
        return out

    def match_prefix(self, req: int, namespace: int, tokens) -> int:
        """Registers req's prompt and gives it the longest indexed prefix.
        req must hold nothing yet.  Returns the matched token count."""
        if self.pending is not None:
            raise AllocatorError("match_prefix while a reservation is open")
        if self.tables.get(req) or req in self.prompts:
            raise AllocatorError("match_prefix on a request that already holds blocks")
        blocks = self.peek_prefix(namespace, tokens)
        self.pfx.lookups += 1
        if blocks:
            self.pfx.hits += 1
            self.pfx.matched_tokens += len(blocks) * self.block_size
            for b in blocks:
                if b in self.cached:
                    self.cached.remove(b)
            self.tables[req] = list(blocks)
            self.tokens[req] = len(blocks) * self.block_size
        self.prompts[req] = (namespace, list(tokens))
        self.indexed_upto[req] = len(blocks)
        self.check()
        return len(blocks) * self.block_size

    def _index_prompt_blocks(self, req: int) -> None:
        if req not in self.prompts:
            return
        ns, toks = self.prompts[req]
        B = self.block_size
        full = min(self.tokens.get(req, 0), len(toks)) // B
        j = self.indexed_upto[req]
        while j < full:
            b = self.tables[req][j]
            parent = -1 if j == 0 else self.tables[req][j - 1]
            key = (ns, parent, tuple(toks[j * B:(j + 1) * B]))
            if (parent != -1 and parent not in self.key_of) or key in self.index:
                j = len(toks) // B + 1   # the chain is someone else's: stop for good
                break
            self.index[key] = b
            self.key_of[b] = key
            j += 1
        self.indexed_upto[req] = j

    def _release(self, b: int) -> None:
        """A block no request holds any more: cached if indexed, else free."""
        if b in self.key_of:
            self.cached.append(b)
        else:
            self.free_list.append(b)

    def _evict(self, n: int) -> None:
        """Evict n cached blocks, each time the oldest one no indexed block extends."""
        children: dict[int, int] = {}
        for key in self.index:
            children[key[1]] = children.get(key[1], 0) + 1
        for _ in range(n):
            for b in self.cached:
                if children.get(b, 0) == 0:
                    break
            else:
                raise AllocatorError("no evictable cached block")
            self.cached.remove(b)
            key = self.key_of.pop(b)
            del self.index[key]
            children[key[1]] -= 1
            self.free_list.append(b)
            self.pfx.evictions += 1

    # -- transitions -------------------------------------------------------------
    def fork(self, parent: int, child: int) -> None:
        """child starts with parent's committed blocks and token count."""
        if self.pending is not None:
            raise AllocatorError("fork while a reservation is open")
        if self.tables.get(child) or child in self.prompts:
            raise AllocatorError("fork into a request that holds blocks")
        if parent not in self.tables:
            raise AllocatorError("fork of a request that holds nothing")
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        self.check()

    def reserve(self, plan) -> bool:
        """plan: [(req, s_i)].  Reserves every new block or none.  Returns False
        (state unchanged) when the plan needs more than q_free + q_cached."""
        if self.pending is not None:
            raise AllocatorError("a reservation is already open")
        reqs = [r for r, _ in plan]
        if len(set(reqs)) != len(reqs):
            raise AllocatorError("request listed twice in one plan")
        need, cows = [], []
        B = self.block_size
        copied_away: dict[int, int] = {}   # source block -> earlier plan entries copying it
        holders: dict[int, int] = {}       # block -> requests holding it
        for t in self.tables.values():
            for b in t:
                holders[b] = holders.get(b, 0) + 1
        for r, s in plan:
            if s < 0:
                raise AllocatorError("negative token count")
            held = self.held_tokens(r)
            d = delta_blocks(held, s, B)
            if blocks_for(held + s, B) > self.max_blocks_per_req:
                raise AllocatorError("block table capacity exceeded")
            cow = False
            if s > 0 and held % B != 0:
                last = self.tables[r][-1]
                # the last writer of a shared partial block keeps the original
                cow = holders[last] - copied_away.get(last, 0) > 1
                if cow:
                    copied_away[last] = copied_away.get(last, 0) + 1
            need.append(d)
            cows.append(cow)
        total = sum(need) + sum(cows)
        if total > self.available():
            self.alloc_failures += 1
            return False
        if len(self.free_list) < total:
            self._evict(total - len(self.free_list))
        pending = []
        for (r, s), d, cow in zip(plan, need, cows):
            c = None
            if cow:
                li = len(self.tables[r]) - 1
                c = (li, self.tables[r][li], self.free_list.pop(0))
            new = [self.free_list.pop(0) for _ in range(d)]
            pending.append((r, s, new, c))
        self.pending = pending
        s_ = self.stats()
        self.peak_used = max(self.peak_used, s_.reserved + s_.committed)
        self.check()
        return True

    def commit(self) -> None:
        if self.pending is None:
            raise AllocatorError("nothing reserved")
        pending, self.pending = self.pending, None
        for r, s, new, c in pending:
            self.tables.setdefault(r, [])
            self.tokens.setdefault(r, 0)
            if c is not None:
                li, src, dst = c
                self.tables[r][li] = dst
                self.pfx.cow_copies += 1
                if self.holders(src) == 0:
                    self._release(src)
            self.tables[r] += new
            self.tokens[r] += s
        for r, _, _, _ in pending:
            self._index_prompt_blocks(r)
        self.check()

    def rollback(self) -> None:
        if self.pending is None:
            raise AllocatorError("nothing reserved")
        back = []
        for _, _, new, c in self.pending:
            back += ([c[2]] if c is not None else []) + new
        self.free_list = back + self.free_list
        self.pending = None
        self.check()

    # -- swapping ---------------------------------------------------------------
    def swap_out(self, req: int):
        """Move req's blocks to the CPU pool.  Returns ([(gpu, cpu)], released
        GPU blocks), or None (state unchanged) if the CPU pool is too small."""
        if self.pending is not None:
            raise AllocatorError("swap_out while a reservation is open")
        if req in self.swapped or not self.tables.get(req):
            raise AllocatorError("swap_out of a request that holds no GPU blocks")
        blocks = list(self.tables[req])
        if len(blocks) > len(self.cpu_free):
            return None
        cpu = [self.cpu_free.pop(0) for _ in blocks]
        tokens = self.tokens[req]
        released = self._release_request(req)
        self.swapped[req] = (cpu, tokens)
        self.check()
        return list(zip(blocks, cpu)), released

    def swap_in_status(self, req: int) -> str:
        n = len(self.swapped[req][0])
        if n > self.capacity:
            return "never"
        return "later" if n > self.available() else "ok"

    def swap_in(self, req: int) -> list[tuple[int, int]]:
        """Bring req back into fresh GPU blocks; returns [(cpu, gpu)]."""
        if self.pending is not None:
            raise AllocatorError("swap_in while a reservation is open")
        if self.swap_in_status(req) != "ok":
            raise AllocatorError("swap_in without the blocks")
        cpu, tokens = self.swapped.pop(req)
        if len(self.free_list) < len(cpu):
            self._evict(len(cpu) - len(self.free_list))
        gpu = [self.free_list.pop(0) for _ in cpu]
        self.tables[req] = gpu
        self.tokens[req] = tokens
        self.cpu_free += cpu
        s_ = self.stats()
        self.peak_used = max(self.peak_used, s_.reserved + s_.committed)
        self.check()
        return list(zip(cpu, gpu))

    def free_request(self, req: int) -> int:
        """Release `req`: its committed blocks in table order (each one no other
        request holds goes to the cache if indexed, else to the back of the free
        list), then any reserved ones to the back of the free list; a swapped
        request releases its CPU blocks.  Returns how many GPU blocks it held
        that no request holds any more."""
        if req in self.swapped:
            self.cpu_free += self.swapped.pop(req)[0]
        released = self._release_request(req)
        self.check()
        return released

    def _release_request(self, req: int) -> int:
        released = 0
        if req in self.tables:
            blocks = self.tables.pop(req)
            self.tokens.pop(req)
            still_held = self.live_blocks()
            for b in blocks:
                if b not in still_held:
                    self._release(b)
                    released += 1
        if self.pending is not None:
            keep = []
            for r, s, new, c in self.pending:
                if r == req:
                    back = ([c[2]] if c is not None else []) + new
                    self.free_list += back
                    released += len(back)
                else:
                    keep.append((r, s, new, c))
            self.pending = keep
        self.prompts.pop(req, None)
        self.indexed_upto.pop(req, None)
        return released
