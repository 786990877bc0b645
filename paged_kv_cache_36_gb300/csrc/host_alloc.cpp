// Host KV block allocator with reserve / execute / commit accounting.
//
// "显存与调度" (ch. 32), section "分配是词元计划的一部分" and Fig. 32.2: a plan's
// new blocks are reserved atomically before execution, committed on success,
// rolled back on failure or cancellation, and
//   q_free + q_reserved + q_committed = q_capacity
// holds after every transition; delta_q_i = ceil((T_i+s_i)/B) - ceil(T_i/B).
// Section "从保留词元到物理块": q_i = ceil(T_i/B), w_i = q_i B - T_i.
// "GPT-5 时代大模型推理调度系统深度实战", section 5.3 BlockManager: allocation
// drains the free list from the front, release pushes on the back.
//
// Prefix sharing: same page, section "共享前缀会改变块的所有权".  Requests with an
// identical KV prefix share its full blocks; q_live = |union of the block
// sets|; r_p counts the requests holding block p plus the prefix index if it
// retains p, and p is recycled only at r_p = 0; the index finds the longest
// reusable prefix and, under memory pressure, drops leaf entries that no
// request holds; full shared blocks are immutable and a shared block still
// being written is copied first.  The index is block-granular: the key of an
// entry is (namespace, the indexed block it extends or -1, its block_size
// token ids), so a key names the whole prefix exactly.  Only full blocks
// wholly inside a registered prompt are indexed, at the commit that
// completes them.  A block held by no request but kept by the index is
// "cached" and sits in a release-ordered list, so
//   q_free + q_reserved + q_live + q_cached = q_capacity.
// A plan that fits in q_free + q_cached but not in q_free first evicts the
// oldest cached blocks that no indexed block extends (to the back of the
// free list).  When a request writes into a partial last block that another
// request also holds, reserve() takes one more block for a copy-on-write: the
// plan's table shows the copy, the (source, destination) pair is listed for
// the device copy, and commit lets go of the source; within one plan the last
// writer of a shared block keeps the original.
//
// Swapping: "vLLM 抢占机制源码精读", sections "Swap 模式" and "Swap-in 恢复流程".
// swap_out needs a free CPU block per GPU block (else nothing changes), lists
// the GPU -> CPU pairs for the transfer and releases the GPU blocks as
// free_request would; swap_in is "never" possible with more blocks than the
// pool, "later" when they are not available, and otherwise takes fresh GPU
// blocks in table order (evicting cached ones as reserve() does), lists the
// CPU -> GPU pairs and releases the CPU blocks.  The CPU pool is a FIFO free
// list too.
//
// The free list is a ring buffer over num_blocks slots, so pop-front,
// push-back and the push-front of a rollback are O(1); the cached list is an
// intrusive doubly linked list over block ids.  Each request keeps one vector
// of block ids: committed blocks first, then the blocks reserved for the open
// plan.
#include "host_alloc.h"

#include <algorithm>
#include <cstring>
#include <functional>
#include <utility>
#include <string>
#include <vector>

#include "pkv_error.h"

namespace pkv {

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

Allocator::Allocator(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_req,
                     int32_t num_cpu_blocks)
    : capacity_(num_blocks), block_size_(block_size), max_blocks_per_req_(max_blocks_per_req),
      ring_(static_cast<size_t>(num_blocks)), head_(0), count_(num_blocks),
      holders_(static_cast<size_t>(num_blocks), 0), children_(static_cast<size_t>(num_blocks), 0),
      parent_(static_cast<size_t>(num_blocks), -2), key_of_(static_cast<size_t>(num_blocks)),
      lru_prev_(static_cast<size_t>(num_blocks), -1), lru_next_(static_cast<size_t>(num_blocks), -1),
      in_cache_(static_cast<size_t>(num_blocks), 0),
      cache_seq_(static_cast<size_t>(num_blocks), 0), cpu_capacity_(num_cpu_blocks),
      cpu_ring_(static_cast<size_t>(num_cpu_blocks > 0 ? num_cpu_blocks : 0)),
      cpu_count_(num_cpu_blocks > 0 ? num_cpu_blocks : 0) {
  for (int32_t i = 0; i < num_blocks; ++i) ring_[i] = i;
  for (int32_t i = 0; i < cpu_count_; ++i) cpu_ring_[i] = i;
  // the index holds at most one entry per block: sized once, it never
  // rehashes in the middle of a step
  index_.reserve(static_cast<size_t>(num_blocks));
}

int32_t Allocator::pop_front() {
  int32_t b = ring_[head_];
  head_ = (head_ + 1) % capacity_;
  --count_;
  return b;
}

void Allocator::push_back(int32_t b) {
  ring_[(head_ + count_) % capacity_] = b;
  ++count_;
}

void Allocator::push_front(int32_t b) {
  head_ = (head_ + capacity_ - 1) % capacity_;
  ring_[head_] = b;
  ++count_;
}

// ---------------------------------------------------------------- holders and the cache
void Allocator::hold(int32_t b) {
  if (holders_[b]++ == 0) ++live_;
}

void Allocator::unhold(int32_t b) {
  if (--holders_[b] == 0) {
    --live_;
    release(b);
  }
}

void Allocator::release(int32_t b) {
  if (parent_[b] != -2) lru_push_back(b);
  else push_back(b);
}

void Allocator::lru_push_back(int32_t b) {
  in_cache_[b] = 1;
  cache_seq_[b] = next_seq_++;
  if (children_[b] == 0) leaf_push(b);
  lru_prev_[b] = lru_tail_;
  lru_next_[b] = -1;
  if (lru_tail_ >= 0) lru_next_[lru_tail_] = b;
  else lru_head_ = b;
  lru_tail_ = b;
  ++cached_;
}

void Allocator::lru_remove(int32_t b) {
  const int32_t p = lru_prev_[b], n = lru_next_[b];
  if (p >= 0) lru_next_[p] = n;
  else lru_head_ = n;
  if (n >= 0) lru_prev_[n] = p;
  else lru_tail_ = p;
  lru_prev_[b] = lru_next_[b] = -1;
  in_cache_[b] = 0;
  --cached_;
}

// A cached block that no indexed block extends becomes an eviction candidate,
// ordered by when it was released to the cache.
void Allocator::leaf_push(int32_t b) {
  if (leaves_.size() >= 2 * static_cast<size_t>(capacity_) + 64) {
    // mostly stale: rebuild from the cached list (amortised over the pushes)
    leaves_.clear();
    for (int32_t c = lru_head_; c >= 0; c = lru_next_[c])
      if (children_[c] == 0 && c != b) leaves_.emplace_back(cache_seq_[c], c);
    std::make_heap(leaves_.begin(), leaves_.end(), std::greater<>());
  }
  leaves_.emplace_back(cache_seq_[b], b);
  std::push_heap(leaves_.begin(), leaves_.end(), std::greater<>());
}

// Evicts the oldest-released cached block that no indexed block extends (a
// leaf of the index): it leaves the index and goes to the back of the free
// list.  Its parent may become a leaf in turn.  Returns false when no cached
// block is a leaf (cannot happen while the index is consistent: the chain
// below a cached block is cached too).
bool Allocator::evict_one() {
  while (!leaves_.empty()) {
    std::pop_heap(leaves_.begin(), leaves_.end(), std::greater<>());
    const auto [seq, b] = leaves_.back();
    leaves_.pop_back();
    if (!in_cache_[b] || cache_seq_[b] != seq || children_[b] != 0) continue;  // stale
    lru_remove(b);
    index_.erase(key_of_[b]);
    key_of_[b].clear();
    const int32_t parent = parent_[b];
    parent_[b] = -2;
    if (parent >= 0 && --children_[parent] == 0 && in_cache_[parent]) leaf_push(parent);
    push_back(b);
    ++evictions_;
    return true;
  }
  return false;
}

std::string Allocator::key(uint64_t ns, int32_t parent, const int32_t* tokens) const {
  std::string k(sizeof(uint64_t) + sizeof(int32_t) * (1 + static_cast<size_t>(block_size_)), '\0');
  char* p = &k[0];
  std::memcpy(p, &ns, sizeof(ns));
  std::memcpy(p + sizeof(ns), &parent, sizeof(parent));
  std::memcpy(p + sizeof(ns) + sizeof(parent), tokens, sizeof(int32_t) * block_size_);
  return k;
}

int32_t Allocator::lookup(uint64_t ns, int32_t parent, const int32_t* tokens) const {
  auto it = index_.find(key(ns, parent, tokens));
  return it == index_.end() ? -1 : it->second;
}

// ---------------------------------------------------------------- prefix index
int Allocator::peek_prefix(uint64_t ns, const int32_t* tokens, int32_t n,
                           int32_t* cached_blocks) const {
  if (n < 0 || (n > 0 && !tokens)) return fail(PKV_E_INVALID, "peek_prefix: bad tokens");
  int32_t m = 0, cached = 0, parent = -1;
  const int32_t m_max = n > 0 ? (n - 1) / block_size_ : 0;
  while (m < m_max) {
    const int32_t b = lookup(ns, parent, tokens + static_cast<int64_t>(m) * block_size_);
    if (b < 0) break;
    if (holders_[b] == 0) ++cached;
    parent = b;
    ++m;
  }
  if (cached_blocks) *cached_blocks = cached;
  return m * block_size_;
}

int Allocator::match_prefix(int32_t req, uint64_t ns, const int32_t* tokens, int32_t n) {
  if (open_) return fail(PKV_E_STATE, "match_prefix: a reservation is open");
  if (n < 0 || (n > 0 && !tokens)) return fail(PKV_E_INVALID, "match_prefix: bad tokens");
  auto it = reqs_.find(req);
  if (it != reqs_.end() && (!it->second.blocks.empty() || it->second.has_prompt))
    return fail(PKV_E_STATE, "match_prefix: request %d already holds blocks", req);
  std::vector<int32_t> matched;
  int32_t parent = -1;
  const int32_t m_max = n > 0 ? (n - 1) / block_size_ : 0;
  while (static_cast<int32_t>(matched.size()) < m_max) {
    const int32_t b =
        lookup(ns, parent, tokens + static_cast<int64_t>(matched.size()) * block_size_);
    if (b < 0) break;
    matched.push_back(b);
    parent = b;
  }
  const int32_t m = static_cast<int32_t>(matched.size());
  ++lookups_;
  if (m > 0) {
    ++hits_;
    matched_tokens_ += static_cast<int64_t>(m) * block_size_;
  }
  ReqBlocks& r = reqs_[req];
  for (int32_t b : matched) {
    if (in_cache_[b]) lru_remove(b);
    hold(b);
  }
  r.blocks = matched;
  r.committed = m;
  r.tokens = static_cast<int64_t>(m) * block_size_;
  r.has_prompt = true;
  r.ns = ns;
  r.prompt.assign(tokens, tokens + n);
  r.indexed_upto = m;
  return m * block_size_;
}

void Allocator::index_prompt_blocks(int32_t req) {
  auto it = reqs_.find(req);
  if (it == reqs_.end() || !it->second.has_prompt) return;
  ReqBlocks& r = it->second;
  const int64_t plen = static_cast<int64_t>(r.prompt.size());
  const int64_t full = std::min<int64_t>(r.tokens, plen) / block_size_;
  int64_t j = r.indexed_upto;
  while (j < full) {
    const int32_t b = r.blocks[j];
    const int32_t parent = j == 0 ? -1 : r.blocks[j - 1];
    const int32_t* toks = r.prompt.data() + j * block_size_;
    std::string k = key(r.ns, parent, toks);
    if ((parent != -1 && parent_[parent] == -2) || index_.count(k)) {
      j = plen / block_size_ + 1;  // the chain is someone else's: stop for good
      break;
    }
    index_.emplace(k, b);
    key_of_[b] = std::move(k);
    parent_[b] = parent;
    if (parent >= 0) ++children_[parent];
    ++j;
  }
  r.indexed_upto = static_cast<int32_t>(j);
}

int Allocator::fork(int32_t parent, int32_t child) {
  if (open_) return fail(PKV_E_STATE, "fork: a reservation is open");
  auto pit = reqs_.find(parent);
  if (pit == reqs_.end()) return fail(PKV_E_UNKNOWN_REQ, "fork: request %d holds nothing", parent);
  auto cit = reqs_.find(child);
  if (cit != reqs_.end() && (!cit->second.blocks.empty() || cit->second.has_prompt))
    return fail(PKV_E_STATE, "fork: request %d already holds blocks", child);
  const std::vector<int32_t> blocks = pit->second.blocks;
  const int64_t tokens = pit->second.tokens;
  ReqBlocks& c = reqs_[child];
  c.blocks = blocks;
  c.committed = static_cast<int32_t>(blocks.size());
  c.tokens = tokens;
  for (int32_t b : blocks) hold(b);
  return ok();
}

// ---------------------------------------------------------------- transitions
int64_t Allocator::held_tokens(int32_t req) const {
  auto it = reqs_.find(req);
  return it == reqs_.end() ? 0 : it->second.tokens;
}

int64_t Allocator::plan_need(int32_t req, int32_t s,
                             std::unordered_map<int32_t, int32_t>* copied_away) const {
  const int64_t held = held_tokens(req);
  int64_t need = ceil_div(held + s, block_size_) - ceil_div(held, block_size_);
  if (s > 0 && held % block_size_ != 0) {
    const ReqBlocks& r = reqs_.at(req);
    const int32_t last = r.blocks[r.committed - 1];
    int32_t& away = (*copied_away)[last];
    if (holders_[last] - away > 1) {  // the last writer keeps the original
      ++away;
      ++need;
    }
  }
  return need;
}

int Allocator::reserve(int32_t n, const int32_t* ids, const int32_t* new_tokens) {
  if (open_) return fail(PKV_E_STATE, "reserve: a reservation is already open");
  if (n < 0 || (n > 0 && (!ids || !new_tokens))) return fail(PKV_E_INVALID, "reserve: bad plan");
  std::vector<int64_t> need(static_cast<size_t>(n));
  std::vector<uint8_t> cow(static_cast<size_t>(n), 0);
  std::unordered_map<int32_t, int32_t> copied_away;
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) {
    for (int32_t j = 0; j < i; ++j)
      if (ids[j] == ids[i]) return fail(PKV_E_INVALID, "reserve: request %d listed twice", ids[i]);
    if (new_tokens[i] < 0) return fail(PKV_E_INVALID, "reserve: negative token count");
    const int64_t held = held_tokens(ids[i]);
    const int64_t after = ceil_div(held + new_tokens[i], block_size_);
    if (after > max_blocks_per_req_)
      return fail(PKV_E_CAPACITY, "reserve: request %d would need %lld blocks (row holds %d)",
                  ids[i], static_cast<long long>(after), max_blocks_per_req_);
    const int64_t delta = after - ceil_div(held, block_size_);
    const int64_t with_copy = plan_need(ids[i], new_tokens[i], &copied_away);
    cow[i] = with_copy > delta;
    need[i] = delta;
    total += with_copy;
  }
  if (total > available()) {
    ++alloc_failures_;
    return fail(PKV_E_NO_BLOCKS, "reserve: %lld blocks needed, %d free and %lld cached",
                static_cast<long long>(total), count_, static_cast<long long>(cached_));
  }
  while (count_ < total)
    if (!evict_one()) return fail(PKV_E_STATE, "reserve: no cached block can be evicted");
  plan_.clear();
  for (int32_t i = 0; i < n; ++i) {
    ReqBlocks& r = reqs_[ids[i]];
    r.committed = static_cast<int32_t>(r.blocks.size());
    PlanEntry e{ids[i], new_tokens[i], static_cast<int32_t>(need[i])};
    if (cow[i]) {
      e.cow_index = r.committed - 1;
      e.cow_src = r.blocks[e.cow_index];
      e.cow_dst = pop_front();
      r.blocks[e.cow_index] = e.cow_dst;
    }
    for (int64_t k = 0; k < need[i]; ++k) r.blocks.push_back(pop_front());
    plan_.push_back(e);
  }
  reserved_ = total;
  open_ = true;
  peak_used_ = std::max<int64_t>(peak_used_, reserved_ + live_);
  return ok();
}

int Allocator::commit() {
  if (!open_) return fail(PKV_E_STATE, "commit: nothing reserved");
  for (const PlanEntry& e : plan_) {
    ReqBlocks& r = reqs_[e.req];
    if (e.cow_index >= 0) {
      ++cow_copies_;
      hold(e.cow_dst);
      unhold(e.cow_src);
    }
    for (size_t k = static_cast<size_t>(r.committed); k < r.blocks.size(); ++k) hold(r.blocks[k]);
    r.tokens += e.tokens;
    r.committed = static_cast<int32_t>(r.blocks.size());
  }
  // a request planned with zero tokens and no blocks holds nothing
  for (const PlanEntry& e : plan_) {
    auto it = reqs_.find(e.req);
    if (it != reqs_.end() && it->second.blocks.empty() && it->second.tokens == 0 &&
        !it->second.has_prompt)
      reqs_.erase(it);
  }
  for (const PlanEntry& e : plan_) index_prompt_blocks(e.req);
  plan_.clear();
  reserved_ = 0;
  open_ = false;
  return ok();
}

int Allocator::rollback() {
  if (!open_) return fail(PKV_E_STATE, "rollback: nothing reserved");
  // undo in reverse so the free list is restored exactly
  for (auto e = plan_.rbegin(); e != plan_.rend(); ++e) {
    ReqBlocks& r = reqs_[e->req];
    for (int32_t k = 0; k < e->blocks; ++k) {
      push_front(r.blocks.back());
      r.blocks.pop_back();
    }
    if (e->cow_index >= 0) {
      r.blocks[e->cow_index] = e->cow_src;
      push_front(e->cow_dst);
    }
    if (r.blocks.empty() && r.tokens == 0 && !r.has_prompt) reqs_.erase(e->req);
  }
  plan_.clear();
  reserved_ = 0;
  open_ = false;
  return ok();
}

int Allocator::free_request(int32_t req) {
  auto sw = swapped_.find(req);
  if (sw != swapped_.end()) {  // a swapped request lets its CPU blocks go
    for (int32_t c : sw->second.cpu) {
      cpu_ring_[(cpu_head_ + cpu_count_) % cpu_capacity_] = c;
      ++cpu_count_;
    }
    swapped_.erase(sw);
  }
  auto it = reqs_.find(req);
  if (it == reqs_.end()) return 0;
  return release_request(it);
}

int32_t Allocator::release_request(std::unordered_map<int32_t, ReqBlocks>::iterator it) {
  const int32_t req = it->first;
  ReqBlocks& r = it->second;
  const PlanEntry* e = nullptr;
  size_t e_at = 0;
  if (open_) {
    for (size_t i = 0; i < plan_.size(); ++i) {
      if (plan_[i].req == req) {
        e = &plan_[i];
        e_at = i;
        break;
      }
    }
  }
  int32_t released = 0;
  // committed blocks, in table order (a copy's source in its own place)
  for (int32_t k = 0; k < r.committed; ++k) {
    const int32_t b = (e && k == e->cow_index) ? e->cow_src : r.blocks[k];
    if (--holders_[b] == 0) {
      --live_;
      release(b);
      ++released;
    }
  }
  // then the reserved ones: the copy's destination, then the new blocks
  if (e) {
    if (e->cow_index >= 0) {
      push_back(e->cow_dst);
      ++released;
    }
    for (size_t k = static_cast<size_t>(r.committed); k < r.blocks.size(); ++k) {
      push_back(r.blocks[k]);
      ++released;
    }
    reserved_ -= e->blocks + (e->cow_index >= 0 ? 1 : 0);
    plan_.erase(plan_.begin() + static_cast<long>(e_at));
  }
  reqs_.erase(it);
  return released;
}

// ---------------------------------------------------------------- swapping
int Allocator::swap_out(int32_t req, int32_t* pairs, int32_t cap_pairs, int32_t* released) {
  if (open_) return fail(PKV_E_STATE, "swap_out: a reservation is open");
  auto it = reqs_.find(req);
  if (it == reqs_.end() || it->second.blocks.empty() || swapped_.count(req))
    return fail(PKV_E_STATE, "swap_out: request %d holds no GPU blocks", req);
  const std::vector<int32_t> blocks = it->second.blocks;
  const int32_t n = static_cast<int32_t>(blocks.size());
  if (n > cpu_count_)
    return fail(PKV_E_NO_BLOCKS, "swap_out: %d blocks, %d free CPU blocks", n, cpu_count_);
  if (n > cap_pairs || !pairs) return fail(PKV_E_INVALID, "swap_out: pair capacity %d < %d", cap_pairs, n);
  Swapped sw;
  sw.tokens = it->second.tokens;
  for (int32_t k = 0; k < n; ++k) {
    const int32_t c = cpu_ring_[cpu_head_];
    cpu_head_ = (cpu_head_ + 1) % cpu_capacity_;
    --cpu_count_;
    sw.cpu.push_back(c);
    pairs[2 * k] = blocks[k];
    pairs[2 * k + 1] = c;
  }
  const int32_t rel = release_request(it);
  if (released) *released = rel;
  swapped_.emplace(req, std::move(sw));
  return n;
}

int Allocator::swap_in_status(int32_t req) const {
  auto it = swapped_.find(req);
  if (it == swapped_.end()) return fail(PKV_E_UNKNOWN_REQ, "swap_in_status: request %d is not swapped", req);
  const int64_t n = static_cast<int64_t>(it->second.cpu.size());
  if (n > capacity_) return 2;
  return n > available() ? 1 : 0;
}

int Allocator::swap_in(int32_t req, int32_t* pairs, int32_t cap_pairs) {
  if (open_) return fail(PKV_E_STATE, "swap_in: a reservation is open");
  const int st = swap_in_status(req);
  if (st < 0) return st;
  if (st != 0) return fail(PKV_E_NO_BLOCKS, "swap_in: request %d cannot be swapped in now", req);
  auto it = swapped_.find(req);
  const int32_t n = static_cast<int32_t>(it->second.cpu.size());
  if (n > cap_pairs || !pairs) return fail(PKV_E_INVALID, "swap_in: pair capacity %d < %d", cap_pairs, n);
  while (count_ < n)
    if (!evict_one()) return fail(PKV_E_STATE, "swap_in: no cached block can be evicted");
  ReqBlocks& r = reqs_[req];
  r = ReqBlocks();
  for (int32_t k = 0; k < n; ++k) {
    const int32_t g = pop_front();
    hold(g);
    r.blocks.push_back(g);
    pairs[2 * k] = it->second.cpu[k];
    pairs[2 * k + 1] = g;
  }
  r.committed = n;
  r.tokens = it->second.tokens;
  for (int32_t c : it->second.cpu) {
    cpu_ring_[(cpu_head_ + cpu_count_) % cpu_capacity_] = c;
    ++cpu_count_;
  }
  swapped_.erase(it);
  peak_used_ = std::max<int64_t>(peak_used_, reserved_ + live_);
  return n;
}

int Allocator::swapped_blocks(int32_t req, int32_t* out, int32_t cap, int64_t* tokens) const {
  auto it = swapped_.find(req);
  if (it == swapped_.end()) return 0;
  const auto& c = it->second.cpu;
  if (static_cast<int64_t>(c.size()) > cap) return fail(PKV_E_INVALID, "swapped_blocks: capacity");
  if (out) std::copy(c.begin(), c.end(), out);
  if (tokens) *tokens = it->second.tokens;
  return static_cast<int>(c.size());
}

int Allocator::cpu_free_list(int32_t* out, int32_t cap) const {
  if (cpu_count_ > cap) return fail(PKV_E_INVALID, "cpu_free_list: capacity %d < %d", cap, cpu_count_);
  for (int32_t i = 0; i < cpu_count_; ++i) out[i] = cpu_ring_[(cpu_head_ + i) % cpu_capacity_];
  return cpu_count_;
}

// ---------------------------------------------------------------- queries
void Allocator::stats(pkv_alloc_stats* s) const {
  s->capacity = capacity_;
  s->free = count_;
  s->reserved = reserved_;
  s->committed = live_;
  int64_t nreq = 0, waste = 0;
  for (const auto& kv : reqs_) {
    if (kv.second.committed == 0) continue;
    ++nreq;
    waste += static_cast<int64_t>(kv.second.committed) * block_size_ - kv.second.tokens;
  }
  s->num_requests = nreq;
  s->tail_waste = waste;
  s->alloc_failures = alloc_failures_;
  s->peak_used = peak_used_;
}

void Allocator::prefix_stats(pkv_prefix_stats* s) const {
  s->lookups = lookups_;
  s->hits = hits_;
  s->matched_tokens = matched_tokens_;
  s->evictions = evictions_;
  s->cow_copies = cow_copies_;
  s->indexed = static_cast<int64_t>(index_.size());
  int64_t shared = 0;
  for (int32_t h : holders_) shared += h >= 2;
  s->shared = shared;
  s->cached = cached_;
}

int Allocator::table(int32_t req, int32_t* out, int32_t cap) const {
  auto it = reqs_.find(req);
  if (it == reqs_.end()) return 0;
  const auto& b = it->second.blocks;
  if (static_cast<int64_t>(b.size()) > cap)
    return fail(PKV_E_INVALID, "table: capacity %d < %zu blocks", cap, b.size());
  std::copy(b.begin(), b.end(), out);
  return static_cast<int>(b.size());
}

const std::vector<int32_t>* Allocator::blocks(int32_t req) const {
  auto it = reqs_.find(req);
  return it == reqs_.end() ? nullptr : &it->second.blocks;
}

int Allocator::free_list(int32_t* out, int32_t cap) const {
  if (count_ > cap) return fail(PKV_E_INVALID, "free_list: capacity %d < %d", cap, count_);
  for (int32_t i = 0; i < count_; ++i) out[i] = ring_[(head_ + i) % capacity_];
  return count_;
}

int Allocator::cached_list(int32_t* out, int32_t cap) const {
  if (cached_ > cap) return fail(PKV_E_INVALID, "cached_list: capacity %d < %lld", cap,
                                 static_cast<long long>(cached_));
  int32_t n = 0;
  for (int32_t b = lru_head_; b >= 0; b = lru_next_[b]) out[n++] = b;
  return n;
}

int Allocator::pending_copies(int32_t* pairs, int32_t cap_pairs) const {
  int32_t n = 0;
  for (const PlanEntry& e : plan_) {
    if (e.cow_index < 0) continue;
    if (n >= cap_pairs) return fail(PKV_E_INVALID, "pending_copies: capacity %d too small", cap_pairs);
    pairs[2 * n] = e.cow_src;
    pairs[2 * n + 1] = e.cow_dst;
    ++n;
  }
  return n;
}

int Allocator::ref_count(int32_t b) const {
  if (b < 0 || b >= capacity_) return fail(PKV_E_INVALID, "ref_count: block %d", b);
  return holders_[b] + (parent_[b] != -2 ? 1 : 0);
}

int Allocator::check() const {
  if (count_ + reserved_ + live_ + cached_ != capacity_)
    return fail(PKV_E_STATE, "conservation violated: %d + %lld + %lld + %lld != %d", count_,
                static_cast<long long>(reserved_), static_cast<long long>(live_),
                static_cast<long long>(cached_), capacity_);
  // 0 unseen, 1 free, 2 cached, 3 live, 4 reserved
  std::vector<uint8_t> where(static_cast<size_t>(capacity_), 0);
  auto mark = [&](int32_t b, uint8_t w) {
    if (b < 0 || b >= capacity_ || where[b]) return false;
    where[b] = w;
    return true;
  };
  for (int32_t i = 0; i < count_; ++i)
    if (!mark(ring_[(head_ + i) % capacity_], 1)) return fail(PKV_E_STATE, "free list corrupt");
  int64_t ncached = 0;
  for (int32_t b = lru_head_; b >= 0; b = lru_next_[b]) {
    if (!mark(b, 2) || !in_cache_[b] || holders_[b] != 0 || parent_[b] == -2)
      return fail(PKV_E_STATE, "cached list corrupt at block %d", b);
    ++ncached;
  }
  if (ncached != cached_) return fail(PKV_E_STATE, "cached count disagrees");
  std::vector<int32_t> holders(static_cast<size_t>(capacity_), 0);
  int64_t reserved = 0;
  for (const auto& kv : reqs_) {
    const ReqBlocks& r = kv.second;
    const PlanEntry* e = nullptr;
    for (const PlanEntry& p : plan_)
      if (p.req == kv.first) e = &p;
    std::vector<int32_t> mine;
    for (int32_t k = 0; k < r.committed; ++k) {
      const int32_t b = (e && k == e->cow_index) ? e->cow_src : r.blocks[k];
      if (b < 0 || b >= capacity_) return fail(PKV_E_STATE, "bad block id %d", b);
      mine.push_back(b);
      ++holders[b];
    }
    std::sort(mine.begin(), mine.end());
    if (std::adjacent_find(mine.begin(), mine.end()) != mine.end())
      return fail(PKV_E_STATE, "request %d holds a block twice", kv.first);
    if (r.committed != ceil_div(r.tokens, block_size_))
      return fail(PKV_E_STATE, "request %d: q_i != ceil(T_i/B)", kv.first);
    if (e) {
      if (e->cow_index >= 0) {
        if (!mark(e->cow_dst, 4)) return fail(PKV_E_STATE, "copy destination reused");
        ++reserved;
      }
      for (size_t k = static_cast<size_t>(r.committed); k < r.blocks.size(); ++k) {
        if (!mark(r.blocks[k], 4)) return fail(PKV_E_STATE, "reserved block reused");
        ++reserved;
      }
    } else if (static_cast<size_t>(r.committed) != r.blocks.size()) {
      return fail(PKV_E_STATE, "request %d has reserved blocks outside a plan", kv.first);
    }
  }
  int64_t live = 0;
  for (int32_t b = 0; b < capacity_; ++b) {
    if (holders[b] != holders_[b]) return fail(PKV_E_STATE, "holder count of block %d", b);
    if (holders[b] > 0) {
      if (!mark(b, 3)) return fail(PKV_E_STATE, "block %d held and listed", b);
      ++live;
    }
  }
  if (live != live_ || reserved != reserved_) return fail(PKV_E_STATE, "counters disagree with tables");
  for (int32_t b = 0; b < capacity_; ++b)
    if (!where[b]) return fail(PKV_E_STATE, "block %d is lost", b);
  std::vector<int32_t> children(static_cast<size_t>(capacity_), 0);
  for (const auto& kv : index_) {
    const int32_t b = kv.second;
    if (b < 0 || b >= capacity_ || key_of_[b] != kv.first || parent_[b] == -2 ||
        (where[b] != 2 && where[b] != 3))
      return fail(PKV_E_STATE, "index entry of block %d", b);
    if (parent_[b] >= 0) {
      if (parent_[parent_[b]] == -2) return fail(PKV_E_STATE, "block %d extends an unindexed block", b);
      ++children[parent_[b]];
    }
  }
  int64_t indexed = 0;
  for (int32_t b = 0; b < capacity_; ++b) {
    if (children[b] != children_[b]) return fail(PKV_E_STATE, "child count of block %d", b);
    indexed += parent_[b] != -2;
  }
  if (indexed != static_cast<int64_t>(index_.size())) return fail(PKV_E_STATE, "index size");
  // every cached leaf of the index has a current entry among the eviction
  // candidates
  std::vector<uint8_t> candidate(static_cast<size_t>(capacity_), 0);
  for (const auto& e : leaves_)
    if (e.second >= 0 && e.second < capacity_ && in_cache_[e.second] &&
        cache_seq_[e.second] == e.first)
      candidate[e.second] = 1;
  for (int32_t b = lru_head_; b >= 0; b = lru_next_[b])
    if (children_[b] == 0 && !candidate[b])
      return fail(PKV_E_STATE, "cached leaf %d is not an eviction candidate", b);
  std::vector<uint8_t> cpu_seen(static_cast<size_t>(cpu_capacity_ > 0 ? cpu_capacity_ : 0), 0);
  for (int32_t i = 0; i < cpu_count_; ++i) {
    const int32_t c = cpu_ring_[(cpu_head_ + i) % cpu_capacity_];
    if (c < 0 || c >= cpu_capacity_ || cpu_seen[c]++) return fail(PKV_E_STATE, "CPU free list corrupt");
  }
  for (const auto& kv : swapped_) {
    if (reqs_.count(kv.first)) return fail(PKV_E_STATE, "request %d swapped and resident", kv.first);
    if (static_cast<int64_t>(kv.second.cpu.size()) != ceil_div(kv.second.tokens, block_size_))
      return fail(PKV_E_STATE, "swapped request %d: q_i != ceil(T_i/B)", kv.first);
    for (int32_t c : kv.second.cpu)
      if (c < 0 || c >= cpu_capacity_ || cpu_seen[c]++) return fail(PKV_E_STATE, "CPU block %d twice", c);
  }
  for (int32_t c = 0; c < cpu_capacity_; ++c)
    if (!cpu_seen[c]) return fail(PKV_E_STATE, "CPU block %d is lost", c);
  return ok();
}

}  // namespace pkv

using pkv::Allocator;
using pkv::fail;

extern "C" {

pkv_alloc* pkv_alloc_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_req) {
  if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_req <= 0) {
    fail(PKV_E_INVALID, "pkv_alloc_create: sizes must be positive");
    return nullptr;
  }
  try {
    return new pkv_alloc(num_blocks, block_size, max_blocks_per_req);
  } catch (...) {
    fail(PKV_E_INVALID, "pkv_alloc_create: out of host memory");
    return nullptr;
  }
}

void pkv_alloc_destroy(pkv_alloc* a) { delete a; }

#define PKV_NEED(a) \
  if (!(a)) return fail(PKV_E_INVALID, "%s: null handle", __func__)

int pkv_alloc_reserve(pkv_alloc* a, int32_t n, const int32_t* ids, const int32_t* toks) {
  PKV_NEED(a);
  return a->impl.reserve(n, ids, toks);
}
int pkv_alloc_commit(pkv_alloc* a) {
  PKV_NEED(a);
  return a->impl.commit();
}
int pkv_alloc_rollback(pkv_alloc* a) {
  PKV_NEED(a);
  return a->impl.rollback();
}
int pkv_alloc_free_request(pkv_alloc* a, int32_t req) {
  PKV_NEED(a);
  return a->impl.free_request(req);
}
int pkv_alloc_get_stats(const pkv_alloc* a, pkv_alloc_stats* out) {
  PKV_NEED(a);
  if (!out) return fail(PKV_E_INVALID, "pkv_alloc_get_stats: null output");
  a->impl.stats(out);
  return PKV_OK;
}
int pkv_alloc_table(const pkv_alloc* a, int32_t req, int32_t* out, int32_t cap) {
  PKV_NEED(a);
  return a->impl.table(req, out, cap);
}
int64_t pkv_alloc_held_tokens(const pkv_alloc* a, int32_t req) {
  return a ? a->impl.held_tokens(req) : 0;
}
int pkv_alloc_free_list(const pkv_alloc* a, int32_t* out, int32_t cap) {
  PKV_NEED(a);
  return a->impl.free_list(out, cap);
}
int pkv_alloc_check(const pkv_alloc* a) {
  PKV_NEED(a);
  return a->impl.check();
}
int pkv_alloc_match_prefix(pkv_alloc* a, int32_t req, uint64_t ns, const int32_t* tokens,
                           int32_t n) {
  PKV_NEED(a);
  return a->impl.match_prefix(req, ns, tokens, n);
}
int pkv_alloc_peek_prefix(const pkv_alloc* a, uint64_t ns, const int32_t* tokens, int32_t n,
                          int32_t* cached_blocks) {
  PKV_NEED(a);
  return a->impl.peek_prefix(ns, tokens, n, cached_blocks);
}
int pkv_alloc_fork(pkv_alloc* a, int32_t parent, int32_t child) {
  PKV_NEED(a);
  return a->impl.fork(parent, child);
}
int pkv_alloc_pending_copies(const pkv_alloc* a, int32_t* pairs, int32_t capacity) {
  PKV_NEED(a);
  if (capacity > 0 && !pairs) return fail(PKV_E_INVALID, "pkv_alloc_pending_copies: null output");
  return a->impl.pending_copies(pairs, capacity);
}
int pkv_alloc_get_prefix_stats(const pkv_alloc* a, pkv_prefix_stats* out) {
  PKV_NEED(a);
  if (!out) return fail(PKV_E_INVALID, "pkv_alloc_get_prefix_stats: null output");
  a->impl.prefix_stats(out);
  return PKV_OK;
}
int pkv_alloc_ref_count(const pkv_alloc* a, int32_t block) {
  PKV_NEED(a);
  return a->impl.ref_count(block);
}
int pkv_alloc_cached_list(const pkv_alloc* a, int32_t* out, int32_t capacity) {
  PKV_NEED(a);
  return a->impl.cached_list(out, capacity);
}
int64_t pkv_alloc_available(const pkv_alloc* a) { return a ? a->impl.available() : 0; }

pkv_alloc* pkv_alloc_create_with_cpu_pool(int32_t num_blocks, int32_t block_size,
                                          int32_t max_blocks_per_req, int32_t num_cpu_blocks) {
  if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_req <= 0 || num_cpu_blocks < 0) {
    fail(PKV_E_INVALID, "pkv_alloc_create_with_cpu_pool: bad sizes");
    return nullptr;
  }
  try {
    return new pkv_alloc(num_blocks, block_size, max_blocks_per_req, num_cpu_blocks);
  } catch (...) {
    fail(PKV_E_INVALID, "pkv_alloc_create_with_cpu_pool: out of host memory");
    return nullptr;
  }
}
int pkv_alloc_swap_out(pkv_alloc* a, int32_t req, int32_t* pairs, int32_t capacity,
                       int32_t* released) {
  PKV_NEED(a);
  return a->impl.swap_out(req, pairs, capacity, released);
}
int pkv_alloc_swap_in_status(const pkv_alloc* a, int32_t req) {
  PKV_NEED(a);
  return a->impl.swap_in_status(req);
}
int pkv_alloc_swap_in(pkv_alloc* a, int32_t req, int32_t* pairs, int32_t capacity) {
  PKV_NEED(a);
  return a->impl.swap_in(req, pairs, capacity);
}
int pkv_alloc_swapped_blocks(const pkv_alloc* a, int32_t req, int32_t* out, int32_t capacity,
                             int64_t* tokens) {
  PKV_NEED(a);
  return a->impl.swapped_blocks(req, out, capacity, tokens);
}
int pkv_alloc_cpu_free_list(const pkv_alloc* a, int32_t* out, int32_t capacity) {
  PKV_NEED(a);
  return a->impl.cpu_free_list(out, capacity);
}

}  // extern "C"
