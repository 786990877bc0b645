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
// The free list is a ring buffer over num_blocks slots, so pop-front,
// push-back and the push-front of a rollback are O(1).  Each request keeps one
// vector of block ids: committed blocks first, then the blocks reserved for the
// open plan.
#include "host_alloc.h"

#include <algorithm>
#include <vector>

#include "pkv_error.h"

namespace pkv {

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

Allocator::Allocator(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_req)
    : capacity_(num_blocks), block_size_(block_size), max_blocks_per_req_(max_blocks_per_req),
      ring_(static_cast<size_t>(num_blocks)), head_(0), count_(num_blocks) {
  for (int32_t i = 0; i < num_blocks; ++i) ring_[i] = i;
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

int64_t Allocator::held_tokens(int32_t req) const {
  auto it = reqs_.find(req);
  return it == reqs_.end() ? 0 : it->second.tokens;
}

int Allocator::reserve(int32_t n, const int32_t* ids, const int32_t* new_tokens) {
  if (open_) return fail(PKV_E_STATE, "reserve: a reservation is already open");
  if (n < 0 || (n > 0 && (!ids || !new_tokens))) return fail(PKV_E_INVALID, "reserve: bad plan");
  std::vector<int64_t> need(static_cast<size_t>(n));
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
    need[i] = after - ceil_div(held, block_size_);
    total += need[i];
  }
  if (total > count_) {
    ++alloc_failures_;
    return fail(PKV_E_NO_BLOCKS, "reserve: %lld blocks needed, %d free",
                static_cast<long long>(total), count_);
  }
  plan_.clear();
  for (int32_t i = 0; i < n; ++i) {
    ReqBlocks& r = reqs_[ids[i]];
    r.committed = static_cast<int32_t>(r.blocks.size());
    for (int64_t k = 0; k < need[i]; ++k) r.blocks.push_back(pop_front());
    plan_.push_back({ids[i], new_tokens[i], static_cast<int32_t>(need[i])});
  }
  reserved_ = total;
  open_ = true;
  peak_used_ = std::max<int64_t>(peak_used_, capacity_ - count_);
  return ok();
}

int Allocator::commit() {
  if (!open_) return fail(PKV_E_STATE, "commit: nothing reserved");
  for (const PlanEntry& e : plan_) {
    ReqBlocks& r = reqs_[e.req];
    r.tokens += e.tokens;
    r.committed = static_cast<int32_t>(r.blocks.size());
    committed_ += e.blocks;
  }
  // a request planned with zero tokens and no blocks holds nothing
  for (const PlanEntry& e : plan_) {
    auto it = reqs_.find(e.req);
    if (it != reqs_.end() && it->second.blocks.empty() && it->second.tokens == 0) reqs_.erase(it);
  }
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
    if (r.blocks.empty() && r.tokens == 0) reqs_.erase(e->req);
  }
  plan_.clear();
  reserved_ = 0;
  open_ = false;
  return ok();
}

int Allocator::free_request(int32_t req) {
  auto it = reqs_.find(req);
  if (it == reqs_.end()) return 0;
  ReqBlocks& r = it->second;
  int32_t released = static_cast<int32_t>(r.blocks.size());
  for (int32_t b : r.blocks) push_back(b);  // committed first, then reserved
  committed_ -= r.committed;
  if (open_) {
    for (size_t i = 0; i < plan_.size(); ++i) {
      if (plan_[i].req == req) {
        reserved_ -= plan_[i].blocks;
        plan_.erase(plan_.begin() + static_cast<long>(i));
        break;
      }
    }
  }
  reqs_.erase(it);
  return released;
}

void Allocator::stats(pkv_alloc_stats* s) const {
  s->capacity = capacity_;
  s->free = count_;
  s->reserved = reserved_;
  s->committed = committed_;
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

int Allocator::check() const {
  if (count_ + reserved_ + committed_ != capacity_)
    return fail(PKV_E_STATE, "conservation violated: %d + %lld + %lld != %d", count_,
                static_cast<long long>(reserved_), static_cast<long long>(committed_), capacity_);
  std::vector<uint8_t> seen(static_cast<size_t>(capacity_), 0);
  auto mark = [&](int32_t b) {
    if (b < 0 || b >= capacity_ || seen[b]) return false;
    seen[b] = 1;
    return true;
  };
  for (int32_t i = 0; i < count_; ++i)
    if (!mark(ring_[(head_ + i) % capacity_])) return fail(PKV_E_STATE, "free list corrupt");
  int64_t committed = 0, reserved = 0;
  for (const auto& kv : reqs_) {
    const ReqBlocks& r = kv.second;
    for (int32_t b : r.blocks)
      if (!mark(b)) return fail(PKV_E_STATE, "block %d referenced twice", b);
    if (r.committed != ceil_div(r.tokens, block_size_))
      return fail(PKV_E_STATE, "request %d: q_i != ceil(T_i/B)", kv.first);
    committed += r.committed;
    reserved += static_cast<int64_t>(r.blocks.size()) - r.committed;
  }
  if (committed != committed_ || reserved != reserved_)
    return fail(PKV_E_STATE, "counters disagree with tables");
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

}  // extern "C"
