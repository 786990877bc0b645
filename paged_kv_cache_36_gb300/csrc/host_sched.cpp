// Host continuous-batching scheduler with recompute preemption, and the
// per-step metadata (block_table rows, query_start_loc, seq_lens,
// num_computed_tokens, slot_mapping) built from its plan.
//
// Policy sources:
// * "AI Infra入门干货总结：大模型是如何高效推理的", section "连续批处理": each step
//   moves num_computed_tokens toward num_tokens under four limits
//   (max_num_seqs, token budget, max_model_len, free blocks); appendix 4
//   ("附4：vLLM调度详细流程"): preemption frees all KV, resets
//   num_computed_tokens to 0 and prepends the request to WAITING; a step that
//   preempted admits nothing.
// * "vLLM 抢占机制源码精读", section "_schedule_running 中的抢占循环": RUNNING is
//   FCFS (head = highest priority); while the current request cannot get
//   slots the queue tail is preempted; with no one left behind it the request
//   preempts itself and the scan ends.  Section "人工抢占测试": a test hook
//   fails the slot check with a fixed probability a bounded number of times.
// * "显存与调度", sections "分配是词元计划的一部分" (delta_q_i, all-or-nothing
//   reservation, commit/rollback) and "分块预填充共享每轮预算" (sum of the
//   step's decode and chunk tokens <= K).
//
// * "显存与调度", sections "共享前缀会改变块的所有权" and "内存压力需要明确策略";
//   "Chunked Prefill 与 Preemption" (a prefix cache lets a recomputed request
//   hit part of its prefix): a request added with its prompt's token ids is
//   matched against the prefix index when admitted and starts at the matched
//   token count; a step may take q_free + q_cached blocks (cached ones are
//   evicted on demand); a preemption gives back the blocks no other request
//   holds.
//
// Where the pages leave a step open this follows the same readings as the
// library's design notes: s_i = min(num_tokens - num_computed, chunk_size,
// remaining budget); a request that catches up samples one token and then
// finishes or grows by one; new blocks are reserved in plan order.
#include <algorithm>
#include <cstring>
#include <deque>
#include <unordered_map>
#include <vector>

#include "host_alloc.h"
#include "pkv_error.h"

namespace pkv {

static inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// splitmix64 as published by Steele, Lea and Flood (OOPSLA 2014).
struct SplitMix64 {
  uint64_t state;
  uint64_t next() {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return static_cast<double>(next() >> 11) * (1.0 / 9007199254740992.0); }
};

enum Status : int32_t { kWaiting = 0, kRunning = 1, kFinished = 2, kSwapped = 3, kIgnored = 4 };

struct Req {
  int32_t id;
  int32_t prompt_len;
  int32_t max_output;
  int32_t outputs = 0;
  int64_t num_tokens;
  int64_t num_computed = 0;
  int32_t preemptions = 0;
  Status status = kWaiting;
  bool has_tokens = false;      // prompt token ids known: prefix sharing applies
  uint64_t ns = 0;
  std::vector<int32_t> tokens;
};

struct Entry {
  int32_t req;
  int32_t s;
  int64_t computed_before;
};

class Scheduler {
 public:
  explicit Scheduler(const pkv_sched_config& c)
      : cfg_(c),
        handle_(c.num_blocks, c.block_size, c.max_blocks_per_req,
                c.preemption_mode == PKV_PREEMPT_SWAP ? c.num_cpu_blocks : 0),
        alloc_(handle_.impl),
        rng_{c.artificial_seed}, inject_left_(c.artificial_preempt_max) {}

  int add_request(int32_t id, int32_t prompt, int32_t max_output, uint64_t ns = 0,
                  const int32_t* tokens = nullptr) {
    if (reqs_.count(id) || prompt < 1 || max_output < 1 || prompt >= cfg_.max_model_len) return 0;
    max_output = std::min<int32_t>(max_output, cfg_.max_model_len - prompt);
    const int64_t largest = ceil_div64(static_cast<int64_t>(prompt) + max_output, cfg_.block_size);
    if (largest > cfg_.num_blocks || largest > cfg_.max_blocks_per_req) return 0;
    Req r;
    r.id = id;
    r.prompt_len = prompt;
    r.max_output = max_output;
    r.num_tokens = prompt;
    if (tokens) {
      r.has_tokens = true;
      r.ns = ns;
      r.tokens.assign(tokens, tokens + prompt);
    }
    reqs_.emplace(id, std::move(r));
    waiting_.push_back(id);
    return 1;
  }

  int step(pkv_step_info* info) {
    if (open_) return fail(PKV_E_STATE, "pkv_sched_step: previous step not finished");
    entries_.clear();
    preempted_.clear();
    admitted_.clear();
    swapped_out_.clear();
    swapped_in_.clear();
    ignored_.clear();
    swap_out_pairs_.clear();
    swap_in_pairs_.clear();
    const int32_t B = cfg_.block_size;
    int64_t budget = cfg_.max_num_batched_tokens;
    int64_t free_blocks = alloc_.available();

    // RUNNING scan, head first.  Requests before position i are scheduled;
    // victims are taken from the back, which is never before i.
    size_t i = 0;
    while (i < running_.size() && budget > 0) {
      Req& r = reqs_.at(running_[i]);
      const int64_t s = std::min<int64_t>({r.num_tokens - r.num_computed, cfg_.chunk_size, budget});
      const int64_t held = alloc_.held_tokens(r.id);
      const int64_t need = ceil_div64(held + s, B) - ceil_div64(held, B);
      bool self_preempted = false;
      for (;;) {
        bool fits = need <= free_blocks;
        if (cfg_.artificial_preempt_prob > 0.0) {
          const double u = rng_.uniform();
          if (u < cfg_.artificial_preempt_prob && inject_left_ > 0) {
            --inject_left_;
            fits = false;
          }
        }
        if (fits) break;
        if (i + 1 < running_.size()) {
          const int32_t victim = running_.back();
          free_blocks += preempt(victim);
        } else {
          free_blocks += preempt(r.id);
          self_preempted = true;
          break;
        }
      }
      if (self_preempted) break;
      entries_.push_back({r.id, static_cast<int32_t>(s), r.num_computed});
      budget -= s;
      free_blocks -= need;
      ++i;
    }

    // SWAPPED, head first, only when nothing was preempted in this step.
    if (preempted_.empty()) {
      while (!swapped_.empty() && budget > 0 &&
             static_cast<int64_t>(running_.size()) < cfg_.max_num_seqs) {
        Req& r = reqs_.at(swapped_.front());
        const int st = alloc_.swap_in_status(r.id);
        if (st < 0) return st;
        if (st == 2) {  // never: more blocks than the pool
          swapped_.pop_front();
          alloc_.free_request(r.id);
          r.status = kIgnored;
          ignored_.push_back(r.id);
          continue;
        }
        int64_t tokens = 0;
        const int n = alloc_.swapped_blocks(r.id, nullptr, 0x7fffffff, &tokens);
        if (n < 0) return n;
        const int64_t s = std::min<int64_t>({r.num_tokens - r.num_computed, cfg_.chunk_size, budget});
        const int64_t need = n + ceil_div64(tokens + s, B) - ceil_div64(tokens, B);
        if (need > free_blocks) break;
        swapped_.pop_front();
        std::vector<int32_t> pairs(2 * static_cast<size_t>(n));
        const int got = alloc_.swap_in(r.id, pairs.data(), n);
        if (got < 0) return got;
        swap_in_pairs_.insert(swap_in_pairs_.end(), pairs.begin(), pairs.end());
        r.status = kRunning;
        running_.push_back(r.id);
        swapped_in_.push_back(r.id);
        entries_.push_back({r.id, static_cast<int32_t>(s), r.num_computed});
        budget -= s;
        free_blocks -= need;
      }
    }

    // WAITING admission, only when nothing was preempted in this step and
    // nothing is left swapped.
    if (preempted_.empty() && swapped_.empty()) {
      while (!waiting_.empty() && budget > 0 &&
             static_cast<int64_t>(running_.size()) < cfg_.max_num_seqs) {
        Req& r = reqs_.at(waiting_.front());
        int64_t matched = 0;
        int32_t from_cache = 0;
        const bool prefix = r.has_tokens && r.num_computed == 0;
        if (prefix)
          matched = alloc_.peek_prefix(r.ns, r.tokens.data(), r.prompt_len, &from_cache);
        const int64_t start = std::max(r.num_computed, matched);
        const int64_t s = std::min<int64_t>({r.num_tokens - start, cfg_.chunk_size, budget});
        const int64_t held = std::max(alloc_.held_tokens(r.id), matched);
        const int64_t need = ceil_div64(held + s, B) - ceil_div64(held, B);
        if (need + from_cache > free_blocks) break;
        if (prefix) {
          const int m = alloc_.match_prefix(r.id, r.ns, r.tokens.data(), r.prompt_len);
          if (m < 0) return m;
          r.num_computed = m;
        }
        waiting_.pop_front();
        running_.push_back(r.id);
        r.status = kRunning;
        admitted_.push_back(r.id);
        entries_.push_back({r.id, static_cast<int32_t>(s), r.num_computed});
        budget -= s;
        free_blocks -= need + from_cache;
      }
    }

    std::vector<int32_t> ids, toks;
    ids.reserve(entries_.size());
    toks.reserve(entries_.size());
    for (const Entry& e : entries_) {
      ids.push_back(e.req);
      toks.push_back(e.s);
    }
    const int rc = alloc_.reserve(static_cast<int32_t>(ids.size()), ids.data(), toks.data());
    if (rc != PKV_OK) return rc;  // cannot happen: the plan was sized to fit
    open_ = true;
    fill_info(info);
    return PKV_OK;
  }

  int finish_step(int32_t ok, int32_t* finished, int32_t cap) {
    if (!open_) return fail(PKV_E_STATE, "pkv_sched_finish_step: no open step");
    open_ = false;
    if (!ok) return alloc_.rollback() == PKV_OK ? 0 : PKV_E_STATE;
    int rc = alloc_.commit();
    if (rc != PKV_OK) return rc;
    int32_t nfin = 0;
    for (const Entry& e : entries_) {
      Req& r = reqs_.at(e.req);
      r.num_computed += e.s;
      if (r.num_computed != r.num_tokens) continue;
      ++r.outputs;
      if (r.outputs >= r.max_output) {
        alloc_.free_request(r.id);
        r.status = kFinished;
        running_.erase(std::find(running_.begin(), running_.end(), r.id));
        ++finished_count_;
        if (finished && nfin < cap) finished[nfin] = r.id;
        ++nfin;
      } else {
        ++r.num_tokens;
      }
    }
    return nfin;
  }

  int build_metadata(int32_t* bt, int32_t stride, int32_t* qsl, int32_t* seq, int32_t* nc,
                     int64_t* slots) const {
    if (!open_) return fail(PKV_E_STATE, "pkv_sched_build_metadata: no open step");
    const int32_t B = cfg_.block_size;
    int64_t t = 0;
    if (qsl) qsl[0] = 0;
    for (size_t k = 0; k < entries_.size(); ++k) {
      const Entry& e = entries_[k];
      const std::vector<int32_t>* row = alloc_.blocks(e.req);
      const int32_t nblk = row ? static_cast<int32_t>(row->size()) : 0;
      if (nblk > stride) return fail(PKV_E_INVALID, "block_table stride %d < %d", stride, nblk);
      if (bt) {
        int32_t* dst = bt + static_cast<int64_t>(k) * stride;
        for (int32_t j = 0; j < stride; ++j) dst[j] = j < nblk ? (*row)[j] : -1;
      }
      if (seq) seq[k] = static_cast<int32_t>(e.computed_before + e.s);
      if (nc) nc[k] = static_cast<int32_t>(e.computed_before);
      if (slots) {
        for (int32_t q = 0; q < e.s; ++q) {
          const int64_t pos = e.computed_before + q;
          slots[t + q] = static_cast<int64_t>((*row)[pos / B]) * B + pos % B;
        }
      }
      t += e.s;
      if (qsl) qsl[k + 1] = static_cast<int32_t>(t);
    }
    return PKV_OK;
  }

  const std::vector<Entry>& entries() const { return entries_; }
  const std::vector<int32_t>& preempted() const { return preempted_; }
  const std::vector<int32_t>& admitted() const { return admitted_; }
  const std::vector<int32_t>& swapped_out() const { return swapped_out_; }
  const std::vector<int32_t>& swapped_in() const { return swapped_in_; }
  const std::vector<int32_t>& ignored() const { return ignored_; }
  const std::vector<int32_t>& swap_out_pairs() const { return swap_out_pairs_; }
  const std::vector<int32_t>& swap_in_pairs() const { return swap_in_pairs_; }
  const std::deque<int32_t>& swapped_queue() const { return swapped_; }
  const std::vector<int32_t>& running() const { return running_; }
  const std::deque<int32_t>& waiting() const { return waiting_; }
  const pkv_alloc* handle() const { return &handle_; }
  const Req* find(int32_t id) const {
    auto it = reqs_.find(id);
    return it == reqs_.end() ? nullptr : &it->second;
  }
  void counters(int64_t* out) const {
    out[0] = total_preemptions_;
    out[1] = recomputed_tokens_;
    out[2] = finished_count_;
    out[3] = inject_left_;
  }
  int64_t swapped_out_blocks() const { return swapped_out_blocks_; }

 private:
  // Swap (if configured and the CPU pool has room) or recompute preemption:
  // returns how many blocks no request holds any more.
  int64_t preempt(int32_t id) {
    Req& r = reqs_.at(id);
    if (cfg_.preemption_mode == PKV_PREEMPT_SWAP) {
      const std::vector<int32_t>* row = alloc_.blocks(id);
      const int32_t n = row ? static_cast<int32_t>(row->size()) : 0;
      if (n > 0 && n <= alloc_.cpu_free()) {
        std::vector<int32_t> pairs(2 * static_cast<size_t>(n));
        int32_t released = 0;
        const int got = alloc_.swap_out(id, pairs.data(), n, &released);
        if (got == n) {
          swap_out_pairs_.insert(swap_out_pairs_.end(), pairs.begin(), pairs.end());
          swapped_out_blocks_ += n;
          r.status = kSwapped;
          ++r.preemptions;
          ++total_preemptions_;
          running_.erase(std::find(running_.begin(), running_.end(), id));
          swapped_.push_back(id);
          preempted_.push_back(id);
          swapped_out_.push_back(id);
          return released;
        }
      }
    }
    recomputed_tokens_ += r.num_computed;
    const int released = alloc_.free_request(id);
    r.num_computed = 0;
    r.status = kWaiting;
    ++r.preemptions;
    ++total_preemptions_;
    running_.erase(std::find(running_.begin(), running_.end(), id));
    waiting_.push_front(id);
    preempted_.push_back(id);
    return released;
  }

  void fill_info(pkv_step_info* info) const {
    if (!info) return;
    std::memset(info, 0, sizeof(*info));
    info->num_reqs = static_cast<int32_t>(entries_.size());
    info->num_preempted = static_cast<int32_t>(preempted_.size());
    info->num_admitted = static_cast<int32_t>(admitted_.size());
    for (const Entry& e : entries_) {
      info->num_tokens += e.s;
      info->max_query_len = std::max(info->max_query_len, e.s);
      const std::vector<int32_t>* row = alloc_.blocks(e.req);
      info->max_blocks = std::max(info->max_blocks, row ? static_cast<int32_t>(row->size()) : 0);
    }
  }

  pkv_sched_config cfg_;
  pkv_alloc handle_;
  Allocator& alloc_;
  SplitMix64 rng_;
  int64_t inject_left_;
  std::unordered_map<int32_t, Req> reqs_;
  std::vector<int32_t> running_;
  std::deque<int32_t> waiting_;
  std::vector<Entry> entries_;
  std::vector<int32_t> preempted_, admitted_;
  std::deque<int32_t> swapped_;
  std::vector<int32_t> swapped_out_, swapped_in_, ignored_, swap_out_pairs_, swap_in_pairs_;
  bool open_ = false;
  int64_t total_preemptions_ = 0, recomputed_tokens_ = 0, finished_count_ = 0;
  int64_t swapped_out_blocks_ = 0;
};

}  // namespace pkv

using pkv::fail;

extern "C" {

struct pkv_sched {
  pkv::Scheduler impl;
  explicit pkv_sched(const pkv_sched_config& c) : impl(c) {}
};

pkv_sched* pkv_sched_create(const pkv_sched_config* c) {
  if (!c || c->max_num_seqs <= 0 || c->max_num_batched_tokens <= 0 || c->chunk_size <= 0 ||
      c->max_model_len <= 1 || c->block_size <= 0 || c->num_blocks <= 0 ||
      c->max_blocks_per_req <= 0 || c->artificial_preempt_prob < 0.0 ||
      c->artificial_preempt_max < 0 ||
      (c->preemption_mode != PKV_PREEMPT_RECOMPUTE && c->preemption_mode != PKV_PREEMPT_SWAP) ||
      c->num_cpu_blocks < 0) {
    fail(PKV_E_INVALID, "pkv_sched_create: invalid configuration");
    return nullptr;
  }
  try {
    return new pkv_sched(*c);
  } catch (...) {
    fail(PKV_E_INVALID, "pkv_sched_create: out of host memory");
    return nullptr;
  }
}

void pkv_sched_destroy(pkv_sched* s) { delete s; }

#define PKV_NEED_S(s) \
  if (!(s)) return fail(PKV_E_INVALID, "%s: null handle", __func__)

int pkv_sched_add_request(pkv_sched* s, int32_t id, int32_t prompt, int32_t max_output) {
  PKV_NEED_S(s);
  return s->impl.add_request(id, prompt, max_output);
}

int pkv_sched_add_request_tokens(pkv_sched* s, int32_t id, int32_t prompt, int32_t max_output,
                                 uint64_t ns, const int32_t* tokens) {
  PKV_NEED_S(s);
  if (!tokens) return fail(PKV_E_INVALID, "pkv_sched_add_request_tokens: null tokens");
  return s->impl.add_request(id, prompt, max_output, ns, tokens);
}

int pkv_sched_step(pkv_sched* s, pkv_step_info* info) {
  PKV_NEED_S(s);
  return s->impl.step(info);
}

int pkv_sched_plan(const pkv_sched* s, int32_t* ids, int32_t* toks, int32_t* before, int32_t cap) {
  PKV_NEED_S(s);
  const auto& e = s->impl.entries();
  if (static_cast<int64_t>(e.size()) > cap) return fail(PKV_E_INVALID, "pkv_sched_plan: capacity");
  for (size_t k = 0; k < e.size(); ++k) {
    if (ids) ids[k] = e[k].req;
    if (toks) toks[k] = e[k].s;
    if (before) before[k] = static_cast<int32_t>(e[k].computed_before);
  }
  return static_cast<int>(e.size());
}

static int copy_ids(const std::vector<int32_t>& v, int32_t* out, int32_t cap) {
  if (static_cast<int64_t>(v.size()) > cap) return fail(PKV_E_INVALID, "capacity %d too small", cap);
  if (out) std::copy(v.begin(), v.end(), out);
  return static_cast<int>(v.size());
}

int pkv_sched_preempted(const pkv_sched* s, int32_t* out, int32_t cap) {
  PKV_NEED_S(s);
  return copy_ids(s->impl.preempted(), out, cap);
}

int pkv_sched_admitted(const pkv_sched* s, int32_t* out, int32_t cap) {
  PKV_NEED_S(s);
  return copy_ids(s->impl.admitted(), out, cap);
}

int pkv_sched_swaps(const pkv_sched* s, int32_t* out_pairs, int32_t out_cap, int32_t* num_out,
                    int32_t* in_pairs, int32_t in_cap, int32_t* num_in) {
  PKV_NEED_S(s);
  const auto& o = s->impl.swap_out_pairs();
  const auto& i = s->impl.swap_in_pairs();
  const int32_t no = static_cast<int32_t>(o.size() / 2), ni = static_cast<int32_t>(i.size() / 2);
  if (num_out) *num_out = no;
  if (num_in) *num_in = ni;
  if (out_pairs) {
    if (no > out_cap) return fail(PKV_E_INVALID, "pkv_sched_swaps: capacity %d < %d", out_cap, no);
    std::copy(o.begin(), o.end(), out_pairs);
  }
  if (in_pairs) {
    if (ni > in_cap) return fail(PKV_E_INVALID, "pkv_sched_swaps: capacity %d < %d", in_cap, ni);
    std::copy(i.begin(), i.end(), in_pairs);
  }
  return PKV_OK;
}

int pkv_sched_swap_events(const pkv_sched* s, int32_t* so, int32_t* nso, int32_t* si, int32_t* nsi,
                          int32_t* ig, int32_t* nig, int32_t cap) {
  PKV_NEED_S(s);
  const int a = copy_ids(s->impl.swapped_out(), so, cap);
  if (a < 0) return a;
  const int b = copy_ids(s->impl.swapped_in(), si, cap);
  if (b < 0) return b;
  const int c = copy_ids(s->impl.ignored(), ig, cap);
  if (c < 0) return c;
  if (nso) *nso = a;
  if (nsi) *nsi = b;
  if (nig) *nig = c;
  return PKV_OK;
}

int pkv_sched_build_metadata(const pkv_sched* s, int32_t* bt, int32_t stride, int32_t* qsl,
                             int32_t* seq, int32_t* nc, int64_t* slots) {
  PKV_NEED_S(s);
  return s->impl.build_metadata(bt, stride, qsl, seq, nc, slots);
}

int pkv_sched_finish_step(pkv_sched* s, int32_t ok, int32_t* finished, int32_t cap) {
  PKV_NEED_S(s);
  return s->impl.finish_step(ok, finished, cap);
}

int pkv_sched_request(const pkv_sched* s, int32_t id, pkv_request_state* out) {
  PKV_NEED_S(s);
  if (!out) return fail(PKV_E_INVALID, "pkv_sched_request: null output");
  std::memset(out, 0, sizeof(*out));
  const pkv::Req* r = s->impl.find(id);
  if (!r) {
    out->status = -1;
    return PKV_E_UNKNOWN_REQ;
  }
  out->status = r->status;
  out->prompt_len = r->prompt_len;
  out->max_output = r->max_output;
  out->outputs = r->outputs;
  out->num_tokens = r->num_tokens;
  out->num_computed = r->num_computed;
  out->preemptions = r->preemptions;
  return PKV_OK;
}

int pkv_sched_queues(const pkv_sched* s, int32_t* running, int32_t* nrun, int32_t* waiting,
                     int32_t* nwait, int32_t cap) {
  PKV_NEED_S(s);
  const auto& r = s->impl.running();
  const auto& w = s->impl.waiting();
  if (static_cast<int64_t>(r.size()) > cap || static_cast<int64_t>(w.size()) > cap)
    return fail(PKV_E_INVALID, "pkv_sched_queues: capacity %d too small", cap);
  if (running) std::copy(r.begin(), r.end(), running);
  if (waiting) std::copy(w.begin(), w.end(), waiting);
  if (nrun) *nrun = static_cast<int32_t>(r.size());
  if (nwait) *nwait = static_cast<int32_t>(w.size());
  return PKV_OK;
}

int pkv_sched_swapped_queue(const pkv_sched* s, int32_t* out, int32_t* num, int32_t cap) {
  PKV_NEED_S(s);
  const auto& q = s->impl.swapped_queue();
  if (static_cast<int64_t>(q.size()) > cap)
    return fail(PKV_E_INVALID, "pkv_sched_swapped_queue: capacity %d too small", cap);
  if (out) std::copy(q.begin(), q.end(), out);
  if (num) *num = static_cast<int32_t>(q.size());
  return PKV_OK;
}

int pkv_sched_counters(const pkv_sched* s, int64_t* out4) {
  PKV_NEED_S(s);
  if (!out4) return fail(PKV_E_INVALID, "pkv_sched_counters: null output");
  s->impl.counters(out4);
  return PKV_OK;
}

const pkv_alloc* pkv_sched_allocator(const pkv_sched* s) {
  return s ? s->impl.handle() : nullptr;
}

}  // extern "C"
