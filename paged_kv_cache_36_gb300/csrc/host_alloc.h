// Host KV block allocator (see host_alloc.cpp for the accounting rules).
#pragma once

#include <cstdint>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pkv.h"

namespace pkv {

class Allocator {
 public:
  Allocator(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_req,
            int32_t num_cpu_blocks = 0);

  int reserve(int32_t n, const int32_t* ids, const int32_t* new_tokens);
  int commit();
  int rollback();
  int free_request(int32_t req);  // blocks no request holds any more, >= 0
  void stats(pkv_alloc_stats* s) const;
  void prefix_stats(pkv_prefix_stats* s) const;
  int table(int32_t req, int32_t* out, int32_t cap) const;
  const std::vector<int32_t>* blocks(int32_t req) const;  // as table(), or null
  int64_t held_tokens(int32_t req) const;
  int free_list(int32_t* out, int32_t cap) const;
  int cached_list(int32_t* out, int32_t cap) const;
  int check() const;
  int32_t num_free() const { return count_; }
  int64_t available() const { return static_cast<int64_t>(count_) + cached_; }
  int32_t block_size() const { return block_size_; }
  bool open() const { return open_; }

  // prefix sharing
  int match_prefix(int32_t req, uint64_t ns, const int32_t* tokens, int32_t n);
  // matched token count without side effects; *cached_blocks = how many of the
  // matched blocks no request holds now (they leave q_cached when matched)
  int peek_prefix(uint64_t ns, const int32_t* tokens, int32_t n, int32_t* cached_blocks) const;
  int fork(int32_t parent, int32_t child);
  int pending_copies(int32_t* pairs, int32_t cap_pairs) const;
  int ref_count(int32_t block) const;
  // blocks a plan entry (req, s) needs: delta_q plus one for a copy-on-write;
  // `copied_away` carries the plan's earlier copies of shared partial blocks
  int64_t plan_need(int32_t req, int32_t s, std::unordered_map<int32_t, int32_t>* copied_away) const;

  // swapping: swap_out returns the pair count (GPU, CPU) written to `pairs`
  // or PKV_E_NO_BLOCKS when the CPU pool is too small (state unchanged);
  // swap_in_status is 0 (ok), 1 (later) or 2 (never); swap_in returns the
  // pair count (CPU, GPU)
  int swap_out(int32_t req, int32_t* pairs, int32_t cap_pairs, int32_t* released);
  int swap_in_status(int32_t req) const;
  int swap_in(int32_t req, int32_t* pairs, int32_t cap_pairs);
  int swapped_blocks(int32_t req, int32_t* out, int32_t cap, int64_t* tokens) const;
  int cpu_free_list(int32_t* out, int32_t cap) const;
  int32_t cpu_free() const { return cpu_count_; }
 private:
  struct ReqBlocks {
    // committed blocks (a copy-on-write destination stands in for its source
    // while a plan is open), then the blocks reserved for the open plan
    std::vector<int32_t> blocks;
    int32_t committed = 0;        // how many of `blocks` are committed
    int64_t tokens = 0;           // T_i, committed tokens
    bool has_prompt = false;      // registered by match_prefix
    uint64_t ns = 0;
    std::vector<int32_t> prompt;
    int32_t indexed_upto = 0;     // prompt blocks already settled
  };
  struct PlanEntry {
    int32_t req;
    int32_t tokens;
    int32_t blocks;               // new blocks (the copy destination not included)
    int32_t cow_index = -1;       // logical block replaced by a copy, or -1
    int32_t cow_src = -1;
    int32_t cow_dst = -1;
  };

  int32_t pop_front();
  void push_back(int32_t b);
  void push_front(int32_t b);
  int32_t release_request(std::unordered_map<int32_t, ReqBlocks>::iterator it);
  struct Swapped {
    std::vector<int32_t> cpu;
    int64_t tokens;
  };
  void hold(int32_t b);
  void unhold(int32_t b);           // a request lets go; releases the block at 0
  void release(int32_t b);          // held by no request: cached if indexed, else free
  void lru_push_back(int32_t b);
  void lru_remove(int32_t b);
  void leaf_push(int32_t b);
  bool evict_one();
  void index_prompt_blocks(int32_t req);
  std::string key(uint64_t ns, int32_t parent, const int32_t* tokens) const;
  int32_t lookup(uint64_t ns, int32_t parent, const int32_t* tokens) const;

  int32_t capacity_, block_size_, max_blocks_per_req_;
  std::vector<int32_t> ring_;
  int32_t head_, count_;
  std::unordered_map<int32_t, ReqBlocks> reqs_;
  std::vector<PlanEntry> plan_;
  bool open_ = false;
  int64_t reserved_ = 0, live_ = 0, alloc_failures_ = 0, peak_used_ = 0;

  // per block
  std::vector<int32_t> holders_;    // requests holding it in their committed tables
  std::vector<int32_t> children_;   // indexed blocks that extend it
  std::vector<int32_t> parent_;     // the indexed block it extends (-1: root); -2 if not indexed
  std::vector<std::string> key_of_;
  std::vector<int32_t> lru_prev_, lru_next_;
  std::vector<uint8_t> in_cache_;
  int32_t lru_head_ = -1, lru_tail_ = -1;
  int64_t cached_ = 0;
  // Eviction candidates: (release sequence number, block) in a min-heap, so
  // the oldest-released cached leaf is found without walking the cached
  // list.  Entries go stale when their block leaves the cache, gains an
  // indexed child or is released again (new sequence number); evict_one()
  // drops stale entries as it meets them, and the heap is rebuilt from the
  // cached list when stale entries outnumber live ones.
  std::vector<uint64_t> cache_seq_;
  uint64_t next_seq_ = 0;
  std::vector<std::pair<uint64_t, int32_t>> leaves_;
  // prefix index: key (namespace, parent, block_size tokens) -> block
  std::unordered_map<std::string, int32_t> index_;
  int64_t lookups_ = 0, hits_ = 0, matched_tokens_ = 0, evictions_ = 0, cow_copies_ = 0;
  // CPU pool for swapping: a FIFO free list (front to take, back to release)
  int32_t cpu_capacity_;
  std::vector<int32_t> cpu_ring_;
  int32_t cpu_head_ = 0, cpu_count_ = 0;
  std::unordered_map<int32_t, Swapped> swapped_;
};

}  // namespace pkv

// The opaque handle of the C interface wraps exactly one allocator.
struct pkv_alloc {
  pkv::Allocator impl;
  pkv_alloc(int32_t nb, int32_t bs, int32_t mb, int32_t ncpu = 0) : impl(nb, bs, mb, ncpu) {}
};
