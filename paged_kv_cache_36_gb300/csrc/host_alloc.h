// Host KV block allocator (see host_alloc.cpp for the accounting rules).
#pragma once

#include <cstdint>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace pkv {

class Allocator {
 public:
  Allocator(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_req);

  int reserve(int32_t n, const int32_t* ids, const int32_t* new_tokens);
  int commit();
  int rollback();
  int free_request(int32_t req);  // blocks released, >= 0
  void stats(pkv_alloc_stats* s) const;
  int table(int32_t req, int32_t* out, int32_t cap) const;
  const std::vector<int32_t>* blocks(int32_t req) const;  // committed + reserved, or null
  int64_t held_tokens(int32_t req) const;
  int free_list(int32_t* out, int32_t cap) const;
  int check() const;
  int32_t num_free() const { return count_; }
  int32_t block_size() const { return block_size_; }
  bool open() const { return open_; }

 private:
  struct ReqBlocks {
    std::vector<int32_t> blocks;  // committed blocks, then reserved ones
    int32_t committed = 0;        // how many of `blocks` are committed
    int64_t tokens = 0;           // T_i, committed tokens
  };
  struct PlanEntry {
    int32_t req;
    int32_t tokens;
    int32_t blocks;
  };

  int32_t pop_front();
  void push_back(int32_t b);
  void push_front(int32_t b);

  int32_t capacity_, block_size_, max_blocks_per_req_;
  std::vector<int32_t> ring_;
  int32_t head_, count_;
  std::unordered_map<int32_t, ReqBlocks> reqs_;
  std::vector<PlanEntry> plan_;
  bool open_ = false;
  int64_t reserved_ = 0, committed_ = 0, alloc_failures_ = 0, peak_used_ = 0;
};

}  // namespace pkv

// The opaque handle of the C interface wraps exactly one allocator.
struct pkv_alloc {
  pkv::Allocator impl;
  pkv_alloc(int32_t nb, int32_t bs, int32_t mb) : impl(nb, bs, mb) {}
};
