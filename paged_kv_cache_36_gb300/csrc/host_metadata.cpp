// slot_mapping builder for a flattened batch (host).
//
// "AI Infra入门干货总结：大模型是如何高效推理的", section "Paged Attention": the
// slot of absolute position pos of request r is
//   block_table[r][pos / block_size] * block_size + pos % block_size.
// Request r's tokens in this step sit at positions num_computed_tokens[r] + k
// for k < query_start_loc[r + 1] - query_start_loc[r].
#include <cstdint>

#include "pkv_error.h"

extern "C" int pkv_build_slot_mapping(const int32_t* block_table, int32_t stride,
                                      const int32_t* qsl, const int32_t* num_computed,
                                      int32_t num_reqs, int32_t block_size, int64_t* slots,
                                      int64_t num_tokens) {
  using pkv::fail;
  if (num_reqs < 0 || block_size <= 0 || stride < 0 || num_tokens < 0)
    return fail(PKV_E_INVALID, "pkv_build_slot_mapping: bad sizes");
  if (num_reqs > 0 && (!block_table || !qsl || !num_computed))
    return fail(PKV_E_INVALID, "pkv_build_slot_mapping: null input");
  if (num_tokens > 0 && !slots) return fail(PKV_E_INVALID, "pkv_build_slot_mapping: null output");
  if (num_reqs > 0 && (qsl[0] != 0 || qsl[num_reqs] != num_tokens))
    return fail(PKV_E_INVALID, "pkv_build_slot_mapping: query_start_loc disagrees with num_tokens");
  for (int32_t r = 0; r < num_reqs; ++r) {
    const int64_t a = qsl[r], b = qsl[r + 1];
    if (b < a) return fail(PKV_E_INVALID, "query_start_loc decreases at request %d", r);
    const int32_t* row = block_table + static_cast<int64_t>(r) * stride;
    for (int64_t t = a; t < b; ++t) {
      const int64_t pos = static_cast<int64_t>(num_computed[r]) + (t - a);
      const int64_t logical = pos / block_size;
      if (logical >= stride)
        return fail(PKV_E_INVALID, "request %d position %lld is past its block-table row", r,
                    static_cast<long long>(pos));
      slots[t] = static_cast<int64_t>(row[logical]) * block_size + pos % block_size;
    }
  }
  return PKV_OK;
}
