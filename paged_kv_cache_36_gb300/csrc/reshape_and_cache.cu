// reshape_and_cache: scatter this step's K/V rows into the paged cache.
//
// "AI Infra入门干货总结：大模型是如何高效推理的", section "Attention Module": after
// the QKV split and RoPE, reshape_and_cache writes the new K/V into the paged
// KV cache by slot_mapping; section "Paged Attention": slot_idx =
// block_idx * block_size + block_offset, with the cache of one layer laid out
// [num_blocks, block_size, num_kv_heads, head_dim].
//
// One CTA per token.  A token's key row and value row (num_kv_heads *
// head_dim elements each, 2 KiB for 8 x 128 bf16) are contiguous both in the
// input and at the destination slot, so the copy is a run of 16-byte vector
// loads and stores: consecutive threads move consecutive 16-byte chunks and
// every warp access is fully coalesced.  Padding tokens (slot < 0) are
// skipped; slots past the pool set PKV_ERR_SLOT and are skipped.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value, int64_t key_stride_v,
    int64_t value_stride_v, uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
    const int64_t* __restrict__ slot_mapping, int64_t num_tokens, int64_t num_slots,
    int32_t vec_per_row, uint32_t* __restrict__ err) {
  // an attention kernel launched as this one's programmatic dependent may
  // start its prologue now; it waits for this grid before reading the caches
  if (threadIdx.x == 0) grid_launch_dependents();
  for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (threadIdx.x == 0 && err) atomicOr(err, PKV_ERR_SLOT);
      continue;
    }
    const uint4* ksrc = key + t * key_stride_v;
    const uint4* vsrc = value + t * value_stride_v;
    uint4* kdst = key_cache + slot * vec_per_row;
    uint4* vdst = value_cache + slot * vec_per_row;
    for (int32_t i = threadIdx.x; i < vec_per_row; i += blockDim.x) {
      const uint4 kv = __ldg(ksrc + i);
      const uint4 vv = __ldg(vsrc + i);
      kdst[i] = kv;
      vdst[i] = vv;
    }
  }
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t key_stride_b,
                                     int64_t value_stride_b, void* key_cache, void* value_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     int64_t num_slots, int64_t row_bytes, uint32_t* err,
                                     cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int32_t vpr = static_cast<int32_t>(row_bytes / 16);
  int threads = ((vpr + 31) / 32) * 32;
  if (threads > 256) threads = 256;
  const int64_t grid = num_tokens < 1048576 ? num_tokens : 1048576;
  reshape_and_cache_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), key_stride_b / 16,
      value_stride_b / 16, static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache),
      slot_mapping, num_tokens, num_slots, vpr, err);
  return cudaGetLastError();
}

}  // namespace pkv
