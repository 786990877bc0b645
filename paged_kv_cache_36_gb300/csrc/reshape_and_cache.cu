// reshape_and_cache: scatter this step's K/V rows into the paged cache.
//
// "AI Infra入门干货总结：大模型是如何高效推理的", section "Attention Module": after
// the QKV split and RoPE, reshape_and_cache writes the new K/V into the paged
// KV cache by slot_mapping; section "Paged Attention": slot_idx =
// block_idx * block_size + block_offset, with the cache of one layer laid out
// [num_blocks, block_size, num_kv_heads, head_dim].
//
// One warp per token.  A token's key row and value row (num_kv_heads *
// head_dim elements each, 2 KiB for 8 x 128 bf16) are contiguous both in the
// input and at the destination slot, so the copy is a run of 16-byte vector
// loads and stores: consecutive lanes move consecutive 16-byte chunks and
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
  // This grid is itself a programmatic dependent of the kernel before it,
  // which may still read the cache or write the new rows: wait for it before
  // any load or store.
  grid_dependency_wait();
  // An attention kernel launched as this one's programmatic dependent may
  // start its prologue now (it waits for this grid before reading the
  // caches).  Released only after the wait above, so that prologue reads
  // metadata that work before this grid wrote.
  if (threadIdx.x == 0) grid_launch_dependents();
  // One warp per token.  The slot and up to four 16-byte chunks of the K row
  // and of the V row per lane are loaded together, so a token costs one
  // memory latency, not two; the stores follow once the slot is known.
  constexpr int kUnroll = 4;
  const int lane = threadIdx.x & 31;
  const int64_t wpb = blockDim.x >> 5;
  for (int64_t t = blockIdx.x * wpb + (threadIdx.x >> 5); t < num_tokens; t += gridDim.x * wpb) {
    const int64_t slot = __ldg(slot_mapping + t);
    const uint4* ksrc = key + t * key_stride_v;
    const uint4* vsrc = value + t * value_stride_v;
    const bool store = slot >= 0 && slot < num_slots;
    if (slot >= num_slots && lane == 0 && err) atomicOr(err, PKV_ERR_SLOT);
    uint4* kdst = key_cache + (store ? slot : 0) * vec_per_row;
    uint4* vdst = value_cache + (store ? slot : 0) * vec_per_row;
    for (int32_t base = 0; base < vec_per_row; base += 32 * kUnroll) {
      uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t i = base + u * 32 + lane;
        if (i < vec_per_row) {
          kr[u] = __ldg(ksrc + i);
          vr[u] = __ldg(vsrc + i);
        }
      }
      if (store) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int32_t i = base + u * 32 + lane;
          if (i < vec_per_row) {
            kdst[i] = kr[u];
            vdst[i] = vr[u];
          }
        }
      }
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
  constexpr int kThreads = 256;  // 8 warps, one token each per iteration
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (num_tokens + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident blocks per SM
  const int64_t grid = blocks < cap ? blocks : cap;
  return launch_programmatic(reshape_and_cache_kernel, dim3(static_cast<unsigned>(grid)),
                             dim3(kThreads), 0, stream, static_cast<const uint4*>(key),
                             static_cast<const uint4*>(value), key_stride_b / 16,
                             value_stride_b / 16, static_cast<uint4*>(key_cache),
                             static_cast<uint4*>(value_cache), slot_mapping, num_tokens, num_slots,
                             vpr, err);
}

}  // namespace pkv
