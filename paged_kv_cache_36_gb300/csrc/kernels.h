// Launchers of the device kernels, called by the C ABI in api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

namespace pkv {

// Raises the dynamic shared-memory limit of kernel `Kern` to `bytes`, once per
// device (the attribute is per function and device; setting it on every launch
// costs host time).
template <auto Kern>
cudaError_t raise_smem_limit_once(size_t bytes) {
  constexpr int kDevices = 64;
  static std::once_flag once[kDevices];
  static cudaError_t status[kDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    status[dev] = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  });
  return status[dev];
}

// Launches `kern` as a programmatic dependent of the kernel before it on
// `stream`: its blocks may become resident while that kernel finishes.  The
// kernel must execute griddepcontrol.wait before touching memory the kernel
// before it may read or write.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Everything an attention kernel needs about one paged_attention_varlen call.
struct AttnArgs {
  const void* q;
  int64_t q_stride;           // elements
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* num_computed;
  void* out;
  int64_t out_stride;         // elements
  int64_t num_tokens;
  int32_t num_reqs;
  int64_t num_blocks;
  int32_t block_size;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  float scale;
  uint32_t* err;              // device error word
};

// Scratch carved out of the caller's workspace for the split-KV decode.
struct DecodeScratch {
  int32_t* counters;          // [num_reqs], zero between calls
  float* part_o;              // [slots][num_heads][head_dim]
  float* part_ml;             // [slots][num_heads][2]: running max (log2 units), sum
  int64_t num_slots;          // = decode grid size + num_reqs
};

cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t key_stride_b,
                                     int64_t value_stride_b, void* key_cache, void* value_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     int64_t num_slots, int64_t row_bytes, uint32_t* err,
                                     cudaStream_t stream);

// Fused RoPE + reshape_and_cache (sizes and strides in elements).
struct RopeArgs {
  const int64_t* positions;
  void* query;
  int64_t query_stride;
  const void* key;
  int64_t key_stride;
  void* key_out;              // may be null
  const void* value;
  int64_t value_stride;
  void* key_cache;
  void* value_cache;
  const int64_t* slot_mapping;
  const float* cos_sin_cache;
  int64_t max_position;
  int64_t num_tokens;
  int64_t num_slots;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t rotary_dim;
  bool is_neox;
  bool bf16;
  uint32_t* err;
};

cudaError_t launch_rope_reshape_and_cache(const RopeArgs& a, cudaStream_t stream);

// Whole-block copies of K and V between two pools (or within one): block
// pairs[2i] of the source pool to block pairs[2i+1] of the destination pool.
cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                               const int32_t* pairs, int32_t n, int64_t block_bytes,
                               int64_t src_blocks, int64_t dst_blocks, uint32_t* err,
                               cudaStream_t stream);

// Grid size (CTAs) of the persistent split-KV decode kernel on this device.
int decode_grid_size(int device);

// This step's new K/V rows for a cache write fused into the decode kernel
// (strides in elements).
struct CacheWrite {
  const void* key;
  const void* value;
  int64_t key_stride;
  int64_t value_stride;
  const int64_t* slot_mapping;
};

// Split-KV decode of a call whose rows all have query length 1 (bf16, mma +
// TMA), launched as a programmatic dependent of the kernel before it.  With
// `write` set, the kernel also does reshape_and_cache of each decode token
// (its row goes to slot_mapping[token] and is used in place of the cache's
// copy of that position).
cudaError_t launch_decode_bf16(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               const DecodeScratch& ws, int grid, cudaStream_t stream,
                               const CacheWrite* write = nullptr);

// A call with rows of query length > 1 (bf16): one persistent kernel of
// `sms` CTAs whose CTAs split between chunked-prefill attention (tcgen05 +
// TMA + TMEM) of those rows and the split-KV decode of the rows of query
// length 1.  qmap is the [T, H, D] query as a (D, H, T) tensor map with a
// 64 x G x 128/G box; kmap/vmap the per-head cache maps; kblk/vblk the
// whole-block cache maps of the decode.  With `write` set the kernel also
// does the call's reshape_and_cache (every row's new K/V to its slot) before
// attending; words 1 and 2 of the workspace header (after the error word)
// are then the prefill CTAs' meeting counter.
cudaError_t launch_varlen_bf16(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, const CUtensorMap& kblk,
                               const CUtensorMap& vblk, const DecodeScratch& ws, int sms,
                               cudaStream_t stream, const CacheWrite* write = nullptr);

// CUDA-core attention, one warp per (query row, head); fp32 path for all rows,
// or only rows of requests with query length > 1 when skip_decode is set.
cudaError_t launch_attn_rows(const AttnArgs& a, bool bf16, bool skip_decode, cudaStream_t stream);

}  // namespace pkv
