// Paged attention on CUDA cores, one warp per (query row, query head).
//
// This is the float32 path of paged_attention_varlen (float32 needs 1e-5
// accuracy, which bf16/tf32 tensor-core tiles cannot give).  It computes the
// same thing as the bf16 kernels ("AI Infra入门干货总结：大模型是如何高效推理的",
// section "Attention Module"; "Chunked Prefill 与 Preemption", section "Chunked
// Prefill：改变调度粒度，不改变 causal 结果"): query row t of request r at absolute
// position p = num_computed[r] + (t - query_start_loc[r]) attends keys
// j = 0..p of its KV head g = h / G, read through block_table, with an online
// softmax (running max and sum, rescaled as each key arrives).
//
// Each lane owns head_dim / 32 dimensions; the dot product is a warp
// all-reduce.  Keys are visited one at a time, so this kernel is meant for
// small problems.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16& d, float x) { d = __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_rows_kernel(const AttnArgs a, int skip_decode,
                                                        float scale_log2) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t t = wid / a.num_heads;
  const int h = static_cast<int>(wid - t * a.num_heads);
  if (t >= a.num_tokens) return;

  // request of row t: the largest r with qsl[r] <= t
  int lo = 0, hi = a.num_reqs;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.qsl + mid) <= t) lo = mid; else hi = mid;
  }
  const int r = lo;
  const int q0 = __ldg(a.qsl + r);
  const int qlen = __ldg(a.qsl + r + 1) - q0;
  if (skip_decode && qlen == 1) return;
  const int nc = __ldg(a.num_computed + r);
  const int seq = __ldg(a.seq_lens + r);
  if (seq != nc + qlen || (seq + a.block_size - 1) / a.block_size > a.bt_stride) {
    if (lane == 0) atomicOr(a.err, PKV_ERR_METADATA);
    return;
  }
  const int pos = nc + static_cast<int>(t - q0);
  const int G = a.num_heads / a.num_kv_heads;
  const int g = h / G;

  const T* qrow = static_cast<const T*>(a.q) + t * a.q_stride + static_cast<int64_t>(h) * D;
  float qv[E];
#pragma unroll
  for (int i = 0; i < E; ++i) qv[i] = to_f32(qrow[lane + 32 * i]);

  const T* kc = static_cast<const T*>(a.key_cache);
  const T* vc = static_cast<const T*>(a.value_cache);
  const int32_t* row = a.block_table + static_cast<int64_t>(r) * a.bt_stride;
  const int64_t tok_stride = static_cast<int64_t>(a.num_kv_heads) * D;
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;

  for (int j = 0; j <= pos; ++j) {
    const int32_t blk = __ldg(row + j / a.block_size);
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) atomicOr(a.err, PKV_ERR_BLOCK_ID);
      continue;
    }
    const int64_t off = (static_cast<int64_t>(blk) * a.block_size + j % a.block_size) * tok_stride +
                        static_cast<int64_t>(g) * D;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) dot += qv[i] * to_f32(kc[off + lane + 32 * i]);
#pragma unroll
    for (int sh = 16; sh; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
    const float s = dot * scale_log2;
    const float mn = fmaxf(m, s);
    const float alpha = exp2f(m - mn);
    const float pj = exp2f(s - mn);
    l = l * alpha + pj;
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = acc[i] * alpha + pj * to_f32(vc[off + lane + 32 * i]);
    m = mn;
  }
  T* orow = static_cast<T*>(a.out) + t * a.out_stride + static_cast<int64_t>(h) * D;
  const float inv = 1.f / l;
#pragma unroll
  for (int i = 0; i < E; ++i) from_f32(orow[lane + 32 * i], acc[i] * inv);
}

cudaError_t launch_attn_rows(const AttnArgs& a, bool bf16, bool skip_decode, cudaStream_t stream) {
  const int64_t warps = a.num_tokens * a.num_heads;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps + (threads / 32) - 1) / (threads / 32);
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  const int sd = skip_decode ? 1 : 0;
  const unsigned grid = static_cast<unsigned>(blocks);
  if (bf16) {
    if (a.head_dim == 128)
      attn_rows_kernel<__nv_bfloat16, 128><<<grid, threads, 0, stream>>>(a, sd, scale_log2);
    else if (a.head_dim == 64)
      attn_rows_kernel<__nv_bfloat16, 64><<<grid, threads, 0, stream>>>(a, sd, scale_log2);
    else
      return cudaErrorNotSupported;
  } else {
    if (a.head_dim == 128)
      attn_rows_kernel<float, 128><<<grid, threads, 0, stream>>>(a, sd, scale_log2);
    else if (a.head_dim == 64)
      attn_rows_kernel<float, 64><<<grid, threads, 0, stream>>>(a, sd, scale_log2);
    else
      return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

}  // namespace pkv
