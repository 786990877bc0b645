// copy_blocks: copy whole KV blocks (K and V) between two block pools, or
// within one.
//
// "显存与调度" (ch. 32), section "共享前缀会改变块的所有权": a shared block that is
// still being written is copied before the write (copy-on-write); the
// allocator lists the (source, destination) pairs of a plan and this kernel
// moves them before the step's cache writes.  The same call moves blocks
// between the HBM pool and a pool in mapped pinned host memory (offload and
// reload, "Chunked Prefill 与 Preemption" and "vLLM 抢占机制源码精读" on swap):
// the GPU reads and writes host memory directly over the CPU-GPU link, so a
// batch of scattered blocks is one launch, not one copy call per block.
//
// Work unit: a 16 KiB chunk of one block of one cache (K or V), taken by one
// CTA: 256 threads, each with four 16-byte loads in flight before its stores.
// The pools may be one and the same (copy-on-write), so their pointers are
// not marked as non-aliasing; the pairs are independent by contract.
// Units are spread over a grid sized to the SMs; a pair whose ids are out of
// range sets PKV_ERR_BLOCK_ID and is skipped.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int64_t kChunkVecs = kThreads * kUnroll;  // 16 KiB

__global__ void __launch_bounds__(kThreads)
    copy_blocks_kernel(const uint4* src_k, const uint4* src_v, uint4* dst_k, uint4* dst_v,
                       const int32_t* __restrict__ pairs, int32_t n, int64_t vecs_per_block,
                       int64_t src_blocks, int64_t dst_blocks, uint32_t* err) {
  const int64_t chunks = (vecs_per_block + kChunkVecs - 1) / kChunkVecs;
  const int64_t units = static_cast<int64_t>(n) * 2 * chunks;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t i = u / (2 * chunks);
    const int64_t rem = u - i * 2 * chunks;
    const int c = rem >= chunks;  // 0: K, 1: V
    const int64_t ch = rem - c * chunks;
    const int64_t s = __ldg(pairs + 2 * i), d = __ldg(pairs + 2 * i + 1);
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
      if (rem == 0 && threadIdx.x == 0 && err) atomicOr(err, PKV_ERR_BLOCK_ID);
      continue;
    }
    const uint4* src = (c ? src_v : src_k) + s * vecs_per_block;
    uint4* dst = (c ? dst_v : dst_k) + d * vecs_per_block;
    const int64_t base = ch * kChunkVecs + threadIdx.x;
    uint4 r[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t x = base + k * kThreads;
      if (x < vecs_per_block) r[k] = src[x];
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t x = base + k * kThreads;
      if (x < vecs_per_block) dst[x] = r[k];
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                               const int32_t* pairs, int32_t n, int64_t block_bytes,
                               int64_t src_blocks, int64_t dst_blocks, uint32_t* err,
                               cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t vpb = block_bytes / 16;
  const int64_t units = static_cast<int64_t>(n) * 2 * ((vpb + kChunkVecs - 1) / kChunkVecs);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident CTAs per SM
  const int64_t grid = units < cap ? units : cap;
  copy_blocks_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
      static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v),
      static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), pairs, n, vpb, src_blocks,
      dst_blocks, err);
  return cudaGetLastError();
}

}  // namespace pkv
