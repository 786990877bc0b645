// paged_attention_varlen for callers that cannot allocate device memory.
//
// Some callers have no way to provide a workspace.  Typical cases:
//   - an engine whose plugin or enqueue hook is forbidden to allocate;
//   - a server that handed every free byte of HBM to the KV block pool at
//     start-up;
//   - a latency-critical loop that must not risk the implicit
//     synchronisation and fragmentation a cudaMalloc / cudaFree can bring.
// This entry point serves them: the split-KV decode's scratch (split
// counters, per-split partial results and the error word) lives in one
// fixed array compiled into this library, so the caller passes only inputs
// and outputs.
//
// The array is file-scope `static __device__` memory of kStaticScratchBytes
// (16 MiB); every GPU that loads the library holds it until the process
// exits.  Batches whose scratch would not fit are rejected with
// PKV_E_WORKSPACE.  Host code cannot use the array's name as an address (on
// the host it is only a stand-in symbol), so the first call on each device
// asks the runtime for its device address with cudaGetSymbolAddress, with
// that device current, and keeps it.  Make that first call before any stream
// capture begins.
//
// All calls share the one array and it keeps the last call's contents.  Each
// call therefore clears the part that must start at zero (error word and
// split counters) with cudaMemsetAsync on the caller's stream before its
// kernels.  Two calls whose work overlaps on the GPU (other streams,
// concurrent graphs) race on the array: serialise them.
//
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pkv.h"
#include "pkv_error.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attention_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkv::fail(PKV_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pkv::fail(PKV_E_UNSUPPORTED, "device %d is beyond the %d supported", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attention_scratch);
    if (e != cudaSuccess || !p)
      return pkv::fail(PKV_E_CUDA, "cudaGetSymbolAddress of the static scratch: %s",
                       cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

// Bytes at the front of the scratch that must be zero when a call starts.
// pkv_paged_attention_varlen lays a workspace out for the largest batch it
// can hold, but the two parts that must start at zero sit at the front for
// every capacity: the 256-byte header with the error word, then the int32
// split counters, one per (request, KV head), at r * num_kv_heads + h.  A
// call touches only the counters of its own num_reqs requests, so clearing
// the header and those num_reqs * num_kv_heads counters is enough.
size_t zeroed_prefix_bytes(int32_t num_reqs, int32_t num_kv_heads) {
  const size_t counters = sizeof(int32_t) * static_cast<size_t>(num_reqs) * num_kv_heads;
  return 256 + ((counters + 255) & ~size_t(255));
}

}  // namespace

extern "C" int pkv_paged_attention_varlen_noalloc(
    const void* q, int64_t q_stride, const void* key_cache, const void* value_cache,
    const int32_t* block_table, int32_t block_table_stride, const int32_t* query_start_loc,
    const int32_t* seq_lens, const int32_t* num_computed_tokens, float scale, void* out,
    int64_t out_stride, int64_t num_tokens, int32_t num_reqs, int64_t num_blocks,
    int32_t block_size, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
    int32_t max_query_len, uint32_t* error_word, void* stream) {
  if (num_reqs < 0 || num_heads <= 0 || head_dim <= 0)
    return pkv::fail(PKV_E_INVALID, "pkv_paged_attention_varlen_noalloc: bad sizes");
  const size_t need = pkv_attention_workspace_bytes(num_reqs, num_heads, head_dim);
  if (need == 0 || need > kStaticScratchBytes)
    return pkv::fail(PKV_E_WORKSPACE,
                     "pkv_paged_attention_varlen_noalloc: this batch needs %zu bytes of scratch; "
                     "the static array holds %zu (use pkv_paged_attention_varlen with a workspace)",
                     need, kStaticScratchBytes);
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != PKV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (num_kv_heads <= 0 || num_kv_heads > num_heads)
    return pkv::fail(PKV_E_INVALID, "pkv_paged_attention_varlen_noalloc: bad num_kv_heads");
  cudaError_t e = cudaMemsetAsync(scratch, 0, zeroed_prefix_bytes(num_reqs, num_kv_heads), st);
  if (e != cudaSuccess)
    return pkv::fail(PKV_E_CUDA, "clearing the static scratch: %s", cudaGetErrorString(e));
  rc = pkv_paged_attention_varlen(q, q_stride, key_cache, value_cache, block_table,
                                  block_table_stride, query_start_loc, seq_lens,
                                  num_computed_tokens, scale, out, out_stride, num_tokens,
                                  num_reqs, num_blocks, block_size, num_heads, num_kv_heads,
                                  head_dim, dtype, max_query_len, scratch, kStaticScratchBytes,
                                  stream);
  if (rc != PKV_OK) return rc;
  if (error_word) {
    e = cudaMemcpyAsync(error_word, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess)
      return pkv::fail(PKV_E_CUDA, "copying the error word: %s", cudaGetErrorString(e));
  }
  return PKV_OK;
}
