// C ABI of the device entry points: argument checks, workspace layout, TMA
// descriptors and kernel launches.  See include/pkv.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "kernels.h"
#include "pkv_error.h"

namespace pkv {
namespace {

constexpr int kVersion = 1;
// error word, the prefill CTAs' two meeting counters, padding
constexpr size_t kHeaderBytes = 256;
constexpr int64_t kMaxTmaRows = 0x7fffffffLL;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct WorkspaceLayout {
  size_t counters, part_ml, part_o, total;
  int64_t slots;
};

WorkspaceLayout workspace_layout(int32_t num_reqs, int32_t num_heads, int32_t head_dim, int grid) {
  WorkspaceLayout w;
  w.slots = static_cast<int64_t>(grid) + num_reqs;
  w.counters = kHeaderBytes;
  w.part_ml = w.counters + align256(sizeof(int32_t) * static_cast<size_t>(num_reqs) * num_heads);
  w.part_o = w.part_ml + align256(sizeof(float) * 2 * static_cast<size_t>(w.slots) * num_heads);
  w.total = w.part_o + align256(sizeof(float) * static_cast<size_t>(w.slots) * num_heads * head_dim);
  return w;
}

// The layout a call uses is the one of the largest batch the workspace can
// hold, not of the call's own batch: the split counters must sit at the same
// place in every call that shares a workspace, or the partials of a small
// batch would land on counters a later, larger batch expects to find zero.
bool layout_for_capacity(size_t bytes, int32_t num_reqs, int32_t num_heads, int32_t head_dim,
                         int grid, WorkspaceLayout* out) {
  if (workspace_layout(num_reqs, num_heads, head_dim, grid).total > bytes) return false;
  int64_t lo = num_reqs, hi = num_reqs;  // layout(lo) fits
  while (hi < (int64_t(1) << 30) &&
         workspace_layout(static_cast<int32_t>(hi * 2 + 1), num_heads, head_dim, grid).total <= bytes)
    hi = hi * 2 + 1;
  hi = hi * 2 + 2;                        // layout(hi) does not fit (or hi is past the search)
  while (hi - lo > 1) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (mid < (int64_t(1) << 30) &&
        workspace_layout(static_cast<int32_t>(mid), num_heads, head_dim, grid).total <= bytes)
      lo = mid;
    else
      hi = mid;
  }
  *out = workspace_layout(static_cast<int32_t>(lo), num_heads, head_dim, grid);
  return true;
}

int current_grid() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  return decode_grid_size(dev);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// One paged block of one cache, all heads, as a single box: the 4-D view
// (64 dims, num_blocks * block_size tokens, head_dim / 64 halves, num_kv_heads)
// with strides (2 B, row, 128 B, head_dim * 2 B) and box (64, block_size,
// head_dim / 64, num_kv_heads).  The box lands as [head][half][token][128 B],
// 128-byte swizzled: one copy per block and cache instead of one per head and
// 64-dim half.
int encode_cache_block_map(CUtensorMap* map, const void* base, int64_t num_blocks,
                           int32_t block_size, int32_t hkv, int32_t d) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t row = static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(hkv);
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(num_blocks * block_size),
                        static_cast<cuuint64_t>(d / 64), static_cast<cuuint64_t>(hkv)};
  cuuint64_t strides[3] = {row, 128, static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(block_size), static_cast<cuuint32_t>(d / 64),
                       static_cast<cuuint32_t>(hkv)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_E_CUDA, "cuTensorMapEncodeTiled (block) failed (%d)", int(r));
  return PKV_OK;
}

// One head of one 16-token paged block as a single box laid out for a
// K-major tensor-core operand: the 5-D view (64 dims, 8 tokens, head_dim / 64
// halves, num_kv_heads, num_blocks * 2 half-blocks) with strides (2 B, row,
// 128 B, head_dim * 2 B, 8 rows) and box (64, 8, head_dim / 64, 1, 2).  The
// box lands as [token half][dim half][8 tokens][128 B]: consecutive groups of
// 8 keys sit head_dim / 64 KiB apart whichever dim half is read.
int encode_cache_head_map(CUtensorMap* map, const void* base, int64_t num_blocks,
                          int32_t block_size, int32_t hkv, int32_t d) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (block_size != 16) return fail(PKV_E_UNSUPPORTED, "block_size must be 16");
  const cuuint64_t row = static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(hkv);
  cuuint64_t dims[5] = {64, 8, static_cast<cuuint64_t>(d / 64), static_cast<cuuint64_t>(hkv),
                        static_cast<cuuint64_t>(num_blocks * 2)};
  cuuint64_t strides[4] = {row, 128, static_cast<cuuint64_t>(d) * 2, row * 8};
  cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(d / 64), 1, 2};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_E_CUDA, "cuTensorMapEncodeTiled (head) failed (%d)", int(r));
  return PKV_OK;
}

// The [T, H, D] query (token stride q_stride elements) as a 3-D tensor
// (D, H, T), box = 64 dims x G heads x 128/G tokens, 128-byte swizzle: one box
// is the 128-row (token, head-in-group) tile of the prefill kernel.
int encode_query_map(CUtensorMap* map, const void* q, int64_t q_stride, int64_t num_tokens,
                     int32_t num_heads, int32_t group, int32_t d) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(num_heads),
                        static_cast<cuuint64_t>(num_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(q_stride) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(128 / group)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_E_CUDA, "cuTensorMapEncodeTiled (query) failed (%d)", int(r));
  return PKV_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// PKV_VALIDATE=1 in the environment: after its launches an entry point waits
// for its stream, reads its device error word (one device-to-host copy) and
// turns any PKV_ERR_* bit into PKV_E_INVALID.  Off by default, so no call
// synchronises.
bool validate_enabled() {
  const char* v = std::getenv("PKV_VALIDATE");
  return v && v[0] == '1';
}

int validate_error_word(const uint32_t* word, cudaStream_t stream, const char* where) {
  if (!word || !validate_enabled()) return PKV_OK;
  uint32_t bits = 0;
  cudaError_t e = cudaMemcpyAsync(&bits, word, sizeof(bits), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, where);
  if (bits)
    return fail(PKV_E_INVALID, "%s: the kernels reported error bits 0x%x (1 block id, 2 slot, "
                "4 metadata, 8 timeout, 16 position)", where, bits);
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_last_error(void) { return last_error_slot().c_str(); }

int pkv_version(void) { return kVersion; }

int pkv_reshape_and_cache(const void* key, const void* value, int64_t key_stride,
                          int64_t value_stride, void* key_cache, void* value_cache,
                          const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                          int32_t dtype, uint32_t* error_word, void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PKV_E_INVALID, "pkv_reshape_and_cache: sizes must be positive");
  if (dtype != PKV_F32 && dtype != PKV_BF16)
    return fail(PKV_E_UNSUPPORTED, "pkv_reshape_and_cache: dtype %d", dtype);
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping)
    return fail(PKV_E_INVALID, "pkv_reshape_and_cache: null pointer");
  const int64_t esize = dtype == PKV_F32 ? 4 : 2;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * esize;
  if (row_bytes % 16 || (key_stride * esize) % 16 || (value_stride * esize) % 16 ||
      !aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_E_INVALID, "pkv_reshape_and_cache: rows, strides and bases must be 16-byte aligned");
  if (key_stride < num_kv_heads * static_cast<int64_t>(head_dim) ||
      value_stride < num_kv_heads * static_cast<int64_t>(head_dim))
    return fail(PKV_E_INVALID, "pkv_reshape_and_cache: token stride shorter than a row");
  cudaError_t e = launch_reshape_and_cache(key, value, key_stride * esize, value_stride * esize,
                                           key_cache, value_cache, slot_mapping, num_tokens,
                                           num_blocks * block_size, row_bytes, error_word,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
  return validate_error_word(error_word, static_cast<cudaStream_t>(stream), "reshape_and_cache");
}

int pkv_rope_reshape_and_cache(const int64_t* positions, void* query, int64_t query_stride,
                               int32_t num_heads, const void* key, int64_t key_stride,
                               void* key_out, const void* value, int64_t value_stride,
                               void* key_cache, void* value_cache, const int64_t* slot_mapping,
                               const float* cos_sin_cache, int64_t max_position,
                               int32_t rotary_dim, int32_t is_neox, int64_t num_tokens,
                               int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                               int32_t head_dim, int32_t dtype, uint32_t* error_word,
                               void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_heads <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0 || max_position <= 0)
    return fail(PKV_E_INVALID, "pkv_rope_reshape_and_cache: sizes must be positive");
  if (dtype != PKV_F32 && dtype != PKV_BF16)
    return fail(PKV_E_UNSUPPORTED, "pkv_rope_reshape_and_cache: dtype %d", dtype);
  if (rotary_dim <= 0 || rotary_dim > head_dim || rotary_dim % 2)
    return fail(PKV_E_INVALID, "pkv_rope_reshape_and_cache: rotary_dim %d (head_dim %d)",
                rotary_dim, head_dim);
  const int64_t esize = dtype == PKV_F32 ? 4 : 2;
  const int64_t item = (is_neox ? rotary_dim / 2 : rotary_dim) * esize;
  if ((head_dim * esize) % 16 || item % 16)
    return fail(PKV_E_UNSUPPORTED,
                "pkv_rope_reshape_and_cache: head_dim and the rotated %s must be multiples of "
                "16 bytes", is_neox ? "half" : "part");
  if (num_tokens == 0) return PKV_OK;
  if (!positions || !query || !key || !value || !key_cache || !value_cache || !slot_mapping ||
      !cos_sin_cache)
    return fail(PKV_E_INVALID, "pkv_rope_reshape_and_cache: null pointer");
  if ((query_stride * esize) % 16 || (key_stride * esize) % 16 || (value_stride * esize) % 16 ||
      !aligned16(query) || !aligned16(key) || !aligned16(value) || !aligned16(key_cache) ||
      !aligned16(value_cache) || !aligned16(cos_sin_cache) || (key_out && !aligned16(key_out)))
    return fail(PKV_E_INVALID, "pkv_rope_reshape_and_cache: strides and bases must be 16-byte aligned");
  const int64_t kv_row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (query_stride < static_cast<int64_t>(num_heads) * head_dim || key_stride < kv_row ||
      value_stride < kv_row)
    return fail(PKV_E_INVALID, "pkv_rope_reshape_and_cache: token stride shorter than a row");
  RopeArgs a;
  a.positions = positions;
  a.query = query;
  a.query_stride = query_stride;
  a.key = key;
  a.key_stride = key_stride;
  a.key_out = key_out;
  a.value = value;
  a.value_stride = value_stride;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.slot_mapping = slot_mapping;
  a.cos_sin_cache = cos_sin_cache;
  a.max_position = max_position;
  a.num_tokens = num_tokens;
  a.num_slots = num_blocks * block_size;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.rotary_dim = rotary_dim;
  a.is_neox = is_neox != 0;
  a.bf16 = dtype == PKV_BF16;
  a.err = error_word;
  cudaError_t e = launch_rope_reshape_and_cache(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope_reshape_and_cache launch");
  return validate_error_word(error_word, static_cast<cudaStream_t>(stream), "rope_reshape_and_cache");
}

int pkv_copy_blocks(const void* src_key_cache, const void* src_value_cache, void* dst_key_cache,
                    void* dst_value_cache, const int32_t* block_pairs, int32_t num_pairs,
                    int64_t src_num_blocks, int64_t dst_num_blocks, int64_t block_bytes,
                    uint32_t* error_word, void* stream) {
  if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_bytes <= 0 ||
      block_bytes % 16)
    return fail(PKV_E_INVALID, "pkv_copy_blocks: bad sizes");
  if (num_pairs == 0) return PKV_OK;
  if (!src_key_cache || !src_value_cache || !dst_key_cache || !dst_value_cache || !block_pairs)
    return fail(PKV_E_INVALID, "pkv_copy_blocks: null pointer");
  if (!aligned16(src_key_cache) || !aligned16(src_value_cache) || !aligned16(dst_key_cache) ||
      !aligned16(dst_value_cache))
    return fail(PKV_E_INVALID, "pkv_copy_blocks: pools must be 16-byte aligned");
  cudaError_t e = launch_copy_blocks(src_key_cache, src_value_cache, dst_key_cache,
                                     dst_value_cache, block_pairs, num_pairs, block_bytes,
                                     src_num_blocks, dst_num_blocks, error_word,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return validate_error_word(error_word, static_cast<cudaStream_t>(stream), "copy_blocks");
}

size_t pkv_attention_workspace_bytes(int32_t num_reqs, int32_t num_heads, int32_t head_dim) {
  if (num_reqs < 0 || num_heads <= 0 || head_dim <= 0) return 0;
  return workspace_layout(num_reqs, num_heads, head_dim, current_grid()).total;
}

static int paged_attention_launch(const void* q, int64_t q_stride, const void* key_cache,
                               const void* value_cache, const int32_t* block_table,
                               int32_t block_table_stride, const int32_t* query_start_loc,
                               const int32_t* seq_lens, const int32_t* num_computed_tokens,
                               float scale, void* out, int64_t out_stride, int64_t num_tokens,
                               int32_t num_reqs, int64_t num_blocks, int32_t block_size,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t dtype, int32_t max_query_len, void* workspace,
                               size_t workspace_bytes, void* stream,
                               const CacheWrite* write = nullptr) {
  if (num_tokens < 0 || num_reqs < 0 || num_blocks <= 0 || num_heads <= 0 || num_kv_heads <= 0)
    return fail(PKV_E_INVALID, "pkv_paged_attention_varlen: bad sizes");
  if (dtype != PKV_F32 && dtype != PKV_BF16)
    return fail(PKV_E_UNSUPPORTED, "pkv_paged_attention_varlen: dtype %d", dtype);
  if (block_size != 16) return fail(PKV_E_UNSUPPORTED, "block_size must be 16 (got %d)", block_size);
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_E_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", head_dim);
  if (num_heads % num_kv_heads) return fail(PKV_E_INVALID, "num_heads %% num_kv_heads != 0");
  if (num_blocks * block_size > kMaxTmaRows)
    return fail(PKV_E_UNSUPPORTED, "pool of %lld blocks is too large", static_cast<long long>(num_blocks));
  if (!workspace) return fail(PKV_E_WORKSPACE, "workspace is required");
  const int grid = current_grid();
  WorkspaceLayout wl;
  if (!layout_for_capacity(workspace_bytes, num_reqs, num_heads, head_dim, grid, &wl))
    return fail(PKV_E_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes,
                workspace_layout(num_reqs, num_heads, head_dim, grid).total);
  if (num_tokens == 0 || num_reqs == 0) return PKV_OK;
  if (!q || !key_cache || !value_cache || !block_table || !query_start_loc || !seq_lens ||
      !num_computed_tokens || !out)
    return fail(PKV_E_INVALID, "pkv_paged_attention_varlen: null pointer");
  const int64_t row = static_cast<int64_t>(num_heads) * head_dim;
  if (q_stride < row || out_stride < row || q_stride % 8 || out_stride % 8 || !aligned16(q) ||
      !aligned16(out) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_E_INVALID, "q/out/caches must be 16-byte aligned with strides >= heads*dim, multiple of 8");
  if (block_table_stride <= 0) return fail(PKV_E_INVALID, "block_table_stride must be positive");

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The cache write of this step's tokens fuses into the bf16 attention
  // kernel; for fp32 reshape_and_cache runs first, launched only once every
  // check of the call has passed.
  const bool fuse_write = write && dtype == PKV_BF16;
  auto write_first = [&]() -> int {
    if (!write || fuse_write) return PKV_OK;
    const int64_t esize = dtype == PKV_F32 ? 4 : 2;
    cudaError_t e = launch_reshape_and_cache(
        write->key, write->value, write->key_stride * esize, write->value_stride * esize,
        const_cast<void*>(key_cache), const_cast<void*>(value_cache), write->slot_mapping,
        num_tokens, num_blocks * block_size, static_cast<int64_t>(num_kv_heads) * head_dim * esize,
        reinterpret_cast<uint32_t*>(ws), st);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "reshape_and_cache launch");
  };
  AttnArgs a;
  a.q = q;
  a.q_stride = q_stride;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.qsl = query_start_loc;
  a.seq_lens = seq_lens;
  a.num_computed = num_computed_tokens;
  a.out = out;
  a.out_stride = out_stride;
  a.num_tokens = num_tokens;
  a.num_reqs = num_reqs;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.err = reinterpret_cast<uint32_t*>(ws);

  if (dtype == PKV_F32) {
    const int wrc = write_first();
    if (wrc != PKV_OK) return wrc;
    cudaError_t e = launch_attn_rows(a, false, false, st);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "attention launch");
  }

  // bf16: decode rows on the split-KV kernel, longer rows on the prefill path
  const int group = num_heads / num_kv_heads;
  if (num_kv_heads > 8 || group > 16 || (group & (group - 1)))
    return fail(PKV_E_UNSUPPORTED, "bf16 path supports num_kv_heads <= 8 and G in {1,2,4,8,16}");
  CUtensorMap kblk, vblk;
  int rc = encode_cache_block_map(&kblk, key_cache, num_blocks, block_size, num_kv_heads, head_dim);
  if (rc != PKV_OK) return rc;
  rc = encode_cache_block_map(&vblk, value_cache, num_blocks, block_size, num_kv_heads, head_dim);
  if (rc != PKV_OK) return rc;
  DecodeScratch ds;
  ds.counters = reinterpret_cast<int32_t*>(ws + wl.counters);
  ds.part_ml = reinterpret_cast<float*>(ws + wl.part_ml);
  ds.part_o = reinterpret_cast<float*>(ws + wl.part_o);
  ds.num_slots = wl.slots;
  // A call with rows of query length > 1 runs one persistent kernel whose
  // CTAs split between the prefill tiles and the decode rows on the device;
  // a decode-only call runs the split-KV decode kernel.  Either is launched
  // as a programmatic dependent of the kernel before it: its set-up and plan
  // read only metadata, and its copies of Q, K and V wait for that kernel
  // (for instance reshape_and_cache) to complete.
  cudaError_t e = cudaSuccess;
  if (max_query_len != 1) {
    CUtensorMap qmap, kmap, vmap;
    rc = encode_query_map(&qmap, q, q_stride, num_tokens, num_heads, num_heads / num_kv_heads,
                          head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_head_map(&kmap, key_cache, num_blocks, block_size, num_kv_heads, head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_head_map(&vmap, value_cache, num_blocks, block_size, num_kv_heads, head_dim);
    if (rc != PKV_OK) return rc;
    e = launch_varlen_bf16(a, qmap, kmap, vmap, kblk, vblk, ds, grid, st,
                           fuse_write ? write : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "varlen attention launch");
    return PKV_OK;
  }
  e = launch_decode_bf16(a, kblk, vblk, ds, grid, st, fuse_write ? write : nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PKV_OK;
}

int pkv_paged_attention_varlen(const void* q, int64_t q_stride, const void* key_cache,
                               const void* value_cache, const int32_t* block_table,
                               int32_t block_table_stride, const int32_t* query_start_loc,
                               const int32_t* seq_lens, const int32_t* num_computed_tokens,
                               float scale, void* out, int64_t out_stride, int64_t num_tokens,
                               int32_t num_reqs, int64_t num_blocks, int32_t block_size,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t dtype, int32_t max_query_len, void* workspace,
                               size_t workspace_bytes, void* stream) {
  const int rc = paged_attention_launch(
      q, q_stride, key_cache, value_cache, block_table, block_table_stride, query_start_loc,
      seq_lens, num_computed_tokens, scale, out, out_stride, num_tokens, num_reqs, num_blocks,
      block_size, num_heads, num_kv_heads, head_dim, dtype, max_query_len, workspace,
      workspace_bytes, stream);
  if (rc != PKV_OK || num_tokens == 0 || num_reqs == 0) return rc;
  return validate_error_word(static_cast<const uint32_t*>(workspace),
                             static_cast<cudaStream_t>(stream), "paged_attention_varlen");
}

int pkv_reshape_and_cache_paged_attention(
    const void* key, int64_t key_stride, const void* value, int64_t value_stride,
    const int64_t* slot_mapping, const void* q, int64_t q_stride, void* key_cache,
    void* value_cache, const int32_t* block_table, int32_t block_table_stride,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* num_computed_tokens,
    float scale, void* out, int64_t out_stride, int64_t num_tokens, int32_t num_reqs,
    int64_t num_blocks, int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t dtype, int32_t max_query_len, void* workspace,
    size_t workspace_bytes, void* stream) {
  if (num_tokens > 0) {
    if (!key || !value || !slot_mapping)
      return fail(PKV_E_INVALID, "pkv_reshape_and_cache_paged_attention: null pointer");
    const int64_t esize = dtype == PKV_F32 ? 4 : 2;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (!aligned16(key) || !aligned16(value) || (key_stride * esize) % 16 ||
        (value_stride * esize) % 16 || (row * esize) % 16)
      return fail(PKV_E_INVALID,
                  "pkv_reshape_and_cache_paged_attention: key/value rows, strides and bases must "
                  "be 16-byte aligned");
    if (key_stride < row || value_stride < row)
      return fail(PKV_E_INVALID,
                  "pkv_reshape_and_cache_paged_attention: token stride shorter than a row");
  }
  CacheWrite w;
  w.key = key;
  w.value = value;
  w.key_stride = key_stride;
  w.value_stride = value_stride;
  w.slot_mapping = slot_mapping;
  const int rc = paged_attention_launch(
      q, q_stride, key_cache, value_cache, block_table, block_table_stride, query_start_loc,
      seq_lens, num_computed_tokens, scale, out, out_stride, num_tokens, num_reqs, num_blocks,
      block_size, num_heads, num_kv_heads, head_dim, dtype, max_query_len, workspace,
      workspace_bytes, stream, &w);
  if (rc != PKV_OK || num_tokens == 0 || num_reqs == 0) return rc;
  return validate_error_word(static_cast<const uint32_t*>(workspace),
                             static_cast<cudaStream_t>(stream), "reshape_and_cache_paged_attention");
}

}  // extern "C"
