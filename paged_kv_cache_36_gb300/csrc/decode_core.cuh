// Split-KV paged decode attention (query length 1) with a fused log-sum-exp
// merge of the splits, bf16 inputs, fp32 accumulation: the body of one CTA,
// shared by the decode kernel and the mixed prefill/decode kernel.
//
// What it computes ("AI Infra入门干货总结：大模型是如何高效推理的", section
// "Attention Module"): for a decode request r (one query row at position
// seq_len - 1) and query head h with KV head g = h / G,
//   out = sum_j softmax_j(scale <q_h, K_r[j][g]>) V_r[j][g],  j < seq_len,
// with K_r / V_r read through block_table.  The closing remarks of the same
// page describe Flash-Decoding: split the KV dimension across SMs and merge the
// per-split results by log-sum-exp.
//
// Work split.  The decode requests' logical blocks are concatenated into one
// sequence of N blocks; persistent CTA c of P = min(grid, N) takes blocks
// [cN/P, (c+1)N/P), at least one each.
// Every CTA streams the same number of bytes whatever the context-length mix,
// and a request spanning several CTAs becomes several splits.  Each split's
// partial (running max m in log2 units, sum l, unnormalised o) goes to
// workspace slot c + r, which is unique because both c and r grow along the
// sequence.  A request that fits in one CTA is normalised and written
// directly.  Otherwise each consumer warp bumps a counter for its (request,
// KV head); the warp that completes the count merges all splits:
//   M = max_s m_s,  out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,
// then resets the counter to zero for the next call.
//
// Data movement.  In the [num_blocks, 16, Hkv, D] cache one physical block of
// all KV heads is one contiguous span (32 KiB for 8 x 128 bf16).  A producer
// warp fetches it with TMA tensor copies - one box of 16 tokens x 64 dims per
// (KV head, 64-dim half), 128-byte swizzled - into a ring of stages holding the
// K and V of one paged block, so every 16-token block is loaded whole and the
// block_table gather stays aligned.  The swizzle makes the per-head row
// accesses below bank-conflict free.
//
// Compute.  One consumer warp per KV head.  With the G query heads of that KV
// head as the N dimension, S^T = K Q^T (16 tokens x 8 heads, K = head_dim) and
// O^T += V^T P^T (head_dim x 8 heads, K = 16 tokens) are m16n8k16 warp MMAs
// fed by ldmatrix from the swizzled stage.  The online softmax runs per head
// column on the accumulator fragments, with the column max reduced by warp
// shuffles, and P is turned into the B operand of the second product by an
// in-register 8x8 transpose.  On GB300 this contraction is small enough
// that the tensor pipe is nearly idle; it is used so the CUDA cores are not
// the bottleneck when G = 8 (4 FMAs per KV byte).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

constexpr int kDecodeMaxStages = 4;
constexpr int kDecodeMaxReqs = 8192;
constexpr int kSmemBudget = 232448;  // 227 KiB opt-in per CTA

struct DecodeParams {
  const __nv_bfloat16* q;
  int64_t q_stride;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* num_computed;
  __nv_bfloat16* out;
  int64_t out_stride;
  int32_t num_reqs;
  int32_t num_blocks;
  int32_t num_heads;
  int32_t hkv;
  int32_t group;
  float scale_log2;
  int32_t* counters;  // [num_reqs * hkv]
  float* part_o;
  float* part_ml;
  uint32_t* err;
  int32_t stages;
  uint32_t stage_bytes;
  // Fused reshape_and_cache (k_new == nullptr: off).  Each decode token's new
  // K/V row is written to its slot and patched into the stage of its block.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t k_new_stride;  // elements per token
  int64_t v_new_stride;
  const int64_t* slot_mapping;
  __nv_bfloat16* key_cache;
  __nv_bfloat16* value_cache;
  int64_t num_slots;
};

// Fills the decode parameters of a call and the dynamic shared memory a CTA
// needs (as many K/V stages as fit in smem_budget, at most kDecodeMaxStages).
// write: fused reshape_and_cache, or null.
inline cudaError_t make_decode_params(const AttnArgs& a, const DecodeScratch& ws,
                                      const CacheWrite* write,
                                      size_t smem_budget, DecodeParams* out, size_t* smem) {
  if (a.num_reqs > kDecodeMaxReqs || a.num_kv_heads > 8) return cudaErrorNotSupported;
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.q_stride = a.q_stride;
  prm.block_table = a.block_table;
  prm.bt_stride = a.bt_stride;
  prm.qsl = a.qsl;
  prm.seq_lens = a.seq_lens;
  prm.num_computed = a.num_computed;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.out_stride = a.out_stride;
  prm.num_reqs = a.num_reqs;
  prm.num_blocks = static_cast<int32_t>(a.num_blocks);
  prm.num_heads = a.num_heads;
  prm.hkv = a.num_kv_heads;
  prm.group = a.num_heads / a.num_kv_heads;
  if (prm.group > 16) return cudaErrorNotSupported;
  prm.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  prm.counters = ws.counters;
  prm.part_o = ws.part_o;
  prm.part_ml = ws.part_ml;
  prm.err = a.err;
  prm.k_new = write ? static_cast<const __nv_bfloat16*>(write->key) : nullptr;
  prm.v_new = write ? static_cast<const __nv_bfloat16*>(write->value) : nullptr;
  prm.k_new_stride = write ? write->key_stride : 0;
  prm.v_new_stride = write ? write->value_stride : 0;
  prm.slot_mapping = write ? write->slot_mapping : nullptr;
  prm.key_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(a.key_cache));
  prm.value_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(a.value_cache));
  prm.num_slots = a.num_blocks * a.block_size;
  prm.stage_bytes = 2u * a.num_kv_heads * (a.head_dim / 64) * 2048u;
  // stage ring, then full/empty barriers, the block prefix [R + 1] and the
  // scan's per-warp sums, after up to 1 KiB of alignment
  const size_t fixed = 1024 + 16 * kDecodeMaxStages + 4 * (a.num_reqs + 1) + 4 * 32 + 64;
  if (smem_budget < fixed) return cudaErrorNotSupported;
  int stages = static_cast<int>((smem_budget - fixed) / prm.stage_bytes);
  if (stages > kDecodeMaxStages) stages = kDecodeMaxStages;
  if (stages < 2) return cudaErrorNotSupported;
  prm.stages = stages;
  *smem = 1024 + static_cast<size_t>(stages) * prm.stage_bytes + 16 * stages +
          4 * (a.num_reqs + 1) + 4 * 32 + 64;
  *out = prm;
  return cudaSuccess;
}

// CTA that owns global decode block x when N blocks are split over P CTAs as
// [cN/P, (c+1)N/P): the largest c with floor(cN/P) <= x.
__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t N, int64_t P) {
  return ((x + 1) * P - 1) / N;
}

// One CTA of the split-KV decode: CTA cta_id of num_ctas.  All threads of
// the CTA call it; warps past the KV-head consumers and the producer return
// after the plan.  smem is the CTA's 1024-byte aligned dynamic shared memory.
template <int D, int NT>
__device__ __forceinline__ void decode_cta(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                           const DecodeParams& p, uint8_t* smem, int cta_id,
                                           int num_ctas) {
  constexpr int NDH = D / 64;       // 128-byte boxes across head_dim
  constexpr int KS = D / 16;        // k-steps of S^T = K Q^T
  constexpr int MT = D / 16;        // m-tiles of O^T
  constexpr uint32_t kBox = 2048;   // 16 rows x 128 bytes

  // A kernel launched as this grid's programmatic dependent (the next call's
  // prefill or decode kernel) may start its metadata-only prologue now; it
  // touches Q, the caches, out and the workspace only after this grid has
  // completed.
  if (threadIdx.x == 0) grid_launch_dependents();
  const int hkv = p.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.num_reqs;
  const uint32_t head_bytes = NDH * kBox;
  const uint32_t kv_region = hkv * head_bytes;

  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes);
  uint64_t* empty_bar = full_bar + p.stages;
  int32_t* prefix = reinterpret_cast<int32_t*>(empty_bar + p.stages);  // [R + 1]
  int32_t* scan_tmp = prefix + R + 1;                                   // [32]

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], hkv);
    }
    fence_mbar_init();
    prefix[0] = 0;
  }
  if (warp == hkv && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }

  // ---- plan: decode blocks per request and their prefix sum ----
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int qlen = __ldg(p.qsl + r + 1) - __ldg(p.qsl + r);
    int nb = 0;
    if (qlen == 1) {
      const int seq = __ldg(p.seq_lens + r);
      nb = (seq + 15) >> 4;
      if (seq != __ldg(p.num_computed + r) + 1 || seq <= 0 || nb > p.bt_stride) {
        if (cta_id == 0) atomicOr(p.err, PKV_ERR_METADATA);
        nb = 0;
      }
    }
    prefix[r + 1] = nb;
  }
  __syncthreads();
  block_inclusive_scan(prefix + 1, R, scan_tmp);
  __syncthreads();

  // With fewer blocks than CTAs only the first N CTAs take part, so every
  // participating CTA owns at least one block and the CTAs a request spans
  // are exactly its splits.
  const int64_t N = prefix[R];
  const int64_t P = N < static_cast<int64_t>(num_ctas) ? N : static_cast<int64_t>(num_ctas);
  const int64_t cta = cta_id;
  // Launched as a programmatic dependent, this grid must not complete before
  // the preceding one: block 0 (here, or in its producer warp below) waits
  // for it before exiting.  The wait returns at once otherwise.
  if (cta >= P) {
    if (cta_id == 0 && threadIdx.x == 0) grid_dependency_wait();
    return;
  }
  const int64_t begin = cta * N / P, end = (cta + 1) * N / P;

  // first request of this CTA: prefix[r] <= begin < prefix[r + 1]
  int r0 = 0;
  {
    int lo = 0, hi = R;  // invariant prefix[lo] <= begin < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= begin) lo = mid; else hi = mid;
    }
    r0 = lo;
  }

  if (warp > hkv) return;  // a launch with more warps than roles
  if (warp == hkv) {
    // ======================= producer warp =======================
    // Launched as a programmatic dependent, this grid may run its prologue
    // while the kernel before it finishes.  That kernel may be the cache
    // write (with or without RoPE, which also rewrites Q), so the caches and
    // Q are read only after it has completed.
    grid_dependency_wait();
    int stage = 0;
    uint32_t phase = 0;
    int r = r0;
    for (int64_t x = begin; x < end;) {
      while (prefix[r + 1] <= x) ++r;
      const int j0 = static_cast<int>(x - prefix[r]);
      const int64_t seg_end = end < prefix[r + 1] ? end : prefix[r + 1];
      const int j1 = static_cast<int>(seg_end - prefix[r]);
      const int32_t* row = p.block_table + static_cast<int64_t>(r) * p.bt_stride;
      for (int jb = j0; jb < j1; jb += 32) {
        const int my = jb + lane;
        int32_t phys = my < j1 ? __ldg(row + my) : 0;
        const bool bad = my < j1 && (phys < 0 || phys >= p.num_blocks);
        if (bad) atomicOr(p.err, PKV_ERR_BLOCK_ID);
        if (phys < 0 || phys >= p.num_blocks) phys = p.num_blocks;  // TMA fills zeros
        const int cnt = (j1 - jb) < 32 ? (j1 - jb) : 32;
        for (int k = 0; k < cnt; ++k) {
          const int32_t pb = __shfl_sync(0xffffffffu, phys, k);
          int alive = 1;
          if (lane == 0) {
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) {
              alive = 0;
            } else {
              mbar_arrive_expect_tx(&full_bar[stage], p.stage_bytes);
              // one box per cache: the whole block, landing [head][dim half][token]
              uint8_t* kdst = smem + stage * p.stage_bytes;
              tma_load_4d(kdst, &kmap, 0, pb * 16, 0, 0, &full_bar[stage]);
              tma_load_4d(kdst + kv_region, &vmap, 0, pb * 16, 0, 0, &full_bar[stage]);
            }
          }
          if (!__shfl_sync(0xffffffffu, alive, 0)) {
            if (cta_id == 0 && lane == 0) grid_dependency_wait();
            return;
          }
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      x = seg_end;
    }
    if (cta_id == 0 && lane == 0) grid_dependency_wait();
    return;
  }

  // ======================= consumer warps (one per KV head) =======================
  // Q may still be being rotated in place by the preceding kernel (see the
  // producer's wait above)
  grid_dependency_wait();
  const int h = warp;
  const int G = p.group;
  const int gid = lane >> 2, tid = lane & 3;
  int stage = 0;
  uint32_t phase = 0;
  int r = r0;
  for (int64_t x = begin; x < end;) {
    while (prefix[r + 1] <= x) ++r;
    const int j0 = static_cast<int>(x - prefix[r]);
    const int64_t seg_end = end < prefix[r + 1] ? end : prefix[r + 1];
    const int j1 = static_cast<int>(seg_end - prefix[r]);
    const int64_t tok = __ldg(p.qsl + r);
    const int seq = __ldg(p.seq_lens + r);
    // Fused cache write: the segment holding the request's last block takes
    // this head's new K row (lanes [0, D/8)) and V row (lanes [D/8, D/4)),
    // one 16-byte chunk per lane, loaded now beside Q.
    const bool patch = p.k_new != nullptr && seg_end == prefix[r + 1];
    constexpr int kChunks = D / 8;  // 16-byte chunks in one head's row
    const bool patch_lane = patch && lane < 2 * kChunks;
    const bool patch_v = lane >= kChunks;
    const int patch_chunk = patch_v ? lane - kChunks : lane;
    uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
    int64_t new_slot = -1, want_slot = -1;
    if (patch_lane) {
      const __nv_bfloat16* src = patch_v ? p.v_new + tok * p.v_new_stride
                                         : p.k_new + tok * p.k_new_stride;
      new_row = __ldg(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(h) * D) + patch_chunk);
      new_slot = __ldg(p.slot_mapping + tok);
      want_slot = static_cast<int64_t>(__ldg(p.block_table + static_cast<int64_t>(r) * p.bt_stride +
                                             (seq - 1) / 16)) * 16 + (seq - 1) % 16;
    }

    // B fragments of Q^T: b0 = Q[g][16ks + 2tid .. +1], b1 = Q[g][16ks + 8 + 2tid .. +1]
    uint32_t qb[NT][KS][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = nt * 8 + gid;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          p.q + tok * p.q_stride + static_cast<int64_t>(h * G + (g < G ? g : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[nt][ks][0] = g < G ? __ldg(qrow + ks * 8 + tid) : 0u;
        qb[nt][ks][1] = g < G ? __ldg(qrow + ks * 8 + 4 + tid) : 0u;
      }
    }

    float o[MT][NT][4];
    float mcol[NT][2], lcol[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[mt][nt][c] = 0.f;
      mcol[nt][0] = mcol[nt][1] = -INFINITY;
      lcol[nt][0] = lcol[nt][1] = 0.f;
    }

    for (int j = j0; j < j1; ++j) {
      if (!mbar_wait(&full_bar[stage], phase, p.err)) return;
      uint8_t* kst = smem + stage * p.stage_bytes + h * head_bytes;
      uint8_t* vst = kst + kv_region;
      const uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);
      const int valid = seq - j * 16 < 16 ? seq - j * 16 : 16;
      if (patch && j == j1 - 1) {
        // The block of position seq - 1: its row valid - 1 is this step's
        // token, which the cache may not hold yet.  Use the new row here and
        // write it to its slot (reshape_and_cache semantics: slot < 0 is
        // padding, a slot past the pool is skipped and flagged).
        if (patch_lane) {
          uint8_t* base = patch_v ? vst : kst;
          *reinterpret_cast<uint4*>(base + (patch_chunk >> 3) * kBox +
                                    swz128(valid - 1, patch_chunk & 7)) = new_row;
          if (new_slot >= 0 && new_slot < p.num_slots) {
            __nv_bfloat16* dst = (patch_v ? p.value_cache : p.key_cache) +
                                 new_slot * (static_cast<int64_t>(hkv) * D) +
                                 static_cast<int64_t>(h) * D;
            reinterpret_cast<uint4*>(dst)[patch_chunk] = new_row;
          } else if (new_slot >= p.num_slots) {
            atomicOr(p.err, PKV_ERR_SLOT);
          }
          // the attention used the new row at the block table's slot
          if (new_slot != want_slot && lane == 0) atomicOr(p.err, PKV_ERR_METADATA);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (valid < 16) {
        // rows past the sequence hold whatever the pool had: zero this head's V rows
        for (int i = lane; i < NDH * (16 - valid) * 8; i += 32) {
          const int box = i / ((16 - valid) * 8);
          const int rem = i - box * (16 - valid) * 8;
          const int row = valid + rem / 8;
          *reinterpret_cast<uint4*>(vst + box * kBox + row * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // ---- S^T = K Q^T ----
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t row = lane & 15;
        const uint32_t chunk = ks * 2 + (lane >> 4);  // 16-byte chunk along head_dim
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + (chunk >> 3) * kBox + swz128(row, chunk & 7), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(s[nt], a0, a1, a2, a3, qb[nt][ks][0], qb[nt][ks][1]);
      }

      // ---- online softmax per head column ----
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pr[4];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const float x0 = gid < valid ? s[nt][cc] * p.scale_log2 : -INFINITY;
          const float x1 = gid + 8 < valid ? s[nt][2 + cc] * p.scale_log2 : -INFINITY;
          float mx = fmaxf(x0, x1);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(mcol[nt][cc], mx);
          const float alpha = exp2_approx(mcol[nt][cc] - mnew);
          mcol[nt][cc] = mnew;
          lcol[nt][cc] *= alpha;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            o[mt][nt][cc] *= alpha;
            o[mt][nt][2 + cc] *= alpha;
          }
          pr[cc] = exp2_approx(x0 - mnew);
          pr[2 + cc] = exp2_approx(x1 - mnew);
        }
        const uint32_t lo = pack_bf16(pr[0], pr[1]);   // token gid,     heads 2tid, 2tid+1
        const uint32_t hi = pack_bf16(pr[2], pr[3]);   // token gid + 8
        // the sums use the same rounded weights the tensor cores see
        lcol[nt][0] += __uint_as_float(lo << 16) + __uint_as_float(hi << 16);
        lcol[nt][1] += __uint_as_float(lo & 0xffff0000u) + __uint_as_float(hi & 0xffff0000u);
        pb[nt][0] = movmatrix_trans(lo);
        pb[nt][1] = movmatrix_trans(hi);
      }

      // ---- O^T += V^T P^T ----
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t row = (lane & 7) | ((lane >> 4) << 3);
        const uint32_t chunk = mt * 2 + ((lane >> 3) & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(vbase + (chunk >> 3) * kBox + swz128(row, chunk & 7), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }

      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[stage]);
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- end of this CTA's part of request r ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float l = lcol[nt][cc];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lcol[nt][cc] = l;
      }
    const int64_t cfirst = cta_of(prefix[r], N, P);
    const int64_t clast = cta_of(prefix[r + 1] - 1, N, P);
    const int nsplit = static_cast<int>(clast - cfirst + 1);
    if (nsplit == 1) {
      __nv_bfloat16* orow = p.out + tok * p.out_stride;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int g = nt * 8 + 2 * tid + cc;
          if (g >= G) continue;
          const float inv = 1.f / lcol[nt][cc];
          __nv_bfloat16* dst = orow + static_cast<int64_t>(h * G + g) * D;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            dst[mt * 16 + gid] = __float2bfloat16_rn(o[mt][nt][cc] * inv);
            dst[mt * 16 + 8 + gid] = __float2bfloat16_rn(o[mt][nt][2 + cc] * inv);
          }
        }
    } else {
      const int64_t slot = cta + r;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int g = nt * 8 + 2 * tid + cc;
          if (g >= G) continue;
          const int64_t hh = h * G + g;
          float* po = p.part_o + (slot * p.num_heads + hh) * D;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            po[mt * 16 + gid] = o[mt][nt][cc];
            po[mt * 16 + 8 + gid] = o[mt][nt][2 + cc];
          }
          if (gid == 0) {
            p.part_ml[(slot * p.num_heads + hh) * 2 + 0] = mcol[nt][cc];
            p.part_ml[(slot * p.num_heads + hh) * 2 + 1] = lcol[nt][cc];
          }
        }
      __threadfence();
      __syncwarp();
      int last = 0;
      int32_t* ctr = p.counters + static_cast<int64_t>(r) * hkv + h;
      if (lane == 0) last = atomicAdd(ctr, 1) == nsplit - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        if (lane == 0) *ctr = 0;  // every split has arrived: ready for the next call
        // Each lane merges one slice of one head: lph lanes per head, dpl
        // dims each, so every head's partials are read at once and the
        // loads of kBatch splits are in flight together (merging one head
        // and one split at a time left its CTA behind the others by the
        // sum of those load latencies).
        constexpr int kMaxV = NT * D / 16;  // float4s per lane at most
        constexpr int kBatch = 4;
        int gp = 1;
        while (gp < G) gp <<= 1;
        const int lph = (32 / gp) < (D / 4) ? (32 / gp) : (D / 4);  // lanes per head
        const int dpl = D / lph;                                      // dims per lane
        const int nv = dpl / 4;
        const int g = lane / lph, sub = lane - g * lph;
        const bool active = g < G;
        const int64_t hh = static_cast<int64_t>(h) * G + (active ? g : 0);
        float mx = -INFINITY;
        for (int s0 = 0; s0 < nsplit; s0 += 8) {
          float mv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mv[k] = s0 + k < nsplit
                        ? __ldcg(p.part_ml + ((cfirst + s0 + k + r) * p.num_heads + hh) * 2)
                        : -INFINITY;
#pragma unroll
          for (int k = 0; k < 8; ++k) mx = fmaxf(mx, mv[k]);
        }
        float4 acc[kMaxV];
#pragma unroll
        for (int v = 0; v < kMaxV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
        for (int s0 = 0; s0 < nsplit; s0 += kBatch) {
          float w[kBatch];
#pragma unroll
          for (int k = 0; k < kBatch; ++k) {
            w[k] = 0.f;
            if (s0 + k < nsplit) {
              const float* ml = p.part_ml + ((cfirst + s0 + k + r) * p.num_heads + hh) * 2;
              w[k] = exp2_approx(__ldcg(ml) - mx);
              den += w[k] * __ldcg(ml + 1);
            }
          }
#pragma unroll
          for (int k = 0; k < kBatch; ++k) {
            if (s0 + k >= nsplit) break;
            const float4* po = reinterpret_cast<const float4*>(
                p.part_o + ((cfirst + s0 + k + r) * p.num_heads + hh) * D + sub * dpl);
#pragma unroll
            for (int v = 0; v < kMaxV; ++v) {
              if (v < nv) {
                const float4 x4 = __ldcg(po + v);
                acc[v].x += w[k] * x4.x;
                acc[v].y += w[k] * x4.y;
                acc[v].z += w[k] * x4.z;
                acc[v].w += w[k] * x4.w;
              }
            }
          }
        }
        if (active) {
          const float inv = 1.f / den;
          uint2* dst = reinterpret_cast<uint2*>(p.out + tok * p.out_stride + hh * D + sub * dpl);
#pragma unroll
          for (int v = 0; v < kMaxV; ++v)
            if (v < nv)
              dst[v] = make_uint2(pack_bf16(acc[v].x * inv, acc[v].y * inv),
                                  pack_bf16(acc[v].z * inv, acc[v].w * inv));
        }
      }
    }
    x = seg_end;
  }
}

}  // namespace pkv
