// Chunked-prefill paged attention on the 5th-generation tensor cores.
//
// What it computes ("AI Infra入门干货总结：大模型是如何高效推理的", section
// "Attention Module"; "Chunked Prefill 与 Preemption", section "Chunked
// Prefill：改变调度粒度，不改变 causal 结果"): for a request with query rows at
// absolute positions p = num_computed + u (u < query_len), every query head h
// attends keys j <= p of KV head h / G, K/V read through block_table:
//   out = softmax(scale * Q K^T + M) V,   M_pj = 0 if j <= p else -inf.
//
// Tiling.  A tile is 128 rows = 128/G query tokens x the G query heads of one
// KV head, so each K/V tile serves all G heads (GQA packing).  Keys come in
// tiles of 128 = eight 16-token paged blocks; each block is one TMA box per
// 64-dim half, landing 128-byte swizzled so that the 8 boxes form one
// [128 keys x 64 dims] operand region.  Per key tile j:
//   S_j = Q K_j^T   (tcgen05.mma M=128 N=128 K=D, fp32 in tensor memory)
//   softmax rows   (one thread per row: tcgen05.ld of its S row, causal mask,
//                   running max, exp2, P as bf16 into a swizzled smem tile)
//   O  += P_j V_j  (tcgen05.mma M=128 N=D K=128, V read MN-major)
// S is double-buffered in tensor memory, so S_{j+1} is computed while the
// softmax of tile j runs.  The running max is only moved (and O, l rescaled)
// when a row's new max exceeds the one in use by more than 2^8; otherwise the
// stale max keeps P <= 256, which is exact arithmetic with a different
// reference point.
//
// Warp roles (6 warps): warp 0 issues TMA (Q once per tile, K/V through a
// 2-stage ring), warp 1 owns the tensor memory and issues MMAs from one
// thread, warps 2-5 (one per 32-lane quadrant of tensor memory) run the
// softmax and the epilogue.  Tiles are handed out persistently by a
// device-side plan over query_start_loc, so no host copy of the metadata is
// needed.  Every wait is bounded; a timeout sets PKV_ERR_TIMEOUT and an abort
// flag that stops all roles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "pkv_device.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;
constexpr int kKeys = 128;
constexpr uint32_t kRegion = 16384;  // 128 rows x 128 bytes
constexpr uint32_t kBox = 2048;      // 16 rows x 128 bytes
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O [256, 256 + D)
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum Bar { kQFull, kQEmpty, kKvFull0, kKvFull1, kKvEmpty0, kKvEmpty1, kSFull0, kSFull1,
           kSFree0, kSFree1, kPFull, kODone, kNumBars };

struct PrefillParams {
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* num_computed;
  __nv_bfloat16* out;
  int64_t out_stride;
  int32_t num_reqs;
  int32_t num_blocks;
  int32_t hkv;
  int32_t group;
  float scale_log2;
  uint32_t* err;
};

struct Tile {
  int r, h, u0, ntok, nkeys, nkt;
  int64_t qs;
  int nc;
};

template <int D>
struct Layout {
  static constexpr int NDH = D / 64;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kQBytes = NDH * kRegion;
  static constexpr uint32_t kKV = kQBytes;
  static constexpr uint32_t kKVHalf = NDH * kRegion;      // K (or V) of one stage
  static constexpr uint32_t kKVStage = 2 * kKVHalf;
  static constexpr uint32_t kP = kKV + 2 * kKVStage;
  static constexpr uint32_t kBars = kP + 2 * kRegion;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;  // tmem slot, abort flag
  static constexpr uint32_t kPrefix = kMisc + 16;
};

__device__ __forceinline__ Tile decode_tile(int tile, const int32_t* prefix, int R,
                                            const PrefillParams& p, int tpt) {
  int lo = 0, hi = R;  // prefix[lo] <= tile < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  Tile t;
  t.r = lo;
  const int rem = tile - prefix[lo];
  const int qt = rem / p.hkv;
  t.h = rem - qt * p.hkv;
  t.qs = __ldg(p.qsl + t.r);
  const int qlen = __ldg(p.qsl + t.r + 1) - static_cast<int>(t.qs);
  t.nc = __ldg(p.num_computed + t.r);
  t.u0 = qt * tpt;
  t.ntok = min(tpt, qlen - t.u0);
  t.nkeys = t.nc + t.u0 + t.ntok;  // keys up to the last row's position
  t.nkt = (t.nkeys + kKeys - 1) / kKeys;
  return t;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(192, 1)
    prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap qmap,
                           const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using L = Layout<D>;
  constexpr int NDH = L::NDH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L::kPrefix);
  int32_t* scan_tmp = prefix + p.num_reqs + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.num_reqs;
  const int G = p.group;
  const int tpt = kRows / G;  // query tokens per tile

  if (threadIdx.x == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      const uint32_t cnt = (b == kSFree0 || b == kSFree1 || b == kPFull) ? 4u : 1u;
      mbar_init(&bars[b], cnt);
    }
    fence_mbar_init();
    *abort_flag = 0;
    prefix[0] = 0;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  // ---- plan: tiles per prefill request ----
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int qlen = __ldg(p.qsl + r + 1) - __ldg(p.qsl + r);
    int nt = 0;
    if (qlen > 1) {
      const int seq = __ldg(p.seq_lens + r);
      if (seq != __ldg(p.num_computed + r) + qlen || (seq + 15) / 16 > p.bt_stride) {
        if (blockIdx.x == 0) atomicOr(p.err, PKV_ERR_METADATA);
      } else {
        nt = ((qlen + tpt - 1) / tpt) * p.hkv;
      }
    }
    prefix[r + 1] = nt;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  block_inclusive_scan(prefix + 1, R, scan_tmp);
  __syncthreads();
  const int total = prefix[R];
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ============================ TMA producer ============================
    uint32_t q_uses = 0, kv_count = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Tile t = decode_tile(tile, prefix, R, p, tpt);
      int qok = 1;
      if (lane == 0) {
        if (q_uses > 0 && !mbar_wait_or_abort(&bars[kQEmpty], (q_uses - 1) & 1, p.err, abort_flag)) {
          qok = 0;
        } else {
          mbar_arrive_expect_tx(&bars[kQFull], L::kQBytes);
          for (int dh = 0; dh < NDH; ++dh)
            tma_load_3d(smem + L::kQ + dh * kRegion, &qmap, dh * 64, t.h * G,
                        static_cast<int32_t>(t.qs + t.u0), &bars[kQFull]);
        }
      }
      if (!__shfl_sync(0xffffffffu, qok, 0)) break;
      ++q_uses;
      const int32_t* row = p.block_table + static_cast<int64_t>(t.r) * p.bt_stride;
      const int nblk = (t.nkeys + 15) / 16;
      for (int j = 0; j < t.nkt; ++j) {
        const int b0 = j * 8;
        const int nvalid = min(8, nblk - b0);
        int32_t phys = 0;
        if (lane < nvalid) {
          phys = __ldg(row + b0 + lane);
          if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, PKV_ERR_BLOCK_ID);
            phys = p.num_blocks;  // out of the tensor: TMA fills zeros
          }
        }
        const int s = kv_count & 1;
        const uint32_t n = kv_count >> 1;
        int ok = 1;
        if (lane == 0) {
          if (n > 0 && !mbar_wait_or_abort(&bars[kKvEmpty0 + s], (n - 1) & 1, p.err, abort_flag)) {
            ok = 0;
          } else {
            mbar_arrive_expect_tx(&bars[kKvFull0 + s], 2u * NDH * kBox * nvalid);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        uint8_t* kst = smem + L::kKV + s * L::kKVStage;
        uint8_t* vst = kst + L::kKVHalf;
        for (int k = 0; k < nvalid; ++k) {
          const int32_t pb = __shfl_sync(0xffffffffu, phys, k);
          if (lane == 0) {
            for (int dh = 0; dh < NDH; ++dh) {
              tma_load_3d(kst + dh * kRegion + k * kBox, &kmap, dh * 64, t.h, pb * 16,
                          &bars[kKvFull0 + s]);
              tma_load_3d(vst + dh * kRegion + k * kBox, &vmap, dh * 64, t.h, pb * 16,
                          &bars[kKvFull0 + s]);
            }
          }
        }
        ++kv_count;
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 1);
    uint32_t q_count = 0, kv_count = 0, s_count = 0, p_count = 0;
    const uint32_t q_base = smem_u32(smem + L::kQ);
    const uint32_t p_base = smem_u32(smem + L::kP);
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Tile t = decode_tile(tile, prefix, R, p, tpt);
      bool ok = true;
      if (lane == 0) ok = mbar_wait_or_abort(&bars[kQFull], q_count & 1, p.err, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ++q_count;
      int s_prev = 0;
      for (int j = 0; j <= t.nkt && ok; ++j) {
        if (j < t.nkt) {
          // ---- S_j = Q K_j^T ----
          const int s = kv_count & 1;
          const int b = s_count & 1;
          if (lane == 0) {
            ok = mbar_wait_or_abort(&bars[kKvFull0 + s], (kv_count >> 1) & 1, p.err, abort_flag);
            if (ok && (s_count >> 1) > 0)
              ok = mbar_wait_or_abort(&bars[kSFree0 + b], ((s_count >> 1) - 1) & 1, p.err,
                                      abort_flag);
            if (ok) {
              tc_fence_after();
              const uint32_t k_base = smem_u32(smem + L::kKV + s * L::kKVStage);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kRegion + (kk & 3) * 32;
                tc_mma_ss(tmem + b * kKeys, smem_desc_sw128(q_base + off, 16, 1024),
                          smem_desc_sw128(k_base + off, 16, 1024), idesc_s, kk > 0);
              }
              tc_commit(&bars[kSFull0 + b]);
            }
          }
        }
        if (j > 0 && ok && lane == 0) {
          // ---- O += P_{j-1} V_{j-1} ----
          ok = mbar_wait_or_abort(&bars[kPFull], p_count & 1, p.err, abort_flag);
          if (ok) {
            tc_fence_after();
            const uint32_t v_base = smem_u32(smem + L::kKV + s_prev * L::kKVStage + L::kKVHalf);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              const uint32_t a_off = (kk >> 2) * kRegion + (kk & 3) * 32;
              tc_mma_ss(tmem + kColO, smem_desc_sw128(p_base + a_off, 16, 1024),
                        smem_desc_sw128(v_base + kk * 16 * 128, kRegion, 1024), idesc_o,
                        (j > 1 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&bars[kODone]);
            tc_commit(&bars[kKvEmpty0 + s_prev]);
            if (j == t.nkt) tc_commit(&bars[kQEmpty]);
          }
        }
        if (j > 0) ++p_count;
        if (j < t.nkt) {
          s_prev = kv_count & 1;
          ++kv_count;
          ++s_count;
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
  } else {
    // ============================ softmax warps ============================
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // tile row = tensor-memory lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    uint8_t* p_tile = smem + L::kP;
    uint32_t s_count = 0, kv_count = 0, o_count = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Tile t = decode_tile(tile, prefix, R, p, tpt);
      const int u = t.u0 + row / G;                   // token of this row within the request
      const bool valid_row = (row / G) < t.ntok && row < tpt * G;
      const int pos = t.nc + (valid_row ? u : t.u0 + t.ntok - 1);
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < t.nkt && ok; ++j) {
        const int b = s_count & 1;
        const int s = kv_count & 1;
        ok = __all_sync(0xffffffffu,
                        mbar_wait_or_abort(&bars[kSFull0 + b], (s_count >> 1) & 1, p.err, abort_flag));
        if (!ok) break;
        tc_fence_after();
        float sv[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) {
          uint32_t r32[32];
          tmem_ld32(lane_addr + b * kKeys + c * 32, r32);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(r32[e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kSFree0 + b]);
        // causal mask and row max (log2 units)
        const int key0 = j * kKeys;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const float x = (key0 + c <= pos) ? sv[c] * p.scale_log2 : -INFINITY;
          sv[c] = x;
          mx = fmaxf(mx, x);
        }
        if (j > 0) {
          // PV_{j-1} must be done before O is touched or the P tile rewritten
          ok = __all_sync(0xffffffffu,
                          mbar_wait_or_abort(&bars[kODone], o_count & 1, p.err, abort_flag));
          ++o_count;
          if (!ok) break;
          tc_fence_after();
          const bool mine = mx > m_used + kRescaleThreshold;
          if (__any_sync(0xffffffffu, mine)) {  // tensor-memory access is warp-collective
            const float alpha = mine ? exp2_approx(m_used - mx) : 1.f;
            if (mine) m_used = mx;
            l *= alpha;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r32[32];
              tmem_ld32(lane_addr + kColO + c * 32, r32);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e)
                r32[e] = __float_as_uint(__uint_as_float(r32[e]) * alpha);
              tmem_st32(lane_addr + kColO + c * 32, r32);
            }
            tmem_wait_st();
          }
        } else {
          m_used = mx;  // key 0 is visible to every row, so mx is finite
        }
        // P row (bf16) into the swizzled P tile; l sums the rounded weights
#pragma unroll
        for (int c = 0; c < kKeys / 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = exp2_approx(sv[c * 8 + 2 * e] - m_used);
            const float p1 = exp2_approx(sv[c * 8 + 2 * e + 1] - m_used);
            w[e] = pack_bf16(p0, p1);
            l += __uint_as_float(w[e] << 16) + __uint_as_float(w[e] & 0xffff0000u);
          }
          *reinterpret_cast<uint4*>(p_tile + (c >> 3) * kRegion + swz128(row, c & 7)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        // keys past the request's end: zero this row's V so 0 * (stale) stays 0
        if (j == t.nkt - 1 && key0 + row >= t.nkeys) {
          uint8_t* vrow = smem + L::kKV + s * L::kKVStage + L::kKVHalf + row * 128;
#pragma unroll
          for (int dh = 0; dh < NDH; ++dh)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + dh * kRegion + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPFull]);
        ++s_count;
        ++kv_count;
      }
      if (!ok) break;
      // ---- epilogue: O / l -> out ----
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bars[kODone], o_count & 1, p.err, abort_flag)))
        break;
      ++o_count;
      tc_fence_after();
      const float inv = 1.f / l;
      __nv_bfloat16* orow =
          p.out + (t.qs + u) * p.out_stride + static_cast<int64_t>(t.h * G + row % G) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r32[32];
        tmem_ld32(lane_addr + kColO + c * 32, r32);
        tmem_wait_ld();
        if (valid_row) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r32[q4 * 8 + 0]) * inv, __uint_as_float(r32[q4 * 8 + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(r32[q4 * 8 + 2]) * inv, __uint_as_float(r32[q4 * 8 + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(r32[q4 * 8 + 4]) * inv, __uint_as_float(r32[q4 * 8 + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(r32[q4 * 8 + 6]) * inv, __uint_as_float(r32[q4 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + q4 * 8) = v;
          }
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Encodes the [T, H, D] query as a 3-D tensor (D, H, T) with a box of
// 64 dims x G heads x 128/G tokens, 128-byte swizzled.
template <int D>
static cudaError_t launch_prefill_t(const PrefillParams& prm, const CUtensorMap& qmap,
                                    const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                                    cudaStream_t stream) {
  using L = Layout<D>;
  const size_t smem = 1024 + L::kPrefix + 4 * (prm.num_reqs + 1) + 4 * 32;
  if (smem > 232448) return cudaErrorNotSupported;
  auto kern = prefill_tcgen05_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, 192, smem, stream>>>(qmap, kmap, vmap, prm);
  return cudaGetLastError();
}

cudaError_t launch_prefill_bf16(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int grid, cudaStream_t stream) {
  const int G = a.num_heads / a.num_kv_heads;
  if (G > 128 || kRows % G) return cudaErrorNotSupported;
  PrefillParams prm;
  prm.block_table = a.block_table;
  prm.bt_stride = a.bt_stride;
  prm.qsl = a.qsl;
  prm.seq_lens = a.seq_lens;
  prm.num_computed = a.num_computed;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.out_stride = a.out_stride;
  prm.num_reqs = a.num_reqs;
  prm.num_blocks = static_cast<int32_t>(a.num_blocks);
  prm.hkv = a.num_kv_heads;
  prm.group = G;
  prm.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  prm.err = a.err;
  if (a.head_dim == 128) return launch_prefill_t<128>(prm, qmap, kmap, vmap, grid, stream);
  if (a.head_dim == 64) return launch_prefill_t<64>(prm, qmap, kmap, vmap, grid, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
