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
// tiles of 128 = eight 16-token paged blocks.  A block of K or V (one head)
// is one TMA box that lands as [token half][dim half][8 keys][128 B],
// 128-byte swizzled: read K-major this is the K operand (groups of 8 keys
// D/64 KiB apart), read MN-major the V operand (64-dim atoms 1 KiB apart,
// groups of 8 keys D/64 KiB apart).  Per key tile j:
//   S_j = Q K_j^T   tcgen05.mma M=128 N=128 K=D from shared memory, fp32 in
//                   tensor memory (three S buffers)
//   softmax        eight warps, two per 32-lane quadrant of tensor memory:
//                   warp half h reads keys [64h, 64h + 64) of every tile; the
//                   two warps of a quadrant exchange their row maxima, so both
//                   use one running max, and each writes its P (bf16) back
//                   over the S columns it has just read
//   O += P_j V_j   tcgen05.mma with A = P from tensor memory and B = V read
//                   MN-major from shared memory, one fp32 accumulator
// A running max is only moved (and O, l rescaled) when it would grow by more
// than 2^8; otherwise the stale max keeps P <= 256, the same arithmetic with a
// different reference point.  With three S buffers, QK of key tile j + 3
// waits only for PV of key tile j, so the tensor core runs ahead of the
// softmax instead of alternating with it.
//
// Warp roles (12 warps): warp 0 streams Q and K (3-stage ring), warp 3
// streams V (2-stage ring); warp 1 owns the tensor memory and issues QK^T;
// warp 2 issues PV; warps 4-11 run the softmax and the epilogue.  Each
// issuer blocks on its own barriers, so neither waits behind the other.
// Tiles are handed out persistently by a device-side plan over
// query_start_loc, heaviest (most keys) first, in rows of one tile per
// CTA that alternate direction, so CTAs end close together when a prompt's
// tiles grow from a few key tiles to many.  Every wait is bounded; a timeout sets PKV_ERR_TIMEOUT and
// an abort flag that stops all roles.
//
// One kernel per call.  The grid is one CTA per SM, and the call's decode
// rows (query length 1) run in the same grid: after the plan every CTA
// knows the step's prefill and decode work and takes the same decision
// (mixed_split.cuh), CTAs [0, n_p) run the prefill tiles as above and CTAs
// [n_p, S) run the split-KV decode body (decode_core.cuh) over the decode
// rows.  The two parts of a mixed step thus overlap on disjoint SMs within
// one launch, with no CTA waiting for another to leave its SM.
//
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_core.cuh"
#include "kernels.h"
#include "mixed_split.cuh"
#include "pkv_device.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;
constexpr int kKeys = 128;
constexpr uint32_t kRegion = 16384;  // 128 rows x 128 bytes
constexpr uint32_t kBox = 2048;      // 16 rows x 128 bytes
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSBufs = 3;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (4 + kSoftmaxWarps) * 32;
// tensor memory: three S/P buffers of 128 fp32 columns (a softmax warp's P
// overwrites the first 32 of its own 64 S columns) and the O accumulator
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = kSBufs * kKeys;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr size_t kPrefillSmemLimit = 232448;  // 227 KiB per CTA

enum Bar {
  kQFull, kQEmpty,
  kKFull0, kKFull1, kKFull2, kKEmpty0, kKEmpty1, kKEmpty2,
  kVFull0, kVFull1, kVEmpty0, kVEmpty1,
  kSFull0, kSFull1, kSFull2, kSFree0, kSFree1, kSFree2,
  kPFull0, kPFull1, kPFull2, kODone0, kODone1, kODone2,
  kOFinal, kPair0, kPair1, kPair2, kPair3,
  kNumBars
};
static_assert(kKFull0 + kKStages == kKEmpty0 && kKEmpty0 + kKStages == kVFull0,
              "one full and one empty barrier per K stage");
static_assert(kVFull0 + kVStages == kVEmpty0 && kVEmpty0 + kVStages == kSFull0,
              "one full and one empty barrier per V stage");
static_assert(kSFull0 + kSBufs == kSFree0 && kSFree0 + kSBufs == kPFull0 &&
                  kPFull0 + kSBufs == kODone0 && kODone0 + kSBufs == kOFinal,
              "S-full, S-free, P-full and O-done: one barrier per S buffer");
static_assert(kColO + 128 <= kTmemCols, "S buffers and O fit in tensor memory");

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
  int32_t cache_reqs;  // query_start_loc and num_computed copied to shared memory
  int32_t head_dim;
  // Fused reshape_and_cache of the prefill rows' tokens (k_new == nullptr:
  // off): row t of k_new / v_new goes to slot_mapping[t] of the caches.
  const uint4* k_new;
  const uint4* v_new;
  int64_t k_new_stride;  // 16-byte vectors per token
  int64_t v_new_stride;
  const int64_t* slot_mapping;
  uint4* key_cache;
  uint4* value_cache;
  int64_t num_slots;
  uint32_t* barrier;     // two zeroed words shared by the prefill CTAs
};

// Batches of up to this many requests keep query_start_loc and num_computed
// in shared memory, so that decoding a tile costs no global load.
constexpr int kReqCache = 2048;

struct Tile {
  int r, h, u0, ntok;
  int nkeys;   // keys loaded: up to the tile's last query row's position
  int nkt;     // key tiles walked
  int64_t qs;
  int nc;
};

template <int D>
struct Layout {
  static constexpr int NDH = D / 64;
  static constexpr uint32_t kHalf = NDH * kRegion;  // one K (or V) tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kHalf;
  static constexpr uint32_t kV = kK + kKStages * kHalf;
  static constexpr uint32_t kBars = kV + kVStages * kHalf;
  static constexpr uint32_t kXch = kBars + 8 * kNumBars;      // [2 parity][2 half][128 rows] floats
  static constexpr uint32_t kMisc = kXch + 2 * 2 * 128 * 4;   // tmem slot, abort flag, n_p
  static constexpr uint32_t kWork = kMisc + 16;                // one MixedWork per warp
  static constexpr uint32_t kPrefix = kWork + 32 * (kThreads / 32);
};

// Tile `ct` -> (request, KV head, query rows).  prefix[r] counts the tiles
// of requests before r; within a request tiles run KV head fastest, then
// query tiles.
__device__ __forceinline__ Tile decode_tile(int ct, const int32_t* prefix, int R,
                                            const PrefillParams& p, int tpt,
                                            const int32_t* qsl, const int32_t* num_computed) {
  int lo = 0, hi = R;  // prefix[lo] <= ct < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= ct) lo = mid; else hi = mid;
  }
  Tile t;
  t.r = lo;
  const int rem = ct - prefix[lo];
  const int qt = rem / p.hkv;
  t.h = rem - qt * p.hkv;
  t.qs = qsl[t.r];
  const int qlen = qsl[t.r + 1] - static_cast<int>(t.qs);
  t.nc = num_computed[t.r];
  t.u0 = qt * tpt;
  t.ntok = min(tpt, qlen - t.u0);
  t.nkeys = t.nc + t.u0 + t.ntok;
  t.nkt = (t.nkeys + kKeys - 1) / kKeys;
  return t;
}

// The it-th tile of CTA cid, or -1 when there is none.  Within a request
// later query tiles see more keys, so tiles are taken from the highest index
// down, ncta at a time, in alternating direction: each CTA starts with one of
// the heaviest tiles and heavy and light ones pair up.
__device__ __forceinline__ int cta_tile(int it, int cid, int ncta, int total) {
  const int lin = it * ncta + ((it & 1) ? ncta - 1 - cid : cid);
  return lin < total ? total - 1 - lin : -1;
}

// The fused cache write of one tile's tokens and KV head: K and V rows of
// tokens [u0, u0 + ntok) of request r, head h, to their slots.  Every (token,
// KV head) of a prefill row belongs to exactly one tile, so the tiles of all
// prefill CTAs write each row once.  The slot must be the one the block table
// gives for the token's position (else PKV_ERR_METADATA); slot < 0 is
// padding and a slot past the pool is skipped with PKV_ERR_SLOT.
template <int D>
__device__ __forceinline__ void write_tile_rows(const PrefillParams& p, const Tile& t) {
  constexpr int kVec = D / 8;  // 16-byte vectors in one head's row
  const int n = t.ntok * 2 * kVec;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int u = i / (2 * kVec);
    const int rem = i - u * 2 * kVec;
    const bool is_v = rem >= kVec;
    const int c = is_v ? rem - kVec : rem;
    const int64_t tok = t.qs + t.u0 + u;
    const int64_t slot = __ldg(p.slot_mapping + tok);
    const int pos = t.nc + t.u0 + u;
    if (c == 0 && !is_v) {
      const int64_t want =
          static_cast<int64_t>(__ldg(p.block_table + static_cast<int64_t>(t.r) * p.bt_stride + pos / 16)) *
              16 + pos % 16;
      if (slot != want) atomicOr(p.err, PKV_ERR_METADATA);
      if (slot >= p.num_slots) atomicOr(p.err, PKV_ERR_SLOT);
    }
    if (slot < 0 || slot >= p.num_slots) continue;
    const uint4 v = __ldg((is_v ? p.v_new + tok * p.v_new_stride : p.k_new + tok * p.k_new_stride) +
                          t.h * kVec + c);
    (is_v ? p.value_cache : p.key_cache)[(slot * p.hkv + t.h) * kVec + c] = v;
  }
}

// Transposes NV x NV blocks of 16-byte values across groups of NV lanes
// (NV a power of two <= 32): afterwards lane NV g + j holds in v[k] what lane
// NV g + k held in v[j].  Butterfly exchanges, log2(NV) rounds of shuffles.
template <int NV>
__device__ __forceinline__ void transpose_lane_groups(uint4 (&v)[NV], int lane) {
#pragma unroll
  for (int s = 1; s < NV; s <<= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (i & s) continue;
      // pair (i, i + s): the low lane sends v[i + s], the high lane v[i]
      const uint4 x = hi ? v[i] : v[i + s];
      uint4 y;
      y.x = __shfl_xor_sync(0xffffffffu, x.x, s);
      y.y = __shfl_xor_sync(0xffffffffu, x.y, s);
      y.z = __shfl_xor_sync(0xffffffffu, x.z, s);
      y.w = __shfl_xor_sync(0xffffffffu, x.w, s);
      if (hi) v[i] = y; else v[i + s] = y;
    }
  }
}

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// All lanes of the calling warp wait; the result is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, err, abort));
}

}  // namespace

static_assert(sizeof(MixedWork) == 32, "one 32-byte slot of work sums per warp");

// qmap/kmap/vmap: the prefill's query and per-head cache maps; kblk/vblk:
// the decode's whole-block cache maps.
template <int D, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    varlen_attention_kernel(const __grid_constant__ CUtensorMap qmap,
                            const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ CUtensorMap kblk,
                            const __grid_constant__ CUtensorMap vblk, const PrefillParams p,
                            const DecodeParams dp) {
  using L = Layout<D>;
  constexpr int NDH = L::NDH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  float* xch = reinterpret_cast<float*>(smem + L::kXch);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int* np_slot = reinterpret_cast<int*>(smem + L::kMisc + 8);
  MixedWork* warp_work = reinterpret_cast<MixedWork*>(smem + L::kWork);  // [warps]
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L::kPrefix);
  int32_t* scan_tmp = prefix + p.num_reqs + 1;
  int32_t* req_qsl = scan_tmp + 32;            // [R + 1] when cached
  int32_t* req_nc = req_qsl + p.num_reqs + 1;  // [R]
  const int32_t* qsl_t = p.cache_reqs ? req_qsl : p.qsl;
  const int32_t* nc_t = p.cache_reqs ? req_nc : p.num_computed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.num_reqs;
  const int cid = blockIdx.x;
  const int G = p.group;
  const int tpt = kRows / G;  // query tokens per tile

  if (threadIdx.x == 0) {
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
  // ---- plan: tiles per prefill request (all of a request's metadata in
  // one round of loads), and the step's prefill and decode work ----
  MixedWork mine = {0, 0, 0, 0, 0};
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int q0 = __ldg(p.qsl + r), q1 = __ldg(p.qsl + r + 1);
    const int seq = __ldg(p.seq_lens + r), nc = __ldg(p.num_computed + r);
    if (p.cache_reqs) {
      req_qsl[r] = q0;
      req_nc[r] = nc;
      if (r == R - 1) req_qsl[R] = q1;
    }
    const int qlen = q1 - q0;
    mixed_work_add(mine, qlen, nc, seq, p.hkv, G, p.head_dim);
    int nt = 0;
    if (qlen > 1) {
      if (nc < 0 || seq != nc + qlen || (seq + 15) / 16 > p.bt_stride) {
        if (blockIdx.x == 0) atomicOr(p.err, PKV_ERR_METADATA);
      } else {
        nt = (qlen + tpt - 1) / tpt * p.hkv;
      }
    }
    prefix[r + 1] = nt;
  }
  mixed_work_warp_sum(mine);
  if (lane == 0) warp_work[warp] = mine;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The roles: every CTA reaches the same n_p from the same sums.  Only a
  // prefill CTA sets up the barriers of the prefill pipeline.
  if (threadIdx.x == 0) {
    MixedWork w = {0, 0, 0, 0, 0};
    for (int i = 0; i < kThreads / 32; ++i) {
      const MixedWork& x = warp_work[i];
      w.prefill_tiles += x.prefill_tiles;
      w.prefill_units += x.prefill_units;
      w.decode_bytes += x.decode_bytes;
      w.prefill_rows += x.prefill_rows;
      w.decode_rows += x.decode_rows;
    }
    const int n_p = mixed_prefill_ctas(w, gridDim.x);
    *np_slot = n_p;
    if (cid < n_p) {
      for (int b = 0; b < kNumBars; ++b) {
        uint32_t n = 1;
        if (b >= kPFull0 && b < kPFull0 + kSBufs) n = kSoftmaxWarps;
        if (b >= kPair0 && b < kPair0 + 4) n = 2;  // the two warps sharing a quadrant
        mbar_init(&bars[b], n);
      }
      fence_mbar_init();
    }
  }
  block_inclusive_scan(prefix + 1, R, scan_tmp);
  __syncthreads();
  const int total = prefix[R];
  const int ncta = *np_slot;
  const uint32_t tmem = *tmem_slot;
  if (cid >= ncta) {
    // ---- decode role: hand back the tensor memory, then the decode body
    // over CTAs [n_p, S) ----
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    __syncthreads();  // every thread has read the slots above; the body reuses the memory
    decode_cta<D, NT>(kblk, vblk, dp, smem, cid - ncta, static_cast<int>(gridDim.x) - ncta);
    return;
  }

  if (p.k_new != nullptr) {
    // ---- fused reshape_and_cache of the prefill rows ----
    // The kernel before this one may still read the caches (or write the new
    // rows): wait for it.  Each CTA writes the rows of its own tiles, then
    // the prefill CTAs meet at a counter in the workspace, so that every
    // tile's copies find every row of its keys in the cache.  The grid is
    // one CTA per SM (its registers admit no second one), and the
    // prefill CTAs have the lowest indices, so all of them are resident once
    // the kernels before this one drain; the wait is bounded all the same.
    grid_dependency_wait();
    for (int it = 0, ct = cta_tile(0, cid, ncta, total); ct >= 0;
         ct = cta_tile(++it, cid, ncta, total))
      write_tile_rows<D>(p, decode_tile(ct, prefix, R, p, tpt, qsl_t, nc_t));
    fence_proxy_async_global();
    __syncthreads();
    if (threadIdx.x == 0 && !cta_group_barrier(p.barrier, ncta, p.err)) *abort_flag = 1;
    __syncthreads();
    fence_proxy_async_global();
  }

  if (warp == 0 || warp == 3) {
    // ============================ TMA producers ============================
    // warp 0 streams Q and K, warp 3 streams V.  They are separate warps so
    // that neither waits on the other's ring: two lanes of one warp would run
    // converged, and K would stall whenever V waits for a free stage.  The
    // whole warp reads the block table, 32 entries per coalesced load and one
    // batch ahead, so no key tile waits on a block-table read; lane 0 waits
    // for free stages and issues the copies.
    const bool is_k = warp == 0;
    const int nst = is_k ? kKStages : kVStages;
    const int full0 = is_k ? kKFull0 : kVFull0;
    const int empty0 = is_k ? kKEmpty0 : kVEmpty0;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    uint8_t* ring = smem + (is_k ? L::kK : L::kV);
    uint32_t q_uses = 0, count = 0;
    bool ok = true;
    bool grid_waited = false;
    for (int it = 0, ct = cta_tile(0, cid, ncta, total); ct >= 0 && ok;
         ct = cta_tile(++it, cid, ncta, total)) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Tile t = decode_tile(ct, prefix, R, p, tpt, qsl_t, nc_t);
      const int32_t* row = p.block_table + static_cast<int64_t>(t.r) * p.bt_stride;
      const int nblk = (t.nkeys + 15) / 16;
      // Block ids [batch, batch + 32) in `cur`, the next 32 in flight in `nxt`.
      // A batch is checked when it becomes current, by which time its loads
      // have long completed, so no key tile waits on a block-table read.
      auto load_ids = [&](int first) -> int32_t {
        const int b = first + lane;
        return b < nblk ? __ldg(row + b) : 0;
      };
      auto check_ids = [&](int32_t v, int first) -> int32_t {
        const int b = first + lane;
        if (b < nblk && (v < 0 || v >= p.num_blocks)) {
          if (is_k) atomicOr(p.err, PKV_ERR_BLOCK_ID);
          v = p.num_blocks;  // out of the tensor: TMA fills zeros
        }
        return v;
      };
      int batch = 0;
      int32_t cur = load_ids(0), nxt = load_ids(32);
      // This grid is a programmatic dependent of the kernel before it, so the
      // set-up and plan above (metadata only) and the first block-table reads
      // overlap that kernel's tail.  Q and the caches may be written by it
      // (the cache write, with RoPE also Q), so the copies start only after
      // it has completed.  Every thread that writes global memory does so
      // after data these copies brought.  The kernel after this one is
      // released here (it waits for this grid to complete before it touches
      // memory this grid uses).
      if (!grid_waited) {
        grid_dependency_wait();
        if (is_k && lane == 0) grid_launch_dependents();
        grid_waited = true;
      }
      if (is_k) {
        if (lane == 0) {
          if (q_uses > 0 && !mbar_wait_or_abort(&bars[kQEmpty], (q_uses - 1) & 1, p.err, abort_flag)) {
            ok = false;
          } else {
            mbar_arrive_expect_tx(&bars[kQFull], L::kHalf);
            for (int dh = 0; dh < NDH; ++dh)
              tma_load_3d(smem + L::kQ + dh * kRegion, &qmap, dh * 64, t.h * G,
                          static_cast<int32_t>(t.qs + t.u0), &bars[kQFull]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++q_uses;
      }
      cur = check_ids(cur, 0);
      for (int j = 0; j < t.nkt && ok; ++j) {
        const int b0 = j * 8;
        if (b0 >= batch + 32) {
          batch += 32;
          cur = check_ids(nxt, batch);
          nxt = load_ids(batch + 32);
        }
        const int nvalid = min(8, nblk - b0);
        int32_t phys[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) phys[k] = __shfl_sync(0xffffffffu, cur, (b0 - batch) + k);
        if (lane == 0) {
          const int st = count % nst;
          const uint32_t n = count / nst;
          if (n > 0 && !mbar_wait_or_abort(&bars[empty0 + st], (n - 1) & 1, p.err, abort_flag)) {
            ok = false;
          } else {
            mbar_arrive_expect_tx(&bars[full0 + st], NDH * kBox * nvalid);
            // one box per block, landing [token half][dim half][8 keys][128 B]
            uint8_t* dst = ring + st * L::kHalf;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (k < nvalid)
                tma_load_5d(dst + k * NDH * kBox, map, 0, 0, 0, t.h, phys[k] * 2,
                            &bars[full0 + st]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++count;
      }
    }
    if (!grid_waited) {  // a CTA without tiles waits and releases the same way
      grid_dependency_wait();
      if (is_k && lane == 0) grid_launch_dependents();
    }
    // drain: every copy into this CTA's ring has landed before the CTA may
    // exit
    if (lane == 0) {
      for (int st = 0; st < nst; ++st) {
        const uint32_t uses = count / nst + (static_cast<uint32_t>(st) < count % nst ? 1u : 0u);
        if (uses == 0) continue;
        mbar_wait(&bars[full0 + st], (uses - 1) & 1, p.err);
      }
      if (is_k && q_uses > 0) mbar_wait(&bars[kQFull], (q_uses - 1) & 1, p.err);
    }
  } else if (warp == 1) {
    // ============================ QK^T issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0);
      // descriptors are built once; a stage or k-step only adds its byte
      // offset >> 4 to the start-address field
      const uint64_t q_desc = smem_desc_sw128(smem_u32(smem + L::kQ), 16, 1024);
      // K stage: groups of 8 keys every NDH KiB, dim half dh at +dh KiB
      const uint64_t k_desc0 = smem_desc_sw128(smem_u32(smem + L::kK), 16, NDH * 1024);
      uint32_t q_count = 0, k_count = 0, s_count = 0;
      bool ok = true;
      for (int it = 0, ct = cta_tile(0, cid, ncta, total); ct >= 0 && ok && !*abort_flag;
           ct = cta_tile(++it, cid, ncta, total)) {
        const Tile t = decode_tile(ct, prefix, R, p, tpt, qsl_t, nc_t);
        ok = mbar_wait_or_abort(&bars[kQFull], q_count & 1, p.err, abort_flag);
        ++q_count;
        for (int j = 0; j < t.nkt && ok; ++j) {
          const int ks = k_count % kKStages;
          const int b = s_count % kSBufs;
          const uint32_t use = s_count / kSBufs;
          ok = mbar_wait_or_abort(&bars[kKFull0 + ks], (k_count / kKStages) & 1, p.err, abort_flag);
          // S/P buffer b is free once PV of the key tile that last used it is done
          if (ok && use > 0)
            ok = mbar_wait_or_abort(&bars[kSFree0 + b], (use - 1) & 1, p.err, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = k_desc0 + ((ks * L::kHalf) >> 4);
          const uint32_t d_s = tmem + kColS + b * kKeys;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t q_off = ((kk >> 2) * kRegion + (kk & 3) * 32) >> 4;
            const uint64_t k_off = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            tc_mma_ss(d_s, q_desc + q_off, kd + k_off, idesc_s, kk > 0);
          }
          tc_commit(&bars[kSFull0 + b]);
          tc_commit(&bars[kKEmpty0 + ks]);
          if (j == t.nkt - 1) tc_commit(&bars[kQEmpty]);
          ++k_count;
          ++s_count;
        }
      }
    }
  } else if (warp == 2) {
    // ============================ PV issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 1);
      // V stage, MN-major: the two 64-dim atoms of a group of 8 keys 1 KiB
      // apart, groups of 8 keys NDH KiB apart
      const uint64_t v_desc0 = smem_desc_sw128(smem_u32(smem + L::kV), 1024, NDH * 1024);
      uint32_t v_count = 0, s_count = 0;
      bool ok = true;
      for (int it = 0, ct = cta_tile(0, cid, ncta, total); ct >= 0 && ok && !*abort_flag;
           ct = cta_tile(++it, cid, ncta, total)) {
        const Tile t = decode_tile(ct, prefix, R, p, tpt, qsl_t, nc_t);
        for (int j = 0; j < t.nkt && ok; ++j) {
          const int vs = v_count % kVStages;
          const int b = s_count % kSBufs;
          const uint32_t use = s_count / kSBufs;
          // P of S buffer b: one barrier per buffer, so that a softmax warp
          // already done with a later key tile cannot complete this tile's
          // phase for a slower warp
          ok = mbar_wait_or_abort(&bars[kPFull0 + b], use & 1, p.err, abort_flag) &&
               mbar_wait_or_abort(&bars[kVFull0 + vs], (v_count / kVStages) & 1, p.err, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd = v_desc0 + ((vs * L::kHalf) >> 4);
          const uint32_t a_p = tmem + kColS + b * kKeys;
          // O += P V over the 128 keys: P columns hold the keys of each warp
          // half in their first 32 (bf16 pairs), V rows [64 half, 64 half + 64)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ts(tmem + kColO, a_p + half * 64 + kk * 8,
                        vd + ((((half * 64 + kk * 16) / 8) * NDH * 1024) >> 4), idesc_o,
                        (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&bars[kODone0 + b]);
          if (j == t.nkt - 1) tc_commit(&bars[kOFinal]);
          tc_commit(&bars[kSFree0 + b]);
          tc_commit(&bars[kVEmpty0 + vs]);
          ++v_count;
          ++s_count;
        }
      }
    }
  } else if (warp >= 4) {
    // ============================ softmax warps ============================
    // Two warps share each 32-lane quadrant of tensor memory (the same 128/4
    // rows): warp half h reads S columns [64 h, 64 h + 64).  They agree on the
    // row maximum every key tile through a small exchange, so one O serves the
    // whole row; each warp keeps the partial sum l of its own columns and
    // rescales its half of O's columns.
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;    // keys [64 half, 64 half + 64) of each tile
    const int row = quad * 32 + lane;    // tile row = tensor-memory lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t o_cols = lane_addr + kColO + half * (D / 2);
    const float sl2 = p.scale_log2;
    uint64_t* pair_bar = &bars[kPair0 + quad];
    uint32_t s_count = 0, v_count = 0, pair_uses = 0, tiles_done = 0;
    // row value exchanged with the partner warp; returns the partner's value
    auto exchange = [&](float mine) -> float {
      float* slot = xch + (pair_uses & 1) * 256;
      slot[half * 128 + row] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(pair_bar);
      const bool done = warp_wait(pair_bar, pair_uses & 1, p.err, abort_flag);
      ++pair_uses;
      return done ? slot[(half ^ 1) * 128 + row] : mine;
    };
    for (int it = 0, ct = cta_tile(0, cid, ncta, total); ct >= 0;
         ct = cta_tile(++it, cid, ncta, total)) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Tile t = decode_tile(ct, prefix, R, p, tpt, qsl_t, nc_t);
      const int u = t.u0 + row / G;  // token of this row within the request
      const bool valid_row = (row / G) < t.ntok;
      const int pos = t.nc + (valid_row ? u : t.u0 + t.ntok - 1);
      const int pos_min = t.nc + t.u0;  // smallest position in the tile
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < t.nkt && ok; ++j) {
        const uint32_t gs = s_count;  // this key tile's index in the CTA's sequence
        const int b = gs % kSBufs;
        if (!warp_wait(&bars[kSFull0 + b], (gs / kSBufs) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_cols = lane_addr + kColS + b * kKeys + half * 64;
        float sv[64];
        {
          uint32_t (&r)[64] = *reinterpret_cast<uint32_t(*)[64]>(&sv);
          tmem_ld32(s_cols, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld32(s_cols + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_wait_ld();
        }
        ++s_count;
        // causal mask (only tiles reaching past the tile's first row) and max
        const int key0 = j * kKeys + half * 64;
        if (key0 + 63 > pos_min) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (key0 + c > pos) sv[c] = -INFINITY;
        }
        // row max: four chains of three-input maxima
        float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
        for (int c = 4; c < 64; c += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], sv[c + k], sv[c + 4 + k]);
        const float m_mine = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
        const float mx = fmaxf(m_mine, exchange(m_mine));  // row max of the key tile
        if (j == 0) {
          m_used = mx;  // finite: key 0 is visible to every row
        } else {
          // both warps of the quadrant see the same mx and m_used, so they
          // take the same decision for every row
          const bool grow = mx > m_used + kRescaleThreshold;
          if (__any_sync(0xffffffffu, grow)) {
            // O must hold PV of the previous key tile before it is rescaled;
            // o_done has one barrier per S buffer because the softmax may run
            // two key tiles ahead of the PV products
            const uint32_t prev = gs - 1;
            if (!warp_wait(&bars[kODone0 + prev % kSBufs], (prev / kSBufs) & 1, p.err, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = grow ? exp2_approx(m_used - mx) : 1.f;
            if (grow) m_used = mx;
            l *= alpha;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              uint32_t r32[32];
              tmem_ld32(o_cols + c * 32, r32);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e)
                r32[e] = __float_as_uint(__uint_as_float(r32[e]) * alpha);
              tmem_st32(o_cols + c * 32, r32);
            }
            tmem_wait_st();
          }
        }
        // P = 2^(s * scale_log2 - m_used) as bf16 pairs over the first 32 of
        // this warp's 64 S columns
        // (two lanes of each packed fma and add: f32x2 operations)
        const float2 sl2x2 = make_float2(sl2, sl2), neg_m2 = make_float2(-m_used, -m_used);
        float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 x = __ffma2_rn(make_float2(sv[2 * e], sv[2 * e + 1]), sl2x2, neg_m2);
          const float2 pe = make_float2(exp2_approx(x.x), exp2_approx(x.y));
          l2[e & 1] = __fadd2_rn(l2[e & 1], pe);
          w[e] = pack_bf16(pe.x, pe.y);
        }
        tmem_st32(s_cols, w);
        l += (l2[0].x + l2[1].x) + (l2[0].y + l2[1].y);
        tmem_wait_st();
        // keys past the tile's last row were not loaded: zero their V rows
        // so that 0 * (stale) stays 0
        if (j == t.nkt - 1 && j * kKeys + kKeys > t.nkeys) {
          // The stage's previous tile (V of key tile gs - 2) may still be in
          // use: this warp can be two key tiles ahead of the PV products.
          // Wait for its release first (PV(gs - 4) is known complete, so that
          // parity is unambiguous), then for this tile's copies.
          const int vs = v_count % kVStages;
          const uint32_t round = v_count / kVStages;
          if ((round > 0 &&
               !warp_wait(&bars[kVEmpty0 + vs], (round - 1) & 1, p.err, abort_flag)) ||
              !warp_wait(&bars[kVFull0 + vs], round & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const int key = j * kKeys + half * 64 + (quad & 1) * 32 + lane;
          if (quad < 2 && key >= t.nkeys) {
            const int k = key - j * kKeys;  // row of key k, dim half dh: group k / 8
            uint8_t* vrow = smem + L::kV + vs * L::kHalf + (k / 8) * NDH * 1024 + (k % 8) * 128;
#pragma unroll
            for (int dh = 0; dh < NDH; ++dh)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vrow + dh * 1024 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        ++v_count;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPFull0 + b]);
      }
      if (!ok) break;
      // ---- epilogue: O / (l_0 + l_1) -> out ----
      // O is final once the tile's last PV is done, waited for on a barrier
      // with one phase per tile
      if (!warp_wait(&bars[kOFinal], tiles_done & 1, p.err, abort_flag)) break;
      ++tiles_done;
      tc_fence_after();
      const float inv = 1.f / (l + exchange(l));
      // This warp holds output dims [half * D/2, half * D/2 + D/2) of its 32
      // rows: NV 16-byte pieces per row.  A transpose among groups of NV
      // lanes turns that into NV rows per group with one piece each per
      // lane, so every store instruction writes whole rows' segments
      // (contiguous bytes) instead of 16 bytes in each of 32 rows.
      constexpr int NV = D / 16;
      uint4 seg[NV];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r0[32];
        tmem_ld32(lane_addr + kColO + half * (D / 2) + c * 32, r0);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4& v = seg[c * 4 + q4];
          v.x = pack_bf16(__uint_as_float(r0[q4 * 8 + 0]) * inv, __uint_as_float(r0[q4 * 8 + 1]) * inv);
          v.y = pack_bf16(__uint_as_float(r0[q4 * 8 + 2]) * inv, __uint_as_float(r0[q4 * 8 + 3]) * inv);
          v.z = pack_bf16(__uint_as_float(r0[q4 * 8 + 4]) * inv, __uint_as_float(r0[q4 * 8 + 5]) * inv);
          v.w = pack_bf16(__uint_as_float(r0[q4 * 8 + 6]) * inv, __uint_as_float(r0[q4 * 8 + 7]) * inv);
        }
      }
      transpose_lane_groups<NV>(seg, lane);
      // lane NV g + j now holds piece j of rows NV g + k (k < NV) of the warp
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int trow = quad * 32 + (lane & ~(NV - 1)) + k;  // tile row
        if (trow / G < t.ntok) {
          __nv_bfloat16* dst = p.out + (t.qs + t.u0 + trow / G) * p.out_stride +
                               static_cast<int64_t>(t.h * G + trow % G) * D + half * (D / 2) +
                               (lane & (NV - 1)) * 8;
          *reinterpret_cast<uint4*>(dst) = seg[k];
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

// Shared memory of one CTA: the layout, the per-request tile prefix and, for
// batches of up to kReqCache requests, query_start_loc and num_computed.
template <int D>
static size_t prefill_smem_bytes(int num_reqs, bool cache_reqs) {
  return 1024 + Layout<D>::kPrefix + 4 * (static_cast<size_t>(num_reqs) + 1) + 4 * 32 +
         (cache_reqs ? 8 * static_cast<size_t>(num_reqs) + 4 : 0);
}

template <int D, int NT>
static cudaError_t launch_varlen_t(const PrefillParams& prm, const DecodeParams& dp,
                                   size_t smem, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, const CUtensorMap& kblk,
                                   const CUtensorMap& vblk, int sms, cudaStream_t stream) {
  auto kern = varlen_attention_kernel<D, NT>;
  cudaError_t e = raise_smem_limit_once<varlen_attention_kernel<D, NT>>(kPrefillSmemLimit);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  // a programmatic dependent of the kernel before it in the stream (see the
  // waits in the producer warps of both roles)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(sms));  // one persistent CTA per SM
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, kblk, vblk, prm, dp);
}

cudaError_t launch_varlen_bf16(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, const CUtensorMap& kblk,
                               const CUtensorMap& vblk, const DecodeScratch& ws, int sms,
                               cudaStream_t stream, const CacheWrite* write) {
  const int G = a.num_heads / a.num_kv_heads;
  if (G > 128 || kRows % G) return cudaErrorNotSupported;
  if (sms < 2) return cudaErrorNotSupported;  // each role keeps a CTA
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
  prm.cache_reqs = a.num_reqs <= kReqCache ? 1 : 0;
  prm.head_dim = a.head_dim;
  prm.k_new = write ? static_cast<const uint4*>(write->key) : nullptr;
  prm.v_new = write ? static_cast<const uint4*>(write->value) : nullptr;
  prm.k_new_stride = write ? write->key_stride / 8 : 0;  // bf16 elements -> 16-byte vectors
  prm.v_new_stride = write ? write->value_stride / 8 : 0;
  prm.slot_mapping = write ? write->slot_mapping : nullptr;
  prm.key_cache = static_cast<uint4*>(const_cast<void*>(a.key_cache));
  prm.value_cache = static_cast<uint4*>(const_cast<void*>(a.value_cache));
  prm.num_slots = a.num_blocks * a.block_size;
  prm.barrier = a.err + 1;  // words 1 and 2 of the workspace header
  // The decode role follows the same kernel before this one as the prefill
  // role, so it waits for it too; it writes the decode rows' new K/V itself.
  DecodeParams dp;
  size_t dsmem = 0;
  cudaError_t e = make_decode_params(a, ws, write, kPrefillSmemLimit, &dp, &dsmem);
  if (e != cudaSuccess) return e;
  const bool wide = G > 8;
  if (a.head_dim == 128) {
    size_t smem = prefill_smem_bytes<128>(prm.num_reqs, prm.cache_reqs != 0);
    if (smem < dsmem) smem = dsmem;
    if (smem > kPrefillSmemLimit) return cudaErrorNotSupported;
    return wide ? launch_varlen_t<128, 2>(prm, dp, smem, qmap, kmap, vmap, kblk, vblk, sms, stream)
                : launch_varlen_t<128, 1>(prm, dp, smem, qmap, kmap, vmap, kblk, vblk, sms, stream);
  }
  if (a.head_dim == 64) {
    size_t smem = prefill_smem_bytes<64>(prm.num_reqs, prm.cache_reqs != 0);
    if (smem < dsmem) smem = dsmem;
    if (smem > kPrefillSmemLimit) return cudaErrorNotSupported;
    return wide ? launch_varlen_t<64, 2>(prm, dp, smem, qmap, kmap, vmap, kblk, vblk, sms, stream)
                : launch_varlen_t<64, 1>(prm, dp, smem, qmap, kmap, vmap, kblk, vblk, sms, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
