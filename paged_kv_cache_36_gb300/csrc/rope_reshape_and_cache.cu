// Fused RoPE + reshape_and_cache: rotate each token's Q and K by the row of
// cos_sin_cache at its position, write Q back in place and scatter the
// rotated K and the unchanged V into the paged cache at slot_mapping.
//
// "AI Infra入门干货总结：大模型是如何高效推理的", section "Attention Module
// (以标准GQA + RoPE为例)": after the QKV split Q and K are rotated (a block-
// diagonal rotation matrix, applied element-wise), then reshape_and_cache
// scatters K/V by slot_mapping; sin/cos come from a table cos_sin_cache
// [max_position_embeddings, rotary_dim] built once and indexed by position.
// Row p holds rotary_dim/2 cosines, then the sines of the same angles.  Pair
// i of a head is (2i, 2i+1) (interleaved) or (i, i + rotary_dim/2) (NeoX);
// (x, y) becomes (x cos - y sin, y cos + x sin); dimensions at and above
// rotary_dim are copied unchanged.
//
// Done as one pass, the rotation costs no HBM traffic beyond the scatter's
// own (plus Q, which the rotation has to read and write anyway): K is read
// once and written straight to its slot.  Two forms, chosen by token count:
// * staged (fewer than 1024 tokens): a CTA takes a run of tokens and moves
//   each token's Q, K, V and table rows with 1-D bulk copies through a ring
//   of shared-memory stages, rotating Q and K there;
// * one warp per token (1024 tokens and more, or rows that do not fit the
//   ring): lanes take 16-byte vectors of a head in order, so every warp
//   access is a run of whole 128-byte lines, and the table row is read
//   through L1 by every head of the token.
// A rotation item is one 16-byte vector (interleaved: the pairs are inside
// it) or two vectors rotary_dim/2 apart (NeoX: the pairs straddle them).
// Arithmetic is fp32 (fma contraction allowed); bf16 results are rounded to
// nearest even.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

namespace {

template <typename T>
struct Vec16;

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// M consecutive floats of the table (M a multiple of 2; 8-byte aligned, and
// 16-byte aligned when M is a multiple of 4).
template <int M>
__device__ __forceinline__ void load_table(const float* p, float (&out)[M]) {
  if constexpr (M % 4 == 0) {
#pragma unroll
    for (int i = 0; i < M; i += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
      out[i] = v.x;
      out[i + 1] = v.y;
      out[i + 2] = v.z;
      out[i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < M; i += 2) {
      const float2 v = __ldg(reinterpret_cast<const float2*>(p + i));
      out[i] = v.x;
      out[i + 1] = v.y;
    }
  }
}

// Plain (coherent) 16-byte load: Q is rewritten in place, and key_out may
// alias key, so these reads must not take the read-only path.
__device__ __forceinline__ uint4 ld16(const uint4* p) { return *p; }

struct RopeParams {
  const int64_t* positions;
  uint4* query;              // in/out
  const uint4* key;
  uint4* key_out;            // may be null
  const uint4* value;
  uint4* key_cache;
  uint4* value_cache;
  const int64_t* slot_mapping;
  const float* cos_sin;
  int64_t q_stride_v;        // token strides in 16-byte vectors
  int64_t k_stride_v;
  int64_t v_stride_v;
  int64_t max_position;
  int64_t num_tokens;
  int64_t num_slots;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_vecs;         // head_dim / N
  int32_t rot_vecs;          // rotary_dim / N
  int32_t rotary_dim;
  uint32_t* err;
};

// Rotation items and copy items of `heads` head rows starting at src.  Item
// j < nrot of a head is a rotation (NeoX: vectors j and j + rot_vecs/2;
// interleaved: vector j); the other items copy vector rot_vecs + (j - nrot).
// Results go to dst0 and dst1 (either may be null) at the same offsets, and
// only if `ok`.  The row's loads are issued before the table row at `pos`
// is touched, so the position's own load latency hides behind them.
template <typename T, bool kNeox, int U>
__device__ __forceinline__ void rope_rows(const uint4* src, uint4* dst0, uint4* dst1, int heads,
                                          int head_vecs, int rot_vecs, int nrot, int npass,
                                          const float* table, int64_t pos, int rotary_dim,
                                          bool ok, int lane) {
  constexpr int N = Vec16<T>::N;
  constexpr int M = kNeox ? N : N / 2;  // table entries one item needs (each of cos, sin)
  const int iph = nrot + npass;
  const int total = heads * iph;
  for (int base = 0; base < total; base += 32 * U) {
    uint4 a[U], b[U];
    int off[U], jj[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * 32 + lane;
      jj[u] = -1;
      if (idx < total) {
        const int h = idx / iph;
        const int j = idx - h * iph;
        jj[u] = j;
        off[u] = h * head_vecs + (j < nrot ? j : rot_vecs + (j - nrot));
        a[u] = ld16(src + off[u]);
        if (kNeox && j < nrot) b[u] = ld16(src + off[u] + (rot_vecs >> 1));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = jj[u];
      if (j < 0 || !ok) continue;
      if (j < nrot) {
        const float* cs = table + pos * rotary_dim;
        const int half = rotary_dim >> 1;
        float c[M], s[M];
        load_table<M>(cs + j * M, c);
        load_table<M>(cs + half + j * M, s);
        float x[N];
        Vec16<T>::unpack(a[u], x);
        if constexpr (kNeox) {
          float y[N];
          Vec16<T>::unpack(b[u], y);
          float xo[N], yo[N];
#pragma unroll
          for (int e = 0; e < N; ++e) {
            xo[e] = x[e] * c[e] - y[e] * s[e];
            yo[e] = y[e] * c[e] + x[e] * s[e];
          }
          const uint4 pa = Vec16<T>::pack(xo), pb = Vec16<T>::pack(yo);
          const int ob = off[u] + (rot_vecs >> 1);
          if (dst0) {
            dst0[off[u]] = pa;
            dst0[ob] = pb;
          }
          if (dst1) {
            dst1[off[u]] = pa;
            dst1[ob] = pb;
          }
        } else {
          float xo[N];
#pragma unroll
          for (int e = 0; e < M; ++e) {
            xo[2 * e] = x[2 * e] * c[e] - x[2 * e + 1] * s[e];
            xo[2 * e + 1] = x[2 * e + 1] * c[e] + x[2 * e] * s[e];
          }
          const uint4 pa = Vec16<T>::pack(xo);
          if (dst0) dst0[off[u]] = pa;
          if (dst1) dst1[off[u]] = pa;
        }
      } else {
        if (dst0) dst0[off[u]] = a[u];
        if (dst1) dst1[off[u]] = a[u];
      }
    }
  }
}

template <typename T, bool kNeox>
__global__ void __launch_bounds__(256) rope_cache_warp_kernel(const RopeParams p) {
  // This grid is itself a programmatic dependent of the kernel before it
  // (which may still read the cache or Q, or write the new rows): wait for
  // it before any load or store.
  grid_dependency_wait();
  // An attention kernel launched as this one's programmatic dependent may
  // start its prologue now (it waits for this grid before reading Q or the
  // caches).  Released only after the wait above, so that prologue reads
  // metadata that work before this grid wrote.
  if (threadIdx.x == 0) grid_launch_dependents();
  // One warp per token.  The V row's loads go out together with the position
  // and slot loads, and the K row's right after; the position's validity is
  // applied only at the stores, so no load waits for it.
  const int lane = threadIdx.x & 31;
  const int nrot = kNeox ? p.rot_vecs / 2 : p.rot_vecs;
  const int npass = p.head_vecs - p.rot_vecs;
  const int64_t row_vecs = static_cast<int64_t>(p.num_kv_heads) * p.head_vecs;
  const int64_t wpb = blockDim.x >> 5;
  for (int64_t t = blockIdx.x * wpb + (threadIdx.x >> 5); t < p.num_tokens;
       t += gridDim.x * wpb) {
    const int64_t pos = __ldg(p.positions + t);
    const int64_t slot = __ldg(p.slot_mapping + t);
    const uint4* vsrc = p.value + t * p.v_stride_v;
    constexpr int kUnroll = 4;
    uint4 r[kUnroll];
#pragma unroll
    for (int v = 0; v < kUnroll; ++v) {
      const int64_t i = v * 32 + lane;
      if (i < row_vecs) r[v] = ld16(vsrc + i);
    }
    const bool ok = pos >= 0 && pos < p.max_position;
    const bool store = ok && slot >= 0 && slot < p.num_slots;
    rope_rows<T, kNeox, 2>(p.key + t * p.k_stride_v,
                           store ? p.key_cache + slot * row_vecs : nullptr,
                           p.key_out ? p.key_out + t * p.k_stride_v : nullptr, p.num_kv_heads,
                           p.head_vecs, p.rot_vecs, nrot, npass, p.cos_sin, pos, p.rotary_dim, ok,
                           lane);
    if (lane == 0 && p.err) {
      if (!ok) atomicOr(p.err, PKV_ERR_POSITION);
      else if (slot >= p.num_slots) atomicOr(p.err, PKV_ERR_SLOT);
    }
    uint4* vdst = p.value_cache + (store ? slot : 0) * row_vecs;
    if (store) {
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int64_t i = v * 32 + lane;
        if (i < row_vecs) vdst[i] = r[v];
      }
    }
    for (int64_t base = 32 * kUnroll; base < row_vecs; base += 32 * kUnroll) {  // longer rows
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int64_t i = base + v * 32 + lane;
        if (i < row_vecs) r[v] = ld16(vsrc + i);
      }
      if (store) {
#pragma unroll
        for (int v = 0; v < kUnroll; ++v) {
          const int64_t i = base + v * 32 + lane;
          if (i < row_vecs) vdst[i] = r[v];
        }
      }
    }
    uint4* q = p.query + t * p.q_stride_v;
    rope_rows<T, kNeox, 4>(q, q, nullptr, p.num_heads, p.head_vecs, p.rot_vecs, nrot, 0, p.cos_sin,
                           pos, p.rotary_dim, ok, lane);
  }
}

template <typename T, bool kNeox>
cudaError_t launch_warp_t(RopeParams p, cudaStream_t stream) {
  constexpr int kThreads = 256;  // 8 warps, one token each per iteration
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (p.num_tokens + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // tokens beyond this loop in the warps
  const int64_t grid = blocks < cap ? blocks : cap;
  return launch_programmatic(rope_cache_warp_kernel<T, kNeox>, dim3(static_cast<unsigned>(grid)),
                             dim3(kThreads), 0, stream, p);
}

// ---------------------------------------------------------------------------
// Staged form: bulk copies through a shared-memory ring.
//
// A CTA takes a contiguous run of tokens.  For each token one thread issues
// four 1-D bulk copies (the Q row, the K row, the V row and the table row at
// the token's position) into a ring stage, S - 1 tokens ahead of the one
// being rotated; the CTA rotates Q and K in shared memory, and the same
// thread writes the stage back with bulk stores (Q in place, K and V to the
// slot, K to key_out).  Bytes in flight are held by the copy engine, not by
// registers: S - 1 stages of 12.5 KiB per CTA for Llama-3-8B rows.
constexpr int kStagedThreads = 128;

struct StageLayout {
  uint32_t q_bytes, kv_bytes, tab_bytes;  // payloads, multiples of 16
  uint32_t off_k, off_v, off_tab;         // offsets in a stage, multiples of 128
  uint32_t stage_bytes;                   // multiple of 128
  int32_t stages;                         // ring depth, >= 3
  int32_t iph;                            // 16-byte rotation items per head; divides kStagedThreads
};

// Rotates the Q rows and the K row of one stage in place.  Thread tid takes
// item w = tid % iph of heads tid / iph, + kStagedThreads / iph, ...; the
// cosines and sines of item w are the same for every head.
template <typename T, bool kNeox>
__device__ __forceinline__ void rotate_stage(uint8_t* st, const RopeParams& p, const StageLayout& L,
                                             int tid) {
  constexpr int N = Vec16<T>::N;
  constexpr int M = kNeox ? N : N / 2;
  const int w = tid & (L.iph - 1);
  const int hstep = kStagedThreads / L.iph;
  const float* tab = reinterpret_cast<const float*>(st + L.off_tab);
  const int half = p.rotary_dim >> 1;
  float c[M], s[M];
#pragma unroll
  for (int e = 0; e < M; ++e) {
    c[e] = tab[w * M + e];
    s[e] = tab[half + w * M + e];
  }
  const int head_bytes = p.head_vecs * 16;
  const int nh = p.num_heads + p.num_kv_heads;
  for (int h = tid / L.iph; h < nh; h += hstep) {
    uint8_t* row = h < p.num_heads ? st + h * head_bytes
                                   : st + L.off_k + (h - p.num_heads) * head_bytes;
    uint4* a = reinterpret_cast<uint4*>(row) + w;
    float x[N];
    Vec16<T>::unpack(*a, x);
    if constexpr (kNeox) {
      uint4* b = a + (p.rot_vecs >> 1);
      float y[N], xo[N], yo[N];
      Vec16<T>::unpack(*b, y);
#pragma unroll
      for (int e = 0; e < N; ++e) {
        xo[e] = x[e] * c[e] - y[e] * s[e];
        yo[e] = y[e] * c[e] + x[e] * s[e];
      }
      *a = Vec16<T>::pack(xo);
      *b = Vec16<T>::pack(yo);
    } else {
      float xo[N];
#pragma unroll
      for (int e = 0; e < M; ++e) {
        xo[2 * e] = x[2 * e] * c[e] - x[2 * e + 1] * s[e];
        xo[2 * e + 1] = x[2 * e + 1] * c[e] + x[2 * e] * s[e];
      }
      *a = Vec16<T>::pack(xo);
    }
  }
}

template <typename T, bool kNeox>
__global__ void __launch_bounds__(kStagedThreads)
    rope_cache_staged_kernel(const RopeParams p, const StageLayout L) {
  // This grid is itself a programmatic dependent of the kernel before it
  // (which may still read the cache or Q, or write the new rows): wait for
  // it before any load or store.
  grid_dependency_wait();
  // An attention kernel launched as this one's programmatic dependent may
  // start its prologue now (it waits for this grid before reading Q or the
  // caches).  Released only after the wait above, so that prologue reads
  // metadata that work before this grid wrote.
  if (threadIdx.x == 0) grid_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * L.stage_bytes);
  // positions and slots of this CTA's tokens, 32 at a time, in a ring of 64
  // entries written and read by warp 0 only
  int64_t* ring_pos = reinterpret_cast<int64_t*>(full + S);
  int64_t* ring_slot = ring_pos + 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t t0 = blockIdx.x * p.num_tokens / G;
  const int64_t n = (blockIdx.x + 1) * p.num_tokens / G - t0;
  const int64_t row_vecs = static_cast<int64_t>(p.num_kv_heads) * p.head_vecs;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  auto load_batch = [&](int64_t j0) {  // warp 0, converged
    const int64_t j = j0 + lane;
    if (j < n) {
      ring_pos[j & 63] = __ldg(p.positions + t0 + j);
      ring_slot[j & 63] = __ldg(p.slot_mapping + t0 + j);
    }
    __syncwarp();
  };
  auto issue = [&](int64_t j) {  // one thread of warp 0
    const int s = static_cast<int>(j % S);
    const int64_t pos = ring_pos[j & 63];
    if (pos < 0 || pos >= p.max_position) {  // nothing to load; the token is skipped
      mbar_arrive(&full[s]);
      return;
    }
    const int64_t tok = t0 + j;
    uint8_t* st = smem + static_cast<size_t>(s) * L.stage_bytes;
    mbar_arrive_expect_tx(&full[s], L.q_bytes + 2 * L.kv_bytes + L.tab_bytes);
    bulk_load(st, p.query + tok * p.q_stride_v, L.q_bytes, &full[s]);
    bulk_load(st + L.off_k, p.key + tok * p.k_stride_v, L.kv_bytes, &full[s]);
    bulk_load(st + L.off_v, p.value + tok * p.v_stride_v, L.kv_bytes, &full[s]);
    bulk_load(st + L.off_tab, p.cos_sin + pos * p.rotary_dim, L.tab_bytes, &full[s]);
  };
  if (warp == 0) load_batch(0);
  __syncthreads();
  if (tid == 0)
    for (int64_t j = 0; j < S - 1 && j < n; ++j) issue(j);

  int64_t i = 0;
  bool timed_out = false;
  for (; i < n; ++i) {
    const int s = static_cast<int>(i % S);
    uint8_t* st = smem + static_cast<size_t>(s) * L.stage_bytes;
    const bool got = mbar_wait(&full[s], static_cast<uint32_t>((i / S) & 1), p.err);
    if (__syncthreads_or(!got)) {
      timed_out = true;
      break;
    }
    // a skipped token's stage holds stale bytes: rotating them is harmless,
    // nothing is written back
    rotate_stage<T, kNeox>(st, p, L, tid);
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0) {
      if (lane == 0) {
        const int64_t pos = ring_pos[i & 63], slot = ring_slot[i & 63];
        const int64_t tok = t0 + i;
        if (pos < 0 || pos >= p.max_position) {
          if (p.err) atomicOr(p.err, PKV_ERR_POSITION);
        } else {
          bulk_store(p.query + tok * p.q_stride_v, st, L.q_bytes);
          if (p.key_out) bulk_store(p.key_out + tok * p.k_stride_v, st + L.off_k, L.kv_bytes);
          if (slot >= 0 && slot < p.num_slots) {
            bulk_store(p.key_cache + slot * row_vecs, st + L.off_k, L.kv_bytes);
            bulk_store(p.value_cache + slot * row_vecs, st + L.off_v, L.kv_bytes);
          } else if (slot >= p.num_slots && p.err) {
            atomicOr(p.err, PKV_ERR_SLOT);
          }
        }
        bulk_commit();
      }
      // refill the previous token's stage once its stores have read it
      const int64_t j = i + S - 1;
      if (j < n) {
        if ((j & 31) == 0) load_batch(j);
        if (lane == 0) {
          bulk_wait_read<1>();
          issue(j);
        }
      }
      __syncwarp();
    }
  }
  if (tid == 0) {
    if (timed_out)  // let the copies still in flight land before leaving
      for (int64_t j = i; j < n && j < i + S - 1; ++j)
        mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1), nullptr);
    bulk_wait_all();
  }
}

constexpr size_t kStagedSmemLimit = 232448;  // 227 KiB, the per-CTA maximum

uint32_t align128(uint64_t x) { return static_cast<uint32_t>((x + 127) & ~uint64_t{127}); }

// The ring layout for these rows, or stages = 0 if the staged form does not
// apply (rows too large for three stages, or items that do not tile a CTA).
template <typename T, bool kNeox>
StageLayout stage_layout(const RopeParams& p) {
  StageLayout L{};
  L.iph = kNeox ? p.rot_vecs / 2 : p.rot_vecs;
  if (L.iph < 1 || L.iph > kStagedThreads || kStagedThreads % L.iph) return L;
  const uint64_t q = static_cast<uint64_t>(p.num_heads) * p.head_vecs * 16;
  const uint64_t kv = static_cast<uint64_t>(p.num_kv_heads) * p.head_vecs * 16;
  const uint64_t tab = static_cast<uint64_t>(p.rotary_dim) * 4;
  const uint64_t stage = align128(align128(q) + 2 * align128(kv) + tab);
  int S = 4;
  while (S >= 3 && S * stage + 8 * S + 1024 > kStagedSmemLimit) --S;
  if (S < 3) return L;
  L.q_bytes = static_cast<uint32_t>(q);
  L.kv_bytes = static_cast<uint32_t>(kv);
  L.tab_bytes = static_cast<uint32_t>(tab);
  L.off_k = align128(q);
  L.off_v = L.off_k + align128(kv);
  L.off_tab = L.off_v + align128(kv);
  L.stage_bytes = static_cast<uint32_t>(stage);
  L.stages = S;
  return L;
}

// Below this many tokens the staged form is faster (its CTAs each take a
// token or a few and have them in flight at once: 5.0 us for 64 Llama-3-8B
// tokens against 8.1 us); from here on the warp form keeps more bytes in
// flight per SM (37.8 us against 40.7 us at 8192 tokens, measured on GB300).
constexpr int64_t kStagedMaxTokens = 1024;

template <typename T, bool kNeox>
cudaError_t launch_t(const RopeParams& p, cudaStream_t stream) {
  const StageLayout L = stage_layout<T, kNeox>(p);
  if (L.stages == 0 || p.num_tokens >= kStagedMaxTokens) return launch_warp_t<T, kNeox>(p, stream);
  auto kern = rope_cache_staged_kernel<T, kNeox>;
  cudaError_t e = raise_smem_limit_once<rope_cache_staged_kernel<T, kNeox>>(kStagedSmemLimit);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(L.stages) * L.stage_bytes + 8 * L.stages + 1024;
  // CTAs per SM for the last smem size seen (the row shape rarely changes)
  static std::atomic<uint64_t> cached{0};  // smem << 16 | CTAs per SM
  uint64_t c = cached.load(std::memory_order_relaxed);
  int per_sm = static_cast<int>(c & 0xffff);
  if ((c >> 16) != smem || per_sm == 0) {
    per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStagedThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    cached.store((static_cast<uint64_t>(smem) << 16) | static_cast<uint64_t>(per_sm),
                 std::memory_order_relaxed);
  }
  static const int sms = [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      return 148;
    return n;
  }();
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  const int64_t grid = p.num_tokens < cap ? p.num_tokens : cap;
  return launch_programmatic(kern, dim3(static_cast<unsigned>(grid)), dim3(kStagedThreads), smem,
                             stream, p, L);
}

}  // namespace

cudaError_t launch_rope_reshape_and_cache(const RopeArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int64_t es = a.bf16 ? 2 : 4;
  RopeParams p;
  p.positions = a.positions;
  p.query = static_cast<uint4*>(a.query);
  p.key = static_cast<const uint4*>(a.key);
  p.key_out = static_cast<uint4*>(a.key_out);
  p.value = static_cast<const uint4*>(a.value);
  p.key_cache = static_cast<uint4*>(a.key_cache);
  p.value_cache = static_cast<uint4*>(a.value_cache);
  p.slot_mapping = a.slot_mapping;
  p.cos_sin = a.cos_sin_cache;
  p.q_stride_v = a.query_stride * es / 16;
  p.k_stride_v = a.key_stride * es / 16;
  p.v_stride_v = a.value_stride * es / 16;
  p.max_position = a.max_position;
  p.num_tokens = a.num_tokens;
  p.num_slots = a.num_slots;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.head_vecs = static_cast<int32_t>(a.head_dim * es / 16);
  p.rot_vecs = static_cast<int32_t>(a.rotary_dim * es / 16);
  p.rotary_dim = a.rotary_dim;
  p.err = a.err;
  if (a.bf16)
    return a.is_neox ? launch_t<__nv_bfloat16, true>(p, stream)
                     : launch_t<__nv_bfloat16, false>(p, stream);
  return a.is_neox ? launch_t<float, true>(p, stream) : launch_t<float, false>(p, stream);
}

}  // namespace pkv
