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
// once and written straight to its slot.  One warp per token, as in
// reshape_and_cache; lanes take 16-byte vectors of a head in order, so every
// warp access is a run of whole 128-byte lines.  A rotation item is one
// 16-byte vector (interleaved: the pairs are inside it) or two vectors
// rotary_dim/2 apart (NeoX: the pairs straddle them).  The table row (512
// bytes for rotary_dim 128) is read through L1 by every head of the token.
// Arithmetic is fp32 (fma contraction allowed); bf16 results are rounded to
// nearest even.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
// Results go to dst0 and dst1 (either may be null) at the same offsets.
template <typename T, bool kNeox, int U>
__device__ __forceinline__ void rope_rows(const uint4* src, uint4* dst0, uint4* dst1, int heads,
                                          int head_vecs, int rot_vecs, int nrot, int npass,
                                          const float* cs, int half, int lane) {
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
      if (j < 0) continue;
      if (j < nrot) {
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
__global__ void __launch_bounds__(256) rope_reshape_and_cache_kernel(const RopeParams p) {
  // an attention kernel launched as this one's programmatic dependent may
  // start its prologue now; it waits for this grid before reading Q or the
  // caches
  if (threadIdx.x == 0) grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int half = p.rotary_dim >> 1;
  const int nrot = kNeox ? p.rot_vecs / 2 : p.rot_vecs;
  const int npass = p.head_vecs - p.rot_vecs;
  const int64_t row_vecs = static_cast<int64_t>(p.num_kv_heads) * p.head_vecs;
  const int64_t wpb = blockDim.x >> 5;
  for (int64_t t = blockIdx.x * wpb + (threadIdx.x >> 5); t < p.num_tokens;
       t += gridDim.x * wpb) {
    const int64_t pos = __ldg(p.positions + t);
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (pos < 0 || pos >= p.max_position) {
      if (lane == 0 && p.err) atomicOr(p.err, PKV_ERR_POSITION);
      continue;
    }
    if (slot >= p.num_slots && lane == 0 && p.err) atomicOr(p.err, PKV_ERR_SLOT);
    const bool store = slot >= 0 && slot < p.num_slots;
    const float* cs = p.cos_sin + pos * p.rotary_dim;
    // V: a plain copy to the slot
    {
      const uint4* vsrc = p.value + t * p.v_stride_v;
      uint4* vdst = p.value_cache + (store ? slot : 0) * row_vecs;
      constexpr int kUnroll = 4;
      for (int64_t base = 0; base < row_vecs; base += 32 * kUnroll) {
        uint4 r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t i = base + u * 32 + lane;
          if (i < row_vecs) r[u] = ld16(vsrc + i);
        }
        if (store) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + u * 32 + lane;
            if (i < row_vecs) vdst[i] = r[u];
          }
        }
      }
    }
    // K: rotated straight into its slot (and into key_out if given)
    rope_rows<T, kNeox, 2>(p.key + t * p.k_stride_v,
                           store ? p.key_cache + slot * row_vecs : nullptr,
                           p.key_out ? p.key_out + t * p.k_stride_v : nullptr, p.num_kv_heads,
                           p.head_vecs, p.rot_vecs, nrot, npass, cs, half, lane);
    // Q: rotated in place; its pass-through part is already where it belongs
    uint4* q = p.query + t * p.q_stride_v;
    rope_rows<T, kNeox, 4>(q, q, nullptr, p.num_heads, p.head_vecs, p.rot_vecs, nrot, 0, cs, half,
                           lane);
  }
}

template <typename T, bool kNeox>
cudaError_t launch_t(const RopeParams& p, cudaStream_t stream) {
  constexpr int kThreads = 256;  // 8 warps, one token each per iteration
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (p.num_tokens + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident blocks per SM
  const int64_t grid = blocks < cap ? blocks : cap;
  rope_reshape_and_cache_kernel<T, kNeox>
      <<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
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
