// How a call with both prefill rows and decode rows shares the SMs between
// its prefill tiles and its decode rows ("AI Infra入门干货总结：大模型是如何高效
// 推理的", section "Attention Module": one varlen call serves the prefill
// chunks and the decode tokens of a step).
//
// Such a call runs one persistent kernel of one CTA per SM (S CTAs).  Every
// CTA sums the step's work from the same metadata and evaluates the same
// integer formula below, so all agree on n_p without talking to each other:
// CTAs [0, n_p) take the prefill role and share the prefill tiles, CTAs
// [n_p, S) take the decode role and share the decode rows' blocks.
//
// The model (times in ns, figures measured on GB300):
//   decode:  t_d = B / 7000, its bytes at the HBM rate.  One SM streams at
//            most about 105 bytes/ns, so the decode keeps that rate down to
//            about 7000 / 105 = 67 SMs and slows below it.
//   prefill: a 128-row query tile of k key tiles costs about 1100 k + 3000
//            ns on one SM, 13/10 of that next to the decode; the tiles are
//            handed out whole, so n CTAs take ceil(tiles / n) tiles each.
// n_p is the fewest CTAs that finish the prefill within half the decode's
// time, raised to a fifth of the SMs (the decode ran no slower on 120-128
// SMs than on all 152, and the prefill then ends well inside the step), and
// capped so that the decode keeps 67 SMs.  When the prefill cannot finish
// within half the decode's time on the SMs it may take, the SMs are split in
// proportion to each role's time on one SM (a decode SM beside a busy
// prefill streams about 70 bytes/ns).  Each role keeps at least one
// CTA while it has rows, so that rows with bad metadata are still reported.
#pragma once

#include <cstdint>

namespace pkv {

struct MixedWork {
  unsigned long long prefill_tiles;  // 128-row query tiles (all KV heads)
  unsigned long long prefill_units;  // their key tiles of 128 keys
  unsigned long long decode_bytes;   // K/V bytes the decode rows read
  unsigned int prefill_rows;         // requests with query length > 1
  unsigned int decode_rows;          // requests with query length 1
};

// Key tiles of the query tiles of one request and one KV head: tile t holds
// tokens [t tpt, (t + 1) tpt) and sees keys up to its last token.
__device__ __forceinline__ unsigned long long prefill_request_units(int nc, int qlen, int tpt) {
  const int tiles = (qlen + tpt - 1) / tpt;
  unsigned long long u = 0;
  if (tpt >= 128) {
    // tpt = 128: tile t sees ceil(nc / 128) + t + 1 key tiles (the last one clipped)
    const unsigned long long base = (nc + 127) / 128;
    const unsigned long long n = tiles - 1;
    u = n * base + n * (n + 1) / 2 + (nc + qlen + 127) / 128;
  } else {
    // tpt divides 128: the count grows by one every 128 / tpt tiles
    const int k = 128 / tpt;
    const int n = tiles - 1;
    const unsigned long long full = n / k, rem = n % k;
    unsigned long long base = 0, tail = 0;
    for (int i = 0; i < k; ++i) {
      const unsigned long long fi = (nc + tpt * (i + 1) + 127) / 128;
      base += fi;
      if (static_cast<unsigned long long>(i) < rem) tail += fi + full;
    }
    u = full * base + k * full * (full - 1) / 2 + tail + (nc + qlen + 127) / 128;
  }
  return u;
}

// Adds one request of the call to w.  qlen > 1: prefill rows; qlen == 1: a
// decode row over seq keys.
__device__ __forceinline__ void mixed_work_add(MixedWork& w, int qlen, int nc, int seq, int hkv,
                                               int group, int head_dim) {
  if (qlen > 1) ++w.prefill_rows;
  if (qlen == 1) ++w.decode_rows;
  if (nc < 0 || nc > (1 << 30) || qlen > (1 << 30)) return;  // the kernels reject such rows
  if (qlen > 1) {
    const int tpt = 128 / group;
    w.prefill_tiles += static_cast<unsigned long long>((qlen + tpt - 1) / tpt) * hkv;
    w.prefill_units += prefill_request_units(nc, qlen, tpt) * hkv;
  } else if (qlen == 1 && seq > 0) {
    w.decode_bytes += static_cast<unsigned long long>(seq) * hkv * head_dim * 4;  // K and V, bf16
  }
}

// Sums w over the lanes of the calling warp (all lanes take part).
__device__ __forceinline__ void mixed_work_warp_sum(MixedWork& w) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    w.prefill_tiles += __shfl_xor_sync(0xffffffffu, w.prefill_tiles, o);
    w.prefill_units += __shfl_xor_sync(0xffffffffu, w.prefill_units, o);
    w.decode_bytes += __shfl_xor_sync(0xffffffffu, w.decode_bytes, o);
    w.prefill_rows += __shfl_xor_sync(0xffffffffu, w.prefill_rows, o);
    w.decode_rows += __shfl_xor_sync(0xffffffffu, w.decode_rows, o);
  }
}

// CTAs of the prefill role out of sms (the decode role takes the other
// sms - n_p).
__device__ __forceinline__ int mixed_prefill_ctas(const MixedWork& w, int sms) {
  if (w.prefill_rows == 0) return 0;
  if (w.decode_rows == 0 || sms < 2) return sms;
  if (w.prefill_tiles == 0) return 1;  // only rows that fail their checks
  if (w.decode_bytes == 0) return sms - 1;
  // the decode saturates HBM (7000 bytes/ns) from about 67 SMs (105 bytes/ns each)
  constexpr unsigned long long kHbmBytesPerNs = 7000, kSatSms = 67;
  const unsigned long long t_d = w.decode_bytes / kHbmBytesPerNs;
  const unsigned long long tile_ns =
      (w.prefill_units * 1100 + w.prefill_tiles * 3000) * 13 / (10 * w.prefill_tiles);
  const int cap = sms > static_cast<int>(kSatSms) + 1 ? sms - static_cast<int>(kSatSms) : 1;
  const unsigned long long per_cta = tile_ns > 0 ? (t_d / 2) / tile_ns : 0;  // tiles per CTA
  if (per_cta >= 1) {
    const unsigned long long need = (w.prefill_tiles + per_cta - 1) / per_cta;
    if (need <= static_cast<unsigned long long>(cap)) {
      const int floor_share = sms / 5 < cap ? sms / 5 : cap;
      const int n = static_cast<int>(need);
      return n > floor_share ? n : (floor_share > 0 ? floor_share : 1);
    }
  }
  // prefill-heavy: split by each role's time on one SM (a decode SM beside
  // a busy prefill streams about 70 bytes/ns)
  constexpr unsigned long long kMixedSmBytesPerNs = 70;
  const unsigned long long t_d1 = w.decode_bytes / kMixedSmBytesPerNs;
  const unsigned long long t_p1 = w.prefill_tiles * tile_ns;
  unsigned long long m = (static_cast<unsigned long long>(sms) * t_d1 + t_d1 + t_p1 - 1) /
                         (t_d1 + t_p1);  // decode SMs, rounded up
  if (m < 1) m = 1;
  if (m > static_cast<unsigned long long>(sms - 1)) m = sms - 1;
  return sms - static_cast<int>(m);
}

}  // namespace pkv
