// evo_bwd_common.cuh — pieces shared by the backward translation units:
// warp roles, shared-memory fill helpers for the key mask, the pair bias and
// the per-query lse / delta values, and the item iterators.  Internal.
#pragma once

#include "evo_internal.h"
#include "evo_ptx.cuh"

namespace evo {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int* status) {
  volatile int never = 0;
  WaitGuard g{limit_ns, status, &never};
  mbar_wait(bar, parity, g);
}

// ============================================================ shared pieces
constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 2) * 32;
constexpr int kProducerWarp = kComputeWarps, kMmaWarp = kComputeWarps + 1;
constexpr size_t kMaxSmem = 232448;  // 227 KB opt-in limit per block

// Pair-bias tile [128 queries][128 keys] in two 64-key halves, 128B swizzle —
// the layout the 3-D TMA map with box (64, 128, 1) writes.  Generic-load fill
// for L % 8 != 0 (no TMA: the row pitch is not a multiple of 16 bytes).
__device__ __forceinline__ void fill_b2_tile_loads(uint8_t* dst, const uint16_t* b2, int L, int i0, int j0,
                                                   int lane) {
  const int cc = lane * 4, half = cc >> 6, chunk = (cc & 63) >> 3, within = cc & 7;
  for (int r = 0; r < kTile; ++r) {
    const int i = i0 + r;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + cc + e;
      const uint32_t val = (i < L && j < L) ? b2[static_cast<size_t>(i) * L + j] : 0u;
      w[e >> 1] |= val << (16 * (e & 1));
    }
    *reinterpret_cast<uint2*>(dst + half * 16384 + swz_offset(r, chunk, 128) + within * 2) =
        make_uint2(w[0], w[1]);
  }
}

// Key-mask chunk for keys j0..j0+127: fp32 × log2(e); -inf past L.
template <bool BF16>
__device__ __forceinline__ void fill_b1_chunk(float* dst, const uint16_t* b1row, int L, int j0, int lane) {
  float4 m4;
  float* mv = reinterpret_cast<float*>(&m4);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = j0 + lane * 4 + e;
    float val = -INFINITY;
    if (j < L) val = b1row ? to_f32<BF16>(b1row[j]) * kLog2e : 0.0f;
    mv[e] = val;
  }
  reinterpret_cast<float4*>(dst)[lane] = m4;
}

// The same chunk in two halves: loads issued one stage ahead (raw values held
// in registers, so their latency overlaps the wait for a free stage), then
// converted and written when the stage is filled.
struct B1Raw {
  uint16_t v[4];
};
__device__ __forceinline__ void b1_prefetch(B1Raw& raw, const uint16_t* b1row, int L, int j0, int lane) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = j0 + lane * 4 + e;
    raw.v[e] = (b1row && j < L) ? b1row[j] : static_cast<uint16_t>(0);
  }
}
template <bool BF16>
__device__ __forceinline__ void b1_store(float* dst, const B1Raw& raw, bool has_b1, int L, int j0, int lane) {
  float4 m4;
  float* mv = reinterpret_cast<float*>(&m4);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = j0 + lane * 4 + e;
    mv[e] = j < L ? (has_b1 ? to_f32<BF16>(raw.v[e]) * kLog2e : 0.0f) : -INFINITY;
  }
  reinterpret_cast<float4*>(dst)[lane] = m4;
}

// lse (× log2 e; +inf for rows past L or with an empty softmax, so P = 0) and
// delta for queries i0..i0+127 of slice bnh, prefetched like the key mask.
struct LdRaw {
  float l[4], d[4];
};
__device__ __forceinline__ void ld_prefetch(LdRaw& raw, const float* lse, const float* delta, size_t bnh, int L,
                                            int i0, int lane) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = i0 + lane * 4 + e;
    raw.l[e] = i < L ? lse[bnh * L + i] : -INFINITY;
    raw.d[e] = i < L ? delta[bnh * L + i] : 0.0f;
  }
}
__device__ __forceinline__ void ld_store(float* dst, const LdRaw& raw, int lane) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x = raw.l[e];
    dst[lane * 4 + e] = (x == -INFINITY) ? INFINITY : x * kLog2e;
    dst[128 + lane * 4 + e] = raw.d[e];
  }
}
__device__ __forceinline__ void fill_lse_delta(float* dst, const float* lse, const float* delta, size_t bnh, int L,
                                               int i0, int lane) {
  LdRaw raw;
  ld_prefetch(raw, lse, delta, bnh, L, i0, lane);
  ld_store(dst, raw, lane);
}

// (b, h, n) slice iterator, n fastest.
struct SlIter {
  int b, h, n;
  __device__ __forceinline__ void init(long long item, const BwdArgs& a) {
    n = static_cast<int>(item % a.N);
    const long long t = item / a.N;
    h = static_cast<int>(t % a.H);
    b = static_cast<int>(t / a.H);
  }
  __device__ __forceinline__ void next(const BwdArgs& a) {
    if (++n == a.N) {
      n = 0;
      if (++h == a.H) {
        h = 0;
        ++b;
      }
    }
  }
};

size_t one_cta_per_sm(size_t bytes) { return bytes > 116u * 1024u ? bytes : 116u * 1024u; }

}  // namespace
}  // namespace evo
