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

// dQ summed over a slice's key tiles in the CTA's own fp32 blocks of the workspace (the
// per-key-tile and the streamed key-major schedules): one block of 32 rows × DP/2 columns
// per compute warp and query tile, staged in shared memory kStg bytes at a time and handed
// to the bulk-copy engine, which stores it (first key tile of the slice) or adds it in L2
// (later key tiles); the last key tile reads the sum back, adds its own tile, scales and
// writes dQ in the dtype.  Successive additions to one block are a query-tile sweep apart,
// and each is issued only once every bulk operation of the warp but the newest is
// complete, so they run one after another in key-tile order: dQ is bitwise reproducible.
template <int DP>
struct DqScr {
  static constexpr uint32_t kBlk = 32u * (DP / 2) * 4u;  // a compute warp's fp32 dQ block
  // staged (and sent) 1 KB at a time: small enough to leave room for the Q/dO stages
  static constexpr uint32_t kStg = kBlk < 1024u ? kBlk : 1024u;
};

// What the compute warps remember of a step until they consume its dQ tile.
struct DqStep {
  int b, n, h, it;
  bool first, last;  // first / last (kept) key tile of its slice
};

template <int DP, bool BF16>
__device__ __forceinline__ bool consume_dq_tile(const BwdArgs& a, const DqStep& d, uint32_t full_bar, uint32_t free_bar,
                                                uint32_t parity, uint32_t col, int r, int w, int hc, int lane,
                                                uint8_t* stg, const WaitGuard& g) {
  constexpr int HD = DP / 2;
  constexpr uint32_t kBlk = DqScr<DP>::kBlk, kStg = DqScr<DP>::kStg;
  constexpr int kPieces = static_cast<int>(kBlk / kStg), kChunks = static_cast<int>(kStg / 512);  // 512 B: 32 rows x 4 floats
  if (!mbar_wait_warp(full_bar, parity, g)) return false;
  tc_fence_after();
  float v[HD];
  if constexpr (HD == 8) {
    uint32_t x[8];
    tmem_ld8(col, x);
    tmem_wait_ld(x);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(x[e]);
  } else {
    uint32_t x[HD / 16][16];
#pragma unroll
    for (int q = 0; q < HD / 16; ++q) tmem_ld16(col + q * 16, x[q]);
#pragma unroll
    for (int q = 0; q < HD / 16; ++q) tmem_wait_ld(x[q]);
#pragma unroll
    for (int q = 0; q < HD / 16; ++q)
#pragma unroll
      for (int e = 0; e < 16; ++e) v[q * 16 + e] = __uint_as_float(x[q][e]);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(free_bar);
  float* blk = a.dq_scr + ((static_cast<size_t>(blockIdx.x) * a.QT + d.it) * kComputeWarps + w) * (kBlk / 4);
  if (!d.last) {
#pragma unroll
    for (int pc = 0; pc < kPieces; ++pc) {
      if (lane == 0) bulk_wait_read_all();  // the previous bulk operation has read the staging block
      __syncwarp();
      float4* sp = reinterpret_cast<float4*>(stg);
#pragma unroll
      for (int q = 0; q < kChunks; ++q) {
        const int c = pc * kChunks + q;
        sp[q * 32 + lane] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        float* dst = blk + pc * (kStg / 4);
        if (d.first) {
          bulk_store_s2g(dst, smem_u32(stg), kStg);
        } else {
          bulk_wait_all_but_newest();  // the piece's previous store or add (a sweep ago) is complete
          bulk_reduce_add_f32(dst, smem_u32(stg), kStg);
        }
        bulk_commit_group();
      }
    }
    return true;
  }
  if (!d.first) {  // the sum of the slice's earlier key tiles
    if (lane == 0) {
      bulk_wait_all_but_newest();
      fence_proxy_async_global();
    }
    __syncwarp();
    const float4* sp = reinterpret_cast<const float4*>(blk);
#pragma unroll
    for (int q = 0; q < HD / 4; ++q) {
      const float4 o = sp[q * 32 + lane];
      v[4 * q] += o.x;
      v[4 * q + 1] += o.y;
      v[4 * q + 2] += o.z;
      v[4 * q + 3] += o.w;
    }
  }
  const int i = d.it * kTile + r;
  if (i >= a.L) return true;
  const long long bn = static_cast<long long>(d.b) * a.N + d.n;
  uint16_t* dq = a.dq + bn * a.r_dq.bn + static_cast<long long>(i) * a.r_dq.l + d.h * a.D + hc * HD;
#pragma unroll
  for (int e = 0; e < HD; e += 8)
    if (hc * HD + e < a.D) {
      uint4 pk;
      pk.x = pack2<BF16>(v[e + 0] * a.scale, v[e + 1] * a.scale);
      pk.y = pack2<BF16>(v[e + 2] * a.scale, v[e + 3] * a.scale);
      pk.z = pack2<BF16>(v[e + 4] * a.scale, v[e + 5] * a.scale);
      pk.w = pack2<BF16>(v[e + 6] * a.scale, v[e + 7] * a.scale);
      *reinterpret_cast<uint4*>(dq + e) = pk;
    }
  return true;
}

size_t one_cta_per_sm(size_t bytes) { return bytes > 116u * 1024u ? bytes : 116u * 1024u; }

}  // namespace
}  // namespace evo
