// evo_fwd.cu — fused forward of memory-efficient biased Evoformer attention
// for sm_103a.
//
// Computes, per (b, n, h) slice, O = softmax(Q Kᵀ D^-1/2 + bias1 + bias2) V
// and the fp32 natural-log row log-sum-exp, never writing the L×L scores to
// device memory.  Definition: web page "DeepSpeed4Science 技术指南：AI4Science
// 大模型长序列训练与 Evoformer 内存高效注意力内核实战" §3.5 (scale, add bias,
// softmax, times V) and §3.7 (fp32 lse saved for the backward; bias1 is
// (B, N, 1, 1, L), bias2 is (B, 1, H, L, L)).
//
// Structure (one CTA per SM, persistent over work items (b, n, h, q-tile)):
//   warp 4      TMA producer: Q tile per item; K, V tiles, the pair-bias tile
//               and the key-mask chunk per key tile, into a 2-stage ring.
//   warp 5      MMA issuer (one thread): S = Q·Kᵀ into TMEM (2 buffers),
//               then O_j = P_j·V_j into TMEM (2 buffers), issued one key tile
//               behind S so the tensor core overlaps the softmax.
//   warps 0..3  softmax, one query row per thread (TMEM lane = row): scale and
//               bias in the log2 domain, online max / sum, P (fp16/bf16) into
//               swizzled shared memory for the P·V MMA, running rescale of the
//               fp32 output accumulator held in registers, epilogue.
// Key columns past L carry a -inf key-mask entry, so no other masking is
// needed; query rows past L are computed and not stored.
#include "evo_internal.h"
#include "evo_ptx.cuh"

namespace evo {
namespace {

constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 320;  // TMEM columns

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

template <int DP>
struct FwdLayout {
  static constexpr uint32_t kTileBytes = kTile * DP * 2;
  uint32_t q, k[kStages], v[kStages], b2[kStages], p[2], b1[kStages], bars, total;
  __host__ __device__ explicit FwdLayout(bool has_b2) {
    uint32_t off = 0;
    q = off;
    off += kTileBytes;
    for (int s = 0; s < kStages; ++s) k[s] = off + s * kTileBytes;
    off += kStages * kTileBytes;
    for (int s = 0; s < kStages; ++s) v[s] = off + s * kTileBytes;
    off += kStages * kTileBytes;
    for (int s = 0; s < kStages; ++s) b2[s] = off + s * 32768u;
    if (has_b2) off += kStages * 32768u;
    for (int b = 0; b < 2; ++b) p[b] = off + b * 32768u;
    off += 2 * 32768u;
    for (int s = 0; s < kStages; ++s) b1[s] = off + s * 512u;
    off += kStages * 512u;
    bars = off;
    off += (sizeof(FwdBars) + 127) & ~127u;
    total = off;
  }
};

struct ItemCoord {
  int b, n, h, qt;
};
__device__ __forceinline__ ItemCoord decode_item(long long item, const FwdArgs& a) {
  ItemCoord c;
  long long t = item;
  c.qt = static_cast<int>(t % a.QT);
  t /= a.QT;
  c.h = static_cast<int>(t % a.H);
  t /= a.H;
  c.n = static_cast<int>(t % a.N);
  c.b = static_cast<int>(t / a.N);
  return c;
}

// Bounded wait that ignores the abort flag: used only to drain work this
// thread itself put in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int* status) {
  volatile int never = 0;
  WaitGuard g{limit_ns, status, &never};
  mbar_wait(bar, parity, g);
}

// ------------------------------------------------------------ producer (warp 4)
template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void fwd_producer(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay,
                                             FwdBars* bars, const WaitGuard& g, int lane) {
  constexpr uint32_t kTB = FwdLayout<DP>::kTileBytes;
  const uint32_t kv_bytes = 2 * kTB + ((HAS_B2 && a.bias2_mode == kBias2Tma) ? 32768u : 0u);
  const int KT = a.QT;
  uint32_t kv_it = 0, q_it = 0;
  bool ok = true;
  for (long long item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
    const ItemCoord c = decode_item(item, a);
    const int bn = c.b * a.N + c.n;
    if (!mbar_wait(smem_u32(&bars->q_empty), (q_it & 1) ^ 1, g)) { ok = false; break; }
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(&bars->q_full), kTB);
      tma_load_4d(smem_u32(base + lay.q), &a.tq, smem_u32(&bars->q_full), 0, c.h, c.qt * kTile, bn);
    }
    ++q_it;
    const uint16_t* b1row = a.bias1 ? a.bias1 + static_cast<size_t>(bn) * a.L : nullptr;
    for (int jt = 0; jt < KT; ++jt, ++kv_it) {
      const uint32_t s = kv_it % kStages, ph = (kv_it / kStages) & 1;
      if (!mbar_wait(smem_u32(&bars->kv_empty[s]), ph ^ 1, g)) { ok = false; break; }
      // key-mask chunk, fp32 in the log2 domain; -inf past L
      {
        float4 m4;
        float* mv = reinterpret_cast<float*>(&m4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = jt * kTile + lane * 4 + e;
          float val = -INFINITY;
          if (j < a.L) val = b1row ? to_f32<BF16>(b1row[j]) * kLog2e : 0.0f;
          mv[e] = val;
        }
        *reinterpret_cast<float4*>(base + lay.b1[s] + lane * 16) = m4;
      }
      if (HAS_B2 && a.bias2_mode == kBias2Loads) {
        // generic path for L % 8 != 0: plain loads into the same swizzled layout
        const uint16_t* b2 = a.bias2 + static_cast<size_t>(c.b * a.H + c.h) * a.L * a.L;
        const int cc = lane * 4, half = cc >> 6, chunk = (cc & 63) >> 3, within = cc & 7;
        for (int r = 0; r < kTile; ++r) {
          const int i = c.qt * kTile + r;
          uint32_t w[2] = {0u, 0u};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = jt * kTile + cc + e;
            const uint32_t val = (i < a.L && j < a.L) ? b2[static_cast<size_t>(i) * a.L + j] : 0u;
            w[e >> 1] |= val << (16 * (e & 1));
          }
          *reinterpret_cast<uint2*>(base + lay.b2[s] + half * 16384 + swz_offset(r, chunk, 128) +
                                    within * 2) = make_uint2(w[0], w[1]);
        }
      }
      const uint32_t full = smem_u32(&bars->kv_full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, kv_bytes);
        tma_load_4d(smem_u32(base + lay.k[s]), &a.tk, full, 0, c.h, jt * kTile, bn);
        tma_load_4d(smem_u32(base + lay.v[s]), &a.tv, full, 0, c.h, jt * kTile, bn);
        if (HAS_B2 && a.bias2_mode == kBias2Tma) {
          const int bh = c.b * a.H + c.h;
          tma_load_3d(smem_u32(base + lay.b2[s]), &a.tb2, full, jt * kTile, c.qt * kTile, bh);
          tma_load_3d(smem_u32(base + lay.b2[s] + 16384), &a.tb2, full, jt * kTile + 64, c.qt * kTile, bh);
        }
      } else {
        mbar_arrive(full);
      }
    }
  }
  // Drain: every copy this warp started has landed before the CTA may exit.
  if (q_it > 0) drain_wait(smem_u32(&bars->q_full), (q_it - 1) & 1, a.wait_ns, a.status);
  for (uint32_t s = 0; s < kStages; ++s) {
    const uint32_t issued = (kv_it + kStages - 1 - s) / kStages;
    if (issued > 0) drain_wait(smem_u32(&bars->kv_full[s]), (issued - 1) & 1, a.wait_ns, a.status);
  }
}

// ------------------------------------------------------------ MMA issuer (warp 5, one thread)
template <int DP, bool BF16>
__device__ __forceinline__ bool fwd_issue_pv(uint32_t u, uint32_t su, uint8_t* base, const FwdLayout<DP>& lay,
                                             FwdBars* bars, uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_o = idesc_f16(128, DP, BF16, false, true);
  const uint32_t ub = u & 1, uph = (u >> 1) & 1;
  if (!mbar_wait(smem_u32(&bars->p_full[ub]), uph, g)) return false;
  if (!mbar_wait(smem_u32(&bars->o_free[ub]), uph ^ 1, g)) return false;
  tc_fence_after();
  const uint32_t p_addr = smem_u32(base + lay.p[ub]);
  const uint32_t v_addr = smem_u32(base + lay.v[su]);
  const uint32_t d = tmem + (ub ? kColO1 : kColO0);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint64_t ad = smem_desc(p_addr + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(v_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ss(d, ad, bd, id_o, k > 0);
  }
  umma_commit(smem_u32(&bars->o_full[ub]));
  umma_commit(smem_u32(&bars->p_empty[ub]));
  umma_commit(smem_u32(&bars->kv_empty[su]));
  return true;
}

template <int DP, bool BF16>
__device__ __forceinline__ void fwd_mma(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay, FwdBars* bars,
                                        uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
  const int KT = a.QT;
  uint32_t kv_it = 0, t_it = 0, q_it = 0, prev_stage = 0;
  bool ok = true;
  for (long long item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
    if (!mbar_wait(smem_u32(&bars->q_full), q_it & 1, g)) { ok = false; break; }
    ++q_it;
    tc_fence_after();
    const uint32_t q_addr = smem_u32(base + lay.q);
    for (int jt = 0; jt < KT; ++jt) {
      const uint32_t s = kv_it % kStages, kph = (kv_it / kStages) & 1;
      if (!mbar_wait(smem_u32(&bars->kv_full[s]), kph, g)) { ok = false; break; }
      const uint32_t buf = t_it & 1, bph = (t_it >> 1) & 1;
      if (!mbar_wait(smem_u32(&bars->s_free[buf]), bph ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      const uint32_t k_addr = smem_u32(base + lay.k[s]);
      const uint32_t d = tmem + (buf ? kColS1 : kColS0);
#pragma unroll
      for (int k = 0; k < DP / 16; ++k) {
        const uint64_t ad = smem_desc(q_addr + k * 32, 16, 8 * RB, SWZ);
        const uint64_t bd = smem_desc(k_addr + k * 32, 16, 8 * RB, SWZ);
        umma_ss(d, ad, bd, id_s, k > 0);
      }
      umma_commit(smem_u32(&bars->s_full[buf]));
      if (jt == KT - 1) umma_commit(smem_u32(&bars->q_empty));
      if (jt > 0 && !fwd_issue_pv<DP, BF16>(t_it - 1, prev_stage, base, lay, bars, tmem, g)) { ok = false; break; }
      prev_stage = s;
      ++t_it;
      ++kv_it;
    }
    if (ok && !fwd_issue_pv<DP, BF16>(t_it - 1, prev_stage, base, lay, bars, tmem, g)) ok = false;
  }
  // Drain: all MMAs this thread issued are complete before TMEM is freed.
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

// ------------------------------------------------------------ softmax (warps 0..3)
template <int DP>
__device__ __forceinline__ bool fwd_consume_o(uint32_t u, float alpha, float (&acc)[DP], FwdBars* bars,
                                              uint32_t trow, int lane, const WaitGuard& g) {
  const uint32_t ub = u & 1, uph = (u >> 1) & 1;
  if (!mbar_wait(smem_u32(&bars->o_full[ub]), uph, g)) return false;
  tc_fence_after();
  const uint32_t col = trow + (ub ? kColO1 : kColO0);
  uint32_t o[DP / 16][16];
#pragma unroll
  for (int c = 0; c < DP / 16; ++c) tmem_ld16(col + c * 16, o[c]);
#pragma unroll
  for (int c = 0; c < DP / 16; ++c) tmem_wait_ld(o[c]);
#pragma unroll
  for (int c = 0; c < DP / 16; ++c)
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[c * 16 + e] = fmaf(acc[c * 16 + e], alpha, __uint_as_float(o[c][e]));
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->o_free[ub]));
  return true;
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void fwd_softmax(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay,
                                            FwdBars* bars, uint32_t tmem, const WaitGuard& g) {
  const int r = threadIdx.x;  // query row within the tile == TMEM lane
  const int warp = r >> 5, lane = r & 31;
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int KT = a.QT;
  uint32_t kv_it = 0, t_it = 0;
  bool ok = true;
  for (long long item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
    const ItemCoord c = decode_item(item, a);
    float m = -INFINITY, l = 0.0f, a_prev = 0.0f;
    float acc[DP];
#pragma unroll
    for (int d = 0; d < DP; ++d) acc[d] = 0.0f;
    for (int jt = 0; jt < KT; ++jt) {
      const uint32_t s = kv_it % kStages, kph = (kv_it / kStages) & 1;
      const uint32_t buf = t_it & 1, bph = (t_it >> 1) & 1;
      if (!mbar_wait(smem_u32(&bars->kv_full[s]), kph, g)) { ok = false; break; }
      if (!mbar_wait(smem_u32(&bars->s_full[buf]), bph, g)) { ok = false; break; }
      tc_fence_after();
      float y[kTile];
      {
        uint32_t sr[4][32];
        const uint32_t col = trow + (buf ? kColS1 : kColS0);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(col + q * 32, sr[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_wait_ld(sr[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e) y[q * 32 + e] = __uint_as_float(sr[q][e]);
      }
      // y = S·s·log2e + bias1·log2e + bias2·log2e ; running max
      float tmax = -INFINITY;
      const float* b1 = reinterpret_cast<const float*>(base + lay.b1[s]);
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        const float4 m0 = *reinterpret_cast<const float4*>(b1 + c8 * 8);
        const float4 m1 = *reinterpret_cast<const float4*>(b1 + c8 * 8 + 4);
        const float mk[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        uint4 pb = make_uint4(0u, 0u, 0u, 0u);
        if (HAS_B2)
          pb = *reinterpret_cast<const uint4*>(base + lay.b2[s] + (c8 >> 3) * 16384 + swz_offset(r, c8 & 7, 128));
        const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float t = fmaf(y[c8 * 8 + e], a.scale_log2, mk[e]);
          if (HAS_B2) {
            const float b2v = (e & 1) ? unpack_hi<BF16>(pw[e >> 1]) : unpack_lo<BF16>(pw[e >> 1]);
            t = fmaf(b2v, kLog2e, t);
          }
          y[c8 * 8 + e] = t;
          tmax = fmaxf(tmax, t);
        }
      }
      // S buffer and the stage's bias tiles are no longer read by this warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->s_free[buf]));
        mbar_arrive(smem_u32(&bars->kv_empty[s]));
      }
      const float m_new = fmaxf(m, tmax);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      const float alpha = ex2(m - m_use);
      float rs = 0.0f;
#pragma unroll
      for (int e = 0; e < kTile; ++e) {
        y[e] = ex2(y[e] - m_use);
        rs += y[e];
      }
      l = fmaf(l, alpha, rs);
      // P -> shared memory (K-major, 128B swizzle, two 64-key halves)
      if (!mbar_wait(smem_u32(&bars->p_empty[buf]), bph ^ 1, g)) { ok = false; break; }
      uint8_t* pbase = base + lay.p[buf];
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint4 pk;
        pk.x = pack2<BF16>(y[c8 * 8 + 0], y[c8 * 8 + 1]);
        pk.y = pack2<BF16>(y[c8 * 8 + 2], y[c8 * 8 + 3]);
        pk.z = pack2<BF16>(y[c8 * 8 + 4], y[c8 * 8 + 5]);
        pk.w = pack2<BF16>(y[c8 * 8 + 6], y[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(pbase + (c8 >> 3) * 16384 + swz_offset(r, c8 & 7, 128)) = pk;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[buf]));
      if (jt > 0 && !fwd_consume_o<DP>(t_it - 1, a_prev, acc, bars, trow, lane, g)) { ok = false; break; }
      a_prev = alpha;
      m = m_new;
      ++t_it;
      ++kv_it;
    }
    if (!ok) break;
    if (!fwd_consume_o<DP>(t_it - 1, a_prev, acc, bars, trow, lane, g)) { ok = false; break; }
    // epilogue
    const int i = c.qt * kTile + r;
    if (i < a.L) {
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const size_t bn = static_cast<size_t>(c.b) * a.N + c.n;
      uint16_t* orow = a.out + ((bn * a.L + i) * a.H + c.h) * a.D;
#pragma unroll
      for (int c8 = 0; c8 < DP / 8; ++c8) {
        if (c8 * 8 < a.D) {
          uint4 pk;
          pk.x = pack2<BF16>(acc[c8 * 8 + 0] * inv, acc[c8 * 8 + 1] * inv);
          pk.y = pack2<BF16>(acc[c8 * 8 + 2] * inv, acc[c8 * 8 + 3] * inv);
          pk.z = pack2<BF16>(acc[c8 * 8 + 4] * inv, acc[c8 * 8 + 5] * inv);
          pk.w = pack2<BF16>(acc[c8 * 8 + 6] * inv, acc[c8 * 8 + 7] * inv);
          *reinterpret_cast<uint4*>(orow + c8 * 8) = pk;
        }
      }
      const float m_fin = (m == -INFINITY) ? 0.0f : m;
      a.lse[(bn * a.H + c.h) * a.L + i] = l > 0.0f ? (m_fin + lg2(l)) * kLn2 : -INFINITY;
    }
  }
}

template <int DP, bool BF16, bool HAS_B2>
__global__ void __launch_bounds__(192, 1) evo_fwd_kernel(const __grid_constant__ FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const FwdLayout<DP> lay(HAS_B2);
  FwdBars* bars = reinterpret_cast<FwdBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1 + 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->s_free[b]), 4);
      mbar_init(smem_u32(&bars->p_full[b]), 4);
      mbar_init(smem_u32(&bars->p_empty[b]), 1);
      mbar_init(smem_u32(&bars->o_full[b]), 1);
      mbar_init(smem_u32(&bars->o_free[b]), 4);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    if (HAS_B2 && a.bias2_mode == kBias2Tma) tma_prefetch_desc(&a.tb2);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&bars->tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const WaitGuard g{a.wait_ns, a.status, &bars->abort};

  if (warp == 4) {
    fwd_producer<DP, BF16, HAS_B2>(a, base, lay, bars, g, lane);
  } else if (warp == 5) {
    if (lane == 0) fwd_mma<DP, BF16>(a, base, lay, bars, tmem, g);
    __syncwarp();
  } else {
    fwd_softmax<DP, BF16, HAS_B2>(a, base, lay, bars, tmem, g);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DP, bool BF16, bool HAS_B2>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t st) {
  const FwdLayout<DP> lay(HAS_B2);
  // At least 116 KB so that two CTAs never share an SM: each allocates all 512
  // TMEM columns, and a second resident CTA would stall in tcgen05.alloc.
  const size_t smem = (lay.total + 1024 > 116u * 1024u) ? lay.total + 1024 : 116u * 1024u;
  auto kern = evo_fwd_kernel<DP, BF16, HAS_B2>;
  static bool limit_set[64] = {};
  cudaError_t e = ensure_smem_limit(kern, smem, limit_set);
  if (e != cudaSuccess) return e;
  const long long grid = a.items < num_sms() ? a.items : num_sms();
  kern<<<static_cast<unsigned>(grid), 192, smem, st>>>(a);
  return cudaGetLastError();
}

template <int DP, bool BF16>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t st) {
  return a.bias2_mode == kBias2None ? launch_fwd_t<DP, BF16, false>(a, st) : launch_fwd_t<DP, BF16, true>(a, st);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int DP, bool bf16, cudaStream_t st) {
  if (a.items <= 0) return cudaSuccess;
  switch (DP) {
    case 16: return bf16 ? launch_fwd_d<16, true>(a, st) : launch_fwd_d<16, false>(a, st);
    case 32: return bf16 ? launch_fwd_d<32, true>(a, st) : launch_fwd_d<32, false>(a, st);
    case 64: return bf16 ? launch_fwd_d<64, true>(a, st) : launch_fwd_d<64, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace evo
