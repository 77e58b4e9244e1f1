// evo_bwd.cu — backward of memory-efficient biased Evoformer attention for
// sm_103a.
//
// Definition: web page "DeepSpeed4Science 技术指南：AI4Science 大模型长序列训练
// 与 Evoformer 内存高效注意力内核实战" §3.7: the backward first forms delta, then
// dQ, dK, dV and the bias gradients, with bias gradients accumulated in fp32
// and cast back to the input dtype; §3.2: the backward recomputes (a little
// extra arithmetic in exchange for not storing the attention matrix).
//
// With P = exp(s·QKᵀ + bias − lse) rebuilt from the saved lse:
//   delta_i = Σ_d dO_id O_id           dP = dO Vᵀ        dS = P ∘ (dP − delta)
//   dV = Pᵀ dO      dK = s·dSᵀ Q      dQ = s·dS K      dbias2[b,h] = Σ_n dS
//
// Kernels, in launch order on the caller's stream:
//   evo_bwd_pre       delta [B,N,H,L] fp32; zeroes the fp32 dQ accumulator.
//   evo_bwd_main      persistent over (b, n, h, key tile).  Per query tile the
//                     MMA thread computes S = Q Kᵀ and dP = dO Vᵀ into TMEM
//                     (lane = query); four compute warps form P and dS (fp16 /
//                     bf16) in swizzled shared memory; the MMA thread then
//                     accumulates dV += Pᵀ dO and dK += dSᵀ Q in TMEM (the same
//                     smem tiles read as MN-major A operands) and forms
//                     dQ_tile = dS K, which the compute warps add into the fp32
//                     accumulator.  dK and dV are written once per item.
//   evo_bwd_dq_cast   dQ = accumulator rounded to the dtype.
//   evo_bwd_db2_part  (pair bias only) per (b, h, query tile, key tile,
//                     n-group): recompute S, dP, P, dS and sum dS over the
//                     group's n in a fixed order in registers; write fp32.
//   evo_bwd_db2_sum   dbias2 = Σ_groups partial in fixed order, cast.
// Both pair-bias stages run in a fixed order, so dbias2 is bitwise
// reproducible.  dQ uses fp32 atomics and is not.
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

// ============================================================ evo_bwd_pre
template <int DP, bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_pre(const BwdArgs a) {
  const long long rows = static_cast<long long>(a.B) * a.N * a.L * a.H;
  for (long long row = blockIdx.x * 256ll + threadIdx.x; row < rows; row += gridDim.x * 256ll) {
    // row enumerates (b, n, i, h) in memory order of [B,N,L,H,D]
    const int h = static_cast<int>(row % a.H);
    long long t = row / a.H;
    const int i = static_cast<int>(t % a.L);
    const long long bn = t / a.L;
    const uint4* o = reinterpret_cast<const uint4*>(a.out + row * a.D);
    const uint4* g = reinterpret_cast<const uint4*>(a.dout + row * a.D);
    float4* acc = reinterpret_cast<float4*>(a.dq_acc + row * a.D);
    float sum = 0.0f;
#pragma unroll
    for (int c = 0; c < DP / 8; ++c) {
      if (c * 8 < a.D) {
        const uint4 ov = o[c], gv = g[c];
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sum = fmaf(unpack_lo<BF16>(ow[e]), unpack_lo<BF16>(gw[e]), sum);
          sum = fmaf(unpack_hi<BF16>(ow[e]), unpack_hi<BF16>(gw[e]), sum);
        }
        acc[2 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
        acc[2 * c + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    a.delta[(bn * a.H + h) * a.L + i] = sum;
  }
}

// ============================================================ evo_bwd_dq_cast
template <bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_dq_cast(const BwdArgs a) {
  const long long n8 = static_cast<long long>(a.B) * a.N * a.L * a.H * a.D / 8;
  for (long long v = blockIdx.x * 256ll + threadIdx.x; v < n8; v += gridDim.x * 256ll) {
    const float4 x = reinterpret_cast<const float4*>(a.dq_acc)[2 * v];
    const float4 y = reinterpret_cast<const float4*>(a.dq_acc)[2 * v + 1];
    uint4 pk;
    pk.x = pack2<BF16>(x.x, x.y);
    pk.y = pack2<BF16>(x.z, x.w);
    pk.z = pack2<BF16>(y.x, y.y);
    pk.w = pack2<BF16>(y.z, y.w);
    reinterpret_cast<uint4*>(a.dq)[v] = pk;
  }
}

// ============================================================ evo_bwd_db2_sum
template <bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_db2_sum(const BwdArgs a) {
  const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
  for (long long e = blockIdx.x * 256ll + threadIdx.x; e < plane; e += gridDim.x * 256ll) {
    float s = 0.0f;
    for (int g = 0; g < a.groups; ++g) s += a.db2_part[g * plane + e];  // fixed group order
    const uint32_t p = pack2<BF16>(s, 0.0f);
    a.dbias2[e] = static_cast<uint16_t>(p & 0xFFFFu);
  }
}

// ============================================================ shared pieces
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

// P (or dS) row of one thread -> [query][key] tile, K-major 128B swizzle, two 64-key halves.
template <bool BF16>
__device__ __forceinline__ void store_row_chunk(uint8_t* tile, int r, int c, const float (&x)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk16 = c * 4 + q;  // 16-byte chunk index 0..15 along the 128 keys
    uint4 pk;
    pk.x = pack2<BF16>(x[q * 8 + 0], x[q * 8 + 1]);
    pk.y = pack2<BF16>(x[q * 8 + 2], x[q * 8 + 3]);
    pk.z = pack2<BF16>(x[q * 8 + 4], x[q * 8 + 5]);
    pk.w = pack2<BF16>(x[q * 8 + 6], x[q * 8 + 7]);
    *reinterpret_cast<uint4*>(tile + (chunk16 >> 3) * 16384 + swz_offset(r, chunk16 & 7, 128)) = pk;
  }
}

// ============================================================ evo_bwd_main
constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 320, kColDQ0 = 384, kColDQ1 = 448;

struct MainBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t st_full, st_free;
  uint64_t ds_full, ds_empty;
  uint64_t dq_full[2], dq_free[2];
  uint64_t dkdv_full, dkdv_free;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

template <int DP>
struct MainLayout {
  static constexpr int kStages = DP == 64 ? 1 : 2;
  static constexpr uint32_t kTB = kTile * DP * 2;
  uint32_t k, v, q[2], d_o[2], b2[2], b1, p, ds, bars, total;
  __host__ __device__ explicit MainLayout(bool has_b2) {
    uint32_t off = 0;
    k = off;
    off += kTB;
    v = off;
    off += kTB;
    for (int s = 0; s < kStages; ++s) q[s] = off + s * kTB;
    off += kStages * kTB;
    for (int s = 0; s < kStages; ++s) d_o[s] = off + s * kTB;
    off += kStages * kTB;
    for (int s = 0; s < kStages; ++s) b2[s] = off + s * 32768u;
    if (has_b2) off += kStages * 32768u;
    p = off;
    off += 32768u;
    ds = off;
    off += 32768u;
    b1 = off;
    off += 1024u;
    bars = off;
    off += (sizeof(MainBars) + 127) & ~127u;
    total = off;
  }
};

struct MainItem {
  int b, n, h, jt;
};
__device__ __forceinline__ MainItem main_item(long long item, const BwdArgs& a) {
  MainItem c;
  long long t = item;
  c.jt = static_cast<int>(t % a.QT);
  t /= a.QT;
  c.h = static_cast<int>(t % a.H);
  t /= a.H;
  c.n = static_cast<int>(t % a.N);
  c.b = static_cast<int>(t / a.N);
  return c;
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void main_producer(const BwdArgs& a, uint8_t* base, const MainLayout<DP>& lay,
                                              MainBars* bars, const WaitGuard& g, int lane, long long items) {
  constexpr int NS = MainLayout<DP>::kStages;
  constexpr uint32_t kTB = MainLayout<DP>::kTB;
  const uint32_t q_bytes = 2 * kTB + ((HAS_B2 && a.bias2_mode == kBias2Tma) ? 32768u : 0u);
  uint32_t it_ctr = 0, item_ctr = 0;
  bool ok = true;
  for (long long item = blockIdx.x; ok && item < items; item += gridDim.x, ++item_ctr) {
    const MainItem c = main_item(item, a);
    const int bn = c.b * a.N + c.n;
    if (!mbar_wait(smem_u32(&bars->kv_empty), (item_ctr & 1) ^ 1, g)) { ok = false; break; }
    fill_b1_chunk<BF16>(reinterpret_cast<float*>(base + lay.b1),
                        a.bias1 ? a.bias1 + static_cast<size_t>(bn) * a.L : nullptr, a.L, c.jt * kTile, lane);
    if (lane == 0) {
      const uint32_t full = smem_u32(&bars->kv_full);
      mbar_arrive_expect_tx(full, 2 * kTB);
      tma_load_4d(smem_u32(base + lay.k), &a.tk, full, 0, c.h, c.jt * kTile, bn);
      tma_load_4d(smem_u32(base + lay.v), &a.tv, full, 0, c.h, c.jt * kTile, bn);
    } else {
      mbar_arrive(smem_u32(&bars->kv_full));
    }
    for (int it = 0; it < a.QT; ++it, ++it_ctr) {
      const uint32_t s = it_ctr % NS, ph = (it_ctr / NS) & 1;
      if (!mbar_wait(smem_u32(&bars->q_empty[s]), ph ^ 1, g)) { ok = false; break; }
      if (HAS_B2 && a.bias2_mode == kBias2Loads)
        fill_b2_tile_loads(base + lay.b2[s], a.bias2 + static_cast<size_t>(c.b * a.H + c.h) * a.L * a.L, a.L,
                           it * kTile, c.jt * kTile, lane);
      const uint32_t full = smem_u32(&bars->q_full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, q_bytes);
        tma_load_4d(smem_u32(base + lay.q[s]), &a.tq, full, 0, c.h, it * kTile, bn);
        tma_load_4d(smem_u32(base + lay.d_o[s]), &a.tdo, full, 0, c.h, it * kTile, bn);
        if (HAS_B2 && a.bias2_mode == kBias2Tma) {
          const int bh = c.b * a.H + c.h;
          tma_load_3d(smem_u32(base + lay.b2[s]), &a.tb2, full, c.jt * kTile, it * kTile, bh);
          tma_load_3d(smem_u32(base + lay.b2[s] + 16384), &a.tb2, full, c.jt * kTile + 64, it * kTile, bh);
        }
      } else {
        mbar_arrive(full);
      }
    }
  }
  if (item_ctr > 0) drain_wait(smem_u32(&bars->kv_full), (item_ctr - 1) & 1, a.wait_ns, a.status);
  for (uint32_t s = 0; s < static_cast<uint32_t>(NS); ++s) {
    const uint32_t issued = (it_ctr + NS - 1 - s) / NS;
    if (issued > 0) drain_wait(smem_u32(&bars->q_full[s]), (issued - 1) & 1, a.wait_ns, a.status);
  }
}

template <int DP, bool BF16>
__device__ __forceinline__ void main_mma(const BwdArgs& a, uint8_t* base, const MainLayout<DP>& lay,
                                         MainBars* bars, uint32_t tmem, const WaitGuard& g, long long items) {
  constexpr int NS = MainLayout<DP>::kStages;
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);   // S, dP: K-major A and B
  constexpr uint32_t id_kv = idesc_f16(128, DP, BF16, true, true);     // dV, dK: MN-major A and B
  constexpr uint32_t id_q = idesc_f16(128, DP, BF16, false, true);     // dQ: K-major A, MN-major B
  const uint32_t p_addr = smem_u32(base + lay.p), ds_addr = smem_u32(base + lay.ds);
  const uint32_t k_addr = smem_u32(base + lay.k), v_addr = smem_u32(base + lay.v);
  uint32_t it_ctr = 0, item_ctr = 0;
  bool ok = true;
  for (long long item = blockIdx.x; ok && item < items; item += gridDim.x, ++item_ctr) {
    if (!mbar_wait(smem_u32(&bars->kv_full), item_ctr & 1, g)) { ok = false; break; }
    // dK / dV of the previous item have been read out of TMEM
    if (!mbar_wait(smem_u32(&bars->dkdv_free), (item_ctr & 1) ^ 1, g)) { ok = false; break; }
    for (int it = 0; it < a.QT; ++it, ++it_ctr) {
      const uint32_t s = it_ctr % NS, ph = (it_ctr / NS) & 1;
      if (!mbar_wait(smem_u32(&bars->q_full[s]), ph, g)) { ok = false; break; }
      if (!mbar_wait(smem_u32(&bars->st_free), (it_ctr & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      const uint32_t q_addr = smem_u32(base + lay.q[s]), do_addr = smem_u32(base + lay.d_o[s]);
#pragma unroll
      for (int k = 0; k < DP / 16; ++k) {
        umma_ss(tmem + kColS, smem_desc(q_addr + k * 32, 16, 8 * RB, SWZ), smem_desc(k_addr + k * 32, 16, 8 * RB, SWZ),
                id_s, k > 0);
      }
#pragma unroll
      for (int k = 0; k < DP / 16; ++k) {
        umma_ss(tmem + kColDP, smem_desc(do_addr + k * 32, 16, 8 * RB, SWZ),
                smem_desc(v_addr + k * 32, 16, 8 * RB, SWZ), id_s, k > 0);
      }
      umma_commit(smem_u32(&bars->st_full));
      // P and dS of this query tile are in shared memory
      if (!mbar_wait(smem_u32(&bars->ds_full), it_ctr & 1, g)) { ok = false; break; }
      const uint32_t qb = it_ctr & 1;
      if (!mbar_wait(smem_u32(&bars->dq_free[qb]), ((it_ctr >> 1) & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // dV += Pᵀ dO   (K = 128 queries)
        const uint64_t ad = smem_desc(p_addr + k * 16 * 128, 16384, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(do_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
        umma_ss(tmem + kColDV, ad, bd, id_kv, (it > 0 || k > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // dK += dSᵀ Q
        const uint64_t ad = smem_desc(ds_addr + k * 16 * 128, 16384, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(q_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
        umma_ss(tmem + kColDK, ad, bd, id_kv, (it > 0 || k > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // dQ_tile = dS K   (K = 128 keys)
        const uint64_t ad = smem_desc(ds_addr + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(k_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
        umma_ss(tmem + (qb ? kColDQ1 : kColDQ0), ad, bd, id_q, k > 0);
      }
      umma_commit(smem_u32(&bars->ds_empty));
      umma_commit(smem_u32(&bars->q_empty[s]));
      umma_commit(smem_u32(&bars->dq_full[qb]));
    }
    if (!ok) break;
    umma_commit(smem_u32(&bars->dkdv_full));
    umma_commit(smem_u32(&bars->kv_empty));
  }
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

// dQ tile (TMEM lanes = queries of tile it) -> fp32 accumulator (scaled by s).
template <int DP>
__device__ __forceinline__ bool main_consume_dq(const BwdArgs& a, const MainItem& c, int it, uint32_t ctr,
                                                MainBars* bars, uint32_t trow, int r, int lane, const WaitGuard& g) {
  const uint32_t qb = ctr & 1;
  if (!mbar_wait(smem_u32(&bars->dq_full[qb]), (ctr >> 1) & 1, g)) return false;
  tc_fence_after();
  uint32_t v[DP / 16][16];
#pragma unroll
  for (int q = 0; q < DP / 16; ++q) tmem_ld16(trow + (qb ? kColDQ1 : kColDQ0) + q * 16, v[q]);
#pragma unroll
  for (int q = 0; q < DP / 16; ++q) tmem_wait_ld(v[q]);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free[qb]));
  const int i = it * kTile + r;
  if (i < a.L) {
    float* dst = a.dq_acc + ((static_cast<size_t>(c.b) * a.N + c.n) * a.L + i) * a.H * a.D + static_cast<size_t>(c.h) * a.D;
#pragma unroll
    for (int q = 0; q < DP / 16; ++q)
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        if (q * 16 + e < a.D)
          red_add_v4(dst + q * 16 + e, __uint_as_float(v[q][e]) * a.scale, __uint_as_float(v[q][e + 1]) * a.scale,
                     __uint_as_float(v[q][e + 2]) * a.scale, __uint_as_float(v[q][e + 3]) * a.scale);
  }
  return true;
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void main_compute(const BwdArgs& a, uint8_t* base, const MainLayout<DP>& lay,
                                             MainBars* bars, uint32_t tmem, const WaitGuard& g, long long items) {
  constexpr int NS = MainLayout<DP>::kStages;
  const int r = threadIdx.x;  // query row within the tile == TMEM lane (for S, dP, dQ) and key row (dK, dV)
  const int warp = r >> 5, lane = r & 31;
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const float* b1s = reinterpret_cast<const float*>(base + lay.b1);
  uint32_t it_ctr = 0, item_ctr = 0;
  bool ok = true;
  for (long long item = blockIdx.x; ok && item < items; item += gridDim.x, ++item_ctr) {
    const MainItem c = main_item(item, a);
    const size_t bnh = (static_cast<size_t>(c.b) * a.N + c.n) * a.H + c.h;
    if (!mbar_wait(smem_u32(&bars->kv_full), item_ctr & 1, g)) { ok = false; break; }
    for (int it = 0; it < a.QT; ++it, ++it_ctr) {
      const uint32_t s = it_ctr % NS, ph = (it_ctr / NS) & 1;
      const int i = it * kTile + r;
      float lse2 = INFINITY, dlt = 0.0f;  // rows past L (and empty rows) get P = 0
      if (i < a.L) {
        const float lv = a.lse[bnh * a.L + i];
        lse2 = (lv == -INFINITY) ? INFINITY : lv * kLog2e;
        dlt = a.delta[bnh * a.L + i];
      }
      if (!mbar_wait(smem_u32(&bars->q_full[s]), ph, g)) { ok = false; break; }
      if (!mbar_wait(smem_u32(&bars->st_full), it_ctr & 1, g)) { ok = false; break; }
      if (!mbar_wait(smem_u32(&bars->ds_empty), (it_ctr & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      const uint8_t* b2t = base + lay.b2[s];
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], pv[32];
        tmem_ld32(trow + kColS + cc * 32, sv);
        tmem_ld32(trow + kColDP + cc * 32, pv);
        tmem_wait_ld(sv);
        tmem_wait_ld(pv);
        float p[32], ds[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk16 = cc * 4 + q;
          uint4 pb = make_uint4(0u, 0u, 0u, 0u);
          if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2t + (chunk16 >> 3) * 16384 + swz_offset(r, chunk16 & 7, 128));
          const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
          const float4 m0 = *reinterpret_cast<const float4*>(b1s + chunk16 * 8);
          const float4 m1 = *reinterpret_cast<const float4*>(b1s + chunk16 * 8 + 4);
          const float mk[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int x = q * 8 + e;
            float y = fmaf(__uint_as_float(sv[x]), a.scale_log2, mk[e]);
            if (HAS_B2) y = fmaf((e & 1) ? unpack_hi<BF16>(pw[e >> 1]) : unpack_lo<BF16>(pw[e >> 1]), kLog2e, y);
            const float pr = ex2(y - lse2);
            p[x] = pr;
            ds[x] = pr * (__uint_as_float(pv[x]) - dlt);
          }
        }
        store_row_chunk<BF16>(base + lay.p, r, cc, p);
        store_row_chunk<BF16>(base + lay.ds, r, cc, ds);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->st_free));
        mbar_arrive(smem_u32(&bars->q_empty[s]));
        mbar_arrive(smem_u32(&bars->ds_full));
      }
      if (it > 0 && !main_consume_dq<DP>(a, c, it - 1, it_ctr - 1, bars, trow, r, lane, g)) { ok = false; break; }
    }
    if (!ok) break;
    if (!main_consume_dq<DP>(a, c, a.QT - 1, it_ctr - 1, bars, trow, r, lane, g)) { ok = false; break; }
    // dK, dV (TMEM lanes = keys of this item's key tile)
    if (!mbar_wait(smem_u32(&bars->dkdv_full), item_ctr & 1, g)) { ok = false; break; }
    tc_fence_after();
    uint32_t kv[DP / 16][16], vv[DP / 16][16];
#pragma unroll
    for (int q = 0; q < DP / 16; ++q) {
      tmem_ld16(trow + kColDK + q * 16, kv[q]);
      tmem_ld16(trow + kColDV + q * 16, vv[q]);
    }
#pragma unroll
    for (int q = 0; q < DP / 16; ++q) {
      tmem_wait_ld(kv[q]);
      tmem_wait_ld(vv[q]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&bars->dkdv_free));
      mbar_arrive(smem_u32(&bars->kv_empty));
    }
    const int j = c.jt * kTile + r;
    if (j < a.L) {
      const size_t off = ((static_cast<size_t>(c.b) * a.N + c.n) * a.L + j) * a.H * a.D + static_cast<size_t>(c.h) * a.D;
#pragma unroll
      for (int q = 0; q < DP / 16; ++q)
#pragma unroll
        for (int e = 0; e < 16; e += 8)
          if (q * 16 + e < a.D) {
            uint4 pk, pv4;
            pk.x = pack2<BF16>(__uint_as_float(kv[q][e + 0]) * a.scale, __uint_as_float(kv[q][e + 1]) * a.scale);
            pk.y = pack2<BF16>(__uint_as_float(kv[q][e + 2]) * a.scale, __uint_as_float(kv[q][e + 3]) * a.scale);
            pk.z = pack2<BF16>(__uint_as_float(kv[q][e + 4]) * a.scale, __uint_as_float(kv[q][e + 5]) * a.scale);
            pk.w = pack2<BF16>(__uint_as_float(kv[q][e + 6]) * a.scale, __uint_as_float(kv[q][e + 7]) * a.scale);
            pv4.x = pack2<BF16>(__uint_as_float(vv[q][e + 0]), __uint_as_float(vv[q][e + 1]));
            pv4.y = pack2<BF16>(__uint_as_float(vv[q][e + 2]), __uint_as_float(vv[q][e + 3]));
            pv4.z = pack2<BF16>(__uint_as_float(vv[q][e + 4]), __uint_as_float(vv[q][e + 5]));
            pv4.w = pack2<BF16>(__uint_as_float(vv[q][e + 6]), __uint_as_float(vv[q][e + 7]));
            *reinterpret_cast<uint4*>(a.dk + off + q * 16 + e) = pk;
            *reinterpret_cast<uint4*>(a.dv + off + q * 16 + e) = pv4;
          }
    }
  }
}

template <int DP, bool BF16, bool HAS_B2>
__global__ void __launch_bounds__(192, 1) evo_bwd_main(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const MainLayout<DP> lay(HAS_B2);
  MainBars* bars = reinterpret_cast<MainBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long items = static_cast<long long>(a.B) * a.N * a.H * a.QT;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->kv_full), 32);
    mbar_init(smem_u32(&bars->kv_empty), 1 + 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 32);
      mbar_init(smem_u32(&bars->q_empty[s]), 1 + 4);
      mbar_init(smem_u32(&bars->dq_full[s]), 1);
      mbar_init(smem_u32(&bars->dq_free[s]), 4);
    }
    mbar_init(smem_u32(&bars->st_full), 1);
    mbar_init(smem_u32(&bars->st_free), 4);
    mbar_init(smem_u32(&bars->ds_full), 4);
    mbar_init(smem_u32(&bars->ds_empty), 1);
    mbar_init(smem_u32(&bars->dkdv_full), 1);
    mbar_init(smem_u32(&bars->dkdv_free), 4);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    tma_prefetch_desc(&a.tdo);
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
    main_producer<DP, BF16, HAS_B2>(a, base, lay, bars, g, lane, items);
  } else if (warp == 5) {
    if (lane == 0) main_mma<DP, BF16>(a, base, lay, bars, tmem, g, items);
    __syncwarp();
  } else {
    main_compute<DP, BF16, HAS_B2>(a, base, lay, bars, tmem, g, items);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ evo_bwd_db2_part
constexpr uint32_t kColS_0 = 0, kColDP_0 = 128, kColS_1 = 256, kColDP_1 = 384;

struct PartBars {
  uint64_t b2_full;
  uint64_t st_full[2], st_free[2];      // stage ring (Q, dO, K, V, key mask)
  uint64_t mm_full[2], mm_free[2];      // TMEM S/dP double buffer
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

template <int DP>
struct PartLayout {
  static constexpr uint32_t kTB = kTile * DP * 2;
  uint32_t q[2], d_o[2], k[2], v[2], b1[2], b2, bars, total;
  __host__ __device__ PartLayout() {
    uint32_t off = 0;
    for (int s = 0; s < 2; ++s) {
      q[s] = off;
      d_o[s] = off + kTB;
      k[s] = off + 2 * kTB;
      v[s] = off + 3 * kTB;
      off += 4 * kTB;
    }
    b2 = off;
    off += 32768u;
    for (int s = 0; s < 2; ++s) b1[s] = off + s * 512u;
    off += 1024u;
    bars = off;
    off += (sizeof(PartBars) + 127) & ~127u;
    total = off;
  }
};

struct PartItem {
  int b, h, it, jt, grp, n0, n1;
};
__device__ __forceinline__ PartItem part_item(const BwdArgs& a) {
  PartItem c;
  long long t = blockIdx.x;
  c.jt = static_cast<int>(t % a.QT);
  t /= a.QT;
  c.it = static_cast<int>(t % a.QT);
  t /= a.QT;
  c.grp = static_cast<int>(t % a.groups);
  t /= a.groups;
  c.h = static_cast<int>(t % a.H);
  c.b = static_cast<int>(t / a.H);
  c.n0 = c.grp * a.group_size;
  c.n1 = min(a.N, c.n0 + a.group_size);
  return c;
}

template <int DP, bool BF16>
__global__ void __launch_bounds__(192, 1) evo_bwd_db2_part(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const PartLayout<DP> lay;
  PartBars* bars = reinterpret_cast<PartBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PartItem c = part_item(a);
  const int nn = c.n1 - c.n0;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->b2_full), 32);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->st_full[s]), 32);
      mbar_init(smem_u32(&bars->st_free[s]), 1 + 4);
      mbar_init(smem_u32(&bars->mm_full[s]), 1);
      mbar_init(smem_u32(&bars->mm_free[s]), 4);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&bars->tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const WaitGuard g{a.wait_ns, a.status, &bars->abort};
  constexpr uint32_t kTB = PartLayout<DP>::kTB;
  const int bh = c.b * a.H + c.h;

  if (warp == 4) {  // ---------------- producer
    if (a.bias2_mode == kBias2Loads)
      fill_b2_tile_loads(base + lay.b2, a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L, c.it * kTile,
                         c.jt * kTile, lane);
    if (lane == 0) {
      const uint32_t full = smem_u32(&bars->b2_full);
      if (a.bias2_mode == kBias2Tma) {
        mbar_arrive_expect_tx(full, 32768u);
        tma_load_3d(smem_u32(base + lay.b2), &a.tb2, full, c.jt * kTile, c.it * kTile, bh);
        tma_load_3d(smem_u32(base + lay.b2 + 16384), &a.tb2, full, c.jt * kTile + 64, c.it * kTile, bh);
      } else {
        mbar_arrive(full);
      }
    } else {
      mbar_arrive(smem_u32(&bars->b2_full));
    }
    int k = 0;
    for (; k < nn; ++k) {
      const int s = k & 1, ph = (k >> 1) & 1;
      if (!mbar_wait(smem_u32(&bars->st_free[s]), ph ^ 1, g)) break;
      const int bn = c.b * a.N + c.n0 + k;
      fill_b1_chunk<BF16>(reinterpret_cast<float*>(base + lay.b1[s]),
                          a.bias1 ? a.bias1 + static_cast<size_t>(bn) * a.L : nullptr, a.L, c.jt * kTile, lane);
      const uint32_t full = smem_u32(&bars->st_full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, 4 * kTB);
        tma_load_4d(smem_u32(base + lay.q[s]), &a.tq, full, 0, c.h, c.it * kTile, bn);
        tma_load_4d(smem_u32(base + lay.d_o[s]), &a.tdo, full, 0, c.h, c.it * kTile, bn);
        tma_load_4d(smem_u32(base + lay.k[s]), &a.tk, full, 0, c.h, c.jt * kTile, bn);
        tma_load_4d(smem_u32(base + lay.v[s]), &a.tv, full, 0, c.h, c.jt * kTile, bn);
      } else {
        mbar_arrive(full);
      }
    }
    drain_wait(smem_u32(&bars->b2_full), 0, a.wait_ns, a.status);
    for (int s = 0; s < 2; ++s) {
      const int issued = (k + 1 - s) / 2;
      if (issued > 0) drain_wait(smem_u32(&bars->st_full[s]), (issued - 1) & 1, a.wait_ns, a.status);
    }
  } else if (warp == 5) {  // ---------------- MMA
    if (lane == 0) {
      constexpr uint32_t RB = DP * 2;
      constexpr uint32_t SWZ = swizzle_for_row(RB);
      constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
      for (int k = 0; k < nn; ++k) {
        const int s = k & 1, ph = (k >> 1) & 1;
        if (!mbar_wait(smem_u32(&bars->st_full[s]), ph, g)) break;
        if (!mbar_wait(smem_u32(&bars->mm_free[s]), ph ^ 1, g)) break;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(base + lay.q[s]), do_addr = smem_u32(base + lay.d_o[s]);
        const uint32_t k_addr = smem_u32(base + lay.k[s]), v_addr = smem_u32(base + lay.v[s]);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk)
          umma_ss(tmem + (s ? kColS_1 : kColS_0), smem_desc(q_addr + kk * 32, 16, 8 * RB, SWZ),
                  smem_desc(k_addr + kk * 32, 16, 8 * RB, SWZ), id_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk)
          umma_ss(tmem + (s ? kColDP_1 : kColDP_0), smem_desc(do_addr + kk * 32, 16, 8 * RB, SWZ),
                  smem_desc(v_addr + kk * 32, 16, 8 * RB, SWZ), id_s, kk > 0);
        umma_commit(smem_u32(&bars->mm_full[s]));
        umma_commit(smem_u32(&bars->st_free[s]));
      }
      umma_commit(smem_u32(&bars->drain));
      drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
    }
    __syncwarp();
  } else {  // ---------------- compute: thread r = query row of the tile
    const int r = threadIdx.x;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int i = c.it * kTile + r;
    float acc[kTile];
#pragma unroll
    for (int e = 0; e < kTile; ++e) acc[e] = 0.0f;
    bool ok = mbar_wait(smem_u32(&bars->b2_full), 0, g);
    for (int k = 0; ok && k < nn; ++k) {
      const int s = k & 1, ph = (k >> 1) & 1;
      const size_t bnh = (static_cast<size_t>(c.b) * a.N + c.n0 + k) * a.H + c.h;
      float lse2 = INFINITY, dlt = 0.0f;
      if (i < a.L) {
        const float lv = a.lse[bnh * a.L + i];
        lse2 = (lv == -INFINITY) ? INFINITY : lv * kLog2e;
        dlt = a.delta[bnh * a.L + i];
      }
      if (!mbar_wait(smem_u32(&bars->st_full[s]), ph, g)) { ok = false; break; }
      if (!mbar_wait(smem_u32(&bars->mm_full[s]), ph, g)) { ok = false; break; }
      tc_fence_after();
      const float* b1s = reinterpret_cast<const float*>(base + lay.b1[s]);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], pv[32];
        tmem_ld32(trow + (s ? kColS_1 : kColS_0) + cc * 32, sv);
        tmem_ld32(trow + (s ? kColDP_1 : kColDP_0) + cc * 32, pv);
        tmem_wait_ld(sv);
        tmem_wait_ld(pv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk16 = cc * 4 + q;
          const uint4 pb = *reinterpret_cast<const uint4*>(base + lay.b2 + (chunk16 >> 3) * 16384 +
                                                           swz_offset(r, chunk16 & 7, 128));
          const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
          const float4 m0 = *reinterpret_cast<const float4*>(b1s + chunk16 * 8);
          const float4 m1 = *reinterpret_cast<const float4*>(b1s + chunk16 * 8 + 4);
          const float mk[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int x = q * 8 + e;
            float y = fmaf(__uint_as_float(sv[x]), a.scale_log2, mk[e]);
            y = fmaf((e & 1) ? unpack_hi<BF16>(pw[e >> 1]) : unpack_lo<BF16>(pw[e >> 1]), kLog2e, y);
            const float pr = ex2(y - lse2);
            acc[cc * 32 + x] += pr * (__uint_as_float(pv[x]) - dlt);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->mm_free[s]));
        mbar_arrive(smem_u32(&bars->st_free[s]));
      }
    }
    if (ok && i < a.L) {
      const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
      float* dst = a.db2_part + c.grp * plane + (static_cast<long long>(bh) * a.L + i) * a.L;
      const int j0 = c.jt * kTile;
#pragma unroll
      for (int e = 0; e < kTile; ++e)
        if (j0 + e < a.L) dst[j0 + e] = acc[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ launch
size_t one_cta_per_sm(size_t bytes) { return bytes > 116u * 1024u ? bytes : 116u * 1024u; }

unsigned grid_for(long long work, long long per_block) {
  long long g = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <int DP, bool BF16, bool HAS_B2>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t st, const ProfileEvents* prof) {
  const long long rows = static_cast<long long>(a.B) * a.N * a.L * a.H;
  prof_record(prof, 2, st);
  evo_bwd_pre<DP, BF16><<<grid_for(rows, 256), 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_record(prof, 3, st);

  {
    const MainLayout<DP> lay(HAS_B2);
    const size_t smem = one_cta_per_sm(lay.total + 1024);
    auto kern = evo_bwd_main<DP, BF16, HAS_B2>;
    static bool limit_set[64] = {};
    if ((e = ensure_smem_limit(kern, smem, limit_set)) != cudaSuccess) return e;
    const long long items = static_cast<long long>(a.B) * a.N * a.H * a.QT;
    const long long grid = items < num_sms() ? items : num_sms();
    kern<<<static_cast<unsigned>(grid), 192, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  prof_record(prof, 4, st);
  evo_bwd_dq_cast<BF16><<<grid_for(rows * a.D / 8, 256), 256, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prof_record(prof, 5, st);

  if (HAS_B2) {
    const PartLayout<DP> lay;
    const size_t smem = one_cta_per_sm(lay.total + 1024);
    auto kern = evo_bwd_db2_part<DP, BF16>;
    static bool limit_set[64] = {};
    if ((e = ensure_smem_limit(kern, smem, limit_set)) != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(a.B) * a.H * a.groups * a.QT * a.QT;
    kern<<<static_cast<unsigned>(blocks), 192, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_record(prof, 6, st);
    const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
    evo_bwd_db2_sum<BF16><<<grid_for(plane, 256), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_record(prof, 7, st);
  }
  return cudaSuccess;
}

template <int DP, bool BF16>
cudaError_t launch_bwd_d(const BwdArgs& a, cudaStream_t st, const ProfileEvents* p) {
  return a.bias2_mode == kBias2None ? launch_bwd_t<DP, BF16, false>(a, st, p) : launch_bwd_t<DP, BF16, true>(a, st, p);
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int DP, bool bf16, cudaStream_t st, const ProfileEvents* p) {
  switch (DP) {
    case 16: return bf16 ? launch_bwd_d<16, true>(a, st, p) : launch_bwd_d<16, false>(a, st, p);
    case 32: return bf16 ? launch_bwd_d<32, true>(a, st, p) : launch_bwd_d<32, false>(a, st, p);
    case 64: return bf16 ? launch_bwd_d<64, true>(a, st, p) : launch_bwd_d<64, false>(a, st, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace evo
