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
//   evo_bwd_pre       delta [B,N,H,L] fp32 (and the transposed pair bias for the
//                     key-major kernel).
//   evo_bwd_main      (shapes whose dQ tiles do not fit in TMEM) persistent over
//                     a contiguous range of whole (b, h, n) slices, streamed as
//                     one sequence of (key tile, query tile) steps.  The MMA
//                     thread computes S = Q Kᵀ and dP = dO Vᵀ into TMEM
//                     (lane = query) one step ahead; eight compute warps (each
//                     32 query rows × 64 keys) form P and dS (fp16 / bf16) in
//                     swizzled shared memory; the MMA thread then forms
//                     dQ_tile = dS K and accumulates dV += Pᵀ dO and dK += dSᵀ Q
//                     in TMEM; the compute warps sum the dQ tiles of a slice in
//                     the CTA's fp32 rows and write dQ at its last key tile.
//   evo_bwd_db2_part  (pair bias only) per (b, h, query tile, key tile,
//                     n-group): recompute S and dP (double-buffered in TMEM),
//                     form P and dS, and sum dS over the group's n in a fixed
//                     order in registers (eight warps, 32 rows × 64 keys each);
//                     write fp32.
//   evo_bwd_db2_sum   dbias2 = Σ_groups partial in fixed order, cast.
// Every sum runs in a fixed order, so all gradients are bitwise reproducible.
#include "evo_bwd_common.cuh"

namespace evo {
namespace {


// x / d in 32-bit arithmetic when x < 2^31 (64-bit division is far slower).
__device__ __forceinline__ long long idiv(long long x, long long d, bool small) {
  return small ? static_cast<long long>(static_cast<uint32_t>(x) / static_cast<uint32_t>(d)) : x / d;
}

// ============================================================ evo_bwd_pre
template <int DP, bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_pre(const BwdArgs a) {
  // the call's own status word starts clear; the later kernels of the call run after this one
  if (a.clear_status && blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
  if (a.b2t) {  // transposed pair bias for the key-major kernel, in 32 x 32 tiles through smem
    __shared__ uint16_t tile[32][34];
    const int TL = (a.L + 31) / 32, lane = threadIdx.x & 31, row0 = threadIdx.x >> 5;
    const long long tiles = static_cast<long long>(a.B) * a.H * TL * TL;
    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int tj = static_cast<int>(t % TL), ti = static_cast<int>((t / TL) % TL);
      const long long bh = t / (static_cast<long long>(TL) * TL);
      const uint16_t* src = a.bias2 + bh * a.L * a.L;
      for (int rr = row0; rr < 32; rr += 8) {
        const int i = ti * 32 + rr, j = tj * 32 + lane;
        tile[rr][lane] = (i < a.L && j < a.L) ? src[static_cast<size_t>(i) * a.L + j] : static_cast<uint16_t>(0);
      }
      __syncthreads();
      uint16_t* dst = a.b2t + bh * a.L * a.b2t_pitch;
      for (int rr = row0; rr < 32; rr += 8) {
        const int j = tj * 32 + rr, i = ti * 32 + lane;
        if (j < a.L && i < a.L) dst[static_cast<size_t>(j) * a.b2t_pitch + i] = tile[lane][rr];
      }
      __syncthreads();
    }
  }
  const long long rows = static_cast<long long>(a.B) * a.N * a.L * a.H;
  if (a.D == 8 || a.D == 16 || a.D == 32 || a.D == 64) {
    // Coalesced: each lane takes one 16-byte chunk (8 elements) of O and dO; the D/8
    // lanes of a row (adjacent) reduce their partial dot products with shuffles.
    const int lpr = a.D / 8;                                   // lanes per row
    const long long chunks = rows * lpr;
    const int lane = threadIdx.x & 31;
    const long long stride = gridDim.x * 256ll;
    constexpr int U = 4;  // chunks per thread per round (all loads issued first)
    for (long long c0 = blockIdx.x * 256ll + threadIdx.x; c0 - lane < chunks; c0 += U * stride) {
      uint4 ov[U], gv[U];
      if (a.packed) {
#pragma unroll
        for (int q = 0; q < U; ++q) {
          const long long ch = c0 + q * stride;
          ov[q] = ch < chunks ? __ldg(reinterpret_cast<const uint4*>(a.out) + ch) : make_uint4(0u, 0u, 0u, 0u);
          gv[q] = ch < chunks ? __ldg(reinterpret_cast<const uint4*>(a.dout) + ch) : make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
        // strided rows: chunk ch is chunk c of token (bn, i), cpt = H*D/8 chunks per token
        const long long cpt = static_cast<long long>(a.H) * lpr;
        const bool small = chunks < (1ll << 31);
#pragma unroll
        for (int q = 0; q < U; ++q) {
          const long long ch = c0 + q * stride;
          ov[q] = gv[q] = make_uint4(0u, 0u, 0u, 0u);
          if (ch < chunks) {
            const long long t = idiv(ch, cpt, small), bn = idiv(t, a.L, small);
            const long long c = ch - t * cpt, i = t - bn * a.L;
            ov[q] = __ldg(reinterpret_cast<const uint4*>(a.out + bn * a.r_out.bn + i * a.r_out.l) + c);
            gv[q] = __ldg(reinterpret_cast<const uint4*>(a.dout + bn * a.r_dout.bn + i * a.r_dout.l) + c);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < U; ++q) {
        const long long ch = c0 + q * stride;
        if (ch - lane >= chunks) break;  // uniform across the warp
        const uint32_t ow[4] = {ov[q].x, ov[q].y, ov[q].z, ov[q].w}, gw[4] = {gv[q].x, gv[q].y, gv[q].z, gv[q].w};
        float sum = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sum = fmaf(unpack_lo<BF16>(ow[e]), unpack_lo<BF16>(gw[e]), sum);
          sum = fmaf(unpack_hi<BF16>(ow[e]), unpack_hi<BF16>(gw[e]), sum);
        }
        for (int off = 1; off < lpr; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (ch < chunks && (lane & (lpr - 1)) == 0) {
          // row (b, n, i, h) in memory order of [B,N,L,H,D] -> delta [B,N,H,L]; 32-bit
          // division when the row count allows it (64-bit division is far slower)
          const long long row = ch / lpr;
          long long dst;
          if (rows < (1ll << 31)) {
            const uint32_t r32 = static_cast<uint32_t>(row), H = a.H, L = a.L;
            const uint32_t t = r32 / H, h = r32 - t * H, bn = t / L, i = t - bn * L;
            dst = (static_cast<long long>(bn) * H + h) * L + i;
          } else {
            const int h = static_cast<int>(row % a.H);
            const long long t = row / a.H;
            dst = (t / a.L * a.H + h) * a.L + t % a.L;
          }
          a.delta[dst] = sum;
        }
      }
    }
  } else
  for (long long row = blockIdx.x * 256ll + threadIdx.x; row < rows; row += gridDim.x * 256ll) {
    // row enumerates (b, n, i, h) in memory order of [B,N,L,H,D]
    const int h = static_cast<int>(row % a.H);
    long long t = row / a.H;
    const int i = static_cast<int>(t % a.L);
    const long long bn = t / a.L;
    const uint4* o = reinterpret_cast<const uint4*>(a.out + bn * a.r_out.bn + i * a.r_out.l + h * a.D);
    const uint4* g = reinterpret_cast<const uint4*>(a.dout + bn * a.r_dout.bn + i * a.r_dout.l + h * a.D);
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
      }
    }
    a.delta[(bn * a.H + h) * a.L + i] = sum;
  }

}

// ============================================================ masked key tiles
// Masked key-tile skipping for the per-key-tile kernel.  evo_bwd_tile_mask: the key
// tiles of each (b, n) row to skip (one warp per row), and zeros for dK and dV of those
// tiles in every head, since the per-key-tile kernel will not run them.  The kernel reads
// the skip bits of each slice it walks.
template <bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_tile_mask(const BwdArgs a) {
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(a.B) * a.N;
  const unsigned long long all = a.QT >= 64 ? ~0ull : ((1ull << a.QT) - 1);
  const int cpr = a.H * a.D / 8;  // 16-byte chunks per token row
  for (long long bn = (blockIdx.x * 256ll + threadIdx.x) >> 5; bn < rows; bn += gridDim.x * 8ll) {
    const unsigned long long kept = kept_tiles<BF16>(a.bias1 + bn * a.L, a.L, a.skip_at, lane);
    const unsigned long long skip = kept ? (~kept & all) : 0ull;
    if (lane == 0) a.tskip[bn] = skip;
    for (unsigned long long rem = skip; rem; rem &= rem - 1) {
      const int j0 = (__ffsll(static_cast<long long>(rem)) - 1) * kTile;
      const int nj = a.L - j0 < kTile ? a.L - j0 : kTile;
      for (int e = lane; e < nj * cpr; e += 32) {
        const int j = j0 + e / cpr, c = e % cpr;
        *reinterpret_cast<uint4*>(a.dk + bn * a.r_dk.bn + static_cast<long long>(j) * a.r_dk.l + c * 8) =
            make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(a.dv + bn * a.r_dv.bn + static_cast<long long>(j) * a.r_dv.l + c * 8) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

// ============================================================ evo_bwd_db2_sum
template <bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_db2_sum(const BwdArgs a) {
  const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
  if ((plane & 3) == 0) {  // four consecutive elements per thread, same fixed group order
    const float4* part = reinterpret_cast<const float4*>(a.db2_part);
    const long long p4 = plane / 4;
    for (long long e = blockIdx.x * 256ll + threadIdx.x; e < p4; e += gridDim.x * 256ll) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      int g = 0;
      for (; g + 16 <= a.groups; g += 16) {
        float4 v[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) v[t] = __ldg(part + (g + t) * p4 + e);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          s.x += v[t].x;
          s.y += v[t].y;
          s.z += v[t].z;
          s.w += v[t].w;
        }
      }
      for (; g + 4 <= a.groups; g += 4) {
        float4 v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = __ldg(part + (g + t) * p4 + e);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          s.x += v[t].x;
          s.y += v[t].y;
          s.z += v[t].z;
          s.w += v[t].w;
        }
      }
      for (; g < a.groups; ++g) {
        const float4 v = __ldg(part + g * p4 + e);
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
      }
      uint2 pk;
      pk.x = pack2<BF16>(s.x, s.y);
      pk.y = pack2<BF16>(s.z, s.w);
      reinterpret_cast<uint2*>(a.dbias2)[e] = pk;
    }
    return;
  }
  for (long long e = blockIdx.x * 256ll + threadIdx.x; e < plane; e += gridDim.x * 256ll) {
    float s = 0.0f;
    int g = 0;
    for (; g + 8 <= a.groups; g += 8) {  // eight loads in flight, added in group order
      float v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) v[t] = __ldg(a.db2_part + (g + t) * plane + e);
#pragma unroll
      for (int t = 0; t < 8; ++t) s += v[t];
    }
    for (; g < a.groups; ++g) s += __ldg(a.db2_part + g * plane + e);
    const uint32_t p = pack2<BF16>(s, 0.0f);
    a.dbias2[e] = static_cast<uint16_t>(p & 0xFFFFu);
  }
}


// ============================================================ evo_bwd_main
// Per-key-tile schedule, for the shapes whose dQ tiles do not all fit in TMEM.  A CTA
// owns a contiguous range of whole (b, h, n) slices.  For each slice it walks the key
// tiles jt in order (with masked-tile skipping, the kept ones) and for each key tile the
// L/128 query tiles it, one step per (jt, it):
//   S = Q Kᵀ, dP = dO Vᵀ into TMEM (lane = query), one step ahead of the compute warps;
//   P and dS in the dtype into swizzled shared-memory tiles (two buffers where they fit,
//   so the compute warps form step u+1 while the gradient MMAs of step u run);
//   dQ_tile = dS K (issued first, so its consumer starts early), dV += Pᵀ dO and
//   dK += dSᵀ Q (the same tiles as MN-major A operands; dK, dV double-buffered across
//   key tiles where TMEM allows).
// dQ of a slice accumulates in the CTA's own fp32 blocks of the workspace (one block of
// 32 rows × DP/2 columns per compute warp and query tile): each compute warp stages its
// dQ_tile block in shared memory and hands it to the bulk-copy engine, which stores it
// (first key tile of the slice) or adds it in L2 (later key tiles); the last key tile
// reads the sum back, adds its own tile, scales and writes dQ in the dtype.  Successive
// additions to one block are a query-tile sweep apart, and each is issued only once every
// bulk operation of the warp but the newest is complete, so they run one after another
// in key-tile order: dQ is bitwise reproducible.  The blocks of one CTA (L × DP floats)
// stay in L2.
__device__ __forceinline__ uint32_t col_s() { return 0u; }
__device__ __forceinline__ uint32_t col_dp() { return 128u; }
template <int DP>
__host__ __device__ constexpr int kv_acc_buffers() { return DP <= 32 ? 2 : 1; }
template <int DP>
__device__ __forceinline__ uint32_t col_dk(uint32_t b) { return 256u + b * 2 * DP; }
template <int DP>
__device__ __forceinline__ uint32_t col_dv(uint32_t b) { return 256u + b * 2 * DP + DP; }
template <int DP>
__device__ __forceinline__ uint32_t col_dq(uint32_t b) { return 256u + kv_acc_buffers<DP>() * 2 * DP + b * DP; }

constexpr int kMaxQStages = 4;

struct MainBars {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t q_full[kMaxQStages], q_empty[kMaxQStages];
  uint64_t st_full, st_free;
  uint64_t ds_full[2], ds_empty[2];
  uint64_t dq_full[2], dq_free[2];
  uint64_t dkdv_full[2], dkdv_free[2];
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

// Shared memory: the P and dS tiles (pds buffers each, 128B-swizzled, so first), K/V
// (two buffers), the Q/dO ring (qs stages), streamed pair-bias tiles (one per Q/dO
// stage), key-mask chunks, lse/delta per stage, barriers.
template <int DP>
struct MainLayout {
  static constexpr uint32_t kTB = kTile * DP * 2;
  static constexpr uint32_t kDqStg = DqScr<DP>::kStg;
  Ring p, ds, k, v, q, d_o, b2s, b1, ld, dqs;
  uint32_t bars, total;
  int kvb;  // K/V buffers
  __host__ __device__ MainLayout(bool has_b2, int qs, int pds, int kv_bufs) : kvb(kv_bufs) {
    uint32_t off = 0;
    p = Ring{off, 32768u};
    off += pds * 32768u;
    ds = Ring{off, 32768u};
    off += pds * 32768u;
    k = Ring{off, 2 * kTB};
    v = Ring{off + kTB, 2 * kTB};
    off += kvb * 2 * kTB;
    q = Ring{off, 2 * kTB};
    d_o = Ring{off + kTB, 2 * kTB};
    off += qs * 2 * kTB;
    b2s = Ring{off, 32768u};
    if (has_b2) off += qs * 32768u;
    b1 = Ring{off, 512u};
    off += 1024u;
    ld = Ring{off, 1024u};
    off += qs * 1024u;
    dqs = Ring{off, kDqStg};  // per compute warp: its dQ block on the way to the workspace
    off += kComputeWarps * kDqStg;
    bars = off;
    off += (sizeof(MainBars) + 127) & ~127u;
    total = off;
  }
};

// K/V buffer of item number c (items alternate between two buffers, or share one) and
// the parity of that buffer's c-th use.
__device__ __forceinline__ uint32_t kv_buf(uint32_t c, int kvb) { return kvb == 2 ? (c & 1) : 0u; }
__device__ __forceinline__ uint32_t kv_par(uint32_t c, int kvb) { return kvb == 2 ? ((c >> 1) & 1) : (c & 1); }

// The walk of one CTA over its steps: slices s0 <= s < s1 (order b, h, n), the kept key
// tiles of each (all, or those not in the row's skip bits), the QT query tiles of each.
struct MainWalk {
  int b, h, n, jt;
  long long s;
  uint64_t skip;  // key tiles of the current slice to skip
  __device__ __forceinline__ bool kept(int t) const { return t >= 64 || !((skip >> t) & 1ull); }
  __device__ __forceinline__ int next_kept(int t, int QT) const {
    do ++t;
    while (t < QT && !kept(t));
    return t;
  }
  __device__ __forceinline__ void enter(const BwdArgs& a) {
    skip = 0;
    if (a.tile_skip && s < a.items) {
      const uint64_t all = a.QT >= 64 ? ~0ull : ((1ull << a.QT) - 1ull);
      skip = a.tskip[static_cast<long long>(b) * a.N + n] & all;
      if (skip == all) skip = 0;  // a row with no kept key skips nothing
    }
    jt = next_kept(-1, a.QT);
  }
  __device__ __forceinline__ void init(long long s0, const BwdArgs& a) {
    s = s0;
    n = static_cast<int>(s0 % a.N);
    const long long t = s0 / a.N;
    h = static_cast<int>(t % a.H);
    b = static_cast<int>(t / a.H);
    enter(a);
  }
  // to the next kept key tile of the slice, or the first of the next slice
  __device__ __forceinline__ void next_item(const BwdArgs& a) {
    jt = next_kept(jt, a.QT);
    if (jt < a.QT) return;
    ++s;
    if (++n == a.N) {
      n = 0;
      if (++h == a.H) {
        h = 0;
        ++b;
      }
    }
    enter(a);
  }
  __device__ __forceinline__ bool first_tile(const BwdArgs& a) const { return next_kept(-1, a.QT) == jt; }
  __device__ __forceinline__ bool last_tile(const BwdArgs& a) const { return next_kept(jt, a.QT) >= a.QT; }
};

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void main_producer(const BwdArgs& a, uint8_t* base, const MainLayout<DP>& lay,
                                              MainBars* bars, const WaitGuard& g, int lane, long long s0,
                                              long long s1) {
  constexpr uint32_t kTB = MainLayout<DP>::kTB;
  const int QS = a.q_stages, QT = a.QT;
  const bool tma_b2 = a.bias2_mode == kBias2Tma;
  const uint32_t q_bytes = 2 * kTB + ((HAS_B2 && tma_b2) ? 32768u : 0u);
  uint32_t it_ctr = 0, item_ctr = 0, s = 0, ph = 0;
  MainWalk w;
  w.init(s0, a);
  bool ok = true;
  for (; ok && w.s < s1; ++item_ctr, w.next_item(a)) {
    const int bn = w.b * a.N + w.n, bh = w.b * a.H + w.h;
    const size_t bnh = static_cast<size_t>(bn) * a.H + w.h;
    const uint32_t kb = kv_buf(item_ctr, lay.kvb);
    if (!mbar_wait_warp(smem_u32(&bars->kv_empty[kb]), kv_par(item_ctr, lay.kvb) ^ 1, g)) { ok = false; break; }
    {
      const uint32_t full = smem_u32(&bars->kv_full[kb]);
      if (lane == 0) {
        mbar_expect_tx(full, 2 * kTB);
        tma_load_4d(smem_u32(base + lay.k[kb]), &a.tk, full, 0, w.h, w.jt * kTile, bn);
        tma_load_4d(smem_u32(base + lay.v[kb]), &a.tv, full, 0, w.h, w.jt * kTile, bn);
      }
      fill_b1_chunk<BF16>(reinterpret_cast<float*>(base + lay.b1[kb]),
                          a.bias1 ? a.bias1 + static_cast<size_t>(bn) * a.L : nullptr, a.L, w.jt * kTile, lane);
      mbar_arrive(full);
    }
    for (int it = 0; it < QT; ++it, ++it_ctr) {
      if (!mbar_wait_warp(smem_u32(&bars->q_empty[s]), ph ^ 1, g)) { ok = false; break; }
      const uint32_t full = smem_u32(&bars->q_full[s]);
      if (lane == 0) {
        mbar_expect_tx(full, q_bytes);
        tma_load_4d(smem_u32(base + lay.q[s]), &a.tq, full, 0, w.h, it * kTile, bn);
        tma_load_4d(smem_u32(base + lay.d_o[s]), &a.tdo, full, 0, w.h, it * kTile, bn);
        if (HAS_B2 && tma_b2) {
          tma_load_3d(smem_u32(base + lay.b2s[s]), &a.tb2, full, w.jt * kTile, it * kTile, bh);
          tma_load_3d(smem_u32(base + lay.b2s[s] + 16384), &a.tb2, full, w.jt * kTile + 64, it * kTile, bh);
        }
      }
      if (HAS_B2 && !tma_b2)
        fill_b2_tile_loads(base + lay.b2s[s], a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L, it * kTile,
                           w.jt * kTile, lane);
      fill_lse_delta(reinterpret_cast<float*>(base + lay.ld[s]), a.lse, a.delta, bnh, a.L, it * kTile, lane);
      mbar_arrive(full);
      if (++s == static_cast<uint32_t>(QS)) {
        s = 0;
        ph ^= 1;
      }
    }
  }
  // Drain: every copy this warp started has landed before the CTA may exit.
  for (uint32_t b = 0; b < static_cast<uint32_t>(lay.kvb); ++b) {
    const uint32_t issued = lay.kvb == 2 ? (item_ctr + 1 - b) / 2 : item_ctr;
    if (issued > 0) drain_wait(smem_u32(&bars->kv_full[b]), (issued - 1) & 1, a.wait_ns, a.status);
  }
  for (uint32_t st = 0; st < static_cast<uint32_t>(QS); ++st) {
    const uint32_t issued = (it_ctr + QS - 1 - st) / QS;
    if (issued > 0) drain_wait(smem_u32(&bars->q_full[st]), (issued - 1) & 1, a.wait_ns, a.status);
  }
}

// Step bookkeeping of the MMA thread: step u = (item index, query tile).
struct Step {
  uint32_t u, item_ctr;
  int it;
  uint32_t qs, qph;  // Q/dO ring stage and phase of this step
};

template <int DP, bool BF16>
__device__ __forceinline__ bool main_issue_sdp(const Step& st, uint8_t* base, const MainLayout<DP>& lay,
                                               MainBars* bars, uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);  // K-major A and B
  const uint32_t kb = kv_buf(st.item_ctr, lay.kvb);
  if (st.it == 0 && !mbar_wait(smem_u32(&bars->kv_full[kb]), kv_par(st.item_ctr, lay.kvb), g)) return false;
  if (!mbar_wait(smem_u32(&bars->q_full[st.qs]), st.qph, g)) return false;
  if (!mbar_wait(smem_u32(&bars->st_free), (st.u & 1) ^ 1, g)) return false;
  tc_fence_after();
  const uint32_t q_addr = smem_u32(base + lay.q[st.qs]), do_addr = smem_u32(base + lay.d_o[st.qs]);
  const uint32_t k_addr = smem_u32(base + lay.k[kb]), v_addr = smem_u32(base + lay.v[kb]);
#pragma unroll
  for (int k = 0; k < DP / 16; ++k)
    umma_ss(tmem + col_s(), smem_desc(q_addr + k * 32, 16, 8 * RB, SWZ), smem_desc(k_addr + k * 32, 16, 8 * RB, SWZ),
            id_s, k > 0);
#pragma unroll
  for (int k = 0; k < DP / 16; ++k)
    umma_ss(tmem + col_dp(), smem_desc(do_addr + k * 32, 16, 8 * RB, SWZ),
            smem_desc(v_addr + k * 32, 16, 8 * RB, SWZ), id_s, k > 0);
  umma_commit(smem_u32(&bars->st_full));
  return true;
}

template <int DP, bool BF16>
__device__ __forceinline__ bool main_issue_grads(const Step& st, int QT, int pds, uint8_t* base,
                                                 const MainLayout<DP>& lay, MainBars* bars, uint32_t tmem,
                                                 const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_kv = idesc_f16(128, DP, BF16, true, true);  // dV, dK: MN-major A and B
  constexpr uint32_t id_q = idesc_f16(128, DP, BF16, false, true);  // dQ: K-major A, MN-major B
  constexpr int NB = kv_acc_buffers<DP>();
  const uint32_t kb = kv_buf(st.item_ctr, lay.kvb);
  const uint32_t db = st.item_ctr % NB, dph = (st.item_ctr / NB) & 1;
  const uint32_t qb = st.u & 1;
  const uint32_t pb = st.u % pds, pph = (st.u / pds) & 1;
  if (!mbar_wait(smem_u32(&bars->ds_full[pb]), pph, g)) return false;
  if (!mbar_wait(smem_u32(&bars->dq_free[qb]), ((st.u >> 1) & 1) ^ 1, g)) return false;
  tc_fence_after();
  const uint32_t p_addr = smem_u32(base + lay.p[pb]), ds_addr = smem_u32(base + lay.ds[pb]);
  const uint32_t q_addr = smem_u32(base + lay.q[st.qs]), do_addr = smem_u32(base + lay.d_o[st.qs]);
  const uint32_t k_addr = smem_u32(base + lay.k[kb]);
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // dQ_tile = dS K   (K = 128 keys)
    const uint64_t ad = smem_desc(ds_addr + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(k_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ss(tmem + col_dq<DP>(qb), ad, bd, id_q, k > 0);
  }
  umma_commit(smem_u32(&bars->dq_full[qb]));
  if (st.it == 0 && !mbar_wait(smem_u32(&bars->dkdv_free[db]), dph ^ 1, g)) return false;
  tc_fence_after();
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // dV += Pᵀ dO   (K = 128 queries)
    const uint64_t ad = smem_desc(p_addr + k * 16 * 128, 16384, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(do_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ss(tmem + col_dv<DP>(db), ad, bd, id_kv, (st.it > 0 || k > 0) ? 1u : 0u);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // dK += dSᵀ Q
    const uint64_t ad = smem_desc(ds_addr + k * 16 * 128, 16384, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(q_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ss(tmem + col_dk<DP>(db), ad, bd, id_kv, (st.it > 0 || k > 0) ? 1u : 0u);
  }
  umma_commit(smem_u32(&bars->ds_empty[pb]));
  umma_commit(smem_u32(&bars->q_empty[st.qs]));
  if (st.it == QT - 1) {
    umma_commit(smem_u32(&bars->dkdv_full[db]));
    umma_commit(smem_u32(&bars->kv_empty[kb]));
  }
  return true;
}

template <int DP, bool BF16>
__device__ __forceinline__ void main_mma(const BwdArgs& a, uint8_t* base, const MainLayout<DP>& lay, MainBars* bars,
                                         uint32_t tmem, const WaitGuard& g, long long s0, long long s1) {
  const int QS = a.q_stages, QT = a.QT, pds = a.pds_bufs;
  auto step_of = [&](Step& st) {  // advance to the next step
    ++st.u;
    if (++st.it == QT) {
      st.it = 0;
      ++st.item_ctr;
    }
    if (++st.qs == static_cast<uint32_t>(QS)) {
      st.qs = 0;
      st.qph ^= 1;
    }
  };
  // the walk only decides how many items (kept key tiles) each slice has
  MainWalk w;
  w.init(s0, a);
  Step cur{0, 0, 0, 0, 0};
  bool ok = w.s < s1;
  auto advance_walk = [&](MainWalk& x, const Step& st) {  // the walk after step st
    if (st.it == QT - 1) x.next_item(a);
  };
  if (QS >= 2) {
    // S/dP of step u+1 go ahead of step u's gradient MMAs, so the compute warps
    // can start on u+1 while the tensor core finishes u.  (Needs a second
    // Q/dO stage: step u's stage is released by its gradient MMAs.)
    // With one K/V buffer, a step that starts a new key tile needs the buffer the
    // previous step's gradient MMAs release: those go first there.
    if (ok) ok = main_issue_sdp<DP, BF16>(cur, base, lay, bars, tmem, g);
    while (ok) {
      Step nxt = cur;
      MainWalk wn = w;
      advance_walk(wn, cur);
      step_of(nxt);
      const bool more = wn.s < s1;
      const bool grads_first = lay.kvb == 1 && nxt.it == 0;
      if (more && !grads_first && !main_issue_sdp<DP, BF16>(nxt, base, lay, bars, tmem, g)) { ok = false; break; }
      if (!main_issue_grads<DP, BF16>(cur, QT, pds, base, lay, bars, tmem, g)) { ok = false; break; }
      if (more && grads_first && !main_issue_sdp<DP, BF16>(nxt, base, lay, bars, tmem, g)) { ok = false; break; }
      if (!more) break;
      cur = nxt;
      w = wn;
    }
  } else {
    while (ok) {
      if (!main_issue_sdp<DP, BF16>(cur, base, lay, bars, tmem, g)) { ok = false; break; }
      if (!main_issue_grads<DP, BF16>(cur, QT, pds, base, lay, bars, tmem, g)) { ok = false; break; }
      advance_walk(w, cur);
      step_of(cur);
      if (w.s >= s1) break;
    }
  }
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

// dQ tile of step u (double-buffered in TMEM by step parity): this warp's DP/2 columns
// into the CTA's fp32 dQ blocks (consume_dq_tile).
template <int DP, bool BF16>
__device__ __forceinline__ bool main_consume_dq(const BwdArgs& a, const DqStep& d, uint32_t u, MainBars* bars,
                                                uint32_t trow, int r, int w, int hc, int lane, uint8_t* stg,
                                                const WaitGuard& g) {
  const uint32_t qb = u & 1;
  return consume_dq_tile<DP, BF16>(a, d, smem_u32(&bars->dq_full[qb]), smem_u32(&bars->dq_free[qb]), (u >> 1) & 1,
                                   trow + col_dq<DP>(qb) + hc * (DP / 2), r, w, hc, lane, stg, g);
}

// What the compute warps remember of an item until they write its dK and dV.
struct KvItem {
  int b, n, h, jt;
};

// dK, dV of a finished item (TMEM lanes = keys of its key tile): this warp's DP/2 columns.
template <int DP, bool BF16>
__device__ __forceinline__ bool main_write_dkdv(const BwdArgs& a, const KvItem& c, uint32_t item_ctr,
                                                MainBars* bars, uint32_t trow, int r, int hc, int lane,
                                                const WaitGuard& g) {
  constexpr int HD = DP / 2;
  constexpr int NB = kv_acc_buffers<DP>();
  const uint32_t db = item_ctr % NB;
  if (!mbar_wait_warp(smem_u32(&bars->dkdv_full[db]), (item_ctr / NB) & 1, g)) return false;
  tc_fence_after();
  float kx[HD], vx[HD];
  const uint32_t ck = trow + col_dk<DP>(db) + hc * HD, cv = trow + col_dv<DP>(db) + hc * HD;
  if constexpr (HD == 8) {
    uint32_t x[8], y[8];
    tmem_ld8(ck, x);
    tmem_ld8(cv, y);
    tmem_wait_ld(x);
    tmem_wait_ld(y);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      kx[e] = __uint_as_float(x[e]);
      vx[e] = __uint_as_float(y[e]);
    }
  } else {
    uint32_t x[HD / 16][16], y[HD / 16][16];
#pragma unroll
    for (int q = 0; q < HD / 16; ++q) {
      tmem_ld16(ck + q * 16, x[q]);
      tmem_ld16(cv + q * 16, y[q]);
    }
#pragma unroll
    for (int q = 0; q < HD / 16; ++q) {
      tmem_wait_ld(x[q]);
      tmem_wait_ld(y[q]);
    }
#pragma unroll
    for (int q = 0; q < HD / 16; ++q)
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        kx[q * 16 + e] = __uint_as_float(x[q][e]);
        vx[q * 16 + e] = __uint_as_float(y[q][e]);
      }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->dkdv_free[db]));
  const int j = c.jt * kTile + r;
  if (j < a.L) {
    const long long bn = static_cast<long long>(c.b) * a.N + c.n, inner = c.h * a.D + hc * HD;
    uint16_t* dk = a.dk + bn * a.r_dk.bn + j * a.r_dk.l + inner;
    uint16_t* dv = a.dv + bn * a.r_dv.bn + j * a.r_dv.l + inner;
#pragma unroll
    for (int e = 0; e < HD; e += 8)
      if (hc * HD + e < a.D) {
        uint4 pk, pv4;
        pk.x = pack2<BF16>(kx[e + 0] * a.scale, kx[e + 1] * a.scale);
        pk.y = pack2<BF16>(kx[e + 2] * a.scale, kx[e + 3] * a.scale);
        pk.z = pack2<BF16>(kx[e + 4] * a.scale, kx[e + 5] * a.scale);
        pk.w = pack2<BF16>(kx[e + 6] * a.scale, kx[e + 7] * a.scale);
        pv4.x = pack2<BF16>(vx[e + 0], vx[e + 1]);
        pv4.y = pack2<BF16>(vx[e + 2], vx[e + 3]);
        pv4.z = pack2<BF16>(vx[e + 4], vx[e + 5]);
        pv4.w = pack2<BF16>(vx[e + 6], vx[e + 7]);
        *reinterpret_cast<uint4*>(dk + e) = pk;
        *reinterpret_cast<uint4*>(dv + e) = pv4;
      }
  }
  return true;
}

// P and dS for one 16-key chunk k (0..3) of this warp's 64 keys (S, dP already loaded
// from TMEM), written to the [query][key] P and dS tiles (K-major, 128B swizzle).
template <bool BF16, bool HAS_B2>
__device__ __forceinline__ void main_chunk16(const uint32_t (&sv)[16], const uint32_t (&pv)[16], const float* b1c,
                                             const uint8_t* b2half, uint8_t* pt, uint8_t* dt, int r, int k,
                                             float lse2, float dlt, float2 sl2) {
  const float2 nl2 = make_float2(-lse2, -lse2), l2e2 = make_float2(kLog2e, kLog2e), nd2 = make_float2(-dlt, -dlt);
#pragma unroll
  for (int q = 0; q < 2; ++q) {  // 8 keys (one 16-byte chunk of the tiles) per q
    const float4 m0 = *reinterpret_cast<const float4*>(b1c + k * 16 + q * 8);
    const float4 m1 = *reinterpret_cast<const float4*>(b1c + k * 16 + q * 8 + 4);
    const float2 mk[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                          make_float2(m1.z, m1.w)};
    const uint32_t off = swz_offset(r, k * 2 + q, 128);
    uint4 pb = make_uint4(0u, 0u, 0u, 0u);
    if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2half + off);
    const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
    uint32_t pp[4], dd[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int x = q * 8 + e2 * 2;
      float2 t = fma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, mk[e2]);
      if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
      t = add2(t, nl2);
      const float p0 = ex2(t.x), p1 = ex2(t.y);
      const float2 dpd = add2(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), nd2);
      const float2 ds = mul2(make_float2(p0, p1), dpd);
      pp[e2] = pack2<BF16>(p0, p1);
      dd[e2] = pack2<BF16>(ds.x, ds.y);
    }
    *reinterpret_cast<uint4*>(pt + off) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
    *reinterpret_cast<uint4*>(dt + off) = make_uint4(dd[0], dd[1], dd[2], dd[3]);
  }
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void main_compute(const BwdArgs& a, uint8_t* base, const MainLayout<DP>& lay,
                                             MainBars* bars, uint32_t tmem, const WaitGuard& g, long long s0,
                                             long long s1) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = w & 3, hc = w >> 2;
  const int r = quad * 32 + lane;  // query row (S, dP, dQ) or key row (dK, dV) within the tile == TMEM lane
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int QS = a.q_stages, QT = a.QT;
  const uint32_t pds = static_cast<uint32_t>(a.pds_bufs);
  uint8_t* dq_stg = base + lay.dqs[w];
  uint32_t u = 0, item_ctr = 0, s = 0, ph = 0;
  MainWalk cur;
  cur.init(s0, a);
  DqStep pd{0, 0, 0, 0, false, false};
  KvItem pk{0, 0, 0, 0};
  bool ok = true;
  for (; ok && cur.s < s1; ++item_ctr, cur.next_item(a)) {
    const uint32_t kb = kv_buf(item_ctr, lay.kvb);
    const bool first = cur.first_tile(a), last = cur.last_tile(a);
    if (!mbar_wait_warp(smem_u32(&bars->kv_full[kb]), kv_par(item_ctr, lay.kvb), g)) { ok = false; break; }
    const float* b1 = reinterpret_cast<const float*>(base + lay.b1[kb]) + hc * 64;
    for (int it = 0; it < QT; ++it, ++u) {
      if (!mbar_wait_warp(smem_u32(&bars->q_full[s]), ph, g)) { ok = false; break; }
      const float* ld = reinterpret_cast<const float*>(base + lay.ld[s]);
      const float lse2 = ld[r], dlt = ld[128 + r];
      const uint8_t* b2half = base + lay.b2s[s] + hc * 16384;
      if (!mbar_wait_warp(smem_u32(&bars->st_full), u & 1, g)) { ok = false; break; }
      // this step's P and dS buffer is free once the gradient MMAs that last read it are done
      const uint32_t pb = u % pds;
      if (!mbar_wait_warp(smem_u32(&bars->ds_empty[pb]), ((u / pds) & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      uint8_t* pt = base + lay.p[pb] + hc * 16384;
      uint8_t* dt = base + lay.ds[pb] + hc * 16384;
      {
        // 16-key chunks of S and dP: chunk k+1's TMEM loads are in flight while chunk k
        // is computed (one pair outstanding, so each wait covers the chunk about to be used)
        const uint32_t cs = trow + col_s() + hc * 64, cp = trow + col_dp() + hc * 64;
        uint32_t s0[16], p0[16], s1[16], p1[16];
        tmem_ld16(cs, s0);
        tmem_ld16(cp, p0);
        tmem_wait_ld(s0);
        tmem_wait_ld(p0);
        tmem_ld16(cs + 16, s1);
        tmem_ld16(cp + 16, p1);
        main_chunk16<BF16, HAS_B2>(s0, p0, b1, b2half, pt, dt, r, 0, lse2, dlt, sl2);
        tmem_wait_ld(s1);
        tmem_wait_ld(p1);
        tmem_ld16(cs + 32, s0);
        tmem_ld16(cp + 32, p0);
        main_chunk16<BF16, HAS_B2>(s1, p1, b1, b2half, pt, dt, r, 1, lse2, dlt, sl2);
        tmem_wait_ld(s0);
        tmem_wait_ld(p0);
        tmem_ld16(cs + 48, s1);
        tmem_ld16(cp + 48, p1);
        main_chunk16<BF16, HAS_B2>(s0, p0, b1, b2half, pt, dt, r, 2, lse2, dlt, sl2);
        tmem_wait_ld(s1);
        tmem_wait_ld(p1);
        // S and dP of this step are in registers: the next step's MMAs may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->st_free));
        main_chunk16<BF16, HAS_B2>(s1, p1, b1, b2half, pt, dt, r, 3, lse2, dlt, sl2);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->ds_full[pb]));
        mbar_arrive(smem_u32(&bars->q_empty[s]));
        if (it == QT - 1) mbar_arrive(smem_u32(&bars->kv_empty[kb]));
      }
      if (u > 0) {
        if (!main_consume_dq<DP, BF16>(a, pd, u - 1, bars, trow, r, w, hc, lane, dq_stg, g)) { ok = false; break; }
        if (it == 0 && !main_write_dkdv<DP, BF16>(a, pk, item_ctr - 1, bars, trow, r, hc, lane, g)) {
          ok = false;
          break;
        }
      }
      pd = DqStep{cur.b, cur.n, cur.h, it, first, last};
      if (++s == static_cast<uint32_t>(QS)) {
        s = 0;
        ph ^= 1;
      }
    }
    pk = KvItem{cur.b, cur.n, cur.h, cur.jt};
  }
  if (ok && u > 0) {
    if (main_consume_dq<DP, BF16>(a, pd, u - 1, bars, trow, r, w, hc, lane, dq_stg, g))
      main_write_dkdv<DP, BF16>(a, pk, item_ctr - 1, bars, trow, r, hc, lane, g);
  }
  if (lane == 0) bulk_wait_all();  // the dQ bulk operations are done with the staging block
}

template <int DP, bool BF16, bool HAS_B2>
__global__ void __launch_bounds__(kThreads, 1) evo_bwd_main(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const MainLayout<DP> lay(HAS_B2, a.q_stages, a.pds_bufs, a.kv_bufs);
  MainBars* bars = reinterpret_cast<MainBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the CTA's contiguous range of whole slices
  const long long s0 = static_cast<long long>(blockIdx.x) * a.chunk;
  const long long s1 = s0 + a.chunk < a.items ? s0 + a.chunk : a.items;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1 + kComputeWarps);
      mbar_init(smem_u32(&bars->ds_full[s]), kComputeWarps);
      mbar_init(smem_u32(&bars->ds_empty[s]), 1);
      mbar_init(smem_u32(&bars->dq_full[s]), 1);
      mbar_init(smem_u32(&bars->dq_free[s]), kComputeWarps);
      mbar_init(smem_u32(&bars->dkdv_full[s]), 1);
      mbar_init(smem_u32(&bars->dkdv_free[s]), kComputeWarps);
    }
    for (int s = 0; s < kMaxQStages; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 32);
      mbar_init(smem_u32(&bars->q_empty[s]), 1 + kComputeWarps);
    }
    mbar_init(smem_u32(&bars->st_full), 1);
    mbar_init(smem_u32(&bars->st_free), kComputeWarps);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    tma_prefetch_desc(&a.tdo);
    if (HAS_B2 && a.bias2_mode == kBias2Tma) tma_prefetch_desc(&a.tb2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const WaitGuard g{a.wait_ns, a.status, &bars->abort};
  if (s0 < s1) {
    if (warp == kProducerWarp) {
      main_producer<DP, BF16, HAS_B2>(a, base, lay, bars, g, lane, s0, s1);
    } else if (warp == kMmaWarp) {
      if (lane == 0) main_mma<DP, BF16>(a, base, lay, bars, tmem, g, s0, s1);
      __syncwarp();
    } else {
      main_compute<DP, BF16, HAS_B2>(a, base, lay, bars, tmem, g, s0, s1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ evo_bwd_slice
// One CTA owns whole (b, n, h) slices (when TMEM has room for every dQ tile of
// a slice): for each key tile jt, for each query tile it, S and dP into TMEM;
// P and dS into the swizzled smem tiles (A operands of dV += Pᵀ dO and
// dK += dSᵀ Q) and dS also into TMEM, where it is the A operand of
// dQ_it += dS·K_jt (TS form; dQ stays in TMEM across key tiles).  dK and dV
// are written per key tile, dQ once per slice: no atomics, no fp32 dQ
// accumulator in device memory.
//
// TMEM columns: S 0..127, dP 128..255, dS (packed pairs) 256..319, dK, dV,
// then the QT dQ tiles.
constexpr uint32_t kSlColS = 0u, kSlColDP = 128u, kSlColDsT = 256u;
// dK/dV accumulators are double-buffered across key tiles when TMEM has room.
__host__ __device__ constexpr int slice_kv_bufs(int DP, int QT) { return 320 + 4 * DP + QT * DP <= 512 ? 2 : 1; }
template <int DP>
__device__ __forceinline__ uint32_t sl_col_dk(uint32_t b) { return 320u + b * 2 * DP; }
template <int DP>
__device__ __forceinline__ uint32_t sl_col_dv(uint32_t b) { return 320u + b * 2 * DP + DP; }
template <int DP>
__device__ __forceinline__ uint32_t sl_col_dq(int it, int nb) { return 320u + nb * 2 * DP + it * DP; }
template <int DP>
__host__ __device__ constexpr bool slice_tmem_fits(int QT) { return 320 + 2 * DP + QT * DP <= 512; }

struct SliceBars {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t q_full[kMaxQStages], q_empty[kMaxQStages];
  uint64_t st_full, st_free, ds_full, ds_empty;
  uint64_t dkdv_full[2], dkdv_free[2], dq_full, dq_free;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

template <int DP>
struct SliceLayout {
  static constexpr uint32_t kTB = kTile * DP * 2;
  Ring k, v, b1, q, d_o, b2s, ld;
  uint32_t p, ds, bars, total;
  __host__ __device__ SliceLayout(bool has_b2, int qs) {
    uint32_t off = 0;
    k = Ring{off, 2 * kTB};
    v = Ring{off + kTB, 2 * kTB};
    off += 4 * kTB;
    q = Ring{off, 2 * kTB};
    d_o = Ring{off + kTB, 2 * kTB};
    off += qs * 2 * kTB;
    b2s = Ring{off, 32768u};
    if (has_b2) off += qs * 32768u;
    p = off;
    off += 32768u;
    ds = off;
    off += 32768u;
    b1 = Ring{off, 512u};
    off += 1024u;
    ld = Ring{off, 1024u};
    off += qs * 1024u;
    bars = off;
    off += (sizeof(SliceBars) + 127) & ~127u;
    total = off;
  }
};


template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void slice_producer(const BwdArgs& a, uint8_t* base, const SliceLayout<DP>& lay,
                                               SliceBars* bars, const WaitGuard& g, int lane, long long i0,
                                               long long i1) {
  constexpr uint32_t kTB = SliceLayout<DP>::kTB;
  const int QS = a.q_stages, QT = a.QT;
  const bool tma_b2 = a.bias2_mode == kBias2Tma;
  const uint32_t q_bytes = 2 * kTB + ((HAS_B2 && tma_b2) ? 32768u : 0u);
  uint32_t grp = 0, steps = 0, s = 0, ph = 0;
  SlIter c;
  c.init(i0, a);
  // next step's lse/delta and next key tile's mask, loaded one step ahead
  SlIter pc = c;
  int pjt = 0, pit = 0;
  LdRaw ldr;
  B1Raw b1r;
  auto prefetch_ld = [&]() {
    if (pc.b < a.B)
      ld_prefetch(ldr, a.lse, a.delta, (static_cast<size_t>(pc.b) * a.N + pc.n) * a.H + pc.h, a.L, pit * kTile,
                  lane);
  };
  auto advance_pf = [&]() {
    if (++pit == QT) {
      pit = 0;
      if (++pjt == QT) {
        pjt = 0;
        pc.next(a);
      }
    }
  };
  b1_prefetch(b1r, a.bias1 ? a.bias1 + (static_cast<size_t>(c.b) * a.N + c.n) * a.L : nullptr, a.L, 0, lane);
  prefetch_ld();
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, c.next(a)) {
    const int bn = c.b * a.N + c.n, bh = c.b * a.H + c.h;
    for (int jt = 0; ok && jt < QT; ++jt, ++grp) {
      const uint32_t kb = grp & 1;
      if (!mbar_wait_warp(smem_u32(&bars->kv_empty[kb]), ((grp >> 1) & 1) ^ 1, g)) { ok = false; break; }
      {
        const uint32_t full = smem_u32(&bars->kv_full[kb]);
        if (lane == 0) {
          mbar_expect_tx(full, 2 * kTB);
          tma_load_4d(smem_u32(base + lay.k[kb]), &a.tk, full, 0, c.h, jt * kTile, bn);
          tma_load_4d(smem_u32(base + lay.v[kb]), &a.tv, full, 0, c.h, jt * kTile, bn);
        }
        b1_store<BF16>(reinterpret_cast<float*>(base + lay.b1[kb]), b1r, a.bias1 != nullptr, a.L, jt * kTile, lane);
        mbar_arrive(full);
        // mask chunk of the next key tile (this slice's next jt, or the next slice's first)
        const int njt = jt + 1 < QT ? jt + 1 : 0;
        SlIter nc = c;
        if (njt == 0) nc.next(a);
        if (nc.b < a.B)
          b1_prefetch(b1r, a.bias1 ? a.bias1 + (static_cast<size_t>(nc.b) * a.N + nc.n) * a.L : nullptr, a.L,
                      njt * kTile, lane);
      }
      for (int it = 0; it < QT; ++it, ++steps) {
        if (!mbar_wait_warp(smem_u32(&bars->q_empty[s]), ph ^ 1, g)) { ok = false; break; }
        const uint32_t full = smem_u32(&bars->q_full[s]);
        if (lane == 0) {
          mbar_expect_tx(full, q_bytes);
          tma_load_4d(smem_u32(base + lay.q[s]), &a.tq, full, 0, c.h, it * kTile, bn);
          tma_load_4d(smem_u32(base + lay.d_o[s]), &a.tdo, full, 0, c.h, it * kTile, bn);
          if (HAS_B2 && tma_b2) {
            tma_load_3d(smem_u32(base + lay.b2s[s]), &a.tb2, full, jt * kTile, it * kTile, bh);
            tma_load_3d(smem_u32(base + lay.b2s[s] + 16384), &a.tb2, full, jt * kTile + 64, it * kTile, bh);
          }
        }
        if (HAS_B2 && !tma_b2)
          fill_b2_tile_loads(base + lay.b2s[s], a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L, it * kTile,
                             jt * kTile, lane);
        ld_store(reinterpret_cast<float*>(base + lay.ld[s]), ldr, lane);
        mbar_arrive(full);
        advance_pf();
        prefetch_ld();
        if (++s == static_cast<uint32_t>(QS)) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  }
  for (uint32_t b = 0; b < 2; ++b) {
    const uint32_t issued = (grp + 1 - b) / 2;
    if (issued > 0) drain_wait(smem_u32(&bars->kv_full[b]), (issued - 1) & 1, a.wait_ns, a.status);
  }
  for (uint32_t st = 0; st < static_cast<uint32_t>(QS); ++st) {
    const uint32_t issued = (steps + QS - 1 - st) / QS;
    if (issued > 0) drain_wait(smem_u32(&bars->q_full[st]), (issued - 1) & 1, a.wait_ns, a.status);
  }
}

struct SlStep {
  uint32_t u, grp, slice;
  int jt, it;
  uint32_t qs, qph;
};

template <int DP, bool BF16>
__device__ __forceinline__ bool slice_issue_sdp(const SlStep& st, uint8_t* base, const SliceLayout<DP>& lay,
                                                SliceBars* bars, uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
  const uint32_t kb = st.grp & 1;
  if (st.it == 0 && !mbar_wait(smem_u32(&bars->kv_full[kb]), (st.grp >> 1) & 1, g)) return false;
  if (!mbar_wait(smem_u32(&bars->q_full[st.qs]), st.qph, g)) return false;
  if (!mbar_wait(smem_u32(&bars->st_free), (st.u & 1) ^ 1, g)) return false;
  tc_fence_after();
  const uint32_t q_addr = smem_u32(base + lay.q[st.qs]), do_addr = smem_u32(base + lay.d_o[st.qs]);
  const uint32_t k_addr = smem_u32(base + lay.k[kb]), v_addr = smem_u32(base + lay.v[kb]);
#pragma unroll
  for (int k = 0; k < DP / 16; ++k)
    umma_ss(tmem + kSlColS, smem_desc(q_addr + k * 32, 16, 8 * RB, SWZ), smem_desc(k_addr + k * 32, 16, 8 * RB, SWZ),
            id_s, k > 0);
#pragma unroll
  for (int k = 0; k < DP / 16; ++k)
    umma_ss(tmem + kSlColDP, smem_desc(do_addr + k * 32, 16, 8 * RB, SWZ),
            smem_desc(v_addr + k * 32, 16, 8 * RB, SWZ), id_s, k > 0);
  umma_commit(smem_u32(&bars->st_full));
  return true;
}

template <int DP, bool BF16>
__device__ __forceinline__ bool slice_issue_grads(const SlStep& st, int QT, uint8_t* base, const SliceLayout<DP>& lay,
                                                  SliceBars* bars, uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_kv = idesc_f16(128, DP, BF16, true, true);  // dV, dK: MN-major A (smem) and B
  constexpr uint32_t id_q = idesc_f16(128, DP, BF16, false, true);  // dQ: A from TMEM, MN-major B
  const uint32_t kb = st.grp & 1;
  const int nb = slice_kv_bufs(DP, QT);
  const uint32_t db = st.grp % nb, dph = (st.grp / nb) & 1;
  if (!mbar_wait(smem_u32(&bars->ds_full), st.u & 1, g)) return false;
  if (st.it == 0 && !mbar_wait(smem_u32(&bars->dkdv_free[db]), dph ^ 1, g)) return false;
  if (st.it == 0 && st.jt == 0 && !mbar_wait(smem_u32(&bars->dq_free), (st.slice & 1) ^ 1, g)) return false;
  tc_fence_after();
  const uint32_t p_addr = smem_u32(base + lay.p), ds_addr = smem_u32(base + lay.ds);
  const uint32_t q_addr = smem_u32(base + lay.q[st.qs]), do_addr = smem_u32(base + lay.d_o[st.qs]);
  const uint32_t k_addr = smem_u32(base + lay.k[kb]);
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // dV += Pᵀ dO   (K = 128 queries)
    const uint64_t ad = smem_desc(p_addr + k * 16 * 128, 16384, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(do_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ss(tmem + sl_col_dv<DP>(db), ad, bd, id_kv, (st.it > 0 || k > 0) ? 1u : 0u);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // dK += dSᵀ Q
    const uint64_t ad = smem_desc(ds_addr + k * 16 * 128, 16384, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(q_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ss(tmem + sl_col_dk<DP>(db), ad, bd, id_kv, (st.it > 0 || k > 0) ? 1u : 0u);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // dQ_it += dS K_jt   (K = 128 keys; dS from TMEM)
    const uint64_t bd = smem_desc(k_addr + k * 16 * RB, kTile * RB, 8 * RB, SWZ);
    umma_ts(tmem + sl_col_dq<DP>(st.it, nb), tmem + kSlColDsT + k * 8, bd, id_q, (st.jt > 0 || k > 0) ? 1u : 0u);
  }
  umma_commit(smem_u32(&bars->ds_empty));
  umma_commit(smem_u32(&bars->q_empty[st.qs]));
  if (st.it == QT - 1) {
    umma_commit(smem_u32(&bars->dkdv_full[db]));
    umma_commit(smem_u32(&bars->kv_empty[kb]));
    if (st.jt == QT - 1) umma_commit(smem_u32(&bars->dq_full));
  }
  return true;
}

template <int DP, bool BF16>
__device__ __forceinline__ void slice_mma(const BwdArgs& a, uint8_t* base, const SliceLayout<DP>& lay,
                                          SliceBars* bars, uint32_t tmem, const WaitGuard& g, long long i0,
                                          long long i1) {
  const int QS = a.q_stages, QT = a.QT;
  const uint32_t total = static_cast<uint32_t>((i1 - i0) * QT * QT);
  auto advance = [&](SlStep& st) {
    ++st.u;
    if (++st.it == QT) {
      st.it = 0;
      ++st.grp;
      if (++st.jt == QT) {
        st.jt = 0;
        ++st.slice;
      }
    }
    if (++st.qs == static_cast<uint32_t>(QS)) {
      st.qs = 0;
      st.qph ^= 1;
    }
  };
  bool ok = total > 0;
  SlStep cur{0, 0, 0, 0, 0, 0, 0};
  if (QS >= 2) {
    if (ok) ok = slice_issue_sdp<DP, BF16>(cur, base, lay, bars, tmem, g);
    for (uint32_t u = 0; ok && u < total; ++u) {
      SlStep nxt = cur;
      advance(nxt);
      if (u + 1 < total && !slice_issue_sdp<DP, BF16>(nxt, base, lay, bars, tmem, g)) { ok = false; break; }
      if (!slice_issue_grads<DP, BF16>(cur, QT, base, lay, bars, tmem, g)) { ok = false; break; }
      cur = nxt;
    }
  } else {
    for (uint32_t u = 0; ok && u < total; ++u) {
      if (!slice_issue_sdp<DP, BF16>(cur, base, lay, bars, tmem, g)) { ok = false; break; }
      if (!slice_issue_grads<DP, BF16>(cur, QT, base, lay, bars, tmem, g)) { ok = false; break; }
      advance(cur);
    }
  }
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

// P and dS for one 32-key chunk: the P/dS smem tiles as in the main kernel, and dS
// (packed pairs, 16 columns) into TMEM for the dQ MMA.
template <bool BF16, bool HAS_B2>
__device__ __forceinline__ void slice_chunk(const uint32_t (&sv)[32], const uint32_t (&pv)[32], const float* b1c,
                                            const uint8_t* b2half, uint8_t* pt, uint8_t* dt, uint32_t ds_tcol, int r,
                                            int c4, float lse2, float dlt, float2 sl2) {
  const float2 nl2 = make_float2(-lse2, -lse2), l2e2 = make_float2(kLog2e, kLog2e), nd2 = make_float2(-dlt, -dlt);
  uint32_t ddt[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 m0 = *reinterpret_cast<const float4*>(b1c + q * 8);
    const float4 m1 = *reinterpret_cast<const float4*>(b1c + q * 8 + 4);
    const float2 mk[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                          make_float2(m1.z, m1.w)};
    uint4 pb = make_uint4(0u, 0u, 0u, 0u);
    if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2half + swz_offset(r, c4 * 4 + q, 128));
    const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
    uint32_t pp[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int x = q * 8 + e2 * 2;
      float2 t = fma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, mk[e2]);
      if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
      t = add2(t, nl2);
      const float p0 = ex2(t.x), p1 = ex2(t.y);
      const float2 dpd = add2(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), nd2);
      const float2 ds = mul2(make_float2(p0, p1), dpd);
      pp[e2] = pack2<BF16>(p0, p1);
      ddt[q * 4 + e2] = pack2<BF16>(ds.x, ds.y);
    }
    const uint32_t off = swz_offset(r, c4 * 4 + q, 128);
    *reinterpret_cast<uint4*>(pt + off) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
    *reinterpret_cast<uint4*>(dt + off) = make_uint4(ddt[q * 4], ddt[q * 4 + 1], ddt[q * 4 + 2], ddt[q * 4 + 3]);
  }
  tmem_st16(ds_tcol, ddt);
}

// dK, dV of key tile jt of slice c (TMEM lanes = keys): this warp's DP/2 columns.
template <int DP, bool BF16>
__device__ __forceinline__ bool slice_write_dkdv(const BwdArgs& a, const SlIter& c, int jt, uint32_t grp,
                                                 SliceBars* bars, uint32_t trow, int r, int hc, int lane,
                                                 const WaitGuard& g) {
  constexpr int HD = DP / 2;
  const int nb = slice_kv_bufs(DP, a.QT);
  const uint32_t db = grp % nb;
  if (!mbar_wait_warp(smem_u32(&bars->dkdv_full[db]), (grp / nb) & 1, g)) return false;
  tc_fence_after();
  float kx[HD], vx[HD];
  const uint32_t ck = trow + sl_col_dk<DP>(db) + hc * HD, cv = trow + sl_col_dv<DP>(db) + hc * HD;
  if constexpr (HD == 8) {
    uint32_t x[8], y[8];
    tmem_ld8(ck, x);
    tmem_ld8(cv, y);
    tmem_wait_ld(x);
    tmem_wait_ld(y);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      kx[e] = __uint_as_float(x[e]);
      vx[e] = __uint_as_float(y[e]);
    }
  } else {
    uint32_t x[HD / 16][16], y[HD / 16][16];
#pragma unroll
    for (int q = 0; q < HD / 16; ++q) {
      tmem_ld16(ck + q * 16, x[q]);
      tmem_ld16(cv + q * 16, y[q]);
    }
#pragma unroll
    for (int q = 0; q < HD / 16; ++q) {
      tmem_wait_ld(x[q]);
      tmem_wait_ld(y[q]);
    }
#pragma unroll
    for (int q = 0; q < HD / 16; ++q)
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        kx[q * 16 + e] = __uint_as_float(x[q][e]);
        vx[q * 16 + e] = __uint_as_float(y[q][e]);
      }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->dkdv_free[db]));
  const int j = jt * kTile + r;
  if (j < a.L) {
    const long long bn = static_cast<long long>(c.b) * a.N + c.n, inner = c.h * a.D + hc * HD;
    uint16_t* dk = a.dk + bn * a.r_dk.bn + j * a.r_dk.l + inner;
    uint16_t* dv = a.dv + bn * a.r_dv.bn + j * a.r_dv.l + inner;
#pragma unroll
    for (int e = 0; e < HD; e += 8)
      if (hc * HD + e < a.D) {
        uint4 pk, pv4;
        pk.x = pack2<BF16>(kx[e + 0] * a.scale, kx[e + 1] * a.scale);
        pk.y = pack2<BF16>(kx[e + 2] * a.scale, kx[e + 3] * a.scale);
        pk.z = pack2<BF16>(kx[e + 4] * a.scale, kx[e + 5] * a.scale);
        pk.w = pack2<BF16>(kx[e + 6] * a.scale, kx[e + 7] * a.scale);
        pv4.x = pack2<BF16>(vx[e + 0], vx[e + 1]);
        pv4.y = pack2<BF16>(vx[e + 2], vx[e + 3]);
        pv4.z = pack2<BF16>(vx[e + 4], vx[e + 5]);
        pv4.w = pack2<BF16>(vx[e + 6], vx[e + 7]);
        *reinterpret_cast<uint4*>(dk + e) = pk;
        *reinterpret_cast<uint4*>(dv + e) = pv4;
      }
  }
  return true;
}

// dQ of slice c (TMEM lanes = queries of each query tile): this warp's DP/2 columns, × s.
template <int DP, bool BF16>
__device__ __forceinline__ bool slice_write_dq(const BwdArgs& a, const SlIter& c, uint32_t slice, SliceBars* bars,
                                               uint32_t trow, int r, int hc, int lane, const WaitGuard& g) {
  constexpr int HD = DP / 2;
  if (!mbar_wait_warp(smem_u32(&bars->dq_full), slice & 1, g)) return false;
  tc_fence_after();
  const long long bn = static_cast<long long>(c.b) * a.N + c.n;
  for (int it = 0; it < a.QT; ++it) {
    float v[HD];
    const uint32_t col = trow + sl_col_dq<DP>(it, slice_kv_bufs(DP, a.QT)) + hc * HD;
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
    const int i = it * kTile + r;
    if (i < a.L) {
      uint16_t* dst = a.dq + bn * a.r_dq.bn + static_cast<long long>(i) * a.r_dq.l + c.h * a.D + hc * HD;
#pragma unroll
      for (int e = 0; e < HD; e += 8)
        if (hc * HD + e < a.D) {
          uint4 pk;
          pk.x = pack2<BF16>(v[e + 0] * a.scale, v[e + 1] * a.scale);
          pk.y = pack2<BF16>(v[e + 2] * a.scale, v[e + 3] * a.scale);
          pk.z = pack2<BF16>(v[e + 4] * a.scale, v[e + 5] * a.scale);
          pk.w = pack2<BF16>(v[e + 6] * a.scale, v[e + 7] * a.scale);
          *reinterpret_cast<uint4*>(dst + e) = pk;
        }
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
  return true;
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void slice_compute(const BwdArgs& a, uint8_t* base, const SliceLayout<DP>& lay,
                                              SliceBars* bars, uint32_t tmem, const WaitGuard& g, long long i0,
                                              long long i1) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = w & 3, hc = w >> 2;
  const int r = quad * 32 + lane;
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int QS = a.q_stages, QT = a.QT;
  uint32_t u = 0, grp = 0, slice = 0, s = 0, ph = 0;
  SlIter cur, prev;
  cur.init(i0, a);
  prev = cur;
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, ++slice) {
    if (item > i0) {
      prev = cur;
      cur.next(a);
    }
    for (int jt = 0; ok && jt < QT; ++jt, ++grp) {
      const uint32_t kb = grp & 1;
      if (!mbar_wait_warp(smem_u32(&bars->kv_full[kb]), (grp >> 1) & 1, g)) { ok = false; break; }
      const float* b1 = reinterpret_cast<const float*>(base + lay.b1[kb]) + hc * 64;
      for (int it = 0; it < QT; ++it, ++u) {
        if (!mbar_wait_warp(smem_u32(&bars->q_full[s]), ph, g)) { ok = false; break; }
        const float* ld = reinterpret_cast<const float*>(base + lay.ld[s]);
        const float lse2 = ld[r], dlt = ld[128 + r];
        const uint8_t* b2half = base + lay.b2s[s] + hc * 16384;
        if (!mbar_wait_warp(smem_u32(&bars->st_full), u & 1, g)) { ok = false; break; }
        if (!mbar_wait_warp(smem_u32(&bars->ds_empty), (u & 1) ^ 1, g)) { ok = false; break; }
        tc_fence_after();
        uint8_t* pt = base + lay.p + hc * 16384;
        uint8_t* dt = base + lay.ds + hc * 16384;
        const uint32_t dst = trow + kSlColDsT + hc * 32;
        {
          uint32_t sv[32], pv[32];
          tmem_ld32(trow + kSlColS + hc * 64, sv);
          tmem_ld32(trow + kSlColDP + hc * 64, pv);
          tmem_wait_ld(sv);
          tmem_wait_ld(pv);
          slice_chunk<BF16, HAS_B2>(sv, pv, b1, b2half, pt, dt, dst, r, 0, lse2, dlt, sl2);
        }
        {
          uint32_t sv[32], pv[32];
          tmem_ld32(trow + kSlColS + hc * 64 + 32, sv);
          tmem_ld32(trow + kSlColDP + hc * 64 + 32, pv);
          tmem_wait_ld(sv);
          tmem_wait_ld(pv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->st_free));
          slice_chunk<BF16, HAS_B2>(sv, pv, b1 + 32, b2half, pt, dt, dst + 16, r, 1, lse2, dlt, sl2);
        }
        tmem_wait_st();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bars->ds_full));
          mbar_arrive(smem_u32(&bars->q_empty[s]));
          if (it == QT - 1) mbar_arrive(smem_u32(&bars->kv_empty[kb]));
        }
        if (it == 0 && grp > 0) {
          // the previous key tile's dK/dV are complete (of this slice, or of the previous one)
          if (!slice_write_dkdv<DP, BF16>(a, jt > 0 ? cur : prev, jt > 0 ? jt - 1 : QT - 1, grp - 1, bars, trow, r,
                                          hc, lane, g)) {
            ok = false;
            break;
          }
          if (jt == 0 && !slice_write_dq<DP, BF16>(a, prev, slice - 1, bars, trow, r, hc, lane, g)) {
            ok = false;
            break;
          }
        }
        if (++s == static_cast<uint32_t>(QS)) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  }
  if (ok && grp > 0) {
    if (slice_write_dkdv<DP, BF16>(a, cur, QT - 1, grp - 1, bars, trow, r, hc, lane, g))
      slice_write_dq<DP, BF16>(a, cur, slice - 1, bars, trow, r, hc, lane, g);
  }
}

template <int DP, bool BF16, bool HAS_B2>
__global__ void __launch_bounds__(kThreads, 1) evo_bwd_slice(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SliceLayout<DP> lay(HAS_B2, a.q_stages);
  SliceBars* bars = reinterpret_cast<SliceBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long i0 = static_cast<long long>(blockIdx.x) * a.chunk;
  const long long i1 = i0 + a.chunk < a.items ? i0 + a.chunk : a.items;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1 + kComputeWarps);
    }
    for (int s = 0; s < kMaxQStages; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 32);
      mbar_init(smem_u32(&bars->q_empty[s]), 1 + kComputeWarps);
    }
    mbar_init(smem_u32(&bars->st_full), 1);
    mbar_init(smem_u32(&bars->st_free), kComputeWarps);
    mbar_init(smem_u32(&bars->ds_full), kComputeWarps);
    mbar_init(smem_u32(&bars->ds_empty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->dkdv_full[b]), 1);
      mbar_init(smem_u32(&bars->dkdv_free[b]), kComputeWarps);
    }
    mbar_init(smem_u32(&bars->dq_full), 1);
    mbar_init(smem_u32(&bars->dq_free), kComputeWarps);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    tma_prefetch_desc(&a.tdo);
    if (HAS_B2 && a.bias2_mode == kBias2Tma) tma_prefetch_desc(&a.tb2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const WaitGuard g{a.wait_ns, a.status, &bars->abort};
  if (warp == kProducerWarp) {
    slice_producer<DP, BF16, HAS_B2>(a, base, lay, bars, g, lane, i0, i1);
  } else if (warp == kMmaWarp) {
    if (lane == 0) slice_mma<DP, BF16>(a, base, lay, bars, tmem, g, i0, i1);
    __syncwarp();
  } else {
    slice_compute<DP, BF16, HAS_B2>(a, base, lay, bars, tmem, g, i0, i1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ evo_bwd_db2_part
constexpr int kMaxPartStages = 3;

struct PartBars {
  uint64_t b2_full;
  uint64_t st_full[kMaxPartStages], st_free[kMaxPartStages];  // stage ring (Q, dO, K, V, key mask, lse, delta)
  uint64_t mm_full[2], mm_free[2];                            // TMEM S/dP double buffer
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

template <int DP>
struct PartLayout {
  static constexpr uint32_t kTB = kTile * DP * 2;
  Ring q, d_o, k, v, b1, ld;
  uint32_t b2, stg, bars, total;
  // stage: also 64 KB of staging for the tile stores of the partial sums (8 KB per compute warp)
  __host__ __device__ PartLayout(int ns, bool stage) {
    uint32_t off = 0;
    q = Ring{off, 4 * kTB};
    d_o = Ring{off + kTB, 4 * kTB};
    k = Ring{off + 2 * kTB, 4 * kTB};
    v = Ring{off + 3 * kTB, 4 * kTB};
    off += ns * 4 * kTB;
    b2 = off;
    off += 32768u;
    stg = off;
    if (stage) off += 65536u;
    b1 = Ring{off, 1536u};
    ld = Ring{off + 512u, 1536u};
    off += ns * 1536u;
    bars = off;
    off += (sizeof(PartBars) + 127) & ~127u;
    total = off;
  }
};

__device__ __forceinline__ uint32_t col_ps(uint32_t b) { return b ? 256u : 0u; }
__device__ __forceinline__ uint32_t col_pdp(uint32_t b) { return b ? 384u : 128u; }

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
__global__ void __launch_bounds__(kThreads, 1) evo_bwd_db2_part(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NS = a.part_stages;
  const PartLayout<DP> lay(NS, a.db2p_tma != 0);
  PartBars* bars = reinterpret_cast<PartBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PartItem c = part_item(a);
  const int nn = c.n1 - c.n0;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->b2_full), 32);
    for (int s = 0; s < kMaxPartStages; ++s) {
      mbar_init(smem_u32(&bars->st_full[s]), 32);
      mbar_init(smem_u32(&bars->st_free[s]), 1 + kComputeWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->mm_full[s]), 1);
      mbar_init(smem_u32(&bars->mm_free[s]), kComputeWarps);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const WaitGuard g{a.wait_ns, a.status, &bars->abort};
  constexpr uint32_t kTB = PartLayout<DP>::kTB;
  const int bh = c.b * a.H + c.h;

  if (warp == kProducerWarp) {  // ---------------- producer
    const uint32_t full_b2 = smem_u32(&bars->b2_full);
    if (a.bias2_mode == kBias2Tma) {
      if (lane == 0) {
        mbar_expect_tx(full_b2, 32768u);
        tma_load_3d(smem_u32(base + lay.b2), &a.tb2, full_b2, c.jt * kTile, c.it * kTile, bh);
        tma_load_3d(smem_u32(base + lay.b2 + 16384), &a.tb2, full_b2, c.jt * kTile + 64, c.it * kTile, bh);
      }
    } else {
      fill_b2_tile_loads(base + lay.b2, a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L, c.it * kTile,
                         c.jt * kTile, lane);
    }
    mbar_arrive(full_b2);
    int k = 0, s = 0, ph = 0;
    B1Raw b1r;
    LdRaw ldr;
    auto prefetch = [&](int kk) {
      const int bn = c.b * a.N + c.n0 + kk;
      b1_prefetch(b1r, a.bias1 ? a.bias1 + static_cast<size_t>(bn) * a.L : nullptr, a.L, c.jt * kTile, lane);
      ld_prefetch(ldr, a.lse, a.delta, static_cast<size_t>(bn) * a.H + c.h, a.L, c.it * kTile, lane);
    };
    if (nn > 0) prefetch(0);
    for (; k < nn; ++k) {
      if (!mbar_wait_warp(smem_u32(&bars->st_free[s]), ph ^ 1, g)) break;
      const int bn = c.b * a.N + c.n0 + k;
      const uint32_t full = smem_u32(&bars->st_full[s]);
      if (lane == 0) {
        mbar_expect_tx(full, 4 * kTB);
        tma_load_4d(smem_u32(base + lay.q[s]), &a.tq, full, 0, c.h, c.it * kTile, bn);
        tma_load_4d(smem_u32(base + lay.d_o[s]), &a.tdo, full, 0, c.h, c.it * kTile, bn);
        tma_load_4d(smem_u32(base + lay.k[s]), &a.tk, full, 0, c.h, c.jt * kTile, bn);
        tma_load_4d(smem_u32(base + lay.v[s]), &a.tv, full, 0, c.h, c.jt * kTile, bn);
      }
      b1_store<BF16>(reinterpret_cast<float*>(base + lay.b1[s]), b1r, a.bias1 != nullptr, a.L, c.jt * kTile, lane);
      ld_store(reinterpret_cast<float*>(base + lay.ld[s]), ldr, lane);
      mbar_arrive(full);
      if (k + 1 < nn) prefetch(k + 1);
      if (++s == NS) {
        s = 0;
        ph ^= 1;
      }
    }
    drain_wait(full_b2, 0, a.wait_ns, a.status);
    for (int st = 0; st < NS; ++st) {
      const int issued = (k + NS - 1 - st) / NS;
      if (issued > 0) drain_wait(smem_u32(&bars->st_full[st]), (issued - 1) & 1, a.wait_ns, a.status);
    }
  } else if (warp == kMmaWarp) {  // ---------------- MMA
    if (lane == 0) {
      constexpr uint32_t RB = DP * 2;
      constexpr uint32_t SWZ = swizzle_for_row(RB);
      constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
      int s = 0, ph = 0;
      for (int k = 0; k < nn; ++k) {
        const uint32_t mb = k & 1;
        if (!mbar_wait(smem_u32(&bars->st_full[s]), ph, g)) break;
        if (!mbar_wait(smem_u32(&bars->mm_free[mb]), ((k >> 1) & 1) ^ 1, g)) break;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(base + lay.q[s]), do_addr = smem_u32(base + lay.d_o[s]);
        const uint32_t k_addr = smem_u32(base + lay.k[s]), v_addr = smem_u32(base + lay.v[s]);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk)
          umma_ss(tmem + col_ps(mb), smem_desc(q_addr + kk * 32, 16, 8 * RB, SWZ),
                  smem_desc(k_addr + kk * 32, 16, 8 * RB, SWZ), id_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk)
          umma_ss(tmem + col_pdp(mb), smem_desc(do_addr + kk * 32, 16, 8 * RB, SWZ),
                  smem_desc(v_addr + kk * 32, 16, 8 * RB, SWZ), id_s, kk > 0);
        umma_commit(smem_u32(&bars->mm_full[mb]));
        umma_commit(smem_u32(&bars->st_free[s]));
        if (++s == NS) {
          s = 0;
          ph ^= 1;
        }
      }
      umma_commit(smem_u32(&bars->drain));
      drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
    }
    __syncwarp();
  } else {  // ---------------- compute: warp (quad, half) = 32 query rows × 64 keys
    const int quad = warp & 3, hc = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
    const uint8_t* b2half = base + lay.b2 + hc * 16384;
    float acc[64];
#pragma unroll
    for (int e = 0; e < 64; ++e) acc[e] = 0.0f;
    bool ok = mbar_wait_warp(smem_u32(&bars->b2_full), 0, g);
    int s = 0, ph = 0;
    for (int k = 0; ok && k < nn; ++k) {
      const uint32_t mb = k & 1;
      if (!mbar_wait_warp(smem_u32(&bars->st_full[s]), ph, g)) { ok = false; break; }
      const float* ld = reinterpret_cast<const float*>(base + lay.ld[s]);
      const float lse2 = ld[r], dlt = ld[128 + r];
      const float* b1 = reinterpret_cast<const float*>(base + lay.b1[s]) + hc * 64;
      if (!mbar_wait_warp(smem_u32(&bars->mm_full[mb]), (k >> 1) & 1, g)) { ok = false; break; }
      tc_fence_after();
      // 16-key chunks of S and dP: chunk k+1's TMEM loads are in flight while chunk k is
      // summed (one pair outstanding, so each wait covers the chunk about to be used)
      const float2 nl2 = make_float2(-lse2, -lse2), l2e2 = make_float2(kLog2e, kLog2e),
                   nd2 = make_float2(-dlt, -dlt);
      const uint32_t cs = trow + col_ps(mb) + hc * 64, cpd = trow + col_pdp(mb) + hc * 64;
      auto chunk16 = [&](const uint32_t (&sv)[16], const uint32_t (&pv)[16], int kc) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float4 m0 = *reinterpret_cast<const float4*>(b1 + kc * 16 + q * 8);
          const float4 m1 = *reinterpret_cast<const float4*>(b1 + kc * 16 + q * 8 + 4);
          const float2 mk[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                                make_float2(m1.z, m1.w)};
          const uint4 pb = *reinterpret_cast<const uint4*>(b2half + swz_offset(r, kc * 2 + q, 128));
          const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int x = q * 8 + e2 * 2, y = kc * 16 + x;
            float2 t = fma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, mk[e2]);
            t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
            t = add2(t, nl2);
            const float2 pr = make_float2(ex2(t.x), ex2(t.y));
            const float2 dpd = add2(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), nd2);
            const float2 a2 = fma2(pr, dpd, make_float2(acc[y], acc[y + 1]));
            acc[y] = a2.x;
            acc[y + 1] = a2.y;
          }
        }
      };
      {
        uint32_t s0[16], p0[16], s1[16], p1[16];
        tmem_ld16(cs, s0);
        tmem_ld16(cpd, p0);
        tmem_wait_ld(s0);
        tmem_wait_ld(p0);
        tmem_ld16(cs + 16, s1);
        tmem_ld16(cpd + 16, p1);
        chunk16(s0, p0, 0);
        tmem_wait_ld(s1);
        tmem_wait_ld(p1);
        tmem_ld16(cs + 32, s0);
        tmem_ld16(cpd + 32, p0);
        chunk16(s1, p1, 1);
        tmem_wait_ld(s0);
        tmem_wait_ld(p0);
        tmem_ld16(cs + 48, s1);
        tmem_ld16(cpd + 48, p1);
        chunk16(s0, p0, 2);
        tmem_wait_ld(s1);
        tmem_wait_ld(p1);
        chunk16(s1, p1, 3);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->mm_free[mb]));
        mbar_arrive(smem_u32(&bars->st_free[s]));
      }
      if (++s == NS) {
        s = 0;
        ph ^= 1;
      }
    }
    const int i = c.it * kTile + r;
    if (ok && a.db2p_tma) {
      // this warp's 32 rows × 64 keys: two [32][32] fp32 blocks (128B swizzle) → two tile stores
      uint8_t* blk = base + lay.stg + warp * 8192;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<float4*>(blk + hb * 4096 + swz_offset(lane, ch, 128)) =
              make_float4(acc[hb * 32 + ch * 4], acc[hb * 32 + ch * 4 + 1], acc[hb * 32 + ch * 4 + 2],
                          acc[hb * 32 + ch * 4 + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int plane = c.grp * a.B * a.H + bh, j0 = c.jt * kTile + hc * 64, i0 = c.it * kTile + quad * 32;
        tma_store_3d(&a.tdb2p, smem_u32(blk), j0, i0, plane);
        tma_store_3d(&a.tdb2p, smem_u32(blk + 4096), j0 + 32, i0, plane);
        bulk_commit_group();
        bulk_wait_all();
      }
    } else if (ok && i < a.L) {
      const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
      float* dst = a.db2_part + c.grp * plane + (static_cast<long long>(bh) * a.L + i) * a.L;
      const int j0 = c.jt * kTile + hc * 64;
#pragma unroll
      for (int e = 0; e < 64; ++e)
        if (j0 + e < a.L) dst[j0 + e] = acc[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ launch

unsigned grid_for(long long work, long long per_block) {
  long long g = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <int DP, bool BF16, bool HAS_B2>
cudaError_t launch_main(BwdArgs a, cudaStream_t st) {
  const MainLayout<DP> lay(HAS_B2, a.q_stages, a.pds_bufs, a.kv_bufs);
  const size_t smem = one_cta_per_sm(lay.total + 1024);
  auto kern = evo_bwd_main<DP, BF16, HAS_B2>;
  static bool limit_set[64] = {};
  cudaError_t e = ensure_smem_limit(kern, kMaxSmem, limit_set);
  if (e != cudaSuccess) return e;
  // whole slices per CTA; at most kMainMaxCtas CTAs (the workspace holds QT × 128 × DP
  // fp32 dQ values for each)
  a.items = static_cast<long long>(a.B) * a.H * a.N;
  long long ctas = num_sms();
  if (ctas > kMainMaxCtas) ctas = kMainMaxCtas;
  a.chunk = (a.items + ctas - 1) / ctas;
  const long long grid = (a.items + a.chunk - 1) / a.chunk;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int DP, bool BF16, bool HAS_B2>
cudaError_t launch_slice(BwdArgs a, cudaStream_t st) {
  const SliceLayout<DP> lay(HAS_B2, a.q_stages);
  const size_t smem = one_cta_per_sm(lay.total + 1024);
  auto kern = evo_bwd_slice<DP, BF16, HAS_B2>;
  static bool limit_set[64] = {};
  cudaError_t e = ensure_smem_limit(kern, kMaxSmem, limit_set);
  if (e != cudaSuccess) return e;
  a.items = static_cast<long long>(a.B) * a.H * a.N;
  const long long sms = num_sms();
  a.chunk = (a.items + sms - 1) / sms;
  const long long grid = (a.items + a.chunk - 1) / a.chunk;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// Query-major slice mode: every dQ tile of a (b, n, h) slice stays in TMEM (no atomics).
template <int DP>
int slice_q_stages(int QT, bool has_b2) {
  if (!slice_tmem_fits<DP>(QT)) return 0;
  for (int q = 3; q >= 2; --q)
    if (SliceLayout<DP>(has_b2, q).total + 1024 <= kMaxSmem) return q;
  return 0;
}

template <int DP, bool BF16>
cudaError_t launch_bwd_d(BwdArgs a, cudaStream_t st, const ProfileEvents* prof) {
  const bool has_b2 = a.bias2_mode != kBias2None;
  const long long rows = static_cast<long long>(a.B) * a.N * a.L * a.H;
  a.items = static_cast<long long>(a.B) * a.H * a.QT * a.N;
  const BwdPlan plan = bwd_plan(DP, a.QT, has_b2);
  const int slice_qs = plan.mode == kBwdSlice ? plan.q_stages : 0;
  // the streamed key-major kernel does not skip masked tiles: with skipping asked for, the
  // per-key-tile kernel runs instead (the workspace covers both)
  const bool km_stream = plan.mode == kBwdKeyMajorStream && !a.tile_skip;
  const bool km_any = plan.mode == kBwdKeyMajor || km_stream;
  if (!km_any && !a.db1p) a.b2t = nullptr;
  prof_record(prof, 2, st);
  evo_bwd_pre<DP, BF16><<<grid_for(rows, 256), 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_record(prof, 3, st);
  if (km_any) {
    // The streamed kernel leaves the key-mask gradient to the separate pass, as the
    // per-key-tile kernel does, so that a call gives the same bytes with or without
    // masked-tile skipping.
    BwdArgs ak = a;
    ak.q_stages = plan.q_stages;
    if (km_stream) ak.db1p = nullptr;
    if ((e = launch_bwd_kmajor(ak, DP, BF16, has_b2, km_stream, st)) != cudaSuccess) return e;
    prof_record(prof, 4, st);
    prof_record(prof, 5, st);  // no dQ cast: dQ stays in TMEM or leaves through the workspace
  } else if (slice_qs > 0) {
    a.q_stages = slice_qs;
    e = has_b2 ? launch_slice<DP, BF16, true>(a, st) : launch_slice<DP, BF16, false>(a, st);
    if (e != cudaSuccess) return e;
    prof_record(prof, 4, st);
    prof_record(prof, 5, st);  // no dQ cast in slice mode
  } else {

  // per-key-tile kernel: double P/dS buffers with the deepest Q/dO ring (at least two
  // stages) that fits; otherwise single buffers
  auto fits = [&](int qs, int pds) { return MainLayout<DP>(has_b2, qs, pds, 2).total + 1024 <= kMaxSmem; };
  int qs = 1, pds = 1;
  for (int q = 4; q >= 2 && pds == 1; --q)
    if (fits(q, 2)) {
      qs = q;
      pds = 2;
    }
  if (pds == 1)
    for (int q = 4; q >= 1; --q)
      if (fits(q, 1)) {
        qs = q;
        break;
      }
  a.q_stages = qs;
  a.pds_bufs = pds;
  a.kv_bufs = 2;
  if (a.tile_skip) {  // masked key tiles: skip bits, and zeros for dK/dV of the skipped tiles
    evo_bwd_tile_mask<BF16><<<grid_for(static_cast<long long>(a.B) * a.N * 32, 256), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  e = has_b2 ? launch_main<DP, BF16, true>(a, st) : launch_main<DP, BF16, false>(a, st);
  if (e != cudaSuccess) return e;
  prof_record(prof, 4, st);
  prof_record(prof, 5, st);  // no dQ cast: the kernel writes dQ
  }

  if (a.db1p) {  // key-mask gradient: partials (by the key-major kernel, or a separate pass), then the sum
    if (plan.mode != kBwdKeyMajor && (e = launch_bwd_db1_partials(a, DP, BF16, has_b2, st)) != cudaSuccess)
      return e;
    if ((e = launch_bwd_db1_sum(a, BF16, st)) != cudaSuccess) return e;
  }
  if (has_b2 && a.dbias2) {
    // deepest ring that fits; staging for tile stores of the partials when it fits too
    auto pfits = [&](int ns, bool stg) { return PartLayout<DP>(ns, stg).total + 1024 <= kMaxSmem; };
    if (a.db2p_tma && !pfits(2, true)) a.db2p_tma = 0;
    const bool stg = a.db2p_tma != 0;
    a.part_stages = pfits(3, stg) ? 3 : 2;
    const PartLayout<DP> lay(a.part_stages, stg);
    const size_t smem = one_cta_per_sm(lay.total + 1024);
    auto kern = evo_bwd_db2_part<DP, BF16>;
    static bool limit_set[64] = {};
    if ((e = ensure_smem_limit(kern, kMaxSmem, limit_set)) != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(a.B) * a.H * a.groups * a.QT * a.QT;
    kern<<<static_cast<unsigned>(blocks), kThreads, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_record(prof, 6, st);
    if (!a.db2_no_sum) {
      const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
      evo_bwd_db2_sum<BF16><<<grid_for(plane, 256), 256, 0, st>>>(a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    prof_record(prof, 7, st);
  }
  return cudaSuccess;
}

template <int DP>
BwdPlan plan_d(int QT, bool has_b2) {
  const int km = kmajor_q_stages(DP, QT, has_b2);
  if (km > 0) return {kBwdKeyMajor, km};
  const int kms = kmajor_stream_q_stages(DP, has_b2);
  if (kms > 0) return {kBwdKeyMajorStream, kms};
  const int sl = slice_q_stages<DP>(QT, has_b2);
  if (sl > 0) return {kBwdSlice, sl};
  return {kBwdMain, 0};
}

}  // namespace

BwdPlan bwd_plan(int DP, int QT, bool has_b2) {
  switch (DP) {
    case 16: return plan_d<16>(QT, has_b2);
    case 32: return plan_d<32>(QT, has_b2);
    default: return plan_d<64>(QT, has_b2);
  }
}

cudaError_t launch_bwd_db2_sum(const BwdArgs& a, bool bf16, cudaStream_t st) {
  const long long plane = static_cast<long long>(a.B) * a.H * a.L * a.L;
  if (plane <= 0 || a.groups <= 0) return cudaSuccess;
  if (bf16)
    evo_bwd_db2_sum<true><<<grid_for(plane, 256), 256, 0, st>>>(a);
  else
    evo_bwd_db2_sum<false><<<grid_for(plane, 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdArgs& a, int DP, bool bf16, cudaStream_t st, const ProfileEvents* p) {
  switch (DP) {
    case 16: return bf16 ? launch_bwd_d<16, true>(a, st, p) : launch_bwd_d<16, false>(a, st, p);
    case 32: return bf16 ? launch_bwd_d<32, true>(a, st, p) : launch_bwd_d<32, false>(a, st, p);
    case 64: return bf16 ? launch_bwd_d<64, true>(a, st, p) : launch_bwd_d<64, false>(a, st, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace evo
