// evo_bwd_kmajor.cu — key-major slice backward of memory-efficient biased
// Evoformer attention for sm_103a.
//
// Definition: web page "DeepSpeed4Science 技术指南：AI4Science 大模型长序列训练
// 与 Evoformer 内存高效注意力内核实战" §3.7 (the backward forms delta, then dQ, dK,
// dV from the probabilities rebuilt with the saved lse) and §3.2 (recompute
// instead of storing the attention matrix).
//
// One CTA owns whole (b, n, h) slices, like the query-major slice kernel, but
// the scores are formed transposed: for key tile jt and query tile it,
//   Sᵀ = K Qᵀ and dPᵀ = V dOᵀ      (TMEM lane = key, column = query)
// so that each compute thread owns one key j of the tile.  It rebuilds
//   Pᵀ_ji = exp2(s·log2e·S_ij + mask_j·log2e + bias2_ij·log2e − lse_i·log2e)
//   dSᵀ_ji = Pᵀ_ji (dP_ij − delta_i)
// writes Pᵀ (fp16 / bf16 pairs) into one of two TMEM buffers, the A operand of
// the TS-form MMA  dV += Pᵀ dO, and dS into one of two swizzled shared-memory
// tiles [key][query], read as the K-major A operand of  dK += dSᵀ Q  and as the
// MN-major A operand of  dQ_it += dS K  (dQ tiles stay in TMEM across key
// tiles).  Both buffers are double, so the compute warps form step u+1 while
// the gradient MMAs of step u run; S and dP of step u+1 are computed while the
// compute warps work on step u.  Finished dK, dV and dQ tiles leave through
// shared memory by TMA tile stores, one step after their last MMA.  The pair
// bias is read from a transposed copy [B,H,L,L'] (L' = L rounded up to 8) that
// the delta kernel writes, so each thread reads its key's row.
//
// TMEM columns: Sᵀ 0..127, dPᵀ 128..255, Pᵀ buffers 256..319 and 320..383
// (packed pairs), then dK, dV (one or two buffers) and the QT dQ tiles.
#include "evo_bwd_common.cuh"

namespace evo {
namespace {

constexpr int kKmMaxQS = 4;
constexpr uint32_t kKmS = 0u, kKmDP = 128u, kKmP = 256u, kKmAcc = 384u;
__device__ __forceinline__ uint32_t km_col_p(uint32_t b) { return kKmP + b * 64u; }

__host__ __device__ constexpr bool km_tmem_fits(int DP, int QT) { return 384 + 2 * DP + QT * DP <= 512; }
__host__ __device__ constexpr int km_kv_bufs(int DP, int QT) { return 384 + 4 * DP + QT * DP <= 512 ? 2 : 1; }
// Streamed dQ (long L): two dQ tile buffers instead of one per query tile.
__host__ __device__ constexpr bool km_stream_fits(int DP) { return 384 + 2 * DP + 2 * DP <= 512; }
__host__ __device__ constexpr int km_stream_kv_bufs(int DP) { return 384 + 4 * DP + 2 * DP <= 512 ? 2 : 1; }
__host__ __device__ constexpr int km_nb(int DP, int QT, bool dqs) { return dqs ? km_stream_kv_bufs(DP) : km_kv_bufs(DP, QT); }
template <int DP>
__device__ __forceinline__ uint32_t km_col_dk(uint32_t b) { return kKmAcc + b * 2 * DP; }
template <int DP>
__device__ __forceinline__ uint32_t km_col_dv(uint32_t b) { return kKmAcc + b * 2 * DP + DP; }
template <int DP>
__device__ __forceinline__ uint32_t km_col_dq(int it, int nb) { return kKmAcc + nb * 2 * DP + it * DP; }
// streamed dQ: the tile of step u in buffer u & 1
template <int DP>
__device__ __forceinline__ uint32_t km_col_dqs(uint32_t b, int nb) { return kKmAcc + nb * 2 * DP + b * DP; }

struct KmBars {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t q_full[kKmMaxQS], q_empty[kKmMaxQS];
  uint64_t st_full, st_free, pds_full, buf_free[2];
  uint64_t dkdv_full[2], dkdv_free[2], dq_full, dq_free;
  uint64_t dqb_full[2], dqb_free[2];  // streamed dQ: per tile buffer
  uint64_t sd_full[2], sd_free[2];  // key-mask gradient pass: Sᵀ / dPᵀ double buffer
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

template <int DP>
struct KmLayout {
  static constexpr uint32_t kTB = kTile * DP * 2;
  Ring ds, stg, b2t, k, v, q, d_o, b1, ld, dqs;
  uint32_t bars, total;
  // grads: the full backward (dS tiles and output staging); without, the key-mask
  // gradient pass that only recomputes dS.  dq_stream: staging of the streamed dQ
  // blocks (one per compute warp).
  __host__ __device__ KmLayout(bool has_b2, int qs, bool grads = true, bool dq_stream = false) {
    uint32_t off = 0;
    ds = Ring{off, 32768u};  // 128B-swizzled tiles first (1024-byte aligned)
    if (grads) off += 2 * 32768u;
    stg = Ring{off, kTB};    // staging of finished dK / dV / dQ: per warp two [32][DP/2] blocks
    if (grads) off += 2 * kTB;
    b2t = Ring{off, 32768u};
    if (has_b2) off += qs * 32768u;
    k = Ring{off, 2 * kTB};
    v = Ring{off + kTB, 2 * kTB};
    off += 4 * kTB;
    q = Ring{off, 2 * kTB};
    d_o = Ring{off + kTB, 2 * kTB};
    off += qs * 2 * kTB;
    b1 = Ring{off, 512u};
    off += 1024u;
    ld = Ring{off, 1024u};
    off += qs * 1024u;
    dqs = Ring{off, DqScr<DP>::kStg};
    if (dq_stream) off += kComputeWarps * DqScr<DP>::kStg;
    bars = off;
    off += (sizeof(KmBars) + 127) & ~127u;
    total = off;
  }
};

// −lse·log2e (−inf for rows past L or with an empty softmax, so P = 0) and
// −delta for the 128 queries of a step: the per-column terms of the exponent
// and of dS.
__device__ __forceinline__ void ld_store_neg(float* dst, const LdRaw& raw, int lane) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x = raw.l[e];
    dst[lane * 4 + e] = (x == -INFINITY) ? -INFINITY : -x * kLog2e;
    dst[128 + lane * 4 + e] = -raw.d[e];
  }
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void km_producer(const BwdArgs& a, uint8_t* base, const KmLayout<DP>& lay, KmBars* bars,
                                            const WaitGuard& g, int lane, long long i0, long long i1) {
  constexpr uint32_t kTB = KmLayout<DP>::kTB;
  const int QS = a.q_stages, QT = a.QT;
  const uint32_t q_bytes = 2 * kTB + (HAS_B2 ? 32768u : 0u);
  uint32_t grp = 0, steps = 0, s = 0, ph = 0;
  SlIter c;
  c.init(i0, a);
  SlIter pc = c;  // lse / delta of the next step and the mask of the next key tile, loaded one step ahead
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
  // L2 prefetch of the Q / dO / pair-bias tiles kPfAhead steps ahead of the load being issued
  constexpr int kPfAhead = 2;
  SlIter fc = c;
  int fjt = 0, fit = 0;
  auto advance_l2 = [&]() {
    if (++fit == QT) {
      fit = 0;
      if (++fjt == QT) {
        fjt = 0;
        fc.next(a);
      }
    }
  };
  auto prefetch_l2 = [&]() {
    if (lane == 0 && fc.b < a.B) {
      const int fbn = fc.b * a.N + fc.n;
      tma_prefetch_4d(&a.tq, 0, fc.h, fit * kTile, fbn);
      tma_prefetch_4d(&a.tdo, 0, fc.h, fit * kTile, fbn);
      if (HAS_B2) {
        const int fbh = fc.b * a.H + fc.h;
        tma_prefetch_3d(&a.tb2t, fit * kTile, fjt * kTile, fbh);
        tma_prefetch_3d(&a.tb2t, fit * kTile + 64, fjt * kTile, fbh);
      }
    }
  };
  for (int k = 0; k < kPfAhead; ++k) {
    advance_l2();
    prefetch_l2();
  }
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
        const int njt = jt + 1 < QT ? jt + 1 : 0;
        SlIter nc = c;
        if (njt == 0) nc.next(a);
        if (lane == 0 && nc.b < a.B) {  // next key tile's K and V into L2
          tma_prefetch_4d(&a.tk, 0, nc.h, njt * kTile, nc.b * a.N + nc.n);
          tma_prefetch_4d(&a.tv, 0, nc.h, njt * kTile, nc.b * a.N + nc.n);
        }
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
          if (HAS_B2) {  // transposed pair bias: rows = keys of tile jt, columns = queries of tile it
            tma_load_3d(smem_u32(base + lay.b2t[s]), &a.tb2t, full, it * kTile, jt * kTile, bh);
            tma_load_3d(smem_u32(base + lay.b2t[s] + 16384), &a.tb2t, full, it * kTile + 64, jt * kTile, bh);
          }
        }
        ld_store_neg(reinterpret_cast<float*>(base + lay.ld[s]), ldr, lane);
        mbar_arrive(full);
        advance_pf();
        prefetch_ld();
        advance_l2();
        prefetch_l2();
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

struct KmStep {
  uint32_t u, grp, slice;
  int jt, it;
  uint32_t qs, qph;
};

// Sᵀ = K Qᵀ and dPᵀ = V dOᵀ of one step into TMEM.
template <int DP, bool BF16>
__device__ __forceinline__ bool km_issue_sdp(const KmStep& st, uint8_t* base, const KmLayout<DP>& lay, KmBars* bars,
                                             uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
  const uint32_t kb = st.grp & 1;
  if (st.it == 0 && !mbar_wait(smem_u32(&bars->kv_full[kb]), (st.grp >> 1) & 1, g)) return false;
  if (!mbar_wait(smem_u32(&bars->q_full[st.qs]), st.qph, g)) return false;
  if (!mbar_wait(smem_u32(&bars->st_free), (st.u & 1) ^ 1, g)) return false;
  tc_fence_after();
  // descriptors: start-address field (bits 0-13, 16-byte units) advanced by constants
  const uint64_t kd = smem_desc(smem_u32(base + lay.k[kb]), 16, 8 * RB, SWZ);
  const uint64_t vd = smem_desc(smem_u32(base + lay.v[kb]), 16, 8 * RB, SWZ);
  const uint64_t qd = smem_desc(smem_u32(base + lay.q[st.qs]), 16, 8 * RB, SWZ);
  const uint64_t dod = smem_desc(smem_u32(base + lay.d_o[st.qs]), 16, 8 * RB, SWZ);
#pragma unroll
  for (int k = 0; k < DP / 16; ++k) umma_ss(tmem + kKmS, kd + k * 2, qd + k * 2, id_s, k > 0);
#pragma unroll
  for (int k = 0; k < DP / 16; ++k) umma_ss(tmem + kKmDP, vd + k * 2, dod + k * 2, id_s, k > 0);
  umma_commit(smem_u32(&bars->st_full));
  return true;
}

// dV += Pᵀ dO (A = Pᵀ in TMEM), dK += dSᵀ Q (A = the dS tile, K-major), then
// dQ_it += dS K (A = the same tile, MN-major).
template <int DP, bool BF16, bool DQS>
__device__ __forceinline__ bool km_issue_grads(const KmStep& st, int QT, uint8_t* base, const KmLayout<DP>& lay,
                                               KmBars* bars, uint32_t tmem, const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_v = idesc_f16(128, DP, BF16, false, true);   // A from TMEM, MN-major B
  constexpr uint32_t id_k = idesc_f16(128, DP, BF16, false, true);   // K-major A (smem), MN-major B
  constexpr uint32_t id_q = idesc_f16(128, DP, BF16, true, true);    // MN-major A, MN-major B
  const uint32_t kb = st.grp & 1;
  const int nb = km_nb(DP, QT, DQS);
  const uint32_t db = st.grp % nb, dph = (st.grp / nb) & 1;
  const uint32_t b = st.u & 1;
  if (!mbar_wait(smem_u32(&bars->pds_full), st.u & 1, g)) return false;
  if (st.it == 0 && !mbar_wait(smem_u32(&bars->dkdv_free[db]), dph ^ 1, g)) return false;
  tc_fence_after();
  // descriptors: start-address field (bits 0-13, 16-byte units) advanced by constants
  const uint64_t dod = smem_desc(smem_u32(base + lay.d_o[st.qs]), kTile * RB, 8 * RB, SWZ);
  const uint64_t qd = smem_desc(smem_u32(base + lay.q[st.qs]), kTile * RB, 8 * RB, SWZ);
  const uint64_t kd = smem_desc(smem_u32(base + lay.k[kb]), kTile * RB, 8 * RB, SWZ);
  const uint32_t ds_addr = smem_u32(base + lay.ds[b]);
  const uint64_t dskd = smem_desc(ds_addr, 16, 1024, kSwizzle128B);         // dSᵀ as K-major A
  const uint64_t dsmd = smem_desc(ds_addr, 16384, 1024, kSwizzle128B);      // dS as MN-major A
  const uint32_t pcol = tmem + km_col_p(b);
  const uint32_t acc_v = (st.it > 0) ? 1u : 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k)  // dV += Pᵀ dO   (K = 128 queries)
    umma_ts(tmem + km_col_dv<DP>(db), pcol + k * 8, dod + k * RB, id_v, (acc_v | k) ? 1u : 0u);
#pragma unroll
  for (int k = 0; k < 8; ++k)  // dK += dSᵀ Q
    umma_ss(tmem + km_col_dk<DP>(db), dskd + (k >> 2) * 1024 + (k & 3) * 2, qd + k * RB, id_k,
            (acc_v | k) ? 1u : 0u);
  umma_commit(smem_u32(&bars->q_empty[st.qs]));
  if (st.it == QT - 1) umma_commit(smem_u32(&bars->dkdv_full[db]));
  if (DQS) {  // this step's dQ tile, into the buffer its consumer has emptied
    if (!mbar_wait(smem_u32(&bars->dqb_free[b]), ((st.u >> 1) & 1) ^ 1, g)) return false;
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < 8; ++k)  // dQ tile = dS K_jt   (K = 128 keys)
      umma_ss(tmem + km_col_dqs<DP>(b, nb), dsmd + k * 128, kd + k * RB, id_q, k > 0 ? 1u : 0u);
    umma_commit(smem_u32(&bars->dqb_full[b]));
    umma_commit(smem_u32(&bars->buf_free[b]));
    if (st.it == QT - 1) umma_commit(smem_u32(&bars->kv_empty[kb]));
    return true;
  }
  if (st.it == 0 && st.jt == 0 && !mbar_wait(smem_u32(&bars->dq_free), (st.slice & 1) ^ 1, g)) return false;
  tc_fence_after();
  const uint32_t acc_q = (st.jt > 0) ? 1u : 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k)  // dQ_it += dS K_jt   (K = 128 keys)
    umma_ss(tmem + km_col_dq<DP>(st.it, nb), dsmd + k * 128, kd + k * RB, id_q, (acc_q | k) ? 1u : 0u);
  umma_commit(smem_u32(&bars->buf_free[b]));
  if (st.it == QT - 1) {
    umma_commit(smem_u32(&bars->kv_empty[kb]));
    if (st.jt == QT - 1) umma_commit(smem_u32(&bars->dq_full));
  }
  return true;
}

template <int DP, bool BF16, bool DQS>
__device__ __forceinline__ void km_mma(const BwdArgs& a, uint8_t* base, const KmLayout<DP>& lay, KmBars* bars,
                                       uint32_t tmem, const WaitGuard& g, long long i0, long long i1) {
  const int QS = a.q_stages, QT = a.QT;
  const uint32_t total = static_cast<uint32_t>((i1 - i0) * QT * QT);
  auto advance = [&](KmStep& st) {
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
  // S/dP of step u+1 are issued before the gradients of step u (needs two Q/dO stages)
  bool ok = total > 0;
  KmStep cur{0, 0, 0, 0, 0, 0, 0};
  if (ok) ok = km_issue_sdp<DP, BF16>(cur, base, lay, bars, tmem, g);
  for (uint32_t u = 0; ok && u < total; ++u) {
    KmStep nxt = cur;
    advance(nxt);
    if (u + 1 < total && !km_issue_sdp<DP, BF16>(nxt, base, lay, bars, tmem, g)) break;
    if (!km_issue_grads<DP, BF16, DQS>(cur, QT, base, lay, bars, tmem, g)) break;
    cur = nxt;
  }
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

// Pᵀ for 32 queries of this thread's key into TMEM (packed pairs) and dS into
// the swizzled smem tile.  nl / nd: −lse·log2e and −delta of the 32 queries.
// DB1: also add this thread's dS values into dsum (the key's share of the key-mask gradient).
template <bool BF16, bool HAS_B2, bool DB1>
__device__ __forceinline__ void km_chunk(const uint32_t (&sv)[32], const uint32_t (&pv)[32], float b1j,
                                         const float* nl, const float* nd, const uint8_t* b2half, uint8_t* dshalf,
                                         uint32_t p_tcol, int r, int c, float2 sl2, float2& dsum) {
  const float2 mk = make_float2(b1j, b1j), l2e2 = make_float2(kLog2e, kLog2e);
  uint32_t pp[16], dd[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 l0 = *reinterpret_cast<const float4*>(nl + q * 8);
    const float4 l1 = *reinterpret_cast<const float4*>(nl + q * 8 + 4);
    const float4 d0 = *reinterpret_cast<const float4*>(nd + q * 8);
    const float4 d1 = *reinterpret_cast<const float4*>(nd + q * 8 + 4);
    const float2 nl2[4] = {make_float2(l0.x, l0.y), make_float2(l0.z, l0.w), make_float2(l1.x, l1.y),
                           make_float2(l1.z, l1.w)};
    const float2 nd2[4] = {make_float2(d0.x, d0.y), make_float2(d0.z, d0.w), make_float2(d1.x, d1.y),
                           make_float2(d1.z, d1.w)};
    uint4 pb = make_uint4(0u, 0u, 0u, 0u);
    if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2half + swz_offset(r, c * 4 + q, 128));
    const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int x = q * 8 + e2 * 2;
      float2 t = fma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, mk);
      if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
      t = add2(t, nl2[e2]);
      const float p0 = ex2(t.x), p1 = ex2(t.y);
      const float2 dpd = add2(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), nd2[e2]);
      const float2 ds = mul2(make_float2(p0, p1), dpd);
      if (DB1) dsum = add2(dsum, ds);
      pp[q * 4 + e2] = pack2<BF16>(p0, p1);
      dd[q * 4 + e2] = pack2<BF16>(ds.x, ds.y);
    }
    *reinterpret_cast<uint4*>(dshalf + swz_offset(r, c * 4 + q, 128)) =
        make_uint4(dd[q * 4], dd[q * 4 + 1], dd[q * 4 + 2], dd[q * 4 + 3]);
  }
  tmem_st16(p_tcol, pp);
}

// The same for one 16-query chunk k (0..3) of this warp's 64 queries: Pᵀ pairs into
// pp[0..7], dSᵀ into the smem tile.
template <bool BF16, bool HAS_B2, bool DB1>
__device__ __forceinline__ void km_chunk16(const uint32_t (&sv)[16], const uint32_t (&pv)[16], float b1j,
                                           const float* nl, const float* nd, const uint8_t* b2half, uint8_t* dshalf,
                                           uint32_t* pp, int r, int k, float2 sl2, float2& dsum) {
  const float2 mk = make_float2(b1j, b1j), l2e2 = make_float2(kLog2e, kLog2e);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float4 l0 = *reinterpret_cast<const float4*>(nl + k * 16 + q * 8);
    const float4 l1 = *reinterpret_cast<const float4*>(nl + k * 16 + q * 8 + 4);
    const float4 d0 = *reinterpret_cast<const float4*>(nd + k * 16 + q * 8);
    const float4 d1 = *reinterpret_cast<const float4*>(nd + k * 16 + q * 8 + 4);
    const float2 nl2[4] = {make_float2(l0.x, l0.y), make_float2(l0.z, l0.w), make_float2(l1.x, l1.y),
                           make_float2(l1.z, l1.w)};
    const float2 nd2[4] = {make_float2(d0.x, d0.y), make_float2(d0.z, d0.w), make_float2(d1.x, d1.y),
                           make_float2(d1.z, d1.w)};
    const uint32_t off = swz_offset(r, k * 2 + q, 128);
    uint4 pb = make_uint4(0u, 0u, 0u, 0u);
    if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2half + off);
    const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
    uint32_t dd[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int x = q * 8 + e2 * 2;
      float2 t = fma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, mk);
      if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
      t = add2(t, nl2[e2]);
      const float p0 = ex2(t.x), p1 = ex2(t.y);
      const float2 dpd = add2(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), nd2[e2]);
      const float2 ds = mul2(make_float2(p0, p1), dpd);
      if (DB1) dsum = add2(dsum, ds);
      pp[q * 4 + e2] = pack2<BF16>(p0, p1);
      dd[e2] = pack2<BF16>(ds.x, ds.y);
    }
    *reinterpret_cast<uint4*>(dshalf + off) = make_uint4(dd[0], dd[1], dd[2], dd[3]);
  }
}

// HD fp32 TMEM columns of this thread's lane into v.
template <int HD>
__device__ __forceinline__ void km_load_cols(uint32_t col, float (&v)[HD]) {
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
}

// Each compute warp writes its own share of a finished tile — its 32 rows
// (TMEM lanes) × DP/2 columns — through a private staging block and one TMA
// store issued by its lane 0, so write-outs need no synchronisation between
// warps.  Block t of warp w: [32][DP/2] fp16/bf16, 32-byte swizzle when the
// rows are 32 bytes (the layout of the output maps' boxes).
template <int DP>
__device__ __forceinline__ uint8_t* km_stage_block(uint8_t* base, const KmLayout<DP>& lay, int w, int t) {
  return base + lay.stg[0] + (w * 2 + t) * (32 * DP);
}

template <int DP, int HD, bool BF16>
__device__ __forceinline__ void km_stage_row(uint8_t* blk, const float (&v)[HD], float mul, int lane) {
#pragma unroll
  for (int e = 0; e < HD; e += 8) {
    uint4 pk;
    pk.x = pack2<BF16>(v[e + 0] * mul, v[e + 1] * mul);
    pk.y = pack2<BF16>(v[e + 2] * mul, v[e + 3] * mul);
    pk.z = pack2<BF16>(v[e + 4] * mul, v[e + 5] * mul);
    pk.w = pack2<BF16>(v[e + 6] * mul, v[e + 7] * mul);
    const uint32_t off = HD == 16 ? swz_offset(lane, e >> 3, 32) : lane * 16u;
    *reinterpret_cast<uint4*>(blk + off) = pk;
  }
}

// Before writing the warp's staging blocks: its previous stores have read them.
__device__ __forceinline__ void km_stage_open(int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
}
__device__ __forceinline__ void km_stage_close() {
  fence_proxy_async_smem();
  __syncwarp();
}

// dK (× s) and dV of key tile jt of slice c.
template <int DP, bool BF16, bool DQS>
__device__ __forceinline__ bool km_write_dkdv(const BwdArgs& a, const SlIter& c, int jt, uint32_t grp, uint8_t* base,
                                              const KmLayout<DP>& lay, KmBars* bars, uint32_t trow, int w, int hc,
                                              int lane, const WaitGuard& g) {
  constexpr int HD = DP / 2;
  const int nb = km_nb(DP, a.QT, DQS);
  const uint32_t db = grp % nb;
  if (!mbar_wait_warp(smem_u32(&bars->dkdv_full[db]), (grp / nb) & 1, g)) return false;
  tc_fence_after();
  float kx[HD], vx[HD];
  km_load_cols<HD>(trow + km_col_dk<DP>(db) + hc * HD, kx);
  km_load_cols<HD>(trow + km_col_dv<DP>(db) + hc * HD, vx);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->dkdv_free[db]));
  uint8_t* bk = km_stage_block<DP>(base, lay, w, 0);
  uint8_t* bv = km_stage_block<DP>(base, lay, w, 1);
  km_stage_open(lane);
  km_stage_row<DP, HD, BF16>(bk, kx, a.scale, lane);
  km_stage_row<DP, HD, BF16>(bv, vx, 1.0f, lane);
  km_stage_close();
  if (lane == 0) {
    const int bn = c.b * a.N + c.n, row = jt * kTile + (w & 3) * 32;
    tma_store_4d(&a.tdk, smem_u32(bk), hc * HD, c.h, row, bn);
    tma_store_4d(&a.tdv, smem_u32(bv), hc * HD, c.h, row, bn);
    bulk_commit_group();
  }
  return true;
}

// dQ (× s) of slice c: every query tile, two per round through the staging blocks.
template <int DP, bool BF16>
__device__ __forceinline__ bool km_write_dq(const BwdArgs& a, const SlIter& c, uint32_t slice, uint8_t* base,
                                            const KmLayout<DP>& lay, KmBars* bars, uint32_t trow, int w, int hc,
                                            int lane, const WaitGuard& g) {
  constexpr int HD = DP / 2;
  if (!mbar_wait_warp(smem_u32(&bars->dq_full), slice & 1, g)) return false;
  tc_fence_after();
  const int nb = km_kv_bufs(DP, a.QT);
  const int bn = c.b * a.N + c.n;
  for (int it0 = 0; it0 < a.QT; it0 += 2) {
    const bool two = it0 + 1 < a.QT;
    float v0[HD], v1[HD];
    km_load_cols<HD>(trow + km_col_dq<DP>(it0, nb) + hc * HD, v0);
    if (two) km_load_cols<HD>(trow + km_col_dq<DP>(it0 + 1, nb) + hc * HD, v1);
    if (it0 + 2 >= a.QT) {  // every dQ column read: the next slice may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
    }
    uint8_t* b0 = km_stage_block<DP>(base, lay, w, 0);
    uint8_t* b1 = km_stage_block<DP>(base, lay, w, 1);
    km_stage_open(lane);
    km_stage_row<DP, HD, BF16>(b0, v0, a.scale, lane);
    if (two) km_stage_row<DP, HD, BF16>(b1, v1, a.scale, lane);
    km_stage_close();
    if (lane == 0) {
      const int row = (w & 3) * 32;
      tma_store_4d(&a.tdq, smem_u32(b0), hc * HD, c.h, it0 * kTile + row, bn);
      if (two) tma_store_4d(&a.tdq, smem_u32(b1), hc * HD, c.h, (it0 + 1) * kTile + row, bn);
      bulk_commit_group();
    }
  }
  return true;
}

// Key-mask gradient partial of key j of slice c, query half hc: [B·N·H][2][L] fp32.
__device__ __forceinline__ void km_store_db1(const BwdArgs& a, const SlIter& c, int hc, int j, float v) {
  if (j < a.L)
    a.db1p[((static_cast<size_t>(c.b * a.N + c.n) * a.H + c.h) * 2 + hc) * a.L + j] = v;
}

template <int DP, bool BF16, bool HAS_B2, bool DB1, bool DQS>
__device__ __forceinline__ void km_compute(const BwdArgs& a, uint8_t* base, const KmLayout<DP>& lay, KmBars* bars,
                                           uint32_t tmem, const WaitGuard& g, long long i0, long long i1) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = w & 3, hc = w >> 2;
  const int r = quad * 32 + lane;  // key row of the tile (TMEM lane)
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int QS = a.q_stages, QT = a.QT;
  uint32_t u = 0, grp = 0, slice = 0, s = 0, ph = 0;
  SlIter cur, prev;
  cur.init(i0, a);
  prev = cur;
  float b1j = 0.0f;
  float2 dsum = make_float2(0.0f, 0.0f);  // DB1: Σ over the key tile's queries of this key's dS
  // DQS: the previous step's dQ tile is consumed one step late (its MMAs are done by then)
  const int nbq = km_nb(DP, QT, DQS);
  uint8_t* dq_stg = base + lay.dqs[w];
  DqStep pd{0, 0, 0, 0, false, false};
  auto consume = [&](uint32_t v) {
    const uint32_t qb = v & 1;
    return consume_dq_tile<DP, BF16>(a, pd, smem_u32(&bars->dqb_full[qb]), smem_u32(&bars->dqb_free[qb]),
                                     (v >> 1) & 1, trow + km_col_dqs<DP>(qb, nbq) + hc * (DP / 2), r, w, hc, lane,
                                     dq_stg, g);
  };
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, ++slice) {
    if (item > i0) {
      prev = cur;
      cur.next(a);
    }
    for (int jt = 0; ok && jt < QT; ++jt, ++grp) {
      const uint32_t kb = grp & 1;
      for (int it = 0; it < QT; ++it, ++u) {
        if (it == 0) {
          if (!mbar_wait_warp(smem_u32(&bars->kv_full[kb]), (grp >> 1) & 1, g)) { ok = false; break; }
          b1j = reinterpret_cast<const float*>(base + lay.b1[kb])[r];
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->kv_empty[kb]));
        }
        if (!mbar_wait_warp(smem_u32(&bars->q_full[s]), ph, g)) { ok = false; break; }
        if (!mbar_wait_warp(smem_u32(&bars->st_full), u & 1, g)) { ok = false; break; }
        if (!mbar_wait_warp(smem_u32(&bars->buf_free[u & 1]), ((u >> 1) & 1) ^ 1, g)) { ok = false; break; }
        tc_fence_after();
        const float* ld = reinterpret_cast<const float*>(base + lay.ld[s]) + hc * 64;
        const uint8_t* b2half = base + lay.b2t[s] + hc * 16384;
        uint8_t* dshalf = base + lay.ds[u & 1] + hc * 16384;
        const uint32_t pcol = trow + km_col_p(u & 1) + hc * 32;
        {
          // 16-query chunks of Sᵀ and dPᵀ: chunk k+1's TMEM loads are in flight while chunk
          // k is computed (one pair outstanding, so each wait covers the chunk about to be
          // used); Pᵀ pairs go to TMEM two chunks at a time
          const uint32_t cs = trow + kKmS + hc * 64, cpd = trow + kKmDP + hc * 64;
          const float* nl = ld;
          const float* nd = ld + 128;
          uint32_t s0[16], p0[16], s1[16], p1[16], pp[16];
          tmem_ld16(cs, s0);
          tmem_ld16(cpd, p0);
          tmem_wait_ld(s0);
          tmem_wait_ld(p0);
          tmem_ld16(cs + 16, s1);
          tmem_ld16(cpd + 16, p1);
          km_chunk16<BF16, HAS_B2, DB1>(s0, p0, b1j, nl, nd, b2half, dshalf, pp, r, 0, sl2, dsum);
          tmem_wait_ld(s1);
          tmem_wait_ld(p1);
          tmem_ld16(cs + 32, s0);
          tmem_ld16(cpd + 32, p0);
          km_chunk16<BF16, HAS_B2, DB1>(s1, p1, b1j, nl, nd, b2half, dshalf, pp + 8, r, 1, sl2, dsum);
          tmem_st16(pcol, pp);
          tmem_wait_ld(s0);
          tmem_wait_ld(p0);
          tmem_ld16(cs + 48, s1);
          tmem_ld16(cpd + 48, p1);
          km_chunk16<BF16, HAS_B2, DB1>(s0, p0, b1j, nl, nd, b2half, dshalf, pp, r, 2, sl2, dsum);
          tmem_wait_ld(s1);
          tmem_wait_ld(p1);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->st_free));
          km_chunk16<BF16, HAS_B2, DB1>(s1, p1, b1j, nl, nd, b2half, dshalf, pp + 8, r, 3, sl2, dsum);
          tmem_st16(pcol + 16, pp);
        }
        tmem_wait_st();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bars->pds_full));
          mbar_arrive(smem_u32(&bars->q_empty[s]));
        }
        if (++s == static_cast<uint32_t>(QS)) {
          s = 0;
          ph ^= 1;
        }
        if (DQS) {
          if (u > 0 && !consume(u - 1)) { ok = false; break; }
          pd = DqStep{cur.b, cur.n, cur.h, it, jt == 0, jt == QT - 1};
        }
        if (DB1 && it == QT - 1) {  // this key's share over the slice's queries, per query half
          km_store_db1(a, cur, hc, jt * kTile + r, dsum.x + dsum.y);
          dsum = make_float2(0.0f, 0.0f);
        }
        // one step late (their MMAs are done by now): dK/dV of the previous key tile and,
        // at a slice boundary, the previous slice's dQ
        if (it == 0 && grp > 0 &&
            !km_write_dkdv<DP, BF16, DQS>(a, jt > 0 ? cur : prev, jt > 0 ? jt - 1 : QT - 1, grp - 1, base, lay,
                                          bars, trow, w, hc, lane, g)) {
          ok = false;
          break;
        }
        if (!DQS && it == 0 && jt == 0 && slice > 0 &&
            !km_write_dq<DP, BF16>(a, prev, slice - 1, base, lay, bars, trow, w, hc, lane, g)) {
          ok = false;
          break;
        }
      }
    }
  }
  if (ok && grp > 0) {
    if (DQS) {
      if (consume(u - 1)) km_write_dkdv<DP, BF16, DQS>(a, cur, QT - 1, grp - 1, base, lay, bars, trow, w, hc, lane, g);
    } else if (km_write_dkdv<DP, BF16, DQS>(a, cur, QT - 1, grp - 1, base, lay, bars, trow, w, hc, lane, g)) {
      km_write_dq<DP, BF16>(a, cur, slice - 1, base, lay, bars, trow, w, hc, lane, g);
    }
  }
  if (lane == 0) bulk_wait_all();  // this warp's tile stores complete before the CTA's smem goes away
}

template <int DP, bool BF16, bool HAS_B2, bool DB1, bool DQS>
__global__ void __launch_bounds__(kThreads, 1) evo_bwd_kmajor(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KmLayout<DP> lay(HAS_B2, a.q_stages, true, DQS);
  KmBars* bars = reinterpret_cast<KmBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long i0 = static_cast<long long>(blockIdx.x) * a.chunk;
  const long long i1 = i0 + a.chunk < a.items ? i0 + a.chunk : a.items;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1 + kComputeWarps);
      mbar_init(smem_u32(&bars->buf_free[s]), 1);
      mbar_init(smem_u32(&bars->dkdv_full[s]), 1);
      mbar_init(smem_u32(&bars->dkdv_free[s]), kComputeWarps);
      mbar_init(smem_u32(&bars->dqb_full[s]), 1);
      mbar_init(smem_u32(&bars->dqb_free[s]), kComputeWarps);
    }
    for (int s = 0; s < kKmMaxQS; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 32);
      mbar_init(smem_u32(&bars->q_empty[s]), 1 + kComputeWarps);
    }
    mbar_init(smem_u32(&bars->st_full), 1);
    mbar_init(smem_u32(&bars->st_free), kComputeWarps);
    mbar_init(smem_u32(&bars->pds_full), kComputeWarps);
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
    if (HAS_B2) tma_prefetch_desc(&a.tb2t);
    tma_prefetch_desc(&a.tdq);
    tma_prefetch_desc(&a.tdk);
    tma_prefetch_desc(&a.tdv);
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
    km_producer<DP, BF16, HAS_B2>(a, base, lay, bars, g, lane, i0, i1);
  } else if (warp == kMmaWarp) {
    if (lane == 0) km_mma<DP, BF16, DQS>(a, base, lay, bars, tmem, g, i0, i1);
    __syncwarp();
  } else {
    km_compute<DP, BF16, HAS_B2, DB1, DQS>(a, base, lay, bars, tmem, g, i0, i1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ key-mask gradient pass
// For the schedules whose main kernel does not produce the key-mask gradient:
// the key-major score recompute alone (Sᵀ, dPᵀ double-buffered in TMEM), each
// thread summing its key's dS over the slice's queries; same producer, same
// partial layout as the key-major kernel with DB1.

template <bool BF16, bool HAS_B2>
__device__ __forceinline__ void km_chunk_sum(const uint32_t (&sv)[32], const uint32_t (&pv)[32], float b1j,
                                             const float* nl, const float* nd, const uint8_t* b2half, int r, int c,
                                             float2 sl2, float2& dsum) {
  const float2 mk = make_float2(b1j, b1j), l2e2 = make_float2(kLog2e, kLog2e);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 l0 = *reinterpret_cast<const float4*>(nl + q * 8);
    const float4 l1 = *reinterpret_cast<const float4*>(nl + q * 8 + 4);
    const float4 d0 = *reinterpret_cast<const float4*>(nd + q * 8);
    const float4 d1 = *reinterpret_cast<const float4*>(nd + q * 8 + 4);
    const float2 nl2[4] = {make_float2(l0.x, l0.y), make_float2(l0.z, l0.w), make_float2(l1.x, l1.y),
                           make_float2(l1.z, l1.w)};
    const float2 nd2[4] = {make_float2(d0.x, d0.y), make_float2(d0.z, d0.w), make_float2(d1.x, d1.y),
                           make_float2(d1.z, d1.w)};
    uint4 pb = make_uint4(0u, 0u, 0u, 0u);
    if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2half + swz_offset(r, c * 4 + q, 128));
    const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int x = q * 8 + e2 * 2;
      float2 t = fma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, mk);
      if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
      t = add2(t, nl2[e2]);
      const float2 dpd = add2(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), nd2[e2]);
      dsum = fma2(make_float2(ex2(t.x), ex2(t.y)), dpd, dsum);
    }
  }
}

template <int DP, bool BF16>
__device__ __forceinline__ void km_db1_mma(const BwdArgs& a, uint8_t* base, const KmLayout<DP>& lay, KmBars* bars,
                                           uint32_t tmem, const WaitGuard& g, long long i0, long long i1) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
  const int QS = a.q_stages, QT = a.QT;
  uint32_t u = 0, grp = 0, qs = 0, qph = 0;
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item) {
    for (int jt = 0; ok && jt < QT; ++jt, ++grp) {
      const uint32_t kb = grp & 1;
      for (int it = 0; it < QT; ++it, ++u) {
        const uint32_t b = u & 1;
        if (it == 0 && !mbar_wait(smem_u32(&bars->kv_full[kb]), (grp >> 1) & 1, g)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&bars->q_full[qs]), qph, g)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&bars->sd_free[b]), ((u >> 1) & 1) ^ 1, g)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kd = smem_desc(smem_u32(base + lay.k[kb]), 16, 8 * RB, SWZ);
        const uint64_t vd = smem_desc(smem_u32(base + lay.v[kb]), 16, 8 * RB, SWZ);
        const uint64_t qd = smem_desc(smem_u32(base + lay.q[qs]), 16, 8 * RB, SWZ);
        const uint64_t dod = smem_desc(smem_u32(base + lay.d_o[qs]), 16, 8 * RB, SWZ);
#pragma unroll
        for (int k = 0; k < DP / 16; ++k) umma_ss(tmem + b * 256u, kd + k * 2, qd + k * 2, id_s, k > 0);
#pragma unroll
        for (int k = 0; k < DP / 16; ++k) umma_ss(tmem + b * 256u + 128u, vd + k * 2, dod + k * 2, id_s, k > 0);
        umma_commit(smem_u32(&bars->sd_full[b]));
        umma_commit(smem_u32(&bars->q_empty[qs]));
        if (it == QT - 1) umma_commit(smem_u32(&bars->kv_empty[kb]));
        if (++qs == static_cast<uint32_t>(QS)) {
          qs = 0;
          qph ^= 1;
        }
      }
    }
  }
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

template <int DP, bool BF16, bool HAS_B2>
__device__ __forceinline__ void km_db1_compute(const BwdArgs& a, uint8_t* base, const KmLayout<DP>& lay,
                                               KmBars* bars, uint32_t tmem, const WaitGuard& g, long long i0,
                                               long long i1) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = w & 3, hc = w >> 2;
  const int r = quad * 32 + lane;
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int QS = a.q_stages, QT = a.QT;
  uint32_t u = 0, grp = 0, s = 0, ph = 0;
  SlIter cur;
  cur.init(i0, a);
  float b1j = 0.0f;
  float2 dsum = make_float2(0.0f, 0.0f);
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item) {
    if (item > i0) cur.next(a);
    for (int jt = 0; ok && jt < QT; ++jt, ++grp) {
      const uint32_t kb = grp & 1;
      for (int it = 0; it < QT; ++it, ++u) {
        const uint32_t b = u & 1;
        if (it == 0) {
          if (!mbar_wait_warp(smem_u32(&bars->kv_full[kb]), (grp >> 1) & 1, g)) { ok = false; break; }
          b1j = reinterpret_cast<const float*>(base + lay.b1[kb])[r];
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->kv_empty[kb]));
        }
        if (!mbar_wait_warp(smem_u32(&bars->q_full[s]), ph, g)) { ok = false; break; }
        if (!mbar_wait_warp(smem_u32(&bars->sd_full[b]), (u >> 1) & 1, g)) { ok = false; break; }
        tc_fence_after();
        const float* ld = reinterpret_cast<const float*>(base + lay.ld[s]) + hc * 64;
        const uint8_t* b2half = base + lay.b2t[s] + hc * 16384;
        const uint32_t cs = trow + b * 256u + hc * 64, cp = cs + 128u;
        {
          uint32_t sv[32], pv[32];
          tmem_ld32(cs, sv);
          tmem_ld32(cp, pv);
          tmem_wait_ld(sv);
          tmem_wait_ld(pv);
          km_chunk_sum<BF16, HAS_B2>(sv, pv, b1j, ld, ld + 128, b2half, r, 0, sl2, dsum);
        }
        {
          uint32_t sv[32], pv[32];
          tmem_ld32(cs + 32, sv);
          tmem_ld32(cp + 32, pv);
          tmem_wait_ld(sv);
          tmem_wait_ld(pv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->sd_free[b]));
          km_chunk_sum<BF16, HAS_B2>(sv, pv, b1j, ld + 32, ld + 160, b2half, r, 1, sl2, dsum);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->q_empty[s]));
        if (++s == static_cast<uint32_t>(QS)) {
          s = 0;
          ph ^= 1;
        }
        if (it == QT - 1) {
          km_store_db1(a, cur, hc, jt * kTile + r, dsum.x + dsum.y);
          dsum = make_float2(0.0f, 0.0f);
        }
      }
    }
  }
}

template <int DP, bool BF16, bool HAS_B2>
__global__ void __launch_bounds__(kThreads, 1) evo_bwd_db1(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KmLayout<DP> lay(HAS_B2, a.q_stages, false);
  KmBars* bars = reinterpret_cast<KmBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long i0 = static_cast<long long>(blockIdx.x) * a.chunk;
  const long long i1 = i0 + a.chunk < a.items ? i0 + a.chunk : a.items;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1 + kComputeWarps);
      mbar_init(smem_u32(&bars->sd_full[s]), 1);
      mbar_init(smem_u32(&bars->sd_free[s]), kComputeWarps);
    }
    for (int s = 0; s < kKmMaxQS; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 32);
      mbar_init(smem_u32(&bars->q_empty[s]), 1 + kComputeWarps);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    tma_prefetch_desc(&a.tdo);
    if (HAS_B2) tma_prefetch_desc(&a.tb2t);
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
    km_producer<DP, BF16, HAS_B2>(a, base, lay, bars, g, lane, i0, i1);
  } else if (warp == kMmaWarp) {
    if (lane == 0) km_db1_mma<DP, BF16>(a, base, lay, bars, tmem, g, i0, i1);
    __syncwarp();
  } else {
    km_db1_compute<DP, BF16, HAS_B2>(a, base, lay, bars, tmem, g, i0, i1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dbias1[b,n,j] = Σ_h Σ_half partial[b,n,h,half,j] in this fixed order, rounded to the dtype.
template <bool BF16>
__global__ void __launch_bounds__(256) evo_bwd_db1_sum(const BwdArgs a) {
  const long long total = static_cast<long long>(a.B) * a.N * a.L;
  for (long long e = blockIdx.x * 256ll + threadIdx.x; e < total; e += gridDim.x * 256ll) {
    const long long bn = e / a.L;
    const int j = static_cast<int>(e - bn * a.L);
    const float* p = a.db1p + bn * a.H * 2 * a.L + j;
    float sum = 0.0f;
    for (int t = 0; t < 2 * a.H; ++t) sum += p[static_cast<size_t>(t) * a.L];
    a.dbias1[e] = static_cast<uint16_t>(pack2<BF16>(sum, 0.0f) & 0xFFFFu);
  }
}

template <int DP, bool BF16, bool HAS_B2>
cudaError_t launch_db1(BwdArgs a, cudaStream_t st) {
  int qs = 0;
  for (int q = kKmMaxQS; q >= 2 && qs == 0; --q)
    if (KmLayout<DP>(HAS_B2, q, false).total + 1024 <= kMaxSmem) qs = q;
  if (qs == 0) return cudaErrorInvalidValue;
  a.q_stages = qs;
  const KmLayout<DP> lay(HAS_B2, qs, false);
  const size_t smem = one_cta_per_sm(lay.total + 1024);
  auto kern = evo_bwd_db1<DP, BF16, HAS_B2>;
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

template <int DP>
cudaError_t launch_db1_d(const BwdArgs& a, bool bf16, bool has_b2, cudaStream_t st) {
  if (bf16) return has_b2 ? launch_db1<DP, true, true>(a, st) : launch_db1<DP, true, false>(a, st);
  return has_b2 ? launch_db1<DP, false, true>(a, st) : launch_db1<DP, false, false>(a, st);
}

template <int DP>
int km_stages(int QT, bool has_b2) {
  if (!km_tmem_fits(DP, QT)) return 0;
  for (int qs = kKmMaxQS; qs >= 2; --qs)
    if (KmLayout<DP>(has_b2, qs).total + 1024 <= kMaxSmem) return qs;
  return 0;
}
// Streamed dQ: any number of query tiles (their dQ leaves through the workspace each step).
template <int DP>
int km_stream_stages(bool has_b2) {
  if (!km_stream_fits(DP)) return 0;
  for (int qs = kKmMaxQS; qs >= 2; --qs)
    if (KmLayout<DP>(has_b2, qs, true, true).total + 1024 <= kMaxSmem) return qs;
  return 0;
}

template <int DP, bool BF16, bool HAS_B2, bool DB1, bool DQS>
cudaError_t launch_km(BwdArgs a, cudaStream_t st) {
  const KmLayout<DP> lay(HAS_B2, a.q_stages, true, DQS);
  const size_t smem = one_cta_per_sm(lay.total + 1024);
  auto kern = evo_bwd_kmajor<DP, BF16, HAS_B2, DB1, DQS>;
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

template <int DP, bool BF16, bool DQS>
cudaError_t launch_km_b(const BwdArgs& a, bool has_b2, cudaStream_t st) {
  if (a.db1p)
    return has_b2 ? launch_km<DP, BF16, true, true, DQS>(a, st) : launch_km<DP, BF16, false, true, DQS>(a, st);
  return has_b2 ? launch_km<DP, BF16, true, false, DQS>(a, st) : launch_km<DP, BF16, false, false, DQS>(a, st);
}

template <int DP>
cudaError_t launch_km_d(const BwdArgs& a, bool bf16, bool has_b2, bool dqs, cudaStream_t st) {
  if (dqs) return bf16 ? launch_km_b<DP, true, true>(a, has_b2, st) : launch_km_b<DP, false, true>(a, has_b2, st);
  return bf16 ? launch_km_b<DP, true, false>(a, has_b2, st) : launch_km_b<DP, false, false>(a, has_b2, st);
}

}  // namespace

int kmajor_q_stages(int DP, int QT, bool has_b2) {
  switch (DP) {
    case 16: return km_stages<16>(QT, has_b2);
    case 32: return km_stages<32>(QT, has_b2);
    default: return 0;
  }
}
int kmajor_stream_q_stages(int DP, bool has_b2) {
  switch (DP) {
    case 16: return km_stream_stages<16>(has_b2);
    case 32: return km_stream_stages<32>(has_b2);
    default: return 0;
  }
}

cudaError_t launch_bwd_db1_partials(const BwdArgs& a, int DP, bool bf16, bool has_b2, cudaStream_t st) {
  switch (DP) {
    case 16: return launch_db1_d<16>(a, bf16, has_b2, st);
    case 32: return launch_db1_d<32>(a, bf16, has_b2, st);
    case 64: return launch_db1_d<64>(a, bf16, has_b2, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_db1_sum(const BwdArgs& a, bool bf16, cudaStream_t st) {
  const long long total = static_cast<long long>(a.B) * a.N * a.L;
  long long grid = (total + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (grid > cap) grid = cap;
  if (bf16)
    evo_bwd_db1_sum<true><<<static_cast<unsigned>(grid), 256, 0, st>>>(a);
  else
    evo_bwd_db1_sum<false><<<static_cast<unsigned>(grid), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_kmajor(const BwdArgs& a, int DP, bool bf16, bool has_b2, bool dq_stream, cudaStream_t st) {
  switch (DP) {
    case 16: return launch_km_d<16>(a, bf16, has_b2, dq_stream, st);
    case 32: return launch_km_d<32>(a, bf16, has_b2, dq_stream, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace evo
