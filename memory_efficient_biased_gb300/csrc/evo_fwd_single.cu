// evo_fwd_single.cu — the forward on one 128-row query tile per work item, for
// the shapes whose pair of query tiles with streamed pair-bias tiles does not fit
// in shared memory (head dimension above 32 with a pair bias and L > 128); every
// other shape runs the paired kernel of evo_fwd.cu.  sm_103a.
//
// Computes, per (b, n, h) slice, O = softmax(Q Kᵀ D^-1/2 + bias1 + bias2) V
// and the fp32 natural-log row log-sum-exp, never writing the L×L scores to
// device memory.  Definition: web page "DeepSpeed4Science 技术指南：AI4Science
// 大模型长序列训练与 Evoformer 内存高效注意力内核实战" §3.5 (scale, add bias,
// softmax, times V) and §3.7 (fp32 lse saved for the backward; bias1 is
// (B, N, 1, 1, L), bias2 is (B, 1, H, L, L)).
//
// Structure (one CTA per SM, persistent over a contiguous range of work items
// ordered (b, h, q-tile, n), so that consecutive items share their pair-bias
// rows).  The kernel streams key tiles across item boundaries:
//   warp 8      TMA producer: Q tile per item (2 buffers); K, V tiles and the
//               key-mask chunk per key tile into a ring of up to 4 stages; the
//               pair-bias tiles of the current (b, h, q-tile) once per group
//               (resident), or per key tile for long sequences (streaming).
//   warp 9      MMA issuer (one thread): S_u = Q·K_uᵀ into TMEM (2 buffers),
//               then O_u = P_u·V_u (P read from TMEM), issued one key tile
//               behind S — also across items, so the tensor core never waits
//               for an epilogue.
//   warps 0..7  softmax.  Warp w owns query rows 32·(w%4).. (its TMEM lane
//               quadrant) and key columns 64·(w/4).. of every tile, and runs an
//               independent online softmax over its key half: its own reference
//               max and sum, its P half (fp16/bf16, into TMEM).  P·V accumulates
//               in TMEM across all key tiles of an item (one accumulator per key
//               half, double-buffered across items).  The reference max moves
//               only when a tile's max exceeds it by more than 2^8 (P stays
//               below 256, exact in fp16/bf16); then the warp rescales its
//               accumulator in TMEM once the previous P·V is done.  The two
//               halves of a row are merged once per item, in the epilogue: each
//               warp reads its DP/2 output columns of both accumulators and the
//               partner's (max, sum) from shared memory, and writes its share
//               of O through shared memory with a TMA tile store.  Scale and
//               biases are applied in the log2 domain with packed f32x2
//               arithmetic.
// Key columns past L carry a -inf key-mask entry, so no other masking is
// needed; query rows past L are computed and not stored.
#include "evo_internal.h"
#include "evo_ptx.cuh"

namespace evo {
namespace {

// This kernel's own item order: (b, h, query tile, n), or with qt_fast (b, h, n, query tile).

constexpr int kMaxStages = 4;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// TMEM columns: S (2 buffers of 128), P (2 buffers of 64 columns of packed
// pairs; half h of the keys in columns 32h..), O (per key half and buffer, DP
// columns each: 2 buffers when DP <= 32, else 1).
__device__ __forceinline__ uint32_t col_s(uint32_t b) { return b ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_p(uint32_t b) { return b ? 320u : 256u; }
template <int DP>
__device__ __forceinline__ uint32_t col_o(uint32_t b, uint32_t half) {
  return 384u + (DP <= 32 ? (b * 2 + half) : half) * DP;
}
template <int DP>
__host__ __device__ constexpr int o_buffers() { return DP <= 32 ? 2 : 1; }

// Pair-bias handling: none, resident per (b, h, q-tile) group, or streamed per key tile.
enum B2Kind : int { kB2None = 0, kB2Resident = 1, kB2Stream = 2 };

struct FwdBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t b2_full, b2_empty;
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_free[2];
  uint64_t pv_done;            // one phase per P·V tile (waited on only before a rescale)
  uint64_t xsum[4], xdone[4];  // per lane quadrant: the two warps sharing those rows (epilogue merge)
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  // per K/V stage, written by the producer before it arrives on kv_full: the key tile
  // held (bits 0-15), first tile of its item (bit 16), last tile of its item (bit 17)
  uint32_t tile_meta[kMaxStages];
};

constexpr uint32_t kTileFirst = 1u << 16, kTileLast = 1u << 17;
// The same tag for tile x of an item that runs all KT tiles (no skipping).
__device__ __forceinline__ uint32_t tile_meta_all(int x, int KT) {
  return static_cast<uint32_t>(x) | (x == 0 ? kTileFirst : 0u) | (x + 1 == KT ? kTileLast : 0u);
}

template <int DP>
struct FwdLayout {
  static constexpr uint32_t kTileBytes = kTile * DP * 2;
  Ring q, k, v, b1, b2s;
  uint32_t b2r, xchg, stg, bars, total;
  __host__ __device__ FwdLayout(int b2kind, int stages, int KT) {
    uint32_t off = 0;
    q = Ring{off, kTileBytes};
    off += 2 * kTileBytes;
    k = Ring{off, 2 * kTileBytes};
    v = Ring{off + kTileBytes, 2 * kTileBytes};
    off += stages * 2 * kTileBytes;
    b2s = Ring{off, 32768u};
    if (b2kind == kB2Stream) off += stages * 32768u;
    b2r = off;
    if (b2kind == kB2Resident) off += KT * 32768u;
    b1 = Ring{off, 512u};
    off += stages * 512u;
    xchg = off;  // epilogue merge: per half, (max, sum) of each row, [value][row]
    off += 2 * 2 * 128 * 4;
    off = (off + 1023u) & ~1023u;
    stg = off;   // O staging: per softmax warp [32 rows][DP/2] (box row swizzle)
    off += kSoftmaxWarps * 32u * DP;
    bars = off;
    off += (sizeof(FwdBars) + 127) & ~127u;
    total = off;
  }
};

// Work items are ordered (b, h, q-tile, n), n fastest, so that the pair-bias tiles of a
// (b, h, q-tile) stay resident across n; without a resident pair bias (qt_fast) they are
// ordered (b, h, n, q-tile), so that the query tiles sharing one (n, h)'s K and V run back
// to back on one CTA and re-read them from L2 instead of DRAM.  A CTA walks a contiguous
// range with an incremental iterator (no integer division per item).
struct ItemIter {
  int b, h, qt, n;
  __device__ __forceinline__ void init(long long item, const FwdArgs& a) {
    long long t = item;
    if (a.qt_fast) {
      qt = static_cast<int>(t % a.QT);
      t /= a.QT;
      n = static_cast<int>(t % a.N);
      t /= a.N;
    } else {
      n = static_cast<int>(t % a.N);
      t /= a.N;
      qt = static_cast<int>(t % a.QT);
      t /= a.QT;
    }
    h = static_cast<int>(t % a.H);
    b = static_cast<int>(t / a.H);
  }
  __device__ __forceinline__ void next(const FwdArgs& a) {
    int& fast = a.qt_fast ? qt : n;
    int& slow = a.qt_fast ? n : qt;
    const int nfast = a.qt_fast ? a.QT : a.N, nslow = a.qt_fast ? a.N : a.QT;
    if (++fast == nfast) {
      fast = 0;
      if (++slow == nslow) {
        slow = 0;
        if (++h == a.H) {
          h = 0;
          ++b;
        }
      }
    }
  }
};

// Bounded wait that ignores the abort flag: used only to drain work this
// thread itself put in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int* status) {
  volatile int never = 0;
  WaitGuard g{limit_ns, status, &never};
  mbar_wait(bar, parity, g);
}

// Pair-bias tile (query rows i0.., key columns j0..) by plain loads into the
// 128B-swizzled two-half layout the TMA map writes (used when L % 8 != 0).
__device__ __forceinline__ void fill_b2_loads(uint8_t* dst, const uint16_t* b2, int L, int i0, int j0, int lane) {
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
    *reinterpret_cast<uint2*>(dst + half * 16384 + swz_offset(r, chunk, 128) + within * 2) = make_uint2(w[0], w[1]);
  }
}

// ------------------------------------------------------------ producer (one warp)
// SKIP: masked-tile skipping; the consumers then follow the stage tags (tile_meta)
// instead of counting the tiles of an item themselves.
template <int DP, bool BF16, int B2, bool SKIP>
__device__ __forceinline__ void fwd_producer(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay,
                                             FwdBars* bars, const WaitGuard& g, int lane, long long i0,
                                             long long i1) {
  constexpr uint32_t kTB = FwdLayout<DP>::kTileBytes;
  const int S = a.stages, KT = a.QT;
  const bool tma_b2 = a.bias2_mode == kBias2Tma;
  const uint32_t kv_bytes = 2 * kTB + ((B2 == kB2Stream && tma_b2) ? 32768u : 0u);
  uint32_t u = 0, q_it = 0, grp_it = 0, s = 0, ph = 0;
  ItemIter c;
  c.init(i0, a);
  // raw key-mask values of the next tile, loaded one tile ahead so that their
  // latency overlaps the wait for a free stage
  uint16_t b1raw[4];
  // the item's key tiles: every tile, or with masked-tile skipping those holding a kept key
  auto tiles_of = [&](const ItemIter& t) -> uint64_t {
    if (!SKIP || !a.bias1 || t.b >= a.B) return 0ull;
    return kept_tiles<BF16>(a.bias1 + (static_cast<size_t>(t.b) * a.N + t.n) * a.L, a.L, a.skip_at, lane);
  };
  auto b1_prefetch = [&](const ItemIter& t, int jt) {
    const uint16_t* row = (a.bias1 && t.b < a.B) ? a.bias1 + (static_cast<size_t>(t.b) * a.N + t.n) * a.L : nullptr;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = jt * kTile + lane * 4 + e;
      b1raw[e] = (row && j < a.L) ? row[j] : static_cast<uint16_t>(0);
    }
  };
  // next item's key-mask row, loaded one item ahead and scanned at the item's last tile
  // (rows too long for registers are scanned at once)
  RowScan nscan;
  const bool scan_ahead = SKIP && a.bias1 && row_scan_fits(a.bias1, a.L);
  uint64_t act = tiles_of(c);
  b1_prefetch(c, next_tile(act, -1, KT));
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, c.next(a)) {
    const int bn = c.b * a.N + c.n, bh = c.b * a.H + c.h;
    ItemIter nc = c;
    nc.next(a);
    if (B2 == kB2Resident && (item == i0 || c.n == 0)) {
      // all softmax warps are done with the previous group's tiles
      if (!mbar_wait(smem_u32(&bars->b2_empty), (grp_it & 1) ^ 1, g)) { ok = false; break; }
      const uint32_t full = smem_u32(&bars->b2_full);
      if (tma_b2) {
        if (lane == 0) {
          mbar_expect_tx(full, KT * 32768u);
          for (int t = 0; t < KT; ++t) {
            tma_load_3d(smem_u32(base + lay.b2r + t * 32768u), &a.tb2, full, t * kTile, c.qt * kTile, bh);
            tma_load_3d(smem_u32(base + lay.b2r + t * 32768u + 16384u), &a.tb2, full, t * kTile + 64,
                        c.qt * kTile, bh);
          }
        }
      } else {
        for (int t = 0; t < KT; ++t)
          fill_b2_loads(base + lay.b2r + t * 32768u, a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L,
                        c.qt * kTile, t * kTile, lane);
      }
      mbar_arrive(full);
      ++grp_it;
    }
    const uint32_t qs = q_it & 1;
    if (!mbar_wait(smem_u32(&bars->q_empty[qs]), ((q_it >> 1) & 1) ^ 1, g)) { ok = false; break; }
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(&bars->q_full[qs]), kTB);
      tma_load_4d(smem_u32(base + lay.q[qs]), &a.tq, smem_u32(&bars->q_full[qs]), 0, c.h, c.qt * kTile, bn);
    }
    ++q_it;
    uint64_t next_act = 0;
    const bool nc_in = nc.b < a.B;
    if (scan_ahead) {
      if (nc_in) row_scan_issue(nscan, a.bias1 + (static_cast<size_t>(nc.b) * a.N + nc.n) * a.L, a.L, lane);
    } else {
      next_act = tiles_of(nc);
    }
    const int jt0 = next_tile(act, -1, KT);
    for (int jt = jt0; jt < KT; ++u) {
      const int jn = next_tile(act, jt, KT);
      if (!mbar_wait(smem_u32(&bars->kv_empty[s]), ph ^ 1, g)) { ok = false; break; }
      const uint32_t full = smem_u32(&bars->kv_full[s]);
      if (lane == 0) {  // copies first: the key-mask loads below must not delay them
        bars->tile_meta[s] = static_cast<uint32_t>(jt) | (jt == jt0 ? kTileFirst : 0u) | (jn >= KT ? kTileLast : 0u);
        mbar_expect_tx(full, kv_bytes);
        tma_load_4d(smem_u32(base + lay.k[s]), &a.tk, full, 0, c.h, jt * kTile, bn);
        tma_load_4d(smem_u32(base + lay.v[s]), &a.tv, full, 0, c.h, jt * kTile, bn);
        if (B2 == kB2Stream && tma_b2) {
          tma_load_3d(smem_u32(base + lay.b2s[s]), &a.tb2, full, jt * kTile, c.qt * kTile, bh);
          tma_load_3d(smem_u32(base + lay.b2s[s] + 16384), &a.tb2, full, jt * kTile + 64, c.qt * kTile, bh);
        }
      }
      if (B2 == kB2Stream && !tma_b2)
        fill_b2_loads(base + lay.b2s[s], a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L, c.qt * kTile,
                      jt * kTile, lane);
      {  // key-mask chunk, fp32 in the log2 domain; -inf past L
        float4 m4;
        float* mv = reinterpret_cast<float*>(&m4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = jt * kTile + lane * 4 + e;
          mv[e] = j < a.L ? (a.bias1 ? to_f32<BF16>(b1raw[e]) * kLog2e : 0.0f) : -INFINITY;
        }
        *reinterpret_cast<float4*>(base + lay.b1[s] + lane * 16) = m4;
      }
      mbar_arrive(full);
      if (jn < KT) {
        b1_prefetch(c, jn);
      } else {
        if (scan_ahead && nc_in) next_act = row_scan_finish<BF16>(nscan, a.L, a.skip_at, lane);
        b1_prefetch(nc, next_tile(next_act, -1, KT));
      }
      if (++s == static_cast<uint32_t>(S)) {
        s = 0;
        ph ^= 1;
      }
      jt = jn;
    }
    act = next_act;
  }
  // Drain: every copy this warp started has landed before the CTA may exit.
  for (uint32_t q = 0; q < 2; ++q) {
    const uint32_t issued = (q_it + 1 - q) / 2;
    if (issued > 0) drain_wait(smem_u32(&bars->q_full[q]), (issued - 1) & 1, a.wait_ns, a.status);
  }
  for (uint32_t st = 0; st < static_cast<uint32_t>(S); ++st) {
    const uint32_t issued = (u + S - 1 - st) / S;
    if (issued > 0) drain_wait(smem_u32(&bars->kv_full[st]), (issued - 1) & 1, a.wait_ns, a.status);
  }
  if (B2 == kB2Resident && grp_it > 0) drain_wait(smem_u32(&bars->b2_full), (grp_it - 1) & 1, a.wait_ns, a.status);
}

// ------------------------------------------------------------ MMA issuer (one thread)
// O_half (+)= P_v,half · V_v,half for both key halves (K = 64 keys each), P from
// TMEM, accumulated over the key tiles of item `item` (meta: first / last tile of it).
template <int DP, bool BF16>
__device__ __forceinline__ bool fwd_issue_pv(uint32_t v, uint32_t sv, uint32_t meta, uint32_t item, uint8_t* base,
                                             const FwdLayout<DP>& lay, FwdBars* bars, uint32_t tmem,
                                             const WaitGuard& g) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_o = idesc_f16(128, DP, BF16, false, true);
  constexpr int NB = o_buffers<DP>();
  const uint32_t vb = v & 1, vph = (v >> 1) & 1;
  const uint32_t ob = item % NB, oph = (item / NB) & 1;
  if (!mbar_wait(smem_u32(&bars->p_full[vb]), vph, g)) return false;
  const bool first = (meta & kTileFirst) != 0;
  if (first && !mbar_wait(smem_u32(&bars->o_free[ob]), oph ^ 1, g)) return false;
  tc_fence_after();
  const uint64_t vd = smem_desc(smem_u32(base + lay.v[sv]), kTile * RB, 8 * RB, SWZ);
  const uint32_t acc = first ? 0u : 1u;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int k = 0; k < 4; ++k)  // 64 keys in steps of 16 (8 TMEM columns of packed pairs)
      umma_ts(tmem + col_o<DP>(ob, half), tmem + col_p(vb) + half * 32 + k * 8, vd + (half * 64 + k * 16) * RB / 16,
              id_o, (acc | k) ? 1u : 0u);
  }
  umma_commit(smem_u32(&bars->pv_done));
  if (meta & kTileLast) umma_commit(smem_u32(&bars->o_full[ob]));
  umma_commit(smem_u32(&bars->p_empty[vb]));
  umma_commit(smem_u32(&bars->kv_empty[sv]));
  return true;
}

template <int DP, bool BF16, bool SKIP>
__device__ __forceinline__ void fwd_mma(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay, FwdBars* bars,
                                        uint32_t tmem, const WaitGuard& g, long long i0, long long i1) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
  const int S = a.stages, KT = a.QT;
  uint32_t u = 0, q_it = 0, prev_stage = 0, s = 0, ph = 0, item_ord = 0, prev_item = 0, prev_meta = 0;
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, ++item_ord) {
    const uint32_t qs = q_it & 1;
    if (!mbar_wait(smem_u32(&bars->q_full[qs]), (q_it >> 1) & 1, g)) { ok = false; break; }
    ++q_it;
    tc_fence_after();
    const uint64_t qd = smem_desc(smem_u32(base + lay.q[qs]), 16, 8 * RB, SWZ);
    for (int x = 0; SKIP || x < KT; ++x) {  // with SKIP, up to the tile tagged last
      if (!mbar_wait(smem_u32(&bars->kv_full[s]), ph, g)) { ok = false; break; }
      const uint32_t meta = SKIP ? bars->tile_meta[s] : tile_meta_all(x, KT);
      const bool last = (meta & kTileLast) != 0;
      const uint32_t buf = u & 1;
      if (!mbar_wait(smem_u32(&bars->s_free[buf]), ((u >> 1) & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      const uint64_t kd = smem_desc(smem_u32(base + lay.k[s]), 16, 8 * RB, SWZ);
#pragma unroll
      for (int k = 0; k < DP / 16; ++k) umma_ss(tmem + col_s(buf), qd + k * 2, kd + k * 2, id_s, k > 0);
      umma_commit(smem_u32(&bars->s_full[buf]));
      if (last) umma_commit(smem_u32(&bars->q_empty[qs]));
      if (u > 0 && !fwd_issue_pv<DP, BF16>(u - 1, prev_stage, prev_meta, prev_item, base, lay, bars, tmem, g)) {
        ok = false;
        break;
      }
      prev_stage = s;
      prev_meta = meta;
      prev_item = item_ord;
      ++u;
      if (++s == static_cast<uint32_t>(S)) {
        s = 0;
        ph ^= 1;
      }
      if (SKIP && last) break;
    }
  }
  if (ok && u > 0) fwd_issue_pv<DP, BF16>(u - 1, prev_stage, prev_meta, prev_item, base, lay, bars, tmem, g);
  // Drain: all MMAs this thread issued are complete before TMEM is freed.
  umma_commit(smem_u32(&bars->drain));
  drain_wait(smem_u32(&bars->drain), 0, a.wait_ns, a.status);
}

// ------------------------------------------------------------ softmax (warps 0..7)
constexpr float kRescaleLog2 = 8.0f;  // the reference max moves only past this margin

// n fp32 TMEM columns of this thread's lane (n a multiple of 8) into v.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t col, float (&v)[N]) {
  if constexpr (N == 8) {
    uint32_t x[8];
    tmem_ld8(col, x);
    tmem_wait_ld(x);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(x[e]);
  } else {
    uint32_t x[N / 16][16];
#pragma unroll
    for (int q = 0; q < N / 16; ++q) tmem_ld16(col + q * 16, x[q]);
#pragma unroll
    for (int q = 0; q < N / 16; ++q) tmem_wait_ld(x[q]);
#pragma unroll
    for (int q = 0; q < N / 16; ++q)
#pragma unroll
      for (int e = 0; e < 16; ++e) v[q * 16 + e] = __uint_as_float(x[q][e]);
  }
}

// This warp's accumulator (its key half, all DP columns) *= alpha, in place.
template <int DP>
__device__ __forceinline__ void fwd_rescale_o(uint32_t col, float alpha) {
#pragma unroll
  for (int c = 0; c < DP / 16; ++c) {
    uint32_t x[16];
    tmem_ld16(col + c * 16, x);
    tmem_wait_ld(x);
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) * alpha);
    tmem_st16(col + c * 16, x);
  }
  tmem_wait_st();
}

// Merge the two key halves of a finished item's rows and write O and lse (m: the
// half's reference max in log2 units, -inf when none of its keys is unmasked).  Each
// warp exchanges its (max, sum) with the partner warp of its lane quadrant, reads
// its DP/2 output columns of both accumulators from TMEM, and stores its
// [32 rows][DP/2] share of O through shared memory with one TMA tile store.
template <int DP, bool BF16>
__device__ __forceinline__ bool fwd_epilogue(const FwdArgs& a, const ItemIter& c, float m, float l, uint32_t fin,
                                             uint8_t* base, const FwdLayout<DP>& lay, FwdBars* bars, uint32_t trow,
                                             int w, int quad, int hc, int r, int lane, const WaitGuard& g) {
  constexpr int HD = DP / 2;
  constexpr int NB = o_buffers<DP>();
  const uint32_t ob = fin % NB;
  float* xchg = reinterpret_cast<float*>(base + lay.xchg);
  if (fin > 0 && !mbar_wait(smem_u32(&bars->xdone[quad]), (fin - 1) & 1, g)) return false;
  float* mine = xchg + hc * 256;
  mine[r] = m;
  mine[128 + r] = l;
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->xsum[quad]));
  if (!mbar_wait(smem_u32(&bars->xsum[quad]), fin & 1, g)) return false;
  const float* other = xchg + (hc ^ 1) * 256;
  const float m_o = other[r], l_o = other[128 + r];
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->xdone[quad]));
  const float mx = fmaxf(m, m_o);
  const float mm = mx == -INFINITY ? 0.0f : mx;  // both halves empty: O = 0, lse = -inf
  const float s_me = ex2(m - mm), s_o = ex2(m_o - mm);
  const float lt = fmaf(l, s_me, l_o * s_o);
  const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
  const float f_me = s_me * inv, f_o = s_o * inv;
  // both accumulators' columns hc·HD.. of this lane, once every P·V of the item is done
  if (!mbar_wait(smem_u32(&bars->o_full[ob]), (fin / NB) & 1, g)) return false;
  tc_fence_after();
  float om[HD], oo[HD];
  tmem_load_cols<HD>(trow + col_o<DP>(ob, hc) + hc * HD, om);
  tmem_load_cols<HD>(trow + col_o<DP>(ob, hc ^ 1) + hc * HD, oo);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->o_free[ob]));
  uint8_t* blk = base + lay.stg + w * 32 * DP;
  if (lane == 0) bulk_wait_read_all();  // the previous item's store has read the staging block
  __syncwarp();
#pragma unroll
  for (int e = 0; e < HD; e += 8) {
    uint4 pk;
    pk.x = pack2<BF16>(fmaf(om[e + 0], f_me, oo[e + 0] * f_o), fmaf(om[e + 1], f_me, oo[e + 1] * f_o));
    pk.y = pack2<BF16>(fmaf(om[e + 2], f_me, oo[e + 2] * f_o), fmaf(om[e + 3], f_me, oo[e + 3] * f_o));
    pk.z = pack2<BF16>(fmaf(om[e + 4], f_me, oo[e + 4] * f_o), fmaf(om[e + 5], f_me, oo[e + 5] * f_o));
    pk.w = pack2<BF16>(fmaf(om[e + 6], f_me, oo[e + 6] * f_o), fmaf(om[e + 7], f_me, oo[e + 7] * f_o));
    const uint32_t off = HD == 8 ? lane * 16u : swz_offset(lane, e >> 3, DP);
    *reinterpret_cast<uint4*>(blk + off) = pk;
  }
  fence_proxy_async_smem();
  __syncwarp();
  const size_t bn = static_cast<size_t>(c.b) * a.N + c.n;
  if (lane == 0) {
    tma_store_4d(&a.tout_half, smem_u32(blk), hc * HD, c.h, c.qt * kTile + quad * 32, static_cast<int>(bn));
    bulk_commit_group();
  }
  const int i = c.qt * kTile + r;
  if (hc == 0 && i < a.L) a.lse[(bn * a.H + c.h) * a.L + i] = lt > 0.0f ? (mm + lg2(lt)) * kLn2 : -INFINITY;
  return true;
}

template <int DP, bool BF16, int B2, bool SKIP>
__device__ __forceinline__ void fwd_softmax(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay,
                                            FwdBars* bars, uint32_t tmem, const WaitGuard& g, long long i0,
                                            long long i1) {
  constexpr bool kHasB2 = B2 != kB2None;
  constexpr int NB = o_buffers<DP>();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = w & 3, hc = w >> 2;  // TMEM lane quadrant, key-column half
  const int r = quad * 32 + lane;       // query row within the tile == TMEM lane
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const float2 l2e2 = make_float2(kLog2e, kLog2e);
  const int S = a.stages, KT = a.QT;
  uint32_t u = 0, fin = 0, grp_it = 0, s = 0, ph = 0, item_ord = 0;
  float m = 0.0f, l = 0.0f, m_fin = 0.0f, l_fin = 0.0f;  // reference max (log2 units) and sum of this half
  bool have = false;
  ItemIter cur, prev;
  cur.init(i0, a);
  prev = cur;
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, ++item_ord) {
    if (item > i0) {
      prev = cur;
      cur.next(a);
    }
    const bool grp_last = item + 1 == i1 || cur.n == a.N - 1;
    if (B2 == kB2Resident && (item == i0 || cur.n == 0)) {
      if (!mbar_wait(smem_u32(&bars->b2_full), grp_it & 1, g)) { ok = false; break; }
      ++grp_it;
    }
    for (int x = 0; SKIP || x < KT; ++x) {  // with SKIP, up to the tile tagged last
      const bool first = x == 0;
      if (first) {  // the previous item's statistics, for its epilogue (-inf: no unmasked key)
        m_fin = have ? m : -INFINITY;
        l_fin = l;
      }
      const uint32_t buf = u & 1, bph = (u >> 1) & 1;
      if (!mbar_wait(smem_u32(&bars->kv_full[s]), ph, g)) { ok = false; break; }
      const uint32_t meta = SKIP ? bars->tile_meta[s] : tile_meta_all(x, KT);
      const int jt = static_cast<int>(meta & 0xffffu);
      const bool last = (meta & kTileLast) != 0;
      if (!mbar_wait(smem_u32(&bars->s_full[buf]), bph, g)) { ok = false; break; }
      tc_fence_after();
      float y[64];
      {
        uint32_t sr[2][32];
        const uint32_t col = trow + col_s(buf) + hc * 64;
        tmem_ld32(col, sr[0]);
        tmem_ld32(col + 32, sr[1]);
        tmem_wait_ld(sr[0]);
        tmem_wait_ld(sr[1]);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          y[e] = __uint_as_float(sr[0][e]);
          y[32 + e] = __uint_as_float(sr[1][e]);
        }
      }
      // y = S·s·log2e + bias1·log2e (+ bias2·log2e); row max over this half (4 chains)
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      const float* b1 = reinterpret_cast<const float*>(base + lay.b1[s]) + hc * 64;
      const uint8_t* b2t = base + (B2 == kB2Resident ? lay.b2r + jt * 32768u : lay.b2s[s]) + hc * 16384;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const float4 m0 = *reinterpret_cast<const float4*>(b1 + c8 * 8);
        const float4 m1 = *reinterpret_cast<const float4*>(b1 + c8 * 8 + 4);
        const float2 mk[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                              make_float2(m1.z, m1.w)};
        uint4 pb = make_uint4(0u, 0u, 0u, 0u);
        if (kHasB2) pb = *reinterpret_cast<const uint4*>(b2t + swz_offset(r, c8, 128));
        const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int x = c8 * 8 + e2 * 2;
          float2 t = fma2(make_float2(y[x], y[x + 1]), sl2, mk[e2]);
          if (kHasB2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
          y[x] = t.x;
          y[x + 1] = t.y;
          mx[e2] = max3(mx[e2], t.x, t.y);
        }
      }
      // this half of S and the stage's bias data are no longer read by this warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->s_free[buf]));
        mbar_arrive(smem_u32(&bars->kv_empty[s]));
        if (B2 == kB2Resident && grp_last && last) mbar_arrive(smem_u32(&bars->b2_empty));
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      // reference max: the first tile's max (0 when every key so far is masked); later
      // tiles move it only past the margin, and then the accumulator is rescaled
      // (have: a finite reference exists; until then every P is exactly 0 and so is
      // the accumulator, so the first unmasked tile just sets the reference)
      float alpha = 1.0f;
      if (first || !have) {
        have = mt != -INFINITY;
        m = have ? mt : 0.0f;
        if (first) l = 0.0f;
      } else if (mt > m + kRescaleLog2) {
        alpha = ex2(m - mt);
        m = mt;
        l *= alpha;
      }
      const float2 nm2 = make_float2(-m, -m);
      float2 rs[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      uint32_t pp[32];
#pragma unroll
      for (int x = 0; x < 64; x += 2) {
        const float2 t = add2(make_float2(y[x], y[x + 1]), nm2);
        const float p0 = ex2(t.x), p1 = ex2(t.y);
        rs[(x >> 1) & 1] = add2(rs[(x >> 1) & 1], make_float2(p0, p1));
        pp[x >> 1] = pack2<BF16>(p0, p1);
      }
      l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
      // P half -> TMEM (64 keys = 32 columns of packed pairs), after P·V of tile u-2
      if (!mbar_wait(smem_u32(&bars->p_empty[buf]), bph ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      // rare: rescale this half's accumulator once P·V of tile u-1 is done.  The TMEM
      // loads and stores are warp-collective, so the whole warp takes this path when any
      // of its rows needs it (the other rows scale by 1).
      if (__any_sync(0xffffffffu, alpha != 1.0f)) {
        if (!mbar_wait(smem_u32(&bars->pv_done), (u - 1) & 1, g)) { ok = false; break; }
        tc_fence_after();
        fwd_rescale_o<DP>(trow + col_o<DP>(item_ord % NB, hc), alpha);
      }
      tmem_st32(trow + col_p(buf) + hc * 32, pp);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[buf]));
      if (first && u > 0 &&
          !fwd_epilogue<DP, BF16>(a, prev, m_fin, l_fin, fin++, base, lay, bars, trow, w, quad, hc, r, lane, g)) {
        ok = false;
        break;
      }
      ++u;
      if (++s == static_cast<uint32_t>(S)) {
        s = 0;
        ph ^= 1;
      }
      if (SKIP && last) break;
    }
  }
  if (ok && u > 0)
    fwd_epilogue<DP, BF16>(a, cur, have ? m : -INFINITY, l, fin++, base, lay, bars, trow, w, quad, hc, r, lane, g);
  if (lane == 0) bulk_wait_all();  // this warp's O stores complete before the CTA's smem goes away
}

template <int DP, bool BF16, int B2, bool SKIP>
__global__ void __launch_bounds__(kThreads, 1) evo_fwd_kernel(const __grid_constant__ FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const FwdLayout<DP> lay(B2, a.stages, a.QT);
  FwdBars* bars = reinterpret_cast<FwdBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long i0 = static_cast<long long>(blockIdx.x) * a.chunk;
  const long long i1 = i0 + a.chunk < a.items ? i0 + a.chunk : a.items;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 1);
      mbar_init(smem_u32(&bars->q_empty[s]), 1);
    }
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1 + kSoftmaxWarps);
    }
    mbar_init(smem_u32(&bars->b2_full), 32);
    mbar_init(smem_u32(&bars->b2_empty), kSoftmaxWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->s_free[b]), kSoftmaxWarps);
      mbar_init(smem_u32(&bars->p_full[b]), kSoftmaxWarps);
      mbar_init(smem_u32(&bars->p_empty[b]), 1);
      mbar_init(smem_u32(&bars->o_full[b]), 1);
      mbar_init(smem_u32(&bars->o_free[b]), kSoftmaxWarps);
    }
    mbar_init(smem_u32(&bars->pv_done), 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(smem_u32(&bars->xsum[q]), 2);
      mbar_init(smem_u32(&bars->xdone[q]), 2);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    if (B2 != kB2None && a.bias2_mode == kBias2Tma) tma_prefetch_desc(&a.tb2);
    tma_prefetch_desc(&a.tout_half);
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
    fwd_producer<DP, BF16, B2, SKIP>(a, base, lay, bars, g, lane, i0, i1);
  } else if (warp == kMmaWarp) {
    if (lane == 0) fwd_mma<DP, BF16, SKIP>(a, base, lay, bars, tmem, g, i0, i1);
    __syncwarp();
  } else {
    fwd_softmax<DP, BF16, B2, SKIP>(a, base, lay, bars, tmem, g, i0, i1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

constexpr size_t kMaxSmem = 232448;  // 227 KB opt-in limit per block

template <int DP, bool BF16, int B2, bool SKIP>
cudaError_t launch_fwd_s(FwdArgs a, cudaStream_t st) {
  const FwdLayout<DP> lay(B2, a.stages, a.QT);
  // At least 116 KB so that two CTAs never share an SM: each allocates all 512
  // TMEM columns, and a second resident CTA would stall in tcgen05.alloc.
  const size_t smem = (lay.total + 1024 > 116u * 1024u) ? lay.total + 1024 : 116u * 1024u;
  auto kern = evo_fwd_kernel<DP, BF16, B2, SKIP>;
  static bool limit_set[64] = {};
  cudaError_t e = ensure_smem_limit(kern, kMaxSmem, limit_set);
  if (e != cudaSuccess) return e;
  const long long sms = num_sms();
  a.chunk = (a.items + sms - 1) / sms;
  const long long grid = (a.items + a.chunk - 1) / a.chunk;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}
template <int DP, bool BF16, int B2>
cudaError_t launch_fwd_t(FwdArgs a, cudaStream_t st) {
  return a.tile_skip ? launch_fwd_s<DP, BF16, B2, true>(a, st) : launch_fwd_s<DP, BF16, B2, false>(a, st);
}

// Deepest K/V ring that fits, and whether the pair-bias tiles of one
// (b, h, q-tile) group can stay resident.
template <int DP, bool BF16>
cudaError_t launch_fwd_d(FwdArgs a, cudaStream_t st) {
  auto fits = [&](int kind, int stages) { return FwdLayout<DP>(kind, stages, a.QT).total + 1024 <= kMaxSmem; };
  if (a.bias2_mode == kBias2None) {
    a.stages = fits(kB2None, 4) ? 4 : 2;
    a.qt_fast = 1;
    return launch_fwd_t<DP, BF16, kB2None>(a, st);
  }
  for (int stages = 4; stages >= 2; --stages) {
    if (a.QT <= 4 && fits(kB2Resident, stages)) {
      a.stages = stages;
      a.b2_resident = 1;
      return launch_fwd_t<DP, BF16, kB2Resident>(a, st);
    }
  }
  a.stages = 2;
  a.b2_resident = 0;
  a.qt_fast = 1;
  return launch_fwd_t<DP, BF16, kB2Stream>(a, st);
}

}  // namespace

cudaError_t launch_fwd_single(const FwdArgs& args, bool bf16, cudaStream_t st) {
  FwdArgs a = args;
  a.items = static_cast<long long>(a.B) * a.H * a.QT * a.N;
  a.qt_fast = 0;
  return bf16 ? launch_fwd_d<64, true>(a, st) : launch_fwd_d<64, false>(a, st);
}

}  // namespace evo
