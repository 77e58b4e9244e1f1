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
// Structure.  One CTA per SM, persistent over a contiguous range of work items;
// an item is a pair of 128-row query tiles (2p, 2p + 1) of one (b, n, h) slice,
// which share its K and V tiles.
//   warp 8      TMA producer: both Q tiles of an item (two buffers); K, V and the
//               key mask (extension rows of the score MMA, or fp32 for the softmax)
//               per key tile into a ring of stages; pair-bias tiles
//               either resident per (b, h, pair) group across n, or streamed with
//               each key tile.
//   warps 9, 10 MMA issuers (one thread each, one per query tile g): per key
//               tile, S_g = Q_g K_jᵀ into TMEM (+ mask_j·D^1/2 without a pair bias,
//               and with one for bf16 at D <= 32: one more K = 16 step, a ones block
//               against the mask split into three bf16 parts, which hold all 24 bits
//               of the fp32 value), and the previous key tile's
//               O_g += P_g [V_{j-1} | 1] (P read from TMEM; the ones columns make
//               the MMA form the row sums of P too).  Neither waits on the other.
//   warps 0..3  softmax of query tile 0, warps 4..7 of query tile 1: one thread
//   and 4..7    per query row.  Each key tile's 128 scores are loaded into
//               registers in two 64-column loads, and S is released at once, so
//               the next tile's scores are computed while this one is worked on.
//               The two groups take turns for the exponentials (a bounded
//               mbarrier hand-off), so one group's exponentials overlap the other's
//               scoring and waits.
//   warp 11     idle (the three warpgroups share the register file: the third
//               gives registers back, the softmax warpgroups take them).
// Online softmax with a lazily moved reference: a row's reference max m moves
// only when a key tile's max exceeds it by more than 2^8 (P then stays below
// 256, exact enough in fp16/bf16); the O accumulator (with its row-sum columns)
// is then rescaled in TMEM once the previous P·V is done.  The tile max is taken
// before P is formed, so each tile is exponentiated once.  Where the score MMA adds
// the mask, P = 2^((S' + bias2·D^1/2)·D^-1/2·log2 e − m) costs a packed f32x2
// multiply-add (two with a pair bias) and an exponential per score; otherwise scale
// and biases are applied in the log2 domain first.  The epilogue divides
// O by the row sum and writes O through shared memory with one TMA tile store per
// warp, and lse.
// Key columns past L carry a -inf mask entry, so no other masking is needed; query rows past L (a partial or absent second query tile) are
// computed and not stored.
#include "evo_internal.h"
#include "evo_ptx.cuh"

namespace evo {
namespace {

constexpr int kMaxStages = 4;
constexpr int kSoftmaxWarps = 8;
// Three warpgroups: two of softmax warps, and one holding the producer and MMA warps
// (its other two warps idle).  Launched at 168 registers a thread (three warps share
// each scheduler's 16K registers); the third warpgroup then gives registers back so
// that the softmax warps can hold a whole row of scores:
// 128 x 104 + 256 x 200 = 384 x 168.
constexpr int kThreads = (kSoftmaxWarps + 4) * 32;
constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;  // MMA warps: kMmaWarp + g
constexpr uint32_t kRegsLaunch = 168, kRegsSoftmax = 200, kRegsOther = 104;
static_assert(128 * kRegsOther + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split exceeds the launch");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;     // the reference max moves only past this margin

// TMEM columns of query tile g: S (128 fp32), P (64 columns of packed pairs; keys
// 2c, 2c+1 in column c), O (DP fp32, then, for DP <= 32, 16 columns that each hold
// the row sum of P: the P·V MMA multiplies P by V with 16 columns of ones appended,
// which costs nothing at these widths, as an MMA with N <= 64 takes as long as one
// with N = 16).
__device__ __forceinline__ uint32_t col_s(uint32_t g) { return g * 256u; }
__device__ __forceinline__ uint32_t col_p(uint32_t g) { return g * 256u + 128u; }
__device__ __forceinline__ uint32_t col_o(uint32_t g) { return g * 256u + 192u; }
template <int DP>
constexpr bool kOnes = DP <= 32;
template <int DP>
constexpr int kOCols = kOnes<DP> ? DP + 16 : DP;

// Pair-bias handling: none, resident per (b, h, pair) group, or streamed per key tile.
enum B2Kind : int { kB2None = 0, kB2Resident = 1, kB2Stream = 2 };
// The key mask is added by the score MMA (one more K = 16 step against a block of ones) without
// a pair bias (a ones tile of its own), and with one for bf16 inputs at D <= 32, where the P·V
// MMA's ones block serves (every element 1.0 in bf16; the K side is zero past its three
// columns); otherwise the softmax warps add it.
__host__ __device__ constexpr bool mask_in_s(int DP, bool bf16, int b2kind) {
  return b2kind == kB2None || (bf16 && DP <= 32);
}

struct FwdBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t b2_full, b2_empty;
  uint64_t s_full[2], s_free[2];    // per query tile: S written / read and decided
  uint64_t p_full[2], p_empty[2];   // per query tile: P written / its P·V done
  uint64_t o_free[2];               // per query tile: the epilogue has read O
  uint64_t turn[2];
  uint64_t drain[2];
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
  static constexpr uint32_t kTB = kTile * DP * 2;
  Ring q, k, v, kx, b1, b2s;
  uint32_t b2r, stg, ones, qx, bars, total;
  // q[2 * buffer + g]; b2s[stage] + g * 32768; b2r + (g * KT + jt) * 32768
  __host__ __device__ FwdLayout(int b2kind, int stages, int KT, bool bf16) {
    uint32_t off = 0;
    b2s = Ring{off, 65536u};
    if (b2kind == kB2Stream) off += stages * 65536u;
    b2r = off;
    if (b2kind == kB2Resident) off += 2 * KT * 32768u;
    q = Ring{off, kTB};
    off += 4 * kTB;
    k = Ring{off, 2 * kTB};
    v = Ring{off + kTB, 2 * kTB};
    off += stages * 2 * kTB;
    stg = off;  // O staging: per softmax warp [32 rows][DP] (row swizzle = 2 DP bytes)
    off += kSoftmaxWarps * 32u * DP * 2u;
    off = (off + 1023u) & ~1023u;
    ones = off;  // 128 rows of ones, read as V's extra columns by the P·V MMA
    if (kOnes<DP>) off += kTile * DP * 2u;
    qx = 0;
    kx = Ring{0, 0};
    b1 = Ring{0, 0};
    if (mask_in_s(DP, bf16, b2kind)) {
      // the key mask enters S through one more K = 16 step of the score MMA: the Q side is a
      // constant [128][16] bf16 tile (columns 0..2 one; with a pair bias the ones block), the K
      // side per stage holds each key's mask·D^1/2 split into three bf16 parts (columns 0..2);
      // rows of 32 bytes, 32-byte swizzle
      if (b2kind == kB2None) {
        qx = off;
        off += kTile * 32u;
      } else {
        qx = ones;
      }
      kx = Ring{off, kTile * 32u};
      off += stages * kTile * 32u;
    } else {  // otherwise the softmax warps add the mask: fp32 × log2 e per key and stage
      b1 = Ring{off, 512u};
      off += stages * 512u;
    }
    bars = off;
    off += (sizeof(FwdBars) + 127) & ~127u;
    total = off;
  }
};

// Work items are pairs of query tiles: ordered (b, h, pair, n), n fastest, so that the
// pair-bias tiles of a (b, h, pair) stay resident across n; otherwise (b, h, n, pair),
// so that the pairs sharing one (n, h)'s K and V run back to back on one CTA.
struct ItemIter {
  int b, h, p, n;
  __device__ __forceinline__ void init(long long item, const FwdArgs& a) {
    long long t = item;
    if (a.qt_fast) {
      p = static_cast<int>(t % a.NP);
      t /= a.NP;
      n = static_cast<int>(t % a.N);
      t /= a.N;
    } else {
      n = static_cast<int>(t % a.N);
      t /= a.N;
      p = static_cast<int>(t % a.NP);
      t /= a.NP;
    }
    h = static_cast<int>(t % a.H);
    b = static_cast<int>(t / a.H);
  }
  __device__ __forceinline__ void next(const FwdArgs& a) {
    int& fast = a.qt_fast ? p : n;
    int& slow = a.qt_fast ? n : p;
    const int nfast = a.qt_fast ? a.NP : a.N, nslow = a.qt_fast ? a.N : a.NP;
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
  mbar_wait_inl(bar, parity, g);
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
  constexpr uint32_t kTB = FwdLayout<DP>::kTB;
  const int S = a.stages, KT = a.QT;
  const bool tma_b2 = a.bias2_mode == kBias2Tma;
  const uint32_t kv_bytes = 2 * kTB + ((B2 == kB2Stream && tma_b2) ? 65536u : 0u);
  uint32_t u = 0, q_it = 0, grp_it = 0, s = 0, ph = 0;
  ItemIter c;
  c.init(i0, a);
  uint16_t b1raw[4];
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
  RowScan nscan;
  const bool scan_ahead = SKIP && a.bias1 && row_scan_fits(a.bias1, a.L);
  const float inv_scale = kLog2e / a.scale_log2;  // the mask in units of Q·Kᵀ
  // the constant parts of the mask extension: the Q side's ones, and columns 8..15 (zero) of
  // every stage's K side; written before this warp's first arrival on a stage
#pragma unroll 1
  for (int row = lane; mask_in_s(DP, BF16, B2) && row < kTile; row += 32) {
    if (B2 == kB2None) {  // (with a pair bias the ones block serves)
      *reinterpret_cast<uint4*>(base + lay.qx + swz_offset(row, 0, 32)) =
          make_uint4(kBf16One | kBf16One << 16, kBf16One, 0u, 0u);
      *reinterpret_cast<uint4*>(base + lay.qx + swz_offset(row, 1, 32)) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int st = 0; st < S; ++st)
      *reinterpret_cast<uint4*>(base + lay.kx[st] + swz_offset(row, 1, 32)) = make_uint4(0u, 0u, 0u, 0u);
  }
  uint64_t act = tiles_of(c);
  b1_prefetch(c, next_tile(act, -1, KT));
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, c.next(a)) {
    const int bn = c.b * a.N + c.n, bh = c.b * a.H + c.h;
    ItemIter nc = c;
    nc.next(a);
    if (B2 == kB2Resident && (item == i0 || c.n == 0)) {
      // every softmax warp is done with the previous group's tiles
      if (!mbar_wait_warp_inl(smem_u32(&bars->b2_empty), (grp_it & 1) ^ 1, g)) { ok = false; break; }
      const uint32_t full = smem_u32(&bars->b2_full);
      for (int gq = 0; gq < 2; ++gq) {
        const int qt = 2 * c.p + gq;
        if (tma_b2) {
          if (lane == 0) {
            if (gq == 0) mbar_expect_tx(full, 2 * KT * 32768u);
            for (int t = 0; t < KT; ++t) {
              const uint32_t dst = smem_u32(base + lay.b2r + (gq * KT + t) * 32768u);
              tma_load_3d(dst, &a.tb2, full, t * kTile, qt * kTile, bh);
              tma_load_3d(dst + 16384u, &a.tb2, full, t * kTile + 64, qt * kTile, bh);
            }
          }
        } else {
          for (int t = 0; t < KT; ++t)
            fill_b2_loads(base + lay.b2r + (gq * KT + t) * 32768u, a.bias2 + static_cast<size_t>(bh) * a.L * a.L,
                          a.L, qt * kTile, t * kTile, lane);
        }
      }
      mbar_arrive(full);
      ++grp_it;
    }
    const uint32_t qb = q_it & 1;
    if (!mbar_wait_warp_inl(smem_u32(&bars->q_empty[qb]), ((q_it >> 1) & 1) ^ 1, g)) { ok = false; break; }
    if (lane == 0) {
      const uint32_t full = smem_u32(&bars->q_full[qb]);
      mbar_arrive_expect_tx(full, 2 * kTB);
      tma_load_4d(smem_u32(base + lay.q[2 * qb]), &a.tq, full, 0, c.h, (2 * c.p) * kTile, bn);
      tma_load_4d(smem_u32(base + lay.q[2 * qb + 1]), &a.tq, full, 0, c.h, (2 * c.p + 1) * kTile, bn);
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
      if (!mbar_wait_warp_inl(smem_u32(&bars->kv_empty[s]), ph ^ 1, g)) { ok = false; break; }
      const uint32_t full = smem_u32(&bars->kv_full[s]);
      if (lane == 0) {  // copies first: the key-mask conversion below must not delay them
        bars->tile_meta[s] = static_cast<uint32_t>(jt) | (jt == jt0 ? kTileFirst : 0u) | (jn >= KT ? kTileLast : 0u);
        mbar_expect_tx(full, kv_bytes);
        tma_load_4d(smem_u32(base + lay.k[s]), &a.tk, full, 0, c.h, jt * kTile, bn);
        tma_load_4d(smem_u32(base + lay.v[s]), &a.tv, full, 0, c.h, jt * kTile, bn);
        if (B2 == kB2Stream && tma_b2) {
          for (int gq = 0; gq < 2; ++gq) {
            const uint32_t dst = smem_u32(base + lay.b2s[s] + gq * 32768u);
            tma_load_3d(dst, &a.tb2, full, jt * kTile, (2 * c.p + gq) * kTile, bh);
            tma_load_3d(dst + 16384u, &a.tb2, full, jt * kTile + 64, (2 * c.p + gq) * kTile, bh);
          }
        }
      }
      if (B2 == kB2Stream && !tma_b2)
        for (int gq = 0; gq < 2; ++gq)
          fill_b2_loads(base + lay.b2s[s] + gq * 32768u, a.bias2 + static_cast<size_t>(bh) * a.L * a.L, a.L,
                        (2 * c.p + gq) * kTile, jt * kTile, lane);
      if constexpr (!mask_in_s(DP, BF16, B2)) {  // key-mask chunk, fp32 in the log2 domain; -inf past L
        float4 m4;
        float* mv = reinterpret_cast<float*>(&m4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = jt * kTile + lane * 4 + e;
          mv[e] = j < a.L ? (a.bias1 ? to_f32<BF16>(b1raw[e]) * kLog2e : 0.0f) : -INFINITY;
        }
        *reinterpret_cast<float4*>(base + lay.b1[s] + lane * 16) = m4;
      } else {  // this lane's four keys of the mask extension: mask·D^1/2 in three bf16 parts; -inf past L
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = jt * kTile + lane * 4 + e;
          const float mk = j < a.L ? (a.bias1 ? to_f32<BF16>(b1raw[e]) * inv_scale : 0.0f) : -INFINITY;
          uint32_t h, m, l;
          split3_bf16(mk, h, m, l);
          *reinterpret_cast<uint4*>(base + lay.kx[s] + swz_offset(lane * 4 + e, 0, 32)) =
              make_uint4(h | m << 16, l, 0u, 0u);
        }
        fence_proxy_async_smem();  // read by the tensor cores
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
  for (uint32_t qb = 0; qb < 2; ++qb) {
    const uint32_t issued = (q_it + 1 - qb) / 2;
    if (issued > 0) drain_wait(smem_u32(&bars->q_full[qb]), (issued - 1) & 1, a.wait_ns, a.status);
  }
  for (uint32_t st = 0; st < static_cast<uint32_t>(S); ++st) {
    const uint32_t issued = (u + S - 1 - st) / S;
    if (issued > 0) drain_wait(smem_u32(&bars->kv_full[st]), (issued - 1) & 1, a.wait_ns, a.status);
  }
  if (B2 == kB2Resident && grp_it > 0) drain_wait(smem_u32(&bars->b2_full), (grp_it - 1) & 1, a.wait_ns, a.status);
}

// ------------------------------------------------------------ MMA issuer (one thread)
// O_g (+)= P_g · [V | 1] (K = 128 keys, P from TMEM) for key tile number v (across
// items), stage sv, tag meta; first tile of an item: wait for the epilogue to have
// read O_g.  V is MN-major: its DP columns are one swizzle atom, and the ones block
// stands in as the next atom (leading byte offset = its distance from the stage).
template <int DP, bool BF16>
__device__ __forceinline__ bool fwd_issue_pv(uint32_t g, uint32_t v, uint32_t sv, uint32_t meta, uint32_t item_ord,
                                             uint8_t* base, const FwdLayout<DP>& lay, FwdBars* bars, uint32_t tmem,
                                             const WaitGuard& gd) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_o = idesc_f16(128, kOCols<DP>, BF16, false, true);
  if (!mbar_wait_inl(smem_u32(&bars->p_full[g]), v & 1, gd)) return false;
  const bool first = (meta & kTileFirst) != 0;
  if (first && !mbar_wait_inl(smem_u32(&bars->o_free[g]), (item_ord & 1) ^ 1, gd)) return false;
  tc_fence_after();
  const uint32_t va = smem_u32(base + lay.v[sv]);
  const uint32_t lbo = kOnes<DP> ? smem_u32(base + lay.ones) - va : kTile * RB;
  const uint64_t vd = smem_desc(va, lbo, 8 * RB, SWZ);
#pragma unroll
  for (int k = 0; k < 8; ++k)  // 128 keys in steps of 16 (8 TMEM columns of packed pairs)
    umma_ts(tmem + col_o(g), tmem + col_p(g) + k * 8, vd + k * 16 * RB / 16, id_o, (!first || k > 0) ? 1u : 0u);
  umma_commit(smem_u32(&bars->p_empty[g]));
  return true;
}

// One issuing thread per query tile g: per key tile, S_g as soon as the group has loaded
// its previous S (s_free), then the group's P·V of the previous key tile as its P
// arrives.  The two threads share the tensor core but never wait on each other.
template <int DP, bool BF16, int B2, bool SKIP>
__device__ __forceinline__ void fwd_mma(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay, FwdBars* bars,
                                        uint32_t tmem, uint32_t gq, const WaitGuard& g, long long i0, long long i1) {
  constexpr uint32_t RB = DP * 2;
  constexpr uint32_t SWZ = swizzle_for_row(RB);
  constexpr uint32_t id_s = idesc_f16(128, 128, BF16, false, false);
  constexpr uint32_t id_x = idesc_f16(128, 128, true, false, false);  // the mask step: bf16 whatever the inputs
  constexpr bool kMaskInS = mask_in_s(DP, BF16, B2);
  const uint64_t qxd = kMaskInS ? smem_desc(smem_u32(base + lay.qx), 16, 8 * 32, kSwizzle32B) : 0ull;
  const int S = a.stages, KT = a.QT;
  uint32_t u = 0, q_it = 0, s = 0, ph = 0, item_ord = 0;
  uint32_t prev_stage = 0, prev_meta = 0, prev_item = 0;
  bool ok = true;
  for (long long item = i0; ok && item < i1; ++item, ++item_ord) {
    const uint32_t qb = q_it & 1;
    if (!mbar_wait_inl(smem_u32(&bars->q_full[qb]), (q_it >> 1) & 1, g)) { ok = false; break; }
    ++q_it;
    tc_fence_after();
    for (int x = 0; SKIP || x < KT; ++x) {  // with SKIP, up to the tile tagged last
      if (!mbar_wait_inl(smem_u32(&bars->kv_full[s]), ph, g)) { ok = false; break; }
      const uint32_t meta = SKIP ? bars->tile_meta[s] : tile_meta_all(x, KT);
      const bool last = (meta & kTileLast) != 0;
      // S_g of this tile once the group has loaded its previous S
      if (!mbar_wait_inl(smem_u32(&bars->s_free[gq]), (u & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      const uint64_t kd = smem_desc(smem_u32(base + lay.k[s]), 16, 8 * RB, SWZ);
      const uint64_t qd = smem_desc(smem_u32(base + lay.q[2 * qb + gq]), 16, 8 * RB, SWZ);
#pragma unroll
      for (int k = 0; k < DP / 16; ++k) umma_ss(tmem + col_s(gq), qd + k * 2, kd + k * 2, id_s, k > 0);
      if (kMaskInS)  // the key mask
        umma_ss(tmem + col_s(gq), qxd, smem_desc(smem_u32(base + lay.kx[s]), 16, 8 * 32, kSwizzle32B), id_x, 1u);
      umma_commit(smem_u32(&bars->s_full[gq]));
      if (last) umma_commit(smem_u32(&bars->q_empty[qb]));
      // the group's P·V of the previous key tile
      if (u > 0) {
        if (!fwd_issue_pv<DP, BF16>(gq, u - 1, prev_stage, prev_meta, prev_item, base, lay, bars, tmem, g)) {
          ok = false;
          break;
        }
        umma_commit(smem_u32(&bars->kv_empty[prev_stage]));
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
  if (ok && u > 0 && fwd_issue_pv<DP, BF16>(gq, u - 1, prev_stage, prev_meta, prev_item, base, lay, bars, tmem, g))
    umma_commit(smem_u32(&bars->kv_empty[prev_stage]));
  // Drain: all MMAs this thread issued are complete before TMEM is freed.
  umma_commit(smem_u32(&bars->drain[gq]));
  drain_wait(smem_u32(&bars->drain[gq]), 0, a.wait_ns, a.status);
}

// ------------------------------------------------------------ softmax (warps 0..7)
// One 32-key chunk of this thread's row, in place; the chunk's max goes into mt.
//   FOLD (the score MMA added the mask): sr holds S' = Q·Kᵀ + mask·D^1/2 (fp32 bits) and
//   becomes y = S' (+ bias2·D^1/2), in units of Q·Kᵀ (bs2: D^1/2 in both lanes).
//   Otherwise sr holds S and becomes y = S·s + mask·log2 e (+ bias2·log2 e), in log2 units
//   (b1c: the chunk's mask × log2 e).
//   (b2h: the 64-key half of the pair-bias tile holding the chunk; c0: the chunk's first
//   16-byte column within that half's 128-byte rows.)
template <bool BF16, bool HAS_B2, bool FOLD>
__device__ __forceinline__ void chunk_scores(uint32_t (&sr)[32], const float* b1c, const uint8_t* b2h, int c0, int r,
                                             float2 sl2, float2 bs2, float& mt) {
  const float2 l2e2 = make_float2(kLog2e, kLog2e);
  float mx[4] = {mt, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // 8 keys per q
    float2 mk[4];
    if constexpr (!FOLD) {
      const float4 m0 = *reinterpret_cast<const float4*>(b1c + q * 8);
      const float4 m1 = *reinterpret_cast<const float4*>(b1c + q * 8 + 4);
      mk[0] = make_float2(m0.x, m0.y), mk[1] = make_float2(m0.z, m0.w);
      mk[2] = make_float2(m1.x, m1.y), mk[3] = make_float2(m1.z, m1.w);
    }
    uint4 pb = make_uint4(0u, 0u, 0u, 0u);
    if (HAS_B2) pb = *reinterpret_cast<const uint4*>(b2h + swz_offset(r, c0 + q, 128));
    const uint32_t pw[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int x = q * 8 + e2 * 2;
      float2 t = make_float2(__uint_as_float(sr[x]), __uint_as_float(sr[x + 1]));
      if constexpr (FOLD) {
        if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), bs2, t);
      } else {
        t = fma2(t, sl2, mk[e2]);
        if (HAS_B2) t = fma2(unpack2<BF16>(pw[e2]), l2e2, t);
      }
      if (HAS_B2 || !FOLD) {
        sr[x] = __float_as_uint(t.x);
        sr[x + 1] = __float_as_uint(t.y);
      }
      mx[e2] = max3(mx[e2], t.x, t.y);
    }
  }
  mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// P = 2^(y·s - m) for one chunk (y in units of Q·Kᵀ, SCALED) or 2^(y - m) (y in log2
// units), y as fp32 bits, packed into pp[0..15]; with ROWSUM, also the row sum into rs
// (otherwise the P·V MMA forms it).
template <bool BF16, bool ROWSUM, bool SCALED>
__device__ __forceinline__ void chunk_probs(const uint32_t (&y)[32], float2 sl2, float m, uint32_t (&pp)[16],
                                            float2& rs) {
  const float2 nm2 = make_float2(-m, -m);
#pragma unroll
  for (int x = 0; x < 32; x += 2) {
    const float2 yy = make_float2(__uint_as_float(y[x]), __uint_as_float(y[x + 1]));
    const float2 t = SCALED ? fma2(yy, sl2, nm2) : add2(yy, nm2);
    const float p0 = ex2(t.x), p1 = ex2(t.y);
    if (ROWSUM) rs = add2(rs, make_float2(p0, p1));
    pp[x >> 1] = pack2<BF16>(p0, p1);
  }
}

// O = acc / l and lse for a finished item: this warp's 32 rows of query tile g through
// shared memory with one TMA tile store.  (m: reference max in log2 units; l: row sum,
// read from the ones columns of the accumulator where the MMA forms it.)
template <int DP, bool BF16>
__device__ __forceinline__ void fwd_epilogue(const FwdArgs& a, const ItemIter& c, uint32_t g, float m, float l,
                                             uint8_t* base, const FwdLayout<DP>& lay, FwdBars* bars, uint32_t trow,
                                             int wq, int r, int lane) {
  constexpr int PC = DP < 32 ? DP : 32;  // columns per TMEM load
  if constexpr (kOnes<DP>) {
    uint32_t x[16];
    tmem_ld16(trow + col_o(g) + DP, x);
    tmem_wait_ld(x);
    l = __uint_as_float(x[0]);
  }
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  uint8_t* blk = base + lay.stg + (g * 4 + wq) * 32 * DP * 2;
  if (lane == 0) bulk_wait_read_all();  // this warp's previous store has read the staging block
  __syncwarp();
#pragma unroll
  for (int q = 0; q < DP / PC; ++q) {
    uint32_t x[PC];
    if constexpr (PC == 16) {
      tmem_ld16(trow + col_o(g) + q * PC, x);
    } else {
      tmem_ld32(trow + col_o(g) + q * PC, x);
    }
    tmem_wait_ld(x);
#pragma unroll
    for (int e = 0; e < PC; e += 8) {
      uint4 pk;
      pk.x = pack2<BF16>(__uint_as_float(x[e + 0]) * inv, __uint_as_float(x[e + 1]) * inv);
      pk.y = pack2<BF16>(__uint_as_float(x[e + 2]) * inv, __uint_as_float(x[e + 3]) * inv);
      pk.z = pack2<BF16>(__uint_as_float(x[e + 4]) * inv, __uint_as_float(x[e + 5]) * inv);
      pk.w = pack2<BF16>(__uint_as_float(x[e + 6]) * inv, __uint_as_float(x[e + 7]) * inv);
      *reinterpret_cast<uint4*>(blk + swz_offset(lane, (q * PC + e) >> 3, DP * 2)) = pk;
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->o_free[g]));
  fence_proxy_async_smem();
  __syncwarp();
  const int qt = 2 * c.p + static_cast<int>(g);
  const int row0 = qt * kTile + wq * 32;
  const size_t bn = static_cast<size_t>(c.b) * a.N + c.n;
  if (lane == 0 && row0 < a.L) {
    tma_store_4d(&a.tout, smem_u32(blk), 0, c.h, row0, static_cast<int>(bn));
    bulk_commit_group();
  }
  const int i = qt * kTile + r;
  if (i < a.L) a.lse[(bn * a.H + c.h) * a.L + i] = l > 0.0f ? (m + lg2(l)) * kLn2 : -INFINITY;
}

// Scales this thread's row of the O accumulator (with its row-sum columns) by alpha.
// Warp-collective.
template <int DP>
__device__ __forceinline__ void rescale_o(uint32_t ocol, float alpha) {
#pragma unroll 1
  for (int c = 0; c < kOCols<DP> / 16; ++c) {
    uint32_t xo[16];
    tmem_ld16(ocol + c * 16, xo);
    tmem_wait_ld(xo);
#pragma unroll
    for (int e = 0; e < 16; ++e) xo[e] = __float_as_uint(__uint_as_float(xo[e]) * alpha);
    tmem_st16(ocol + c * 16, xo);
  }
}

// Per key tile: load the row's 128 scores from TMEM into registers (S is then free
// for the next tile's scores), apply scale and biases, take the tile max, move the
// reference if needed, and write P = 2^(y - m) to TMEM for the P·V MMA.
template <int DP, bool BF16, int B2, bool SKIP>
__device__ __forceinline__ void fwd_softmax(const FwdArgs& a, uint8_t* base, const FwdLayout<DP>& lay,
                                            FwdBars* bars, uint32_t tmem, const WaitGuard& g, long long i0,
                                            long long i1) {
  constexpr bool kHasB2 = B2 != kB2None;
  constexpr bool kFold = mask_in_s(DP, BF16, B2);  // the score MMA added the mask
  constexpr bool kRowSum = !kOnes<DP>;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t grp = static_cast<uint32_t>(w >> 2);  // query tile of the item
  const int wq = w & 3;                                 // TMEM lane quadrant
  const int r = wq * 32 + lane;                         // query row within the tile == TMEM lane
  const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t scol = trow + col_s(grp), pcol = trow + col_p(grp), ocol = trow + col_o(grp);
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const float inv_scale = kLog2e / a.scale_log2;  // D^1/2: the pair bias in units of Q·Kᵀ
  const float2 bs2 = make_float2(inv_scale, inv_scale);
  const int S = a.stages, KT = a.QT;
  uint32_t u = 0, grp_it = 0, s = 0, ph = 0;
  float m = 0.0f, l = 0.0f;  // reference max (log2 units); row sum (kept here only without ones columns)
  bool have = false;         // a finite reference exists (until then every P is 0)
  ItemIter cur, prev;
  cur.init(i0, a);
  prev = cur;
  bool ok = true;
  if (grp == 1 && lane == 0) mbar_arrive(smem_u32(&bars->turn[0]));  // query tile 0 goes first
  for (long long item = i0; ok && item < i1; ++item) {
    if (item > i0) {
      prev = cur;
      cur.next(a);
    }
    const bool grp_last = item + 1 == i1 || cur.n == a.N - 1;
    if (B2 == kB2Resident && (item == i0 || cur.n == 0)) {
      if (!mbar_wait_warp_inl(smem_u32(&bars->b2_full), grp_it & 1, g)) { ok = false; break; }
      ++grp_it;
    }
    float m_fin = 0.0f, l_fin = 0.0f;  // the previous item's statistics, for its epilogue
    for (int x = 0; SKIP || x < KT; ++x) {  // with SKIP, up to the tile tagged last
      const bool first = x == 0;
      if (first) {
        m_fin = have ? m : 0.0f;
        l_fin = l;
        have = false;
        m = 0.0f;
        l = 0.0f;
      }
      if (!mbar_wait_warp_inl(smem_u32(&bars->kv_full[s]), ph, g)) { ok = false; break; }
      const uint32_t meta = SKIP ? bars->tile_meta[s] : tile_meta_all(x, KT);
      const int jt = static_cast<int>(meta & 0xffffu);
      const bool last = (meta & kTileLast) != 0;
      if (!mbar_wait_warp_inl(smem_u32(&bars->s_full[grp]), u & 1, g)) { ok = false; break; }
      tc_fence_after();
      const float* b1 = reinterpret_cast<const float*>(base + lay.b1[s]);  // (where the softmax adds the mask)
      const uint8_t* b2t =
          base + (B2 == kB2Resident ? lay.b2r + (grp * KT + jt) * 32768u : lay.b2s[s] + grp * 32768u);
      // S in two 64-column loads: the second is in flight while the first half is scored
      uint32_t ya[64], yb[64];
      uint32_t(&y0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ya[0]);
      uint32_t(&y1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ya[32]);
      uint32_t(&y2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&yb[0]);
      uint32_t(&y3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&yb[32]);
      float mt = -INFINITY;
      tmem_ld64(scol, ya);
      tmem_wait_ld(ya);
      tmem_ld64(scol + 64, yb);
      chunk_scores<BF16, kHasB2, kFold>(y0, b1, b2t, 0, r, sl2, bs2, mt);
      chunk_scores<BF16, kHasB2, kFold>(y1, b1 + 32, b2t, 4, r, sl2, bs2, mt);
      tmem_wait_ld(yb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->s_free[grp]));  // S may be overwritten
      chunk_scores<BF16, kHasB2, kFold>(y2, b1 + 64, b2t + 16384, 0, r, sl2, bs2, mt);
      chunk_scores<BF16, kHasB2, kFold>(y3, b1 + 96, b2t + 16384, 4, r, sl2, bs2, mt);
      if (kFold) mt *= a.scale_log2;  // to the log2 units of the reference max (a positive factor keeps the max)
      __syncwarp();
      if (lane == 0) {  // the stage's bias data are no longer read by this warp
        mbar_arrive(smem_u32(&bars->kv_empty[s]));
        if (B2 == kB2Resident && grp_last && last) mbar_arrive(smem_u32(&bars->b2_empty));
      }
      // The reference moves to the tile max where the row has none yet, or where the
      // tile max passes it by more than the margin (P then stays below 2^8).
      bool resc = false;
      float alpha = 1.0f;
      if (mt != -INFINITY && (!have || mt > m + kRescaleLog2)) {
        resc = have;
        alpha = have ? ex2(m - mt) : 1.0f;
        m = mt;
        have = true;
      }
      // P goes to TMEM once the previous tile's P·V has read it (and, on the first tile
      // of an item, the previous item's O is complete)
      if (!mbar_wait_warp_inl(smem_u32(&bars->p_empty[grp]), (u & 1) ^ 1, g)) { ok = false; break; }
      tc_fence_after();
      if (!mbar_wait_warp_inl(smem_u32(&bars->turn[grp]), u & 1, g)) { ok = false; break; }
      float2 rs = make_float2(0.0f, 0.0f);
      {  // P in two 32-column stores
        uint32_t pp[32];
        uint32_t(&p0)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pp[0]);
        uint32_t(&p1)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pp[16]);
        chunk_probs<BF16, kRowSum, kFold>(y0, sl2, m, p0, rs);
        chunk_probs<BF16, kRowSum, kFold>(y1, sl2, m, p1, rs);
        tmem_st32(pcol, pp);
        chunk_probs<BF16, kRowSum, kFold>(y2, sl2, m, p0, rs);
        // the other group's turn begins with this tile's last quarter (the turns only share
        // out the exponential unit; nothing in either group's data depends on them)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->turn[grp ^ 1]));
        chunk_probs<BF16, kRowSum, kFold>(y3, sl2, m, p1, rs);
        tmem_st32(pcol + 32, pp);
      }
      // The accumulator of the previous tiles (complete: p_empty) is rescaled before this
      // tile's P·V adds to it (that P·V waits for p_full below).
      if (!first && __any_sync(0xffffffffu, resc)) {
        rescale_o<DP>(ocol, alpha);
        l *= alpha;
      }
      if (kRowSum) l += rs.x + rs.y;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[grp]));
      // The previous item's O is complete (p_empty above); this item's first P·V, which
      // overwrites it, waits for the epilogue (o_free).
      if (first && item > i0) fwd_epilogue<DP, BF16>(a, prev, grp, m_fin, l_fin, base, lay, bars, trow, wq, r, lane);
      ++u;
      if (++s == static_cast<uint32_t>(S)) {
        s = 0;
        ph ^= 1;
      }
      if (SKIP && last) break;
    }
  }
  if (ok && u > 0) {
    // the last item: its last P·V
    if (mbar_wait_warp_inl(smem_u32(&bars->p_empty[grp]), ((u - 1) & 1), g)) {
      tc_fence_after();
      fwd_epilogue<DP, BF16>(a, cur, grp, have ? m : 0.0f, l, base, lay, bars, trow, wq, r, lane);
    }
  }
  if (lane == 0) bulk_wait_all();  // this warp's O stores complete before the CTA's smem goes away
}

template <int DP, bool BF16, int B2, bool SKIP>
__global__ void __launch_bounds__(kThreads, 1) evo_fwd_kernel(const __grid_constant__ FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const FwdLayout<DP> lay(B2, a.stages, a.QT, BF16);
  FwdBars* bars = reinterpret_cast<FwdBars*>(base + lay.bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long i0 = static_cast<long long>(blockIdx.x) * a.chunk;
  const long long i1 = i0 + a.chunk < a.items ? i0 + a.chunk : a.items;
  if (threadIdx.x == 0) {
    bars->abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 1);
      mbar_init(smem_u32(&bars->q_empty[s]), 2);  // both MMA threads
      mbar_init(smem_u32(&bars->drain[s]), 1);
      mbar_init(smem_u32(&bars->s_full[s]), 1);
      mbar_init(smem_u32(&bars->s_free[s]), 4);
      mbar_init(smem_u32(&bars->p_full[s]), 4);
      mbar_init(smem_u32(&bars->p_empty[s]), 1);
      mbar_init(smem_u32(&bars->o_free[s]), 4);
      mbar_init(smem_u32(&bars->turn[s]), 4);
    }
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 32);
      mbar_init(smem_u32(&bars->kv_empty[s]), 2 + kSoftmaxWarps);  // both MMA threads, every softmax warp
    }
    mbar_init(smem_u32(&bars->b2_full), 32);
    mbar_init(smem_u32(&bars->b2_empty), kSoftmaxWarps);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&a.tq);
    tma_prefetch_desc(&a.tk);
    tma_prefetch_desc(&a.tv);
    if (B2 != kB2None && a.bias2_mode == kBias2Tma) tma_prefetch_desc(&a.tb2);
    tma_prefetch_desc(&a.tout);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_slot), 512);
    tmem_relinquish();
  }
  if constexpr (kOnes<DP>) {  // the row-sum columns' operand: every element 1.0
    const uint32_t one2 = BF16 ? 0x3F803F80u : 0x3C003C00u;
    uint4* ones = reinterpret_cast<uint4*>(base + lay.ones);
    for (int e = threadIdx.x; e < kTile * DP * 2 / 16; e += kThreads) ones[e] = make_uint4(one2, one2, one2, one2);
    fence_proxy_async_smem();  // seen by the tensor core's reads
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const WaitGuard g{a.wait_ns, a.status, &bars->abort};

  if (warp >= kSoftmaxWarps) {
    setmaxnreg_dec<kRegsOther>();
    if (warp == kProducerWarp) {
      fwd_producer<DP, BF16, B2, SKIP>(a, base, lay, bars, g, lane, i0, i1);
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
      if (lane == 0) fwd_mma<DP, BF16, B2, SKIP>(a, base, lay, bars, tmem, static_cast<uint32_t>(warp - kMmaWarp), g, i0, i1);
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
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
  const FwdLayout<DP> lay(B2, a.stages, a.QT, BF16);
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

// Deepest K/V ring that fits, and whether the pair-bias tiles of one (b, h, pair)
// group can stay resident.  The ring needs two stages (a stage is released by the P·V
// of its tile, issued after the next tile's scores); where two stages of K, V and both
// query tiles' pair-bias tiles do not fit (D = 64), the single-tile kernel runs.
template <int DP, bool BF16>
cudaError_t launch_fwd_d(FwdArgs a, cudaStream_t st) {
  auto fits = [&](int kind, int stages) { return FwdLayout<DP>(kind, stages, a.QT, BF16).total + 1024 <= kMaxSmem; };
  a.NP = (a.QT + 1) / 2;
  a.items = static_cast<long long>(a.B) * a.H * a.N * a.NP;
  if (a.bias2_mode == kBias2None) {
    a.stages = fits(kB2None, 4) ? 4 : 2;
    a.qt_fast = 1;
    return launch_fwd_t<DP, BF16, kB2None>(a, st);
  }
  for (int stages = 3; stages >= 2; --stages) {
    if (fits(kB2Resident, stages)) {
      a.stages = stages;
      a.b2_resident = 1;
      a.qt_fast = 0;
      return launch_fwd_t<DP, BF16, kB2Resident>(a, st);
    }
  }
  // D > 32 with a long pair bias: the single-tile kernel, built for 64 columns only (its tile
  // loads would not fill its stages for another width); with D <= 32 the streamed layout
  // always fits, so anything else is a layout error
  if (!fits(kB2Stream, 2)) return DP == 64 ? launch_fwd_single(a, BF16, st) : cudaErrorInvalidValue;
  a.stages = 2;
  a.b2_resident = 0;
  a.qt_fast = 1;
  return launch_fwd_t<DP, BF16, kB2Stream>(a, st);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int DP, bool bf16, cudaStream_t st) {
  if (a.B <= 0 || a.N <= 0 || a.H <= 0 || a.QT <= 0) return cudaSuccess;
  switch (DP) {
    case 16: return bf16 ? launch_fwd_d<16, true>(a, st) : launch_fwd_d<16, false>(a, st);
    case 32: return bf16 ? launch_fwd_d<32, true>(a, st) : launch_fwd_d<32, false>(a, st);
    case 64: return bf16 ? launch_fwd_d<64, true>(a, st) : launch_fwd_d<64, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace evo
