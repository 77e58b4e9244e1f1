// evo_internal.h — launch interfaces between the C-ABI host layer
// (evo_host.cu) and the kernel translation units.  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace evo {

constexpr int kTile = 128;  // queries (and keys) per tile

// Element strides of the (b·n) and token dimensions of one [B,N,L,H,D] tensor
// whose H·D elements per token are packed: element (bn, l, h, d) sits at
// bn·bn_stride + l·l_stride + h·D + d.  Packed: bn = L·H·D, l = H·D.
struct Rows {
  long long bn, l;
};

// How the pair bias reaches shared memory.
enum Bias2Mode : int { kBias2None = 0, kBias2Tma = 1, kBias2Loads = 2 };

struct FwdArgs {
  CUtensorMap tq, tk, tv;   // 4-D (D, H, L, B*N) views with the tensors' own strides, box (DP, 1, 128, 1)
  CUtensorMap tb2;          // 3-D [B*H][L][L] view, box (64, 128, 1), 128B swizzle (kBias2Tma)
  CUtensorMap tout;         // O as the 4-D view with box (DP, 1, 32, 1): one softmax warp's 32 rows
  CUtensorMap tout_half;    // the same with box (DP/2, 1, 32, 1) (single-tile forward)
  const uint16_t* bias1;    // [B,N,L] or nullptr
  const uint16_t* bias2;    // [B,H,L,L] or nullptr
  uint16_t* out;            // [B,N,L,H,D]
  float* lse;               // [B,N,H,L]
  int B, N, L, H, D;
  int QT;                   // ceil(L / 128)
  int NP;                   // ceil(QT / 2): pairs of query tiles
  long long items;          // B*H*NP*N work items (query-tile pairs), ordered (b, h, pair, n), or with
                            // qt_fast (b, h, n, pair)
  int qt_fast;              // no resident pair bias: an (n, h)'s pairs run back to back (K/V reuse in L2)
  long long chunk;          // consecutive items per CTA
  int stages;               // depth of the K/V ring (2..4)
  int b2_resident;          // pair-bias tiles of the current (b, h, q-tile) kept in smem
  float scale_log2;         // D^-1/2 * log2(e)
  int bias2_mode;
  int tile_skip;            // skip key tiles whose every key mask is <= skip_at (QT <= 64 only)
  float skip_at;
  uint64_t wait_ns;
  int* status;
};

struct BwdArgs {
  CUtensorMap tq, tk, tv, tdo;  // 4-D views like the forward, box (DP, 1, 128, 1)
  CUtensorMap tb2;              // 3-D [B*H][L][L] view, box (64, 128, 1), 128B swizzle
  CUtensorMap tb2t;             // key-major kernel: the transposed copy b2t, same box and swizzle
  CUtensorMap tdq, tdk, tdv;    // key-major kernel: output views, box (DP/2, 1, 32, 1) = one warp's share
  CUtensorMap tdb2p;            // fp32 partial planes as 3-D (j, i, G*B*H), box (32, 32, 1), 128B swizzle
  const uint16_t* q;
  const uint16_t* out;
  const uint16_t* dout;
  const uint16_t* bias1;
  const uint16_t* bias2;
  const float* lse;
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  uint16_t* dbias2;
  Rows r_out, r_dout;       // row strides of the plain (non-TMA) reads of O and dO
  Rows r_dq, r_dk, r_dv;    // row strides of the plain writes of dQ, dK, dV
  int packed;               // all five of the above are packed [B*N][L][H*D]
  float* delta;             // workspace [B,N,H,L]
  float* dq_scr;            // workspace: per-key-tile kernel, QT × 128 × DP fp32 dQ values per CTA
  float* db2_part;          // workspace [G][B,H,L,L]
  uint16_t* dbias1;         // [B,N,L] or nullptr
  float* db1p;              // workspace [B*N*H][2][L]: key-mask gradient partials (per key half of the queries)
  uint16_t* b2t;            // workspace [B,H,L,b2t_pitch]: b2t[bh][j][i] = bias2[bh][i][j] (key-major kernel)
  int b2t_pitch;            // L rounded up to a multiple of 8 (16-byte rows for TMA)
  int B, N, L, H, D;
  int QT;
  int groups;               // G: n-groups of the pair-bias gradient
  int group_size;           // ceil(N / G)
  long long items;          // main kernel: B*H*N whole (b, h, n) slices
  long long chunk;          // main kernel: consecutive slices per CTA
  int q_stages;             // main kernel: depth of the Q/dO ring
  int pds_bufs;             // main kernel: P and dS shared-memory buffers (1 or 2)
  int kv_bufs;              // main kernel: K/V buffers (2: the next key tile loads ahead; 1)
  int part_stages;          // pair-bias partial kernel: depth of its ring
  int db2p_tma;             // pair-bias partial kernel: tile stores through tdb2p (L % 4 == 0)
  int db2_no_sum;           // pair-bias gradient: write the partial planes only (the caller sums them)
  // Masked key-tile skipping in the per-key-tile kernel (tile_skip; QT <= 64): it skips
  // the key tiles of each slice whose every key mask is <= skip_at (rows with no kept key
  // skip nothing); dK and dV of the skipped key tiles are written as zeros beforehand.
  int tile_skip;
  float skip_at;
  unsigned long long* tskip;  // workspace [B*N]: key tiles of each row to skip, as bits
  float scale;              // D^-1/2
  float scale_log2;         // D^-1/2 * log2(e)
  int bias2_mode;
  uint64_t wait_ns;
  int* status;
  int clear_status;         // the first kernel zeroes *status (the workspace's own status word)
};

// Caller-owned CUDA events recorded around the library's launches (profiling hook).
struct ProfileEvents {
  void* ev[8];
  int count;
};
// Under stream capture the record must be external to become a timestamped
// event-record node of the graph (a plain record would only become a
// dependency edge); outside capture the external flag is invalid.
inline void prof_record(const ProfileEvents* p, int idx, cudaStream_t st) {
  if (!p || idx >= p->count || !p->ev[idx]) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
  const cudaEvent_t ev = static_cast<cudaEvent_t>(p->ev[idx]);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}

// At most this many CTAs run the per-key-tile backward kernel; the workspace holds
// L × DP fp32 dQ rows for each.
constexpr int kMainMaxCtas = 256;

// Raise a kernel's dynamic shared-memory limit once per device (so that later
// launches, including those under stream capture, issue nothing but the launch).
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kern, size_t bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// Which backward kernel runs for a shape (shared by workspace sizing and launch):
// key-major slice kernel, query-major slice kernel (both keep dQ in TMEM), or the
// per-key-tile kernel with an fp32 dQ accumulator in the workspace.
enum BwdMode : int { kBwdKeyMajor = 0, kBwdSlice = 1, kBwdMain = 2, kBwdKeyMajorStream = 3 };
struct BwdPlan {
  int mode;
  int q_stages;
};
BwdPlan bwd_plan(int DP, int QT, bool has_b2);
int kmajor_q_stages(int DP, int QT, bool has_b2);
int kmajor_stream_q_stages(int DP, bool has_b2);
cudaError_t launch_bwd_kmajor(const BwdArgs& a, int DP, bool bf16, bool has_b2, bool dq_stream, cudaStream_t st);
// The pair-bias gradient's fixed-order sum over a.groups partial planes at a.db2_part.
cudaError_t launch_bwd_db2_sum(const BwdArgs& a, bool bf16, cudaStream_t st);
// Key-mask gradient partials (a.db1p) by the key-major score recompute alone, for the
// schedules whose main kernel does not produce them; then the fixed-order sum into a.dbias1.
cudaError_t launch_bwd_db1_partials(const BwdArgs& a, int DP, bool bf16, bool has_b2, cudaStream_t st);
cudaError_t launch_bwd_db1_sum(const BwdArgs& a, bool bf16, cudaStream_t st);

int num_sms();
cudaError_t launch_fwd(const FwdArgs& a, int DP, bool bf16, cudaStream_t st);
// The single-query-tile forward (DP = 64 only), for the shapes the paired kernel cannot fit.
cudaError_t launch_fwd_single(const FwdArgs& a, bool bf16, cudaStream_t st);
cudaError_t launch_bwd(const BwdArgs& a, int DP, bool bf16, cudaStream_t st, const ProfileEvents* prof);
cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, cudaStream_t st);

}  // namespace evo
