// evo_host.cu — the C ABI of libevo_attn.so (declared in include/evo_attn.h):
// argument validation, TMA tensor-map construction, workspace carving and
// dispatch to the sm_103a kernels.  The operation is the one defined on the
// web page "DeepSpeed4Science 技术指南：AI4Science 大模型长序列训练与 Evoformer
// 内存高效注意力内核实战" §3.5-§3.7; §3.7 also fixes the validation this layer
// performs (bias1 (B, N, 1, 1, L), bias2 (B, 1, H, L, L), fp16/bf16 inputs,
// device-resident tensors, backward head dimension <= 64).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "evo_attn.h"
#include "evo_internal.h"
#include "evo_ptx.cuh"
#include <cstdio>

namespace evo {

// Fallback device status word: kernels of calls given no status location of their
// own record a bounded wait that ran out here (evo_attn_device_status reads it).
__device__ int g_evo_status = 0;

constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// What made this thread's last call return EVO_ERR_CUDA (evo_attn_last_error_detail).
static thread_local char g_detail[192] = "";
static void set_detail(const char* what, int code, const char* name) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", what, name ? name : "?", code);
}
evo_status_t cuda_fail(const char* what, cudaError_t e) {
  set_detail(what, static_cast<int>(e), cudaGetErrorName(e));
  return EVO_ERR_CUDA;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  int cc_major = 0, cc_minor = 0, sms = 0;
  int* status = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&d, dev]() {
    cudaError_t e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_evo_status);
    d.err = e;
  });
  if (dev_out) *dev_out = dev;
  return &d;
}

// The settings of one call: from its evo_options_t, or the defaults.
struct CallOpts {
  bool skip = false;
  float skip_at = -1.0e4f;
  uint64_t wait_ns = kDefaultWaitNs;
  int* status = nullptr;  // where kernels record a timeout; nullptr = the call's default location
  bool no_db2 = false;
  ProfileEvents prof{{nullptr}, 0};
  // internal (the host-buffer step's row chunks): the pair-bias gradient's n-group size
  // (0: the shape's own rule), the partial planes written to db2_planes (one per group
  // of this call, H planes of L x L each) and not summed
  int db2_group_size = 0;
  float* db2_planes = nullptr;
};

// Reads *o into c; false when the struct is malformed.
bool read_opts(const evo_options_t* o, CallOpts* c) {
  if (!o) return true;
  if (o->size < sizeof(evo_options_t)) return false;
  if (o->flags & ~static_cast<uint32_t>(EVO_OPT_SKIP_MASKED_TILES | EVO_OPT_NO_DBIAS2)) return false;
  if (o->num_events < 0 || (o->num_events > 0 && !o->events)) return false;
  c->skip = (o->flags & EVO_OPT_SKIP_MASKED_TILES) != 0;
  c->skip_at = o->skip_threshold;
  c->no_db2 = (o->flags & EVO_OPT_NO_DBIAS2) != 0;
  if (o->wait_limit_ns) c->wait_ns = o->wait_limit_ns < 1000 ? 1000 : o->wait_limit_ns;
  c->status = o->status;
  c->prof.count = o->num_events > 8 ? 8 : o->num_events;
  for (int i = 0; i < c->prof.count; ++i) c->prof.ev[i] = o->events[i];
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// l2: how far the L2 widens a request beyond the box's bytes.  Tiles of whole contiguous
// rows (pair bias, partial planes) take 256 bytes; one head's rows of a [B,N,L,H,D] tensor
// take none, since the neighbouring heads' bytes a wider fetch brings in are read by other
// work items much later (after eviction when the tensors outgrow L2).
bool encode_t(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz,
              CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  auto fn = tmap_encoder();
  if (!fn) {
    set_detail("cuTensorMapEncodeTiled entry point", 0, "not found");
    return false;
  }
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dt,
                  static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) set_detail("cuTensorMapEncodeTiled", static_cast<int>(r), "CUresult");
  return r == CUDA_SUCCESS;
}
bool encode(CUtensorMap* m, const void* base, bool bf16, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz,
            CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  return encode_t(m, base, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, dims,
                  strides, box, swz, l2);
}

// fp32 pair-bias partial planes [G*B*H][L][L] as 3-D (j, i, plane); box (32, 32, 1), 128B swizzle.
bool map_db2_part(CUtensorMap* m, const void* p, const evo_shape_t& s, int groups) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(s.L), static_cast<cuuint64_t>(s.L),
                        static_cast<cuuint64_t>(groups) * s.B * s.H};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(s.L) * 4, static_cast<cuuint64_t>(s.L) * s.L * 4};
  cuuint32_t box[3] = {32, 32, 1};
  return encode_t(m, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

int padded_dim(int64_t D) { return D <= 16 ? 16 : (D <= 32 ? 32 : 64); }

Rows packed_rows(const evo_shape_t& s) { return {s.L * s.H * s.D, s.H * s.D}; }

// [B,N,L,H,D] with row strides r viewed as 4-D (D, H, L, B*N); box (DP, 1, 128, 1),
// swizzle = 2*DP bytes.
bool map_qkv(CUtensorMap* m, const void* p, const evo_shape_t& s, bool bf16, const Rows& r) {
  const int DP = padded_dim(s.D);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(s.D), static_cast<cuuint64_t>(s.H), static_cast<cuuint64_t>(s.L),
                        static_cast<cuuint64_t>(s.B * s.N)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.D * 2), static_cast<cuuint64_t>(r.l * 2),
                           static_cast<cuuint64_t>(r.bn * 2)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(DP), 1, static_cast<cuuint32_t>(kTile), 1};
  const CUtensorMapSwizzle swz = DP == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : DP == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
  return encode(m, p, bf16, 4, dims, strides, box, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// The same 4-D view with a box of one warp's share of an output tile: (DP/2, 1, 32, 1);
// swizzle = the box row (DP bytes): none for 16, 32B for 32, 64B for 64.
bool map_rows_half(CUtensorMap* m, const void* p, const evo_shape_t& s, bool bf16, const Rows& r) {
  const int DP = padded_dim(s.D);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(s.D), static_cast<cuuint64_t>(s.H), static_cast<cuuint64_t>(s.L),
                        static_cast<cuuint64_t>(s.B * s.N)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.D * 2), static_cast<cuuint64_t>(r.l * 2),
                           static_cast<cuuint64_t>(r.bn * 2)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(DP / 2), 1, 32, 1};
  return encode(m, p, bf16, 4, dims, strides, box,
                DP == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                : DP == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                           : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// The same 4-D view with a box of 32 whole rows: (DP, 1, 32, 1); swizzle = the box row
// (2·DP bytes).
bool map_rows32(CUtensorMap* m, const void* p, const evo_shape_t& s, bool bf16, const Rows& r) {
  const int DP = padded_dim(s.D);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(s.D), static_cast<cuuint64_t>(s.H), static_cast<cuuint64_t>(s.L),
                        static_cast<cuuint64_t>(s.B * s.N)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.D * 2), static_cast<cuuint64_t>(r.l * 2),
                           static_cast<cuuint64_t>(r.bn * 2)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(DP), 1, 32, 1};
  return encode(m, p, bf16, 4, dims, strides, box,
                DP == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                : DP == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B,
                CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// [B,1,H,L,L] viewed as 3-D (key j, query i, B*H).
bool map_bias2(CUtensorMap* m, const void* p, const evo_shape_t& s, bool bf16, int box_j, CUtensorMapSwizzle swz) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(s.L), static_cast<cuuint64_t>(s.L),
                        static_cast<cuuint64_t>(s.B * s.H)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(s.L * 2), static_cast<cuuint64_t>(s.L * s.L * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_j), static_cast<cuuint32_t>(kTile), 1};
  return encode(m, p, bf16, 3, dims, strides, box, swz);
}

// Transposed pair-bias copy [B*H][L][pitch] (pitch = L rounded up to 8) viewed as
// 3-D (query i, key j, B*H); box (64, 128, 1), 128B swizzle.
bool map_b2t(CUtensorMap* m, const void* p, const evo_shape_t& s, bool bf16, int pitch) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(s.L), static_cast<cuuint64_t>(s.L),
                        static_cast<cuuint64_t>(s.B * s.H)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch) * 2, static_cast<cuuint64_t>(s.L) * pitch * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTile), 1};
  return encode(m, p, bf16, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
  const void* p;
  size_t bytes;
};
bool overlap(const Range& a, const Range& b) {
  if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// ---- strided [B,N,L,H,D] tensors (evo_attn_fwd_strided / evo_attn_bwd_strided)

evo_strides_t packed_strides(const evo_shape_t& s) { return {s.N * s.L * s.H * s.D, s.L * s.H * s.D, s.H * s.D}; }

// Strides of extent-1 dimensions address nothing: replace them by the packed values.
evo_strides_t normalised(evo_strides_t t, const evo_shape_t& s) {
  const evo_strides_t p = packed_strides(s);
  if (s.B == 1) t.b = p.b;
  if (s.N == 1) t.n = p.n;
  if (s.L == 1) t.l = p.l;
  return t;
}

// Every stride a positive multiple of 8 elements (16 bytes, the tensor-map rule)
// below 2^36 elements; no two token rows (H*D elements each) overlap: taken in
// order of stride, each dimension's stride covers the whole extent of the
// dimensions inside it; the addressed span stays below 2^44 elements.
bool strides_ok(const evo_strides_t& t, const evo_shape_t& s) {
  struct Dim {
    int64_t ext, str;
  } d[3] = {{s.B, t.b}, {s.N, t.n}, {s.L, t.l}};
  for (const Dim& x : d)
    if (x.str <= 0 || x.str % 8 != 0 || x.str >= (int64_t(1) << 36)) return false;
  auto order = [](Dim& x, Dim& y) {
    if (y.str < x.str) {
      const Dim z = x;
      x = y;
      y = z;
    }
  };
  order(d[0], d[1]);
  order(d[1], d[2]);
  order(d[0], d[1]);
  double need = double(s.H) * double(s.D);
  for (const Dim& x : d) {
    if (x.ext == 1) continue;
    if (double(x.str) < need) return false;
    need = double(x.str) * double(x.ext);
  }
  return need < 17592186044416.0;
}

// Bytes from the tensor's first element to one past its last.
size_t span_bytes(const evo_strides_t& t, const evo_shape_t& s) {
  return size_t((s.B - 1) * t.b + (s.N - 1) * t.n + (s.L - 1) * t.l + s.H * s.D) * 2;
}

// The kernels address (b, n) as one tensor-map dimension of extent B*N: possible
// when B == 1, N == 1, or the batch stride is N times the row stride.  Otherwise
// the call runs batch by batch.
bool merges(const evo_strides_t& t, const evo_shape_t& s) { return s.B == 1 || s.N == 1 || t.b == s.N * t.n; }
Rows rows_of(const evo_strides_t& t, const evo_shape_t& s) { return {s.N == 1 ? t.b : t.n, t.l}; }
bool same_rows(const Rows& x, const Rows& y) { return x.bn == y.bn && x.l == y.l; }

evo_status_t check_shape(const evo_shape_t& s) {
  if (s.B < 1 || s.N < 1 || s.H < 1 || s.L < 1 || s.L > 32768) return EVO_ERR_BAD_SHAPE;
  if (s.D < 8 || s.D > 64 || (s.D % 8) != 0) return EVO_ERR_BAD_SHAPE;
  const int64_t lim = int64_t(1) << 31;
  if (s.B > lim / s.N || s.B > lim / s.H) return EVO_ERR_BAD_SHAPE;  // TMA coordinates are int32
  // element counts must stay far from size_t overflow: B*N*L*H*D and B*H*L*L below 2^44
  const double e1 = double(s.B) * s.N * s.L * s.H * s.D, e2 = double(s.B) * s.H * s.L * s.L;
  if (e1 >= 17592186044416.0 || e2 >= 17592186044416.0) return EVO_ERR_BAD_SHAPE;
  if (double(s.B) * s.N * s.H * ((s.L + kTile - 1) / kTile) >= 9.0e18) return EVO_ERR_BAD_SHAPE;
  return EVO_OK;
}

evo_status_t check_device(DeviceInfo** out) {
  int dev = 0;
  DeviceInfo* d = device_info(&dev);
  if (!d || d->err != cudaSuccess) return d ? cuda_fail("device query", d->err) : EVO_ERR_CUDA;
  if (d->cc_major != 10 || d->cc_minor != 3) return EVO_ERR_ARCH;
  // Make the device's primary context current on this thread: the tensor maps are
  // encoded through the driver API, which needs one (e.g. on a framework's worker
  // thread whose first CUDA call is ours).
  const cudaError_t e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_fail("cudaSetDevice", e);
  *out = d;
  return EVO_OK;
}

size_t qkv_bytes(const evo_shape_t& s) { return size_t(s.B) * s.N * s.L * s.H * s.D * 2; }
size_t lse_bytes(const evo_shape_t& s) { return size_t(s.B) * s.N * s.H * s.L * 4; }
size_t bias1_bytes(const evo_shape_t& s) { return size_t(s.B) * s.N * s.L * 2; }
size_t bias2_bytes(const evo_shape_t& s) { return size_t(s.B) * s.H * s.L * s.L * 2; }
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// n-groups of the deterministic two-stage pair-bias gradient: enough
// (b, h, q-tile, k-tile, group) blocks for two waves over 152 SMs.
// n-groups of the pair-bias partial kernel (one CTA per (b, h, query tile, key tile,
// group)): at least two waves of 152 CTAs, and, among up to four times that many
// groups, the fewest whose CTAs fill the last wave to 95 % (else the fullest last wave),
// so that no SM idles through a nearly empty last wave.
void bwd_groups(const evo_shape_t& s, int* groups, int* group_size) {
  constexpr int64_t kWave = 152;
  const int64_t QT = (s.L + kTile - 1) / kTile;
  const int64_t tiles = s.B * s.H * QT * QT;
  const int64_t n = s.N > 0 ? s.N : 1;
  int64_t g0 = (2 * kWave + tiles - 1) / tiles;
  if (g0 < 1) g0 = 1;
  if (g0 > n) g0 = n;
  int64_t best_g = 0, best_gs = 0;
  double best_eff = -1.0;
  for (int64_t g = g0; g <= 4 * g0 && g <= n; ++g) {
    const int64_t gs = (n + g - 1) / g, ge = (n + gs - 1) / gs;  // groups after rounding the size
    const int64_t ctas = tiles * ge, waves = (ctas + kWave - 1) / kWave;
    const double eff = static_cast<double>(ctas) / static_cast<double>(waves * kWave);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best_g = ge;
      best_gs = gs;
    }
    if (eff >= 0.95) break;
  }
  *groups = static_cast<int>(best_g);
  *group_size = static_cast<int>(best_gs);
}

int b2t_pitch(const evo_shape_t& s) { return static_cast<int>((s.L + 7) / 8 * 8); }

// Backward workspace: delta always; for the per-key-tile kernel, L × DP fp32 dQ
// rows per CTA (at most kMainMaxCtas CTAs) and the skip bits of masked-tile
// skipping; the transposed pair bias wherever a key-major kernel reads it (the
// key-major schedule, or the key-mask gradient pass); the key-mask gradient
// partials when dbias1 is wanted; the pair-bias partial planes whenever there
// is a pair bias.
struct WsLayout {
  BwdPlan plan;
  size_t status, delta, dq_scr, b2t, db1p, db2, skip, total;
  bool can_skip;  // room for the skip bits (per-key-tile schedule, at most 64 key tiles)
};
// has_db2: the call computes the pair-bias gradient (its partial planes)
WsLayout ws_layout(const evo_shape_t& s, bool has_bias2, bool has_db1 = false, bool has_db2 = true) {
  WsLayout w{};
  w.plan = bwd_plan(padded_dim(s.D), static_cast<int>((s.L + kTile - 1) / kTile), has_bias2);
  size_t off = 0;
  w.status = off;  // the call's device status word (evo_attn_bwd_status)
  off += 256;
  w.delta = off;
  off += round256(size_t(s.B) * s.N * s.H * s.L * 4);
  w.dq_scr = off;
  if (w.plan.mode == kBwdMain || w.plan.mode == kBwdKeyMajorStream) {
    const int64_t slices = s.B * s.H * s.N;
    const int64_t ctas = slices < kMainMaxCtas ? slices : kMainMaxCtas;
    off += round256(size_t(ctas) * ((s.L + kTile - 1) / kTile) * kTile * padded_dim(s.D) * 4);
  }
  w.b2t = off;
  if ((w.plan.mode == kBwdKeyMajor || w.plan.mode == kBwdKeyMajorStream || has_db1) && has_bias2)
    off += round256(size_t(s.B) * s.H * s.L * b2t_pitch(s) * 2);
  w.db1p = off;
  if (has_db1) off += round256(size_t(s.B) * s.N * s.H * 2 * s.L * 4);
  w.db2 = off;
  if (has_bias2 && has_db2) {
    int g = 0, gs = 0;
    bwd_groups(s, &g, &gs);
    off += round256(size_t(g) * s.B * s.H * s.L * s.L * 4);
  }
  // masked-tile skipping of the per-key-tile kernel: skip bits [B*N] u64
  const int64_t QT = (s.L + kTile - 1) / kTile;
  w.skip = off;
  w.can_skip = (w.plan.mode == kBwdMain || w.plan.mode == kBwdKeyMajorStream) && QT <= 64;
  if (w.can_skip) off += round256(size_t(s.B) * s.N * 8);
  w.total = off;
  return w;
}

}  // namespace

int num_sms() {
  DeviceInfo* d = device_info(nullptr);
  return (d && d->sms > 0) ? d->sms : 148;
}

// ------------------------------------------------------------ self-test kernel
__global__ void evo_wait_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  const WaitGuard g{limit_ns, status, &abort_flag};
  // Nothing ever arrives on `bar`: the wait runs out and records the timeout.
  mbar_wait(smem_u32(&bar), 0, g);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, cudaStream_t st) {
  evo_wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace evo

using namespace evo;

extern "C" {

int evo_attn_abi_version(void) { return EVO_ATTN_ABI_VERSION; }

const char* evo_status_string(evo_status_t s) {
  switch (s) {
    case EVO_OK: return "ok";
    case EVO_ERR_NULL_POINTER: return "a required pointer is NULL";
    case EVO_ERR_BAD_SHAPE: return "unsupported shape (B,N,H>=1, 1<=L<=32768, D in 8..64 step 8)";
    case EVO_ERR_BAD_DTYPE: return "dtype must be EVO_F16 or EVO_BF16";
    case EVO_ERR_MISALIGNED: return "a pointer is not suitably aligned (16 B tensors, 2 B bias1, 4 B lse, 256 B workspace)";
    case EVO_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than evo_attn_bwd_workspace_bytes()";
    case EVO_ERR_ARCH: return "current device is not compute capability 10.3 (GB300, sm_103a)";
    case EVO_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case EVO_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out; outputs are undefined";
    case EVO_ERR_ALIASING: return "an output buffer overlaps an input buffer";
    case EVO_ERR_BAD_ARGUMENT: return "invalid argument combination";
    case EVO_ERR_SCRATCH_LIMIT:
      return "backward workspace exceeds the fixed 16 MiB scratch of evo_attn_bwd_noalloc; use evo_attn_bwd";
    case EVO_ERR_BAD_LAYOUT:
      return "a stride breaks the layout rules (multiples of 8, rows must not overlap)";
  }
  return "unknown status";
}

evo_status_t evo_attn_fwd(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                          void* out, float* lse, evo_shape_t shape, evo_dtype_t dtype, void* stream) {
  return evo_attn_fwd_opts(q, k, v, bias1, bias2, out, lse, shape, dtype, nullptr, nullptr, stream);
}

evo_status_t evo_attn_fwd_strided(const void* q, const void* k, const void* v, const void* bias1,
                                  const void* bias2, void* out, float* lse, evo_shape_t shape, evo_dtype_t dtype,
                                  const evo_layout_t* layout, void* stream) {
  return evo_attn_fwd_opts(q, k, v, bias1, bias2, out, lse, shape, dtype, layout, nullptr, stream);
}

evo_status_t evo_attn_fwd_opts(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                               void* out, float* lse, evo_shape_t shape, evo_dtype_t dtype,
                               const evo_layout_t* layout, const evo_options_t* opts, void* stream) {
  CallOpts co;
  if (!read_opts(opts, &co)) return EVO_ERR_BAD_ARGUMENT;
  if (co.no_db2) return EVO_ERR_BAD_ARGUMENT;  // a backward-only option
  if (!q || !k || !v || !out || !lse) return EVO_ERR_NULL_POINTER;
  if (dtype != EVO_F16 && dtype != EVO_BF16) return EVO_ERR_BAD_DTYPE;
  evo_status_t st = check_shape(shape);
  if (st != EVO_OK) return st;
  evo_strides_t t[4];  // q, k, v, out
  for (int i = 0; i < 4; ++i) {
    const evo_strides_t* given = layout ? (i == 0 ? &layout->q : i == 1 ? &layout->k : i == 2 ? &layout->v
                                                                                       : &layout->out)
                                        : nullptr;
    t[i] = normalised(given ? *given : packed_strides(shape), shape);
    if (!strides_ok(t[i], shape)) return EVO_ERR_BAD_LAYOUT;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      (bias1 && !aligned(bias1, 2)) || (bias2 && !aligned(bias2, 16)))
    return EVO_ERR_MISALIGNED;
  const Range ins[5] = {{q, span_bytes(t[0], shape)}, {k, span_bytes(t[1], shape)}, {v, span_bytes(t[2], shape)},
                        {bias1, bias1 ? bias1_bytes(shape) : 0}, {bias2, bias2 ? bias2_bytes(shape) : 0}};
  const Range outs[2] = {{out, span_bytes(t[3], shape)}, {lse, lse_bytes(shape)}};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return EVO_ERR_ALIASING;
  if (overlap(outs[0], outs[1])) return EVO_ERR_ALIASING;
  DeviceInfo* dev = nullptr;
  if ((st = check_device(&dev)) != EVO_OK) return st;

  const bool bf16 = dtype == EVO_BF16;
  bool whole = true;
  for (const evo_strides_t& x : t) whole = whole && merges(x, shape);
  evo_shape_t sub = shape;
  sub.B = whole ? shape.B : 1;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  prof_record(&co.prof, 0, cs);
  for (int64_t b = 0; b < shape.B; b += sub.B) {
    const auto at = [&](const void* p, const evo_strides_t& x) {
      return static_cast<const uint8_t*>(p) + size_t(b * x.b) * 2;
    };
    FwdArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!map_qkv(&a.tq, at(q, t[0]), sub, bf16, rows_of(t[0], sub)) ||
        !map_qkv(&a.tk, at(k, t[1]), sub, bf16, rows_of(t[1], sub)) ||
        !map_qkv(&a.tv, at(v, t[2]), sub, bf16, rows_of(t[2], sub)) ||
        !map_rows32(&a.tout, at(out, t[3]), sub, bf16, rows_of(t[3], sub)) ||
        !map_rows_half(&a.tout_half, at(out, t[3]), sub, bf16, rows_of(t[3], sub)))
      return EVO_ERR_CUDA;
    const uint16_t* b2 = bias2 ? static_cast<const uint16_t*>(bias2) + b * shape.H * shape.L * shape.L : nullptr;
    a.bias2_mode = kBias2None;
    if (b2) {
      if (shape.L % 8 == 0) {
        if (!map_bias2(&a.tb2, b2, sub, bf16, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return EVO_ERR_CUDA;
        a.bias2_mode = kBias2Tma;
      } else {
        a.bias2_mode = kBias2Loads;
      }
    }
    a.bias1 = bias1 ? static_cast<const uint16_t*>(bias1) + b * shape.N * shape.L : nullptr;
    a.bias2 = b2;
    a.out = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(out) + size_t(b * t[3].b) * 2);
    a.lse = lse + b * shape.N * shape.H * shape.L;
    a.B = static_cast<int>(sub.B);
    a.N = static_cast<int>(shape.N);
    a.L = static_cast<int>(shape.L);
    a.H = static_cast<int>(shape.H);
    a.D = static_cast<int>(shape.D);
    a.QT = static_cast<int>((shape.L + kTile - 1) / kTile);
    a.NP = (a.QT + 1) / 2;
    a.items = sub.B * shape.N * shape.H * a.NP;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(shape.D)));
    a.tile_skip = co.skip && bias1 && a.QT <= 64;
    a.skip_at = co.skip_at;
    a.wait_ns = co.wait_ns;
    a.status = co.status ? co.status : dev->status;
    const cudaError_t e = launch_fwd(a, padded_dim(shape.D), bf16, cs);
    if (e != cudaSuccess) return cuda_fail("forward launch", e);
  }
  prof_record(&co.prof, 1, cs);
  return EVO_OK;
}

size_t evo_attn_bwd_workspace_bytes(evo_shape_t shape, evo_dtype_t dtype, int flags) {
  if (dtype != EVO_F16 && dtype != EVO_BF16) return 0;
  if (check_shape(shape) != EVO_OK) return 0;
  if (flags & ~(EVO_WS_BIAS2 | EVO_WS_DBIAS1 | EVO_WS_NO_DBIAS2)) return 0;
  const bool b2 = (flags & EVO_WS_BIAS2) != 0, db1 = (flags & EVO_WS_DBIAS1) != 0;
  const bool db2 = (flags & EVO_WS_NO_DBIAS2) == 0;
  // enough for the whole batch at once and for one batch at a time (strided layouts
  // whose batch and row dimensions do not merge)
  evo_shape_t one = shape;
  one.B = 1;
  const size_t whole = ws_layout(shape, b2, db1, db2).total, each = ws_layout(one, b2, db1, db2).total;
  return whole > each ? whole : each;
}

namespace {
// The legacy entry points: default settings, timeouts recorded in the fallback word.
evo_status_t bwd_impl(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                      const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      void* dbias1, void* dbias2, void* workspace, size_t workspace_bytes, evo_shape_t shape,
                      evo_dtype_t dtype, const evo_layout_t* layout, const CallOpts& co, bool fallback_status,
                      void* stream);
}  // namespace

evo_status_t evo_attn_bwd(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                          const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          void* dbias2, void* workspace, size_t workspace_bytes, evo_shape_t shape,
                          evo_dtype_t dtype, void* stream) {
  return bwd_impl(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, nullptr, dbias2, workspace, workspace_bytes,
                  shape, dtype, nullptr, CallOpts{}, true, stream);
}

evo_status_t evo_attn_bwd_ex(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                             const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                             void* dbias1, void* dbias2, void* workspace, size_t workspace_bytes,
                             evo_shape_t shape, evo_dtype_t dtype, void* stream) {
  return bwd_impl(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, dbias1, dbias2, workspace, workspace_bytes,
                  shape, dtype, nullptr, CallOpts{}, true, stream);
}

evo_status_t evo_attn_bwd_strided(const void* q, const void* k, const void* v, const void* bias1,
                                  const void* bias2, const void* out, const float* lse, const void* dout, void* dq,
                                  void* dk, void* dv, void* dbias1, void* dbias2, void* workspace,
                                  size_t workspace_bytes, evo_shape_t shape, evo_dtype_t dtype,
                                  const evo_layout_t* layout, void* stream) {
  return bwd_impl(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, dbias1, dbias2, workspace, workspace_bytes,
                  shape, dtype, layout, CallOpts{}, true, stream);
}

evo_status_t evo_attn_bwd_opts(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                               const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* dbias1, void* dbias2, void* workspace, size_t workspace_bytes,
                               evo_shape_t shape, evo_dtype_t dtype, const evo_layout_t* layout,
                               const evo_options_t* opts, void* stream) {
  CallOpts co;
  if (!read_opts(opts, &co)) return EVO_ERR_BAD_ARGUMENT;
  return bwd_impl(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, dbias1, dbias2, workspace, workspace_bytes,
                  shape, dtype, layout, co, false, stream);
}

evo_status_t evo_attn_bwd_status(const void* workspace, void* stream) {
  if (!workspace) return EVO_ERR_NULL_POINTER;
  if (!aligned(workspace, 256)) return EVO_ERR_MISALIGNED;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return EVO_ERR_CUDA;
  int v = 0;
  const cudaError_t e = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail("status read", e);
  return v == 0 ? EVO_OK : EVO_ERR_DEVICE_TIMEOUT;
}

namespace {
evo_status_t bwd_impl(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                      const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      void* dbias1, void* dbias2, void* workspace, size_t workspace_bytes, evo_shape_t shape,
                      evo_dtype_t dtype, const evo_layout_t* layout, const CallOpts& co, bool fallback_status,
                      void* stream) {
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace) return EVO_ERR_NULL_POINTER;
  if (dtype != EVO_F16 && dtype != EVO_BF16) return EVO_ERR_BAD_DTYPE;
  evo_status_t st = check_shape(shape);
  if (st != EVO_OK) return st;
  if (dbias2 && !bias2) return EVO_ERR_BAD_ARGUMENT;
  if (bias2 && !dbias2 && !co.no_db2) return EVO_ERR_BAD_ARGUMENT;
  if (co.no_db2 && dbias2) return EVO_ERR_BAD_ARGUMENT;
  if (dbias1 && !bias1) return EVO_ERR_BAD_ARGUMENT;
  enum { Q, K, V, O, DO, DQ, DK, DV };
  evo_strides_t t[8];
  for (int i = 0; i < 8; ++i) {
    const evo_strides_t* g = nullptr;
    if (layout) {
      const evo_strides_t* all[8] = {&layout->q,    &layout->k,  &layout->v,  &layout->out,
                                     &layout->dout, &layout->dq, &layout->dk, &layout->dv};
      g = all[i];
    }
    t[i] = normalised(g ? *g : packed_strides(shape), shape);
    if (!strides_ok(t[i], shape)) return EVO_ERR_BAD_LAYOUT;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) ||
      (bias1 && !aligned(bias1, 2)) || (bias2 && !aligned(bias2, 16)) || (dbias2 && !aligned(dbias2, 16)) ||
      (dbias1 && !aligned(dbias1, 2)) || !aligned(workspace, 256))
    return EVO_ERR_MISALIGNED;
  bool whole = true;
  for (const evo_strides_t& x : t) whole = whole && merges(x, shape);
  evo_shape_t sub = shape;
  sub.B = whole ? shape.B : 1;
  // (partial planes written elsewhere take no room in the workspace)
  const WsLayout w = ws_layout(sub, bias2 != nullptr, dbias1 != nullptr, dbias2 != nullptr && !co.db2_planes);
  if (workspace_bytes < w.total) return EVO_ERR_WORKSPACE_TOO_SMALL;
  const Range ins[8] = {{q, span_bytes(t[Q], shape)},      {k, span_bytes(t[K], shape)},
                        {v, span_bytes(t[V], shape)},      {bias1, bias1 ? bias1_bytes(shape) : 0},
                        {bias2, bias2 ? bias2_bytes(shape) : 0}, {out, span_bytes(t[O], shape)},
                        {lse, lse_bytes(shape)},           {dout, span_bytes(t[DO], shape)}};
  const Range outs[6] = {{dq, span_bytes(t[DQ], shape)},
                         {dk, span_bytes(t[DK], shape)},
                         {dv, span_bytes(t[DV], shape)},
                         {dbias2, dbias2 ? bias2_bytes(shape) : 0},
                         {dbias1, dbias1 ? bias1_bytes(shape) : 0},
                         {workspace, w.total}};
  for (int i = 0; i < 6; ++i) {
    for (const Range& r : ins)
      if (overlap(outs[i], r)) return EVO_ERR_ALIASING;
    for (int j = i + 1; j < 6; ++j)
      if (overlap(outs[i], outs[j])) return EVO_ERR_ALIASING;
  }
  DeviceInfo* dev = nullptr;
  if ((st = check_device(&dev)) != EVO_OK) return st;

  const bool bf16 = dtype == EVO_BF16;
  const Rows packed = packed_rows(sub);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (int64_t b = 0; b < shape.B; b += sub.B) {
    const auto at = [&](const void* p, int which) {
      return const_cast<uint16_t*>(reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(p) +
                                                                     size_t(b * t[which].b) * 2));
    };
    const size_t b1_off = size_t(b * shape.N * shape.L), b2_off = size_t(b * shape.H * shape.L * shape.L);
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!map_qkv(&a.tq, at(q, Q), sub, bf16, rows_of(t[Q], sub)) ||
        !map_qkv(&a.tk, at(k, K), sub, bf16, rows_of(t[K], sub)) ||
        !map_qkv(&a.tv, at(v, V), sub, bf16, rows_of(t[V], sub)) ||
        !map_qkv(&a.tdo, at(dout, DO), sub, bf16, rows_of(t[DO], sub)))
      return EVO_ERR_CUDA;
    if (padded_dim(shape.D) <= 32 && (!map_rows_half(&a.tdq, at(dq, DQ), sub, bf16, rows_of(t[DQ], sub)) ||
                                      !map_rows_half(&a.tdk, at(dk, DK), sub, bf16, rows_of(t[DK], sub)) ||
                                      !map_rows_half(&a.tdv, at(dv, DV), sub, bf16, rows_of(t[DV], sub))))
      return EVO_ERR_CUDA;
    a.bias1 = bias1 ? static_cast<const uint16_t*>(bias1) + b1_off : nullptr;
    a.bias2 = bias2 ? static_cast<const uint16_t*>(bias2) + b2_off : nullptr;
    a.bias2_mode = kBias2None;
    if (a.bias2) {
      if (shape.L % 8 == 0) {
        if (!map_bias2(&a.tb2, a.bias2, sub, bf16, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return EVO_ERR_CUDA;
        a.bias2_mode = kBias2Tma;
      } else {
        a.bias2_mode = kBias2Loads;
      }
    }
    a.q = at(q, Q);
    a.out = at(out, O);
    a.dout = at(dout, DO);
    a.lse = lse + b * shape.N * shape.H * shape.L;
    a.dq = at(dq, DQ);
    a.dk = at(dk, DK);
    a.dv = at(dv, DV);
    a.r_out = rows_of(t[O], sub);
    a.r_dout = rows_of(t[DO], sub);
    a.r_dq = rows_of(t[DQ], sub);
    a.r_dk = rows_of(t[DK], sub);
    a.r_dv = rows_of(t[DV], sub);
    a.packed = same_rows(a.r_out, packed) && same_rows(a.r_dout, packed) && same_rows(a.r_dq, packed) &&
               same_rows(a.r_dk, packed) && same_rows(a.r_dv, packed);
    a.dbias2 = dbias2 ? static_cast<uint16_t*>(dbias2) + b2_off : nullptr;
    a.delta = reinterpret_cast<float*>(ws + w.delta);
    a.dq_scr = reinterpret_cast<float*>(ws + w.dq_scr);
    a.db2_part = dbias2 ? reinterpret_cast<float*>(ws + w.db2) : nullptr;
    if (dbias1) {
      a.dbias1 = static_cast<uint16_t*>(dbias1) + b1_off;
      a.db1p = reinterpret_cast<float*>(ws + w.db1p);
    }
    if (bias2 && (w.plan.mode == kBwdKeyMajor || w.plan.mode == kBwdKeyMajorStream || dbias1)) {
      a.b2t = reinterpret_cast<uint16_t*>(ws + w.b2t);
      a.b2t_pitch = b2t_pitch(sub);
      if (!map_b2t(&a.tb2t, a.b2t, sub, bf16, a.b2t_pitch)) return EVO_ERR_CUDA;
    }
    a.B = static_cast<int>(sub.B);
    a.N = static_cast<int>(shape.N);
    a.L = static_cast<int>(shape.L);
    a.H = static_cast<int>(shape.H);
    a.D = static_cast<int>(shape.D);
    a.QT = static_cast<int>((shape.L + kTile - 1) / kTile);
    bwd_groups(sub, &a.groups, &a.group_size);
    if (co.db2_group_size > 0) {
      a.group_size = co.db2_group_size;
      a.groups = static_cast<int>((sub.N + a.group_size - 1) / a.group_size);
    }
    if (co.db2_planes && dbias2) {
      a.db2_part = co.db2_planes;
      a.db2_no_sum = 1;
    }
    if (dbias2 && shape.L % 4 == 0) {
      if (!map_db2_part(&a.tdb2p, a.db2_part, sub, a.groups)) return EVO_ERR_CUDA;
      a.db2p_tma = 1;
    }
    a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(shape.D)));
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(shape.D)));
    if (co.skip && bias1 && w.can_skip) {
      a.tile_skip = 1;
      a.skip_at = co.skip_at;
      a.tskip = reinterpret_cast<unsigned long long*>(ws + w.skip);
    }
    a.wait_ns = co.wait_ns;
    // the call's status word: given, the workspace's own (cleared by the first kernel), or
    // the fallback word
    a.status = co.status ? co.status : (fallback_status ? dev->status : reinterpret_cast<int*>(ws + w.status));
    a.clear_status = !co.status && !fallback_status && b == 0;
    const cudaError_t e = launch_bwd(a, padded_dim(shape.D), bf16, static_cast<cudaStream_t>(stream), &co.prof);
    if (e != cudaSuccess) return cuda_fail("backward launches", e);
  }
  return EVO_OK;
}
}  // namespace

const char* evo_attn_last_error_detail(void) { return g_detail; }

evo_status_t evo_attn_device_status(void* stream) {
  DeviceInfo* dev = device_info(nullptr);
  if (!dev || dev->err != cudaSuccess) return EVO_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return EVO_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_evo_status, sizeof(int)) != cudaSuccess) return EVO_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_evo_status, &zero, sizeof(int)) != cudaSuccess) return EVO_ERR_CUDA;
    return EVO_ERR_DEVICE_TIMEOUT;
  }
  return EVO_OK;
}

evo_status_t evo_attn_selftest_wait_timeout(uint64_t limit_ns, int* status, void* stream) {
  DeviceInfo* dev = nullptr;
  evo_status_t st = check_device(&dev);
  if (st != EVO_OK) return st;
  if (status && !aligned(status, 4)) return EVO_ERR_MISALIGNED;
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
  return launch_wait_selftest(limit_ns, status ? status : dev->status, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? EVO_OK
             : EVO_ERR_CUDA;
}

namespace {
struct ArenaLayout {
  size_t q, k, v, dout, out, dq, dk, dv, b1, b2, db2, db2p, lse, ws, total;
};
// The host-buffer step runs the backward chunk by chunk with a pair bias too when B = 1:
// each chunk writes the pair-bias partial planes of its n-groups (the whole call's
// groups, so that the chunk boundaries fall on group boundaries) into one buffer, summed
// once at the end in the same fixed order as an unchunked call.
bool chunked_db2(const evo_shape_t& s, bool has_b2) { return has_b2 && s.B == 1; }
ArenaLayout arena_layout(const evo_shape_t& s, bool has_b1, bool has_b2) {
  ArenaLayout a{};
  size_t off = 0;
  const size_t nq = round256(qkv_bytes(s));
  size_t* qkv[8] = {&a.q, &a.k, &a.v, &a.dout, &a.out, &a.dq, &a.dk, &a.dv};
  for (size_t* p : qkv) {
    *p = off;
    off += nq;
  }
  a.b1 = off;
  if (has_b1) off += round256(bias1_bytes(s));
  a.b2 = off;
  if (has_b2) off += round256(bias2_bytes(s));
  a.db2 = off;
  if (has_b2) off += round256(bias2_bytes(s));
  a.db2p = off;
  if (chunked_db2(s, has_b2)) {
    int g = 0, gs = 0;
    bwd_groups(s, &g, &gs);
    off += round256(size_t(g) * s.H * s.L * s.L * 4);
  }
  a.lse = off;
  off += round256(lse_bytes(s));
  a.ws = off;
  off += ws_layout(s, has_b2).total;
  a.total = off;
  return a;
}
}  // namespace

size_t evo_attn_step_host_arena_bytes(evo_shape_t shape, evo_dtype_t dtype, int has_bias1, int has_bias2) {
  if (dtype != EVO_F16 && dtype != EVO_BF16) return 0;
  if (check_shape(shape) != EVO_OK) return 0;
  return arena_layout(shape, has_bias1 != 0, has_bias2 != 0).total;
}

evo_status_t evo_attn_step_host(const void* q, const void* k, const void* v, const void* bias1, const void* bias2,
                                const void* dout, void* out, float* lse, void* dq, void* dk, void* dv, void* dbias2,
                                void* arena, size_t arena_bytes, evo_shape_t shape, evo_dtype_t dtype,
                                void* stream) {
  if (!q || !k || !v || !dout || !out || !dq || !dk || !dv || !arena) return EVO_ERR_NULL_POINTER;
  if (dtype != EVO_F16 && dtype != EVO_BF16) return EVO_ERR_BAD_DTYPE;
  evo_status_t st = check_shape(shape);
  if (st != EVO_OK) return st;
  if ((bias2 != nullptr) != (dbias2 != nullptr)) return EVO_ERR_BAD_ARGUMENT;
  if (!aligned(arena, 256)) return EVO_ERR_MISALIGNED;
  const ArenaLayout L = arena_layout(shape, bias1 != nullptr, bias2 != nullptr);
  if (arena_bytes < L.total) return EVO_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* dev = nullptr;
  if ((st = check_device(&dev)) != EVO_OK) return st;
  uint8_t* A = static_cast<uint8_t*>(arena);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);

  // Chunks of rows (b, n0 .. n0+nn) so that copies overlap compute: the host-to-device
  // copies of chunk c+1 (stream ci) run while chunk c computes (the caller's stream),
  // and chunk c-1's results travel back (stream co).  Without a pair bias the backward
  // runs chunk by chunk too; with one it runs once over all rows (its gradient sums
  // over every n), and dQ, dK, dV start back as soon as its main kernel is done.
  // With a pair bias and B = 1 the backward runs in chunks too (whole n-groups of the
  // pair-bias gradient per chunk): four chunks measured best on triangle, many_head and
  // msa_row.  With a pair bias and B > 1 only the forward runs in chunks, and smaller
  // forward launches cost more than the overlap gains past two.
  const bool db2_chunks = chunked_db2(shape, bias2 != nullptr);
  const int64_t sms = dev->sms > 0 ? dev->sms : 148;
  const int64_t slices = shape.B * shape.N * shape.H;
  int64_t target = slices / (2 * sms);
  target = target < 1 ? 1 : (target > 8 ? 8 : target);
  if (db2_chunks && slices >= 4 * sms) target = 4;
  if (bias2 != nullptr && !db2_chunks && target > 2) target = 2;
  int64_t per_b = (target + shape.B - 1) / shape.B;
  if (per_b > shape.N) per_b = shape.N;
  const int64_t nc = (shape.N + per_b - 1) / per_b;  // rows per chunk
  const int64_t chunks_per_b = (shape.N + nc - 1) / nc;
  int64_t chunks = shape.B * chunks_per_b;
  if (chunks > 64) return EVO_ERR_BAD_SHAPE;  // cannot happen: target <= 8 and B * ceil(8 / B) <= 8 + B
  const bool chunk_bwd = bias2 == nullptr || db2_chunks;
  int db2_groups = 0, db2_gs = 0;
  int64_t nc_rows = nc;  // rows per chunk
  if (db2_chunks) {  // whole pair-bias n-groups per chunk
    bwd_groups(shape, &db2_groups, &db2_gs);
    const int64_t gpc = (db2_groups + target - 1) / target;
    nc_rows = gpc * db2_gs;
    if (nc_rows > shape.N) nc_rows = shape.N;
    chunks = (shape.N + nc_rows - 1) / nc_rows;
  }

  struct Res {
    cudaStream_t ci = nullptr, co = nullptr;
    cudaEvent_t ev[4 * 64 + 3] = {};
    int nev = 0;
    ~Res() {  // released once their pending work is done
      for (int i = 0; i < nev; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
      if (ci) cudaStreamDestroy(ci);
      if (co) cudaStreamDestroy(co);
    }
  } r;
  cudaError_t e = cudaStreamCreateWithFlags(&r.ci, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&r.co, cudaStreamNonBlocking);
  const int nev = static_cast<int>(4 * chunks + 3);
  for (int i = 0; e == cudaSuccess && i < nev; ++i) {
    e = cudaEventCreateWithFlags(&r.ev[i], cudaEventDisableTiming);
    r.nev = i + 1;
  }
  if (e != cudaSuccess) return cuda_fail("host step: streams and events", e);
  cudaEvent_t ev_start = r.ev[0], ev_mid = r.ev[1], ev_done = r.ev[2];
  auto ev_in = [&](int64_t c) { return r.ev[3 + 4 * c]; };       // all of the chunk's inputs are up
  auto ev_fwd = [&](int64_t c) { return r.ev[3 + 4 * c + 1]; };
  auto ev_bwd = [&](int64_t c) { return r.ev[3 + 4 * c + 2]; };
  auto ev_fwd_in = [&](int64_t c) { return r.ev[3 + 4 * c + 3]; };  // the forward's inputs are up
  auto ok = [&](cudaError_t x) {
    if (x != cudaSuccess && e == cudaSuccess) e = x;
    return x == cudaSuccess;
  };
  // the arena may still be in use by earlier work on the caller's stream
  ok(cudaEventRecord(ev_start, s));
  ok(cudaStreamWaitEvent(r.ci, ev_start, 0));
  ok(cudaStreamWaitEvent(r.co, ev_start, 0));

  const size_t row_qkv = size_t(shape.L) * shape.H * shape.D * 2, row_b1 = size_t(shape.L) * 2;
  const size_t row_lse = size_t(shape.H) * shape.L * 4;
  auto h2d = [&](size_t off, const void* src, size_t bytes) {
    ok(cudaMemcpyAsync(A + off, src, bytes, cudaMemcpyHostToDevice, r.ci));
  };
  auto d2h = [&](void* dst, size_t off, size_t bytes) {
    ok(cudaMemcpyAsync(dst, A + off, bytes, cudaMemcpyDeviceToHost, r.co));
  };
  const auto hp = [](const void* p, size_t off) { return static_cast<const uint8_t*>(p) + off; };
  const auto hw = [](void* p, size_t off) { return static_cast<uint8_t*>(p) + off; };
  // chunk c: batch b, rows n0 .. n0 + nn
  const int64_t cpb = db2_chunks ? chunks : chunks_per_b, rpc = db2_chunks ? nc_rows : nc;
  auto chunk_rows = [&](int64_t c, int64_t* b, int64_t* n0, int64_t* nn) {
    *b = c / cpb;
    *n0 = (c % cpb) * rpc;
    *nn = shape.N - *n0 < rpc ? shape.N - *n0 : rpc;
  };
  if (bias2) h2d(L.b2, bias2, bias2_bytes(shape));
  for (int64_t c = 0; c < chunks; ++c) {
    int64_t b, n0, nn;
    chunk_rows(c, &b, &n0, &nn);
    const size_t row0 = size_t(b * shape.N + n0), rows = size_t(nn);
    h2d(L.q + row0 * row_qkv, hp(q, row0 * row_qkv), rows * row_qkv);
    h2d(L.k + row0 * row_qkv, hp(k, row0 * row_qkv), rows * row_qkv);
    h2d(L.v + row0 * row_qkv, hp(v, row0 * row_qkv), rows * row_qkv);
    if (bias1) h2d(L.b1 + row0 * row_b1, hp(bias1, row0 * row_b1), rows * row_b1);
    ok(cudaEventRecord(ev_fwd_in(c), r.ci));  // the forward need not wait for dO
    h2d(L.dout + row0 * row_qkv, hp(dout, row0 * row_qkv), rows * row_qkv);
    ok(cudaEventRecord(ev_in(c), r.ci));
  }
  for (int64_t c = 0; c < chunks && e == cudaSuccess && st == EVO_OK; ++c) {
    int64_t b, n0, nn;
    chunk_rows(c, &b, &n0, &nn);
    const size_t row0 = size_t(b * shape.N + n0), rows = size_t(nn);
    const evo_shape_t sub{1, nn, shape.L, shape.H, shape.D};
    uint8_t* cq = A + L.q + row0 * row_qkv;
    uint8_t* ck = A + L.k + row0 * row_qkv;
    uint8_t* cv = A + L.v + row0 * row_qkv;
    uint8_t* cout = A + L.out + row0 * row_qkv;
    uint8_t* cdo = A + L.dout + row0 * row_qkv;
    const void* cb1 = bias1 ? A + L.b1 + row0 * row_b1 : nullptr;
    const void* cb2 = bias2 ? A + L.b2 + size_t(b) * shape.H * shape.L * shape.L * 2 : nullptr;
    float* clse = reinterpret_cast<float*>(A + L.lse + row0 * row_lse);
    ok(cudaStreamWaitEvent(s, ev_fwd_in(c), 0));
    st = evo_attn_fwd(cq, ck, cv, cb1, cb2, cout, clse, sub, dtype, stream);
    if (st != EVO_OK) break;
    ok(cudaEventRecord(ev_fwd(c), s));
    if (chunk_bwd) ok(cudaStreamWaitEvent(s, ev_in(c), 0));  // dO of this chunk
    if (chunk_bwd && !db2_chunks) {
      st = evo_attn_bwd(cq, ck, cv, cb1, nullptr, cout, clse, cdo, A + L.dq + row0 * row_qkv,
                        A + L.dk + row0 * row_qkv, A + L.dv + row0 * row_qkv, nullptr, A + L.ws, arena_bytes - L.ws,
                        sub, dtype, stream);
      if (st != EVO_OK) break;
      ok(cudaEventRecord(ev_bwd(c), s));
    } else if (db2_chunks) {  // this chunk's n-groups of pair-bias partials, summed after the last chunk
      CallOpts co;
      co.db2_group_size = db2_gs;
      co.db2_planes = reinterpret_cast<float*>(A + L.db2p) + size_t(n0 / db2_gs) * shape.H * shape.L * shape.L;
      st = bwd_impl(cq, ck, cv, cb1, cb2, cout, clse, cdo, A + L.dq + row0 * row_qkv, A + L.dk + row0 * row_qkv,
                    A + L.dv + row0 * row_qkv, nullptr, A + L.db2, A + L.ws, arena_bytes - L.ws, sub, dtype, nullptr,
                    co, true, stream);
      if (st != EVO_OK) break;
      ok(cudaEventRecord(ev_bwd(c), s));
    }
    ok(cudaStreamWaitEvent(r.co, ev_fwd(c), 0));
    d2h(hw(out, row0 * row_qkv), L.out + row0 * row_qkv, rows * row_qkv);
    if (lse) d2h(hw(lse, row0 * row_lse), L.lse + row0 * row_lse, rows * row_lse);
    if (chunk_bwd) {
      ok(cudaStreamWaitEvent(r.co, ev_bwd(c), 0));
      d2h(hw(dq, row0 * row_qkv), L.dq + row0 * row_qkv, rows * row_qkv);
      d2h(hw(dk, row0 * row_qkv), L.dk + row0 * row_qkv, rows * row_qkv);
      d2h(hw(dv, row0 * row_qkv), L.dv + row0 * row_qkv, rows * row_qkv);
    }
  }
  if (db2_chunks && e == cudaSuccess && st == EVO_OK) {  // the pair-bias gradient: every group's planes
    BwdArgs sa;
    std::memset(&sa, 0, sizeof(sa));
    sa.B = 1;
    sa.N = static_cast<int>(shape.N);
    sa.H = static_cast<int>(shape.H);
    sa.L = static_cast<int>(shape.L);
    sa.groups = db2_groups;
    sa.db2_part = reinterpret_cast<float*>(A + L.db2p);
    sa.dbias2 = reinterpret_cast<uint16_t*>(A + L.db2);
    ok(launch_bwd_db2_sum(sa, dtype == EVO_BF16, s));
    ok(cudaEventRecord(ev_mid, s));
    ok(cudaStreamWaitEvent(r.co, ev_mid, 0));
    d2h(dbias2, L.db2, bias2_bytes(shape));
  }
  if (!chunk_bwd && e == cudaSuccess && st == EVO_OK) {
    ok(cudaStreamWaitEvent(s, ev_in(chunks - 1), 0));  // every chunk's dO (the copies run in order)
    CallOpts co;
    co.prof.count = 6;
    co.prof.ev[5] = ev_mid;  // recorded once the main backward kernel is done
    st = bwd_impl(A + L.q, A + L.k, A + L.v, bias1 ? A + L.b1 : nullptr, A + L.b2, A + L.out,
                  reinterpret_cast<const float*>(A + L.lse), A + L.dout, A + L.dq, A + L.dk, A + L.dv, nullptr,
                  A + L.db2, A + L.ws, arena_bytes - L.ws, shape, dtype, nullptr, co, true, stream);
    if (st == EVO_OK) {
      ok(cudaEventRecord(ev_bwd(0), s));
      const size_t nq = qkv_bytes(shape);
      ok(cudaStreamWaitEvent(r.co, ev_mid, 0));
      d2h(dq, L.dq, nq);
      d2h(dk, L.dk, nq);
      d2h(dv, L.dv, nq);
      ok(cudaStreamWaitEvent(r.co, ev_bwd(0), 0));
      d2h(dbias2, L.db2, bias2_bytes(shape));
    }
  }
  // the caller's stream completes with the last copy back
  ok(cudaEventRecord(ev_done, r.co));
  ok(cudaStreamWaitEvent(s, ev_done, 0));
  if (st != EVO_OK) return st;
  if (e != cudaSuccess) return cuda_fail("host step: copies", e);
  return EVO_OK;
}

}  // extern "C"
