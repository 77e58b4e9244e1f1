// evo_micro.cu — throughput microbenchmarks behind the kernels' design choices
// (not part of the attention library: built into its own libevo_micro.so and
// run by `python bench.py --micro`).
//
//  * exponentials: sustained rate of the special-function unit for
//    ex2.approx.ftz.f32, ex2.approx.f16x2 and ex2.approx.ftz.bf16x2, of the
//    FMA-pipe polynomial 2^x used to offload part of the softmax exponentials,
//    scalar and packed f32x2, and of plain fma / fma.f32x2 for scale;
//  * tcgen05.mma issue cost: cycles per kind::f16 instruction (M = 128,
//    K = 16) with both operands in shared memory (SS) or A in tensor memory
//    (TS), for N = 32 .. 256.
//
// Every kernel records clock64() deltas per block, so the rates come out per SM
// clock independently of the clock the GPU ran at.  All waits are bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../evo_ptx.cuh"

#define EVO_MICRO_API extern "C" __attribute__((visibility("default")))

namespace {

using namespace evo;

// ---------------------------------------------------------------- exponentials
constexpr int kChains = 8;  // independent dependency chains per thread

__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm volatile("{\n\t.reg .b32 t;\n\tneg.f16x2 t, %1;\n\tex2.approx.f16x2 %0, t;\n\t}" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
  uint32_t y;
  asm volatile("{\n\t.reg .b32 t;\n\tneg.bf16x2 t, %1;\n\tex2.approx.ftz.bf16x2 %0, t;\n\t}" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ float ex2_neg(float x) {
  float y;
  asm volatile("{\n\t.reg .f32 t;\n\tneg.f32 t, %1;\n\tex2.approx.ftz.f32 %0, t;\n\t}" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA pipe: x = j + f with j = round(x) (the 1.5·2^23 rounding
// trick), f in [-1/2, 1/2]; 2^f by a degree-3 polynomial fitted for minimal
// relative error (coefficients from fit_exp2_poly.py in this directory's
// parent; max relative error 7.5e-5); 2^j added to the exponent field.
// Valid for x >= -125 (callers clamp), exact powers of two aside.
constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
constexpr float kP0 = 0.9999281167984009f, kP1 = 0.6932609677314758f, kP2 = 0.24261054396629333f,
                kP3 = 0.05517132207751274f;
__device__ __forceinline__ float exp2_poly(float x) {
  x = fmaxf(x, -125.0f);
  const float t = x + kRound;
  const float f = x - (t - kRound);
  float p = fmaf(kP3, f, kP2);
  p = fmaf(p, f, kP1);
  p = fmaf(p, f, kP0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  x.x = fmaxf(x.x, -125.0f);
  x.y = fmaxf(x.y, -125.0f);
  const float2 r = make_float2(kRound, kRound), nr = make_float2(-kRound, -kRound);
  const float2 t = add2(x, r);
  const float2 f = fma2(add2(t, nr), make_float2(-1.0f, -1.0f), x);
  float2 p = fma2(make_float2(kP3, kP3), f, make_float2(kP2, kP2));
  p = fma2(p, f, make_float2(kP1, kP1));
  p = fma2(p, f, make_float2(kP0, kP0));
  return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                     __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}

enum ExpKind : int {
  kEx2F32 = 0,     // ex2.approx.ftz.f32 (1 exp / instruction)
  kEx2F16x2 = 1,   // ex2.approx.f16x2 (2 exps / instruction)
  kEx2BF16x2 = 2,  // ex2.approx.ftz.bf16x2 (2 exps / instruction)
  kPoly = 3,       // FMA-pipe polynomial, scalar
  kPoly2 = 4,      // FMA-pipe polynomial, packed f32x2
  kFma = 5,        // fma.rn.f32 (1 op / instruction)
  kFma2 = 6,       // fma.rn.f32x2 (2 ops / instruction)
  kMix31 = 7,      // 3 ex2.f32 : 1 packed polynomial pair (the softmax offload mix)
};

template <int K>
__global__ void __launch_bounds__(512, 4) micro_exp(float* sink, long long* cyc, int iters) {
  float x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = 0.25f + 0.01f * ((threadIdx.x + c) & 15);
  __syncthreads();
  const long long t0 = clock64();
#pragma unroll 4
  for (int i = 0; i < iters; ++i) {  // unrolled so that loop overhead stays small next to 32 ops
    if constexpr (K == kEx2F32) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) x[c] = ex2_neg(x[c]);
    } else if constexpr (K == kEx2F16x2 || K == kEx2BF16x2) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) {
        uint32_t v = __float_as_uint(x[c]);
        v = K == kEx2F16x2 ? ex2_f16x2(v) : ex2_bf16x2(v);
        x[c] = __uint_as_float(v);
      }
    } else if constexpr (K == kPoly) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) x[c] = exp2_poly(-x[c]);
    } else if constexpr (K == kPoly2) {
#pragma unroll
      for (int c = 0; c < kChains; c += 2) {
        const float2 r = exp2_poly2(make_float2(-x[c], -x[c + 1]));
        x[c] = r.x;
        x[c + 1] = r.y;
      }
    } else if constexpr (K == kFma) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) x[c] = fmaf(x[c], 0.999f, 0.001f);
    } else if constexpr (K == kFma2) {
#pragma unroll
      for (int c = 0; c < kChains; c += 2) {
        const float2 r = fma2(make_float2(x[c], x[c + 1]), make_float2(0.999f, 0.999f), make_float2(0.001f, 0.001f));
        x[c] = r.x;
        x[c + 1] = r.y;
      }
    } else {  // kMix31: chains 0..5 on the SFU, 6..7 by the packed polynomial
#pragma unroll
      for (int c = 0; c < 6; ++c) x[c] = ex2_neg(x[c]);
      const float2 r = exp2_poly2(make_float2(-x[6], -x[7]));
      x[6] = r.x;
      x[7] = r.y;
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c];
  if (s == 12345.0f) sink[threadIdx.x] = s;  // keeps the chains live
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// ---------------------------------------------------------------- MMA issue cost
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s bound on the completion wait

struct MmaSmem {
  alignas(1024) uint8_t a[128 * 64];  // 128 rows x 64 bytes, 64B swizzle
  alignas(1024) uint8_t b[256 * 64];  // up to 256 rows x 64 bytes
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
};

// One thread issues `reps` MMAs (M = 128, N, K = 16; reps a multiple of 16),
// round robin over ACCS independent accumulators (ACCS * N <= 256 columns), in
// straight-line groups of 16 with compile-time addresses so that the issue loop
// itself costs next to nothing; the block reports the cycles from the first issue
// to the completion of the last.  Operand contents are whatever shared/tensor
// memory holds: only time matters.
template <int N, bool TS, int ACCS>
__global__ void __launch_bounds__(128, 1) micro_mma(long long* cyc, int reps, int* status) {
  __shared__ MmaSmem sm;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(smem_u32(&sm.done), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t id = idesc_f16(128, N, true, false, false);
    const uint64_t ad = smem_desc(smem_u32(sm.a), 16, 8 * 64, kSwizzle64B);
    const uint64_t bd = smem_desc(smem_u32(sm.b), 16, 8 * 64, kSwizzle64B);
    const long long t0 = clock64();
#pragma unroll 1
    for (int r = 0; r < reps; r += 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t k = i & 1;  // alternate the two K = 16 slices of the 32-wide rows
        const uint32_t d = tmem + static_cast<uint32_t>((i % ACCS) * N);
        const uint32_t acc = (r > 0 || i >= ACCS) ? 1u : 0u;
        if (TS)
          umma_ts(d, tmem + 256 + k * 8, bd + k * 2, id, acc);
        else
          umma_ss(d, ad + k * 2, bd + k * 2, id, acc);
      }
    }
    umma_commit(smem_u32(&sm.done));
    WaitGuard g{kWaitNs, status, &sm.abort};
    mbar_wait(smem_u32(&sm.done), 0, g);
    const long long t1 = clock64();
    cyc[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- tensor-memory loads
// Four warps (one per TMEM lane quadrant) each run `reps` rounds of `per_wait`
// tcgen05.ld.32x32b.x32 loads followed by one tcgen05.wait::ld; the block reports the
// cycles of warp 0 (so cycles / reps is the cost of a round: latency when per_wait = 1).
template <int PW>
__global__ void __launch_bounds__(128, 1) micro_tmem_ld(long long* cyc, int reps, float* sink) {
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    tmem_alloc(smem_u32(&slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot + (static_cast<uint32_t>(warp * 32) << 16);
  float acc = 0.0f;
  __syncwarp();
  const long long t0 = clock64();
#pragma unroll 1
  for (int r = 0; r < reps; ++r) {
    uint32_t x[PW][32];
#pragma unroll
    for (int q = 0; q < PW; ++q) tmem_ld32(tmem + q * 32 + (r & 1) * 128, x[q]);
#pragma unroll
    for (int q = 0; q < PW; ++q) tmem_wait_ld(x[q]);
#pragma unroll
    for (int q = 0; q < PW; ++q)
#pragma unroll
      for (int e = 0; e < 32; e += 8) acc += __uint_as_float(x[q][e]);  // compile-time indices only
  }
  const long long t1 = clock64();
  if (acc == 12345.0f) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(slot, 512);
  }
}

// The operand forms of the attention kernels' small-N MMAs (M = 128, N = 32, K = 16),
// 16 per round into one accumulator, from one thread:
//   FORM 0  A from TMEM, B MN-major 64B swizzle (rows of 32 bf16)   — forward O += P V
//   FORM 1  A MN-major 128B swizzle, B MN-major 64B swizzle           — backward dV, dK
//   FORM 2  A K-major 128B swizzle, B MN-major 64B swizzle            — backward dQ
//   FORM 3  A K-major 64B swizzle, B K-major 64B swizzle              — reference (both K-major)
struct FormSmem {
  alignas(1024) uint8_t a[128 * 256];  // a 128 x 128 bf16 tile (two 64-column halves of 128B rows)
  alignas(1024) uint8_t b[128 * 64];   // a 128 x 32 bf16 tile (rows of 64 bytes)
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
};
template <int FORM>
__global__ void __launch_bounds__(128, 1) micro_form(long long* cyc, int reps, int* status) {
  extern __shared__ uint8_t dyn[];
  FormSmem& sm = *reinterpret_cast<FormSmem*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(smem_u32(&sm.done), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t RB = 64, kTile = 128;
    constexpr uint32_t id = FORM == 0 ? idesc_f16(128, 32, true, false, true)
                          : FORM == 1 ? idesc_f16(128, 32, true, true, true)
                          : FORM == 2 ? idesc_f16(128, 32, true, false, true)
                                      : idesc_f16(128, 32, true, false, false);
    const uint32_t a_addr = smem_u32(sm.a), b_addr = smem_u32(sm.b);
    const long long t0 = clock64();
#pragma unroll 1
    for (int r = 0; r < reps; r += 16) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int kk = k & 7;
        const uint32_t acc = (r > 0 || k > 0) ? 1u : 0u;
        if (FORM == 0) {
          const uint64_t bd = smem_desc(b_addr, kTile * RB, 8 * RB, kSwizzle64B) + kk * 16 * RB / 16;
          umma_ts(tmem, tmem + 256 + kk * 8, bd, id, acc);
        } else if (FORM == 1) {
          const uint64_t ad = smem_desc(a_addr + kk * 16 * 128, 16384, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(b_addr + kk * 16 * RB, kTile * RB, 8 * RB, kSwizzle64B);
          umma_ss(tmem, ad, bd, id, acc);
        } else if (FORM == 2) {
          const uint64_t ad = smem_desc(a_addr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(b_addr + kk * 16 * RB, kTile * RB, 8 * RB, kSwizzle64B);
          umma_ss(tmem, ad, bd, id, acc);
        } else {
          const uint64_t ad = smem_desc(a_addr, 16, 8 * 64, kSwizzle64B) + (k & 1) * 2;
          const uint64_t bd = smem_desc(b_addr, 16, 8 * 64, kSwizzle64B) + (k & 1) * 2;
          umma_ss(tmem, ad, bd, id, acc);
        }
      }
    }
    umma_commit(smem_u32(&sm.done));
    WaitGuard g{kWaitNs, status, &sm.abort};
    mbar_wait(smem_u32(&sm.done), 0, g);
    cyc[blockIdx.x] = clock64() - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// 32 lanes x 64 columns in one load, and its wait tied to the 64 registers.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63]) : : "memory");
}

// The forward's P·V MMA form (A = P from TMEM, B = V MN-major 64B, N = 32, or 48 with
// a second B atom standing for the ones columns) issued by one thread while eight
// other warps load from / store to TMEM, or use shared memory, or the MUFU, as the
// softmax warps do: how much each kind of traffic slows the MMAs.
// MODE: 0 none, 1 TMEM loads (4 x32 per wait), 2 TMEM stores (4 x16 per wait),
// 3 loads then stores, 4 shared-memory loads and stores, 5 ex2 chains, 6 TMEM loads
// (2 x64 per wait), 7 TMEM loads (8 x16 per wait).  ccyc: the first traffic warp's
// own loop time.
struct ContendSmem {
  alignas(1024) uint8_t a[128 * 256];
  alignas(1024) uint8_t b[128 * 64];
  alignas(1024) uint8_t ones[128 * 64];
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
};

template <int MODE, int N, bool SS>
__global__ void __launch_bounds__(384, 1) micro_contend(long long* cyc, long long* ccyc, int reps, int creps,
                                                        float* sink, int* status) {
  extern __shared__ uint8_t dyn[];
  ContendSmem& sm = *reinterpret_cast<ContendSmem*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(smem_u32(&sm.done), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t RB = 64, kTile = 128;
    constexpr uint32_t id = idesc_f16(128, N, true, false, true);
    const uint32_t a_addr = smem_u32(sm.a), b_addr = smem_u32(sm.b);
    const uint32_t lbo = N > 32 ? smem_u32(sm.ones) - b_addr : kTile * RB;
    const long long t0 = clock64();
#pragma unroll 1
    for (int r = 0; r < reps; r += 16) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int kk = k & 7;
        const uint64_t bd = smem_desc(b_addr, lbo, 8 * RB, kSwizzle64B) + kk * 16 * RB / 16;
        if (SS) {  // A = a 128 x 128 K-major tile, 128B swizzle (two 64-key halves)
          const uint64_t ad = smem_desc(a_addr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          umma_ss(tmem, ad, bd, id, (r > 0 || k > 0) ? 1u : 0u);
        } else {
          umma_ts(tmem, tmem + 256 + kk * 8, bd, id, (r > 0 || k > 0) ? 1u : 0u);
        }
      }
    }
    umma_commit(smem_u32(&sm.done));
    WaitGuard g{kWaitNs, status, &sm.abort};
    mbar_wait(smem_u32(&sm.done), 0, g);
    cyc[blockIdx.x] = clock64() - t0;
  } else if (warp >= 4 && MODE != 0) {
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t half = static_cast<uint32_t>((warp >> 3) & 1);  // two warps per lane quadrant
    float acc = 0.0f;
    const long long c0 = clock64();
#pragma unroll 1
    for (int it = 0; it < creps; ++it) {
      if (MODE == 6) {
        uint32_t x0[64], x1[64];
        const uint32_t c = trow + 64 + half * 64;
        tmem_ld64(c, x0);
        tmem_ld64(c, x1);
        tmem_wait_ld64(x0);
        tmem_wait_ld64(x1);
#pragma unroll
        for (int e = 0; e < 64; ++e) acc += __uint_as_float(x0[e]) + __uint_as_float(x1[e]);
      }
      if (MODE == 7) {
        const uint32_t c = trow + 64 + half * 64;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t x0[16], x1[16], x2[16], x3[16];
          tmem_ld16(c + q * 32, x0);
          tmem_ld16(c + q * 32 + 16, x1);
          tmem_ld16(c + q * 32, x2);
          tmem_ld16(c + q * 32 + 16, x3);
          tmem_wait_ld(x0);
          tmem_wait_ld(x1);
          tmem_wait_ld(x2);
          tmem_wait_ld(x3);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            acc += __uint_as_float(x0[e]) + __uint_as_float(x1[e]) + __uint_as_float(x2[e]) + __uint_as_float(x3[e]);
        }
      }
      if (MODE == 1 || MODE == 3) {
        uint32_t x0[32], x1[32], x2[32], x3[32];
        const uint32_t c = trow + 64 + half * 64;  // columns 64..191 (D uses 0..N-1 <= 63)
        tmem_ld32(c, x0);
        tmem_ld32(c + 32, x1);
        tmem_ld32(c, x2);
        tmem_ld32(c + 32, x3);
        tmem_wait_ld(x0);
        tmem_wait_ld(x1);
        tmem_wait_ld(x2);
        tmem_wait_ld(x3);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          acc += __uint_as_float(x0[e]) + __uint_as_float(x1[e]) + __uint_as_float(x2[e]) + __uint_as_float(x3[e]);
      }
      if (MODE == 2 || MODE == 3) {
        uint32_t y[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] = static_cast<uint32_t>(it + e);
        const uint32_t c = trow + 384 + half * 64;  // columns 384..511
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_st16(c + q * 16, y);
        tmem_wait_st();
      }
      if (MODE == 4) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(sm.a);
        uint32_t* dst = reinterpret_cast<uint32_t*>(sm.a) + 4096;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint4 v = reinterpret_cast<const uint4*>(src)[(q * 32 + lane + it) & 1023];
          acc += __uint_as_float(v.x ^ v.y ^ v.z ^ v.w);
          reinterpret_cast<uint4*>(dst)[(q * 32 + lane) & 1023] = v;
        }
      }
      if (MODE == 5) {
#pragma unroll
        for (int q = 0; q < 64; ++q) acc = ex2(acc * -0.5f);
      }
    }
    if (warp == 4 && lane == 0) ccyc[blockIdx.x] = clock64() - c0;
    if (acc == 1234.5f) sink[threadIdx.x] = acc;  // keeps the traffic from being removed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int K>
cudaError_t run_exp(int blocks, int iters, float* sink, long long* cyc, cudaStream_t st) {
  micro_exp<K><<<blocks, 512, 0, st>>>(sink, cyc, iters);
  return cudaGetLastError();
}

template <int N, bool TS>
cudaError_t run_mma_t(int blocks, int reps, int accs, long long* cyc, int* status, cudaStream_t st) {
  switch (accs) {
    case 1: micro_mma<N, TS, 1><<<blocks, 128, 0, st>>>(cyc, reps, status); break;
    case 2: micro_mma<N, TS, 2><<<blocks, 128, 0, st>>>(cyc, reps, status); break;
    case 4:
      if (4 * N > 256) return cudaErrorInvalidValue;
      micro_mma<N, TS, (4 * N <= 256 ? 4 : 1)><<<blocks, 128, 0, st>>>(cyc, reps, status);
      break;
    case 8:
      if (8 * N > 256) return cudaErrorInvalidValue;
      micro_mma<N, TS, (8 * N <= 256 ? 8 : 1)><<<blocks, 128, 0, st>>>(cyc, reps, status);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
template <int N>
cudaError_t run_mma(int ts, int blocks, int reps, int accs, long long* cyc, int* status, cudaStream_t st) {
  if (accs < 1 || accs * N > 256 || reps % 16 != 0) return cudaErrorInvalidValue;
  return ts ? run_mma_t<N, true>(blocks, reps, accs, cyc, status, st)
            : run_mma_t<N, false>(blocks, reps, accs, cyc, status, st);
}

}  // namespace

// Exponential / FMA throughput: `blocks` blocks of 512 threads, each thread running
// `iters` iterations of 8 independent chains of the op `kind` (ExpKind above).
// sink: device float[512] (never written in practice); cycles: device int64[blocks],
// the clock64() span of each block.  Returns a cudaError_t value.
EVO_MICRO_API int evo_micro_exp(int kind, int blocks, int iters, void* sink, void* cycles, void* stream) {
  float* s = static_cast<float*>(sink);
  long long* c = static_cast<long long*>(cycles);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (blocks <= 0 || iters <= 0 || !sink || !cycles) return cudaErrorInvalidValue;
  switch (kind) {
    case kEx2F32: return run_exp<kEx2F32>(blocks, iters, s, c, st);
    case kEx2F16x2: return run_exp<kEx2F16x2>(blocks, iters, s, c, st);
    case kEx2BF16x2: return run_exp<kEx2BF16x2>(blocks, iters, s, c, st);
    case kPoly: return run_exp<kPoly>(blocks, iters, s, c, st);
    case kPoly2: return run_exp<kPoly2>(blocks, iters, s, c, st);
    case kFma: return run_exp<kFma>(blocks, iters, s, c, st);
    case kFma2: return run_exp<kFma2>(blocks, iters, s, c, st);
    case kMix31: return run_exp<kMix31>(blocks, iters, s, c, st);
    default: return cudaErrorInvalidValue;
  }
}

// Small-N MMA operand forms (FORM 0..3 above): `blocks` blocks, `reps` MMAs each
// (a multiple of 16); cycles: device int64[blocks]; status as evo_micro_mma.
EVO_MICRO_API int evo_micro_mma_form(int form, int blocks, int reps, void* cycles, void* status, void* stream) {
  long long* c = static_cast<long long*>(cycles);
  int* s = static_cast<int*>(status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (blocks <= 0 || reps <= 0 || reps % 16 != 0 || !cycles || !status) return cudaErrorInvalidValue;
  const size_t smem = sizeof(FormSmem) + 1024;
  switch (form) {
#define EVO_FORM(F)                                                                              \
  case F: {                                                                                      \
    cudaError_t e = cudaFuncSetAttribute(micro_form<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                         static_cast<int>(smem));                                \
    if (e != cudaSuccess) return e;                                                              \
    micro_form<F><<<blocks, 128, smem, st>>>(c, reps, s);                                        \
    break;                                                                                       \
  }
    EVO_FORM(0)
    EVO_FORM(1)
    EVO_FORM(2)
    EVO_FORM(3)
#undef EVO_FORM
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// P·V MMAs under other warps' traffic (micro_contend): mode 0..5, n 32 or 48; `reps`
// MMAs (a multiple of 16) while the eight other warps run `creps` rounds of traffic.
EVO_MICRO_API int evo_micro_contend(int mode, int n, int ss, int blocks, int reps, int creps, void* cycles,
                                    void* ccycles, void* sink, void* status, void* stream) {
  long long* c = static_cast<long long*>(cycles);
  long long* cc = static_cast<long long*>(ccycles);
  float* sk = static_cast<float*>(sink);
  int* s = static_cast<int*>(status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (blocks <= 0 || reps <= 0 || reps % 16 != 0 || creps < 0 || !cycles || !sink || !status ||
      !ccycles || (n != 32 && n != 48) || mode < 0 || mode > 7)
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ContendSmem) + 1024;
#define EVO_CONT(M, NN, SSF)                                                                      \
  if (mode == M && n == NN && (ss != 0) == SSF) {                                                  \
    auto kern = micro_contend<M, NN, SSF>;                                                         \
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                         static_cast<int>(smem));                                  \
    if (e != cudaSuccess) return e;                                                                \
    kern<<<blocks, 384, smem, st>>>(c, cc, reps, creps, sk, s);                                    \
    return cudaGetLastError();                                                                     \
  }
#define EVO_CONT_N(M) EVO_CONT(M, 32, false) EVO_CONT(M, 48, false) EVO_CONT(M, 32, true) EVO_CONT(M, 48, true)
  EVO_CONT_N(0) EVO_CONT_N(1) EVO_CONT_N(2) EVO_CONT_N(3) EVO_CONT_N(4) EVO_CONT_N(5) EVO_CONT_N(6)
  EVO_CONT_N(7)
#undef EVO_CONT_N
#undef EVO_CONT
  return cudaErrorInvalidValue;
}

// tcgen05.ld cost: `blocks` blocks (one per SM) of four warps, each round `per_wait`
// (1, 2 or 4) x32 loads then one wait; cycles: device int64[blocks] over `reps` rounds.
EVO_MICRO_API int evo_micro_tmem_ld(int per_wait, int blocks, int reps, void* cycles, void* sink, void* stream) {
  long long* c = static_cast<long long*>(cycles);
  float* s = static_cast<float*>(sink);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (blocks <= 0 || reps <= 0 || !cycles || !sink) return cudaErrorInvalidValue;
  switch (per_wait) {
    case 1: micro_tmem_ld<1><<<blocks, 128, 0, st>>>(c, reps, s); break;
    case 2: micro_tmem_ld<2><<<blocks, 128, 0, st>>>(c, reps, s); break;
    case 4: micro_tmem_ld<4><<<blocks, 128, 0, st>>>(c, reps, s); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// tcgen05.mma issue cost: `blocks` blocks (one per SM), each issuing `reps` MMAs of
// M = 128, the given N (32, 64, 128 or 256), K = 16, round robin over `accs`
// independent accumulators (accs * N <= 256); ts != 0 reads A from tensor memory.
// cycles: device int64[blocks]; status: device int, set to 8 if the completion wait
// ran out.  Returns a cudaError_t value.
EVO_MICRO_API int evo_micro_mma(int n, int ts, int accs, int blocks, int reps, void* cycles, void* status,
                                void* stream) {
  long long* c = static_cast<long long*>(cycles);
  int* s = static_cast<int*>(status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (blocks <= 0 || reps <= 0 || !cycles || !status) return cudaErrorInvalidValue;
  switch (n) {
    case 32: return run_mma<32>(ts, blocks, reps, accs, c, s, st);
    case 64: return run_mma<64>(ts, blocks, reps, accs, c, s, st);
    case 128: return run_mma<128>(ts, blocks, reps, accs, c, s, st);
    case 256: return run_mma<256>(ts, blocks, reps, accs, c, s, st);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------- host link
// Copies driven by the SMs: a grid-stride loop of 16-byte loads and stores, for host ↔
// device copies through mapped pinned host memory (against the copy engines' rate).
__global__ void micro_copy16(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += step) dst[i] = src[i];
}

// dst[0 .. bytes) = src[0 .. bytes); both 16-byte aligned device-accessible pointers (device
// memory, or the device pointer of mapped pinned host memory), bytes a multiple of 16.
EVO_MICRO_API int evo_micro_copy(const void* src, void* dst, size_t bytes, int blocks, void* stream) {
  if (!src || !dst || blocks <= 0 || bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(src) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(dst) & 15) != 0)
    return cudaErrorInvalidValue;
  micro_copy16<<<blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(src),
                                                                     static_cast<uint4*>(dst), bytes / 16);
  return cudaGetLastError();
}

// The device pointer of pinned host memory (cudaHostGetDevicePointer); *dev = nullptr and an
// error when the memory is not mapped.
EVO_MICRO_API int evo_micro_host_ptr(void* host, void** dev) {
  *dev = nullptr;
  const cudaError_t e = cudaHostGetDevicePointer(dev, host, 0);
  if (e != cudaSuccess) *dev = nullptr;
  return static_cast<int>(e);
}
