// evo_noalloc.cu — evo_attn_bwd_noalloc: the backward for callers that
// cannot allocate device memory (see include/evo_attn.h).
//
// The scratch lives in a fixed file-scope device array instead of a
// caller-provided workspace.  This file is its own module, so the array is
// only reserved on a GPU once this entry point is first used there.  Host
// code never passes the array's name to a kernel (on the host the name is a
// stand-in, not a device address); it passes the device address that
// cudaGetSymbolAddress returns for the current device.
#include <cuda_runtime.h>

#include <mutex>

#include "evo_attn.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[EVO_NOALLOC_SCRATCH_BYTES];

struct ScratchSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  ScratchSlot& s = g_slots[dev];
  std::call_once(s.once, [&s]() {
    void* p = nullptr;
    s.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (s.err == cudaSuccess) s.ptr = p;
  });
  return s.err == cudaSuccess ? s.ptr : nullptr;
}

}  // namespace

extern "C" evo_status_t evo_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* bias1,
                                             const void* bias2, const void* out, const float* lse,
                                             const void* dout, void* dq, void* dk, void* dv, void* dbias2,
                                             evo_shape_t shape, evo_dtype_t dtype, void* stream) {
  if (dtype != EVO_F16 && dtype != EVO_BF16) return EVO_ERR_BAD_DTYPE;
  const size_t need = evo_attn_bwd_workspace_bytes(shape, dtype, bias2 != nullptr);
  if (need == 0) return EVO_ERR_BAD_SHAPE;
  if (need > EVO_NOALLOC_SCRATCH_BYTES) return EVO_ERR_SCRATCH_LIMIT;
  void* scratch = scratch_on_current_device();
  if (!scratch) return EVO_ERR_CUDA;
  // The backward clears its dQ accumulator itself and overwrites every other
  // scratch byte it reads, so stale contents from an earlier call are harmless.
  return evo_attn_bwd(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, dbias2, scratch,
                      EVO_NOALLOC_SCRATCH_BYTES, shape, dtype, stream);
}
