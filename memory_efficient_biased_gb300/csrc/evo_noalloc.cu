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

#include <atomic>
#include <mutex>

#include "evo_attn.h"

namespace evo {
evo_status_t cuda_fail(const char* what, cudaError_t e);  // evo_host.cu: records the last-error text
}

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[EVO_NOALLOC_SCRATCH_BYTES];

struct ScratchSlot {
  std::mutex lock;
  std::atomic<void*> ptr{nullptr};
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the scratch array on the current device, looked up with that
// device current.  Only a successful lookup is kept: a failed one (for instance the
// device out of memory when lazy module loading reserves the array at this first
// use) is reported and tried again by the next call.
evo_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return evo::cuda_fail("noalloc scratch: cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return evo::cuda_fail("noalloc scratch: device index", cudaErrorInvalidDevice);
  ScratchSlot& s = g_slots[dev];
  void* p = s.ptr.load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> g(s.lock);
    p = s.ptr.load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return evo::cuda_fail("noalloc scratch lookup (cudaGetSymbolAddress)", e);
      s.ptr.store(p, std::memory_order_release);
    }
  }
  *out = p;
  return EVO_OK;
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
  void* scratch = nullptr;
  const evo_status_t st = scratch_on_current_device(&scratch);
  if (st != EVO_OK) return st;
  // The backward writes every scratch byte before it reads it (the first key tile of a
  // slice stores its dQ rows, later ones add to them), so stale contents from an
  // earlier call are harmless.
  return evo_attn_bwd(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, dbias2, scratch,
                      EVO_NOALLOC_SCRATCH_BYTES, shape, dtype, stream);
}
