// lora_linear_fused_noalloc: the fused layer for callers that cannot
// allocate device memory.
//
// Some callers of this library have no way to hand it a workspace.  Code
// running inside a framework whose allocator already owns all device memory
// (a serving engine that reserved the rest of HBM for KV cache), plugins that
// the host process does not allow to allocate, and real-time paths that
// forbid allocation after start-up all fall in this group.  For them this
// entry point keeps its scratch (error word, segment arrays, shrink partials)
// in a fixed array that lives in the library itself, sized
// LORA_NOALLOC_SCRATCH_BYTES, and otherwise runs exactly lora_linear_fused.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "lora.h"

namespace {

// The scratch lives here.  Its device memory is committed when the library's
// device code is loaded on a GPU: with CUDA's lazy module loading (the
// default) that is the first lookup of the address below, i.e. the first
// call on that device; with CUDA_MODULE_LOADING=EAGER it is when the process
// first uses that GPU.  It is held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LORA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code
// the array's name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
lora_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return LORA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_linear_fused_noalloc(const void* x, const void* W0,
                                                   const void* A_pool, const void* B_pool,
                                                   const int32_t* slot_ids, const float* scale,
                                                   void* y, int32_t T, int32_t d_in,
                                                   int32_t d_out, int32_t r, int32_t n_slots,
                                                   lora_dtype_t dt, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  // batches whose scratch does not fit the fixed array are refused up front
  const size_t need = lora_workspace_bytes(LORA_OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots);
  if (need > LORA_NOALLOC_SCRATCH_BYTES) return LORA_ERR_WORKSPACE;
  void* scratch = nullptr;
  lora_status_t s = scratch_for_current_device(&scratch);
  if (s != LORA_OK) return s;
  // the error word must start at zero (everything else is overwritten); it
  // is cleared only once every argument has been validated, so a refused
  // call enqueues nothing at all
  return lora::linear_fused_impl(x, W0, A_pool, B_pool, slot_ids, scale, y, T, d_in, d_out, r,
                                 n_slots, dt, scratch, LORA_NOALLOC_SCRATCH_BYTES, stream, true);
}
