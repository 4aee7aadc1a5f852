// noalloc.cu -- moe_forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run the MoE layer: code inside a plugin or serving engine
// whose device memory is owned and pre-carved by the host framework, loops
// that must not allocate after start-up (allocation can block, synchronise
// the device or fail under memory pressure), and callers that cannot hold a
// workspace of their own.  For them this file keeps the forward's scratch in
// one statically sized device array that is part of the library itself.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it (MOE_STATIC_SCRATCH_BYTES each).  Its device address is looked up
// once per device, with that device current, the first time this entry point
// runs there.  Every call on a device shares the same array and finds the
// previous call's intermediates in it; the forward clears the one word that
// must start at zero (its status word).  Calls that overlap on the GPU (on
// different streams, or from several host threads without ordering) race on
// the array and must not be issued.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[MOE_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_forward_noalloc(const moe_problem_t* p, const void* x, const int32_t* topk_ids,
                                   const float* topk_weights, const void* w13,
                                   const uint8_t* w13_scale, const void* w2,
                                   const uint8_t* w2_scale, void* out, void* stream) {
  // the same argument checks, and so the same status codes, as moe_forward;
  // the size limit of the static array comes after them
  int rc = moe::validate_forward_problem(p);
  if (rc != MOE_OK) return rc;
  if (moe_workspace_size(p) > static_cast<size_t>(MOE_STATIC_SCRATCH_BYTES))
    return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_forward(p, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, out, scratch,
                     static_cast<size_t>(MOE_STATIC_SCRATCH_BYTES), stream);
}

// The status word of the last moe_forward_noalloc on the current device
// sits at offset 0 of the static array (moe_forward's workspace layout puts
// it first).  Reading it needs the array's device address, which only this
// file knows, and a copy of 4 bytes to the host: nothing is allocated.
extern "C" int moe_forward_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_get_device_status(static_cast<const int32_t*>(scratch), stream);
}
