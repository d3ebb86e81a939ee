// moe_forward_noalloc: moe_forward for callers that cannot allocate device
// memory, with its scratch in a fixed array inside this library.
//
// Some callers have no way to call cudaMalloc when they run the block: an
// inference engine plugin whose host forbids allocation while a request is
// being served, a real-time loop with a no-allocation rule, or code embedded
// in a framework that owns every device buffer and hands out only inputs and
// outputs.  For them this entry point takes the same inputs and outputs as
// moe_forward but supplies the workspace itself, from the file-scope device
// array below.  It is a convenience wrapper with no counterpart on the pages
// the block follows.
//
// The array is sized for decode-sized batches (up to 144 tokens at
// d = W = 2880, top-4); every GPU that loads the library holds it until the
// process exits.  Every call shares it: calls that overlap on the GPU (on two
// streams, or from two threads) race on the same scratch and must not be
// issued.  Nothing in it needs clearing between calls: each call writes every
// part of the scratch it reads, status word included.
#include "moe.h"

#include <cuda_runtime.h>

#include <mutex>
#include <string>

namespace moe {
void set_last_error(const std::string& msg);   // defined with moe_last_error
}

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

// The scratch.  In host code `g_scratch` is only a host-side stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DevicePtrs {
  std::mutex mu;
  void* ptr[64] = {};
};

DevicePtrs& device_ptrs() {
  static DevicePtrs p;
  return p;
}

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does this set-up).  The cached address
// belongs to the device's current context: after cudaDeviceReset the module is
// loaded again and the array may move, so this library must not be used
// across a reset of a device it has already run on.
moe_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    moe::set_last_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) {
    moe::set_last_error("device ordinal out of range");
    return MOE_ERR_UNSUPPORTED;
  }
  DevicePtrs& p = device_ptrs();
  std::lock_guard<std::mutex> lock(p.mu);
  if (!p.ptr[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_scratch);
    if (e != cudaSuccess || !a) {
      moe::set_last_error(std::string("cudaGetSymbolAddress of the scratch array: ") +
                          cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    p.ptr[dev] = a;
  }
  *out = p.ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward_noalloc(const void* x_bf16, int64_t T, int d, int W,
                               const float* router_w, const float* router_b,
                               const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale,
                               const void* b_gu_bf16, const uint8_t* w_dn_fp4,
                               const uint8_t* w_dn_scale, const void* b_dn_bf16, int E, int k,
                               float limit, float alpha, void* out_bf16, void* stream) {
  if (T == 0) {
    // nothing to run, but the arguments get moe_forward's checks (shape,
    // alignment, NaN clamp); no scratch is needed for them
    return moe_forward(x_bf16, T, d, W, router_w, router_b, w_gu_fp4, w_gu_scale, b_gu_bf16,
                       w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16, nullptr, 0,
                       stream);
  }
  const size_t need = moe_workspace_bytes(T, d, W, E, k);
  if (need == 0) return MOE_ERR_SHAPE;   // invalid shape; moe_last_error() says which
  if (need > kScratchBytes) {
    moe::set_last_error("moe_forward_noalloc: this shape needs " + std::to_string(need) +
                        " bytes of scratch but the built-in array holds " +
                        std::to_string(kScratchBytes) +
                        " (up to 144 tokens at d = W = 2880, k = 4); use moe_forward with a"
                        " workspace");
    return MOE_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  return moe_forward(x_bf16, T, d, W, router_w, router_b, w_gu_fp4, w_gu_scale, b_gu_bf16,
                     w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16, scratch,
                     kScratchBytes, stream);
}

moe_status moe_poll_status_noalloc(void* stream) {
  void* scratch = nullptr;
  const moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  // the status word is the first word of the scratch, as of any workspace
  return moe_poll_status(scratch, stream);
}

}  // extern "C"
