// route_noalloc.cu - moe_route_noalloc: router logits, top-k selection and
// renormalised routing weights without a handle and without allocating.
//
// The routing arithmetic is the forward's own: the kernels moe_forward runs
// above 64 tokens (router_logits_kernel, topk_kernel); at or below 64 tokens
// moe_forward forms the logits inside front_small_kernel in the same
// canonical FP32 order and selects with the same warp top-k, so the result is
// bit-identical to the routing moe_forward computes.  The only difference is
// where the intermediate lives: the FP32 logits [T, E] go to one file-scope
// device array of fixed size instead of a handle's workspace.
//
// The first call on a device does the set-up for that device (looks the
// array's address up and raises the router kernel's shared-memory cap).  With
// CUDA's lazy module loading, that look-up is also what loads this file's
// device code on the device and so reserves the array there; the first call
// should therefore come before any stream capture, and before a memory pool
// claims the device's free memory.  Calls whose work overlaps on one
// device share the array and race: order them on one stream.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe_nvfp4.h"

static constexpr size_t LOGITS_BYTES = sizeof(float) * (size_t)MOE_ROUTE_NOALLOC_MAX_LOGITS;

// The whole scratch of the routing: the logits, MOE_ROUTE_NOALLOC_MAX_LOGITS
// floats (4 MiB).  One copy per device, created when the library's device
// code is loaded on that device.
static __device__ __align__(256) unsigned char g_route_scratch[LOGITS_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceScratch {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_route_scratch on this device
  int smem_cap = 0;               // router shared-memory cap raised at set-up
};

std::mutex g_setup_mutex;
DeviceScratch g_devices[MAX_DEVICES];

// Once per device, with that device current: look up the array's address on
// it and raise the router kernel's shared-memory cap to the device's opt-in
// maximum (raised only, so handles created later cannot lower it).
moe_status setup_current_device(const DeviceScratch** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceScratch& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
    void* base = nullptr;
    if (cudaGetSymbolAddress(&base, g_route_scratch) != cudaSuccess || base == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    if (moe::router_setup_max(optin) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    d.base = static_cast<unsigned char*>(base);
    d.smem_cap = optin;
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" {

moe_status moe_route_noalloc(const void* x, const void* gate_w, const float* gate_bias, int num_tokens, int hidden,
                             int num_experts, int top_k, int32_t* topk_ids, float* topk_w, void* stream) {
  const int T = num_tokens, H = hidden, E = num_experts, K = top_k;
  if (T < 0 || H <= 0 || E <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 256 || E % 8 || E > 256 || K > E || K > 16) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * E > MOE_ROUTE_NOALLOC_MAX_LOGITS) return MOE_ERR_TOO_MANY_TOKENS;
  const DeviceScratch* d = nullptr;
  const moe_status st = setup_current_device(&d);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x || !gate_w || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(gate_w) || (gate_bias && !aligned16(gate_bias))) return MOE_ERR_INVALID_ARG;
  if (moe::router_smem_bytes(H, E) > d->smem_cap) return MOE_ERR_UNSUPPORTED;

  float* logits = reinterpret_cast<float*>(d->base);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = moe::launch_router_logits(x, gate_w, gate_bias, logits, T, H, E, s);
  if (e == cudaSuccess) e = moe::launch_topk(logits, T, E, K, topk_ids, topk_w, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // extern "C"
