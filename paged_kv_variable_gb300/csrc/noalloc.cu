// Attention entry point that allocates nothing and needs no caller workspace.
//
// Some callers cannot hand the library a device workspace: a host that owns
// all device memory through its own pool and forbids other allocations, code
// that must not call cudaMalloc because it synchronises the device and would
// stall a latency-critical serving loop, or bindings that have no allocator
// at all.  For them this file keeps the scratch the attention call needs (work
// list, split-KV partials, status word) in a fixed device array that every GPU
// loading the library reserves until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace pkv {
namespace {

// The fixed scratch: 32 MiB per device.  A plan whose workspace is larger is
// rejected (split-KV partials dominate: 8 KiB per KV chunk at head_dim 128).
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, resolved once per device.
pkv_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(PKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_attn_varlen_kvcache_fwd_noalloc(const pkv_problem* problem, const pkv_fwd_args* args,
                                                          pkv_plan_t plan, void* stream) {
  // every host check first: a rejected call leaves the shared scratch alone
  pkv_status st = validate_call(problem, args, plan);
  if (st != PKV_OK) return st;
  if (plan->layout.total > kStaticScratchBytes)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL,
                "this plan needs %zu bytes of scratch but the fixed scratch holds %zu bytes; use "
                "pkv_attn_varlen_kvcache_fwd with a caller workspace",
                plan->layout.total, kStaticScratchBytes);
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  st = pkv_plan_upload(plan, scratch, kStaticScratchBytes, stream);
  if (st != PKV_OK) return st;
  return pkv_attn_varlen_kvcache_fwd(problem, args, plan, scratch, kStaticScratchBytes, stream);
}

extern "C" pkv_status pkv_get_status_noalloc(void* stream, int32_t* device_status) {
  if (!device_status) return fail(PKV_ERR_INVALID_ARG, "NULL output");
  void* scratch = nullptr;
  pkv_status st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  // the status word sits at the head of every plan's workspace layout
  return pkv_get_status(scratch, stream, device_status);
}
