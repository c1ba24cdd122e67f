// tva_noalloc.cu - tree_verify_attn_varlen_noalloc: the batched attention for callers
// that may not allocate device memory.
//
// Some callers cannot hand this library a workspace: code running inside a host
// engine that owns every device allocation and forbids cudaMalloc (or its own pool)
// on its execution path, plugins whose per-call interface has no workspace argument,
// and latency-critical loops that must not risk an allocation.  For them the
// partials this path needs live in one fixed array in this file, held on each GPU
// until the process exits.  The array is reserved when this file's module is loaded
// on a device: under CUDA's default lazy module loading (this module has no kernels)
// that is the first cudaGetSymbolAddress below, i.e. the entry point's first call on
// the device, which then fails with TVA_ERR_CUDA if the device has no 32 MiB left;
// with CUDA_MODULE_LOADING=EAGER it is when the library's device code is loaded.
#include <cstdio>
#include <mutex>

#include "tva.h"
#include "tva_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB per GPU

// The scratch.  In host code this name is only a stand-in for the device symbol, never
// a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
void* scratch_on_current_device() {
  int dev = 0;
  if (tva::check_cuda(cudaGetDevice(&dev), "cudaGetDevice") != cudaSuccess || dev < 0 ||
      dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (tva::check_cuda(cudaGetSymbolAddress(&p, g_static_scratch),
                        "cudaGetSymbolAddress(static scratch)") != cudaSuccess)
      return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" tva_status tree_verify_attn_varlen_noalloc(const tva_params* p, const void* q,
                                                      const void* k_cache, const void* v_cache,
                                                      const void* tree_k, const void* tree_v,
                                                      const int32_t* parent, void* out, float* lse,
                                                      int32_t* dev_status, void* stream) {
  if (p == nullptr) return TVA_ERR_INVALID_ARG;
  const size_t need = tva_workspace_size(p);
  if (need > kStaticScratchBytes) {
    char what[128];
    snprintf(what, sizeof(what), "problem needs %zu bytes of scratch, the static buffer holds %zu",
             need, kStaticScratchBytes);
    tva::record_error("tree_verify_attn_varlen_noalloc", 0, what);
    return TVA_ERR_WORKSPACE;
  }
  void* ws = scratch_on_current_device();
  if (ws == nullptr) return TVA_ERR_CUDA;
  // Invalid parameters (need == 0) are reported by the workspace form's own checks.
  return tree_verify_attn_varlen(p, q, k_cache, v_cache, tree_k, tree_v, parent, out, lse, ws,
                                 kStaticScratchBytes, dev_status, stream);
}
