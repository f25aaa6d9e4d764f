// nystrom_attn_fwd_noalloc: the forward pass for callers that cannot
// allocate device memory (declared in include/nystrom.h). Its scratch is a
// fixed file-scope device array instead of a cudaMalloc'd workspace.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "nys_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// The scratch itself. Every device that loads this library reserves it for
// the life of the process. In host code `g_noalloc_scratch` names a host-side
// stand-in, never a device address: the device address comes from
// cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on device `dev` (which is current).
// Looked up once per device; later calls reuse it.
int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return nys::set_cuda_error(e);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return NYS_OK;
}

}  // namespace

extern "C" int nystrom_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                        const float* conv_w, void* out, int B, int H, int n,
                                        int d, int m, int iters, int conv_ks, int dtype,
                                        nys_stream_t stream) {
  int rc = nys::check_args(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  nys::Shape s{B, H, n, d, m, iters, conv_ks, dtype};
  if (nys::make_layout(s).total > kNoAllocScratchBytes) return NYS_ERR_NOMEM;
  int dev = 0;
  rc = nys::check_device(&dev);
  if (rc != NYS_OK) return rc;
  if (dev >= kMaxDevices) return NYS_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  rc = scratch_address(dev, &scratch);
  if (rc != NYS_OK) return rc;
  return nys::run(s, q, k, v, conv_w, out, static_cast<char*>(scratch), stream, dev);
}
